// microbench.cu -- instruction throughput probes for the attention kernel's
// building blocks on sm_103a, after the method of "Kernel Bottleneck Tuning",
// section "1. Measure instruction throughputs in isolation": 8 independent
// dependency chains per thread, results fed back so the loop cannot be
// hoisted, %clock64 around the timed loop with a memory clobber.
//
// fmha_microbench_alu(which): 0 ex2.approx.ftz.f32, 1 cvt.rn.bf16x2.f32,
//   2 fma.rn.f32x2 (512 threads per SM); 3 the softmax exp loop of one
//   128-score row per thread, 4 ex2 alone (128 threads per SM).
// fmha_microbench_mma(...): back-to-back tcgen05.mma kind::f16 M=128 from
//   `issuers` warps, each rotating nothing (one accumulator per issuer):
//   a_tmem   0 = A from shared memory (SS), 1 = A from tensor memory (TS)
//   b_mn     B stored MN-major (as V in O += P V) instead of K-major
//   n        64, 128 or 256
//   uniform  1 = the whole warp runs the loop and one lane issues through a
//              predicate (warp-uniform operands); 0 = lane 0 inside a branch
// fmha_microbench_tmem_ld: tcgen05.ld 32x32b.x32 + wait, 4 warps.
// fmha_microbench_mma_mix / _boundary / _handoff / _pingpong: the attention
//   kernel's MMA stream, the issuing thread's cost at a step boundary,
//   barrier hand-off latency while MMAs run, and two alternating issuers
//   (each documented at its kernel below).
// fmha_microbench_empty_launch: an empty one-wave kernel, for the launch
//   envelope inside a pair of timing events.
// Each writes the per-CTA cycle count of its timed region to out_cycles
// (host memory, n_ctas entries) and returns 0, 1 on a bad argument, 2 on a
// CUDA error, 3 if a completion wait expired (bounded at 1 s).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "sm103_ptx.cuh"

namespace {

using namespace fmha;

// Probe-only arithmetic (the attention kernel does not use these).
namespace ptx_probe {
// 2^x of a pair on the FMA pipe instead of the MUFU: range reduction
// 2^x = 2^n * 2^f with n = round(x), f = x - n in [-0.5, 0.5] (n taken from
// the low mantissa bits of x + 1.5 * 2^23), and 2^f from a degree-3
// polynomial whose coefficients were fitted here for minimal relative error
// on [-0.5, 0.5] (Lawson-weighted least squares; max relative error 7.5e-5,
// below half a bf16 ulp by a factor of 26).  x is clamped at -126, where 2^x
// is below every normal fp32.
__device__ __forceinline__ float2 exp2_poly2(float2 x) {
  x.x = fmaxf(x.x, -126.f);
  x.y = fmaxf(x.y, -126.f);
  const float2 t = __fadd2_rn(x, make_float2(12582912.f, 12582912.f));
  const float2 n = __fadd2_rn(t, make_float2(-12582912.f, -12582912.f));
  const float2 f = __ffma2_rn(n, make_float2(-1.f, -1.f), x);
  float2 p = __ffma2_rn(make_float2(0.0551716648f, 0.0551716648f), f, make_float2(0.242611125f, 0.242611125f));
  p = __ffma2_rn(p, f, make_float2(0.693260968f, 0.693260968f));
  p = __ffma2_rn(p, f, make_float2(0.999928057f, 0.999928057f));
  const uint32_t bx = __float_as_uint(p.x) + (__float_as_uint(t.x) << 23);
  const uint32_t by = __float_as_uint(p.y) + (__float_as_uint(t.y) << 23);
  return make_float2(__uint_as_float(bx), __uint_as_float(by));
}

// Two fp32 values -> packed f16x2 (round to nearest), lo in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// 2^x of both halves of a packed f16x2 (one MUFU instruction for two values).
__device__ __forceinline__ uint32_t ex2_approx_f16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Packed f16x2 -> two fp32 (lo = low half).
__device__ __forceinline__ float2 unpack_f16x2(uint32_t h) {
  float lo, hi;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
  return make_float2(lo, hi);
}

// bf16x2 pack by integer rounding (round half up on the magnitude): the
// alternative to cvt.rn.bf16x2.f32 that the exp-loop probe compares.
__device__ __forceinline__ uint32_t pack_bf16x2_alu(float lo, float hi) {
  return __byte_perm(__float_as_uint(lo) + 0x8000u, __float_as_uint(hi) + 0x8000u, 0x7632);
}
}  // namespace ptx_probe

constexpr int kAluThreads = 512;
constexpr int kTcThreads = 128;
// shared memory: zeroed A tile (32 KiB) and B tile (64 KiB), barriers
constexpr uint32_t kMbA = 0, kMbB = 32768, kMbBar = 32768 + 65536, kMbSmem = kMbBar + 128 + 1024;

__global__ void __launch_bounds__(kAluThreads, 1) alu_probe(int which, int reps, long long* out, float* sink) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = 0.001f * (threadIdx.x + i);
  float2 w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = make_float2(v[i], v[i] + 1.f);
  __syncthreads();
  long long t0, t1;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0)::"memory");
  if (which == 0) {
    for (int r = 0; r < reps; ++r) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = ptx::ex2_approx(v[i]) * -0.5f;
    }
  } else if (which == 1) {
    for (int r = 0; r < reps; ++r) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t d = ptx::pack_bf16x2(v[i], v[i]);
        v[i] = __uint_as_float((d & 0xffff0000u) ^ 0x00800000u);
      }
    }
  } else {
    const float2 a = make_float2(0.999f, 0.999f), c = make_float2(1e-3f, 1e-3f);
    for (int r = 0; r < reps; ++r) {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = __ffma2_rn(w[i], a, c);
    }
  }
  __syncthreads();
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1)::"memory");
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc += v[i] + w[i].x + w[i].y;
  sink[blockIdx.x * kAluThreads + threadIdx.x] = acc;
  if (threadIdx.x == 0) out[blockIdx.x] = t1 - t0;
}

// The attention softmax's exp loop in isolation, 128 threads (one warp per SM
// sub-partition, as in the kernel): per row 128 scores -> one packed FMA per
// pair, two ex2, packed row-sum add, bf16x2 pack; the packed P goes to shared
// memory so nothing is dead code.  which 3: as is; which 4: ex2 only at one
// warp per sub-partition (8 chains).
__global__ void __launch_bounds__(128, 1) softmax_exp_probe(int which, int reps, long long* out, float* sink) {
  __shared__ uint32_t sp[128 * 65];
  float s[128];
#pragma unroll
  for (int k = 0; k < 128; ++k) s[k] = 0.01f * ((threadIdx.x * 7 + k * 13) & 255) - 1.f;
  const float c = 0.1275f, neg_mc = -1.5f;
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = 0.001f * (threadIdx.x + i);
  __syncthreads();
  long long t0, t1;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0)::"memory");
  if (which == 3) {
    const float2 c2 = make_float2(c, c), nm2 = make_float2(neg_mc, neg_mc);
    for (int r = 0; r < reps; ++r) {
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float2 x = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), c2, nm2);
        const float p0 = ptx::ex2_approx(x.x);
        const float p1 = ptx::ex2_approx(x.y);
        acc[i & 3] = __fadd2_rn(acc[i & 3], make_float2(p0, p1));
        sp[threadIdx.x * 65 + i] = ptx::pack_bf16x2(p0, p1);
      }
      s[r & 127] += 1e-7f;  // the next repetition depends on this one
    }
  } else {
    for (int r = 0; r < reps; ++r) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = ptx::ex2_approx(v[i]) * -0.5f;
    }
  }
  __syncthreads();
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1)::"memory");
  float a = acc[0].x + acc[1].y + acc[2].x + acc[3].y + static_cast<float>(sp[threadIdx.x * 65 + 3] & 1u);
#pragma unroll
  for (int i = 0; i < 8; ++i) a += v[i];
  sink[blockIdx.x * 128 + threadIdx.x] = a;
  if (threadIdx.x == 0) out[blockIdx.x] = t1 - t0;
}

// Variants of the exp loop, `threads` = 128 (one warp per sub-partition, as
// the kernel) or 256 (two): per repetition each thread turns 128 scores into
// 64 packed pairs.  variant 0: packed FMA, two ex2, packed row-sum add,
// cvt.rn bf16x2 pack; 1: without the pack; 2: ex2 + row sum only (no FMA, no
// pack; hoisted by the compiler, not meaningful); 3: without the ex2 (FMA,
// sum, pack); 4: as 0 with the integer pack; 5: the pair's exponent in f16x2
// (one packed ex2 for two scores, then back to fp32 for the sum and the bf16
// pack); 6: packed f16x2 ex2 alone, 8 chains, 64 per repetition; 7: as 0 with
// one pair in four on the FMA pipe (exp2_poly2); 8: one pair in eight.
// Packed words go to shared memory as 16-byte vectors; the offset the scores
// are shifted by changes every repetition so nothing is hoisted.
template <int variant, int threads>
__global__ void __launch_bounds__(threads, 1) exp_loop_probe(int reps, long long* out, float* sink) {
  __shared__ uint4 sp[threads * 8];
  float s[128];
#pragma unroll
  for (int k = 0; k < 128; ++k) s[k] = 0.01f * ((threadIdx.x * 7 + k * 13) & 255) - 1.f;
  const float c = 0.1275f;
  float neg_mc = -1.5f;
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  uint32_t hv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) hv[i] = 0x3c00bc00u + threadIdx.x + i;  // (-1, 1) and nearby
  __syncthreads();
  long long t0, t1;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0)::"memory");
  const float2 c2 = make_float2(c, c);
  if (variant == 6) {
    for (int r = 0; r < reps; ++r) {
#pragma unroll
      for (int rep8 = 0; rep8 < 8; ++rep8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) hv[i] = ptx_probe::ex2_approx_f16x2(hv[i]) ^ 0x80008000u;
      }
    }
  }
  for (int r = 0; r < (variant == 6 ? 0 : reps); ++r) {
    const float2 nm2 = make_float2(neg_mc, neg_mc);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      uint32_t pk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = 8 * q + 2 * i;
        float2 x = make_float2(s[k], s[k + 1]);
        if (variant != 2) x = __ffma2_rn(x, c2, nm2);
        float p0 = x.x, p1 = x.y;
        if ((variant == 7 && i == 3) || (variant == 8 && i == 3 && (q & 1))) {
          const float2 e = ptx_probe::exp2_poly2(x);
          p0 = e.x;
          p1 = e.y;
        } else if (variant == 5) {
          const float2 e = ptx_probe::unpack_f16x2(ptx_probe::ex2_approx_f16x2(ptx_probe::pack_f16x2(x.x, x.y)));
          p0 = e.x;
          p1 = e.y;
        } else if (variant != 3) {
          p0 = ptx::ex2_approx(x.x);
          p1 = ptx::ex2_approx(x.y);
        }
        acc[i] = __fadd2_rn(acc[i], make_float2(p0, p1));
        if (variant == 4)
          pk[i] = ptx_probe::pack_bf16x2_alu(p0, p1);
        else
          pk[i] = ptx::pack_bf16x2(p0, p1);
      }
      if (variant != 1 && variant != 2) sp[threadIdx.x * 8 + (q & 7)] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    neg_mc += 1e-7f;
  }
  __syncthreads();
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1)::"memory");
  const uint4 w = sp[threadIdx.x * 8 + 3];
  sink[blockIdx.x * threads + threadIdx.x] = acc[0].x + acc[1].y + acc[2].x + acc[3].y +
                                             static_cast<float>((w.x ^ w.w ^ hv[0] ^ hv[5]) & 1u);
  if (threadIdx.x == 0) out[blockIdx.x] = t1 - t0;
}

// Shared set-up of the tensor-core probes: zero the operand tiles, init one
// barrier per warp, allocate all 512 TMEM columns.
__device__ __forceinline__ uint32_t tc_setup(uint8_t* smem, uint32_t base) {
  uint32_t* z = reinterpret_cast<uint32_t*>(smem);
  for (uint32_t i = threadIdx.x; i < kMbBar / 4; i += kTcThreads) z[i] = 0u;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kMbBar + 64);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) ptx::mbar_init(base + kMbBar + 8u * i, 1);
    ptx::fence_mbar_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // zeros visible to the tensor core
  if ((threadIdx.x >> 5) == 0) {
    ptx::tmem_alloc(ptx::smem_addr(tslot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  return *tslot;
}

__device__ __forceinline__ void tc_teardown(uint32_t tmem) {
  ptx::tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

__device__ __forceinline__ bool bounded_wait(uint32_t bar) {
  const uint64_t g0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, 0))
    if (ptx::globaltimer_ns() - g0 > 1000000000ull) return false;
  return true;
}

template <int a_tmem, int b_mn, int n, int uniform>
__global__ void __launch_bounds__(kTcThreads, 1) mma_probe(int issuers, int reps, long long* out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t tmem = tc_setup(smem, base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long t0 = 0, t1 = 0;
  const bool issuer_warp = warp < issuers;
  if (issuer_warp && (uniform || lane == 0)) {
    const uint32_t leader = lane == 0 ? 1u : 0u;
    // accumulators: issuer w owns columns [w * n, (w + 1) * n) (below 384);
    // a TMEM A operand sits at columns [448, 512)
    const uint32_t d = tmem + static_cast<uint32_t>(warp * n);
    const uint32_t idesc = ptx::idesc_bf16_f32(128, n, false, b_mn != 0);
    const uint64_t a0 = ptx::smem_desc_sw128(base + kMbA, 16, 1024);
    // B: K-major rows of 128 bytes (n rows, 8-row groups 1024 apart, 16 KiB
    // per 64 K) or MN-major (64-wide atoms 16 KiB apart, 16 K rows per step)
    const uint64_t b0 = b_mn ? ptx::smem_desc_sw128(base + kMbB, 16384, 1024)
                             : ptx::smem_desc_sw128(base + kMbB, 16, 1024);
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0)::"memory");
    for (int r = 0; r < reps; ++r) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint64_t a_off = ((k >> 2) * 16384u + (k & 3) * 32u) >> 4;
        const uint64_t b_off = b_mn ? ((2048u * k) >> 4) : (((k >> 2) * (n * 128u) + (k & 3) * 32u) >> 4);
        if (uniform) {
          if (a_tmem)
            ptx::mma_ts_leader(d, tmem + 448u + 8u * k, b0 + b_off, idesc, 1u, leader);
          else
            ptx::mma_ss_leader(d, a0 + a_off, b0 + b_off, idesc, 1u, leader);
        } else {
          if (a_tmem)
            ptx::mma_ts(d, tmem + 448u + 8u * k, b0 + b_off, idesc, 1u);
          else
            ptx::mma_ss(d, a0 + a_off, b0 + b_off, idesc, 1u);
        }
      }
    }
    const uint32_t bar = base + kMbBar + 8u * warp;
    if (uniform)
      ptx::mma_commit_leader(bar, leader);
    else
      ptx::mma_commit(bar);
    if (!bounded_wait(bar)) status[0] = 1;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1)::"memory");
  }
  __syncwarp();
  tc_teardown(tmem);
  if (threadIdx.x == 0) out[blockIdx.x] = t1 - t0;
}

// Issuing-thread cost of the step boundary: each round issues the 16 MMAs of
// one tile group (8 PV + 8 QK^T), then mode 0: tcgen05.commit then
// mbarrier.try_wait on an already-completed barrier; 1: the try_wait alone;
// 2: the commit alone.  Modes 3-5: the same three after 16 MMAs of N=256
// (128 cycles each, so more work is still in flight at the boundary).
// Mode 6: mode 0 while warps 1-3 poll (try_wait, every lane) a barrier that
// never completes; 7: mode 0 while warps 1-3 wait for each commit's phase of
// the committed barrier (as softmax warps wait for S); 8: the commit then a
// dependent shared-memory load instead of the try_wait.
// Returns the summed cycles of that boundary sequence.
template <int mode>
__global__ void __launch_bounds__(kTcThreads, 1) boundary_probe(int reps, long long* out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t tmem = tc_setup(smem, base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile uint32_t* done_flag = reinterpret_cast<volatile uint32_t*>(smem + kMbBar + 96);
  if (threadIdx.x == 0) *done_flag = 0u;
  __syncthreads();
  long long acc = 0;
  if (mode == 6 && warp > 0) {
    const uint64_t g0 = ptx::globaltimer_ns();
    while (*done_flag == 0u && ptx::globaltimer_ns() - g0 < 1000000000ull)
      if (ptx::mbar_try_wait(base + kMbBar + 16u, 0)) status[0] = 1;  // never completes
  } else if (mode == 7 && warp > 0) {
    for (int r = 0; r < reps; ++r) {
      const uint64_t g0 = ptx::globaltimer_ns();
      bool ok = true;
      while (!ptx::mbar_try_wait(base + kMbBar + 8u, static_cast<uint32_t>(r & 1)))
        if (ptx::globaltimer_ns() - g0 > 1000000000ull) {
          ok = false;
          break;
        }
      if (!ok) {
        status[0] = 1;
        break;
      }
    }
  } else if (warp == 0 && lane == 0) {
    const uint32_t done_bar = base + kMbBar + 24u;
    ptx::mbar_arrive(done_bar);  // count 1: phase 0 completes now
    const uint32_t id_qk = ptx::idesc_bf16_f32(128, 128, false, false);
    const uint32_t id_pv = ptx::idesc_bf16_f32(128, 128, false, true);
    const uint64_t q0 = ptx::smem_desc_sw128(base + kMbA, 16, 1024);
    const uint64_t k0 = ptx::smem_desc_sw128(base + kMbB, 16, 1024);
    const uint64_t v0 = ptx::smem_desc_sw128(base + kMbB + 32768u, 16384, 1024);
    int fails = 0;
    const uint32_t id_wide = ptx::idesc_bf16_f32(128, 256, false, false);
    for (int r = 0; r < reps; ++r) {
      if (mode < 3) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          ptx::mma_ts(tmem + 256u, tmem + 8u * k, v0 + ((2048u * k) >> 4), id_pv, 1u);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t off = ((k >> 2) * 16384u + (k & 3) * 32u) >> 4;
          ptx::mma_ss(tmem, q0 + off, k0 + off, id_qk, k > 0 ? 1u : 0u);
        }
      } else {
        // D = columns [0, 256); B = 256 K-major rows (the whole 64 KiB B tile)
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint64_t a_off = (((k & 7) >> 2) * 16384u + (k & 3) * 32u) >> 4;
          const uint64_t b_off = (((k & 7) >> 2) * 32768u + (k & 3) * 32u) >> 4;
          ptx::mma_ss(tmem, q0 + a_off, k0 + b_off, id_wide, k > 0 ? 1u : 0u);
        }
      }
      long long a, b;
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(a)::"memory");
      if (mode != 1 && mode != 4) ptx::mma_commit(base + kMbBar + 8u);
      if (mode == 8) {
        if (*done_flag != 0u) ++fails;
      } else if (mode != 2 && mode != 5 && !ptx::mbar_try_wait(done_bar, 0)) {
        ++fails;
      }
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(b)::"memory");
      acc += b - a;
    }
    const uint32_t bar = base + kMbBar;
    ptx::mma_commit(bar);
    if (!bounded_wait(bar) || fails) status[0] = 1;
    *done_flag = 1u;
  }
  __syncwarp();
  tc_teardown(tmem);
  if (threadIdx.x == 0) out[blockIdx.x] = acc;
}

// The attention kernel's MMA stream without its waits: per tile t (0, 1) a
// group of 8 PV MMAs (A = P from TMEM columns [128 t, 128 t + 64), B = V
// MN-major) into O_t at columns 256 + 128 t, then 8 QK^T MMAs (A = Q, B = K,
// both K-major in shared memory) into S_t at columns 128 t.  mode 0: that
// stream; 1: only the QK^T MMAs; 2: only the PV MMAs; 3: the stream while
// warps 1-3 write 16-byte vectors to a separate shared-memory buffer (TMA-like
// write traffic) until the issuer is done; 4: tile 0's stream only while warps
// 1-3 load TMEM columns [128, 256) and store columns [384, 512), which no MMA
// of this mode touches (softmax-like TMEM traffic); 5: tile 0's stream alone;
// 6: the two-tile stream with a tcgen05.commit after every 8 MMAs (as the
// kernel signals S ready and frees ring slots); 7: a commit after every MMA;
// 8: one commit per 32 MMAs; 9: tile 0's QK^T only, a commit after every 8.
// 10: the stream of mode 0 on random operands (bf16 of magnitude [0.5, 4)
// and random sign in Q, K and V, so S and P are random too) instead of zeros;
// 11: mode 1 on random operands.
// In-loop commits go to a barrier nobody waits on.  P and S share columns
// exactly as in the kernel (the next QK^T of a tile follows its PV).
template <int mode>
__global__ void __launch_bounds__(kTcThreads, 1) mma_mix_probe(int reps, long long* out, int* status) {
  constexpr int n_tiles = (mode == 4 || mode == 5 || mode == 9) ? 1 : 2;
  constexpr bool do_pv = mode != 1 && mode != 9 && mode != 11;
  constexpr bool do_qk = mode != 2;
  constexpr bool commit_group = mode == 6 || mode == 9;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t tmem = tc_setup(smem, base);
  if constexpr (mode >= 10) {
    uint32_t* w = reinterpret_cast<uint32_t*>(smem);
    for (uint32_t i = threadIdx.x; i < kMbBar / 4; i += kTcThreads) {
      uint32_t h = i * 2654435761u + 0x9e3779b9u;
      h ^= h >> 15;
      h *= 2246822519u;
      h ^= h >> 13;
      const uint32_t lo = (h & 0x8000u) | ((126u + (h >> 4) % 3u) << 7) | (h & 0x7Fu);
      const uint32_t hi = ((h >> 16) & 0x8000u) | ((126u + (h >> 20) % 3u) << 7) | ((h >> 8) & 0x7Fu);
      w[i] = lo | (hi << 16);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
  }
  volatile uint32_t* done_flag = reinterpret_cast<volatile uint32_t*>(smem + kMbBar + 96);
  if (threadIdx.x == 0) *done_flag = 0u;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long t0 = 0, t1 = 0;
  if (warp == 0) {
    const uint32_t leader = lane == 0 ? 1u : 0u;
    const uint32_t id_qk = ptx::idesc_bf16_f32(128, 128, false, false);
    const uint32_t id_pv = ptx::idesc_bf16_f32(128, 128, false, true);
    const uint64_t q0 = ptx::smem_desc_sw128(base + kMbA, 16, 1024);
    const uint64_t k0 = ptx::smem_desc_sw128(base + kMbB, 16, 1024);
    const uint64_t v0 = ptx::smem_desc_sw128(base + kMbB + 32768u, 16384, 1024);
    const uint32_t spare = base + kMbBar + 8u;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0)::"memory");
    for (int r = 0; r < reps; ++r) {
#pragma unroll
      for (int tl = 0; tl < n_tiles; ++tl) {
        if (do_pv) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            ptx::mma_ts_leader(tmem + 256u + 128u * tl, tmem + 128u * tl + 8u * k, v0 + ((2048u * k) >> 4), id_pv,
                               1u, leader);
            if (mode == 7) ptx::mma_commit_leader(spare, leader);
          }
          if (commit_group) ptx::mma_commit_leader(spare, leader);
        }
        if (do_qk) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t off = ((k >> 2) * 16384u + (k & 3) * 32u) >> 4;
            ptx::mma_ss_leader(tmem + 128u * tl, q0 + off, k0 + off, id_qk, k > 0 ? 1u : 0u, leader);
            if (mode == 7) ptx::mma_commit_leader(spare, leader);
          }
          if (commit_group) ptx::mma_commit_leader(spare, leader);
        }
      }
      if (mode == 8) ptx::mma_commit_leader(spare, leader);
    }
    const uint32_t bar = base + kMbBar;
    ptx::mma_commit_leader(bar, leader);
    if (!bounded_wait(bar)) status[0] = 1;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1)::"memory");
    if (lane == 0) *done_flag = 1u;
  } else if (mode == 4) {
    const uint32_t lanes = (static_cast<uint32_t>(warp) * 32u) << 16;
    float acc = 0.f;
    for (int it = 0; it < (1 << 20) && *done_flag == 0u; ++it) {
      float x[32];
      ptx::tmem_ld32_wait(tmem + lanes + 128u + 32u * (it & 3), x);
      uint32_t u[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(x[i] + 1.f);
      ptx::tmem_st32(tmem + lanes + 384u + 32u * (it & 3), u);
      ptx::tmem_wait_st();
      acc += x[5];
    }
    if (acc == 12345.f) status[1] = 1;  // keeps the loads
  } else if (mode == 3) {
    // write traffic into [kMbBar + 128, + 32 KiB) (inside the launch's extra
    // 32 KiB); bounded in iterations
    uint4* dst = reinterpret_cast<uint4*>(smem + kMbBar + 128);
    const uint4 val = make_uint4(threadIdx.x, 1u, 2u, 3u);
    for (int it = 0; it < (1 << 22) && *done_flag == 0u; ++it) {
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[((it * 8 + i) * 96 + threadIdx.x - 32) & 2047] = val;
    }
  }
  __syncwarp();
  tc_teardown(tmem);
  if (threadIdx.x == 0) out[blockIdx.x] = t1 - t0;
}

// Hand-off latency while an MMA stream runs.  Warp 0 (one lane) issues MMAs
// until the measuring warps are done: mode 0 none, 1 QK^T-like (A and B in
// shared memory, N = 128), 2 PV-like (A = P in tensor memory, B = V in shared
// memory, N = 128), 3 the attention stream (per tile 8 PV then 8 QK^T, two
// tiles).  what 0: warps 1 and 2 (one lane each) ping-pong `rounds` times
// through two count-1 mbarriers (arrive, the other side polls with
// try_wait); out = summed round-trip cycles.  what 1: warp 1 chases a
// pointer through shared memory `rounds` times (dependent ld.shared); out =
// summed cycles.  what 2: the ping-pong of what 0 through two named barriers
// (bar.arrive / bar.sync, whole warps; both sides run all rounds, so every
// bar.sync is matched).  Every mbarrier or flag wait is bounded (1 s, status 1).
template <int mode>
__global__ void __launch_bounds__(kTcThreads, 1) handoff_probe(int what, int rounds, long long* out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t tmem = tc_setup(smem, base);
  volatile uint32_t* started = reinterpret_cast<volatile uint32_t*>(smem + kMbBar + 96);
  volatile uint32_t* done_flag = reinterpret_cast<volatile uint32_t*>(smem + kMbBar + 100);
  uint32_t* chain = reinterpret_cast<uint32_t*>(smem + kMbBar + 128);  // 256 words, in the extra 32 KiB
  if (threadIdx.x == 0) {
    *started = 0u;
    *done_flag = 0u;
  }
  for (int i = threadIdx.x; i < 256; i += kTcThreads) chain[i] = static_cast<uint32_t>((i * 97 + 13) & 255);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar_x = base + kMbBar + 16u, bar_y = base + kMbBar + 24u;
  auto wait_parity = [&](uint32_t bar, uint32_t parity) {
    const uint64_t g0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity))
      if (ptx::globaltimer_ns() - g0 > 1000000000ull) return false;
    return true;
  };
  auto wait_flag = [&](volatile uint32_t* f) {
    const uint64_t g0 = ptx::globaltimer_ns();
    while (*f == 0u)
      if (ptx::globaltimer_ns() - g0 > 1000000000ull) return false;
    return true;
  };
  long long acc = 0;
  if (warp == 0 && lane == 0) {
    const uint32_t id_qk = ptx::idesc_bf16_f32(128, 128, false, false);
    const uint32_t id_pv = ptx::idesc_bf16_f32(128, 128, false, true);
    const uint64_t q0 = ptx::smem_desc_sw128(base + kMbA, 16, 1024);
    const uint64_t k0 = ptx::smem_desc_sw128(base + kMbB, 16, 1024);
    const uint64_t v0 = ptx::smem_desc_sw128(base + kMbB + 32768u, 16384, 1024);
    bool any = false;
    const uint64_t g0 = ptx::globaltimer_ns();
    for (int r = 0; r < (1 << 16) && *done_flag == 0u; ++r) {
      if constexpr (mode == 0) {
        *started = 1u;
        if (ptx::globaltimer_ns() - g0 > 1000000000ull) break;
        continue;
      } else {
#pragma unroll
        for (int tl = 0; tl < (mode == 3 ? 2 : 1); ++tl) {
          if (mode == 2 || mode == 3) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              ptx::mma_ts_leader(tmem + 256u + 128u * tl, tmem + 128u * tl + 8u * k, v0 + ((2048u * k) >> 4), id_pv, 1u,
                                 1u);
          }
          if (mode == 1 || mode == 3) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t off = ((k >> 2) * 16384u + (k & 3) * 32u) >> 4;
              ptx::mma_ss_leader(tmem + 128u * tl, q0 + off, k0 + off, id_qk, k > 0 ? 1u : 0u, 1u);
            }
          }
        }
        any = true;
        if (r == 1) *started = 1u;
      }
    }
    *started = 1u;
    if (any) {
      const uint32_t bar = base + kMbBar;
      ptx::mma_commit_leader(bar, 1u);
      if (!bounded_wait(bar)) status[0] = 1;
    }
  } else if (warp == 1 && what == 2) {
    if (!wait_flag(started)) status[0] = 1;
    __syncwarp();
    for (int r = 0; r < rounds; ++r) {
      long long a, b;
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(a)::"memory");
      asm volatile("bar.arrive 1, 64;" ::: "memory");
      asm volatile("bar.sync 2, 64;" ::: "memory");
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(b)::"memory");
      acc += b - a;
    }
    if (lane == 0) *done_flag = 1u;
  } else if (warp == 2 && what == 2) {
    for (int r = 0; r < rounds; ++r) {
      asm volatile("bar.sync 1, 64;" ::: "memory");
      asm volatile("bar.arrive 2, 64;" ::: "memory");
    }
  } else if (warp == 1 && lane == 0) {
    if (!wait_flag(started)) status[0] = 1;
    if (what == 0) {
      for (int r = 0; r < rounds; ++r) {
        long long a, b;
        asm volatile("mov.u64 %0, %%clock64;" : "=l"(a)::"memory");
        ptx::mbar_arrive(bar_x);
        const bool ok = wait_parity(bar_y, static_cast<uint32_t>(r & 1));
        asm volatile("mov.u64 %0, %%clock64;" : "=l"(b)::"memory");
        if (!ok) {
          status[0] = 1;
          break;
        }
        acc += b - a;
      }
    } else {
      uint32_t i = 0;
      long long a, b;
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(a)::"memory");
      for (int r = 0; r < rounds; ++r) i = reinterpret_cast<volatile uint32_t*>(chain)[i];
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(b)::"memory");
      acc = b - a;
      if (i == 12345u) status[1] = 1;  // keeps the chain
    }
    *done_flag = 1u;
  } else if (warp == 2 && lane == 0 && what == 0) {
    for (int r = 0; r < rounds; ++r) {
      if (!wait_parity(bar_x, static_cast<uint32_t>(r & 1))) {
        status[0] = 1;
        break;
      }
      ptx::mbar_arrive(bar_y);
    }
  }
  __syncwarp();
  tc_teardown(tmem);
  if (threadIdx.x == 32) out[blockIdx.x] = acc;
}

// Two issuing threads alternating MMA groups.  Each round is one KV step of
// the attention stream: tile 0's group (8 PV into O_0, then 8 QK^T into S_0)
// and tile 1's group.  variant 0: one thread issues both groups with a
// commit after each (the attention kernel's schedule); 1: tile t's group is
// issued by warp t, which then commits and hands a token (a count-1
// mbarrier) to the other issuer, which waits for it before its group; 2: as
// 1 with the token handed over before the commit; 3: as 1 without commits.
// out = cycles of `reps` rounds (32 MMAs each) on the thread that issues the
// last group.  Every wait is bounded (1 s, status 1).
template <int variant>
__global__ void __launch_bounds__(kTcThreads, 1) pingpong_probe(int reps, long long* out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t tmem = tc_setup(smem, base);
  const uint32_t tok[2] = {base + kMbBar + 32u, base + kMbBar + 40u};
  const uint32_t spare[2] = {base + kMbBar + 48u, base + kMbBar + 56u};
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(tok[i], 1);
      ptx::mbar_init(spare[i], 1);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t id_qk = ptx::idesc_bf16_f32(128, 128, false, false);
  const uint32_t id_pv = ptx::idesc_bf16_f32(128, 128, false, true);
  const uint64_t q0 = ptx::smem_desc_sw128(base + kMbA, 16, 1024);
  const uint64_t k0 = ptx::smem_desc_sw128(base + kMbB, 16, 1024);
  const uint64_t v0 = ptx::smem_desc_sw128(base + kMbB + 32768u, 16384, 1024);
  auto group = [&](int tl) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      ptx::mma_ts(tmem + 256u + 128u * tl, tmem + 128u * tl + 8u * k, v0 + ((2048u * k) >> 4), id_pv, 1u);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint64_t off = ((k >> 2) * 16384u + (k & 3) * 32u) >> 4;
      ptx::mma_ss(tmem + 128u * tl, q0 + off, k0 + off, id_qk, k > 0 ? 1u : 0u);
    }
  };
  auto wait = [&](uint32_t bar, uint32_t parity) {
    const uint64_t g0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity))
      if (ptx::globaltimer_ns() - g0 > 1000000000ull) return false;
    return true;
  };
  long long t0 = 0, t1 = 0;
  if (variant == 0 && warp == 0 && lane == 0) {
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0)::"memory");
    for (int r = 0; r < reps; ++r) {
      group(0);
      ptx::mma_commit(spare[0]);
      group(1);
      ptx::mma_commit(spare[1]);
    }
    ptx::mma_commit(base + kMbBar);
    if (!bounded_wait(base + kMbBar)) status[0] = 1;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1)::"memory");
  } else if (variant > 0 && warp < 2 && lane == 0) {
    const int me = warp;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0)::"memory");
    for (int r = 0; r < reps; ++r) {
      // tile 0 at round r follows tile 1's group of round r - 1; tile 1 follows tile 0's of round r
      bool ok = true;
      if (me == 0 && r > 0) ok = wait(tok[0], static_cast<uint32_t>((r - 1) & 1));
      if (me == 1) ok = wait(tok[1], static_cast<uint32_t>(r & 1));
      if (!ok) {
        status[0] = 1;
        break;
      }
      group(me);
      if (variant == 1) ptx::mma_commit(spare[me]);
      ptx::mbar_arrive(tok[1 - me]);
      if (variant == 2) ptx::mma_commit(spare[me]);
    }
    ptx::mma_commit(base + kMbBar + 8u * me);
    if (!bounded_wait(base + kMbBar + 8u * me)) status[0] = 1;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1)::"memory");
  }
  __syncwarp();
  tc_teardown(tmem);
  if (threadIdx.x == (variant == 0 ? 0 : 32)) out[blockIdx.x] = t1 - t0;
}

__global__ void __launch_bounds__(kTcThreads, 1) tmem_ld_probe(int reps, long long* out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t tmem = tc_setup(smem, base);
  const int warp = threadIdx.x >> 5;
  const uint32_t ta = tmem + ((static_cast<uint32_t>(warp) * 32u) << 16);
  float acc = 0.f;
  long long t0, t1;
  __syncthreads();
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0)::"memory");
  for (int r = 0; r < reps; ++r) {
    float x[32];
    ptx::tmem_ld32_wait(ta + 32u * (r & 7), x);
    acc += x[0] + x[17] + x[31];
  }
  __syncthreads();
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1)::"memory");
  if (acc == 12345.f) status[1] = 1;  // keeps the loads
  tc_teardown(tmem);
  if (threadIdx.x == 0) out[blockIdx.x] = t1 - t0;
}

int finish(long long* d_out, int* d_status, float* d_sink, long long* out_cycles, int n_ctas) {
  int rc = 0;
  int st[2] = {0, 0};
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) fprintf(stderr, "microbench: %s\n", cudaGetErrorString(e));
  if (e != cudaSuccess ||
      cudaMemcpy(out_cycles, d_out, sizeof(long long) * n_ctas, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(st, d_status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    rc = 2;
  else if (st[0] != 0)
    rc = 3;
  cudaFree(d_out);
  cudaFree(d_status);
  if (d_sink) cudaFree(d_sink);
  return rc;
}

bool alloc(long long** d_out, int** d_status, int n_ctas) {
  if (cudaMalloc(d_out, sizeof(long long) * n_ctas) != cudaSuccess) return false;
  if (cudaMalloc(d_status, 2 * sizeof(int)) != cudaSuccess) return false;
  return cudaMemset(*d_status, 0, 2 * sizeof(int)) == cudaSuccess;
}

}  // namespace

namespace {
// Accuracy probe of exp2_poly2: y_poly[i] = exp2_poly2(x[i]), y_ref[i] = exp2f(x[i]).
__global__ void exp2_poly_values(const float* x, float* y_poly, float* y_ref, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float x1 = i + 1 < n ? x[i + 1] : 0.f;
  const float2 y = ptx_probe::exp2_poly2(make_float2(x[i], x1));
  y_poly[i] = y.x;
  y_ref[i] = exp2f(x[i]);
  if (i + 1 < n) {
    y_poly[i + 1] = y.y;
    y_ref[i + 1] = exp2f(x1);
  }
}
}  // namespace

// Evaluates the FMA-pipe exp2 of the exp-loop probe (and exp2f beside it) on
// n host inputs; results to host arrays.  Returns 0, 1 on a bad argument, 2 on
// a CUDA error.
extern "C" int fmha_probe_exp2_poly(const float* x, float* y_poly, float* y_ref, int n) {
  if (x == nullptr || y_poly == nullptr || y_ref == nullptr || n < 1) return 1;
  float* d = nullptr;
  const size_t bytes = sizeof(float) * static_cast<size_t>(n);
  if (cudaMalloc(&d, 3 * bytes) != cudaSuccess) return 2;
  int rc = 0;
  if (cudaMemcpy(d, x, bytes, cudaMemcpyHostToDevice) != cudaSuccess) rc = 2;
  if (rc == 0) {
    const int pairs = (n + 1) / 2;
    exp2_poly_values<<<(pairs + 255) / 256, 256>>>(d, d + n, d + 2 * static_cast<size_t>(n), n);
    if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) rc = 2;
  }
  if (rc == 0 && (cudaMemcpy(y_poly, d + n, bytes, cudaMemcpyDeviceToHost) != cudaSuccess ||
                  cudaMemcpy(y_ref, d + 2 * static_cast<size_t>(n), bytes, cudaMemcpyDeviceToHost) != cudaSuccess))
    rc = 2;
  cudaFree(d);
  return rc;
}

extern "C" int fmha_microbench_alu(int which, int reps, long long* out_cycles, int n_ctas) {
  if (which < 0 || which > 4 || reps < 1 || n_ctas < 1 || out_cycles == nullptr) return 1;
  long long* d_out = nullptr;
  int* d_status = nullptr;
  float* d_sink = nullptr;
  if (!alloc(&d_out, &d_status, n_ctas) ||
      cudaMalloc(&d_sink, sizeof(float) * n_ctas * kAluThreads) != cudaSuccess)
    return 2;
  if (which <= 2)
    alu_probe<<<n_ctas, kAluThreads>>>(which, reps, d_out, d_sink);
  else
    softmax_exp_probe<<<n_ctas, 128>>>(which, reps, d_out, d_sink);
  return finish(d_out, d_status, d_sink, out_cycles, n_ctas);
}

extern "C" int fmha_microbench_mma(int a_tmem, int b_mn, int n, int issuers, int uniform, int reps,
                                   long long* out_cycles, int n_ctas) {
  if ((n != 64 && n != 128 && n != 256) || issuers < 1 || issuers > 3 || issuers * n > 384 || reps < 1 ||
      n_ctas < 1 || out_cycles == nullptr || (a_tmem && n != 128))
    return 1;
  long long* d_out = nullptr;
  int* d_status = nullptr;
  if (!alloc(&d_out, &d_status, n_ctas)) return 2;
  // operand arrangement fixed at compile time, so the loop holds only the MMAs
  auto launch = [&](auto kernel) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMbSmem));
    kernel<<<n_ctas, kTcThreads, kMbSmem>>>(issuers, reps, d_out, d_status);
  };
  const int key = (a_tmem ? 1 : 0) | (b_mn ? 2 : 0) | (uniform ? 4 : 0);
  if (n == 64) {
    if (key == 4) launch(mma_probe<0, 0, 64, 1>); else return 1;
  } else if (n == 256) {
    if (key == 4) launch(mma_probe<0, 0, 256, 1>); else if (key == 0) launch(mma_probe<0, 0, 256, 0>); else return 1;
  } else {
    switch (key) {
      case 0: launch(mma_probe<0, 0, 128, 0>); break;
      case 1: launch(mma_probe<1, 0, 128, 0>); break;
      case 2: launch(mma_probe<0, 1, 128, 0>); break;
      case 3: launch(mma_probe<1, 1, 128, 0>); break;
      case 4: launch(mma_probe<0, 0, 128, 1>); break;
      case 5: launch(mma_probe<1, 0, 128, 1>); break;
      case 6: launch(mma_probe<0, 1, 128, 1>); break;
      default: launch(mma_probe<1, 1, 128, 1>); break;
    }
  }
  return finish(d_out, d_status, nullptr, out_cycles, n_ctas);
}

// Cycles of `reps` rounds of the attention MMA stream (32 MMAs a round) in
// the given mode of mma_mix_probe.  Returns as fmha_microbench_mma.
extern "C" int fmha_microbench_mma_mix(int mode, int reps, long long* out_cycles, int n_ctas) {
  if (mode < 0 || mode > 11 || reps < 1 || n_ctas < 1 || out_cycles == nullptr) return 1;
  long long* d_out = nullptr;
  int* d_status = nullptr;
  if (!alloc(&d_out, &d_status, n_ctas)) return 2;
  const int smem = static_cast<int>(kMbSmem) + 32768;
  auto launch = [&](auto kernel) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    kernel<<<n_ctas, kTcThreads, smem>>>(reps, d_out, d_status);
  };
  switch (mode) {
    case 0: launch(mma_mix_probe<0>); break;
    case 1: launch(mma_mix_probe<1>); break;
    case 2: launch(mma_mix_probe<2>); break;
    case 3: launch(mma_mix_probe<3>); break;
    case 4: launch(mma_mix_probe<4>); break;
    case 5: launch(mma_mix_probe<5>); break;
    case 6: launch(mma_mix_probe<6>); break;
    case 7: launch(mma_mix_probe<7>); break;
    case 8: launch(mma_mix_probe<8>); break;
    case 9: launch(mma_mix_probe<9>); break;
    case 10: launch(mma_mix_probe<10>); break;
    default: launch(mma_mix_probe<11>); break;
  }
  return finish(d_out, d_status, nullptr, out_cycles, n_ctas);
}

// Summed cycles of handoff_probe (mode: the MMA stream; what: 0 mbarrier
// ping-pong round trips, 1 dependent shared-memory loads, 2 named-barrier
// ping-pong round trips) over `rounds`.  Returns as
// fmha_microbench_mma.
extern "C" int fmha_microbench_handoff(int mode, int what, int rounds, long long* out_cycles, int n_ctas) {
  if (mode < 0 || mode > 3 || what < 0 || what > 2 || rounds < 1 || rounds > (1 << 20) || n_ctas < 1 ||
      out_cycles == nullptr)
    return 1;
  long long* d_out = nullptr;
  int* d_status = nullptr;
  if (!alloc(&d_out, &d_status, n_ctas)) return 2;
  const int smem = static_cast<int>(kMbSmem) + 32768;
  auto launch = [&](auto kernel) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    kernel<<<n_ctas, kTcThreads, smem>>>(what, rounds, d_out, d_status);
  };
  switch (mode) {
    case 0: launch(handoff_probe<0>); break;
    case 1: launch(handoff_probe<1>); break;
    case 2: launch(handoff_probe<2>); break;
    default: launch(handoff_probe<3>); break;
  }
  return finish(d_out, d_status, nullptr, out_cycles, n_ctas);
}

namespace {
__global__ void __launch_bounds__(512, 1) empty_probe() {}
}  // namespace

// Launches an empty kernel of `grid` CTAs of `block` threads with `smem`
// bytes of dynamic shared memory on `stream` (asynchronous): the launch
// envelope a one-wave kernel pays inside a pair of timing events.  Returns 0,
// 1 on a bad argument, 2 on a launch error.
extern "C" int fmha_microbench_empty_launch(int grid, int block, int smem, void* stream) {
  if (grid < 1 || block < 32 || block > 512 || smem < 0 || smem > 232448) return 1;
  if (cudaFuncSetAttribute(empty_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 2;
  empty_probe<<<grid, block, smem, static_cast<cudaStream_t>(stream)>>>();
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

// Cycles of `reps` rounds of pingpong_probe<variant>.  Returns as
// fmha_microbench_mma.
extern "C" int fmha_microbench_pingpong(int variant, int reps, long long* out_cycles, int n_ctas) {
  if (variant < 0 || variant > 3 || reps < 1 || reps > (1 << 20) || n_ctas < 1 || out_cycles == nullptr) return 1;
  long long* d_out = nullptr;
  int* d_status = nullptr;
  if (!alloc(&d_out, &d_status, n_ctas)) return 2;
  auto launch = [&](auto kernel) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMbSmem));
    kernel<<<n_ctas, kTcThreads, kMbSmem>>>(reps, d_out, d_status);
  };
  switch (variant) {
    case 0: launch(pingpong_probe<0>); break;
    case 1: launch(pingpong_probe<1>); break;
    case 2: launch(pingpong_probe<2>); break;
    default: launch(pingpong_probe<3>); break;
  }
  return finish(d_out, d_status, nullptr, out_cycles, n_ctas);
}

// Summed cycles of the step-boundary sequence of boundary_probe over `reps`
// rounds.  Returns as fmha_microbench_mma.
extern "C" int fmha_microbench_boundary(int mode, int reps, long long* out_cycles, int n_ctas) {
  if (mode < 0 || mode > 8 || reps < 1 || n_ctas < 1 || out_cycles == nullptr) return 1;
  long long* d_out = nullptr;
  int* d_status = nullptr;
  if (!alloc(&d_out, &d_status, n_ctas)) return 2;
  auto launch = [&](auto kernel) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMbSmem));
    kernel<<<n_ctas, kTcThreads, kMbSmem>>>(reps, d_out, d_status);
  };
  switch (mode) {
    case 0: launch(boundary_probe<0>); break;
    case 1: launch(boundary_probe<1>); break;
    case 2: launch(boundary_probe<2>); break;
    case 3: launch(boundary_probe<3>); break;
    case 4: launch(boundary_probe<4>); break;
    case 5: launch(boundary_probe<5>); break;
    case 6: launch(boundary_probe<6>); break;
    case 7: launch(boundary_probe<7>); break;
    default: launch(boundary_probe<8>); break;
  }
  return finish(d_out, d_status, nullptr, out_cycles, n_ctas);
}

// Cycles for `reps` repetitions of exp_loop_probe<variant, threads>.
extern "C" int fmha_microbench_exp_loop(int variant, int threads, int reps, long long* out_cycles, int n_ctas) {
  if (variant < 0 || variant > 8 || (threads != 128 && threads != 256) || reps < 1 || n_ctas < 1 ||
      out_cycles == nullptr)
    return 1;
  long long* d_out = nullptr;
  int* d_status = nullptr;
  float* d_sink = nullptr;
  if (!alloc(&d_out, &d_status, n_ctas) || cudaMalloc(&d_sink, sizeof(float) * n_ctas * 256) != cudaSuccess)
    return 2;
#define FMHA_EXP_CASE(V)                                                   \
  case V:                                                                  \
    if (threads == 128)                                                    \
      exp_loop_probe<V, 128><<<n_ctas, 128>>>(reps, d_out, d_sink);        \
    else                                                                   \
      exp_loop_probe<V, 256><<<n_ctas, 256>>>(reps, d_out, d_sink);        \
    break;
  switch (variant) {
    FMHA_EXP_CASE(0)
    FMHA_EXP_CASE(1)
    FMHA_EXP_CASE(2)
    FMHA_EXP_CASE(3)
    FMHA_EXP_CASE(4)
    FMHA_EXP_CASE(5)
    FMHA_EXP_CASE(6)
    FMHA_EXP_CASE(7)
    FMHA_EXP_CASE(8)
  }
#undef FMHA_EXP_CASE
  return finish(d_out, d_status, d_sink, out_cycles, n_ctas);
}

extern "C" int fmha_microbench_tmem_ld(int reps, long long* out_cycles, int n_ctas) {
  if (reps < 1 || n_ctas < 1 || out_cycles == nullptr) return 1;
  long long* d_out = nullptr;
  int* d_status = nullptr;
  if (!alloc(&d_out, &d_status, n_ctas)) return 2;
  cudaFuncSetAttribute(tmem_ld_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMbSmem));
  tmem_ld_probe<<<n_ctas, kTcThreads, kMbSmem>>>(reps, d_out, d_status);
  return finish(d_out, d_status, nullptr, out_cycles, n_ctas);
}
