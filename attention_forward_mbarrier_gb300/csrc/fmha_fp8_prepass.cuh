// fmha_fp8_prepass.cuh -- V in e4m3 for the FP8 PV variant of the forward.
//
// "Kernel Bottleneck Tuning" (sections "4. If scheduling has no headroom:
// eliminate instructions algebraically" and "5. Tune the producer->consumer
// handoff split") describes an attention forward whose O += P V product runs
// on FP8 operands.  A tcgen05.mma of kind::f8f6f4 takes both operands in 8
// bits, so V is quantised as well: per K/V head, V8 = e4m3(V / s) with
// s = max|V| / 448 (448 = the largest finite e4m3), and s is folded into the
// epilogue's 1 / l.
//
// Layout of the quantised V (workspace, written here): Vt[kv_head][d][x],
// bytes, d = 0..head_dim-1 rows of Kpad bytes, keys contiguous (the K-major B
// operand of the PV product).  Sequence b's keys start at padded position
// pk0(b) = 16 * (ceil(k0(b) / 16) + b), so every TMA box starts on a 16-byte
// boundary; the gaps between sequences hold e4m3 zeros.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace fmha {
namespace fp8 {

constexpr float kE4m3Max = 448.f;

__host__ __device__ __forceinline__ int64_t padded_start(int64_t k0, int b) { return 16 * ((k0 + 15) / 16 + b); }
__host__ __device__ __forceinline__ int64_t padded_keys(int64_t total_k, int batch) {
  return padded_start(total_k, batch);
}

struct PrepassParams {
  const __nv_bfloat16* v;  // [total_k, kv_heads, head_dim]
  uint32_t* amax_bits;     // [kv_heads]: max |V| as float bits (zeroed before the first kernel)
  uint8_t* vt;             // [kv_heads, head_dim, kpad]
  const int32_t* cu_k;     // [batch + 1] or nullptr (dense)
  int batch, total_k, max_seqlen_k, kv_heads, head_dim;
  int64_t kpad;
};

__device__ __forceinline__ int64_t seq_key_start(const PrepassParams& p, int b) {
  return p.cu_k != nullptr ? static_cast<int64_t>(p.cu_k[b]) : static_cast<int64_t>(b) * p.max_seqlen_k;
}

// max |V| per K/V head: one CTA per (token chunk, K/V head); each warp takes
// tokens of the chunk (16 lanes per 256-byte row, two rows per instruction),
// the CTA reduces in shared memory and makes one atomicMax (non-negative
// floats order as their bits), so the atomics stay few per head.
constexpr int kAmaxThreads = 256;
constexpr int kAmaxTokens = 64;  // tokens per CTA (many CTAs: the pass is latency-bound)
__global__ void __launch_bounds__(kAmaxThreads) v_amax_kernel(const PrepassParams p) {
  __shared__ float warp_max[kAmaxThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane >> 4, sub = lane & 15;
  const int h = static_cast<int>(blockIdx.y);
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kAmaxTokens;
  const int64_t t1 = min(t0 + kAmaxTokens, static_cast<int64_t>(p.total_k));
  float m = 0.f;
  for (int64_t t = t0 + 2 * warp + half; t < t1; t += 2 * (kAmaxThreads / 32)) {
    const uint4 v4 = *reinterpret_cast<const uint4*>(p.v + (t * p.kv_heads + h) * p.head_dim + 8 * sub);
    const uint32_t w[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) warp_max[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.f;
#pragma unroll
    for (int i = 0; i < kAmaxThreads / 32; ++i) b = fmaxf(b, warp_max[i]);
    if (b > 0.f) atomicMax(p.amax_bits + h, __float_as_uint(b));
  }
}

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Quantise and transpose: one CTA (256 threads) per (128 padded key
// positions, K/V head), head_dim 128.  Positions outside every sequence get
// e4m3 zero.
constexpr int kQuantThreads = 256;
__global__ void __launch_bounds__(kQuantThreads) v_quant_kernel(const PrepassParams p) {
  __shared__ __align__(16) uint8_t tile[128][128 + 16];  // [d][key]
  const int h = static_cast<int>(blockIdx.y);
  const int64_t x0 = static_cast<int64_t>(blockIdx.x) * 128;
  const uint32_t bits = p.amax_bits[h];
  const float amax = __uint_as_float(bits);
  const float inv = amax > 0.f ? kE4m3Max / amax : 1.f;
  // phase 1: one padded key position per lane (warps 0-3 head dims 0..63,
  // warps 4-7 head dims 64..127): each byte store of a warp writes 32
  // consecutive bytes of one row of the tile (no bank conflicts)
  {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = 32 * (warp & 3) + lane;
    const int64_t x = x0 + r;
    // the sequence whose padded range holds x (binary search on padded starts)
    int lo = 0, hi = p.batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (padded_start(seq_key_start(p, mid), mid) <= x)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int64_t ks = seq_key_start(p, lo);
    const int64_t len = p.cu_k != nullptr ? static_cast<int64_t>(p.cu_k[lo + 1]) - ks : p.max_seqlen_k;
    const int64_t i = x - padded_start(ks, lo);
    const bool in_seq = p.batch > 0 && i >= 0 && i < len;
    const __nv_bfloat16* src = p.v + ((ks + i) * p.kv_heads + h) * p.head_dim;
    uint4 rowv[8];  // this lane's 8 chunks of 8 head dims, all loads in flight at once
#pragma unroll
    for (int i = 0; i < 8; ++i)
      rowv[i] = in_seq ? *reinterpret_cast<const uint4*>(src + 8 * (8 * (warp >> 2) + i)) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = 8 * (warp >> 2) + i;
      uint16_t q[4] = {0, 0, 0, 0};
      if (in_seq) {
        const uint4 v4 = rowv[i];
        const uint32_t w[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
          q[k] = e4m3x2(f.x * inv, f.y * inv);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tile[8 * c + 2 * k][r] = static_cast<uint8_t>(q[k] & 0xffu);
        tile[8 * c + 2 * k + 1][r] = static_cast<uint8_t>(q[k] >> 8);
      }
    }
  }
  __syncthreads();
  // phase 2: 128 rows (d) x 8 chunks of 16 bytes
  for (int it = threadIdx.x; it < 128 * 8; it += kQuantThreads) {
    const int d = it >> 3, c = it & 7;
    const int64_t x = x0 + 16 * c;
    if (x >= p.kpad) continue;  // kpad is a multiple of 16
    const uint4 v = *reinterpret_cast<const uint4*>(&tile[d][16 * c]);
    *reinterpret_cast<uint4*>(p.vt + (static_cast<int64_t>(h) * p.head_dim + d) * p.kpad + x) = v;
  }
}

}  // namespace fp8
}  // namespace fmha
