// fmha_bwd_kernel.cuh -- backward pass of the fused attention forward, sm_103a.
//
// Given q, k, v, the forward's output O and log-sum-exp, and the upstream
// gradient dO, computes dQ, dK, dV of L = sum dO . O for head_dim 128 bf16
// [tokens, heads, 128] tensors, dense or varlen, causal or not, with grouped
// K/V heads.  The benchmark step of "[BUG] CuTe DSL 4.7/4.8 regression:
// FlashAttention-4 SM100 forward kernel spills registers" (section
// "Steps/Code to reproduce bug") runs this pass after the varlen causal
// forward.  With P = exp(scale * q k^T - LSE) (the forward's softmax,
// recomputed from its LSE):
//   dV = P^T dO,  dP = dO V^T,  D_i = dO_i . O_i,  dS = P * (dP - D),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Three kernels, no atomics (every output row is written by one CTA):
//   fmha_bwd_dot_kernel   D_i = dO_i . O_i for every row, into the workspace
//                         (coalesced, bandwidth-bound);
//   fmha_bwd_dq_kernel    one CTA per (head, 128 query rows, sequence): per
//                         128-key block S = Q K^T and dP = dO V^T into
//                         TMEM, dS in bf16 over S, dQ += dS K; S is
//                         double-buffered and dP released as soon as it is in
//                         registers, so the next blocks' products overlap the
//                         gradient math.
//   fmha_bwd_dkdv_kernel  one CTA per (K/V head, 128 keys, sequence): per query
//                         block of every query head of the group, in two
//                         halves of 64 queries, S^T = K Q^T and dP^T = V dO^T
//                         into TMEM, P^T and dS^T in bf16 over them, dV += P^T
//                         dO and dK += dS^T Q; one half's gradient math
//                         overlaps the other half's products.
// Every GEMM is a tcgen05.mma of one of the forward's two forms: both operands
// K-major in shared memory, or A from TMEM with an MN-major B.  Warp roles
// (224 threads): warps 0-3 the gradient math on one TMEM lane (row) each and
// the epilogue; warp 4 the TMA producer; warps 5 and 6 issue MMAs (two
// streams, see each kernel), warp 5 owns TMEM.
// Every mbarrier wait is bounded as in the forward kernel.
#pragma once

#include "fmha_fwd_kernel.cuh"

namespace fmha {
namespace bwd {

constexpr int kWarpProducer = 4;
constexpr int kWarpMma = 5;
// the dQ kernel has a second MMA-issuing warp for dP (224 threads)
constexpr int kDqThreads = 224;
constexpr int kWarpMmaDp = 6;
constexpr uint32_t kTile = kBlockM * 128 * 2;  // a 128 x 128 bf16 tile: two swizzled 64-column halves
constexpr float kLog2e = 1.4426950408889634f;

struct alignas(64) BwdParams {
  CUtensorMap tmap_q;   // [total_q, heads * 128]
  CUtensorMap tmap_do;  // [total_q, heads * 128]
  CUtensorMap tmap_k;   // [total_k, kv_heads * 128]
  CUtensorMap tmap_v;
  const __nv_bfloat16* out;   // O
  const __nv_bfloat16* dout;  // dO
  const float* lse;           // [heads, total_q], natural log
  float* dvec;                // D, [heads, total_q] (workspace)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int batch, total_q, total_k, max_seqlen_q, max_seqlen_k, heads, kv_heads;
  int causal, kv_group;
  float scale;       // dQ, dK factor
  float scale_log2;  // scale * log2(e)
};

// Opt-in coarse trace (build with -DFMHA_TRACE): %clock64 stamps of the CTAs
// of head (K/V head) 0, sequence 0, one row of kTraceSlots per query (key)
// block: per block / item j < 64 at slot 8 j + event, the dK/dV kernel's
// issuing threads per item j < 60 at slot 512 + 8 j + event, set-up and exit
// at 1000 + event.
#ifdef FMHA_TRACE
__device__ unsigned long long* g_trace_dq;
__device__ unsigned long long* g_trace_dkdv;
#define FMHA_BWD_TRACE(row, slot)                                                            \
  do {                                                                                       \
    if ((row) != nullptr) (row)[(slot)] = static_cast<unsigned long long>(clock64());       \
  } while (0)
#else
#define FMHA_BWD_TRACE(row, slot) \
  do {                            \
  } while (0)
#endif

__device__ __forceinline__ void seq_bounds(const BwdParams& p, int b, int& q0, int& lq, int& k0, int& lk) {
  if (p.cu_q != nullptr) {
    q0 = p.cu_q[b];
    lq = p.cu_q[b + 1] - q0;
    k0 = p.cu_k[b];
    lk = p.cu_k[b + 1] - k0;
  } else {
    q0 = b * p.max_seqlen_q;
    lq = p.max_seqlen_q;
    k0 = b * p.max_seqlen_k;
    lk = p.max_seqlen_k;
  }
  if (lq < 0) lq = 0;
  if (lk < 0) lk = 0;
}

// -LSE * log2(e) of a query row, the additive term of its exponent; -inf for a
// row with no visible key (LSE = -inf), whose P must be 0 (its keys are all
// masked anyway).
__device__ __forceinline__ float neg_lse2(float lse) { return lse == -INFINITY ? -INFINITY : -lse * kLog2e; }

// ============================================================================ D
// D_i = dO_i . O_i (fp32) for every (token, head) row, into the workspace
// [heads, total_q].  Coalesced: 16 lanes per 256-byte row, two rows per warp
// instruction, grid-stride over the rows.  (Rows of no sequence get a value
// that nothing reads.)
constexpr int kDotThreads = 256;
__global__ void __launch_bounds__(kDotThreads) fmha_bwd_dot_kernel(const __grid_constant__ BwdParams p) {
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, sub = lane & 15;
  const int64_t rows = static_cast<int64_t>(p.total_q) * p.heads;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r2 = warp0; 2 * r2 < rows; r2 += nwarps) {
    const int64_t r = 2 * r2 + half;  // row = token * heads + head
    float acc = 0.f;
    if (r < rows) {
      const uint4 a = *reinterpret_cast<const uint4*>(p.out + r * 128 + 8 * sub);
      const uint4 g = *reinterpret_cast<const uint4*>(p.dout + r * 128 + 8 * sub);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 af = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[k]));
        const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[k]));
        acc = fmaf(af.x, gf.x, acc);
        acc = fmaf(af.y, gf.y, acc);
      }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);  // within each 16-lane half
    if (sub == 0 && r < rows) {
      const int64_t tok = r / p.heads;
      const int h = static_cast<int>(r - tok * p.heads);
      p.dvec[static_cast<int64_t>(h) * p.total_q + tok] = acc;
    }
  }
}

// ============================================================================ dQ
// Shared memory: Q and dO tiles, a 3-slot ring of K blocks and a 2-slot ring
// of V blocks, barriers.
struct DqSmem {
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffDo = kTile;
  static constexpr uint32_t kOffK = 2 * kTile;  // slot s at + s kTile (3 slots)
  static constexpr uint32_t kOffV = 5 * kTile;  // slot s at + s kTile (2 slots)
  static constexpr uint32_t kOffBar = 7 * kTile;
  static constexpr uint32_t kOffMisc = kOffBar + 128;
  static constexpr uint32_t kBytes = kOffBar + 256 + 1024;
  static_assert(kBytes <= 232448, "shared memory per CTA");
};
constexpr int kDqKSlots = 3, kDqVSlots = 2;
// barrier ids
constexpr int kDqQFull = 0;     // Q and dO landed
constexpr int kDqKFull = 1;     // [3] K_j of slot j % 3 landed
constexpr int kDqVFull = 4;     // [2] V_j of slot j % 2 landed
constexpr int kDqKFree = 6;     // [3] dQ(j) retired: K_j no longer read
constexpr int kDqBlkReady = 9;  // [2] S(j) and dP(j) in TMEM, barrier j & 1 (two arrivals: the S
                                // issuer's and the dP issuer's commits); also tells the producer
                                // that V_j (read only by dP(j)) is free
constexpr int kDqDpFree = 11;   // dP(j) read into registers (4 warps)
constexpr int kDqPReady = 12;   // [2] dS(j) stored, barrier j & 1 (4 warps)
constexpr int kDqDone = 14;     // every MMA of the S / dQ issuer retired
constexpr int kDqDpDone = 15;   // every MMA of the dP issuer retired
// Pairs of alternating barriers where a waiter could otherwise find a barrier
// two phases on: dP(j+1) lets the gradient warps finish block j+1 before the
// MMA thread polls for dS(j), and dP(j+1) may retire before the producer polls
// for dP(j).  With two barriers the next phase of each needs a step the waiter
// itself has not yet allowed.
// TMEM columns: S of block j at 128 (j & 1) (dS as bf16 over its first 64
// columns, chunk c of 32 scores to columns 16 c .. 16 c + 15, already read),
// dP at 256, dQ at 384.
constexpr uint32_t kDqColDp = 256, kDqColDq = 384;
__device__ __forceinline__ uint32_t dq_col_s(int j) { return 128u * static_cast<uint32_t>(j & 1); }

// Schedule (two MMA-issuing threads; issue is paced by the tensor pipe, so a
// thread blocked on its own queue cannot react to a hand-off): the S / dQ
// issuer issues S(0), S(1), then per block j dQ(j) once dS(j) is stored and
// S(j+2) into the S buffer dQ(j) just read; the dP issuer issues dP(j+1) as
// soon as the gradient warps have dP(j) in registers.  The gradient math of
// block j thus overlaps dP(j+1) and the S products of later blocks.
__global__ void __launch_bounds__(kDqThreads, 1) fmha_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (warp == kWarpProducer && lane == 0) {
    ptx::prefetch_tensormap(&p.tmap_q);
    ptx::prefetch_tensormap(&p.tmap_do);
    ptx::prefetch_tensormap(&p.tmap_k);
    ptx::prefetch_tensormap(&p.tmap_v);
  }
  const int h = static_cast<int>(blockIdx.x);
  const int r0 = static_cast<int>(blockIdx.y) * kBlockM;
  const int b = static_cast<int>(blockIdx.z);
  int q0, lq, k0, lk;
  seq_bounds(p, b, q0, lq, k0, lk);
  if (r0 >= lq) return;  // uniform, before any shared state
  const int off = lk - lq;
  const int nb = tile_blocks(r0, lq, lk, p.causal);
  const int xq = h * 128;
#ifdef FMHA_TRACE
  unsigned long long* trow = (g_trace_dq != nullptr && h == 0 && b == 0) ? g_trace_dq + blockIdx.y * 1024ull : nullptr;
#else
  unsigned long long* trow = nullptr;
#endif
  if (threadIdx.x == 0) FMHA_BWD_TRACE(trow, 1000);
  const int xkv = (h / p.kv_group) * 128;

  Ctx ctx;
  ctx.bar0 = base + DqSmem::kOffBar;
  ctx.abort_flag = reinterpret_cast<volatile uint32_t*>(smem + DqSmem::kOffMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + DqSmem::kOffMisc);

  auto load_tile = [&](const CUtensorMap* m, uint32_t dst, uint32_t bar, int x, int y, uint64_t pol) {
    ptx::tma_load_2d(dst, m, bar, x, y, pol);
    ptx::tma_load_2d(dst + kHalfBytes, m, bar, x + 64, y, pol);
  };
  auto load_k = [&](int j, uint64_t pol) {
    const uint32_t bar = ctx.bar(kDqKFull + j % kDqKSlots);
    ptx::mbar_arrive_expect_tx(bar, kTile);
    load_tile(&p.tmap_k, base + DqSmem::kOffK + (j % kDqKSlots) * kTile, bar, xkv, k0 + kBlockN * j, pol);
  };
  auto load_v = [&](int j, uint64_t pol) {
    const uint32_t bar = ctx.bar(kDqVFull + j % kDqVSlots);
    ptx::mbar_arrive_expect_tx(bar, kTile);
    load_tile(&p.tmap_v, base + DqSmem::kOffV + (j % kDqVSlots) * kTile, bar, xkv, k0 + kBlockN * j, pol);
  };
  // loads before the set-up sync: K_0, V_0, K_1, V_1, K_2 (every slot once)
  const int early_k = min(kDqKSlots, nb), early_v = min(kDqVSlots, nb);

  if (warp == kWarpProducer && lane == 0) {
    ptx::mbar_init(ctx.bar(kDqQFull), 1);
    for (int s = 0; s < kDqKSlots; ++s) {
      ptx::mbar_init(ctx.bar(kDqKFull + s), 1);
      ptx::mbar_init(ctx.bar(kDqKFree + s), 1);
    }
    for (int s = 0; s < kDqVSlots; ++s) ptx::mbar_init(ctx.bar(kDqVFull + s), 1);
    ptx::mbar_init(ctx.bar(kDqBlkReady), 2);
    ptx::mbar_init(ctx.bar(kDqBlkReady + 1), 2);
    ptx::mbar_init(ctx.bar(kDqDpDone), 1);
    ptx::mbar_init(ctx.bar(kDqDpFree), 4);
    ptx::mbar_init(ctx.bar(kDqPReady), 4);
    ptx::mbar_init(ctx.bar(kDqPReady + 1), 4);
    ptx::mbar_init(ctx.bar(kDqDone), 1);
    *ctx.abort_flag = 0u;
    ptx::fence_mbar_init();
    if (nb > 0) {
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint64_t pol_kv = ptx::policy_evict_last();
      const uint32_t bar = ctx.bar(kDqQFull);
      ptx::mbar_arrive_expect_tx(bar, 2 * kTile);
      load_tile(&p.tmap_q, base + DqSmem::kOffQ, bar, xq, q0 + r0, pol_q);
      load_tile(&p.tmap_do, base + DqSmem::kOffDo, bar, xq, q0 + r0, pol_q);
      for (int j = 0; j < early_k; ++j) {
        load_k(j, pol_kv);
        if (j < early_v) load_v(j, pol_kv);
      }
    }
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ================================ gradient math: one query row per thread
    const int r = warp * 32 + lane;
    const int row = r0 + r;
    const bool valid = row < lq;
    const uint32_t lane_base = tmem + ((static_cast<uint32_t>(warp) * 32u) << 16);
    float dval = 0.f;
    float nl2 = -INFINITY;  // rows past the sequence end: P = 0
    if (valid) {
      // D_i (from the pre-pass) and the row's LSE
      const size_t li = static_cast<size_t>(h) * p.total_q + q0 + row;
      dval = p.dvec[li];
      nl2 = neg_lse2(p.lse[li]);
    }
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    const float2 nl2_2 = make_float2(nl2, nl2);
    const float2 nd2 = make_float2(-dval, -dval);
    const int key_end = p.causal ? min(row + off + 1, lk) : lk;      // this row's visible keys
    const int tile_key_end = p.causal ? min(r0 + off + 1, lk) : lk;  // the tile's first row's
    const bool tr = r == 0 && trow != nullptr;
    if (tr) FMHA_BWD_TRACE(trow, 1001);
    for (int j = 0; j < nb; ++j) {
      if (!wait_bar_warp(ctx, kDqBlkReady + (j & 1), (j >> 1) & 1, kRoleSoftmax)) break;
      if (tr && j < 64) FMHA_BWD_TRACE(trow, 8 * j + 0);
      ptx::tc_fence_after();
      // dP(j) into registers at once, then its columns are released for dP(j+1)
      float dp[128];
      ptx::tmem_ld128_wait(lane_base + kDqColDp, dp);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ctx.bar(kDqDpFree));
      if (tr && j < 64) FMHA_BWD_TRACE(trow, 8 * j + 1);
      const uint32_t col_s = dq_col_s(j);
      const bool need_mask = tile_key_end - j * kBlockN < kBlockN;  // diagonal or key tail
      const int lim = key_end - j * kBlockN;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float s[32];
        ptx::tmem_ld32_wait(lane_base + col_s + 32u * cc, s);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int kk = 32 * cc + 2 * i;
          const float2 x = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), c2, nl2_2);
          float p0 = ptx::ex2_approx(x.x);
          float p1 = ptx::ex2_approx(x.y);
          if (need_mask) {
            p0 = kk < lim ? p0 : 0.f;
            p1 = kk + 1 < lim ? p1 : 0.f;
          }
          const float2 g = __fadd2_rn(make_float2(dp[kk], dp[kk + 1]), nd2);  // dP - D
          const float2 ds = __fmul2_rn(make_float2(p0, p1), g);
          pk[i] = ptx::pack_bf16x2(ds.x, ds.y);
        }
        ptx::tmem_st16(lane_base + col_s + 16u * cc, pk);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ctx.bar(kDqPReady + (j & 1)));
      if (tr && j < 64) FMHA_BWD_TRACE(trow, 8 * j + 2);
    }
    if (tr) FMHA_BWD_TRACE(trow, 1002);
    // ---- epilogue: dQ * scale -> bf16
    const bool have = nb > 0 && wait_bar_warp(ctx, kDqDone, 0, kRoleSoftmax);
    if (have) ptx::tc_fence_after();
    __nv_bfloat16* dst = p.dq + (static_cast<size_t>(q0 + row) * p.heads + h) * 128;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      float o[32];
      if (have) {
        ptx::tmem_ld32_wait(lane_base + kDqColDq + 32u * cc, o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0.f;
      }
      if (valid) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * cc);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          uint4 w;
          w.x = ptx::pack_bf16x2(o[8 * v4 + 0] * p.scale, o[8 * v4 + 1] * p.scale);
          w.y = ptx::pack_bf16x2(o[8 * v4 + 2] * p.scale, o[8 * v4 + 3] * p.scale);
          w.z = ptx::pack_bf16x2(o[8 * v4 + 4] * p.scale, o[8 * v4 + 5] * p.scale);
          w.w = ptx::pack_bf16x2(o[8 * v4 + 6] * p.scale, o[8 * v4 + 7] * p.scale);
          d4[v4] = w;
        }
      }
    }
  } else if (warp == kWarpProducer) {
    // ================================ TMA producer: the remaining K and V blocks in block order
    if (lane == 0) {
      const uint64_t pol_kv = ptx::policy_evict_last();
      int issued_k = early_k, issued_v = early_v;
      bool ok = true;
      for (int j = 0; j < nb && ok; ++j) {
        // K_j reuses the slot of K_(j-3), free once dQ(j-3) retired; V_j the
        // slot of V_(j-2), free once dP(j-2) retired (its block-ready commit)
        if (j >= kDqKSlots) {
          const int prev = j - kDqKSlots;
          ok = wait_bar(ctx, kDqKFree + prev % kDqKSlots, (prev / kDqKSlots) & 1, kRoleLoad);
          if (!ok) break;
          load_k(j, pol_kv);
          ++issued_k;
        }
        if (j >= kDqVSlots) {
          const int prev = j - kDqVSlots;
          ok = wait_bar(ctx, kDqBlkReady + (prev & 1), (prev >> 1) & 1, kRoleLoad);
          if (!ok) break;
          load_v(j, pol_kv);
          ++issued_v;
        }
      }
      for (int j = max(0, issued_k - kDqKSlots); j < issued_k; ++j)
        wait_drain(ctx, kDqKFull + j % kDqKSlots, (j / kDqKSlots) & 1);
      for (int j = max(0, issued_v - kDqVSlots); j < issued_v; ++j)
        wait_drain(ctx, kDqVFull + j % kDqVSlots, (j / kDqVSlots) & 1);
      if (nb > 0) wait_drain(ctx, kDqQFull, 0);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ================================ S / dQ issuer
    if (lane == 0 && nb > 0) {
      const uint64_t q_desc = desc_kmajor(base + DqSmem::kOffQ);
      const uint64_t k_kmaj = desc_kmajor(base + DqSmem::kOffK);
      const uint64_t k_mn = desc_mnmajor(base + DqSmem::kOffK);
      constexpr uint64_t kStep = kTile >> 4;  // descriptor units of one tile
      auto wait_k = [&](int j) { return wait_bar(ctx, kDqKFull + j % kDqKSlots, (j / kDqKSlots) & 1, kRoleMma); };
      auto issue_s = [&](int j) {
        issue_qk<128>(tmem + dq_col_s(j), q_desc, k_kmaj + (j % kDqKSlots) * kStep);
        ptx::mma_commit(ctx.bar(kDqBlkReady + (j & 1)));  // S(j): one of block j's two arrivals
      };
      bool issued_any = false;
      bool ok = wait_bar(ctx, kDqQFull, 0, kRoleMma) && wait_k(0);
      if (ok) {
        ptx::tc_fence_after();
        issue_s(0);
        issued_any = true;
        if (nb > 1) {
          ok = wait_k(1);
          if (ok) {
            ptx::tc_fence_after();
            issue_s(1);
          }
        }
      }
      for (int j = 0; j < nb && ok; ++j) {
        if (!wait_bar(ctx, kDqPReady + (j & 1), (j >> 1) & 1, kRoleMma)) break;
        if (j < 64) FMHA_BWD_TRACE(trow, 8 * j + 4);
        ptx::tc_fence_after();
        // dQ += dS(j) K_j: A = dS (bf16 over S(j)), B = K_j MN-major
        issue_pv<128>(tmem + kDqColDq, tmem + dq_col_s(j), k_mn + (j % kDqKSlots) * kStep, j > 0);
        ptx::mma_commit(ctx.bar(kDqKFree + j % kDqKSlots));
        if (j + 2 < nb) {
          if (!wait_k(j + 2)) break;
          if (j < 64) FMHA_BWD_TRACE(trow, 8 * j + 5);
          ptx::tc_fence_after();
          issue_s(j + 2);  // into the S buffer dQ(j) has just read (in order)
        }
      }
      if (issued_any) {
        ptx::mma_commit(ctx.bar(kDqDone));
        wait_drain(ctx, kDqDone, 0);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMmaDp) {
    // ================================ dP issuer
    if (lane == 0 && nb > 0) {
      const uint64_t do_desc = desc_kmajor(base + DqSmem::kOffDo);
      const uint64_t v_kmaj = desc_kmajor(base + DqSmem::kOffV);
      constexpr uint64_t kStep = kTile >> 4;
      bool issued_any = false;
      bool ok = wait_bar(ctx, kDqQFull, 0, kRoleMma);
      for (int j = 0; j < nb && ok; ++j) {
        if (j > 0) {
          // dP(j-1) is in the gradient warps' registers: dP(j) into its columns
          if (!wait_bar(ctx, kDqDpFree, (j - 1) & 1, kRoleMma)) break;
          if (j - 1 < 64) FMHA_BWD_TRACE(trow, 8 * (j - 1) + 3);
        }
        if (!wait_bar(ctx, kDqVFull + j % kDqVSlots, (j / kDqVSlots) & 1, kRoleMma)) break;
        if (j > 0 && j - 1 < 64) FMHA_BWD_TRACE(trow, 8 * (j - 1) + 6);
        ptx::tc_fence_after();
        issue_qk<128>(tmem + kDqColDp, do_desc, v_kmaj + (j % kDqVSlots) * kStep);  // dP(j) = dO V_j^T
        ptx::mma_commit(ctx.bar(kDqBlkReady + (j & 1)));  // dP(j): block j's other arrival
        issued_any = true;
      }
      if (issued_any) {
        ptx::mma_commit(ctx.bar(kDqDpDone));
        wait_drain(ctx, kDqDpDone, 0);
      }
    }
    __syncwarp();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ============================================================================ dK, dV
// Shared memory: K, V tiles, a 2-stage ring of (Q, dO) tiles with their rows'
// -LSE log2(e) and -D, barriers.
struct DkvSmem {
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffV = kTile;
  static constexpr uint32_t kOffRing = 2 * kTile;  // stage s: Q at + 2 s kTile, dO at + (2 s + 1) kTile
  static constexpr uint32_t kOffRow = kOffRing + 4 * kTile;  // stage s: -LSE log2e [128] at + 1024 s, -D [128] at + 1024 s + 512
  static constexpr uint32_t kOffBar = kOffRow + 2048;
  static constexpr uint32_t kOffMisc = kOffBar + 128;
  static constexpr uint32_t kBytes = kOffBar + 256 + 1024;
  static_assert(kBytes <= 232448, "shared memory per CTA");
};
constexpr int kKvKVFull = 0;      // K, V landed
constexpr int kKvStageFull = 1;   // [2] Q, dO and the row terms of stage s
constexpr int kKvStageFree = 3;   // [2] the MMAs reading stage s retired
constexpr int kKvHalfReady = 5;   // [2] S^T, dP^T of query half h in TMEM
constexpr int kKvPReady = 7;      // [2] P^T, dS^T of query half h stored (4 warps)
constexpr int kKvDone = 9;        // every MMA of the dV / dK issuer retired
constexpr int kKvDvDone = 10;     // [2] dV, dK of query half h retired: its TMEM columns are free
constexpr int kKvScoreDone = 12;  // every MMA of the score issuer retired
constexpr int kDkvThreads = 224;  // two MMA-issuing warps: scores (warp 5), dV / dK (warp 6)
// TMEM columns.  Each 128-query block is processed as two halves of 64
// queries: S^T of half h at 64 h, dP^T at 128 + 64 h (P^T and dS^T as bf16
// over their first 32 columns), dV at 256, dK at 384.
constexpr uint32_t kKvColDp = 128, kKvColDv = 256, kKvColDk = 384;
constexpr uint32_t kQHalfBytes = 64 * 128;  // 64 rows of a swizzled 64-column half

// S^T_h = K Q_h^T (or dP^T_h = V dO_h^T): M=128 keys, N=64 queries (rows
// 64 h .. 64 h + 63 of the Q tile, 8 KiB into each swizzled half), K=128 head
// dims in 8 steps.
__device__ __forceinline__ void issue_half_qk(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBlockM, 64, false, false);
  ptx::mma_ss_imm<false>(tmem_d, a_desc, b_desc, idesc);
#pragma unroll
  for (int k = 1; k < 8; ++k) {
    const uint64_t off = ((k >> 2) * kHalfBytes + (k & 3) * 32u) >> 4;
    ptx::mma_ss_imm<true>(tmem_d, a_desc + off, b_desc + off, idesc);
  }
}

// dV += P^T_h dO_h (or dK += dS^T_h Q_h): M=128 keys, N=128 head dims, K=64
// queries in 4 steps; A from TMEM (8 columns per step), B MN-major from the
// rows of half h.
__device__ __forceinline__ void issue_half_pv(uint32_t tmem_d, uint32_t tmem_a, uint64_t b_desc, bool accumulate) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBlockM, 128, false, true);
  if (accumulate)
    ptx::mma_ts_imm<true>(tmem_d, tmem_a, b_desc, idesc);
  else
    ptx::mma_ts_imm<false>(tmem_d, tmem_a, b_desc, idesc);
#pragma unroll
  for (int k = 1; k < 4; ++k) ptx::mma_ts_imm<true>(tmem_d, tmem_a + 8u * k, b_desc + ((2048u * k) >> 4), idesc);
}

__global__ void __launch_bounds__(kDkvThreads, 1) fmha_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (warp == kWarpProducer && lane == 0) {
    ptx::prefetch_tensormap(&p.tmap_q);
    ptx::prefetch_tensormap(&p.tmap_do);
    ptx::prefetch_tensormap(&p.tmap_k);
    ptx::prefetch_tensormap(&p.tmap_v);
  }
  const int hk = static_cast<int>(blockIdx.x);
  const int j0 = static_cast<int>(blockIdx.y) * kBlockN;
  const int b = static_cast<int>(blockIdx.z);
  int q0, lq, k0, lk;
  seq_bounds(p, b, q0, lq, k0, lk);
  if (j0 >= lk) return;
  const int off = lk - lq;
#ifdef FMHA_TRACE
  unsigned long long* trow =
      (g_trace_dkdv != nullptr && hk == 0 && b == 0) ? g_trace_dkdv + blockIdx.y * 1024ull : nullptr;
#else
  unsigned long long* trow = nullptr;
#endif
  if (threadIdx.x == 0) FMHA_BWD_TRACE(trow, 1000);
  // query blocks that see some key of this block: causal rows i see keys j <= i + off
  const int m_end = (lq + kBlockM - 1) / kBlockM;
  const int m_start = p.causal ? max(0, j0 - off) / kBlockM : 0;
  const int nm = max(0, m_end - m_start);
  const int group = p.kv_group;
  const int n_items = group * nm;  // item it: query head hk * group + it / nm, query block m_start + it % nm
  const int xkv = hk * 128;

  Ctx ctx;
  ctx.bar0 = base + DkvSmem::kOffBar;
  ctx.abort_flag = reinterpret_cast<volatile uint32_t*>(smem + DkvSmem::kOffMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + DkvSmem::kOffMisc);

  if (warp == kWarpProducer && lane == 0) {
    ptx::mbar_init(ctx.bar(kKvKVFull), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ctx.bar(kKvStageFull + s), 1);
      ptx::mbar_init(ctx.bar(kKvStageFree + s), 1);
      ptx::mbar_init(ctx.bar(kKvHalfReady + s), 1);
      ptx::mbar_init(ctx.bar(kKvPReady + s), 4);
      ptx::mbar_init(ctx.bar(kKvDvDone + s), 1);
    }
    ptx::mbar_init(ctx.bar(kKvDone), 1);
    ptx::mbar_init(ctx.bar(kKvScoreDone), 1);
    *ctx.abort_flag = 0u;
    ptx::fence_mbar_init();
    if (n_items > 0) {
      const uint64_t pol = ptx::policy_evict_first();
      const uint32_t bar = ctx.bar(kKvKVFull);
      ptx::mbar_arrive_expect_tx(bar, 2 * kTile);
      const int y = k0 + j0;
      ptx::tma_load_2d(base + DkvSmem::kOffK, &p.tmap_k, bar, xkv, y, pol);
      ptx::tma_load_2d(base + DkvSmem::kOffK + kHalfBytes, &p.tmap_k, bar, xkv + 64, y, pol);
      ptx::tma_load_2d(base + DkvSmem::kOffV, &p.tmap_v, bar, xkv, y, pol);
      ptx::tma_load_2d(base + DkvSmem::kOffV + kHalfBytes, &p.tmap_v, bar, xkv + 64, y, pol);
    }
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ================================ gradient math: one key row per thread
    const int r = warp * 32 + lane;
    const int jr = j0 + r;  // sequence-local key index
    const uint32_t lane_base = tmem + ((static_cast<uint32_t>(warp) * 32u) << 16);
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    const bool tr = r == 0 && trow != nullptr;
    if (tr) FMHA_BWD_TRACE(trow, 1001);
    bool ok = true;
    for (int it = 0; it < n_items && ok; ++it) {
      const int s = it & 1;
      const int m = m_start + it % nm;
      // the row terms of this stage (written by the producer's threads)
      if (!wait_bar_warp(ctx, kKvStageFull + s, (it >> 1) & 1, kRoleSoftmax)) break;
      if (tr && it < 64) FMHA_BWD_TRACE(trow, 8 * it + 0);
      // causal: key jr is visible to query column cq iff jr <= m * 128 + cq + off
      const bool need_mask = p.causal && (m * kBlockM + off < j0 + kBlockN - 1);
      const int cmin = jr - off - m * kBlockM;  // first visible column
      const uint32_t rowterms = base + DkvSmem::kOffRow + 1024u * s;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        if (!wait_bar_warp(ctx, kKvHalfReady + hf, it & 1, kRoleSoftmax)) {
          ok = false;
          break;
        }
        if (tr && it < 64) FMHA_BWD_TRACE(trow, 8 * it + 1 + 2 * hf);
        ptx::tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float st[32], dpt[32];
          ptx::tmem_ld32x2_wait(lane_base + 64u * hf + 32u * cc, st, lane_base + kKvColDp + 64u * hf + 32u * cc,
                                dpt);
          uint32_t pk[16], dk16[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = 64 * hf + 32 * cc + 2 * i;
            const float2 nl = ptx::ld_shared_v2f(rowterms + 4u * col);
            const float2 nd = ptx::ld_shared_v2f(rowterms + 512u + 4u * col);
            const float2 x = __ffma2_rn(make_float2(st[2 * i], st[2 * i + 1]), c2, nl);
            float p0 = ptx::ex2_approx(x.x);
            float p1 = ptx::ex2_approx(x.y);
            if (need_mask) {
              p0 = col >= cmin ? p0 : 0.f;
              p1 = col + 1 >= cmin ? p1 : 0.f;
            }
            const float2 g = __fadd2_rn(make_float2(dpt[2 * i], dpt[2 * i + 1]), nd);  // dP - D
            const float2 ds = __fmul2_rn(make_float2(p0, p1), g);
            pk[i] = ptx::pack_bf16x2(p0, p1);
            dk16[i] = ptx::pack_bf16x2(ds.x, ds.y);
          }
          ptx::tmem_st16(lane_base + 64u * hf + 16u * cc, pk);
          ptx::tmem_st16(lane_base + kKvColDp + 64u * hf + 16u * cc, dk16);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ctx.bar(kKvPReady + hf));
        if (tr && it < 64) FMHA_BWD_TRACE(trow, 8 * it + 2 + 2 * hf);
      }
    }
    if (tr) FMHA_BWD_TRACE(trow, 1002);
    // ---- epilogue: dV, dK * scale -> bf16 (keys of the sequence only)
    const bool have = n_items > 0 && wait_bar_warp(ctx, kKvDone, 0, kRoleSoftmax);
    if (have) ptx::tc_fence_after();
    const bool valid = jr < lk;
    const size_t e = (static_cast<size_t>(k0 + jr) * p.kv_heads + hk) * 128;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      __nv_bfloat16* dst = (which == 0 ? p.dv : p.dk) + e;
      const float f = which == 0 ? 1.f : p.scale;
      const uint32_t col0 = which == 0 ? kKvColDv : kKvColDk;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float o[32];
        if (have) {
          ptx::tmem_ld32_wait(lane_base + col0 + 32u * cc, o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
        }
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * cc);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 w;
            w.x = ptx::pack_bf16x2(o[8 * v4 + 0] * f, o[8 * v4 + 1] * f);
            w.y = ptx::pack_bf16x2(o[8 * v4 + 2] * f, o[8 * v4 + 3] * f);
            w.z = ptx::pack_bf16x2(o[8 * v4 + 4] * f, o[8 * v4 + 5] * f);
            w.w = ptx::pack_bf16x2(o[8 * v4 + 6] * f, o[8 * v4 + 7] * f);
            d4[v4] = w;
          }
        }
      }
    }
  } else if (warp == kWarpProducer) {
    // ================================ producer: (Q, dO) tiles and their row terms
    const uint64_t pol = ptx::policy_evict_last();
    int issued = 0;
    bool ok = true;
    for (int it = 0; it < n_items && ok; ++it) {
      const int s = it & 1;
      const int h = hk * group + it / nm;
      const int m = m_start + it % nm;
      // row terms: -LSE log2(e) and -D of the block's 128 query rows (rows
      // past the sequence end get -inf, so their P is 0), read from global
      // memory before waiting for the stage so that the wait hides them
      float nl[4], dd[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int qr = m * kBlockM + 4 * lane + i;
        nl[i] = -INFINITY;
        dd[i] = 0.f;
        if (qr < lq) {
          const size_t li = static_cast<size_t>(h) * p.total_q + q0 + qr;
          nl[i] = neg_lse2(p.lse[li]);
          dd[i] = -p.dvec[li];
        }
      }
      if (it >= 2) ok = wait_bar_warp(ctx, kKvStageFree + s, ((it >> 1) - 1) & 1, kRoleLoad);
      if (!ok) break;
      if (lane == 0 && it < 64) FMHA_BWD_TRACE(trow, 8 * it + 7);
      const uint32_t rowterms = base + DkvSmem::kOffRow + 1024u * s;
      ptx::st_shared_v4f(rowterms + 16u * lane, nl[0], nl[1], nl[2], nl[3]);
      ptx::st_shared_v4f(rowterms + 512u + 16u * lane, dd[0], dd[1], dd[2], dd[3]);
      __syncwarp();
      if (lane == 0) {
        const uint32_t bar = ctx.bar(kKvStageFull + s);
        ptx::mbar_arrive_expect_tx(bar, 2 * kTile);
        const uint32_t dst = base + DkvSmem::kOffRing + 2u * s * kTile;
        const int y = q0 + m * kBlockM;
        const int x = h * 128;
        ptx::tma_load_2d(dst, &p.tmap_q, bar, x, y, pol);
        ptx::tma_load_2d(dst + kHalfBytes, &p.tmap_q, bar, x + 64, y, pol);
        ptx::tma_load_2d(dst + kTile, &p.tmap_do, bar, x, y, pol);
        ptx::tma_load_2d(dst + kTile + kHalfBytes, &p.tmap_do, bar, x + 64, y, pol);
      }
      ++issued;
    }
    if (lane == 0) {
      for (int it = max(0, issued - 2); it < issued; ++it) wait_drain(ctx, kKvStageFull + (it & 1), (it >> 1) & 1);
      if (n_items > 0) wait_drain(ctx, kKvKVFull, 0);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ================================ score issuer
    // Per item (query block), per half h of 64 queries: S^T and dP^T into the
    // half's columns once the dV / dK issuer's products of the previous item
    // have read them.  Two issuing threads because issue is paced by the
    // tensor pipe: one thread blocked on its own queue would see the other
    // stream's hand-offs late.
    if (lane == 0 && n_items > 0) {
      const uint64_t k_desc = desc_kmajor(base + DkvSmem::kOffK);
      const uint64_t v_desc = desc_kmajor(base + DkvSmem::kOffV);
      constexpr uint64_t kHalfRows = kQHalfBytes >> 4;  // rows 64.. of a tile, in descriptor units
      bool issued_any = false;
      bool ok = wait_bar(ctx, kKvKVFull, 0, kRoleMma);
      for (int it = 0; it < n_items && ok; ++it) {
        const uint32_t q_tile = base + DkvSmem::kOffRing + 2u * (it & 1) * kTile;
        if (!wait_bar(ctx, kKvStageFull + (it & 1), (it >> 1) & 1, kRoleMma)) break;
        if (it < 60) FMHA_BWD_TRACE(trow, 512 + 8 * it + 0);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (it > 0 && !wait_bar(ctx, kKvDvDone + hf, (it - 1) & 1, kRoleMma)) {
            ok = false;
            break;
          }
          if (it < 60) FMHA_BWD_TRACE(trow, 512 + 8 * it + 1 + hf);
          ptx::tc_fence_after();
          const uint64_t q_kmaj = desc_kmajor(q_tile) + hf * kHalfRows;
          const uint64_t do_kmaj = desc_kmajor(q_tile + kTile) + hf * kHalfRows;
          issue_half_qk(tmem + 64u * hf, k_desc, q_kmaj);             // S^T_h = K Q_h^T
          issue_half_qk(tmem + kKvColDp + 64u * hf, v_desc, do_kmaj);  // dP^T_h = V dO_h^T
          ptx::mma_commit(ctx.bar(kKvHalfReady + hf));
          if (hf == 1 && it < 60) FMHA_BWD_TRACE(trow, 512 + 8 * it + 3);
          issued_any = true;
        }
      }
      if (issued_any) {
        ptx::mma_commit(ctx.bar(kKvScoreDone));
        wait_drain(ctx, kKvScoreDone, 0);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma + 1) {
    // ================================ dV / dK issuer
    if (lane == 0 && n_items > 0) {
      constexpr uint64_t kHalfRows = kQHalfBytes >> 4;
      bool issued_any = false;
      bool ok = true;
      for (int it = 0; it < n_items && ok; ++it) {
        const uint32_t q_tile = base + DkvSmem::kOffRing + 2u * (it & 1) * kTile;
        // the item's Q and dO tiles (complete by now; observed by this thread too)
        if (!wait_bar(ctx, kKvStageFull + (it & 1), (it >> 1) & 1, kRoleMma)) break;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (!wait_bar(ctx, kKvPReady + hf, it & 1, kRoleMma)) {
            ok = false;
            break;
          }
          if (it < 64) FMHA_BWD_TRACE(trow, 8 * it + 5 + hf);
          ptx::tc_fence_after();
          const bool acc = it > 0 || hf > 0;
          const uint64_t q_mn = desc_mnmajor(q_tile) + hf * kHalfRows;
          const uint64_t do_mn = desc_mnmajor(q_tile + kTile) + hf * kHalfRows;
          issue_half_pv(tmem + kKvColDv, tmem + 64u * hf, do_mn, acc);             // dV += P^T_h dO_h
          issue_half_pv(tmem + kKvColDk, tmem + kKvColDp + 64u * hf, q_mn, acc);   // dK += dS^T_h Q_h
          ptx::mma_commit(ctx.bar(kKvDvDone + hf));
          if (hf == 1) ptx::mma_commit(ctx.bar(kKvStageFree + (it & 1)));  // the item's Q, dO read by both issuers
          if (it < 60) FMHA_BWD_TRACE(trow, 512 + 8 * it + 4 + hf);
          issued_any = true;
        }
      }
      if (issued_any) {
        ptx::mma_commit(ctx.bar(kKvDone));
        wait_drain(ctx, kKvDone, 0);
      }
    }
    __syncwarp();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace bwd
}  // namespace fmha
