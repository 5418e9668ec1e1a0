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
// Two kernels, no atomics (every output row is written by one CTA):
//   fmha_bwd_dq_kernel    one CTA per (head, 128 query rows, sequence): first
//                         D_i (written to the workspace for the second kernel),
//                         then per 128-key block S = Q K^T and dP = dO V^T into
//                         TMEM, dS in bf16 over S, dQ += dS K.
//   fmha_bwd_dkdv_kernel  one CTA per (K/V head, 128 keys, sequence): per query
//                         block of every query head of the group, S^T = K Q^T
//                         and dP^T = V dO^T into TMEM, P^T and dS^T in bf16 over
//                         them, dV += P^T dO and dK += dS^T Q.
// Every GEMM is a tcgen05.mma of one of the forward's two forms: both operands
// K-major in shared memory, or A from TMEM with an MN-major B.  Warp roles
// (192 threads): warps 0-3 the gradient math on one TMEM lane (row) each and
// the epilogue; warp 4 the TMA producer; warp 5 the MMA issuer and TMEM owner.
// Every mbarrier wait is bounded as in the forward kernel.
#pragma once

#include "fmha_fwd_kernel.cuh"

namespace fmha {
namespace bwd {

constexpr int kThreads = 192;
constexpr int kWarpProducer = 4;
constexpr int kWarpMma = 5;
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

// ============================================================================ dQ
// Shared memory: Q, dO tiles, a 2-stage ring of (K, V) blocks, barriers.
struct DqSmem {
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffDo = kTile;
  static constexpr uint32_t kOffRing = 2 * kTile;  // stage s: K at + 2 s kTile, V at + (2 s + 1) kTile
  static constexpr uint32_t kOffBar = kOffRing + 4 * kTile;
  static constexpr uint32_t kOffMisc = kOffBar + 128;
  static constexpr uint32_t kBytes = kOffBar + 256 + 1024;
  static_assert(kBytes <= 232448, "shared memory per CTA");
};
// barrier ids
constexpr int kDqQFull = 0;      // Q and dO landed
constexpr int kDqKVFull = 1;     // [2] K_j, V_j of stage j & 1 landed
constexpr int kDqStageFree = 3;  // [2] the MMAs reading stage s retired
constexpr int kDqSReady = 5;     // S(j), dP(j) in TMEM
constexpr int kDqPReady = 6;     // dS(j) stored (4 warps)
constexpr int kDqDone = 7;       // every MMA retired
// TMEM columns.  The bf16 pairs of a 32-column chunk of S (or dP) are stored
// over columns 16 c .. 16 c + 15 of the same tensor, which the chunk loads of
// this row have already read.
constexpr uint32_t kDqColS = 0, kDqColDp = 128, kDqColDq = 256;

__global__ void __launch_bounds__(kThreads, 1) fmha_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
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
  const int xkv = (h / p.kv_group) * 128;

  Ctx ctx;
  ctx.bar0 = base + DqSmem::kOffBar;
  ctx.abort_flag = reinterpret_cast<volatile uint32_t*>(smem + DqSmem::kOffMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + DqSmem::kOffMisc);

  auto load_kv = [&](int j, uint64_t pol) {
    const int s = j & 1;
    const uint32_t bar = ctx.bar(kDqKVFull + s);
    ptx::mbar_arrive_expect_tx(bar, 2 * kTile);
    const uint32_t dk = base + DqSmem::kOffRing + 2u * s * kTile;
    const int y = k0 + kBlockN * j;
    ptx::tma_load_2d(dk, &p.tmap_k, bar, xkv, y, pol);
    ptx::tma_load_2d(dk + kHalfBytes, &p.tmap_k, bar, xkv + 64, y, pol);
    ptx::tma_load_2d(dk + kTile, &p.tmap_v, bar, xkv, y, pol);
    ptx::tma_load_2d(dk + kTile + kHalfBytes, &p.tmap_v, bar, xkv + 64, y, pol);
  };
  const int early = min(2, nb);

  if (warp == kWarpProducer && lane == 0) {
    ptx::mbar_init(ctx.bar(kDqQFull), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ctx.bar(kDqKVFull + s), 1);
      ptx::mbar_init(ctx.bar(kDqStageFree + s), 1);
    }
    ptx::mbar_init(ctx.bar(kDqSReady), 1);
    ptx::mbar_init(ctx.bar(kDqPReady), 4);
    ptx::mbar_init(ctx.bar(kDqDone), 1);
    *ctx.abort_flag = 0u;
    ptx::fence_mbar_init();
    if (nb > 0) {
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint64_t pol_kv = ptx::policy_evict_last();
      const uint32_t bar = ctx.bar(kDqQFull);
      ptx::mbar_arrive_expect_tx(bar, 2 * kTile);
      const int y = q0 + r0;
      ptx::tma_load_2d(base + DqSmem::kOffQ, &p.tmap_q, bar, xq, y, pol_q);
      ptx::tma_load_2d(base + DqSmem::kOffQ + kHalfBytes, &p.tmap_q, bar, xq + 64, y, pol_q);
      ptx::tma_load_2d(base + DqSmem::kOffDo, &p.tmap_do, bar, xq, y, pol_q);
      ptx::tma_load_2d(base + DqSmem::kOffDo + kHalfBytes, &p.tmap_do, bar, xq + 64, y, pol_q);
      for (int j = 0; j < early; ++j) load_kv(j, pol_kv);
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
      // D_i = dO_i . O_i (fp32), also kept for the dK/dV kernel
      const size_t e = (static_cast<size_t>(q0 + row) * p.heads + h) * 128;
      const uint4* o4 = reinterpret_cast<const uint4*>(p.out + e);
      const uint4* g4 = reinterpret_cast<const uint4*>(p.dout + e);
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const uint4 a = o4[i], g = g4[i];
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 af = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[k]));
          const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[k]));
          acc0 = fmaf(af.x, gf.x, acc0);
          acc1 = fmaf(af.y, gf.y, acc1);
        }
      }
      dval = acc0 + acc1;
      const size_t li = static_cast<size_t>(h) * p.total_q + q0 + row;
      p.dvec[li] = dval;
      nl2 = neg_lse2(p.lse[li]);
    }
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    const float2 nl2_2 = make_float2(nl2, nl2);
    const float2 nd2 = make_float2(-dval, -dval);
    const int key_end = p.causal ? min(row + off + 1, lk) : lk;              // this row's visible keys
    const int tile_key_end = p.causal ? min(r0 + off + 1, lk) : lk;          // the tile's first row's
    for (int j = 0; j < nb; ++j) {
      if (!wait_bar_warp(ctx, kDqSReady, j & 1, kRoleSoftmax)) break;
      ptx::tc_fence_after();
      const bool need_mask = tile_key_end - j * kBlockN < kBlockN;  // diagonal or key tail
      const int lim = key_end - j * kBlockN;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float s[32], dp[32];
        ptx::tmem_ld32x2_wait(lane_base + kDqColS + 32u * cc, s, lane_base + kDqColDp + 32u * cc, dp);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 x = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), c2, nl2_2);
          float p0 = ptx::ex2_approx(x.x);
          float p1 = ptx::ex2_approx(x.y);
          if (need_mask) {
            const int col = 32 * cc + 2 * i;
            p0 = col < lim ? p0 : 0.f;
            p1 = col + 1 < lim ? p1 : 0.f;
          }
          const float2 g = __fadd2_rn(make_float2(dp[2 * i], dp[2 * i + 1]), nd2);  // dP - D
          const float2 ds = __fmul2_rn(make_float2(p0, p1), g);
          pk[i] = ptx::pack_bf16x2(ds.x, ds.y);
        }
        ptx::tmem_st16(lane_base + kDqColS + 16u * cc, pk);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ctx.bar(kDqPReady));
    }
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
    // ================================ TMA producer: K/V blocks 2.. through the ring
    if (lane == 0) {
      const uint64_t pol_kv = ptx::policy_evict_last();
      int issued = early;
      for (int j = early; j < nb; ++j) {
        // stage j & 1 last held block j - 2, read by the MMAs of step j - 2
        if (!wait_bar(ctx, kDqStageFree + (j & 1), ((j >> 1) - 1) & 1, kRoleLoad)) break;
        load_kv(j, pol_kv);
        ++issued;
      }
      for (int j = max(0, issued - 2); j < issued; ++j) wait_drain(ctx, kDqKVFull + (j & 1), (j >> 1) & 1);
      if (nb > 0) wait_drain(ctx, kDqQFull, 0);
    }
    __syncwarp();
  } else {
    // ================================ MMA issuer
    if (lane == 0 && nb > 0) {
      const uint64_t q_desc = desc_kmajor(base + DqSmem::kOffQ);
      const uint64_t do_desc = desc_kmajor(base + DqSmem::kOffDo);
      const uint64_t ring_kmaj = desc_kmajor(base + DqSmem::kOffRing);
      const uint64_t ring_mn = desc_mnmajor(base + DqSmem::kOffRing);
      constexpr uint64_t kStep = kTile >> 4;  // descriptor units of one tile
      bool issued_any = false;
      bool ok = wait_bar(ctx, kDqQFull, 0, kRoleMma) && wait_bar(ctx, kDqKVFull, 0, kRoleMma);
      if (ok) {
        ptx::tc_fence_after();
        issue_qk<128>(tmem + kDqColS, q_desc, ring_kmaj);               // S(0) = Q K_0^T
        issue_qk<128>(tmem + kDqColDp, do_desc, ring_kmaj + kStep);     // dP(0) = dO V_0^T
        ptx::mma_commit(ctx.bar(kDqSReady));
        issued_any = true;
      }
      for (int j = 0; j < nb && ok; ++j) {
        const int s = j & 1;
        if (!wait_bar(ctx, kDqPReady, j & 1, kRoleMma)) break;
        ptx::tc_fence_after();
        // dQ += dS(j) K_j: A = dS (bf16 over S), B = K_j MN-major
        issue_pv<128>(tmem + kDqColDq, tmem + kDqColS, ring_mn + 2 * s * kStep, j > 0);
        ptx::mma_commit(ctx.bar(kDqStageFree + s));
        if (j + 1 < nb) {
          const int s1 = (j + 1) & 1;
          if (!wait_bar(ctx, kDqKVFull + s1, ((j + 1) >> 1) & 1, kRoleMma)) break;
          ptx::tc_fence_after();
          issue_qk<128>(tmem + kDqColS, q_desc, ring_kmaj + 2 * s1 * kStep);
          issue_qk<128>(tmem + kDqColDp, do_desc, ring_kmaj + (2 * s1 + 1) * kStep);
          ptx::mma_commit(ctx.bar(kDqSReady));
        }
      }
      if (issued_any) {
        ptx::mma_commit(ctx.bar(kDqDone));
        wait_drain(ctx, kDqDone, 0);
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
constexpr int kKvSReady = 5;      // S^T, dP^T in TMEM
constexpr int kKvPReady = 6;      // P^T, dS^T stored (4 warps)
constexpr int kKvDone = 7;        // every MMA retired
constexpr uint32_t kKvColS = 0, kKvColDp = 128, kKvColDv = 256, kKvColDk = 384;

__global__ void __launch_bounds__(kThreads, 1) fmha_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
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
    }
    ptx::mbar_init(ctx.bar(kKvSReady), 1);
    ptx::mbar_init(ctx.bar(kKvPReady), 4);
    ptx::mbar_init(ctx.bar(kKvDone), 1);
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
    for (int it = 0; it < n_items; ++it) {
      const int s = it & 1;
      const int m = m_start + it % nm;
      // the row terms of this stage (written by the producer's threads) and S^T, dP^T
      if (!wait_bar_warp(ctx, kKvStageFull + s, (it >> 1) & 1, kRoleSoftmax)) break;
      if (!wait_bar_warp(ctx, kKvSReady, it & 1, kRoleSoftmax)) break;
      ptx::tc_fence_after();
      // causal: key jr is visible to query column cq iff jr <= m * 128 + cq + off
      const bool need_mask = p.causal && (m * kBlockM + off < j0 + kBlockN - 1);
      const int cmin = jr - off - m * kBlockM;  // first visible column
      const uint32_t rowterms = base + DkvSmem::kOffRow + 1024u * s;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float st[32], dpt[32];
        ptx::tmem_ld32x2_wait(lane_base + kKvColS + 32u * cc, st, lane_base + kKvColDp + 32u * cc, dpt);
        uint32_t pk[16], dk16[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = 32 * cc + 2 * i;
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
        ptx::tmem_st16(lane_base + kKvColS + 16u * cc, pk);
        ptx::tmem_st16(lane_base + kKvColDp + 16u * cc, dk16);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ctx.bar(kKvPReady));
    }
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
      if (it >= 2) ok = wait_bar_warp(ctx, kKvStageFree + s, ((it >> 1) - 1) & 1, kRoleLoad);
      if (!ok) break;
      // row terms: -LSE log2(e) and -D of the block's 128 query rows (rows
      // past the sequence end get -inf, so their P is 0)
      const uint32_t rowterms = base + DkvSmem::kOffRow + 1024u * s;
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
  } else {
    // ================================ MMA issuer
    if (lane == 0 && n_items > 0) {
      const uint64_t k_desc = desc_kmajor(base + DkvSmem::kOffK);
      const uint64_t v_desc = desc_kmajor(base + DkvSmem::kOffV);
      const uint64_t ring_kmaj = desc_kmajor(base + DkvSmem::kOffRing);
      const uint64_t ring_mn = desc_mnmajor(base + DkvSmem::kOffRing);
      constexpr uint64_t kStep = kTile >> 4;
      bool issued_any = false;
      bool ok = wait_bar(ctx, kKvKVFull, 0, kRoleMma) && wait_bar(ctx, kKvStageFull, 0, kRoleMma);
      if (ok) {
        ptx::tc_fence_after();
        issue_qk<128>(tmem + kKvColS, k_desc, ring_kmaj);            // S^T(0) = K Q_0^T
        issue_qk<128>(tmem + kKvColDp, v_desc, ring_kmaj + kStep);   // dP^T(0) = V dO_0^T
        ptx::mma_commit(ctx.bar(kKvSReady));
        issued_any = true;
      }
      for (int it = 0; it < n_items && ok; ++it) {
        const int s = it & 1;
        if (!wait_bar(ctx, kKvPReady, it & 1, kRoleMma)) break;
        ptx::tc_fence_after();
        issue_pv<128>(tmem + kKvColDv, tmem + kKvColS, ring_mn + (2 * s + 1) * kStep, it > 0);  // dV += P^T dO
        issue_pv<128>(tmem + kKvColDk, tmem + kKvColDp, ring_mn + 2 * s * kStep, it > 0);       // dK += dS^T Q
        ptx::mma_commit(ctx.bar(kKvStageFree + s));
        if (it + 1 < n_items) {
          const int s1 = (it + 1) & 1;
          if (!wait_bar(ctx, kKvStageFull + s1, ((it + 1) >> 1) & 1, kRoleMma)) break;
          ptx::tc_fence_after();
          issue_qk<128>(tmem + kKvColS, k_desc, ring_kmaj + 2 * s1 * kStep);
          issue_qk<128>(tmem + kKvColDp, v_desc, ring_kmaj + (2 * s1 + 1) * kStep);
          ptx::mma_commit(ctx.bar(kKvSReady));
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
