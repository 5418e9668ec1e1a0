// fmha_fwd_kernel.cuh -- fused attention forward for sm_103a.
//
// O = softmax(scale * Q K^T [+ causal mask]) V and the per-row log-sum-exp, for
// bf16 [tokens, heads, head_dim] tensors (head_dim 128 or 64), dense or varlen
// (cu_seqlens), after
// "[BUG] Unexpected Slower Performance in C++ CuTe (77_blackwell_fmha) vs
// Python CuTe DSL (fmha.py) on Jetson Thor" (sections "Test Commands" and
// "Implementation Differences in softmax_step") and "[BUG] CuTe DSL 4.7/4.8
// regression: FlashAttention-4 SM100 forward kernel spills registers"
// (section "Steps/Code to reproduce bug": varlen causal forward, 512 threads
// per CTA at a 128-register entry budget).
//
// One CTA owns a work unit (sequence b, head h, 256 query rows = two 128-row
// tiles) and walks the unit's 128-key blocks.  Warp roles (512 threads):
//   warpgroup 0, 1  softmax for tile 0 / tile 1: tcgen05.ld the S row, track
//                   the running max, fold scale and -max into one packed FMA,
//                   ex2, row sum, convert P to bf16 and tcgen05.st it over S;
//                   then the tile's epilogue (O / l -> bf16 global, LSE);
//                   when a row max moved past the lazy threshold the softmax
//                   warps rescale their own O rows in TMEM;
//   warpgroup 2     idle (its registers go to the softmax warpgroups);
//   warp 12         TMA producer: Q tiles once, then a K/V ring in shared
//                   memory whose slots the MMA warp's step commits free;
//   warp 13         MMA issuer: tcgen05.mma S = Q K^T (both operands in
//                   shared memory) and O += P V (P from TMEM), completion
//                   signalled with tcgen05.commit on mbarriers;
//   warps 14, 15    idle (barrier observers in the trace build).
// Tensor memory (512 columns): S0/P0 [0,128), S1/P1 [128,256), O0 [256,384),
// O1 [384,512) (head_dim 64 uses the first 64 columns of each O).  P (bf16
// pairs) overwrites the first 64 columns of its S.
//
// Every mbarrier wait is bounded in time: on expiry the kernel records an
// error word, raises a CTA-wide abort flag, lets in-flight copies and MMAs
// drain (again bounded), frees its tensor memory and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace fmha {

constexpr int kBlockM = 128;   // query rows per tile (MMA M)
constexpr int kBlockN = 128;   // keys per block (MMA N of QK^T, K of PV)
constexpr int kTiles = 2;      // query tiles per CTA (at most; barriers exist for both)
constexpr int kThreads = 512;

// A tile (128 rows: queries, keys or values) is stored as 64-column halves
// of 128 rows x 128 bytes (16 KiB, 128-byte swizzle): one half for head_dim
// 64, two for head_dim 128.
constexpr uint32_t kHalfBytes = kBlockM * 64 * 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kNumBars = 16;
static_assert(kNumBars * 8 <= 256, "barrier area");

// Sizes that depend on the head dimension (64, 128 or 256).  Shared memory
// map, offsets from a 1024-byte aligned base: Q tiles, the K/V ring, barriers,
// misc words.
//   head_dim 64, 128: two query tiles per CTA, a K/V ring of four slots (two
//     key blocks in flight), TMEM S0 S1 O0 O1 of 128 columns each.
//   head_dim 256: one query tile per CTA (O alone takes 256 TMEM columns: S
//     [0, 128), O [256, 512)), a ring of two 64 KiB slots (K_j, V_j).
// The slot-release protocol (load idx reuses the slot of load idx - kStages,
// freed by a step commit) holds for either ring: a K slot is refilled after
// the QK^T that read it has committed and a V slot after its PV, so no
// barrier is ever waited on more than one phase late.
template <int HD>
struct Dims {
  static_assert(HD == 64 || HD == 128 || HD == 256, "head_dim");
  static constexpr int kHeadDim = HD;
  static constexpr int kHalves = HD / 64;
  static constexpr int kTiles = HD == 256 ? 1 : 2;   // query tiles per CTA
  static constexpr int kStages = HD == 256 ? 2 : 4;  // K/V ring slots
  static constexpr uint32_t kTileBytes = kBlockM * HD * 2;  // one Q tile / K or V block
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKV = kOffQ + kTiles * kTileBytes;
  static constexpr uint32_t kOffBar = kOffKV + kStages * kTileBytes;
  static constexpr uint32_t kOffMisc = kOffBar + 256;  // tmem base slot, abort flag
  static constexpr uint32_t kSmemBytes = kOffBar + 512 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Barrier ids.  Every tcgen05.commit stalls the tensor pipe for ~70-140
// cycles (measured), so the MMA warp commits twice per KV step: S ready for
// tile 0 when both tiles run, and one step commit.  Step commit n (n = 0 after
// the first QK^T, n = j + 1 after step j) goes to StepDone[n & 1]; it tells the
// last tile of the step that its S is ready and the producer that the step's
// ring slots are free.
constexpr int kBarQFull = 0;     // [2]
constexpr int kBarKVFull = 2;    // [4] (the ring's slots)
constexpr int kBarStepDone = 6;  // [2]  step commit n, alternating
constexpr int kBarSFull0 = 8;    //      QK^T of tile 0 landed (tile 0 not the last tile)
constexpr int kBarPVReady = 9;   // [2]  P of tile t stored (and its O rows rescaled)
constexpr int kBarOFinal = 11;   // [2]  last PV of tile t complete
constexpr int kBarMmaDone = 13;  //      every MMA retired
constexpr int kBarPVPart = 14;   // [2]  first part of P of tile t stored (split hand-off only)
// one query tile per CTA (two ring slots): V_m's slot free after PV(m), on the
// ring barriers the two-slot ring leaves unused
constexpr int kBarVFree = kBarKVFull + 2;  // [2]
static_assert(kBarPVPart + 2 == static_cast<int>(kNumBars), "ids");

// P hand-off split ("Kernel Bottleneck Tuning", section "5. Tune the
// producer->consumer handoff split"): the softmax stores P in four chunks of
// 32 keys and signals after the first FMHA_P_SPLIT of them, so that the MMA
// warp starts O += P V on those keys while the rest is exponentiated; 4 (the
// default) is one hand-off after the whole row.
#ifndef FMHA_P_SPLIT
#define FMHA_P_SPLIT 4
#endif
constexpr int kPSplit = FMHA_P_SPLIT;
static_assert(kPSplit >= 1 && kPSplit <= 4, "P split in quarters of the key block");
// Safety contract of the split: the PV K-steps the MMA warp issues after the
// first signal (16 keys each) must not reach past the keys the softmax stored
// before it, or an MMA reads P columns not yet written.
constexpr int kPvStepsBeforeFull = 2 * kPSplit;
static_assert(kPvStepsBeforeFull * 16 <= kPSplit * 32, "P split: consumer ahead of producer");
// The same knob for the FP8 PV variant (its PV K-steps are 32 keys, one per
// quarter), tuned separately: the pages report a 3/4 split best for an FP8 PV
// on B300.
#ifndef FMHA_P_SPLIT_FP8
#define FMHA_P_SPLIT_FP8 4
#endif
constexpr int kPSplitFp8 = FMHA_P_SPLIT_FP8;
static_assert(kPSplitFp8 >= 1 && kPSplitFp8 <= 4, "FP8 P split in quarters of the key block");


// Warpgroup of each role.  Warp w reaches TMEM lanes 32 (w % 4) .. + 31, so
// any warpgroup could hold a tile's softmax (placing the control warpgroup
// first measured the same).
constexpr int kWgControl = 3;
constexpr int kWgSoftmax0 = 0;  // softmax of tile 0; tile 1 is the next warpgroup
constexpr int kWgIdle = 2;
constexpr int kWarpProducer = 4 * kWgControl;      // TMA producer, barrier set-up
constexpr int kWarpMma = 4 * kWgControl + 1;       // MMA issuer, TMEM owner

// roles, for the timeout detail word
constexpr int kRoleSoftmax = 1, kRoleLoad = 3, kRoleMma = 4, kRoleDrain = 5;

#ifndef FMHA_WAIT_LIMIT_NS
#define FMHA_WAIT_LIMIT_NS 1000000000ull
#endif
constexpr uint64_t kWaitLimitNs = FMHA_WAIT_LIMIT_NS;  // per wait (1 s by default)

// Register budgets per warpgroup after the split (sum x 128 threads = 64K).
// Helper calls in these regions must be inlined: ptxas cannot place an ABI
// call inside a setmaxnreg region.
// Warpgroup 2 has no work (the softmax warps rescale their own O rows) and
// gives its registers to the softmax.
constexpr int kRegsSoftmax = 200, kRegsIdle = 32, kRegsControl = 80;
static_assert(2 * kRegsSoftmax + kRegsIdle + kRegsControl == 512, "register split");
// head_dim 256 (one query tile): warpgroup 1 has no tile and idles too; its
// registers go to the softmax warpgroup (eight 32-column O chunks in the
// rescale and the epilogue) and to the control warpgroup (its MMA issuer holds
// the descriptors of 16 K-steps per QK^T).
constexpr int kRegsSoftmax1 = 224, kRegsIdle1 = 32, kRegsControl1 = 512 - kRegsSoftmax1 - 2 * kRegsIdle1;
static_assert(kRegsControl1 % 8 == 0 && kRegsControl1 <= 256 && kRegsControl1 > 128, "register split, one tile");

struct alignas(64) FwdParams {
  CUtensorMap tmap_q;  // [total_q, heads*128] bf16, box 64 x 128, 128B swizzle
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  __nv_bfloat16* out;
  float* lse;  // [heads, total_q] or nullptr
  const int32_t* cu_q;
  const int32_t* cu_k;
  int batch, total_q, total_k, max_seqlen_q, max_seqlen_k, heads;
  int causal;
  int kv_group;             // query heads per K/V head (heads / kv_heads)
  float scale_log2;         // scale * log2(e)
  float rescale_threshold;  // skip the O rescale while the max grew by <= this (log2 units)
  // FP8 PV variant only
  const uint32_t* v_amax_bits;  // max |V| per K/V head (float bits)
  CUtensorMap tmap_vt;          // e4m3 V^T [kv_heads * 128, kpad] bytes, box 128 x 128, 128B swizzle
  // persistent variant only
  unsigned int* work;  // the launch's counter slot: {units fetched beyond the grid size, CTAs finished}
  int units;           // heads * query blocks * sequences, in the plain grid's order
};

__device__ int g_status;  // 0 = ok, else 1 + (role * 256 + barrier id) of the first expired wait

// Opt-in coarse pipeline trace (build with -DFMHA_TRACE): %clock64 stamps at
// the hand-off points of each role for the CTAs of head 0, sequence 0, one
// row of kTraceSlots per query block.  Off by default: each stamp is a
// side-effecting instruction that blocks some scheduling across it.
constexpr int kTraceSlots = 2048;
constexpr int kTrSoftmax = 16;      // + t * 512 + j * 8 + event
constexpr int kTrMma = 1040;        // + j * 8 + event
constexpr int kTrLoad = 1600;       // + ring index
constexpr int kTrMaxBlocks = 32;
constexpr int kTrObsLoad = 272;  // + ring index (< 256): ring load landed
constexpr int kTrObsStep = 784;  // + step commit n (< 128): its MMAs completed
constexpr int kTrEpilogue = 1560;  // + 4 t + {0 O final seen, 1 O stored, 2 O staged}; 1568 after the final sync
// set-up stamps: 2 entry, 3 barriers initialised, 4 first copies issued,
// 5 TMEM allocated, 6 before the set-up sync (0 = after it)
#ifdef FMHA_TRACE
__device__ unsigned long long* g_trace;
// per-CTA table (every CTA, linear block id): %globaltimer at entry, after the
// set-up sync and at exit, and the SM id
__device__ unsigned long long* g_trace_ctas;
// The stamps go to shared memory (a global store would delay the thread's
// next mbarrier arrive, which waits for its earlier stores, and so lengthen
// the hand-offs being measured) and are copied to the row at exit.
constexpr uint32_t kTraceSmemBytes = kTraceSlots * 8;
#define FMHA_TRACE_AT(slot)                                                                  \
  do {                                                                                       \
    if (trace_row != nullptr) trace_smem[(slot)] = static_cast<unsigned long long>(clock64()); \
  } while (0)
#else
constexpr uint32_t kTraceSmemBytes = 0;
#define FMHA_TRACE_AT(slot) \
  do {                      \
  } while (0)
#endif

struct Ctx {
  uint32_t bar0;                  // shared address of barrier 0
  volatile uint32_t* abort_flag;  // shared
  __device__ __forceinline__ uint32_t bar(int id) const { return bar0 + 8u * id; }
};

// Wait for the phase of `bar` with the given parity; false on abort or expiry.
__device__ __forceinline__ bool wait_slow(const Ctx& c, uint32_t bar, uint32_t parity, int code) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity))
      return true;
    if (*c.abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
      *c.abort_flag = 1u;
      atomicCAS(&g_status, 0, 1 + code);
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bar(const Ctx& c, int id, uint32_t parity, int role) {
  const uint32_t b = c.bar(id);
  if (ptx::mbar_try_wait(b, parity)) return true;
  return wait_slow(c, b, parity, role * 256 + id);
}

// Whole-warp wait: every lane polls, and the warp agrees on the outcome so
// that the .sync.aligned tcgen05 ops and warp votes after it stay convergent.
__device__ __forceinline__ bool wait_bar_warp(const Ctx& c, int id, uint32_t parity, int role) {
  return __all_sync(0xffffffffu, wait_bar(c, id, parity, role));
}

// Drain wait used on the way out: ignores the abort flag, still bounded.
__device__ __forceinline__ void wait_drain(const Ctx& c, int id, uint32_t parity) {
  const uint32_t b = c.bar(id);
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(b, parity)) {
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(&g_status, 0, 1 + kRoleDrain * 256 + id);
      return;
    }
  }
}

// Key blocks a 128-row query tile starting at sequence row r0 must visit; 0 if
// the tile is past the sequence end or every row is fully masked.  Causal
// rows see keys j <= i + (lk - lq).
__device__ __forceinline__ int tile_blocks(int r0, int lq, int lk, int causal) {
  if (r0 >= lq) return 0;
  if (!causal) return (lk + kBlockN - 1) / kBlockN;
  const int last = min(r0 + kBlockM - 1, lq - 1);
  const int lim = min(last + lk - lq, lk - 1);
  return lim >= 0 ? lim / kBlockN + 1 : 0;
}

// Heads per rasterisation group of the head-grouped grid order.
constexpr int kHeadGroup = 4;

// Work unit of a CTA in the head-grouped grid order, (heads x query blocks,
// sequences): blockIdx.x runs over the query blocks of a group of kHeadGroup
// heads in launch order, the group's heads fastest, so that the CTAs in
// flight share the K/V of a few heads in L2 (used when one sequence's K/V
// exceeds it).  Returns the head and sets the query block's launch-order index.
// The CTA index is read through an opaque move so that a second call
// recomputes the head instead of keeping it in a register across the kernel.
__device__ __forceinline__ int decode_grouped(int heads, int& launch_pair) {
  uint32_t x, nx;
  asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(x));
  asm volatile("mov.u32 %0, %%nctaid.x;" : "=r"(nx));
  const int pairs = static_cast<int>(nx) / heads;
  const int u = static_cast<int>(x);
  const int g = u / (kHeadGroup * pairs);
  const int gh = min(kHeadGroup, heads - g * kHeadGroup);  // heads in this (possibly last, partial) group
  const int rem = u - g * kHeadGroup * pairs;
  launch_pair = rem / gh;
  return g * kHeadGroup + (rem - launch_pair * gh);
}

__device__ __forceinline__ uint32_t col_s(int t) { return 128u * t; }
__device__ __forceinline__ uint32_t col_o(int t) { return 256u + 128u * t; }

// ---------------------------------------------------------------------------
// MMA issue helpers (one thread)
// S_t = Q_t K^T: M=128 queries, N=128 keys, K=128 head dims in 8 steps of 16.
// Q and K tiles are K-major with 128-byte swizzle: two 16 KiB halves (head dims
// 0..63 and 64..127), rows 128 bytes apart, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) { return ptx::smem_desc_sw128(saddr, 16, 1024); }
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr) {
  return ptx::smem_desc_sw128(saddr, kHalfBytes, 1024);
}
// A descriptor's start address is its low 14 bits in 16-byte units; every
// offset below stays inside the 256 KiB window, so offsets add without carry.

// Each MMA is one instruction with a base descriptor plus an immediate offset:
// a single issuing thread then keeps the tensor core fed (M128 N128 K16 every
// 64 cycles, measured).
template <int HD>
__device__ __forceinline__ void issue_qk(uint32_t tmem_d, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBlockM, kBlockN, false, false);
  if constexpr (HD > 128) {
    // 16 K-steps: keep the base + offset sums at issue time rather than
    // hoisted out of the caller's loop (they would not fit the issuer's
    // register budget)
    asm volatile("" : "+l"(q_desc), "+l"(k_desc));
  }
  ptx::mma_ss_imm<false>(tmem_d, q_desc, k_desc, idesc);
#pragma unroll
  for (int k = 1; k < HD / 16; ++k) {
    const uint64_t off = ((k >> 2) * kHalfBytes + (k & 3) * 32u) >> 4;
    ptx::mma_ss_imm<true>(tmem_d, q_desc + off, k_desc + off, idesc);
  }
}

// O_t (+)= P_t V: M=128 queries, N=128 head dims, K=128 keys in 8 steps of 16.
// P comes from TMEM (8 columns of bf16 pairs per step); V is MN-major in the
// same swizzled layout as K: head dims contiguous within a 128-byte row, the
// second 64 head dims 16 KiB further (leading offset), 8-key groups 1024
// bytes apart (stride offset), 16 keys = 2048 bytes per step.
template <int HD>
__device__ __forceinline__ void issue_pv(uint32_t tmem_d, uint32_t tmem_p, uint64_t v_desc, bool accumulate) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBlockM, HD, false, true);
  if constexpr (HD > 128) asm volatile("" : "+l"(v_desc), "+r"(tmem_p));  // as in issue_qk
  if (accumulate)
    ptx::mma_ts_imm<true>(tmem_d, tmem_p, v_desc, idesc);
  else
    ptx::mma_ts_imm<false>(tmem_d, tmem_p, v_desc, idesc);
#pragma unroll
  for (int k = 1; k < kBlockN / 16; ++k)
    ptx::mma_ts_imm<true>(tmem_d, tmem_p + 8u * k, v_desc + ((2048u * k) >> 4), idesc);
}

// Row max of 128 scores: three-input max, four independent chains.  (The
// max is bound by min/max throughput, ~250 cycles a row: more chains or a
// two-input tree measured no faster.)
__device__ __forceinline__ float row_max128(const float (&s)[128]) {
  float mx[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float a = ptx::fmax3(s[32 * q + 0], s[32 * q + 1], s[32 * q + 2]);
#pragma unroll
    for (int k = 3; k < 31; k += 2) a = ptx::fmax3(a, s[32 * q + k], s[32 * q + k + 1]);
    mx[q] = fmaxf(a, s[32 * q + 31]);
  }
  return ptx::fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
}

// Row min, the same way: with a negative scale the largest scaled score
// s * scale belongs to the smallest raw score s.
__device__ __forceinline__ float row_min128(const float (&s)[128]) {
  float mn[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float a = ptx::fmin3(s[32 * q + 0], s[32 * q + 1], s[32 * q + 2]);
#pragma unroll
    for (int k = 3; k < 31; k += 2) a = ptx::fmin3(a, s[32 * q + k], s[32 * q + k + 1]);
    mn[q] = fminf(a, s[32 * q + 31]);
  }
  return ptx::fmin3(fminf(mn[0], mn[1]), mn[2], mn[3]);
}

// Ring load idx -> (K or V, key block).  Default order: K_0, V_0, K_1, V_1,
// ...  Double-buffered S (one query tile per CTA), the order the MMA groups
// read them in: K_0, K_1, V_0, K_2, V_1, K_3, ..., V_(n-2), V_(n-1) (group g
// issues PV(g - 2) then QK^T(g)).
template <bool kDoubleS>
__device__ __forceinline__ void ring_block(int idx, int n_kv, bool& is_v, int& blk) {
  if constexpr (!kDoubleS) {
    is_v = idx & 1;
    blk = idx >> 1;
  } else {
    if (idx == 0) {
      is_v = false;
      blk = 0;
    } else if (n_kv == 1) {
      is_v = true;
      blk = 0;
    } else if (idx == 1) {
      is_v = false;
      blk = 1;
    } else if (idx == 2 * n_kv - 1) {
      is_v = true;
      blk = n_kv - 1;
    } else {
      const int r = idx - 2;
      is_v = !(r & 1);
      blk = (r >> 1) + (r & 1) * 2;
    }
  }
}

// The barrier and phase parity of the commit after which ring load idx's
// block has been read for the last time (its slot is free).  Default: K_s by
// QK^T(s) (step commit s), V_s by PV(s) (step commit s + 1), step commit n on
// StepDone[n % 2].  Double-buffered S: K_g by the commit after QK^T(g)
// (StepDone[g % 2]), V_m by the commit after PV(m) (VFree[m % 2]).
template <bool kDoubleS>
__device__ __forceinline__ void ring_release(int idx, int n_kv, int& bar, uint32_t& parity) {
  if constexpr (!kDoubleS) {
    const int n = (idx >> 1) + (idx & 1);
    bar = kBarStepDone + (n & 1);
    parity = static_cast<uint32_t>(n >> 1) & 1u;
  } else {
    bool is_v;
    int blk;
    ring_block<true>(idx, n_kv, is_v, blk);
    bar = (is_v ? kBarVFree : kBarStepDone) + (blk & 1);
    parity = static_cast<uint32_t>(blk >> 1) & 1u;
  }
}

// The lazy-rescale reference for a block: its row max (min for a negative
// scale) replaces the reference in use m_used only when the scaled extreme
// grew by more than `threshold` (log2 units); NaN while both are the mask
// value compares false: keep.
__device__ __forceinline__ float lazy_reference(const float (&s)[128], bool neg, float m_used, float c,
                                                float threshold) {
  const float m_blk = neg ? row_min128(s) : row_max128(s);
  return (m_blk - m_used) * c > threshold ? m_blk : m_used;
}

// One softmax exp pass over a row of 128 scores with reference score m_ref
// (the raw score whose scaled value is the row's largest): P = 2^(s c - m_ref c)
// (one packed FMA per pair, ex2), bf16 pairs stored to TMEM at t_s (64
// columns); returns the row sum of P.  Masked scores hold +-inf with the sign
// that makes s c = -inf, so they give P = 0; m_ref is infinite only while
// every score so far was masked.
__device__ __forceinline__ float exp_pass(const float (&s)[128], float c, float m_ref, uint32_t t_s) {
  const float neg_mc = isinf(m_ref) ? 0.f : -m_ref * c;
  const float2 c2 = make_float2(c, c);
  const float2 nm2 = make_float2(neg_mc, neg_mc);
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t pk[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int k = half * 64 + 2 * i;
      const float2 x = __ffma2_rn(make_float2(s[k], s[k + 1]), c2, nm2);
      const float p0 = ptx::ex2_approx(x.x);
      const float p1 = ptx::ex2_approx(x.y);
      acc[i & 3] = __fadd2_rn(acc[i & 3], make_float2(p0, p1));
      pk[i] = ptx::pack_bf16x2(p0, p1);
    }
    ptx::tmem_st32(t_s + 32u * half, pk);
  }
  const float2 a01 = __fadd2_rn(acc[0], acc[1]);
  const float2 a23 = __fadd2_rn(acc[2], acc[3]);
  const float2 a = __fadd2_rn(a01, a23);
  return a.x + a.y;
}

// The exp pass in four 32-key chunks; after chunk kPSplit - 1, `before` runs
// (the O rescale, which must precede the first PV), the stores so far are made
// visible (wait::st, fence) and `signal` is called (split hand-off).  Running
// the rescale there rather than before the pass keeps fewer scores live.
template <int kSplit, typename Before, typename Signal>
__device__ __forceinline__ float exp_pass_split(const float (&s)[128], float c, float m_ref, uint32_t t_s,
                                                Before&& before, Signal&& signal) {
  const float neg_mc = isinf(m_ref) ? 0.f : -m_ref * c;
  const float2 c2 = make_float2(c, c);
  const float2 nm2 = make_float2(neg_mc, neg_mc);
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int k = q * 32 + 2 * i;
      const float2 x = __ffma2_rn(make_float2(s[k], s[k + 1]), c2, nm2);
      const float p0 = ptx::ex2_approx(x.x);
      const float p1 = ptx::ex2_approx(x.y);
      acc[i & 3] = __fadd2_rn(acc[i & 3], make_float2(p0, p1));
      pk[i] = ptx::pack_bf16x2(p0, p1);
    }
    ptx::tmem_st16(t_s + 16u * q, pk);
    if (q == kSplit - 1 && q < 3) {
      before();
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      signal();
    }
  }
  const float2 a01 = __fadd2_rn(acc[0], acc[1]);
  const float2 a23 = __fadd2_rn(acc[2], acc[3]);
  const float2 a = __fadd2_rn(a01, a23);
  return a.x + a.y;
}

// O (+)= P V over the PV K-steps [k0, k1) (16 keys each); the first K-step of a
// key block accumulates unless `accumulate` is false.
template <int HD>
__device__ __forceinline__ void issue_pv_steps(uint32_t tmem_d, uint32_t tmem_p, uint64_t v_desc, bool accumulate,
                                               int k0, int k1) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBlockM, HD, false, true);
#pragma unroll
  for (int k = 0; k < kBlockN / 16; ++k) {
    if (k < k0 || k >= k1) continue;
    if (k == 0 && !accumulate)
      ptx::mma_ts_imm<false>(tmem_d, tmem_p, v_desc, idesc);
    else
      ptx::mma_ts_imm<true>(tmem_d, tmem_p + 8u * k, v_desc + ((2048u * k) >> 4), idesc);
  }
}

// e4m3 pair (round to nearest, saturating to +-448): lo in bits 0..7.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// The exp pass of the FP8 variant: P = 2^(s c - m_ref c) as above, stored as
// e4m3, four keys per 32-bit TMEM column (key 4 i + b in byte b of column i):
// 32 columns at t_s.  P <= 2^8 (the lazy-rescale threshold) fits e4m3's 448.
// Returns the row sum of the unrounded P.
__device__ __forceinline__ float exp_pass_fp8(const float (&s)[128], float c, float m_ref, uint32_t t_s) {
  const float neg_mc = isinf(m_ref) ? 0.f : -m_ref * c;
  const float2 c2 = make_float2(c, c);
  const float2 nm2 = make_float2(neg_mc, neg_mc);
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int k = half * 64 + 4 * i;
      const float2 x0 = __ffma2_rn(make_float2(s[k], s[k + 1]), c2, nm2);
      const float2 x1 = __ffma2_rn(make_float2(s[k + 2], s[k + 3]), c2, nm2);
      const float p0 = ptx::ex2_approx(x0.x), p1 = ptx::ex2_approx(x0.y);
      const float p2 = ptx::ex2_approx(x1.x), p3 = ptx::ex2_approx(x1.y);
      acc[(2 * i) & 3] = __fadd2_rn(acc[(2 * i) & 3], make_float2(p0, p1));
      acc[(2 * i + 1) & 3] = __fadd2_rn(acc[(2 * i + 1) & 3], make_float2(p2, p3));
      pk[i] = pack_e4m3x2(p0, p1) | (pack_e4m3x2(p2, p3) << 16);
    }
    ptx::tmem_st16(t_s + 16u * half, pk);
  }
  const float2 a01 = __fadd2_rn(acc[0], acc[1]);
  const float2 a23 = __fadd2_rn(acc[2], acc[3]);
  const float2 a = __fadd2_rn(a01, a23);
  return a.x + a.y;
}

// The FP8 exp pass in four 32-key chunks (8 TMEM columns each), with the
// split hand-off of exp_pass_split after chunk kSplit - 1.
template <int kSplit, typename Before, typename Signal>
__device__ __forceinline__ float exp_pass_fp8_split(const float (&s)[128], float c, float m_ref, uint32_t t_s,
                                                    Before&& before, Signal&& signal) {
  const float neg_mc = isinf(m_ref) ? 0.f : -m_ref * c;
  const float2 c2 = make_float2(c, c);
  const float2 nm2 = make_float2(neg_mc, neg_mc);
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k = q * 32 + 4 * i;
      const float2 x0 = __ffma2_rn(make_float2(s[k], s[k + 1]), c2, nm2);
      const float2 x1 = __ffma2_rn(make_float2(s[k + 2], s[k + 3]), c2, nm2);
      const float p0 = ptx::ex2_approx(x0.x), p1 = ptx::ex2_approx(x0.y);
      const float p2 = ptx::ex2_approx(x1.x), p3 = ptx::ex2_approx(x1.y);
      acc[(2 * i) & 3] = __fadd2_rn(acc[(2 * i) & 3], make_float2(p0, p1));
      acc[(2 * i + 1) & 3] = __fadd2_rn(acc[(2 * i + 1) & 3], make_float2(p2, p3));
      pk[i] = pack_e4m3x2(p0, p1) | (pack_e4m3x2(p2, p3) << 16);
    }
    ptx::tmem_st8(t_s + 8u * q, pk);
    if (q == kSplit - 1 && q < 3) {
      before();
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      signal();
    }
  }
  const float2 a01 = __fadd2_rn(acc[0], acc[1]);
  const float2 a23 = __fadd2_rn(acc[2], acc[3]);
  const float2 a = __fadd2_rn(a01, a23);
  return a.x + a.y;
}

// O (+)= P V with e4m3 operands: M=128 queries, N=128 head dims, K=128 keys in
// 4 steps of 32.  P from TMEM (8 columns of four keys per step); V^T K-major
// in shared memory (128 head-dim rows of 128 key bytes, 128-byte swizzle):
// a step of 32 keys is 32 bytes along the row.
__device__ __forceinline__ void issue_pv_fp8(uint32_t tmem_d, uint32_t tmem_p, uint64_t vt_desc, bool accumulate) {
  constexpr uint32_t idesc = ptx::idesc_e4m3_f32(kBlockM, 128);
  if (accumulate)
    ptx::mma_ts_f8_imm<true>(tmem_d, tmem_p, vt_desc, idesc);
  else
    ptx::mma_ts_f8_imm<false>(tmem_d, tmem_p, vt_desc, idesc);
#pragma unroll
  for (int k = 1; k < kBlockN / 32; ++k) ptx::mma_ts_f8_imm<true>(tmem_d, tmem_p + 8u * k, vt_desc + ((32u * k) >> 4), idesc);
}

// The FP8 PV over the K-steps [k0, k1) (32 keys each).
__device__ __forceinline__ void issue_pv_fp8_steps(uint32_t tmem_d, uint32_t tmem_p, uint64_t vt_desc, bool accumulate,
                                                   int k0, int k1) {
  constexpr uint32_t idesc = ptx::idesc_e4m3_f32(kBlockM, 128);
#pragma unroll
  for (int k = 0; k < kBlockN / 32; ++k) {
    if (k < k0 || k >= k1) continue;
    if (k == 0 && !accumulate)
      ptx::mma_ts_f8_imm<false>(tmem_d, tmem_p, vt_desc, idesc);
    else
      ptx::mma_ts_f8_imm<true>(tmem_d, tmem_p + 8u * k, vt_desc + ((32u * k) >> 4), idesc);
  }
}

// ---------------------------------------------------------------------------
// kGrouped: the head-grouped grid order (see decode_grouped); else the grid
// is (heads, query blocks, sequences).
// kFp8: O += P V with P and V in e4m3 (kind::f8f6f4); V comes from the
// pre-pass's transposed e4m3 copy (tmap_vt), its per-head scale folds into the
// epilogue's 1 / l.
template <int HD, bool kGrouped, bool kFp8 = false>
__global__ void __launch_bounds__(kThreads, 1) fmha_fwd_kernel(const __grid_constant__ FwdParams p) {
  static_assert(!kFp8 || HD == 128, "FP8 PV: head_dim 128");
  // the P hand-off split of this variant, and the PV K-steps issued after its first signal
  constexpr int kSplit = kFp8 ? kPSplitFp8 : kPSplit;
  constexpr int kStepsBeforeFull = kFp8 ? kSplit : kPvStepsBeforeFull;
  static_assert(kStepsBeforeFull * (kFp8 ? 32 : 16) <= kSplit * 32, "P split: consumer ahead of producer");
  using D = Dims<HD>;
  constexpr int kHeadDim = HD;
  constexpr int kStages = D::kStages;
  constexpr uint32_t kTileBytes = D::kTileBytes;
  constexpr uint32_t kOffQ = D::kOffQ, kOffKV = D::kOffKV, kOffBar = D::kOffBar, kOffMisc = D::kOffMisc;
  constexpr uint64_t kSlotDescStep = kTileBytes >> 4;
  // one query tile per CTA (head_dim 256): two S buffers, so that the next
  // block's QK^T runs during this block's softmax
  constexpr bool kDoubleS = D::kTiles == 1;
  static_assert(!kDoubleS || (kSplit == 4 && D::kStages == 2), "double-buffered S: one P hand-off, two ring slots");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // first: start the descriptor fetches, which need no parameter loads, so
  // they overlap the (cold) loads of the scalar parameters below
  if (warp == kWarpProducer && lane == 0) {
    ptx::prefetch_tensormap(&p.tmap_q);
    ptx::prefetch_tensormap(&p.tmap_k);
    ptx::prefetch_tensormap(&p.tmap_v);
    if constexpr (kFp8) ptx::prefetch_tensormap(&p.tmap_vt);
  }
#ifdef FMHA_TRACE
  const unsigned long long t_entry = static_cast<unsigned long long>(clock64());
  const size_t cta_lin = blockIdx.x + static_cast<size_t>(gridDim.x) * (blockIdx.y + static_cast<size_t>(gridDim.y) * blockIdx.z);
  if (threadIdx.x == 0 && g_trace_ctas != nullptr) {
    g_trace_ctas[cta_lin * 4 + 0] = ptx::globaltimer_ns();
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    g_trace_ctas[cta_lin * 4 + 3] = smid;
  }
#endif

  // ---- work unit: head, 256-row query block (causal launches start with the
  // last, longest one), sequence
  int h, launch_pair, pairs, b;
  if constexpr (kGrouped) {
    h = decode_grouped(p.heads, launch_pair);
    pairs = static_cast<int>(gridDim.x) / p.heads;
    b = static_cast<int>(blockIdx.y);
  } else {
    h = static_cast<int>(blockIdx.x);
    launch_pair = static_cast<int>(blockIdx.y);
    pairs = static_cast<int>(gridDim.y);
    b = static_cast<int>(blockIdx.z);
  }
  const int pair = p.causal ? pairs - 1 - launch_pair : launch_pair;
#ifdef FMHA_TRACE
  unsigned long long* trace_row =
      (g_trace != nullptr && h == 0 && b == 0) ? g_trace + static_cast<size_t>(launch_pair) * kTraceSlots : nullptr;
  // stamps in shared memory past the misc words (the trace build allocates kTraceSmemBytes more)
  volatile unsigned long long* trace_smem = reinterpret_cast<volatile unsigned long long*>(smem + kOffMisc + 256);
  if (trace_row != nullptr)
    for (int i = threadIdx.x; i < kTraceSlots; i += blockDim.x) trace_smem[i] = 0ull;
  if (threadIdx.x == 0 && trace_row != nullptr) trace_smem[2] = t_entry;
#endif
  int q0, lq, k0, lk;
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
  if (lk < 0) lk = 0;
  const int m0 = pair * (D::kTiles * kBlockM);
  if (m0 >= lq) return;  // uniform across the CTA, before any shared state

  // key blocks per tile; causal rows see keys j <= i + (lk - lq)
  const int off = lk - lq;
  const int n_blk0 = tile_blocks(m0, lq, lk, p.causal);
  const int n_blk1 = D::kTiles > 1 ? tile_blocks(m0 + kBlockM, lq, lk, p.causal) : 0;
  const bool active1 = D::kTiles > 1 && m0 + kBlockM < lq;  // tile 0 is active whenever the unit exists
  const int n_kv = max(n_blk0, n_blk1);
  // The last tile of every KV step: tile 1 whenever it has blocks (it never has
  // fewer than tile 0: causal rows further down see more keys), else tile 0.
  const int t_last = n_blk1 > 0 ? 1 : 0;
  auto n_blk = [&](int t) { return t ? n_blk1 : n_blk0; };
  auto active = [&](int t) { return t ? active1 : true; };

  Ctx ctx;
  ctx.bar0 = base + kOffBar;
  ctx.abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);

  // TMA producer steps (one thread): the Q tiles, and ring load idx = K (even) or
  // V (odd) of key block idx / 2 into slot idx % kStages.
  const int xh = h * kHeadDim;                    // this head's columns in q / out
  const int xkv = (h / p.kv_group) * kHeadDim;    // its K/V head's columns in k / v
  auto load_q = [&](int t, uint64_t pol) {
    if (n_blk(t) > 0) {
      const uint32_t bar = ctx.bar(kBarQFull + t);
      ptx::mbar_arrive_expect_tx(bar, kTileBytes);
      const uint32_t dst = base + kOffQ + t * kTileBytes;
      const int y = q0 + m0 + kBlockM * t;
#pragma unroll
      for (int hf = 0; hf < D::kHalves; ++hf) ptx::tma_load_2d(dst + hf * kHalfBytes, &p.tmap_q, bar, xh + 64 * hf, y, pol);
    }
  };
  auto load_kv = [&](int idx, uint64_t pol) {
    const int slot = idx % kStages;
    const uint32_t bar = ctx.bar(kBarKVFull + slot);
    const uint32_t dst = base + kOffKV + slot * kTileBytes;
    if constexpr (kFp8) {
      if (idx & 1) {  // e4m3 V^T block: 128 head-dim rows of 128 key bytes at the sequence's padded start
        ptx::mbar_arrive_expect_tx(bar, kTileBytes / 2);
        const int x = static_cast<int>(16 * ((k0 + 15) / 16 + b)) + kBlockN * (idx >> 1);
        ptx::tma_load_2d(dst, &p.tmap_vt, bar, x, (h / p.kv_group) * kHeadDim, pol);
        return;
      }
    }
    ptx::mbar_arrive_expect_tx(bar, kTileBytes);
    bool is_v;
    int blk;
    ring_block<kDoubleS>(idx, n_kv, is_v, blk);
    const CUtensorMap* m = is_v ? &p.tmap_v : &p.tmap_k;
    const int y = k0 + kBlockN * blk;
#pragma unroll
    for (int hf = 0; hf < D::kHalves; ++hf) ptx::tma_load_2d(dst + hf * kHalfBytes, m, bar, xkv + 64 * hf, y, pol);
  };
  // ring loads issued before the CTA-wide set-up sync (the ring starts empty)
  const int early_loads = min(kStages, 2 * n_kv);

  if (warp == kWarpProducer && lane == 0) {
    for (int t = 0; t < kTiles; ++t) {
      ptx::mbar_init(ctx.bar(kBarQFull + t), 1);
      ptx::mbar_init(ctx.bar(kBarStepDone + t), 1);
      ptx::mbar_init(ctx.bar(kBarPVReady + t), 4);  // the tile's 4 softmax warps
      ptx::mbar_init(ctx.bar(kBarOFinal + t), 1);
    }
    for (int s = 0; s < 4; ++s) ptx::mbar_init(ctx.bar(kBarKVFull + s), 1);
    for (int t = 0; t < kTiles; ++t) ptx::mbar_init(ctx.bar(kBarPVPart + t), 4);
    ptx::mbar_init(ctx.bar(kBarSFull0), 1);
    ptx::mbar_init(ctx.bar(kBarMmaDone), 1);
    *ctx.abort_flag = 0u;
    ptx::fence_mbar_init();
    FMHA_TRACE_AT(3);
    // start the first copies now: they overlap the TMEM allocation and the sync
    // what the first S needs first (Q_0, K_0), then the rest: at launch every
    // CTA loads at once and DRAM bandwidth orders the arrivals
    const uint64_t pol_q = ptx::policy_evict_first();
    const uint64_t pol_kv = ptx::policy_evict_last();
    load_q(0, pol_q);
    if (early_loads > 0) load_kv(0, pol_kv);
    load_q(1, pol_q);
    for (int idx = 1; idx < early_loads; ++idx) load_kv(idx, pol_kv);
    FMHA_TRACE_AT(4);
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
    if (lane == 0) FMHA_TRACE_AT(5);
  }
#ifdef FMHA_TRACE
  if (threadIdx.x == 0) FMHA_TRACE_AT(6);
#endif
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
#ifdef FMHA_TRACE
  if (threadIdx.x == 0) FMHA_TRACE_AT(0);
  if (threadIdx.x == 0 && g_trace_ctas != nullptr) g_trace_ctas[cta_lin * 4 + 1] = ptx::globaltimer_ns();
#endif

  const int wg = warp >> 2;
  if (wg == kWgSoftmax0 || (D::kTiles > 1 && wg == kWgSoftmax0 + 1)) {
    // =============================== softmax (tile t = wg)
    ptx::setmaxnreg_inc<(D::kTiles > 1 ? kRegsSoftmax : kRegsSoftmax1)>();
    const int t = wg - kWgSoftmax0;
    const int r = (warp & 3) * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t t_s = tmem + ((static_cast<uint32_t>(warp & 3) * 32u) << 16) + col_s(t);
    const int row = m0 + kBlockM * t + r;  // sequence-local query index
    const int nb = n_blk(t);
    const float c = p.scale_log2;  // nonzero: the launcher passes 2^-126 for a zero scale
    const float sum_limit = exp2f(p.rescale_threshold);  // row sums below it: every P below it
    // Softmax order is the order of s * c: for a negative scale the reference
    // score is the row minimum and masked scores hold +inf (s * c = -inf).
    const bool neg = c < 0.f;
    const float s_mask = neg ? INFINITY : -INFINITY;
    const int key_end = p.causal ? min(row + off + 1, lk) : lk;  // this row's visible keys [0, key_end)
    const int tile_key_end = p.causal ? min(m0 + kBlockM * t + off + 1, lk) : lk;  // the tile's first row
    float m_used = s_mask;
    float l = 0.f;
    for (int j = 0; j < nb; ++j) {
      // S_t(j): step commit j for the step's last tile, else tile 0's own commit
      const bool s_ok = t == t_last ? wait_bar_warp(ctx, kBarStepDone + (j & 1), (j >> 1) & 1, kRoleSoftmax)
                                    : wait_bar_warp(ctx, kBarSFull0, j & 1, kRoleSoftmax);
      if (!s_ok) break;
      const bool tr = (r == 0 && j < kTrMaxBlocks);
      if (tr) FMHA_TRACE_AT(kTrSoftmax + t * 512 + j * 8 + 0);
      ptx::tc_fence_after();
      // this block's S buffer (two alternate with one query tile per CTA)
      const uint32_t t_sj = kDoubleS ? t_s + col_s(j & 1) : t_s;
      float s[128];
      ptx::tmem_ld128_wait(t_sj, s);
      if (tr) FMHA_TRACE_AT(kTrSoftmax + t * 512 + j * 8 + 1);
      const int c0 = j * kBlockN;
      if (tile_key_end - c0 < kBlockN) {  // block crosses the diagonal or the key tail
        const int lim = key_end - c0;
#pragma unroll
        for (int k = 0; k < 128; ++k)
          if (k >= lim) s[k] = s_mask;
      }
      // Reference score of this block (lazy rescale): the block max of s * c
      // replaces the reference in use only when it grew by more than the
      // threshold.  With one P hand-off in bf16 and two query tiles, after the
      // row's first visible block the exponents are taken against the
      // reference in use first, and the block max is found only when some
      // row's sum exceeds 2^threshold: below that every P is below it too, so
      // the rule keeps the reference and those P stand; above it the rule
      // decides and, if it moves the reference, the pass is redone.
      constexpr bool kStaleFirst = !kFp8 && kSplit == 4 && D::kTiles > 1;
      bool stale = kStaleFirst && j > 0 && !__any_sync(0xffffffffu, isinf(m_used));
      float m_ref = stale ? m_used : lazy_reference(s, neg, m_used, c, p.rescale_threshold);
      if (tr) FMHA_TRACE_AT(kTrSoftmax + t * 512 + j * 8 + 2);
      float alpha = 1.f;
      // Rescale this warp's O rows.  PV_t(j-1) has completed (two tiles: S_t(j)
      // is committed after it; one tile with two S buffers: waited for below)
      // and PV_t(j) waits for this warp's P hand-off (with a split hand-off,
      // the first one: hence the rescale before that signal).
      auto rescale_o = [&]() {
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if constexpr (kDoubleS) {
            // PV(j - 1) may still run (S(j) came from group j, before it)
            if (!wait_bar_warp(ctx, kBarVFree + ((j - 1) & 1), ((j - 1) >> 1) & 1, kRoleSoftmax)) return;
            ptx::tc_fence_after();
          }
          const uint32_t t_o = tmem + ((static_cast<uint32_t>(warp & 3) * 32u) << 16) + col_o(t);
#pragma unroll
          for (int cc = 0; cc < HD / 32; ++cc) {
            float o[32];
            ptx::tmem_ld32_wait(t_o + 32u * cc, o);
            uint32_t u[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(o[i] * alpha);
            ptx::tmem_st32(t_o + 32u * cc, u);
          }
        }
      };
      float row_sum;
      auto signal_part = [&]() {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ctx.bar(kBarPVPart + t));
      };
      if constexpr (kFp8 && kSplit < 4) {
        alpha = (m_ref == m_used) ? 1.f : ptx::ex2_approx((m_used - m_ref) * c);
        row_sum = exp_pass_fp8_split<kSplit>(s, c, m_ref, t_sj, rescale_o, signal_part);
      } else if constexpr (kFp8) {
        alpha = (m_ref == m_used) ? 1.f : ptx::ex2_approx((m_used - m_ref) * c);
        row_sum = exp_pass_fp8(s, c, m_ref, t_sj);
        rescale_o();
      } else if constexpr (kSplit < 4) {
        alpha = (m_ref == m_used) ? 1.f : ptx::ex2_approx((m_used - m_ref) * c);
        row_sum = exp_pass_split<kSplit>(s, c, m_ref, t_sj, rescale_o, signal_part);
      } else {
        // one exp pass; true when it must be redone against a moved reference
        auto pass_redo = [&]() -> bool {
          row_sum = exp_pass(s, c, m_ref, t_sj);
          if (!stale || !__any_sync(0xffffffffu, row_sum > sum_limit)) return false;
          stale = false;
          const float m_new = lazy_reference(s, neg, m_used, c, p.rescale_threshold);
          if (!__any_sync(0xffffffffu, m_new != m_used)) return false;
          m_ref = m_new;
          ptx::tmem_wait_st();  // the first pass's stores land before they are overwritten
          return true;
        };
        if constexpr (HD == 64) {  // both passes inlined (measured faster there)
#pragma unroll
          for (int pass = 0; pass < 2; ++pass)
            if (!pass_redo()) break;
        } else {  // one copy of the pass
#pragma unroll 1
          for (int pass = 0; pass < 2; ++pass)
            if (!pass_redo()) break;
        }
        // an infinite m_used (nothing visible yet) gives alpha 0 (its O rows and l are still 0)
        alpha = (m_ref == m_used) ? 1.f : ptx::ex2_approx((m_used - m_ref) * c);
        rescale_o();
      }
      if (tr) FMHA_TRACE_AT(kTrSoftmax + t * 512 + j * 8 + 3);
      l = l * alpha + row_sum;
      m_used = m_ref;
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      // (double-buffered S: the softmax can be two blocks ahead of the PVs,
      // so P hand-offs alternate between the two barriers)
      if (lane == 0) ptx::mbar_arrive(ctx.bar(kBarPVReady + (kDoubleS ? (j & 1) : t)));
      if (tr) FMHA_TRACE_AT(kTrSoftmax + t * 512 + j * 8 + 4);
      // the other three warps of the warpgroup stamp their own hand-off (skew)
      if (lane == 0 && (warp & 3) != 0 && j < kTrMaxBlocks) FMHA_TRACE_AT(kTrSoftmax + t * 512 + j * 8 + 4 + (warp & 3));
    }
    // ---- epilogue of this tile: LSE and O / l -> bf16 (rows of the sequence only),
    // as soon as this tile's last PV completed
    const bool valid = active(t) && row < lq;
    int lp_unused;
    // recomputed rather than held through the loop
    const int h = kGrouped ? decode_grouped(p.heads, lp_unused) : static_cast<int>(blockIdx.x);
    if (p.lse != nullptr && valid) {
      const float lse = (l > 0.f) ? (m_used * c + log2f(l)) * 0.69314718055994531f : -INFINITY;
      p.lse[static_cast<size_t>(h) * p.total_q + q0 + row] = lse;
    }
    if (active(t) && (nb == 0 || wait_bar_warp(ctx, kBarOFinal + t, 0, kRoleSoftmax))) {
      if (nb > 0) ptx::tc_fence_after();
      if (r == 0) FMHA_TRACE_AT(kTrEpilogue + 4 * t + 0);
      float v_scale = 1.f;  // FP8 variant: V was stored as V / s, s = max|V| / 448
      if constexpr (kFp8) {
        const float amax = __uint_as_float(p.v_amax_bits[h / p.kv_group]);
        v_scale = amax > 0.f ? amax / 448.f : 1.f;
      }
      const float inv = l > 0.f ? v_scale / l : 0.f;
      const uint32_t t_o = tmem + ((static_cast<uint32_t>(warp & 3) * 32u) << 16) + col_o(t);
      // Whole warp inside the sequence: stage its 32 rows of O in this tile's Q
      // buffer (free once the tile's last MMA completed) in the 128-byte
      // swizzled layout (conflict-free both ways), then read back so that each
      // 16-byte store instruction of the warp covers two complete 256-byte
      // rows.  A warp with rows past the sequence end stores its valid rows
      // directly, one row per thread.
      const bool staged_out = nb > 0 && __all_sync(0xffffffffu, valid);
      if (staged_out) {
        const uint32_t tile_smem = base + kOffQ + static_cast<uint32_t>(t) * kTileBytes;
        const uint32_t row_addr = tile_smem + static_cast<uint32_t>(r) * 128u;
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
          float o[32];
          ptx::tmem_ld32_wait(t_o + 32u * cc, o);
          const uint32_t half_addr = row_addr + static_cast<uint32_t>(cc >> 1) * kHalfBytes;
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const uint32_t chunk = static_cast<uint32_t>((cc & 1) * 4 + v4);  // 16-byte chunk in the 128-byte row
            ptx::st_shared_v4(half_addr + ((chunk ^ static_cast<uint32_t>(r & 7)) << 4),
                              ptx::pack_bf16x2(o[8 * v4 + 0] * inv, o[8 * v4 + 1] * inv),
                              ptx::pack_bf16x2(o[8 * v4 + 2] * inv, o[8 * v4 + 3] * inv),
                              ptx::pack_bf16x2(o[8 * v4 + 4] * inv, o[8 * v4 + 5] * inv),
                              ptx::pack_bf16x2(o[8 * v4 + 6] * inv, o[8 * v4 + 7] * inv));
          }
        }
        if (r == 0) FMHA_TRACE_AT(kTrEpilogue + 4 * t + 2);
        __syncwarp();
        // HD / 8 lanes per row, each one 16-byte chunk (8 head dims): every
        // store instruction of the warp covers 32 / (HD / 8) complete rows
        constexpr int kLanesPerRow = HD / 8, kRowsPerInst = 32 / kLanesPerRow;
        const int kc = lane % kLanesPerRow;
        const uint32_t hf = static_cast<uint32_t>(kc >> 3), c = static_cast<uint32_t>(kc & 7);
#pragma unroll
        for (int i = 0; i < 32 / kRowsPerInst; ++i) {
          const int rt = 32 * (warp & 3) + kRowsPerInst * i + lane / kLanesPerRow;  // row within the tile
          const uint4 v = ptx::ld_shared_v4(tile_smem + hf * kHalfBytes + static_cast<uint32_t>(rt) * 128u +
                                            ((c ^ static_cast<uint32_t>(rt & 7)) << 4));
          __nv_bfloat16* dst =
              p.out + (static_cast<size_t>(q0 + m0 + kBlockM * t + rt) * p.heads + h) * kHeadDim + 64 * hf + 8 * c;
          *reinterpret_cast<uint4*>(dst) = v;
        }
      } else {
        __nv_bfloat16* dst =
            p.out + (static_cast<size_t>(q0 + row) * p.heads + h) * static_cast<size_t>(kHeadDim);
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
          float o[32];
          if (nb > 0) {
            ptx::tmem_ld32_wait(t_o + 32u * cc, o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0.f;
          }
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * cc);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = ptx::pack_bf16x2(o[8 * v4 + 0] * inv, o[8 * v4 + 1] * inv);
              w.y = ptx::pack_bf16x2(o[8 * v4 + 2] * inv, o[8 * v4 + 3] * inv);
              w.z = ptx::pack_bf16x2(o[8 * v4 + 4] * inv, o[8 * v4 + 5] * inv);
              w.w = ptx::pack_bf16x2(o[8 * v4 + 6] * inv, o[8 * v4 + 7] * inv);
              d4[v4] = w;
            }
          }
        }
      }
      if (r == 0) FMHA_TRACE_AT(kTrEpilogue + 4 * t + 1);
    }
  } else if (wg == kWgIdle || wg == kWgSoftmax0 + 1) {
    // =============================== idle (its registers go to the softmax)
    ptx::setmaxnreg_dec<(D::kTiles > 1 ? kRegsIdle : kRegsIdle1)>();
  } else {
    if constexpr (D::kTiles > 1)
      ptx::setmaxnreg_dec<kRegsControl>();
    else
      ptx::setmaxnreg_inc<kRegsControl1>();
    if (warp == kWarpProducer) {
      // =============================== TMA producer (continues after the early loads)
      if (lane == 0) {
        const uint64_t pol_kv = ptx::policy_evict_last();
        int issued = early_loads;
        for (int idx = early_loads; idx < 2 * n_kv; ++idx) {
          // the slot's previous block (load idx - 4) was last read by the MMAs
          // of step commit n: K_s by QK^T(s) (commit s), V_s by PV(s) (commit s + 1);
          // the first kStages loads find their slots empty
          const int prev = idx - kStages;
          if (prev >= 0) {
            int rel_bar;
            uint32_t rel_parity;
            ring_release<kDoubleS>(prev, n_kv, rel_bar, rel_parity);
            if (!wait_bar(ctx, rel_bar, rel_parity, kRoleLoad)) break;
          }
          if (idx < 400) FMHA_TRACE_AT(kTrLoad + idx);
          load_kv(idx, pol_kv);
          ++issued;
        }
        // every issued copy has landed before the CTA may exit
        for (int idx = max(0, issued - kStages); idx < issued; ++idx)
          wait_drain(ctx, kBarKVFull + idx % kStages, (idx / kStages) & 1);
#pragma unroll
        for (int t = 0; t < kTiles; ++t)
          if (n_blk(t) > 0) wait_drain(ctx, kBarQFull + t, 0);
      }
      __syncwarp();
    } else if (warp == kWarpMma) {
      // =============================== MMA issuer
      // Per KV step j: for each tile with block j, PV_t(j) then QK^T_t(j + 1)
      // (S_t and P_t share TMEM columns, so the next QK^T follows the PV), a
      // commit for tile 0's S unless tile 0 is the step's last tile, and one
      // step commit.
      if (lane == 0) {
        const uint64_t q_desc[kTiles] = {desc_kmajor(base + kOffQ), desc_kmajor(base + kOffQ + kTileBytes)};
        const uint64_t kv_desc = desc_kmajor(base + kOffKV);
        const uint64_t kv_desc_mn = desc_mnmajor(base + kOffKV);
        bool issued_any = false;
        bool ok = true;
        if constexpr (kDoubleS) {
          // Group g (0 .. n_kv + 1): PV(g - 2) reading P from S buffer g % 2,
          // then QK^T(g) into the same buffer; a commit after each (VFree:
          // V's slot free and O updated; StepDone: S(g) ready, K_g's slot
          // free), so that a slot is refilled as soon as its reader is done
          // and the next block's copy runs behind the other MMA.  Block j's
          // softmax overlaps QK^T(j + 1) and PV(j - 1).  P(m) arrives on
          // PVReady[m % 2] (phase m / 2): the softmax may run two blocks
          // ahead of the PVs.
          if (n_kv > 0) ok = wait_bar(ctx, kBarQFull + 0, 0, kRoleMma);
          for (int g = 0; ok && n_kv > 0 && g < n_kv + 2; ++g) {
            if (g >= 2) {
              const int m = g - 2;
              const int vidx = m < n_kv - 1 ? 2 + 2 * m : (n_kv == 1 ? 1 : 2 * n_kv - 1);
              if (!wait_bar(ctx, kBarKVFull + vidx % kStages, (vidx / kStages) & 1, kRoleMma) ||
                  !wait_bar(ctx, kBarPVReady + (m & 1), (m >> 1) & 1, kRoleMma)) {
                ok = false;
                break;
              }
              if (m < kTrMaxBlocks) FMHA_TRACE_AT(kTrMma + m * 8 + 1);
              ptx::tc_fence_after();
              issue_pv<HD>(tmem + col_o(0), tmem + col_s(m & 1), kv_desc_mn + kSlotDescStep * (vidx % kStages), m > 0);
              ptx::mma_commit(ctx.bar(kBarVFree + (m & 1)));  // V_m's slot free, O has PV(m)
              if (m == n_kv - 1) ptx::mma_commit(ctx.bar(kBarOFinal + 0));
            }
            if (g < n_kv) {
              const int kidx = g < 2 ? g : 2 * g - 1;
              if (!wait_bar(ctx, kBarKVFull + kidx % kStages, (kidx / kStages) & 1, kRoleMma)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              issue_qk<HD>(tmem + col_s(g & 1), q_desc[0], kv_desc + kSlotDescStep * (kidx % kStages));
              issued_any = true;
              ptx::mma_commit(ctx.bar(kBarStepDone + (g & 1)));  // S(g) ready, K_g's slot free
            }
          }
        } else if (n_kv > 0) {
          ok = wait_bar(ctx, kBarKVFull + 0, 0, kRoleMma);
        }
        if (!kDoubleS && ok && n_kv > 0) {
          // each tile's first QK^T as soon as its own Q tile has landed
#pragma unroll
          for (int t = 0; t < kTiles; ++t) {
            if (ok && n_blk(t) > 0) {
              ok = wait_bar(ctx, kBarQFull + t, 0, kRoleMma);
              if (!ok) break;
              ptx::tc_fence_after();
              issue_qk<HD>(tmem + col_s(t), q_desc[t], kv_desc);
              issued_any = true;
              if (t != t_last) ptx::mma_commit(ctx.bar(kBarSFull0));
            }
          }
#ifndef FMHA_TEST_DROP_STEP_COMMIT
          ptx::mma_commit(ctx.bar(kBarStepDone + 0));  // step commit 0
#else
          // test build only: step commit 0 is never made, so the waits on it
          // expire and the kernel must report a timeout and shut down cleanly
#endif
          for (int j = 0; j < n_kv && ok; ++j) {
            const int vidx = 2 * j + 1, vslot = vidx % kStages;
            if (!wait_bar(ctx, kBarKVFull + vslot, (vidx / kStages) & 1, kRoleMma)) break;
            const bool tr = j < kTrMaxBlocks;
            if (tr) FMHA_TRACE_AT(kTrMma + j * 8 + 0);
            ptx::tc_fence_after();
            const int kidx = 2 * j + 2, kslot = kidx % kStages;
            bool k_ready = false;
#pragma unroll
            for (int t = 0; t < kTiles; ++t) {
              if (!ok || j >= n_blk(t)) continue;
              if constexpr (kSplit < 4) {
                // split hand-off: the K-steps of the first P chunks after the
                // first signal, the rest after the full one
                if (!wait_bar(ctx, kBarPVPart + t, j & 1, kRoleMma)) {
                  ok = false;
                  break;
                }
                ptx::tc_fence_after();
                if constexpr (kFp8)
                  issue_pv_fp8_steps(tmem + col_o(t), tmem + col_s(t), kv_desc + kSlotDescStep * vslot, j > 0, 0,
                                     kStepsBeforeFull);
                else
                  issue_pv_steps<HD>(tmem + col_o(t), tmem + col_s(t), kv_desc_mn + kSlotDescStep * vslot, j > 0, 0,
                                     kStepsBeforeFull);
              }
              if (!wait_bar(ctx, kBarPVReady + t, j & 1, kRoleMma)) {
                ok = false;
                break;
              }
              if (tr) FMHA_TRACE_AT(kTrMma + j * 8 + 1 + 2 * t);
              ptx::tc_fence_after();
              if constexpr (kFp8 && kSplit < 4)
                issue_pv_fp8_steps(tmem + col_o(t), tmem + col_s(t), kv_desc + kSlotDescStep * vslot, j > 0,
                                   kStepsBeforeFull, kBlockN / 32);
              else if constexpr (kSplit < 4)
                issue_pv_steps<HD>(tmem + col_o(t), tmem + col_s(t), kv_desc_mn + kSlotDescStep * vslot, j > 0,
                                   kStepsBeforeFull, kBlockN / 16);
              else if constexpr (kFp8)
                issue_pv_fp8(tmem + col_o(t), tmem + col_s(t), kv_desc + kSlotDescStep * vslot, j > 0);
              else
                issue_pv<HD>(tmem + col_o(t), tmem + col_s(t), kv_desc_mn + kSlotDescStep * vslot, j > 0);
              if (j + 1 < n_blk(t)) {
                if (!k_ready) {
                  if (!wait_bar(ctx, kBarKVFull + kslot, (kidx / kStages) & 1, kRoleMma)) {
                    ok = false;
                    break;
                  }
                  ptx::tc_fence_after();
                  k_ready = true;
                }
                if (tr) FMHA_TRACE_AT(kTrMma + j * 8 + 6 + t);
                issue_qk<HD>(tmem + col_s(t), q_desc[t], kv_desc + kSlotDescStep * kslot);
                if (t != t_last) ptx::mma_commit(ctx.bar(kBarSFull0));
              } else {
                ptx::mma_commit(ctx.bar(kBarOFinal + t));
              }
              if (tr) FMHA_TRACE_AT(kTrMma + j * 8 + 2 + 2 * t);
            }
            if (!ok) break;
            const int n = j + 1;  // step commit n: frees V_j's and K_(j+1)'s slots
            ptx::mma_commit(ctx.bar(kBarStepDone + (n & 1)));
            if (tr) FMHA_TRACE_AT(kTrMma + j * 8 + 5);
          }
        }
        if (issued_any) {  // all MMAs retired before TMEM is released
          ptx::mma_commit(ctx.bar(kBarMmaDone));
          wait_drain(ctx, kBarMmaDone, 0);
        }
      }
      __syncwarp();
    }
#ifdef FMHA_TRACE
    else if (lane == 0 && trace_row != nullptr) {
      // trace build only: warp 14 stamps when each ring load lands, warp 15
      // when the MMAs of each step commit complete (short bounded polls that
      // never raise the error word; a miss ends the observation)
      auto observe = [&](int id, uint32_t parity) {
        const uint64_t g0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(ctx.bar(id), parity))
          if (ptx::globaltimer_ns() - g0 > 200000ull) return false;
        return true;
      };
      if (warp == kWarpMma + 1) {
        for (int idx = 0; idx < min(2 * n_kv, 256); ++idx) {
          if (!observe(kBarKVFull + idx % kStages, (idx / kStages) & 1)) break;
          FMHA_TRACE_AT(kTrObsLoad + idx);
        }
      } else {
        for (int n = 0; n <= min(n_kv, 127); ++n) {
          if (!observe(kBarStepDone + (n & 1), (n >> 1) & 1)) break;
          FMHA_TRACE_AT(kTrObsStep + n);
        }
      }
    }
#endif
  }

#ifdef FMHA_TRACE
  if (warp == 4 * kWgIdle && lane == 0) FMHA_TRACE_AT(1);
#endif
  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) FMHA_TRACE_AT(kTrEpilogue + 8);
  if (warp == kWarpMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
#ifdef FMHA_TRACE
    if (lane == 0 && g_trace_ctas != nullptr) g_trace_ctas[cta_lin * 4 + 2] = ptx::globaltimer_ns();
#endif
  }
#ifdef FMHA_TRACE
  __syncthreads();
  if (trace_row != nullptr)
    for (int i = threadIdx.x; i < kTraceSlots; i += blockDim.x) trace_row[i] = trace_smem[i];
#endif
}

}  // namespace fmha
