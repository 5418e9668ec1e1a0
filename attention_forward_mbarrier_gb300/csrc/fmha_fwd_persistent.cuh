// fmha_fwd_persistent.cuh -- the forward as a persistent kernel, for launches
// made of many short work units.
//
// The plain kernel (fmha_fwd_kernel.cuh) runs one CTA per work unit (head,
// 256-row query block, sequence), so every unit pays for its own set-up, its
// first loads and its epilogue: on causal batches of sequences of a few
// thousand tokens a unit walks ~10 key blocks, and those fixed costs are a
// fifth of it.  Here min(units, SMs) CTAs stay resident and run the units one
// after another, and consecutive units of a CTA overlap:
//   * the producer loads the next unit's Q tiles and first K/V blocks while
//     the current unit's last steps run (its Q tile is refilled once the
//     tile's last QK^T has completed);
//   * the MMA warp issues the next unit's first QK^T right after the current
//     unit's last PV (S and P share TMEM columns, and the tensor pipe runs
//     MMAs in issue order), and its first PV once the softmax warps have read
//     the previous O out of TMEM;
//   * the softmax warps write the previous unit's O and LSE while the next
//     unit's first scores are computed.
// Units keep the plain grid's launch order (heads fastest, then query blocks
// longest-first for causal launches, then sequences): CTA c starts with unit
// c, and every later unit comes from a counter in global memory, so the
// longest units start first and the CTAs finish close together, as the
// hardware's own block scheduler would have it.
//
// The counter: one of kWorkSlots slots per launch (the host hands out slots
// round-robin, so launches in flight on different streams use different
// ones), {units taken beyond the first grid-size, CTAs finished}; the last CTA
// to finish resets both words to zero for the slot's next launch.
//
// Per-CTA roles and tensor memory are those of the plain kernel (two 128-row
// query tiles, head_dim 64 or 128, bf16 P).  Barrier phases run on across
// units: every role derives the same per-unit block counts and keeps the same
// running counters, so each wait knows its phase.
#pragma once

#include "fmha_fwd_kernel.cuh"

namespace fmha {

constexpr int kWorkSlots = 64;
// {units fetched beyond the grid size, CTAs finished} per launch slot
__device__ unsigned int g_work[kWorkSlots][2];

namespace pers {

// Barrier ids.  A parity wait is only unambiguous while its barrier is at
// most one phase away from the phase waited for, and here a waiter may skip
// units, so:
//   * step commits (which free ring slots) rotate over four barriers: the
//     producer waits the commits in order, never more than three behind the
//     MMA warp (each ring load lets it commit at most one more step);
//   * tile 0's S is always signalled on its own barrier (SFull0), which only
//     tile 0's softmax waits, phase by phase;
//   * tile 1's S is the step commit; in a unit where tile 1 has no key block,
//     its softmax warps still wait each step's commit and acknowledge it on
//     PVReady1, and the MMA warp waits for that before the next step commit,
//     so tile 1 never falls behind the step commits nor runs ahead of them.
constexpr int kBarQFull = 0;       // [2]
constexpr int kBarKVFull = 2;      // [4] ring slots
constexpr int kBarSFull0 = 6;      //     S of tile 0 ready
constexpr int kBarPVReady = 7;     // [2] P of tile t stored (4 softmax warps)
constexpr int kBarOFinal = 9;      // [2] last PV of tile t complete
constexpr int kBarMmaDone = 11;    //     every MMA retired
constexpr int kBarStepDone = 12;   // [4] step commit n at n % 4
constexpr int kBarODrained = 16;   // [2] the tile's 4 softmax warps have read O_t out of TMEM
constexpr int kBarUnitFull = 18;   // [4] unit ring entry written by the producer
constexpr int kBarUnitFree = 22;   // [4] unit ring entry read by every consumer
constexpr int kBarQFree = 26;      // [2] the unit's last QK^T of tile t has completed (Q_t may be refilled)
constexpr int kStepBars = 4;
constexpr int kUnitRing = 4;
constexpr int kUnitConsumers = 1 + 2 * 4;  // the MMA thread and the 8 softmax warps
static_assert(kBarQFree + 2 <= 32, "barrier area holds 32 barriers");
// misc words (after the tmem base slot and the abort flag): the release step
// commit of the last load into each ring slot (producer only), then the unit
// ring: each entry a unit decoded by the producer (so that no other role reads
// the sequence bounds from global memory on its way into the next unit)
#ifndef FMHA_PERS_REGS_SOFTMAX
#define FMHA_PERS_REGS_SOFTMAX 192
#endif
// register split after setmaxnreg (softmax, idle, control warpgroups)
#ifndef FMHA_PERS_REGS_IDLE
#define FMHA_PERS_REGS_IDLE 32
#endif
constexpr int kRegsSoftmax = FMHA_PERS_REGS_SOFTMAX, kRegsIdle = FMHA_PERS_REGS_IDLE;
constexpr int kRegsControl = 512 - 2 * kRegsSoftmax - kRegsIdle;
static_assert(kRegsControl % 8 == 0 && kRegsControl >= 24 && kRegsControl <= 256, "register split");
constexpr uint32_t kMiscObsStop = 8;  // trace build: the MMA warp is done
constexpr uint32_t kMiscRelease = 16;
constexpr uint32_t kMiscUnits = 32;
constexpr int kUnitInts = 12;  // one ring entry: unit index (-1: no more units), then the Unit fields
static_assert(kMiscUnits + kUnitRing * kUnitInts * 4 <= 256, "misc area");

struct Unit {
  int h, q0, lq, k0, lk, m0;
  int n_blk0, n_blk1, n_kv;  // key blocks of tile 0, of tile 1 (never fewer), of the unit
};

// Unit u in the plain grid's order: u = h + heads * (launch_pair + pairs * b).
// False if its query block lies past the sequence end (no work at all).
__device__ __forceinline__ bool unit_at(const FwdParams& p, int pairs, int u, Unit& w) {
  w.h = u % p.heads;
  const int rest = u / p.heads;
  const int lp = rest % pairs;
  const int b = rest / pairs;
  const int pair = p.causal ? pairs - 1 - lp : lp;
  if (p.cu_q != nullptr) {
    w.q0 = p.cu_q[b];
    w.lq = p.cu_q[b + 1] - w.q0;
    w.k0 = p.cu_k[b];
    w.lk = p.cu_k[b + 1] - w.k0;
  } else {
    w.q0 = b * p.max_seqlen_q;
    w.lq = p.max_seqlen_q;
    w.k0 = b * p.max_seqlen_k;
    w.lk = p.max_seqlen_k;
  }
  if (w.lk < 0) w.lk = 0;
  w.m0 = pair * (kTiles * kBlockM);
  if (w.m0 >= w.lq) return false;
  w.n_blk0 = tile_blocks(w.m0, w.lq, w.lk, p.causal);
  w.n_blk1 = tile_blocks(w.m0 + kBlockM, w.lq, w.lk, p.causal);
  w.n_kv = max(w.n_blk0, w.n_blk1);
  return true;
}

__device__ __forceinline__ void put_unit(volatile int* e, int u, const Unit& w) {
  e[1] = w.h, e[2] = w.q0, e[3] = w.lq, e[4] = w.k0, e[5] = w.lk, e[6] = w.m0;
  e[7] = w.n_blk0, e[8] = w.n_blk1, e[9] = w.n_kv;
  e[0] = u;
}
__device__ __forceinline__ int get_unit(const volatile int* e, Unit& w) {
  w.h = e[1], w.q0 = e[2], w.lq = e[3], w.k0 = e[4], w.lk = e[5], w.m0 = e[6];
  w.n_blk0 = e[7], w.n_blk1 = e[8], w.n_kv = e[9];
  return e[0];
}

// Step commits of a unit: commit 0 after the first QK^T, commit j + 1 after step j.
__device__ __forceinline__ int unit_commits(const Unit& w) { return w.n_kv > 0 ? w.n_kv + 1 : 0; }

__device__ __forceinline__ bool wait_step(const Ctx& c, int n, int role) {
  return wait_bar(c, kBarStepDone + (n % kStepBars), static_cast<uint32_t>(n / kStepBars) & 1u, role);
}
__device__ __forceinline__ bool wait_step_warp(const Ctx& c, int n, int role) {
  return __all_sync(0xffffffffu, wait_step(c, n, role));
}

// Opt-in trace (build with -DFMHA_TRACE): per CTA, per unit k < kTrUnits,
// kTrEvents %clock64 stamps at slot (cta * kTrUnits + k) * kTrEvents + event:
// 0 unit index, 1 MMA took the unit, 2 its first QK^T issued, 3 its last step
// commit issued, 4 tile 0 saw its first S, 5 tile 1 saw its first S, 6 tile 1
// finished the epilogue, 7 key blocks of the unit, 8 producer published the
// unit, 9 / 10 / 11 producer issued Q_0 / K_0 / Q_1, 12 / 13 / 14 MMA saw
// K_0 / Q_0 / Q_1 landed; for units k < kTrUnits - 1.
// Unit slot kTrUnits - 1 holds the CTA's %globaltimer and %clock64 at entry and
// at exit (events 0, 1 and 2, 3).
constexpr int kTrUnits = 64, kTrEvents = 16;
// The stamps go to shared memory first (a global store would delay the
// thread's next mbarrier arrive, which waits for its earlier stores) and are
// copied out at exit.
#ifdef FMHA_TRACE
constexpr uint32_t kTraceSmemBytes = kTrUnits * kTrEvents * 8;
#else
constexpr uint32_t kTraceSmemBytes = 0;
#endif

// Shared memory: the plain kernel's map, then the trace stamps of a trace build.
template <int HD>
struct Smem {
  static constexpr uint32_t kOffTrace = Dims<HD>::kOffBar + 1024;  // after the barriers and misc words
  static constexpr uint32_t kBytes = kOffTrace + kTraceSmemBytes + 1024;  // + alignment slack
  static_assert(kBytes <= 232448, "shared memory per CTA");
};
#ifdef FMHA_TRACE
__device__ unsigned long long* g_trace_pers;
// observers (warps 14, 15 of the trace build): per CTA two rows of 1024
// %clock64 stamps, when step commit n completed and when ring load g landed
__device__ unsigned long long* g_trace_obs;
#define FMHA_PERS_TRACE(k, e, v)                                             \
  do {                                                                        \
    if (tr_pers != nullptr && (k) < pers::kTrUnits - 1)                       \
      tr_smem[static_cast<size_t>(k) * pers::kTrEvents + (e)] = (v);          \
  } while (0)
#else
#define FMHA_PERS_TRACE(k, e, v) \
  do {                           \
  } while (0)
#endif

}  // namespace pers

template <int HD>
__global__ void __launch_bounds__(kThreads, 1) fmha_fwd_persistent_kernel(const __grid_constant__ FwdParams p) {
  static_assert(HD == 64 || HD == 128, "two query tiles per CTA");
  using D = Dims<HD>;
  using pers::Unit;
  using pers::kBarQFull, pers::kBarKVFull, pers::kBarSFull0, pers::kBarPVReady, pers::kBarOFinal, pers::kBarMmaDone,
      pers::kBarStepDone;
  constexpr int kHeadDim = HD;
  constexpr int kStages = D::kStages;
  static_assert(kStages == 4, "ring of four slots");
  constexpr uint32_t kTileBytes = D::kTileBytes;
  constexpr uint32_t kOffQ = D::kOffQ, kOffKV = D::kOffKV, kOffBar = D::kOffBar, kOffMisc = D::kOffMisc;
  constexpr uint64_t kSlotDescStep = kTileBytes >> 4;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (warp == kWarpProducer && lane == 0) {
    ptx::prefetch_tensormap(&p.tmap_q);
    ptx::prefetch_tensormap(&p.tmap_k);
    ptx::prefetch_tensormap(&p.tmap_v);
  }
#ifdef FMHA_TRACE
  unsigned long long* const tr_pers = pers::g_trace_pers;  // read once
  volatile unsigned long long* const tr_smem =
      reinterpret_cast<volatile unsigned long long*>(smem + pers::Smem<HD>::kOffTrace);
  for (int i = threadIdx.x; i < pers::kTrUnits * pers::kTrEvents; i += blockDim.x) tr_smem[i] = 0ull;
  if (threadIdx.x == 0 && tr_pers != nullptr) {
    tr_smem[(pers::kTrUnits - 1) * pers::kTrEvents + 0] = ptx::globaltimer_ns();
    tr_smem[(pers::kTrUnits - 1) * pers::kTrEvents + 2] = static_cast<unsigned long long>(clock64());
  }
#endif
  const int pairs = (p.max_seqlen_q + kTiles * kBlockM - 1) / (kTiles * kBlockM);
  const int grid = static_cast<int>(gridDim.x);

  Ctx ctx;
  ctx.bar0 = base + kOffBar;
  ctx.abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem + kOffMisc + pers::kMiscUnits);
  volatile int* release = reinterpret_cast<volatile int*>(smem + kOffMisc + pers::kMiscRelease);
#ifdef FMHA_TRACE
  if (threadIdx.x == 0) *reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + pers::kMiscObsStop) = 0u;
#endif

  if (warp == kWarpProducer && lane == 0) {
    for (int t = 0; t < kTiles; ++t) {
      ptx::mbar_init(ctx.bar(kBarQFull + t), 1);
      ptx::mbar_init(ctx.bar(kBarPVReady + t), 4);  // the tile's 4 softmax warps
      ptx::mbar_init(ctx.bar(kBarOFinal + t), 1);
      ptx::mbar_init(ctx.bar(pers::kBarODrained + t), 4);
      ptx::mbar_init(ctx.bar(pers::kBarQFree + t), 1);
    }
    for (int s = 0; s < kStages; ++s) ptx::mbar_init(ctx.bar(kBarKVFull + s), 1);
    for (int s = 0; s < pers::kStepBars; ++s) ptx::mbar_init(ctx.bar(kBarStepDone + s), 1);
    for (int s = 0; s < pers::kUnitRing; ++s) {
      ptx::mbar_init(ctx.bar(pers::kBarUnitFull + s), 1);
      ptx::mbar_init(ctx.bar(pers::kBarUnitFree + s), pers::kUnitConsumers);
    }
    ptx::mbar_init(ctx.bar(kBarSFull0), 1);
    ptx::mbar_init(ctx.bar(kBarMmaDone), 1);
    *ctx.abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // the next published unit (ring entry nu) into w; -1 ends the CTA's work
  auto take_unit = [&](int nu, bool& ok, Unit& w) -> int {
    const int slot = nu & (pers::kUnitRing - 1);
    ok = wait_bar(ctx, pers::kBarUnitFull + slot, static_cast<uint32_t>(nu / pers::kUnitRing) & 1u, kRoleMma);
    return ok ? pers::get_unit(unit_ring + slot * pers::kUnitInts, w) : -1;
  };

  const int wg = warp >> 2;
  if (wg == kWgSoftmax0 || wg == kWgSoftmax0 + 1) {
    // =============================== softmax (tile t = wg), unit after unit
    ptx::setmaxnreg_inc<pers::kRegsSoftmax>();
    const int t = wg - kWgSoftmax0;
    const int r = (warp & 3) * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_off = (static_cast<uint32_t>(warp & 3) * 32u) << 16;
    const uint32_t t_s = tmem + lane_off + col_s(t);
    const uint32_t t_o = tmem + lane_off + col_o(t);
    const float c = p.scale_log2;
    const bool neg = c < 0.f;
    const float s_mask = neg ? INFINITY : -INFINITY;
    int cn = 0;   // step commits of the units before this one (tile 1)
    int s0n = 0;  // S commits of tile 0 before this unit (tile 0)
    int ofn = 0;  // O-final phases waited for
    // ring entry nu into (w, u), the whole warp; false on abort
    auto take = [&](int nu, Unit& w, int& u) -> bool {
      const int slot = nu & (pers::kUnitRing - 1);
      if (!wait_bar_warp(ctx, pers::kBarUnitFull + slot, static_cast<uint32_t>(nu / pers::kUnitRing) & 1u,
                         kRoleSoftmax))
        return false;
      u = pers::get_unit(unit_ring + slot * pers::kUnitInts, w);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ctx.bar(pers::kBarUnitFree + slot));
      return true;
    };
    Unit w;
    int u = -1;
    bool live = take(0, w, u);
    for (int nu = 0; live && u >= 0; ++nu) {
      const int nb = t ? w.n_blk1 : w.n_blk0;
      const bool active = t == 0 || w.m0 + kBlockM < w.lq;
      const int row = w.m0 + kBlockM * t + r;  // sequence-local query index
      const int off = w.lk - w.lq;
      const int key_end = p.causal ? min(row + off + 1, w.lk) : w.lk;
      const int tile_key_end = p.causal ? min(w.m0 + kBlockM * t + off + 1, w.lk) : w.lk;
      float m_used = s_mask;
      float l = 0.f;
      bool ok = true;
      if (t == 1 && nb == 0) {
        // no key block for tile 1: acknowledge each step commit of the unit
        // (S_0(j) ready) so that tile 1 keeps pace with the step commits
        for (int j = 0; j < w.n_kv && ok; ++j) {
          ok = pers::wait_step_warp(ctx, cn + j, kRoleSoftmax);
          if (ok && lane == 0) ptx::mbar_arrive(ctx.bar(kBarPVReady + 1));
        }
      }
      for (int j = 0; j < nb && ok; ++j) {
        const bool s_ok = t == 1 ? pers::wait_step_warp(ctx, cn + j, kRoleSoftmax)
                                 : wait_bar_warp(ctx, kBarSFull0, static_cast<uint32_t>(s0n + j) & 1u, kRoleSoftmax);
        if (!s_ok) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if (j == 0 && r == 0) FMHA_PERS_TRACE(nu, 4 + t, static_cast<unsigned long long>(clock64()));
        float s[128];
        ptx::tmem_ld128_wait(t_s, s);
        const int c0 = j * kBlockN;
        if (tile_key_end - c0 < kBlockN) {  // block crosses the diagonal or the key tail
          const int lim = key_end - c0;
#pragma unroll
          for (int k = 0; k < 128; ++k)
            if (k >= lim) s[k] = s_mask;
        }
        const float m_blk = neg ? row_min128(s) : row_max128(s);
        const float m_ref = (m_blk - m_used) * c > p.rescale_threshold ? m_blk : m_used;
        const float alpha = (m_ref == m_used) ? 1.f : ptx::ex2_approx((m_used - m_ref) * c);
        const float row_sum = exp_pass(s, c, m_ref, t_s);
        // rescale this warp's O rows: PV_t(j - 1) has completed (S_t(j) is
        // committed after it) and PV_t(j) waits for this warp's hand-off
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int cc = 0; cc < HD / 32; ++cc) {
            float o[32];
            ptx::tmem_ld32_wait(t_o + 32u * cc, o);
            uint32_t uo[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) uo[i] = __float_as_uint(o[i] * alpha);
            ptx::tmem_st32(t_o + 32u * cc, uo);
          }
        }
        l = l * alpha + row_sum;
        m_used = m_ref;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ctx.bar(kBarPVReady + t));
      }
      if (!ok) break;
      Unit wn;
      int un = -1;
      // ---- epilogue: O / l -> bf16 and the LSE, one row per thread (the Q
      // buffers already hold the next unit's tiles, so O is not staged).  All
      // of O_t is read out of TMEM and released before the global stores: an
      // mbarrier arrive waits for the thread's earlier stores, and the next
      // unit's first PV waits for this arrive.
      const bool valid = active && row < w.lq;
      if (active) {
        float o[HD];
        if (nb > 0) {
          if (!wait_bar_warp(ctx, kBarOFinal + t, static_cast<uint32_t>(ofn) & 1u, kRoleSoftmax)) break;
          ++ofn;
          ptx::tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < HD / 32; ++cc)
            ptx::tmem_ld32_wait(t_o + 32u * cc, *reinterpret_cast<float(*)[32]>(o + 32 * cc));
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(ctx.bar(pers::kBarODrained + t));
        } else {
#pragma unroll
          for (int i = 0; i < HD; ++i) o[i] = 0.f;
        }
        // the next unit's entry is taken (and released) before the stores too
        live = take(nu + 1, wn, un);
        if (valid) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
          uint4* d4 = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(w.q0 + row) * p.heads + w.h) *
                                                           static_cast<size_t>(kHeadDim));
#pragma unroll
          for (int v4 = 0; v4 < HD / 8; ++v4) {
            uint4 x;
            x.x = ptx::pack_bf16x2(o[8 * v4 + 0] * inv, o[8 * v4 + 1] * inv);
            x.y = ptx::pack_bf16x2(o[8 * v4 + 2] * inv, o[8 * v4 + 3] * inv);
            x.z = ptx::pack_bf16x2(o[8 * v4 + 4] * inv, o[8 * v4 + 5] * inv);
            x.w = ptx::pack_bf16x2(o[8 * v4 + 6] * inv, o[8 * v4 + 7] * inv);
            d4[v4] = x;
          }
        }
      }
      if (!active) live = take(nu + 1, wn, un);
      if (p.lse != nullptr && valid) {
        const float lse = (l > 0.f) ? (m_used * c + log2f(l)) * 0.69314718055994531f : -INFINITY;
        p.lse[static_cast<size_t>(w.h) * p.total_q + w.q0 + row] = lse;
      }
      if (t == 1 && r == 0) FMHA_PERS_TRACE(nu, 6, static_cast<unsigned long long>(clock64()));
      cn += pers::unit_commits(w);
      s0n += w.n_blk0;
      w = wn;
      u = un;
    }
  } else if (wg == kWgIdle) {
    // =============================== idle (its registers go to the softmax)
    ptx::setmaxnreg_dec<pers::kRegsIdle>();
  } else {
    ptx::setmaxnreg_dec<pers::kRegsControl>();
    if (warp == kWarpProducer) {
      // =============================== producer: fetches units, publishes
      // them in the unit ring, loads their Q tiles and K/V blocks
      if (lane == 0) {
        const uint64_t pol_q = ptx::policy_evict_first();
        const uint64_t pol_kv = ptx::policy_evict_last();
        int nu = 0;     // units published
        int ld = 0;     // ring loads issued
        int cbase = 0;  // step commit 0 of the current unit (= step commits of the units before it)
        int qloads[kTiles] = {0, 0};
        bool ok = true;
        // the first unit with work from u on (later candidates from the counter), or >= units
        auto claim = [&](int u, Unit& w) -> int {
          while (u < p.units && !pers::unit_at(p, pairs, u, w)) u = grid + static_cast<int>(atomicAdd(p.work, 1u));
          return u;
        };
        // publish unit u (-1: no more) in the unit ring
        auto publish = [&](int u, const Unit& w) -> bool {
          const int slot = nu & (pers::kUnitRing - 1);
          if (nu >= pers::kUnitRing &&
              !wait_bar(ctx, pers::kBarUnitFree + slot, static_cast<uint32_t>(nu / pers::kUnitRing - 1) & 1u,
                        kRoleLoad))
            return false;
          pers::put_unit(unit_ring + slot * pers::kUnitInts, u < p.units ? u : -1, w);
          ptx::mbar_arrive(ctx.bar(pers::kBarUnitFull + slot));
          FMHA_PERS_TRACE(nu, 8, static_cast<unsigned long long>(clock64()));
          ++nu;
          return true;
        };
        Unit w;
        int u = claim(static_cast<int>(blockIdx.x), w);
        ok = publish(u, w);
        while (ok && u < p.units) {
          int pending = -1;  // the counter value taken for the next unit
          const int xh = w.h * kHeadDim;
          const int xkv = (w.h / p.kv_group) * kHeadDim;
          // Q_t, once the previous unit's last QK^T of tile t has completed
          auto load_q = [&](int t) -> bool {
            if ((t ? w.n_blk1 : w.n_blk0) == 0) return true;
            if (qloads[t] > 0 &&
                !wait_bar(ctx, pers::kBarQFree + t, static_cast<uint32_t>(qloads[t] - 1) & 1u, kRoleLoad))
              return false;
            const uint32_t bar = ctx.bar(kBarQFull + t);
            ptx::mbar_arrive_expect_tx(bar, kTileBytes);
            const uint32_t dst = base + kOffQ + t * kTileBytes;
            const int y = w.q0 + w.m0 + kBlockM * t;
#pragma unroll
            for (int hf = 0; hf < D::kHalves; ++hf)
              ptx::tma_load_2d(dst + hf * kHalfBytes, &p.tmap_q, bar, xh + 64 * hf, y, pol_q);
            FMHA_PERS_TRACE(nu - 1, 9 + 2 * t, static_cast<unsigned long long>(clock64()));
            ++qloads[t];
            return true;
          };
          // what the unit's first S needs first: Q_0, K_0, then Q_1 and the rest
          if (!load_q(0)) break;
          for (int i = 0; i < 2 * w.n_kv && ok; ++i) {
            if (i == 1) {
              // Q_1 and V_0 wait for the previous unit's last steps: start
              // their DRAM reads into L2 now
              if (w.n_blk1 > 0)
#pragma unroll
                for (int hf = 0; hf < D::kHalves; ++hf)
                  ptx::tma_prefetch_2d(&p.tmap_q, xh + 64 * hf, w.q0 + w.m0 + kBlockM);
#pragma unroll
              for (int hf = 0; hf < D::kHalves; ++hf) ptx::tma_prefetch_2d(&p.tmap_v, xkv + 64 * hf, w.k0);
              if (!load_q(1)) {
                ok = false;
                break;
              }
            }
            // Two key blocks before the unit's last load (a few steps before its
            // end) take the next unit from the counter, so that the CTAs that
            // finish first take the remaining units; the atomic's latency
            // passes while the last loads wait for their slots.
            if (i == max(0, 2 * w.n_kv - 4)) pending = static_cast<int>(atomicAdd(p.work, 1u));
            const int g = ld++;
            const int s = g & (kStages - 1);
            // the slot's previous block was last read by the MMAs of step commit release[s]
            if (g >= kStages && !pers::wait_step(ctx, release[s], kRoleLoad)) {
              ok = false;
              break;
            }
            const uint32_t bar = ctx.bar(kBarKVFull + s);
            ptx::mbar_arrive_expect_tx(bar, kTileBytes);
            const uint32_t dst = base + kOffKV + s * kTileBytes;
            const CUtensorMap* m = (i & 1) ? &p.tmap_v : &p.tmap_k;
            const int y = w.k0 + kBlockN * (i >> 1);
#pragma unroll
            for (int hf = 0; hf < D::kHalves; ++hf)
              ptx::tma_load_2d(dst + hf * kHalfBytes, m, bar, xkv + 64 * hf, y, pol_kv);
            // K_b is last read by QK^T(b) (step commit b), V_b by PV(b) (commit b + 1)
            release[s] = cbase + (i >> 1) + (i & 1);
            if (i == 0) FMHA_PERS_TRACE(nu - 1, 10, static_cast<unsigned long long>(clock64()));
          }
          if (!ok) break;
          cbase += pers::unit_commits(w);
          if (pending < 0) pending = static_cast<int>(atomicAdd(p.work, 1u));  // a unit without key blocks
          // every load of this unit is issued: publish the next, whose first
          // loads (Q_0, K_0) can usually go out at once
          u = claim(grid + pending, w);
          if (!publish(u, w)) break;
        }
        // every issued copy has landed before the CTA may exit
        for (int g = max(0, ld - kStages); g < ld; ++g)
          wait_drain(ctx, kBarKVFull + (g & (kStages - 1)), static_cast<uint32_t>(g / kStages) & 1u);
#pragma unroll
        for (int t = 0; t < kTiles; ++t)
          if (qloads[t] > 0) wait_drain(ctx, kBarQFull + t, static_cast<uint32_t>(qloads[t] - 1) & 1u);
      }
      __syncwarp();
    } else if (warp == kWarpMma) {
      // =============================== MMA issuer, unit after unit (the plain
      // kernel's per-step order), plus: the first PV_t of a unit waits until
      // the softmax warps have read the previous unit's O_t
      if (lane == 0) {
        const uint64_t q_desc[kTiles] = {desc_kmajor(base + kOffQ), desc_kmajor(base + kOffQ + kTileBytes)};
        const uint64_t kv_desc = desc_kmajor(base + kOffKV);
        const uint64_t kv_desc_mn = desc_mnmajor(base + kOffKV);
        int ld = 0;                          // ring loads consumed
        int cn = 0;                          // step commits made
        int qn[kTiles] = {0, 0};             // Q_t phases consumed
        int pvn[kTiles] = {0, 0};            // P_t hand-offs consumed
        int on[kTiles] = {0, 0};             // units whose O_t was final
        bool issued_any = false;
        bool ok = true;
        for (int nu = 0; ok; ++nu) {
          Unit w;
          const int u = take_unit(nu, ok, w);
          if (!ok) break;
          ptx::mbar_arrive(ctx.bar(pers::kBarUnitFree + (nu & (pers::kUnitRing - 1))));
          if (u < 0) break;
          FMHA_PERS_TRACE(nu, 1, static_cast<unsigned long long>(clock64()));
          FMHA_PERS_TRACE(nu, 0, static_cast<unsigned long long>(u));
          FMHA_PERS_TRACE(nu, 7, static_cast<unsigned long long>(w.n_kv));
          if (w.n_kv == 0) continue;
          auto n_blk = [&](int t) { return t ? w.n_blk1 : w.n_blk0; };
          {
            const int ks = ld & (kStages - 1);
            if (!wait_bar(ctx, kBarKVFull + ks, static_cast<uint32_t>(ld / kStages) & 1u, kRoleMma)) break;
            FMHA_PERS_TRACE(nu, 12, static_cast<unsigned long long>(clock64()));
#pragma unroll
            for (int t = 0; t < kTiles; ++t) {
              if (ok && n_blk(t) > 0) {
                ok = wait_bar(ctx, kBarQFull + t, static_cast<uint32_t>(qn[t]) & 1u, kRoleMma);
                if (!ok) break;
                FMHA_PERS_TRACE(nu, 13 + t, static_cast<unsigned long long>(clock64()));
                ++qn[t];
                ptx::tc_fence_after();
                issue_qk<HD>(tmem + col_s(t), q_desc[t], kv_desc + kSlotDescStep * ks);
                if (t == 1) FMHA_PERS_TRACE(nu, 15, static_cast<unsigned long long>(clock64()));
                issued_any = true;
                if (t == 0) ptx::mma_commit(ctx.bar(kBarSFull0));
                if (n_blk(t) == 1) ptx::mma_commit(ctx.bar(pers::kBarQFree + t));  // the tile's last QK^T
              }
            }
            if (!ok) break;
            ptx::mma_commit(ctx.bar(kBarStepDone + cn % pers::kStepBars));
            ++cn;
            FMHA_PERS_TRACE(nu, 2, static_cast<unsigned long long>(clock64()));
          }
          for (int j = 0; j < w.n_kv && ok; ++j) {
            const int vidx = ld + 2 * j + 1, vs = vidx & (kStages - 1);
            if (!wait_bar(ctx, kBarKVFull + vs, static_cast<uint32_t>(vidx / kStages) & 1u, kRoleMma)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const int kidx = ld + 2 * j + 2, ks = kidx & (kStages - 1);
            bool k_ready = false;
#pragma unroll
            for (int t = 0; t < kTiles; ++t) {
              if (!ok || j >= n_blk(t)) continue;
              if (!wait_bar(ctx, kBarPVReady + t, static_cast<uint32_t>(pvn[t]) & 1u, kRoleMma)) {
                ok = false;
                break;
              }
              ++pvn[t];
              if (j == 0 && on[t] > 0 &&
                  !wait_bar(ctx, pers::kBarODrained + t, static_cast<uint32_t>(on[t] - 1) & 1u, kRoleMma)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              issue_pv<HD>(tmem + col_o(t), tmem + col_s(t), kv_desc_mn + kSlotDescStep * vs, j > 0);
              if (j + 1 < n_blk(t)) {
                if (!k_ready) {
                  if (!wait_bar(ctx, kBarKVFull + ks, static_cast<uint32_t>(kidx / kStages) & 1u, kRoleMma)) {
                    ok = false;
                    break;
                  }
                  ptx::tc_fence_after();
                  k_ready = true;
                }
                issue_qk<HD>(tmem + col_s(t), q_desc[t], kv_desc + kSlotDescStep * ks);
                if (t == 0) ptx::mma_commit(ctx.bar(kBarSFull0));
                if (j + 2 == n_blk(t)) ptx::mma_commit(ctx.bar(pers::kBarQFree + t));  // the tile's last QK^T
              } else {
                ptx::mma_commit(ctx.bar(kBarOFinal + t));
                ++on[t];
              }
            }
            if (!ok) break;
            // tile 1 without key blocks acknowledges every step (see the barrier ids)
            if (w.n_blk1 == 0) {
              if (!wait_bar(ctx, kBarPVReady + 1, static_cast<uint32_t>(pvn[1]) & 1u, kRoleMma)) {
                ok = false;
                break;
              }
              ++pvn[1];
            }
            ptx::mma_commit(ctx.bar(kBarStepDone + cn % pers::kStepBars));
            ++cn;
          }
          ld += 2 * w.n_kv;
          FMHA_PERS_TRACE(nu, 3, static_cast<unsigned long long>(clock64()));
        }
        if (issued_any) {  // all MMAs retired before TMEM is released
          ptx::mma_commit(ctx.bar(kBarMmaDone));
          wait_drain(ctx, kBarMmaDone, 0);
        }
#ifdef FMHA_TRACE
        *reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + pers::kMiscObsStop) = 1u;
#endif
      }
      __syncwarp();
    }
#ifdef FMHA_TRACE
    else if (lane == 0 && pers::g_trace_obs != nullptr) {
      // trace build only: warp 14 stamps step commits completing, warp 15 ring
      // loads landing, in order, until the MMA warp is done
      volatile uint32_t* stop = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + pers::kMiscObsStop);
      unsigned long long* row =
          pers::g_trace_obs + (static_cast<size_t>(blockIdx.x) * 2 + (warp - kWarpMma - 1)) * 1024;
      for (int n = 0; n < 1024; ++n) {
        const int id = warp == kWarpMma + 1 ? kBarStepDone + n % pers::kStepBars : kBarKVFull + n % kStages;
        const uint32_t par = static_cast<uint32_t>(warp == kWarpMma + 1 ? n / pers::kStepBars : n / kStages) & 1u;
        bool seen = false;
        const uint64_t g0 = ptx::globaltimer_ns();
        while (!*stop && ptx::globaltimer_ns() - g0 < 200000ull)
          if (ptx::mbar_try_wait(ctx.bar(id), par)) {
            seen = true;
            break;
          }
        if (!seen) break;
        row[n] = static_cast<unsigned long long>(clock64());
      }
    }
#endif
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
#ifdef FMHA_TRACE
  if (threadIdx.x == 0 && tr_pers != nullptr) {
    tr_smem[(pers::kTrUnits - 1) * pers::kTrEvents + 1] = ptx::globaltimer_ns();
    tr_smem[(pers::kTrUnits - 1) * pers::kTrEvents + 3] = static_cast<unsigned long long>(clock64());
  }
  __syncthreads();
  if (tr_pers != nullptr)
    for (int i = threadIdx.x; i < pers::kTrUnits * pers::kTrEvents; i += blockDim.x)
      tr_pers[static_cast<size_t>(blockIdx.x) * pers::kTrUnits * pers::kTrEvents + i] = tr_smem[i];
#endif
  if (threadIdx.x == 0) {
    // the last CTA of the launch resets the counter slot for its next launch;
    // every CTA's fetches were made before its own increment below
    __threadfence();
    if (atomicAdd(p.work + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.work, 0u);
      atomicExch(p.work + 1, 0u);
    }
  }
}

}  // namespace fmha
