// fmha_api.cu -- host launcher and C ABI of libfmha.so (declared in fmha.h).
//
// Validates arguments without touching the GPU, encodes the three TMA tensor
// maps (Q, K, V viewed as 2-D [tokens, heads * head_dim] bf16, 64 x 128 boxes
// with 128-byte swizzle), and launches the kernel for head_dim 64, 128 or 256:
// one CTA per (head, 256-row query block, sequence), or 128-row blocks for
// head_dim 256.  The kernel orders the units in groups of a few heads, and causal
// launches walk query blocks from the last to the first so the longest units
// start first.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <mutex>

#include "fmha.h"
#include "fmha_fwd_kernel.cuh"
#include "fmha_fwd_persistent.cuh"
#include "fmha_bwd_kernel.cuh"
#include "fmha_fp8_prepass.cuh"

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [tokens, heads * head_dim] bf16, row stride heads * head_dim * 2 bytes, box 64 x 128,
// 128B swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int tokens, int heads, int head_dim) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads) * head_dim, static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads) * head_dim * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Per-sequence K/V size above which the head-grouped grid order is used (a
// little under the 129 MB L2, which also holds the Q and O streams).  A test
// build lowers it so that small problems, which the oracle checks in full,
// take the head-grouped order too.
#ifndef FMHA_L2_GROUP_BYTES
#define FMHA_L2_GROUP_BYTES (int64_t(96) << 20)
#endif
constexpr int64_t kL2GroupBytes = FMHA_L2_GROUP_BYTES;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <int HD, bool kGrouped, bool kFp8 = false>
int configure_kernel() {
  static int rc = -1;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  // per-process attribute; re-applied cheaply if a previous attempt failed
  if (rc != 0) {
    rc = cudaFuncSetAttribute(fmha::fmha_fwd_kernel<HD, kGrouped, kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(fmha::Dims<HD>::kSmemBytes + fmha::kTraceSmemBytes)) == cudaSuccess
             ? 0
             : 1;
  }
  return rc;
}

template <int HD, bool kGrouped, bool kFp8 = false>
int launch(const fmha::FwdParams& p, dim3 grid, fmha_stream_t stream) {
  if (configure_kernel<HD, kGrouped, kFp8>() != 0) return FMHA_ERR_CUDA;
  fmha::fmha_fwd_kernel<HD, kGrouped, kFp8><<<grid, fmha::kThreads, fmha::Dims<HD>::kSmemBytes + fmha::kTraceSmemBytes,
                                              reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? FMHA_OK : FMHA_ERR_CUDA;
}

// The persistent kernel runs when the plain grid would take more than
// FMHA_PERSISTENT_WAVES waves of CTAs (one CTA per SM), i.e. when many units
// would each pay their own set-up and epilogue.  Test builds lower the
// threshold and cap the grid (FMHA_PERSISTENT_MAX_CTAS) so that small problems
// run many units per CTA.
#ifndef FMHA_PERSISTENT_WAVES
#define FMHA_PERSISTENT_WAVES 1
#endif
#ifndef FMHA_PERSISTENT_MAX_CTAS
#define FMHA_PERSISTENT_MAX_CTAS 0
#endif

template <int HD>
int configure_persistent() {
  static int rc = -1;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (rc != 0) {
    rc = cudaFuncSetAttribute(fmha::fmha_fwd_persistent_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(fmha::pers::Smem<HD>::kBytes)) == cudaSuccess
             ? 0
             : 1;
  }
  return rc;
}

// SM count of the current device (cached per device).
int sm_count() {
  static int counts[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    counts[dev] = n;
  }
  return counts[dev];
}

// A counter slot of the persistent kernel for this launch: slots are handed
// out round-robin, so launches in flight at the same time use different ones.
unsigned int* work_slot() {
  static void* base[64] = {nullptr};
  static std::mutex mu;
  static unsigned int next = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (base[dev] == nullptr && cudaGetSymbolAddress(&base[dev], fmha::g_work) != cudaSuccess) {
    base[dev] = nullptr;
    return nullptr;
  }
  const unsigned int s = next++ % fmha::kWorkSlots;
  return static_cast<unsigned int*>(base[dev]) + 2 * s;
}

template <int HD>
int launch_persistent(fmha::FwdParams& p, int ctas, fmha_stream_t stream) {
  if (configure_persistent<HD>() != 0) return FMHA_ERR_CUDA;
  p.work = work_slot();
  if (p.work == nullptr) return FMHA_ERR_CUDA;
  fmha::fmha_fwd_persistent_kernel<HD><<<ctas, fmha::kThreads, fmha::pers::Smem<HD>::kBytes,
                                         reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? FMHA_OK : FMHA_ERR_CUDA;
}

// The backward pass's dK/dV kernel runs on a second stream of the library's,
// forked from the caller's stream once D is written and joined back before
// the call returns, so that the dQ and dK/dV CTAs fill each other's last
// waves (when one sequence's K/V fits in L2).  One stream and two events per device, created on first use; the
// fork, the launch and the join are made under a lock, so that calls from
// several host threads do not interleave their event records.  A stream
// capture follows the fork and the join (the second stream joins the capture
// through the first event).  -DFMHA_BWD_FORK=0 runs both on the caller's stream.
#ifndef FMHA_BWD_FORK
#define FMHA_BWD_FORK 1
#endif
struct BwdFork {
  cudaStream_t aux = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool ready = false;
};
std::mutex g_bwd_fork_mu;

// this device's fork objects (under g_bwd_fork_mu), or nullptr
BwdFork* bwd_fork_locked() {
  static BwdFork forks[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  BwdFork& f = forks[dev];
  if (!f.ready) {
    if (cudaStreamCreateWithFlags(&f.aux, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
    f.ready = true;
  }
  return &f;
}

// e4m3 V^T [rows, kpad] bytes (keys contiguous), box 128 keys x 128 rows, 128B swizzle.
bool make_map_vt(CUtensorMap* m, const void* ptr, int64_t rows, int64_t kpad) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kpad), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kpad)};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Workspace of the FP8 variant: per-K/V-head max |V| (float bits), then the
// e4m3 V^T at a 256-byte boundary.
size_t fp8_amax_bytes(int kv_heads) { return (static_cast<size_t>(kv_heads) * 4 + 255) / 256 * 256; }

}  // namespace

extern "C" int fmha_fwd_gqa(const void* q, const void* k, const void* v, void* out, float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
                            int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int heads,
                            int kv_heads, int head_dim, float scale, int causal, fmha_stream_t stream) {
  // ---- validation: no GPU work before this point
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return FMHA_ERR_INVALID_ARG;
  if (heads < 1 || kv_heads < 1 || heads % kv_heads != 0) return FMHA_ERR_INVALID_ARG;
  if ((cu_seqlens_q == nullptr) != (cu_seqlens_k == nullptr)) return FMHA_ERR_INVALID_ARG;
  if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || heads < 1)
    return FMHA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FMHA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FMHA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      (lse != nullptr && !aligned(lse, 4)))
    return FMHA_ERR_INVALID_ARG;
  if (cu_seqlens_q == nullptr) {
    if (static_cast<int64_t>(batch) * max_seqlen_q != total_q ||
        static_cast<int64_t>(batch) * max_seqlen_k != total_k)
      return FMHA_ERR_INVALID_ARG;
  }
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return FMHA_ERR_UNSUPPORTED;
  if (batch > 65535) return FMHA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(heads) * head_dim * 2 >= (int64_t(1) << 32)) return FMHA_ERR_UNSUPPORTED;

  // query rows per CTA: two 128-row tiles, one for head_dim 256
  const int unit_rows = (head_dim == 256 ? 1 : fmha::kTiles) * fmha::kBlockM;
  const int pairs = (max_seqlen_q + unit_rows - 1) / unit_rows;
  if (batch == 0 || total_q == 0 || pairs == 0) return FMHA_OK;  // nothing to compute
  // Rasterise in groups of kHeadGroup heads when one sequence's K/V does not fit
  // in L2: the CTAs in flight then read the K/V of about kHeadGroup heads.
  const int64_t kv_bytes = static_cast<int64_t>(kv_heads) * max_seqlen_k * head_dim * 4;  // K and V, bf16
  // (head_dim 256 keeps the plain order: its grouped variant would spill registers)
  const bool grouped = head_dim != 256 && kv_bytes > kL2GroupBytes && heads > fmha::kHeadGroup;
  if (grouped ? static_cast<int64_t>(heads) * pairs > INT32_MAX : pairs > 65535) return FMHA_ERR_UNSUPPORTED;

  fmha::FwdParams p;
  // a k/v tensor with no rows still needs a valid map extent; it is never read then
  const int tk = total_k > 0 ? total_k : 1;
  if (!make_map(&p.tmap_q, q, total_q, heads, head_dim) || !make_map(&p.tmap_k, k, tk, kv_heads, head_dim) ||
      !make_map(&p.tmap_v, v, tk, kv_heads, head_dim))
    return FMHA_ERR_CUDA;
  p.kv_group = heads / kv_heads;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.batch = batch;
  p.total_q = total_q;
  p.total_k = total_k;
  p.max_seqlen_q = max_seqlen_q;
  p.max_seqlen_k = max_seqlen_k;
  p.heads = heads;
  p.causal = causal;
  // scale * log2(e), folded into the softmax FMA.  A zero (or denormal) scale
  // runs as +-2^-126, the smallest normal float: every visible key then gets
  // the weight 2^(s * 2^-126 - m * 2^-126), which is 1 in fp32, and masked keys
  // keep -inf instead of the NaN of -inf * 0.
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  if (std::fabs(p.scale_log2) < FLT_MIN) p.scale_log2 = std::signbit(scale) ? -FLT_MIN : FLT_MIN;
  p.rescale_threshold = 8.0f;

  if (grouped) {
    const dim3 grid(static_cast<unsigned>(heads * pairs), static_cast<unsigned>(batch), 1u);
    return head_dim == 64 ? launch<64, true>(p, grid, stream) : launch<128, true>(p, grid, stream);
  }
  const int64_t units = static_cast<int64_t>(heads) * pairs * batch;
  const int sms = sm_count();
  if (head_dim != 256 && sms > 0 && units > static_cast<int64_t>(FMHA_PERSISTENT_WAVES) * sms && units <= INT32_MAX / 2) {
    int ctas = sms;
    if (FMHA_PERSISTENT_MAX_CTAS > 0) ctas = std::min(ctas, FMHA_PERSISTENT_MAX_CTAS);
    ctas = static_cast<int>(std::min<int64_t>(ctas, units));
    p.units = static_cast<int>(units);
    return head_dim == 64 ? launch_persistent<64>(p, ctas, stream) : launch_persistent<128>(p, ctas, stream);
  }
  const dim3 grid(static_cast<unsigned>(heads), static_cast<unsigned>(pairs), static_cast<unsigned>(batch));
  if (head_dim == 64) return launch<64, false>(p, grid, stream);
  return head_dim == 128 ? launch<128, false>(p, grid, stream) : launch<256, false>(p, grid, stream);
}

extern "C" size_t fmha_fwd_fp8pv_workspace_size(int batch, int total_k, int kv_heads, int head_dim) {
  if (batch < 0 || total_k < 0 || kv_heads < 1 || head_dim < 1) return 0;
  const int64_t kpad = fmha::fp8::padded_keys(total_k, batch);
  return fp8_amax_bytes(kv_heads) + static_cast<size_t>(kv_heads) * head_dim * static_cast<size_t>(kpad);
}

extern "C" int fmha_fwd_fp8pv(const void* q, const void* k, const void* v, void* out, float* lse, void* workspace,
                              const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch, int total_q,
                              int total_k, int max_seqlen_q, int max_seqlen_k, int heads, int kv_heads,
                              int head_dim, float scale, int causal, fmha_stream_t stream) {
  // ---- validation: no GPU work before this point
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || workspace == nullptr)
    return FMHA_ERR_INVALID_ARG;
  if (heads < 1 || kv_heads < 1 || heads % kv_heads != 0) return FMHA_ERR_INVALID_ARG;
  if ((cu_seqlens_q == nullptr) != (cu_seqlens_k == nullptr)) return FMHA_ERR_INVALID_ARG;
  if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0) return FMHA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FMHA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FMHA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(workspace, 256) ||
      (lse != nullptr && !aligned(lse, 4)))
    return FMHA_ERR_INVALID_ARG;
  if (cu_seqlens_q == nullptr) {
    if (static_cast<int64_t>(batch) * max_seqlen_q != total_q ||
        static_cast<int64_t>(batch) * max_seqlen_k != total_k)
      return FMHA_ERR_INVALID_ARG;
  }
  if (head_dim != 128) return FMHA_ERR_UNSUPPORTED;
  if (batch > 65535) return FMHA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(heads) * head_dim * 2 >= (int64_t(1) << 32)) return FMHA_ERR_UNSUPPORTED;
  const int64_t kpad = fmha::fp8::padded_keys(total_k, batch);
  if (kpad + fmha::kBlockN >= (int64_t(1) << 31)) return FMHA_ERR_UNSUPPORTED;  // TMA x coordinates are int32
  const int pairs = (max_seqlen_q + fmha::kTiles * fmha::kBlockM - 1) / (fmha::kTiles * fmha::kBlockM);
  if (batch == 0 || total_q == 0 || pairs == 0) return FMHA_OK;
  const int64_t kv_bytes = static_cast<int64_t>(kv_heads) * max_seqlen_k * head_dim * 4;
  const bool grouped = kv_bytes > kL2GroupBytes && heads > fmha::kHeadGroup;
  if (grouped ? static_cast<int64_t>(heads) * pairs > INT32_MAX : pairs > 65535) return FMHA_ERR_UNSUPPORTED;

  fmha::FwdParams p;
  const int tk = total_k > 0 ? total_k : 1;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* amax = reinterpret_cast<uint32_t*>(ws);
  uint8_t* vt = ws + fp8_amax_bytes(kv_heads);
  if (!make_map(&p.tmap_q, q, total_q, heads, head_dim) || !make_map(&p.tmap_k, k, tk, kv_heads, head_dim) ||
      !make_map(&p.tmap_v, v, tk, kv_heads, head_dim) ||
      !make_map_vt(&p.tmap_vt, vt, static_cast<int64_t>(kv_heads) * head_dim, kpad > 0 ? kpad : 16))
    return FMHA_ERR_CUDA;
  p.v_amax_bits = amax;
  p.kv_group = heads / kv_heads;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.batch = batch;
  p.total_q = total_q;
  p.total_k = total_k;
  p.max_seqlen_q = max_seqlen_q;
  p.max_seqlen_k = max_seqlen_k;
  p.heads = heads;
  p.causal = causal;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  if (std::fabs(p.scale_log2) < FLT_MIN) p.scale_log2 = std::signbit(scale) ? -FLT_MIN : FLT_MIN;
  p.rescale_threshold = 8.0f;

  // V -> e4m3 V^T (max |V| per K/V head, then quantise and transpose)
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  fmha::fp8::PrepassParams pp;
  pp.v = static_cast<const __nv_bfloat16*>(v);
  pp.amax_bits = amax;
  pp.vt = vt;
  pp.cu_k = cu_seqlens_k;
  pp.batch = batch;
  pp.total_k = total_k;
  pp.max_seqlen_k = max_seqlen_k;
  pp.kv_heads = kv_heads;
  pp.head_dim = head_dim;
  pp.kpad = kpad;
  if (cudaMemsetAsync(amax, 0, static_cast<size_t>(kv_heads) * 4, st) != cudaSuccess) return FMHA_ERR_CUDA;
  if (total_k > 0) {
    const int64_t chunks = (static_cast<int64_t>(total_k) + fmha::fp8::kAmaxTokens - 1) / fmha::fp8::kAmaxTokens;
    fmha::fp8::v_amax_kernel<<<dim3(static_cast<unsigned>(chunks), kv_heads), fmha::fp8::kAmaxThreads, 0, st>>>(pp);
    if (cudaGetLastError() != cudaSuccess) return FMHA_ERR_CUDA;
  }
  if (kpad > 0) {
    fmha::fp8::v_quant_kernel<<<dim3(static_cast<unsigned>((kpad + 127) / 128), kv_heads), fmha::fp8::kQuantThreads,
                                0, st>>>(pp);
    if (cudaGetLastError() != cudaSuccess) return FMHA_ERR_CUDA;
  }
  if (grouped) return launch<128, true, true>(p, dim3(static_cast<unsigned>(heads * pairs), batch, 1u), stream);
  return launch<128, false, true>(p, dim3(heads, pairs, batch), stream);
}

extern "C" int fmha_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int heads,
                        int head_dim, float scale, int causal, fmha_stream_t stream) {
  return fmha_fwd_gqa(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, max_seqlen_q,
                      max_seqlen_k, heads, heads, head_dim, scale, causal, stream);
}

namespace {

template <typename Kernel>
int set_smem(Kernel kernel, uint32_t bytes, int& rc, std::mutex& mu) {
  std::lock_guard<std::mutex> lock(mu);
  if (rc != 0)
    rc = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) ==
                 cudaSuccess
             ? 0
             : 1;
  return rc;
}

int configure_bwd() {
  static int rc_dq = -1, rc_kv = -1;
  static std::mutex mu;
  if (set_smem(fmha::bwd::fmha_bwd_dq_kernel, fmha::bwd::DqSmem::kBytes, rc_dq, mu) != 0) return 1;
  return set_smem(fmha::bwd::fmha_bwd_dkdv_kernel, fmha::bwd::DkvSmem::kBytes, rc_kv, mu);
}

}  // namespace

extern "C" size_t fmha_bwd_workspace_size(int heads, int total_q) {
  if (heads < 0 || total_q < 0) return 0;
  return static_cast<size_t>(heads) * static_cast<size_t>(total_q) * sizeof(float);
}

extern "C" int fmha_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, float* workspace,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch, int total_q,
                        int total_k, int max_seqlen_q, int max_seqlen_k, int heads, int kv_heads, int head_dim,
                        float scale, int causal, fmha_stream_t stream) {
  // ---- validation: no GPU work before this point
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || dout == nullptr || lse == nullptr ||
      dq == nullptr || dk == nullptr || dv == nullptr || workspace == nullptr)
    return FMHA_ERR_INVALID_ARG;
  if (heads < 1 || kv_heads < 1 || heads % kv_heads != 0) return FMHA_ERR_INVALID_ARG;
  if ((cu_seqlens_q == nullptr) != (cu_seqlens_k == nullptr)) return FMHA_ERR_INVALID_ARG;
  if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0) return FMHA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FMHA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FMHA_ERR_INVALID_ARG;
  const void* p16[] = {q, k, v, out, dout, dq, dk, dv};
  for (const void* x : p16)
    if (!aligned(x, 16)) return FMHA_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || !aligned(workspace, 4)) return FMHA_ERR_INVALID_ARG;
  if (cu_seqlens_q == nullptr) {
    if (static_cast<int64_t>(batch) * max_seqlen_q != total_q ||
        static_cast<int64_t>(batch) * max_seqlen_k != total_k)
      return FMHA_ERR_INVALID_ARG;
  }
  if (head_dim != 128) return FMHA_ERR_UNSUPPORTED;
  if (batch > 65535) return FMHA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(heads) * head_dim * 2 >= (int64_t(1) << 32)) return FMHA_ERR_UNSUPPORTED;
  const int qblocks = (max_seqlen_q + fmha::kBlockM - 1) / fmha::kBlockM;
  const int kblocks = (max_seqlen_k + fmha::kBlockN - 1) / fmha::kBlockN;
  if (qblocks > 65535 || kblocks > 65535) return FMHA_ERR_UNSUPPORTED;
  if (batch == 0 || (total_q == 0 && total_k == 0)) return FMHA_OK;

  fmha::bwd::BwdParams p;
  const int tq = total_q > 0 ? total_q : 1;  // a map needs a nonzero extent; it is never read then
  const int tk = total_k > 0 ? total_k : 1;
  if (!make_map(&p.tmap_q, q, tq, heads, head_dim) || !make_map(&p.tmap_do, dout, tq, heads, head_dim) ||
      !make_map(&p.tmap_k, k, tk, kv_heads, head_dim) || !make_map(&p.tmap_v, v, tk, kv_heads, head_dim))
    return FMHA_ERR_CUDA;
  p.out = static_cast<const __nv_bfloat16*>(out);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  p.dvec = workspace;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.batch = batch;
  p.total_q = total_q;
  p.total_k = total_k;
  p.max_seqlen_q = max_seqlen_q;
  p.max_seqlen_k = max_seqlen_k;
  p.heads = heads;
  p.kv_heads = kv_heads;
  p.causal = causal;
  p.kv_group = heads / kv_heads;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);

  if (configure_bwd() != 0) return FMHA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // D = rowsum(dO * O) into the workspace, then dQ, then dK / dV (both read D)
  if (total_q > 0) {
    const int64_t rows = static_cast<int64_t>(total_q) * heads;
    const int64_t blocks = std::min<int64_t>((rows + 15) / 16, 152 * 32);  // 16 rows per 256-thread block pass
    fmha::bwd::fmha_bwd_dot_kernel<<<static_cast<unsigned>(blocks), fmha::bwd::kDotThreads, 0, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FMHA_ERR_CUDA;
  }
  const bool run_dq = qblocks > 0 && total_q > 0, run_dkdv = kblocks > 0 && total_k > 0;
  std::unique_lock<std::mutex> lock(g_bwd_fork_mu, std::defer_lock);
  BwdFork* fork = nullptr;
  // (a sequence whose K/V exceeds L2 keeps both kernels on the caller's stream:
  // run at once, their CTAs would split L2 between two working sets)
  const bool kv_fits_l2 = static_cast<int64_t>(kv_heads) * max_seqlen_k * head_dim * 4 <= kL2GroupBytes;
  if (FMHA_BWD_FORK && run_dq && run_dkdv && kv_fits_l2) {
    lock.lock();
    fork = bwd_fork_locked();
    if (fork != nullptr && (cudaEventRecord(fork->fork, st) != cudaSuccess ||
                            cudaStreamWaitEvent(fork->aux, fork->fork, 0) != cudaSuccess))
      return FMHA_ERR_CUDA;
  }
  if (run_dq) {
    fmha::bwd::fmha_bwd_dq_kernel<<<dim3(heads, qblocks, batch), fmha::bwd::kDqThreads, fmha::bwd::DqSmem::kBytes,
                                    st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FMHA_ERR_CUDA;
  }
  if (run_dkdv) {
    fmha::bwd::fmha_bwd_dkdv_kernel<<<dim3(kv_heads, kblocks, batch), fmha::bwd::kDkvThreads,
                                      fmha::bwd::DkvSmem::kBytes, fork != nullptr ? fork->aux : st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FMHA_ERR_CUDA;
  }
  if (fork != nullptr &&
      (cudaEventRecord(fork->join, fork->aux) != cudaSuccess || cudaStreamWaitEvent(st, fork->join, 0) != cudaSuccess))
    return FMHA_ERR_CUDA;
  return FMHA_OK;
}

// ---------------------------------------------------------------------------
// fmha_bwd_noalloc: fmha_bwd for callers that cannot allocate device memory
// (code running where cudaMalloc is unavailable or forbidden, e.g. inside a
// host allocator's own hooks, a plugin whose host owns all memory, or a
// process that has reserved the whole device up front).  The backward pass's
// one scratch buffer, D = rowsum(dO * O), then lives in the fixed array below,
// which every GPU that loads this library holds until the process exits.
namespace {

constexpr size_t kStaticScratchFloats = size_t(1) << 21;  // 8 MiB: heads * total_q <= 2,097,152
__device__ __align__(256) float g_bwd_static_scratch[kStaticScratchFloats];

// The array's device address, looked up once per device with that device
// current.  In host code the array's name is only a stand-in, never a device
// address.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_addr[kMaxDevices] = {};

int static_scratch(float** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FMHA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (dev >= 0 && dev < kMaxDevices && g_scratch_addr[dev] != nullptr) {
    *ptr = g_scratch_addr[dev];
    return FMHA_OK;
  }
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_bwd_static_scratch) != cudaSuccess || addr == nullptr) return FMHA_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevices) g_scratch_addr[dev] = static_cast<float*>(addr);
  *ptr = static_cast<float*>(addr);
  return FMHA_OK;
}

}  // namespace

extern "C" int fmha_bwd_noalloc(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_seqlens_q,
                                const int32_t* cu_seqlens_k, int batch, int total_q, int total_k,
                                int max_seqlen_q, int max_seqlen_k, int heads, int kv_heads, int head_dim,
                                float scale, int causal, fmha_stream_t stream) {
  if (heads < 1 || total_q < 0) return FMHA_ERR_INVALID_ARG;
  if (static_cast<size_t>(heads) * static_cast<size_t>(total_q) > kStaticScratchFloats)
    return FMHA_ERR_UNSUPPORTED;  // D would not fit the fixed scratch array
  float* scratch = nullptr;
  const int rc = static_scratch(&scratch);
  if (rc != FMHA_OK) return rc;
  // Nothing in the array needs to start at zero: the dQ kernel writes every
  // entry of D that the dK/dV kernel then reads.
  return fmha_bwd(q, k, v, out, dout, lse, dq, dk, dv, scratch, cu_seqlens_q, cu_seqlens_k, batch, total_q,
                  total_k, max_seqlen_q, max_seqlen_k, heads, kv_heads, head_dim, scale, causal, stream);
}

extern "C" int fmha_get_device_status(fmha_stream_t stream, int* detail) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FMHA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, fmha::g_status, sizeof(int)) != cudaSuccess) return FMHA_ERR_CUDA;
  if (word == 0) {
    if (detail) *detail = 0;
    return FMHA_OK;
  }
  const int zero = 0;
  if (cudaMemcpyToSymbol(fmha::g_status, &zero, sizeof(int)) != cudaSuccess) return FMHA_ERR_CUDA;
  if (detail) *detail = word - 1;
  return FMHA_ERR_TIMEOUT;
}

extern "C" const char* fmha_status_string(int status) {
  switch (status) {
    case FMHA_OK: return "ok";
    case FMHA_ERR_INVALID_ARG: return "invalid argument";
    case FMHA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FMHA_ERR_CUDA: return "CUDA error";
    case FMHA_ERR_TIMEOUT: return "device pipeline wait timed out";
    default: return "unknown status";
  }
}

extern "C" int fmha_version(void) { return 10100; }

#ifdef FMHA_TRACE
// Trace builds only: point the kernel's trace at a device buffer of
// (query blocks) x 2048 uint64 slots (see fmha_trace.h), or nullptr to stop.
extern "C" int fmha_debug_set_trace(void* device_buffer) {
  unsigned long long* p = static_cast<unsigned long long*>(device_buffer);
  return cudaMemcpyToSymbol(fmha::g_trace, &p, sizeof(p)) == cudaSuccess ? FMHA_OK : FMHA_ERR_CUDA;
}

// Trace builds only: backward-pass stamps, (query blocks) x 1024 and (key
// blocks) x 1024 uint64 slots for the dQ and dK/dV kernels, or nullptr.
extern "C" int fmha_debug_set_bwd_trace(void* dq_buffer, void* dkdv_buffer) {
  unsigned long long* a = static_cast<unsigned long long*>(dq_buffer);
  unsigned long long* b = static_cast<unsigned long long*>(dkdv_buffer);
  if (cudaMemcpyToSymbol(fmha::bwd::g_trace_dq, &a, sizeof(a)) != cudaSuccess) return FMHA_ERR_CUDA;
  return cudaMemcpyToSymbol(fmha::bwd::g_trace_dkdv, &b, sizeof(b)) == cudaSuccess ? FMHA_OK : FMHA_ERR_CUDA;
}

// Trace builds only: persistent-kernel stamps, (grid size) x 64 units x 16
// uint64 slots, or nullptr.
extern "C" int fmha_debug_set_pers_trace(void* device_buffer) {
  unsigned long long* p = static_cast<unsigned long long*>(device_buffer);
  return cudaMemcpyToSymbol(fmha::pers::g_trace_pers, &p, sizeof(p)) == cudaSuccess ? FMHA_OK : FMHA_ERR_CUDA;
}

// Trace builds only: persistent-kernel observer stamps, (grid size) x 2 x 1024
// uint64 slots, or nullptr.
extern "C" int fmha_debug_set_pers_obs_trace(void* device_buffer) {
  unsigned long long* p = static_cast<unsigned long long*>(device_buffer);
  return cudaMemcpyToSymbol(fmha::pers::g_trace_obs, &p, sizeof(p)) == cudaSuccess ? FMHA_OK : FMHA_ERR_CUDA;
}

// Trace builds only: per-CTA table of 4 uint64 per CTA (grid size x 4), or nullptr.
extern "C" int fmha_debug_set_cta_trace(void* device_buffer) {
  unsigned long long* p = static_cast<unsigned long long*>(device_buffer);
  return cudaMemcpyToSymbol(fmha::g_trace_ctas, &p, sizeof(p)) == cudaSuccess ? FMHA_OK : FMHA_ERR_CUDA;
}
#endif
