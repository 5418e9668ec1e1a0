/*
 * fmha.h -- C ABI of libfmha.so, a fused multi-head attention forward for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (after "[BUG] Unexpected Slower Performance in C++ CuTe
 * (77_blackwell_fmha) vs Python CuTe DSL (fmha.py) on Jetson Thor", sections
 * "Test Commands" and "Implementation Differences in softmax_step", and
 * "[BUG] CuTe DSL 4.7/4.8 regression: FlashAttention-4 SM100 forward kernel
 * spills registers", section "Steps/Code to reproduce bug"):
 *
 *   for every sequence b, head h and query row i of b:
 *     s_ij  = scale * q_i . k_j   over keys j of sequence b,
 *             keys with j >= Lk, or (causal) j > i + Lk - Lq, are masked out
 *     O_i   = sum_j softmax_j(s_ij) v_j            (bf16 output)
 *     LSE_i = log(sum_j exp(s_ij))                  (natural log, fp32)
 *
 * A row with no visible key (Lk = 0, or causal with i + Lk - Lq < 0) gets
 * O_i = 0 and LSE_i = -inf.  The causal diagonal is aligned to the
 * bottom-right corner, which is the usual top-left one when Lq == Lk.
 *
 * Threading / ownership: every pointer argument is device memory owned by
 * the caller.  The library allocates no device memory per call and keeps no
 * per-call state; calls are asynchronous on `stream` and never synchronise
 * it.  The host never reads device memory (cu_seqlens are read on the GPU).
 */
#ifndef FMHA_H_
#define FMHA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (0 = the legacy default stream). */
typedef struct CUstream_st *fmha_stream_t;

enum fmha_status_code {
    FMHA_OK = 0,
    FMHA_ERR_INVALID_ARG = 1, /* a null or misaligned pointer, inconsistent sizes */
    FMHA_ERR_UNSUPPORTED = 2, /* a valid request this build does not handle (e.g. head_dim not 64, 128, 256) */
    FMHA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, tensor map) */
    FMHA_ERR_TIMEOUT = 4      /* a device-side pipeline wait gave up (see fmha_get_device_status) */
};

/*
 * fmha_fwd -- O = softmax(scale * Q K^T [+ causal mask]) V and the per-row LSE.
 *
 * q            bf16 [total_q, heads, head_dim], contiguous, 16-byte aligned.
 * k, v         bf16 [total_k, heads, head_dim], contiguous, 16-byte aligned.
 * out          bf16 [total_q, heads, head_dim], contiguous, 16-byte aligned.
 *              Rows of every sequence are written; nothing else is touched.
 * lse          fp32 [heads, total_q], 4-byte aligned, or NULL (not written).
 * cu_seqlens_q int32 [batch + 1] device array of prefix offsets into the
 * cu_seqlens_k token dimension (cu[0] = 0, non-decreasing, cu[batch] =
 *              total), as in the varlen layout of the page above.  Both NULL
 *              selects dense batches: sequence b holds rows
 *              [b * max_seqlen, (b + 1) * max_seqlen) -- the [b, s, h, d]
 *              layout -- and then total_q == batch * max_seqlen_q and
 *              total_k == batch * max_seqlen_k are required.
 * batch        number of sequences (>= 0; <= 65535).
 * total_q,     token counts of q/out and of k/v.  The library needs them for
 * total_k      the tensor-map bounds and the LSE layout because it never
 *              reads cu_seqlens on the host.
 * max_seqlen_q an upper bound on every sequence's query / key length, as in
 * max_seqlen_k the page's varlen call (the caller's responsibility; a longer
 *              sequence is not fully computed).  The launch has one CTA per
 *              head, 256-query-row block and sequence: FMHA_ERR_UNSUPPORTED
 *              if ceil(max_seqlen_q / 256) > 65535, or, when one sequence's
 *              K/V exceeds 96 MiB (the grid is then ordered in head groups),
 *              if heads * ceil(max_seqlen_q / 256) > 2^31 - 1.
 * heads        >= 1.
 * head_dim     64, 128 or 256 (else FMHA_ERR_UNSUPPORTED).  The pages' runs
 *              use 128; 64 and 256 are adjacent sizes their command line also
 *              takes.  head_dim 256 runs one 128-row query block per CTA.
 * scale        finite softmax scale of any sign, e.g. 1/sqrt(128); no default
 *              is applied.  scale = 0 gives every visible key the same weight
 *              (O = mean of the visible V rows, LSE = log of their count).
 * causal       0 or 1.
 * stream       CUDA stream the kernel is enqueued on.
 *
 * Returns FMHA_OK once the kernel is enqueued (or when there is no work),
 * FMHA_ERR_INVALID_ARG / FMHA_ERR_UNSUPPORTED before touching the GPU, or
 * FMHA_ERR_CUDA if encoding the tensor maps or the launch failed.  A device
 * pipeline wait that gives up does not fault the GPU: the kernel stops, its
 * outputs are unspecified, and fmha_get_device_status reports it.
 */
int fmha_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
             const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
             int batch, int total_q, int total_k,
             int max_seqlen_q, int max_seqlen_k, int heads, int head_dim,
             float scale, int causal, fmha_stream_t stream);

/*
 * fmha_fwd_gqa -- fmha_fwd with grouped K/V heads (grouped-query attention;
 * kv_heads == 1 is multi-query attention).  Not on the pages above; the
 * plainest extension of their operation: query head h attends with K/V head
 * h / (heads / kv_heads), so consecutive query heads share one K/V head.
 *
 * k, v         bf16 [total_k, kv_heads, head_dim], contiguous, 16-byte aligned.
 * kv_heads     >= 1 and a divisor of heads (else FMHA_ERR_INVALID_ARG).
 * Every other argument, the return values and the error behaviour are those
 * of fmha_fwd, which is fmha_fwd_gqa with kv_heads == heads.
 */
int fmha_fwd_gqa(const void *q, const void *k, const void *v, void *out, float *lse,
                 const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                 int batch, int total_q, int total_k,
                 int max_seqlen_q, int max_seqlen_k, int heads, int kv_heads, int head_dim,
                 float scale, int causal, fmha_stream_t stream);

/*
 * fmha_fwd_fp8pv -- fmha_fwd_gqa with the O += P V product on FP8 (e4m3)
 * operands, after "Kernel Bottleneck Tuning" (sections "4. If scheduling has
 * no headroom: eliminate instructions algebraically" and "5. Tune the
 * producer->consumer handoff split"), whose attention forward runs P V in
 * FP8.  Opt-in: the result is less accurate than fmha_fwd's.
 *
 * P is rounded to e4m3 after the exponent (P <= 2^8 by the lazy-rescale
 * threshold, inside e4m3's range); V is rounded to e4m3 as V / s with one scale
 * s = max|V| / 448 per K/V head, folded into the epilogue's 1 / l; the row sum
 * l and the LSE use the unrounded P (the LSE is as accurate as fmha_fwd's).
 * Expected error of O against exact attention: relative RMS a few 1e-2, and
 * at most about 2^-3 * max|V| for any element (half an e4m3 unit on P and on V).
 *
 * workspace    device memory of fmha_fwd_fp8pv_workspace_size(batch, total_k,
 *              kv_heads, head_dim) bytes, 256-byte aligned, owned by the
 *              caller, contents on entry irrelevant.  The call writes into it:
 *              at offset 0, max|V| per K/V head as float bits; at offset
 *              ceil(kv_heads * 4 / 256) * 256, the e4m3 values of V / s as
 *              [kv_heads][head_dim][kpad] bytes with keys contiguous, sequence
 *              b's key i at column 16 * (ceil(k0(b) / 16) + b) + i (k0(b) its
 *              first key token, kpad = 16 * (ceil(total_k / 16) + batch)) and
 *              zeros between sequences.  Calls that share a workspace must
 *              not overlap on the GPU.
 * head_dim     128 (else FMHA_ERR_UNSUPPORTED).
 * All other arguments, return values and errors are those of fmha_fwd_gqa.
 * Three kernels are enqueued on `stream` (max |V|, quantise and transpose V,
 * attention) after a cudaMemsetAsync of the max words; nothing is allocated.
 */
int fmha_fwd_fp8pv(const void *q, const void *k, const void *v, void *out, float *lse, void *workspace,
                   const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                   int batch, int total_q, int total_k,
                   int max_seqlen_q, int max_seqlen_k, int heads, int kv_heads, int head_dim,
                   float scale, int causal, fmha_stream_t stream);

/* Bytes of workspace fmha_fwd_fp8pv needs (0 for an invalid argument). */
size_t fmha_fwd_fp8pv_workspace_size(int batch, int total_k, int kv_heads, int head_dim);

/*
 * fmha_bwd -- gradients of the forward pass: dQ, dK, dV of L = sum(dO * O).
 *
 * The benchmark step of "[BUG] CuTe DSL 4.7/4.8 regression: FlashAttention-4
 * SM100 forward kernel spills registers" (section "Steps/Code to reproduce
 * bug") runs this pass after the varlen causal forward.  With
 * P_ij = exp(scale * q_i . k_j - LSE_i) over the visible keys (0 elsewhere):
 *
 *   dV_j = sum_i P_ij dO_i               D_i   = dO_i . O_i
 *   dS_ij = P_ij (dO_i . v_j - D_i)      dQ_i  = scale * sum_j dS_ij k_j
 *                                        dK_j  = scale * sum_i dS_ij q_i
 *
 * summed over every query head that reads a K/V head (grouped K/V heads as
 * in fmha_fwd_gqa).
 *
 * q, out, dout bf16 [total_q, heads, head_dim]; out and lse are the outputs
 *              of fmha_fwd / fmha_fwd_gqa for these q, k, v (lse required).
 * k, v         bf16 [total_k, kv_heads, head_dim].
 * dq           bf16 [total_q, heads, head_dim]: rows of every sequence written.
 * dk, dv       bf16 [total_k, kv_heads, head_dim]: keys of every sequence
 *              written (0 for a key no query sees).
 * workspace    fp32 device scratch of fmha_bwd_workspace_size(heads, total_q)
 *              bytes, 4-byte aligned, owned by the caller; it receives D.  Its
 *              contents on entry do not matter; two calls in flight at the
 *              same time must not share it.
 * All other arguments are those of fmha_fwd_gqa (kv_heads == heads for
 * multi-head attention).  head_dim must be 128 (else FMHA_ERR_UNSUPPORTED);
 * ceil(max_seqlen_q / 128) and ceil(max_seqlen_k / 128) at most 65535.
 * Every 16-byte alignment rule of fmha_fwd applies to q, k, v, out, dout,
 * dq, dk and dv.
 *
 * Three kernels are enqueued on `stream` (D, then dQ, then dK and dV); the
 * call allocates nothing and never synchronises.  Returns as fmha_fwd does.
 */
int fmha_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout,
             const float *lse, void *dq, void *dk, void *dv, float *workspace,
             const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
             int batch, int total_q, int total_k,
             int max_seqlen_q, int max_seqlen_k, int heads, int kv_heads, int head_dim,
             float scale, int causal, fmha_stream_t stream);

/* Bytes of device workspace fmha_bwd needs: heads * total_q * 4 (0 for a
 * negative argument). */
size_t fmha_bwd_workspace_size(int heads, int total_q);

/*
 * fmha_bwd_noalloc -- fmha_bwd without the workspace argument, for callers
 * that cannot allocate device memory: code that runs where cudaMalloc is
 * unavailable or not allowed (inside an allocator's own hooks, a plugin whose
 * host owns every byte of device memory, a process that reserved the whole
 * device up front).  The pages have no counterpart of this entry point.
 *
 * The scratch that fmha_bwd takes from the caller (D, heads * total_q
 * floats) lives instead in one fixed array of 8 MiB inside this library,
 * which every GPU that loads the library holds until the process exits.
 * heads * total_q must be at most 2,097,152 (2^21); a larger problem is
 * refused with FMHA_ERR_UNSUPPORTED before any GPU work.  The call allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).
 *
 * The first call on each device looks the array's device address up with
 * that device current (cudaGetSymbolAddress); make that first call before
 * any stream capture.  Every call shares the one array per device and leaves
 * its contents behind (nothing in it has to start at zero), so calls whose
 * work overlaps on the GPU race on it: issue them on one stream, or order
 * them.  Arguments, outputs and return values are otherwise those of
 * fmha_bwd.
 */
int fmha_bwd_noalloc(const void *q, const void *k, const void *v, const void *out, const void *dout,
                     const float *lse, void *dq, void *dk, void *dv,
                     const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                     int batch, int total_q, int total_k,
                     int max_seqlen_q, int max_seqlen_k, int heads, int kv_heads, int head_dim,
                     float scale, int causal, fmha_stream_t stream);

/*
 * fmha_get_device_status -- synchronise `stream`, then read and clear the
 * device status word of the current device.  Returns FMHA_OK if no kernel
 * reported a problem since the last call, FMHA_ERR_TIMEOUT if a pipeline wait
 * gave up (then *detail, if non-NULL, receives which wait: role * 256 +
 * barrier id), or FMHA_ERR_CUDA if the synchronisation itself failed.
 */
int fmha_get_device_status(fmha_stream_t stream, int *detail);

/* Human-readable name of a status code (static storage, never NULL). */
const char *fmha_status_string(int status);

/* ABI version of this library: major * 10000 + minor * 100 + patch. */
int fmha_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FMHA_H_ */
