/*
 * fmha_trace.h -- debug hook of trace builds of libfmha.so (compiled with
 * -DFMHA_TRACE); the default build does not export it.
 *
 * The coarse pipeline trace follows the method of "Kernel Bottleneck Tuning",
 * section "2. Trace the real pipeline, coarsely": timestamps only at role
 * hand-off points, so that the instrumented kernel keeps its schedule.
 */
#ifndef FMHA_TRACE_H_
#define FMHA_TRACE_H_
#ifdef __cplusplus
extern "C" {
#endif

/*
 * fmha_debug_set_trace -- device_buffer: caller-owned device memory of
 * gridDim.y (query blocks of 256 rows) x 2048 uint64 slots, or NULL.  The
 * CTAs of head 0 / sequence 0 write %clock64 stamps into row blockIdx.y; the
 * slot map is the kTr* constants of fmha_fwd_kernel.cuh.  Returns FMHA_OK or
 * FMHA_ERR_CUDA.
 */
int fmha_debug_set_trace(void *device_buffer);

/*
 * fmha_debug_set_cta_trace -- device_buffer: caller-owned device memory of
 * (grid size) x 4 uint64, or NULL.  Every CTA writes, at its linear block id,
 * %globaltimer (ns) at entry, after the set-up sync and at exit, and its SM
 * id.  Returns FMHA_OK or FMHA_ERR_CUDA.
 */
int fmha_debug_set_cta_trace(void *device_buffer);

/*
 * fmha_debug_set_bwd_trace -- caller-owned device buffers of
 * ceil(max_seqlen_q / 128) x 1024 and ceil(max_seqlen_k / 128) x 1024 uint64
 * for the %clock64 stamps of the backward pass's dQ and dK/dV kernels (CTAs
 * of head 0, sequence 0), or NULL to stop.
 */
int fmha_debug_set_bwd_trace(void *dq_buffer, void *dkdv_buffer);

/*
 * fmha_debug_set_pers_trace -- caller-owned device memory of (grid size) x 64
 * x 16 uint64, or NULL: the persistent forward kernel's stamps, per CTA and per
 * unit it ran (the first 63), at the slots that fmha_fwd_persistent.cuh
 * lists (unit index, %clock64 at the MMA warp's and the softmax warps'
 * hand-offs, key blocks).  Returns FMHA_OK or FMHA_ERR_CUDA.
 */
int fmha_debug_set_pers_trace(void *device_buffer);

/*
 * fmha_debug_set_pers_obs_trace -- caller-owned device memory of (grid size)
 * x 2 x 1024 uint64, or NULL: in the persistent forward kernel's trace build,
 * two otherwise idle warps stamp (%clock64) when each step commit completes
 * and when each ring load lands, in order (the first 1024 of each).
 */
int fmha_debug_set_pers_obs_trace(void *device_buffer);

#ifdef __cplusplus
}
#endif
#endif
