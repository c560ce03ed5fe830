/*
 * moe_probe.h -- measurement aid of the GB300 MoE layer library (libmoe_gb300.so); not part of the
 * layer's computation.
 *
 * The pages report that the engine's decode kernels reach 97.9 % of memory bandwidth on matrix
 * operations and that removing all arithmetic changes decode speed by only 0.2 % ("Perplexity
 * открыла код Lily - движка для локальных моделей на Mac", section "Спекулятивное декодирование
 * не взлетело").  The entry point below reproduces that experiment for this library's decode
 * kernel: it moves exactly the weight bytes one token's decode layer call moves, with the same
 * grid, thread-block clusters, shared-memory plan, copy instructions and programmatic dependent
 * launch, and does no arithmetic.  Its time per call is the bandwidth ceiling of the decode
 * kernel's access pattern.  A second entry point makes the library's bounded device waits run out
 * on purpose, so that tests can see the timeout reported and the context survive it.
 */
#ifndef MOE_GB300_PROBE_H_
#define MOE_GB300_PROBE_H_

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Loads-only replica of moe_layer_forward's one-token decode launch.
 *   dims       as for moe_layer_forward, with T == 1 and dims the decode kernel takes
 *              (MOE_ERR_UNSUPPORTED otherwise);
 *   idx        int32 [k] device pointer: the token's experts in slot order (as moe_route writes
 *              them), each in 0..E-1 (not checked on the device: an index out of range reads
 *              outside the weights);
 *   routed, shared, workspace, workspace_bytes, stream: as for moe_layer_forward (only the
 *              workspace's error word is used; bit 1 is set if a copy never landed).
 * Nothing is written except the error word.  T == 0 is a no-op. */
moe_status moe_decode_stream_probe(const moe_dims* dims, const int32_t* idx, const moe_experts* routed,
                                   const moe_experts* shared, void* workspace, size_t workspace_bytes, void* stream);

/* Test aid for the library's bounded waits: one CTA waits on an mbarrier that nothing completes,
 * through the same wait every kernel of the library uses, but giving up after limit_cycles SM
 * cycles instead of the kernels' fixed limit (about two seconds).  The wait gives up, sets bit 1
 * (a bounded device wait timed out) of the workspace's error word, and the kernel returns; the
 * context stays usable.  limit_cycles must lie in 1 .. 4e9 (MOE_ERR_INVALID_ARG otherwise); the
 * workspace must hold at least the error word (256 bytes, 16-byte aligned: MOE_ERR_WORKSPACE /
 * MOE_ERR_MISALIGNED otherwise).  Nothing is written except the error word. */
moe_status moe_wait_timeout_probe(void* workspace, size_t workspace_bytes, long long limit_cycles, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_PROBE_H_ */
