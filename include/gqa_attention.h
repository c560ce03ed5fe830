/*
 * gqa_attention.h -- C ABI of the grouped-query decode attention over a bf16 key/value cache
 * (GB300, sm_103a).  Part of libmoe_gb300.so; shares its status codes and its workspace error
 * word with moe.h.
 *
 * What the call computes (sources: news pages about Perplexity's "Lily" engine):
 *   - The model's full-attention layers use grouped-query attention with sixteen query heads and
 *     two key/value heads.  ("Perplexity libera Lily: inferencia en Rust y Metal para Mac",
 *     section "Tres formas de carga en un mismo modelo".)
 *   - At decode, attention reads a key/value cache that grows with the context.  The query heads
 *     of one group share one thread group, so every key and value row is loaded once (GQA
 *     packing), and long contexts are laid out in fixed blocks.  (Same page, section "Decode:
 *     mover menos bytes por token"; "Прибавка к MLX-LM в цифрах" on neuro-ai.ru lists the same
 *     two techniques.)
 * Readings where the pages are silent: head size 128; query head h reads key/value head
 * h / (Hq / Hkv); scores q . k / sqrt(128); softmax over the N cached positions (the new token's
 * key and value are already appended); one sequence per call; fp32 output.
 *
 * For each query head h with group g = h / (Hq / Hkv):
 *   o[h, :] = sum_n softmax_n(q[h, :] . K[g, n, :] / sqrt(128)) V[g, n, :],  n = 0 .. N-1.
 *
 * How it runs: the N positions are cut into fixed tiles of 64 positions; each CTA of the first
 * launch takes a contiguous run of tiles of one key/value head (about one CTA per SM over all
 * heads), streams them through shared memory with tensor-map copies, and keeps a running softmax
 * for all query heads of the group; a second launch merges the runs of each head in a fixed order.
 * Results are identical from run to run.
 *
 * Conventions are those of moe.h: device pointers owned by the caller, 16-byte aligned; work is
 * enqueued on `stream` (a cudaStream_t, NULL = legacy default stream); argument checks on the host
 * before any launch; inputs never written.  Scratch and the error word live in the caller's
 * workspace (clear its first 4 bytes once with moe_clear_error_flags; read them with
 * moe_read_error_flags).  Bits this call may set: 1 (a bounded wait timed out; o invalid) and
 * 8 (an output is not finite, which only non-finite or overflowing inputs cause).
 */
#ifndef GQA_ATTENTION_GB300_H_
#define GQA_ATTENTION_GB300_H_

#include <stddef.h>
#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Shapes of one decode-attention call.
 *   n_heads     Hq, query heads, >= 1
 *   n_kv_heads  Hkv, key/value heads, >= 1, Hq % Hkv == 0, Hq / Hkv <= 8, Hkv <= 65535
 *   head_dim    D, must be 128
 *   n_ctx       N, cached positions to attend over, 1 <= N <= capacity
 *   capacity    positions allocated per key/value head (row stride of the cache), < 2^31 */
typedef struct gqa_dims {
  int32_t n_heads, n_kv_heads, head_dim, n_ctx, capacity;
} gqa_dims;

/* Workspace bytes for these dims (the 256-byte head holding the error word, then per-block
 * partial results: Hkv * min(ceil(N / 64), 256) blocks of 4160 bytes).  0 for invalid dims. */
size_t gqa_decode_workspace_bytes(const gqa_dims* dims);

/* One decode step of grouped-query attention.
 *   q        bf16 [Hq, 128]                    the new token's queries (uint16 bit patterns)
 *   k_cache  bf16 [Hkv, capacity, 128]         keys; positions 0 .. N-1 are read, the rest never
 *   v_cache  bf16 [Hkv, capacity, 128]         values, same layout
 *   o        fp32 [Hq, 128]                    output
 *   workspace / workspace_bytes                >= gqa_decode_workspace_bytes(dims)
 * Returns MOE_ERR_INVALID_ARG for a null pointer, Hq % Hkv != 0, N < 1 or N > capacity;
 * MOE_ERR_UNSUPPORTED for head_dim != 128, Hq / Hkv > 8 or the size limits above;
 * MOE_ERR_MISALIGNED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA as in moe.h.  Two launches on `stream`:
 * the block pass and the merge (the merge under programmatic dependent launch).
 * Ordering: copies of the cached positions below 64 * floor((N - 1) / 64) (every 64-position tile
 * but the last) may start before the work enqueued just before this call on `stream` has finished
 * (programmatic dependent launch); q and the last tile, which holds position N - 1 (the new token's
 * key and value), are read only after it has finished.  So no work still in flight when the call
 * is enqueued may write those earlier positions. */
moe_status gqa_decode_attention(const gqa_dims* dims, const uint16_t* q, const uint16_t* k_cache,
                                const uint16_t* v_cache, float* o, void* workspace, size_t workspace_bytes,
                                void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTENTION_GB300_H_ */
