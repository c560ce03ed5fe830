/*
 * deltanet_scan.h -- C ABI of the Gated DeltaNet recurrent scan (GB300, sm_103a).  Part of
 * libmoe_gb300.so; shares its status codes and its workspace error word with moe.h.
 *
 * What the call computes.  The model's thirty recurrent layers are Gated DeltaNet layers, and the
 * engine scans their recurrence with the state carried in registers ("Perplexity libera Lily:
 * inferencia en Rust y Metal para Mac", sections "Tres formas de carga en un mismo modelo" and
 * "Prefill: pesos comprimidos y enrutamiento en la GPU"; "Perplexity ouvre le code de Lily...",
 * lefilia.fr, article body).  The recurrence is the gated delta rule of the published Gated DeltaNet
 * (Yang, Kautz and Hatamizadeh, ICLR 2025); for each head, with the state S of shape [128, 128]
 * (value rows by key columns):
 *
 *   k^_t = k_t / sqrt(|k_t|^2 + 1e-6),   q^_t = q_t / sqrt(|q_t|^2 + 1e-6) / sqrt(128)
 *   S_t  = exp(g_t) S_{t-1} + beta_t (v_t - exp(g_t) S_{t-1} k^_t) k^_t^T
 *   o_t  = S_t q^_t
 *
 * Readings where the pages are silent: key and value size 128; q and k normalised per head and
 * token as the published layer does; the decay g (log scale, <= 0) and the write strength beta
 * come from the caller (the gate projections are outside the scan).
 *
 * How it runs: the rows of S are independent given the keys, so each CTA holds 16 rows of one
 * head's state in registers (eight lanes per row, sixteen fp32 values a lane) for the whole
 * sequence and walks the tokens in order; a fifth warp stages the next 32 tokens' keys, queries and
 * values by tensor-map copies and normalises them while the scan runs.  The state is read once at
 * the start and written once at the end.
 *
 * Conventions are those of moe.h: device pointers owned by the caller, 16-byte aligned; work is
 * enqueued on `stream`; argument checks on the host before any launch; inputs never written except
 * that state_out may be the same buffer as state_in (an in-place update).  Error bits this call may
 * set in the workspace's error word: 1 (a bounded wait timed out; outputs invalid) and 8 (the final
 * state is not finite).
 */
#ifndef DELTANET_SCAN_GB300_H_
#define DELTANET_SCAN_GB300_H_

#include <stddef.h>
#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* T tokens, H heads, key size d_k and value size d_v (both must be 128). */
typedef struct gdn_dims {
  int32_t T, H, d_k, d_v;
} gdn_dims;

/* Workspace bytes: the 256-byte head that holds the error word.  0 for invalid dims. */
size_t gdn_scan_workspace_bytes(const gdn_dims* dims);

/* The scan over T tokens of one sequence.
 *   q, k      bf16 [T, H, 128]   (uint16 bit patterns)
 *   v         bf16 [T, H, 128]
 *   g         fp32 [T, H]        log decay
 *   beta      fp32 [T, H]        write strength
 *   state_in  fp32 [H, 128, 128] S before the first token (row = value index, column = key index)
 *   state_out fp32 [H, 128, 128] S after the last token; may equal state_in
 *   o         fp32 [T, H, 128]
 * Returns MOE_ERR_INVALID_ARG for a null pointer or T < 0 or H < 1; MOE_ERR_UNSUPPORTED for
 * d_k or d_v other than 128, H > 65535 or T * H * 128 >= 2^31; MOE_ERR_MISALIGNED, MOE_ERR_WORKSPACE,
 * MOE_ERR_CUDA as in moe.h.  T == 0 copies state_in to state_out (when they differ).  One launch
 * on `stream`, under programmatic dependent launch (every input is read after the preceding work
 * on the stream has finished). */
moe_status gdn_scan(const gdn_dims* dims, const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* g,
                    const float* beta, const float* state_in, float* state_out, float* o, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Option bits of gdn_scan_opts. */
#define GDN_OPT_STATE_EARLY 1u

/* gdn_scan with options; options == 0 is gdn_scan.
 * GDN_OPT_STATE_EARLY: state_in is read before the preceding work on the stream has finished (the
 * scan warps load their rows of S before the programmatic-launch wait, so the load overlaps the
 * end of that work; q, k, v, g and beta are still read after it).  The caller promises that the
 * work immediately preceding this call on the stream does not write state_in: in a decode loop
 * each layer's state was last written by that layer's own scan of the previous token, many
 * launches earlier.  Results are identical to gdn_scan's.
 * Returns MOE_ERR_INVALID_ARG for an unknown option bit; otherwise as gdn_scan. */
moe_status gdn_scan_opts(const gdn_dims* dims, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const float* g, const float* beta, const float* state_in, float* state_out, float* o,
                         void* workspace, size_t workspace_bytes, void* stream, uint32_t options);

#ifdef __cplusplus
}
#endif

#endif /* DELTANET_SCAN_GB300_H_ */
