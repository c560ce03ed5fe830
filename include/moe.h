/*
 * moe.h -- C ABI of the GB300 (sm_103a) mixture-of-experts layer with 4-bit affine experts.
 *
 * What the layer computes (sources: four news pages about Perplexity's "Lily" engine):
 *   - Weights are 4-bit affine codes in groups of 64 with one bf16 scale and one bf16 bias per
 *     group, w = q * scale + bias; the GPU rebuilds them tile by tile inside the grouped GEMM and
 *     accumulates in FP32, so the expanded weights never reach memory.  ("Perplexity libera
 *     Lily: inferencia en Rust y Metal para Mac", section "Prefill: pesos comprimidos y
 *     enrutamiento en la GPU".)
 *   - A router scores 256 experts and keeps eight; a shared expert sees every token.  (Same
 *     page, section "Tres formas de carga en un mismo modelo"; "Perplexity ouvre le code de
 *     Lily...", article body.)
 *   - The routing histogram, prefix scan, scatter and block map stay on the GPU with no host
 *     synchronisation inside the layer.  (Same page and section as the weight format.)
 *   - At batch 1 the layer is bound by weight bandwidth.  (Same page, section "Decode: mover
 *     menos bytes por token".)
 * Readings where the pages are silent: top-k in descending logit order, ties to the lower
 * expert index; routing weights are the softmax of the k selected logits; SwiGLU experts
 * h = silu(x Wg^T) * (x Wu^T), y = h Wd^T; shared-expert gate sigmoid(x . w_sg); eight codes
 * per uint32 with the lowest nibble holding the lowest column.
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers owned by the caller, 16-byte aligned.  The library
 *     allocates no memory and keeps no per-call state; scratch lives in the caller's workspace.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     No call synchronises with the host except moe_read_error_flags.
 *   - Inputs are never written.  Calls are reentrant; two calls may run concurrently only with
 *     distinct workspaces and outputs.
 *   - Errors are returned, never thrown.  Argument checks happen on the host before any launch.
 *     Conditions only the GPU can see set bits in the workspace's error word (sticky until read):
 *       1  a bounded wait timed out (outputs invalid);
 *       2  a value of the grouped-GEMM path left the fp16 operand range: above 65504, or a block
 *          that sits in fp16's subnormal range and loses precision there (a token whose largest
 *          |x| is below 2^-12, a weight row whose largest |w| is below 2^-12, or a token whose h
 *          is below 2^-12 over a 32-row block of F);
 *       4  routing tables inconsistent with the dims;
 *       8  an activation of the decode path (x or h) is not finite.
 *     Calls whose inputs may leave the fp16 operand range (more than eight tokens per call) must
 *     check the word with moe_read_error_flags before trusting y; the decode path (up to eight
 *     tokens) computes in exact integers and fp32 and has no range limit below fp32's.
 *   - T == 0 is a no-op that returns MOE_OK.
 *
 * Dimension limits: 1 <= k <= 32, k <= E <= 1024, d and F multiples of 128, F_shared == 0 (no
 * shared expert) or F_shared == F, T * (k + 1) < 2^31.  (The tensor-core tiles take 128 rows of d
 * and of F; the grouped-GEMM path also needs d % 256 == 0.)
 */
#ifndef MOE_GB300_H_
#define MOE_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, k > E, T < 0, tile_n outside 16..128 or not a multiple of 16 */
  MOE_ERR_UNSUPPORTED = 2, /* dims outside the limits above */
  MOE_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
  MOE_ERR_WORKSPACE = 4,   /* workspace null or smaller than moe_workspace_bytes() */
  MOE_ERR_CUDA = 5         /* a CUDA runtime call or kernel launch failed */
} moe_status;

/* Layer dimensions.  T tokens, hidden size d, E routed experts, top-k, expert FFN width F,
 * shared-expert FFN width F_shared (0 or F).  Quantisation group size is fixed at 64. */
typedef struct moe_dims {
  int32_t T, d, E, k, F, F_shared;
} moe_dims;

/* One 4-bit matrix of R output rows and C input columns (a "qmat"), stacked over a leading
 * expert axis:
 *   codes  uint32 [n, R, C/8]   column c of row r in bits 4*(c%8)..4*(c%8)+3 of word (r, c/8)
 *   scales bf16   [n, R, C/64]  (stored as uint16 bit patterns)
 *   biases bf16   [n, R, C/64]
 *   w[r, c] = q * scales[r, c/64] + biases[r, c/64]. */
typedef struct moe_qmat {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
} moe_qmat;

/* An expert set: gate [n, F, d], up [n, F, d], down [n, d, F].  n = E for the routed experts,
 * n = 1 for the shared expert. */
typedef struct moe_experts {
  moe_qmat gate, up, down;
} moe_experts;

/* Routing tables (all device memory, caller-owned; assignment a = t*k + j routes token t to its
 * j-th expert):
 *   idx       int32 [T, k]   experts in descending logit order, ties to the lower index
 *   w         fp32  [T, k]   softmax of the selected logits
 *   counts    int32 [E]      assignments per expert (histogram)
 *   offsets   int32 [E + 1]  exclusive prefix sum of counts; offsets[E] = T*k
 *   perm      int32 [T*k]    assignment held by slot p; slots sorted by (expert, token)
 *   inv       int32 [T*k]    slot of assignment a
 *   tiles     int32 [moe_max_tiles(), 4]  block map rows (e, first slot, rows, 0): for each
 *             expert with counts[e] > 0 in increasing e, ceil(counts[e]/tile_n) tiles of at
 *             most tile_n consecutive slots; then the shared expert as group e = E over slots
 *             T*k .. T*k+T-1 (token order), in tiles of at most tile_n
 *   num_tiles int32 [1]      number of block-map rows written
 *   tile_n    rows per tile (16..128, a multiple of 16)
 * Every field is bit-exact given the same fp32 logits. */
typedef struct moe_routing {
  int32_t* idx;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  int32_t* tiles;
  int32_t* num_tiles;
  int32_t tile_n;
} moe_routing;

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status s);

/* Upper bound on the number of block-map rows for these dims: floor(T*k/tile_n) + min(E, T*k)
 * + ceil(T/tile_n).  Returns 0 for invalid arguments. */
size_t moe_max_tiles(const moe_dims* dims, int32_t tile_n);

/* Workspace bytes needed by moe_route, moe_expert_forward and moe_layer_forward for these dims
 * (one size serves all three).  Returns 0 for invalid dims.  The first 4 bytes of the workspace are
 * its error word: kernels only ever set bits in it, so it is sticky across calls.  Clear it once
 * after allocating the workspace (moe_clear_error_flags); the rest needs no initialisation. */
size_t moe_workspace_bytes(const moe_dims* dims);

/* Routing: top-k, weights, histogram, exclusive scan, permutation and block map of fp32
 * router logits [T, E], all on the GPU with no host synchronisation ("Perplexity libera Lily...",
 * section "Prefill: pesos comprimidos y enrutamiento en la GPU": histogram, prefix scan, scatter
 * and block map in one command buffer).  Writes every field of *out (out->tile_n is an input).
 * The workspace holds scratch for the tables. */
moe_status moe_route(const moe_dims* dims, const float* logits, const moe_routing* out, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Expert outputs per slot: the fused-dequant grouped GEMM ("Perplexity libera Lily...", section
 * "Prefill: pesos comprimidos y enrutamiento en la GPU": 4-bit weights rebuilt tile by tile on
 * chip, FP32 accumulation).  Needs d % 256 == 0 and routing->tile_n <= 112 (the activation stages
 * hold 112 rows); MOE_ERR_UNSUPPORTED otherwise.
 * y_perm[p] = FFN_{e(p)}(x[token(p)]) for the T*k routed slots of
 * `routing`, followed (when `shared` is non-NULL) by the shared expert's outputs for the T
 * tokens in slots T*k .. T*k+T-1.  x bf16 [T, d]; y_perm fp32 [T*k + T, d] (or [T*k, d] without
 * a shared expert).  GEMM operands are rounded to fp16 (dequantised weights, x, h), products
 * accumulate in fp32. */
moe_status moe_expert_forward(const moe_dims* dims, const uint16_t* x, const moe_routing* routing,
                              const moe_experts* routed, const moe_experts* shared, float* y_perm,
                              void* workspace, size_t workspace_bytes, void* stream);

/* The whole layer: y[t] = sum_j w[t,j] FFN_{idx[t,j]}(x_t) + sigmoid(x_t . w_sg) FFN_shared(x_t)
 * (a router keeping 8 of 256 experts plus a shared expert every token uses: "Perplexity libera
 * Lily...", section "Tres formas de carga en un mismo modelo"; at batch 1 the layer is bound by
 * weight bandwidth: section "Decode: mover menos bytes por token").
 * x bf16 [T, d]; logits fp32 [T, E]; w_shared_gate bf16 [d] (ignored when shared is NULL);
 * y fp32 [T, d].  routing_out may be NULL; when given, its tables are filled as by moe_route.
 * T <= 8 runs the decode path when d <= 2048 and k + 1 <= 32: two launches per call (the fused
 * kernel -- routing in the kernel, exact integer dot products of the 4-bit codes with fixed-point
 * activations, fp32 everywhere else; each expert slot takes the tokens in turn -- and a small
 * kernel that sums its partial outputs in a fixed order).  Otherwise, and for T > 8, the
 * grouped-GEMM path (fp16 tensor-core operands, fp32 accumulation; needs d % 256 == 0, and
 * routing_out->tile_n <= 112 when routing_out is given; MOE_ERR_UNSUPPORTED otherwise); its own
 * block map uses tiles of 112 rows.  The decode path's workspace holds
 * 512 * ceil(d / 512) * (k + 1) * F / 128 floats of partial outputs per token. */
moe_status moe_layer_forward(const moe_dims* dims, const uint16_t* x, const float* logits,
                             const moe_experts* routed, const moe_experts* shared, const uint16_t* w_shared_gate,
                             float* y, const moe_routing* routing_out, void* workspace, size_t workspace_bytes,
                             void* stream);

/* Option bits of moe_layer_forward_opts. */
#define MOE_OPT_BF16_OPERANDS 1u

/* moe_layer_forward with options; options == 0 is moe_layer_forward.
 * MOE_OPT_BF16_OPERANDS: the grouped-GEMM path takes bf16 tensor-core operands instead of fp16
 * (the MMA rate is the same): w = q * s + b rounded once to bf16, x as given, h and the expert
 * outputs rounded to bf16; accumulation and the weighted combine stay fp32.  bf16 has fp32's
 * exponent range, so this path raises none of fp16's range flags (error bit 2), at about twice
 * the rounding error of fp16 operands (8 significant bits against 11).  Calls that run the decode
 * path (T <= 8) are unaffected: it has no tensor-core operands.
 * Returns MOE_ERR_INVALID_ARG for an unknown option bit; otherwise as moe_layer_forward. */
moe_status moe_layer_forward_opts(const moe_dims* dims, const uint16_t* x, const float* logits,
                                  const moe_experts* routed, const moe_experts* shared,
                                  const uint16_t* w_shared_gate, float* y, const moe_routing* routing_out,
                                  void* workspace, size_t workspace_bytes, void* stream, uint32_t options);

/* moe_layer_forward with the input and output in host memory: copies x_host (bf16 [T, d]) and
 * logits_host (fp32 [T, E]) to a staging area at the end of the workspace, runs the layer, and
 * copies y (fp32 [T, d]) back to y_host -- the copies and the kernels queued on `stream` in that
 * order; the call returns before they finish, so synchronise the stream before reading y_host.
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to be
 * asynchronous; pageable buffers work but the runtime may stage them synchronously.  The
 * workspace must hold moe_workspace_bytes_host(dims) bytes (the first moe_workspace_bytes(dims)
 * of it serve as the layer's workspace, error word included).  No routing tables are returned.
 * With T <= 8 on the fused decode kernel, all three buffers page-locked, mapped into the
 * device's address space (unified addressing) and 16-byte aligned, and y_host allocated by
 * cudaHostAlloc / cudaMallocHost (registered memory may be read-only for the device), no copies
 * are queued: a one-CTA kernel reads x and logits from host memory into the workspace and the
 * decode kernel writes y into host memory itself. */
size_t moe_workspace_bytes_host(const moe_dims* dims);
moe_status moe_layer_forward_host(const moe_dims* dims, const uint16_t* x_host, const float* logits_host,
                                  const moe_experts* routed, const moe_experts* shared,
                                  const uint16_t* w_shared_gate, float* y_host, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Option bits of moe_layer_forward_host_opts. */
#define MOE_OPT_HOST_INPUTS_READY 1u

/* moe_layer_forward_host with options; options == 0 is moe_layer_forward_host.
 * MOE_OPT_HOST_INPUTS_READY: x_host and logits_host hold their final values when the call is made
 * (no work queued on the stream before the call writes them).  On the staging-kernel path (T <= 8,
 * page-locked mapped buffers) the kernel then reads them before the preceding work on the stream
 * has finished, so their latency across the CPU-GPU link overlaps that work; the workspace is
 * still written only after it.  Results are identical to moe_layer_forward_host's; the copy path
 * is unaffected.  Returns MOE_ERR_INVALID_ARG for an unknown option bit; otherwise as
 * moe_layer_forward_host. */
moe_status moe_layer_forward_host_opts(const moe_dims* dims, const uint16_t* x_host, const float* logits_host,
                                       const moe_experts* routed, const moe_experts* shared,
                                       const uint16_t* w_shared_gate, float* y_host, void* workspace,
                                       size_t workspace_bytes, void* stream, uint32_t options);

/* Pre-norm block of a stack of MoE layers (the step between two layers, not part of the layer; an
 * addition for the 40-layer stack workload -- the pages' router scores 256 experts from the
 * normalised hidden state, a linear router being the reading):
 * when y_prev is non-NULL, x_resid += y_prev (written back); then h = RMSNorm(x_resid) * gamma
 * = x / sqrt(mean(x^2) + eps) * gamma rounded to bf16, and router logits = h W_r^T with bf16
 * operands and fp32 accumulation on the tensor cores.  x_resid fp32 [T, d] (in/out); y_prev fp32
 * [T, d] or NULL; gamma bf16 [d]; w_router bf16 [E, d]; h_out bf16 [T, d]; logits_out fp32 [T, E].
 * The workspace is only used for its error word (any size >= 4 bytes). */
moe_status moe_rmsnorm_router(const moe_dims* dims, float* x_resid, const float* y_prev, const uint16_t* gamma,
                              const uint16_t* w_router, float eps, uint16_t* h_out, float* logits_out,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Decode (T == 1) layer forward that allocates nothing and takes no workspace.  The pages have
 * no counterpart: this entry point exists for callers that cannot allocate device memory when
 * they run the layer -- an engine whose memory planner hands out all of HBM once at start-up and
 * forbids later cudaMalloc calls, a latency-critical decode loop that must never enter
 * cudaMalloc/cudaFree (they may synchronise the device), or a host program that holds only
 * pointers to weights, inputs and outputs.  Arguments and results are those of
 * moe_layer_forward with T == 1 (same kernels), and dims outside moe_layer_forward's rules return
 * its status codes.
 *   - Scratch: a library-owned device array of 512 KB (+256 B) that every GPU which loads the
 *     library keeps until the process exits; it bounds the decode path's partial outputs,
 *     512 * ceil(d / 512) * (k + 1) * F / 128 <= 131072 floats (the decode workload, d 2048,
 *     k 8, F 512, needs 73728).  Larger dims, T > 1, or dims the decode path does not take return
 *     MOE_ERR_UNSUPPORTED; T == 0 returns MOE_OK.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 *     that device current; make that first call before any stream capture.
 *   - All calls share the array: calls whose work overlaps on the GPU (different streams, or
 *     different host threads) race.  Serialise them, e.g. on one stream.
 *   - Device-side error bits (a timed-out wait) land in the shared array and are not reported;
 *     use moe_layer_forward with a workspace to read them. */
moe_status moe_layer_forward_decode_noalloc(const moe_dims* dims, const uint16_t* x, const float* logits,
                                            const moe_experts* routed, const moe_experts* shared,
                                            const uint16_t* w_shared_gate, float* y, void* stream);

/* Enqueues the clearing of the workspace's error word on `stream` (no host synchronisation). */
moe_status moe_clear_error_flags(void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises `stream`, copies the workspace's error word to *flags, then clears it.  Bits (see
 * the conventions above): 1 = a bounded device wait timed out, 2 = a value left the fp16 operand
 * range of the grouped-GEMM path, 4 = routing tables inconsistent with the dims, 8 = a decode-path
 * activation is not finite.  0 means every call since the last clear completed cleanly. */
moe_status moe_read_error_flags(void* workspace, size_t workspace_bytes, uint32_t* flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H_ */
