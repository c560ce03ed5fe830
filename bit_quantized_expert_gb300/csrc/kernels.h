// Internal launch interface between the C ABI (api.cu) and the kernels.  Plain structs of
// device pointers and sizes; no allocation happens behind any of these functions.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// ---------------------------------------------------------------- routing (route.cu)
struct RouteArgs {
  const float* logits;   // [T, E]
  int T, E, k, d;
  int32_t* idx;          // [T, k]
  float* w;              // [T, k]
  const uint16_t* x;     // bf16 [T, d] or null (no fp16 copy / gate)
  const uint16_t* w_sg;  // bf16 [d] or null
  float* gs;             // [T] shared gate, or null
  uint32_t* err;
  int bf16;              // the GEMM takes x as bf16: no fp16 range check of x
};
cudaError_t launch_topk(const RouteArgs& a, cudaStream_t st);

struct TablesArgs {
  const int32_t* idx;
  int T, E, k, tile_n, has_shared;
  int32_t *counts, *offsets, *perm, *inv, *tiles, *num_tiles;
  int32_t* chunk;          // scratch [ceil(T/32)][E]: per-chunk counts, then per-chunk bases
  uint32_t* err;
  int32_t* sched;          // or null: also write the grouped GEMM's walk order (launch_schedule's)
};
size_t tables_scratch_bytes(int T, int E);

// Order in which the grouped GEMM walks the block map: full tiles first (in block-map order), then
// the partial tiles by decreasing width (ties in block-map order), so that the round-robin split
// of units over the persistent CTAs gives every CTA a similar amount of work.
struct ScheduleArgs {
  const int32_t* tiles;     // block map rows (e, row0, rows, 0)
  const int32_t* num_tiles;
  int tile_n;
  int32_t* sched;           // [>= num_tiles] tile index of the u-th scheduled tile
  uint32_t* err;
};
cudaError_t launch_schedule(const ScheduleArgs& a, cudaStream_t st);
// One CTA whose waits on an mbarrier that nothing completes give up after `limit` cycles (route.cu).
cudaError_t launch_wait_probe(uint32_t* err, long long limit, cudaStream_t st);
cudaError_t launch_tables(const TablesArgs& a, cudaStream_t st);

// ---------------------------------------------------------------- grouped GEMM (gemm.cu)
struct QPtr {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
};

// Tensor maps of one launch: packed codes of each operand matrix for the routed and the
// shared expert set, and (down projection) the h operand.
// Widest block-map tile the grouped GEMM takes (its activation stages hold this many rows).
constexpr int kGemmMaxTileN = 112;

struct GemmMaps {
  CUtensorMap codes[2][2];   // [matrix][0 = routed, 1 = shared]
  CUtensorMap h;             // down projection: h [slots, F] fp16, 112-row boxes
  CUtensorMap x;             // gate/up projection: x rows in slot order [slots, d] fp16, 112-row boxes
  CUtensorMap h16;           // the same two tensors with 16-row boxes (tiles narrower than 128)
  CUtensorMap x16;
};

struct GemmArgs {
  const int32_t* tiles;      // block map rows (e, row0, rows, 0)
  const int32_t* num_tiles;
  const int32_t* sched;      // walk order of the block map (launch_schedule)
  const int32_t* perm;       // slot -> assignment (gate/up gathers x rows)
  QPtr mat[2][2];            // [matrix][routed/shared]: scales and biases read by the dequant warps
  int T, k, E, d, F;
  uint16_t* h;               // gate/up output: 16-bit [slots, F], operand chunk order
  float* y_perm;             // down output: fp32 [slots, d] (when y16 is null)
  uint16_t* y16;             // down output: 16-bit [slots, d], or null
  uint32_t* err;
  int bf16;                  // operands (weights, x, h) and y16 in bf16 rather than fp16
};
size_t gemm_smem_bytes(int mode);
cudaError_t launch_gemm(int mode, const GemmMaps& maps, const GemmArgs& a, int grid, cudaStream_t st);

struct CombineArgs {
  const float* y_perm;    // [T*k + T, d] fp32, or null
  const uint16_t* y16;    // [T*k + T, d] fp16 (used when non-null)
  const int32_t* inv;     // [T*k]
  const float* w;         // [T, k]
  const float* gs;        // [T] or null (no shared expert)
  int T, k, d;
  float* y;               // [T, d]
  int bf16;               // y16 holds bf16 rather than fp16
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st);

struct PermuteArgs {
  const uint16_t* x;      // bf16 [T, d]
  const int32_t* perm;    // [T*k] slot -> assignment t*k + j
  int T, k, d, slots;     // slots = T*k (+ T with a shared expert)
  uint16_t* xperm;        // fp16 (bf16 when bf16 is set) [slots, d] operand chunk order: row s = x[token(s)]
  uint32_t* err;
  int bf16;
};
cudaError_t launch_permute_x(const PermuteArgs& a, cudaStream_t st);

// ---------------------------------------------------------------- decode T <= 8 (decode.cu)
struct DecodeArgs {
  const uint16_t* x;       // bf16 [T][d]
  const float* logits;     // [T][E]
  QPtr gate[2], up[2], down[2];   // [0] routed (stacked over E), [1] shared (may be null)
  const uint16_t* w_sg;    // bf16 [d] or null
  int d, E, k, F, has_shared;
  int T;                   // tokens, 1 .. kDecodeMaxTokens (0 reads as 1)
  float* part;             // scratch: fp32 [T][decode_scratch_floats] partial outputs per row slice
  float* y;                // fp32 [T][d]
  uint32_t* err;
};
// Tensor maps of a decode launch: the down-projection codes of the routed [0] and shared [1]
// expert sets as 2-D uint32 tensors {F/8 words, n*d rows}, box 16 words x decode_box_rows rows.
struct DecodeMaps {
  CUtensorMap down[2];
};
int decode_box_rows(int d, int F);
bool decode_supported(int d, int E, int k, int F);
constexpr int kDecodeMaxTokens = 8;   // tokens one decode launch can take (one routing warp each)
constexpr int kDecodeLayerMaxT = 8;    // layer calls of up to this many tokens take the decode kernel
size_t decode_scratch_floats(int d, int k, int F);   // floats of DecodeArgs::part per token
// The decode launch's second kernel: y from the partials (DecodeArgs::part, ::y; k1 expert slots).
struct ReduceArgs {
  const float* part;
  float* y;
  int d, F, k1;
};
cudaError_t launch_decode(const DecodeMaps& maps, const DecodeArgs& a, cudaStream_t st, bool pdl);
// Loads-only replica of the decode kernel's weight copies for one token whose k experts are given
// (a measurement aid; see decode_stream_kernel).
struct StreamArgs {
  QPtr gate[2], up[2], down[2];
  const int32_t* idx;      // [k] experts of the token, in slot order
  int d, E, k, F, has_shared;
  uint32_t* err;
};
cudaError_t launch_decode_stream(const DecodeMaps& maps, const StreamArgs& a, cudaStream_t st);
// Encodes DecodeMaps::down[i] for n stacked [d, F] down matrices (api.cu); false on failure.
// cuTensorMapEncodeTiled, fetched once from the driver (null if the driver lacks it).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();
bool encode_decode_down(CUtensorMap* m, const uint32_t* codes, int n, int d, int F);

// Workspace head shared by the C ABI and the allocation-free entry point: the error word at 0.
constexpr size_t kWsHeadBytes = 256;

// Host-side dims rules of every layer call (api.cu); MOE_OK = 0.
int check_layer_dims(int T, int d, int E, int k, int F, int F_shared);

// One CTA copies a token's x (x_bytes, a multiple of 16) and logits (lg_bytes, a multiple of 4)
// from page-locked, mapped host memory (16-byte aligned) into device buffers, once, so that the
// decode kernel's many readers hit device memory; launched with programmatic serialisation, it
// waits for the previous kernel on the stream before writing.
struct StageArgs {
  const uint4* x_src;
  uint4* x_dst;
  const float* lg_src;
  float* lg_dst;
  int x_units;   // 16-byte units of x
  int lg_n;      // floats of logits
  int early;     // the first round of host reads goes out before the dependency wait
};
cudaError_t launch_stage_in(const StageArgs& a, cudaStream_t st);

// ---------------------------------------------------------------- pre-norm block (router.cu)
struct NormArgs {
  float* x;               // fp32 [T, d] residual stream (updated when y_prev is given)
  const float* y_prev;    // fp32 [T, d] or null
  const uint16_t* gamma;  // bf16 [d]
  int T, d;
  float eps;
  uint16_t* h;            // bf16 [T, d]
};
cudaError_t launch_rmsnorm(const NormArgs& a, cudaStream_t st);

struct RouterMaps {
  CUtensorMap w;          // W_r bf16 [E, d], box 64 x 128, 128-byte swizzle
  CUtensorMap h;          // h bf16 [T, d], box 64 x 128, 128-byte swizzle
};
struct RouterArgs {
  int T, d, E;
  float* logits;          // fp32 [T, E]
  uint32_t* err;
};
cudaError_t launch_router(const RouterMaps& maps, const RouterArgs& a, cudaStream_t st);

}  // namespace moe
