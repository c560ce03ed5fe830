// C ABI of the MoE layer (declarations and contracts in include/moe.h).  Host-side argument
// checks, workspace layout, TMA descriptor encoding and launch order; no allocation and no
// host synchronisation except moe_read_error_flags.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "../../include/moe.h"
#include "../../include/moe_probe.h"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kTileN = kGemmMaxTileN;   // block-map tile of the layer call (token rows per MMA tile)

struct Layout {
  size_t err, xperm, gs, idx, w, counts, offsets, perm, inv, tiles, num_tiles, sched, chunk, h, yperm, hdec, total;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// The first kWsHeadBytes of a workspace: the error word at 0 (zero before the first call).

size_t max_tiles_of(long long T, long long k, long long E, long long tile_n, bool shared) {
  return (size_t)(T * k / tile_n + std::min(E, T * k) + (shared ? (T + tile_n - 1) / tile_n : 0));
}

Layout layout_of(const moe_dims& d) {
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  const size_t T = d.T, k = d.k, E = d.E, D = d.d, F = d.F;
  const bool sh = d.F_shared > 0;
  const size_t slots = T * k + (sh ? T : 0);
  L.err = take(kWsHeadBytes);
  L.xperm = take(slots * D * 2);
  L.gs = take(T * 4);
  L.idx = take(T * k * 4);
  L.w = take(T * k * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm = take(T * k * 4);
  L.inv = take(T * k * 4);
  L.tiles = take(max_tiles_of(d.T, d.k, d.E, kTileN, sh) * 16);
  L.num_tiles = take(16);
  L.sched = take(max_tiles_of(d.T, d.k, d.E, 16, sh) * 4);   // GEMM walk order (any tile_n >= 16)
  L.chunk = take(tables_scratch_bytes((int)T, (int)E));   // routing-table scratch
  L.h = take(slots * F * 2);
  L.yperm = take(slots * D * 2);   // fp16 expert outputs of the layer path
  L.hdec = take(T >= 1 && T <= (size_t)kDecodeLayerMaxT ? T * decode_scratch_floats((int)D, (int)k, (int)F) * 4 : 0);   // decode partials
  L.total = o;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int check_layer_dims(int T, int d, int E, int k, int F, int F_shared) {
  if (T < 0 || k < 1 || E < 1 || k > E || d < 1 || F < 1 || F_shared < 0) return MOE_ERR_INVALID_ARG;
  if (k > 32 || E > 1024) return MOE_ERR_UNSUPPORTED;
  if (d % 128 != 0 || F % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (F_shared != 0 && F_shared != F) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * (k + 1) >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if ((long long)d * F >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

namespace {

moe_status check_dims(const moe_dims* d) {
  if (d == nullptr) return MOE_ERR_INVALID_ARG;
  return static_cast<moe_status>(check_layer_dims(d->T, d->d, d->E, d->k, d->F, d->F_shared));
}

moe_status check_qmat(const moe_qmat& q) {
  if (!q.codes || !q.scales || !q.biases) return MOE_ERR_INVALID_ARG;
  if (!aligned16(q.codes) || !aligned16(q.scales) || !aligned16(q.biases)) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

moe_status check_experts(const moe_experts* x) {
  if (x == nullptr) return MOE_ERR_INVALID_ARG;
  moe_status s;
  if ((s = check_qmat(x->gate)) != MOE_OK) return s;
  if ((s = check_qmat(x->up)) != MOE_OK) return s;
  return check_qmat(x->down);
}

moe_status check_ptr(const void* p) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  return aligned16(p) ? MOE_OK : MOE_ERR_MISALIGNED;
}

moe_status check_routing(const moe_routing* r) {
  if (r == nullptr) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {r->idx, r->w, r->counts, r->offsets, r->perm, r->inv, r->tiles, r->num_tiles};
  for (const void* p : ps) {
    moe_status s = check_ptr(p);
    if (s != MOE_OK) return s;
  }
  if (r->tile_n < 16 || r->tile_n > 128 || r->tile_n % 16 != 0) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

// ---------------------------------------------------------------- TMA descriptors
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

namespace {

// Packed codes of n stacked [R, C] matrices as a 3-D uint32 tensor {C/8, R, n}; box 16 x 128 x 1
// (128 codes of 128 rows = two quantisation groups of a tile, 64 bytes per row) in the 64-byte
// swizzle.
bool encode_codes(CUtensorMap* m, const uint32_t* codes, int n, int R, int C) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)(C / 8), (cuuint64_t)R, (cuuint64_t)n};
  const cuuint64_t strides[2] = {(cuuint64_t)(C / 8) * 4, (cuuint64_t)R * (C / 8) * 4};
  const cuuint32_t box[3] = {16, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(codes), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major fp16 matrix [rows, cols] (h, or x in slot order) with a box of 64 columns x box_rows
// rows in the 128-byte swizzle (the MMA operand layout).
bool encode_f16_rows(CUtensorMap* m, const uint16_t* p, long long rows, int cols, int box_rows) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(p), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Down-projection codes of n stacked [d, F] matrices as a 2-D uint32 tensor {F/8, n*d}, box of 16
// words (the 128 columns of one decode cluster) by decode_box_rows rows, no swizzle.
bool encode_decode_down(CUtensorMap* m, const uint32_t* codes, int n, int d, int F) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(F / 8), (cuuint64_t)n * (cuuint64_t)d};
  const cuuint64_t strides[1] = {(cuuint64_t)(F / 8) * 4};
  const cuuint32_t box[2] = {16, (cuuint32_t)decode_box_rows(d, F)};
  const cuuint32_t es[2] = {1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(codes), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Row-major bf16 matrix [rows, cols] with a 64 x 128 box in the 128-byte swizzle.
bool encode_bf16_rows(CUtensorMap* m, const uint16_t* p, long long rows, int cols) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int counts[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 0 || dev >= 64) return 1;
  if (counts[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    counts[dev] = n > 0 ? n : 1;
  }
  return counts[dev];
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

struct RoutingPtrs {
  int32_t *idx, *counts, *offsets, *perm, *inv, *tiles, *num_tiles;
  float* w;
  int tile_n;
};

RoutingPtrs internal_routing(void* ws, const Layout& L) {
  return {at<int32_t>(ws, L.idx),   at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets),
          at<int32_t>(ws, L.perm),  at<int32_t>(ws, L.inv),    at<int32_t>(ws, L.tiles),
          at<int32_t>(ws, L.num_tiles), at<float>(ws, L.w),    kTileN};
}

RoutingPtrs caller_routing(const moe_routing* r) {
  return {r->idx, r->counts, r->offsets, r->perm, r->inv, r->tiles, r->num_tiles, r->w, r->tile_n};
}

cudaError_t run_routing(const moe_dims& d, const float* logits, const RoutingPtrs& R, const uint16_t* x,
                        const uint16_t* w_sg, float* gs, int32_t* chunk, uint32_t* err, cudaStream_t st,
                        int32_t* sched = nullptr, bool bf = false) {
  RouteArgs ra{logits, d.T, d.E, d.k, d.d, R.idx, R.w, x, w_sg, gs, err, bf ? 1 : 0};
  cudaError_t e = launch_topk(ra, st);
  if (e != cudaSuccess) return e;
  TablesArgs ta{R.idx, d.T, d.E, d.k, R.tile_n, d.F_shared > 0 ? 1 : 0, R.counts, R.offsets, R.perm, R.inv,
                R.tiles, R.num_tiles, chunk, err, sched};
  return launch_tables(ta, st);
}

QPtr qptr(const moe_qmat& q) { return QPtr{q.codes, q.scales, q.biases}; }

// x rows in slot order (fp16, or bf16 when bf is set), gate/up GEMM (h), then down GEMM (expert
// outputs: fp32 y_perm, or 16-bit y16 when y16 is non-null) over the block map in R.
moe_status run_experts(const moe_dims& d, const RoutingPtrs& R, const moe_experts* routed, const moe_experts* shared,
                       const uint16_t* x, uint16_t* xperm, uint16_t* h, float* y_perm, uint16_t* y16,
                       int32_t* sched, uint32_t* err, cudaStream_t st, bool sched_ready = false, bool bf = false) {
  // the down GEMM pairs 128-row blocks of the output dimension; activation stages hold 112 rows
  if (d.d % 256 != 0 || R.tile_n > kGemmMaxTileN) return MOE_ERR_UNSUPPORTED;
  const bool sh = shared != nullptr && d.F_shared > 0;
  const long long slots = (long long)d.T * d.k + (sh ? d.T : 0);
  const moe_experts* s_or_r = sh ? shared : routed;
  const int ns = sh ? 1 : d.E;

  GemmMaps m0{}, m1{};
  bool ok = encode_codes(&m0.codes[0][0], routed->gate.codes, d.E, d.F, d.d) &&
            encode_codes(&m0.codes[0][1], s_or_r->gate.codes, ns, d.F, d.d) &&
            encode_codes(&m0.codes[1][0], routed->up.codes, d.E, d.F, d.d) &&
            encode_codes(&m0.codes[1][1], s_or_r->up.codes, ns, d.F, d.d) &&
            encode_codes(&m1.codes[0][0], routed->down.codes, d.E, d.d, d.F) &&
            encode_codes(&m1.codes[0][1], s_or_r->down.codes, ns, d.d, d.F) &&
            encode_f16_rows(&m1.h, h, slots, d.F, kGemmMaxTileN) &&
            encode_f16_rows(&m0.x, xperm, slots, d.d, kGemmMaxTileN) &&
            encode_f16_rows(&m1.h16, h, slots, d.F, 16) && encode_f16_rows(&m0.x16, xperm, slots, d.d, 16);
  if (!ok) return MOE_ERR_CUDA;
  PermuteArgs pa{x, R.perm, d.T, d.k, d.d, (int)slots, xperm, err, bf ? 1 : 0};
  if (launch_permute_x(pa, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (!sched_ready) {   // the layer path's routing already wrote it
    ScheduleArgs sa{R.tiles, R.num_tiles, R.tile_n, sched, err};
    if (launch_schedule(sa, st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  m0.h = m1.h;
  m0.h16 = m1.h16;
  m1.codes[1][0] = m1.codes[0][0];
  m1.codes[1][1] = m1.codes[0][1];

  const size_t maxt = max_tiles_of(d.T, d.k, d.E, R.tile_n, sh);
  GemmArgs a{};
  a.tiles = R.tiles;
  a.num_tiles = R.num_tiles;
  a.sched = sched;
  a.perm = R.perm;
  a.T = d.T;
  a.k = d.k;
  a.E = d.E;
  a.d = d.d;
  a.F = d.F;
  a.h = h;
  a.y_perm = y_perm;
  a.y16 = y16;
  a.err = err;
  a.bf16 = bf ? 1 : 0;
  a.mat[0][0] = qptr(routed->gate);
  a.mat[0][1] = qptr(s_or_r->gate);
  a.mat[1][0] = qptr(routed->up);
  a.mat[1][1] = qptr(s_or_r->up);
  const int sms = sm_count();
  const int g0 = (int)std::max<size_t>(1, std::min<size_t>((size_t)sms, maxt * (d.F / 128)));
  cudaError_t e = launch_gemm(0, m0, a, g0, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  a.mat[0][0] = qptr(routed->down);
  a.mat[0][1] = qptr(s_or_r->down);
  a.mat[1][0] = a.mat[0][0];
  a.mat[1][1] = a.mat[0][1];
  const int g1 = (int)std::max<size_t>(1, std::min<size_t>((size_t)sms, maxt * (d.d / 256)));
  e = launch_gemm(1, m1, a, g1, st);
  return cuda_status(e);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null pointer or argument out of range";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: dimensions outside the supported limits";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED: a pointer is not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing or too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or kernel launch failed";
  }
  return "unknown moe_status";
}

size_t moe_max_tiles(const moe_dims* dims, int32_t tile_n) {
  if (check_dims(dims) != MOE_OK || tile_n < 16 || tile_n > 128 || tile_n % 16 != 0) return 0;
  return max_tiles_of(dims->T, dims->k, dims->E, tile_n, dims->F_shared > 0);
}

size_t moe_workspace_bytes(const moe_dims* dims) {
  if (check_dims(dims) != MOE_OK) return 0;
  return layout_of(*dims).total;
}

moe_status moe_route(const moe_dims* dims, const float* logits, const moe_routing* out, void* workspace,
                     size_t workspace_bytes, void* stream) {
  moe_status s = check_dims(dims);
  if (s != MOE_OK) return s;
  if ((s = check_routing(out)) != MOE_OK) return s;
  if (dims->T == 0) return MOE_OK;
  if ((s = check_ptr(logits)) != MOE_OK) return s;
  if ((s = check_ptr(workspace)) != MOE_OK) return s == MOE_ERR_INVALID_ARG ? MOE_ERR_WORKSPACE : s;
  const Layout L = layout_of(*dims);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = at<uint32_t>(workspace, L.err);
  return cuda_status(run_routing(*dims, logits, caller_routing(out), nullptr, nullptr, nullptr,
                                 at<int32_t>(workspace, L.chunk), err, st));
}

moe_status moe_expert_forward(const moe_dims* dims, const uint16_t* x, const moe_routing* routing,
                              const moe_experts* routed, const moe_experts* shared, float* y_perm, void* workspace,
                              size_t workspace_bytes, void* stream) {
  moe_status s = check_dims(dims);
  if (s != MOE_OK) return s;
  if ((s = check_routing(routing)) != MOE_OK) return s;
  if ((s = check_experts(routed)) != MOE_OK) return s;
  if (shared != nullptr && (s = check_experts(shared)) != MOE_OK) return s;
  if (shared != nullptr && dims->F_shared == 0) return MOE_ERR_INVALID_ARG;
  if (shared == nullptr && dims->F_shared != 0) return MOE_ERR_INVALID_ARG;
  if (dims->T == 0) return MOE_OK;
  if (dims->d % 256 != 0) return MOE_ERR_UNSUPPORTED;   // grouped-GEMM path
  if ((s = check_ptr(x)) != MOE_OK) return s;
  if ((s = check_ptr(y_perm)) != MOE_OK) return s;
  if ((s = check_ptr(workspace)) != MOE_OK) return s == MOE_ERR_INVALID_ARG ? MOE_ERR_WORKSPACE : s;
  const Layout L = layout_of(*dims);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = at<uint32_t>(workspace, L.err);
  return run_experts(*dims, caller_routing(routing), routed, shared, x, at<uint16_t>(workspace, L.xperm),
                     at<uint16_t>(workspace, L.h), y_perm, nullptr, at<int32_t>(workspace, L.sched), err, st);
}

moe_status moe_layer_forward(const moe_dims* dims, const uint16_t* x, const float* logits, const moe_experts* routed,
                             const moe_experts* shared, const uint16_t* w_shared_gate, float* y,
                             const moe_routing* routing_out, void* workspace, size_t workspace_bytes, void* stream) {
  return moe_layer_forward_opts(dims, x, logits, routed, shared, w_shared_gate, y, routing_out, workspace,
                                workspace_bytes, stream, 0u);
}

moe_status moe_layer_forward_opts(const moe_dims* dims, const uint16_t* x, const float* logits,
                                  const moe_experts* routed, const moe_experts* shared,
                                  const uint16_t* w_shared_gate, float* y, const moe_routing* routing_out,
                                  void* workspace, size_t workspace_bytes, void* stream, uint32_t options) {
  if (options & ~(uint32_t)MOE_OPT_BF16_OPERANDS) return MOE_ERR_INVALID_ARG;
  const bool bf = (options & MOE_OPT_BF16_OPERANDS) != 0;
  moe_status s = check_dims(dims);
  if (s != MOE_OK) return s;
  if ((s = check_experts(routed)) != MOE_OK) return s;
  if (shared != nullptr && (s = check_experts(shared)) != MOE_OK) return s;
  if (shared != nullptr && dims->F_shared == 0) return MOE_ERR_INVALID_ARG;
  if (shared == nullptr && dims->F_shared != 0) return MOE_ERR_INVALID_ARG;
  if (routing_out != nullptr && (s = check_routing(routing_out)) != MOE_OK) return s;
  if (dims->T == 0) return MOE_OK;
  if ((s = check_ptr(x)) != MOE_OK) return s;
  if ((s = check_ptr(logits)) != MOE_OK) return s;
  if ((s = check_ptr(y)) != MOE_OK) return s;
  if (shared != nullptr && (s = check_ptr(w_shared_gate)) != MOE_OK) return s;
  if ((s = check_ptr(workspace)) != MOE_OK) return s == MOE_ERR_INVALID_ARG ? MOE_ERR_WORKSPACE : s;
  const Layout L = layout_of(*dims);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = at<uint32_t>(workspace, L.err);
  const bool sh = shared != nullptr;
  const moe_dims& d = *dims;

  // One to kDecodeLayerMaxT tokens: the fused decode kernel, one launch for all of them (each CTA
  // takes its expert slot of every token in turn; per-token arrival counters for the combine).
  if (d.T <= kDecodeLayerMaxT && decode_supported(d.d, d.E, d.k, d.F)) {
    DecodeArgs da{};
    da.x = x;
    da.logits = logits;
    da.gate[0] = qptr(routed->gate);
    da.up[0] = qptr(routed->up);
    da.down[0] = qptr(routed->down);
    if (sh) {
      da.gate[1] = qptr(shared->gate);
      da.up[1] = qptr(shared->up);
      da.down[1] = qptr(shared->down);
    }
    da.w_sg = sh ? w_shared_gate : nullptr;
    da.d = d.d;
    da.E = d.E;
    da.k = d.k;
    da.F = d.F;
    da.has_shared = sh ? 1 : 0;
    da.part = at<float>(workspace, L.hdec);
    da.y = y;
    da.err = err;
    da.T = d.T;
    DecodeMaps dmaps{};
    if (!encode_decode_down(&dmaps.down[0], routed->down.codes, d.E, d.d, d.F) ||
        !encode_decode_down(&dmaps.down[1], sh ? shared->down.codes : routed->down.codes, sh ? 1 : d.E, d.d, d.F))
      return MOE_ERR_CUDA;
    if (launch_decode(dmaps, da, st, true) != cudaSuccess) return MOE_ERR_CUDA;
    if (routing_out != nullptr)
      return cuda_status(run_routing(d, logits, caller_routing(routing_out), nullptr, nullptr, nullptr,
                                     at<int32_t>(workspace, L.chunk), err, st));
    return MOE_OK;
  }

  if (d.d % 256 != 0) return MOE_ERR_UNSUPPORTED;   // grouped-GEMM path
  const RoutingPtrs R = routing_out ? caller_routing(routing_out) : internal_routing(workspace, L);
  uint16_t* xperm = at<uint16_t>(workspace, L.xperm);
  float* gs = sh ? at<float>(workspace, L.gs) : nullptr;
  cudaError_t e = run_routing(d, logits, R, x, sh ? w_shared_gate : nullptr, gs, at<int32_t>(workspace, L.chunk), err, st,
                              at<int32_t>(workspace, L.sched), bf);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  uint16_t* y16 = at<uint16_t>(workspace, L.yperm);
  s = run_experts(d, R, routed, sh ? shared : nullptr, x, xperm, at<uint16_t>(workspace, L.h), nullptr, y16,
                  at<int32_t>(workspace, L.sched), err, st, true, bf);
  if (s != MOE_OK) return s;
  CombineArgs cb{nullptr, y16, R.inv, R.w, gs, d.T, d.k, d.d, y, bf ? 1 : 0};
  return cuda_status(launch_combine(cb, st));
}

// Device address of page-locked host memory registered with CUDA and mapped into the device's
// address space, 16-byte aligned; null for anything else (pageable memory included).
static void* mapped_host(const void* p) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();   // clear the sticky-free error of an unknown pointer
    return nullptr;
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return nullptr;
  if ((reinterpret_cast<uintptr_t>(attr.devicePointer) & 15u) != 0) return nullptr;
  return attr.devicePointer;
}

// True for memory from cudaHostAlloc / cudaMallocHost, which the device may always write.  Memory
// registered with cudaHostRegister can be read-only for the device (cudaHostRegisterReadOnly) and
// its flags cannot be queried here, so an output buffer of that kind takes the copy instead.
static bool host_alloc_writable(const void* p) {
  unsigned int flags = 0;
  if (cudaHostGetFlags(&flags, const_cast<void*>(p)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}

static size_t host_staging_at(const moe_dims& d, size_t* x_off, size_t* lg_off, size_t* y_off) {
  const size_t base = (layout_of(d).total + 255) & ~(size_t)255;
  const size_t xb = ((size_t)d.T * d.d * 2 + 255) & ~(size_t)255;
  const size_t lb = ((size_t)d.T * d.E * 4 + 255) & ~(size_t)255;
  const size_t yb = ((size_t)d.T * d.d * 4 + 255) & ~(size_t)255;
  *x_off = base;
  *lg_off = base + xb;
  *y_off = base + xb + lb;
  return base + xb + lb + yb;
}

size_t moe_workspace_bytes_host(const moe_dims* dims) {
  if (check_dims(dims) != MOE_OK) return 0;
  size_t xo, lo, yo;
  return host_staging_at(*dims, &xo, &lo, &yo);
}

moe_status moe_layer_forward_host(const moe_dims* dims, const uint16_t* x_host, const float* logits_host,
                                  const moe_experts* routed, const moe_experts* shared,
                                  const uint16_t* w_shared_gate, float* y_host, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return moe_layer_forward_host_opts(dims, x_host, logits_host, routed, shared, w_shared_gate, y_host, workspace,
                                     workspace_bytes, stream, 0u);
}

moe_status moe_layer_forward_host_opts(const moe_dims* dims, const uint16_t* x_host, const float* logits_host,
                                       const moe_experts* routed, const moe_experts* shared,
                                       const uint16_t* w_shared_gate, float* y_host, void* workspace,
                                       size_t workspace_bytes, void* stream, uint32_t options) {
  if (options & ~(uint32_t)MOE_OPT_HOST_INPUTS_READY) return MOE_ERR_INVALID_ARG;
  moe_status s = check_dims(dims);
  if (s != MOE_OK) return s;
  if (dims->T == 0) return MOE_OK;
  if (x_host == nullptr || logits_host == nullptr || y_host == nullptr) return MOE_ERR_INVALID_ARG;
  if ((s = check_ptr(workspace)) != MOE_OK) return s == MOE_ERR_INVALID_ARG ? MOE_ERR_WORKSPACE : s;
  size_t xo, lo, yo;
  if (workspace_bytes < host_staging_at(*dims, &xo, &lo, &yo)) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* x = reinterpret_cast<uint16_t*>(ws + xo);
  float* logits = reinterpret_cast<float*>(ws + lo);
  float* y = reinterpret_cast<float*>(ws + yo);
  const size_t T = (size_t)dims->T;
  // Tokens on the fused decode kernel (T <= kDecodeLayerMaxT): when all three buffers are
  // page-locked host memory mapped into the device's address space, one small kernel reads x and
  // logits across the CPU-GPU link into the workspace (once, instead of once per CTA of the
  // decode kernel), and the decode kernel writes y into host memory itself -- no copy-engine
  // transfers on the stream.  Anything else (pageable memory, unaligned pointers, more tokens)
  // takes the copies.
  if (T <= (size_t)kDecodeLayerMaxT && decode_supported(dims->d, dims->E, dims->k, dims->F)) {
    void* xm = mapped_host(x_host);
    void* lm = mapped_host(logits_host);
    void* ym = host_alloc_writable(y_host) ? mapped_host(y_host) : nullptr;
    if (xm != nullptr && lm != nullptr && ym != nullptr) {
      StageArgs sa{};
      sa.x_src = static_cast<const uint4*>(xm);
      sa.x_dst = reinterpret_cast<uint4*>(x);
      sa.lg_src = static_cast<const float*>(lm);
      sa.lg_dst = logits;
      sa.x_units = (int)T * dims->d * 2 / 16;
      sa.lg_n = (int)T * dims->E;
      sa.early = (options & MOE_OPT_HOST_INPUTS_READY) ? 1 : 0;
      if (launch_stage_in(sa, st) != cudaSuccess) return MOE_ERR_CUDA;
      return moe_layer_forward(dims, x, logits, routed, shared, w_shared_gate, static_cast<float*>(ym), nullptr,
                               workspace, layout_of(*dims).total, stream);
    }
  }
  if (cudaMemcpyAsync(x, x_host, T * dims->d * 2, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(logits, logits_host, T * dims->E * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  s = moe_layer_forward(dims, x, logits, routed, shared, w_shared_gate, y, nullptr, workspace, layout_of(*dims).total,
                        stream);
  if (s != MOE_OK) return s;
  return cudaMemcpyAsync(y_host, y, T * dims->d * 4, cudaMemcpyDeviceToHost, st) == cudaSuccess ? MOE_OK
                                                                                               : MOE_ERR_CUDA;
}

moe_status moe_rmsnorm_router(const moe_dims* dims, float* x_resid, const float* y_prev, const uint16_t* gamma,
                              const uint16_t* w_router, float eps, uint16_t* h_out, float* logits_out,
                              void* workspace, size_t workspace_bytes, void* stream) {
  moe_status s = check_dims(dims);
  if (s != MOE_OK) return s;
  if (!(eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
  if (dims->T == 0) return MOE_OK;
  const void* ps[] = {x_resid, gamma, w_router, h_out, logits_out};
  for (const void* p : ps)
    if ((s = check_ptr(p)) != MOE_OK) return s;
  if (y_prev != nullptr && (s = check_ptr(y_prev)) != MOE_OK) return s;
  if ((s = check_ptr(workspace)) != MOE_OK) return s == MOE_ERR_INVALID_ARG ? MOE_ERR_WORKSPACE : s;
  if (workspace_bytes < 4) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  NormArgs na{x_resid, y_prev, gamma, dims->T, dims->d, eps, h_out};
  if (launch_rmsnorm(na, st) != cudaSuccess) return MOE_ERR_CUDA;
  RouterMaps maps{};
  if (!encode_bf16_rows(&maps.w, w_router, dims->E, dims->d) || !encode_bf16_rows(&maps.h, h_out, dims->T, dims->d))
    return MOE_ERR_CUDA;
  RouterArgs ra{dims->T, dims->d, dims->E, logits_out, at<uint32_t>(workspace, 0)};
  return cuda_status(launch_router(maps, ra, st));
}

moe_status moe_wait_timeout_probe(void* workspace, size_t workspace_bytes, long long limit_cycles, void* stream) {
  if (limit_cycles < 1 || limit_cycles > 4000000000ll) return MOE_ERR_INVALID_ARG;
  moe_status s = check_ptr(workspace);
  if (s != MOE_OK) return s == MOE_ERR_INVALID_ARG ? MOE_ERR_WORKSPACE : s;
  if (workspace_bytes < kWsHeadBytes) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_wait_probe(static_cast<uint32_t*>(workspace), limit_cycles,
                                       static_cast<cudaStream_t>(stream)));
}

moe_status moe_decode_stream_probe(const moe_dims* dims, const int32_t* idx, const moe_experts* routed,
                                   const moe_experts* shared, void* workspace, size_t workspace_bytes, void* stream) {
  moe_status s = check_dims(dims);
  if (s != MOE_OK) return s;
  if ((s = check_experts(routed)) != MOE_OK) return s;
  if (shared != nullptr && (s = check_experts(shared)) != MOE_OK) return s;
  if ((shared != nullptr) != (dims->F_shared > 0)) return MOE_ERR_INVALID_ARG;
  if (dims->T == 0) return MOE_OK;
  if (dims->T != 1 || !decode_supported(dims->d, dims->E, dims->k, dims->F)) return MOE_ERR_UNSUPPORTED;
  if ((s = check_ptr(idx)) != MOE_OK) return s;
  if ((s = check_ptr(workspace)) != MOE_OK) return s == MOE_ERR_INVALID_ARG ? MOE_ERR_WORKSPACE : s;
  if (workspace_bytes < 4) return MOE_ERR_WORKSPACE;
  const moe_dims& d = *dims;
  const bool sh = shared != nullptr;
  StreamArgs a{};
  a.gate[0] = qptr(routed->gate);
  a.up[0] = qptr(routed->up);
  a.down[0] = qptr(routed->down);
  if (sh) {
    a.gate[1] = qptr(shared->gate);
    a.up[1] = qptr(shared->up);
    a.down[1] = qptr(shared->down);
  }
  a.idx = idx;
  a.d = d.d;
  a.E = d.E;
  a.k = d.k;
  a.F = d.F;
  a.has_shared = sh ? 1 : 0;
  a.err = at<uint32_t>(workspace, 0);
  DecodeMaps maps{};
  if (!encode_decode_down(&maps.down[0], routed->down.codes, d.E, d.d, d.F) ||
      !encode_decode_down(&maps.down[1], sh ? shared->down.codes : routed->down.codes, sh ? 1 : d.E, d.d, d.F))
    return MOE_ERR_CUDA;
  return cuda_status(launch_decode_stream(maps, a, static_cast<cudaStream_t>(stream)));
}

moe_status moe_clear_error_flags(void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < 4) return MOE_ERR_WORKSPACE;
  const size_t n = 4;   // the error word
  return cuda_status(cudaMemsetAsync(workspace, 0, n, static_cast<cudaStream_t>(stream)));
}

moe_status moe_read_error_flags(void* workspace, size_t workspace_bytes, uint32_t* flags, void* stream) {
  if (workspace == nullptr || flags == nullptr) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < 4) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(flags, workspace, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(workspace, 0, 4) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // extern "C"
