// Allocation-free variant of the one-token (decode) layer call.
//
// moe_layer_forward needs a workspace that the caller allocates.  Some callers cannot allocate
// device memory when they call the layer: an engine whose memory planner hands out every byte
// of HBM once, at start-up, to weights and caches and forbids later cudaMalloc calls; a
// latency-critical decode loop that must never enter cudaMalloc or cudaFree, which may
// synchronise the whole device; or a host program that only holds pointers to weights, inputs
// and outputs and has no allocator of its own.  moe_layer_forward_decode_noalloc serves them: the
// only scratch it needs (an error word and the decode kernel's partial outputs per row slice)
// lives in the file-scope device array below, which every GPU that loads
// this library holds until the process exits.
#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

namespace moe {
namespace {

// The first kWsHeadBytes hold the error word, as in a workspace; then the decode kernel's partial
// outputs of one token (decode_scratch_floats).
constexpr int kNoAllocHeadFloats = (int)(kWsHeadBytes / 4);
constexpr size_t kNoAllocMaxPart = 131072;   // upper bound on the partial outputs: 512 KB
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocHeadFloats + kNoAllocMaxPart];

constexpr int kMaxDevices = 64;
float* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the array on the current device.  In host code the array's name is only a
// stand-in for the symbol, not an address a kernel may use; the address comes from
// cudaGetSymbolAddress, asked once per device with that device current.
cudaError_t scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

moe_status check_qmat_ptrs(const moe_qmat& q) {
  const void* ps[] = {q.codes, q.scales, q.biases};
  for (const void* p : ps) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p) & 15u) return MOE_ERR_MISALIGNED;
  }
  return MOE_OK;
}

moe_status check_expert_ptrs(const moe_experts& x) {
  moe_status s;
  if ((s = check_qmat_ptrs(x.gate)) != MOE_OK) return s;
  if ((s = check_qmat_ptrs(x.up)) != MOE_OK) return s;
  return check_qmat_ptrs(x.down);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_layer_forward_decode_noalloc(const moe_dims* dims, const uint16_t* x, const float* logits,
                                                       const moe_experts* routed, const moe_experts* shared,
                                                       const uint16_t* w_shared_gate, float* y, void* stream) {
  if (dims == nullptr || routed == nullptr) return MOE_ERR_INVALID_ARG;
  // the dims rules of moe_layer_forward, with its status codes
  const int ds = check_layer_dims(dims->T, dims->d, dims->E, dims->k, dims->F, dims->F_shared);
  if (ds != MOE_OK) return static_cast<moe_status>(ds);
  if (dims->T == 0) return MOE_OK;
  if (dims->T != 1) return MOE_ERR_UNSUPPORTED;                      // one token per call
  const bool sh = shared != nullptr;
  if (sh != (dims->F_shared > 0)) return MOE_ERR_INVALID_ARG;
  if (!decode_supported(dims->d, dims->E, dims->k, dims->F)) return MOE_ERR_UNSUPPORTED;
  if (decode_scratch_floats(dims->d, dims->k, dims->F) > kNoAllocMaxPart) return MOE_ERR_UNSUPPORTED;
  moe_status s;
  if ((s = check_expert_ptrs(*routed)) != MOE_OK) return s;
  if (sh && (s = check_expert_ptrs(*shared)) != MOE_OK) return s;
  const void* ps[] = {x, logits, y, sh ? static_cast<const void*>(w_shared_gate) : static_cast<const void*>(x)};
  for (const void* p : ps) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p) & 15u) return MOE_ERR_MISALIGNED;
  }

  float* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = reinterpret_cast<uint32_t*>(scratch);
  // The array keeps the previous call's contents: the error word starts every call at zero.  Every
  // partial is written by the decode kernel before the reduce kernel of the same call reads it.
  if (cudaMemsetAsync(err, 0, 4, st) != cudaSuccess) return MOE_ERR_CUDA;

  DecodeArgs da{};
  da.x = x;
  da.logits = logits;
  da.gate[0] = QPtr{routed->gate.codes, routed->gate.scales, routed->gate.biases};
  da.up[0] = QPtr{routed->up.codes, routed->up.scales, routed->up.biases};
  da.down[0] = QPtr{routed->down.codes, routed->down.scales, routed->down.biases};
  if (sh) {
    da.gate[1] = QPtr{shared->gate.codes, shared->gate.scales, shared->gate.biases};
    da.up[1] = QPtr{shared->up.codes, shared->up.scales, shared->up.biases};
    da.down[1] = QPtr{shared->down.codes, shared->down.scales, shared->down.biases};
  }
  da.w_sg = sh ? w_shared_gate : nullptr;
  da.d = dims->d;
  da.E = dims->E;
  da.k = dims->k;
  da.F = dims->F;
  da.has_shared = sh ? 1 : 0;
  da.T = 1;
  da.part = scratch + kNoAllocHeadFloats;
  da.y = y;
  da.err = err;
  DecodeMaps dmaps{};
  if (!encode_decode_down(&dmaps.down[0], routed->down.codes, dims->E, dims->d, dims->F) ||
      !encode_decode_down(&dmaps.down[1], sh ? shared->down.codes : routed->down.codes, sh ? 1 : dims->E, dims->d,
                          dims->F))
    return MOE_ERR_CUDA;
  return launch_decode(dmaps, da, st, true) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
