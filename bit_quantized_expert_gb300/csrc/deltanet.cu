// Gated DeltaNet recurrent scan with the state resident in registers (declarations and contracts
// in include/deltanet_scan.h).
//
// The recurrence of one head, S_t = a_t S_{t-1} + b_t (v_t - a_t S_{t-1} k_t) k_t^T, o_t = S_t q_t,
// acts on each row i of S on its own once k_t is known:
//   x_i = S_{t-1}[i, :] . k_t,  y_i = S_{t-1}[i, :] . q_t,  c_i = b_t (v_t[i] - a_t x_i),
//   S_t[i, :] = a_t S_{t-1}[i, :] + c_i k_t,  o_t[i] = a_t y_i + c_i (k_t . q_t).
// So the 128 x 128 state of a head is cut into row blocks: a CTA holds 16 rows in registers (eight
// lanes per row, sixteen columns a lane, interleaved so that the eight lanes of a row read one
// contiguous 128-byte line of k_t and of q_t), and the only per-token communication is the
// three-step butterfly that sums x_i and y_i over a row's eight lanes.  The state is read once
// and written once per call.
//
// Four staging warps feed the scan: tensor-map copies bring 32 tokens of raw bf16 keys, queries
// and this CTA's 16 value rows into a two-deep ring; each staging warp normalises eight of the
// tokens' keys and queries (fp32), computes k_t . q_t, the decay a_t = exp(g_t) and converts the
// values, and the chunk is published through an mbarrier while the scan warps work on the previous
// one.  The scan warps keep each chunk's outputs in shared memory and store them a chunk at a time.

#include <cmath>
#include <cstring>

#include <cuda_bf16.h>

#include "../../include/deltanet_scan.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kSD = 128;                  // key and value size
constexpr int kRowsPerCta = 16;
constexpr int kScanWarps = 4;             // four rows a warp, eight lanes a row
constexpr int kStageWarps = 4;            // eight tokens of a chunk each
constexpr int kThreadsScan = (kScanWarps + kStageWarps) * 32;
constexpr int kChunk = 32;                // tokens per staged chunk
constexpr int kBufs = 2;
constexpr float kL2Eps = 1e-6f;

// Shared-memory loads the compiler may schedule freely (no memory side effects as far as it
// knows): they read data that is constant between two mbarrier waits.  The address they use is
// passed through pin() after each wait, a volatile step that keeps them after it.
__device__ __forceinline__ float4 lds4(uint32_t addr) {
  float4 v;
  asm("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds1(uint32_t addr) {
  float v;
  asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t pin(uint32_t x) {
  asm volatile("mov.b32 %0, %0;" : "+r"(x)::"memory");
  return x;
}
__device__ __forceinline__ void sts1(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float4 lds4_v(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// Dynamic shared memory plan (bytes).
constexpr int kRawKQ = kChunk * kSD * 2;                       // one chunk of k (or q), bf16
constexpr int kRawV = kChunk * kRowsPerCta * 2;                // one chunk of this CTA's v rows
constexpr int kOffRawK = 0;
constexpr int kOffRawQ = kOffRawK + kBufs * kRawKQ;
constexpr int kOffRawV = kOffRawQ + kBufs * kRawKQ;
constexpr int kOffNK = kOffRawV + kBufs * kRawV;               // normalised k, fp32 [kChunk][128]
constexpr int kOffNQ = kOffNK + kBufs * kChunk * kSD * 4;
constexpr int kOffSc = kOffNQ + kBufs * kChunk * kSD * 4;      // {a_t, b_t, k.q, 0} per token
constexpr int kOffV = kOffSc + kBufs * kChunk * 16;            // v rows, fp32 [kChunk][16]
constexpr int kOffO = kOffV + kBufs * kChunk * kRowsPerCta * 4;  // outputs, fp32 [kChunk][16]
constexpr int kScanSmem = kOffO + kBufs * kChunk * kRowsPerCta * 4 + 128;   // + alignment slack
constexpr int kChunkTx = 2 * kRawKQ + kRawV;
static_assert(kOffRawV % 128 == 0 && kOffNK % 16 == 0 && kOffSc % 16 == 0 && kOffO % 16 == 0, "alignment");
static_assert(kChunk == kStageWarps * 8, "eight tokens per staging warp");

struct ScanMaps {
  CUtensorMap qk[2];   // bf16 {128, H, T}, box {128, 1, 32}: q, k
  CUtensorMap v;       // bf16 {128, H, T}, box {16, 1, 32}
};

struct ScanArgs {
  const float* g;
  const float* beta;
  const float* s_in;
  float* s_out;
  float* o;
  uint32_t* err;
  int T, H;
  int early_state;   // state_in may be read before the dependency wait (GDN_OPT_STATE_EARLY)
};

__global__ void __launch_bounds__(kThreadsScan, 1)
    gdn_scan_kernel(const __grid_constant__ ScanMaps maps, const ScanArgs a) {
  extern __shared__ uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t raw_full[kBufs], ready[kBufs], done[kBufs];
  uint8_t* sm = sm_raw + ((128u - (smem_u32(sm_raw) & 127u)) & 127u);   // tensor-copy targets: 128-byte aligned
  __shared__ int abort_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, r0 = blockIdx.x * kRowsPerCta;
  const int nchunks = (a.T + kChunk - 1) / kChunk;
  if (tid == 0) {
    for (int b = 0; b < kBufs; ++b) {
      mbar_init(smem_u32(&raw_full[b]), 1);
      mbar_init(smem_u32(&ready[b]), kStageWarps);
      mbar_init(smem_u32(&done[b]), kScanWarps);
    }
    abort_s = 0;
    mbar_fence_init();
  }
  __syncthreads();
  // Every input may come from the kernel before this one -- except, with early_state, the state,
  // which the scan warps then read before their own wait.
  if (!a.early_state || warp >= kScanWarps) {
    pdl_wait();
    pdl_launch_dependents();
  }

  int issued = 0;   // chunks whose copies the issuing lane (staging warp 0, lane 0) has issued
  if (warp >= kScanWarps) {
    // ------------------------------------------------------------------ staging warps
    const int sw = warp - kScanWarps;
    const bool issuer = (sw == 0 && lane == 0);
    auto issue = [&](int c) {
      const int b = c % kBufs;
      issued = c + 1;
      const uint32_t bar = smem_u32(&raw_full[b]);
      mbar_arrive_expect_tx(bar, kChunkTx);
      tma_load_3d(smem_u32(sm + kOffRawK + b * kRawKQ), &maps.qk[1], bar, 0, h, c * kChunk);
      tma_load_3d(smem_u32(sm + kOffRawQ + b * kRawKQ), &maps.qk[0], bar, 0, h, c * kChunk);
      tma_load_3d(smem_u32(sm + kOffRawV + b * kRawV), &maps.v, bar, r0, h, c * kChunk);
    };
    if (issuer) {
      prefetch_tmap(&maps.qk[0]);
      prefetch_tmap(&maps.qk[1]);
      prefetch_tmap(&maps.v);
      for (int c = 0; c < kBufs && c < nchunks; ++c) issue(c);
    }
    // decay and write strength of this warp's eight tokens, one token a lane, one chunk ahead
    auto load_gb = [&](int c, float& gv, float& bv) {
      const int t = c * kChunk + sw * 8 + lane;
      gv = 0.f;
      bv = 0.f;
      if (lane < 8 && c < nchunks && t < a.T) {
        gv = __ldg(a.g + (size_t)t * a.H + h);
        bv = __ldg(a.beta + (size_t)t * a.H + h);
      }
    };
    float g_cur, b_cur, g_nxt, b_nxt;
    load_gb(0, g_cur, b_cur);
    for (int c = 0; c < nchunks; ++c) {
      const int b = c % kBufs;
      load_gb(c + 1, g_nxt, b_nxt);
      const float a_lane = expf(g_cur);
      if (!mbar_wait_warp(smem_u32(&raw_full[b]), (c / kBufs) & 1, &abort_s, a.err)) break;
      if (c >= kBufs && !mbar_wait_warp(smem_u32(&done[b]), ((c / kBufs) - 1) & 1, &abort_s, a.err)) break;
      const __nv_bfloat16* __restrict__ rk = reinterpret_cast<const __nv_bfloat16*>(sm + kOffRawK + b * kRawKQ);
      const __nv_bfloat16* __restrict__ rq = reinterpret_cast<const __nv_bfloat16*>(sm + kOffRawQ + b * kRawKQ);
      const __nv_bfloat16* __restrict__ rv = reinterpret_cast<const __nv_bfloat16*>(sm + kOffRawV + b * kRawV);
      float* __restrict__ nk = reinterpret_cast<float*>(sm + kOffNK + b * kChunk * kSD * 4);
      float* __restrict__ nq = reinterpret_cast<float*>(sm + kOffNQ + b * kChunk * kSD * 4);
      float4* __restrict__ scs = reinterpret_cast<float4*>(sm + kOffSc + b * kChunk * 16);
      float* __restrict__ vs = reinterpret_cast<float*>(sm + kOffV + b * kChunk * kRowsPerCta * 4);
      const int nt = min(kChunk, a.T - c * kChunk);
      const int t_end = min(sw * 8 + 8, nt);
#pragma unroll 2
      for (int t = sw * 8; t < t_end; ++t) {
        const uint2 kw = *reinterpret_cast<const uint2*>(rk + t * kSD + 4 * lane);
        const uint2 qw = *reinterpret_cast<const uint2*>(rq + t * kSD + 4 * lane);
        const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kw.x));
        const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kw.y));
        const float2 q01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qw.x));
        const float2 q23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qw.y));
        float kk = k01.x * k01.x + k01.y * k01.y + k23.x * k23.x + k23.y * k23.y;
        float qq = q01.x * q01.x + q01.y * q01.y + q23.x * q23.x + q23.y * q23.y;
        float kq = k01.x * q01.x + k01.y * q01.y + k23.x * q23.x + k23.y * q23.y;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          kk += __shfl_xor_sync(0xFFFFFFFFu, kk, off);
          qq += __shfl_xor_sync(0xFFFFFFFFu, qq, off);
          kq += __shfl_xor_sync(0xFFFFFFFFu, kq, off);
        }
        const float rk_n = rsqrtf(kk + kL2Eps);
        const float rq_n = rsqrtf(qq + kL2Eps) * 0.08838834764831845f;   // 1 / sqrt(128)
        *reinterpret_cast<float4*>(nk + t * kSD + 4 * lane) =
            make_float4(k01.x * rk_n, k01.y * rk_n, k23.x * rk_n, k23.y * rk_n);
        *reinterpret_cast<float4*>(nq + t * kSD + 4 * lane) =
            make_float4(q01.x * rq_n, q01.y * rq_n, q23.x * rq_n, q23.y * rq_n);
        const float at = __shfl_sync(0xFFFFFFFFu, a_lane, t - sw * 8);
        const float bt = __shfl_sync(0xFFFFFFFFu, b_cur, t - sw * 8);
        if (lane == 0) scs[t] = make_float4(at, bt, kq * rk_n * rq_n, 0.f);
        if (lane < kRowsPerCta) vs[t * kRowsPerCta + lane] = __bfloat162float(rv[t * kRowsPerCta + lane]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ready[b]));
      // The raw buffer is refilled once all four staging warps have read it (ready[b] complete).
      // (No early exit from this lane alone: the warp's next collective wait needs every lane; after
      // a timeout that wait fails for all of them together.)
      if (issuer && c + kBufs < nchunks && mbar_wait(smem_u32(&ready[b]), (c / kBufs) & 1, &abort_s, a.err)) {
        fence_proxy_async_smem();
        issue(c + kBufs);
      }
      g_cur = g_nxt;
      b_cur = b_nxt;
    }
  } else {
    // ------------------------------------------------------------------ scan warps
    const int row = warp * 4 + (lane >> 3), lr = lane & 7;
    const int i_glob = r0 + row;
    float s[16];   // S[i, 32 j + 4 lr + e] in s[4 j + e]
    {
      const float4* src = reinterpret_cast<const float4*>(a.s_in + ((size_t)h * kSD + i_glob) * kSD) + lr;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 v4 = __ldg(src + 8 * j);
        s[4 * j] = v4.x;
        s[4 * j + 1] = v4.y;
        s[4 * j + 2] = v4.z;
        s[4 * j + 3] = v4.w;
      }
    }
    if (a.early_state) {   // the state is in registers; the token inputs come after the wait
      pdl_wait();
      pdl_launch_dependents();
    }
    const size_t o_step = (size_t)a.H * kSD;
    float* __restrict__ o_out = a.o + (size_t)h * kSD + r0 + warp * 4;
    const uint32_t sm_base = smem_u32(sm);
    // Token t of the staged ring: buffer (t / 32) % 2, slot t % 32.  `base` is re-pinned after
    // every wait so that no load of a chunk moves above the wait that publishes it.
    uint32_t base = sm_base;
    auto kq_addr = [&](int off, int t) {
      return base + off + ((t / kChunk) % kBufs) * (kChunk * kSD * 4) + ((t % kChunk) * kSD + 4 * lr) * 4;
    };
    auto slice = [&](uint32_t addr, float (&dst)[16]) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 v4 = lds4(addr + 128 * j);
        dst[4 * j] = v4.x, dst[4 * j + 1] = v4.y, dst[4 * j + 2] = v4.z, dst[4 * j + 3] = v4.w;
      }
    };
    for (int c = 0; c < nchunks; ++c) {
      const int b = c % kBufs;
      if (!mbar_wait_warp(smem_u32(&ready[b]), (c / kBufs) & 1, &abort_s, a.err)) break;
      base = pin(sm_base);
      const int nt = min(kChunk, a.T - c * kChunk);
      // Each token's output is stored during the next token, after that token's operand loads:
      // a store placed before them would keep them (possible alias) behind this token's chain.
      float o_prev = 0.f;
      uint32_t o_prev_addr = 0u;
#pragma unroll 2
      for (int tt = 0; tt < nt; ++tt) {
        const int t = c * kChunk + tt;
        float kv[16], qv[16];
        slice(kq_addr(kOffNK, t), kv);
        slice(kq_addr(kOffNQ, t), qv);
        const float4 sc = lds4(base + kOffSc + b * (kChunk * 16) + tt * 16);
        const float vi = lds1(base + kOffV + b * (kChunk * kRowsPerCta * 4) + (tt * kRowsPerCta + row) * 4);
        if (tt > 0 && lr == 0) sts1(o_prev_addr, o_prev);
        float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f, y0 = 0.f, y1 = 0.f, y2 = 0.f, y3 = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          x0 = fmaf(s[4 * j], kv[4 * j], x0);
          x1 = fmaf(s[4 * j + 1], kv[4 * j + 1], x1);
          x2 = fmaf(s[4 * j + 2], kv[4 * j + 2], x2);
          x3 = fmaf(s[4 * j + 3], kv[4 * j + 3], x3);
          y0 = fmaf(s[4 * j], qv[4 * j], y0);
          y1 = fmaf(s[4 * j + 1], qv[4 * j + 1], y1);
          y2 = fmaf(s[4 * j + 2], qv[4 * j + 2], y2);
          y3 = fmaf(s[4 * j + 3], qv[4 * j + 3], y3);
        }
        float x = (x0 + x1) + (x2 + x3), y = (y0 + y1) + (y2 + y3);
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) {
          x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
          y += __shfl_xor_sync(0xFFFFFFFFu, y, off);
        }
        const float at = sc.x, ci = sc.y * (vi - at * x);
#pragma unroll
        for (int e = 0; e < 16; ++e) s[e] = fmaf(ci, kv[e], at * s[e]);
        o_prev = fmaf(at, y, ci * sc.z);
        o_prev_addr = sm_base + kOffO + b * (kChunk * kRowsPerCta * 4) + (tt * kRowsPerCta + row) * 4;
      }
      if (nt > 0 && lr == 0) sts1(o_prev_addr, o_prev);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&done[b]));
      if (lane < nt) {
        const float4 ov = lds4_v(sm_base + kOffO + b * (kChunk * kRowsPerCta * 4) + (lane * kRowsPerCta + warp * 4) * 4);
        *reinterpret_cast<float4*>(o_out + (size_t)(c * kChunk + lane) * o_step) = ov;
      }
    }
    bool finite = true;
    float4* dst = reinterpret_cast<float4*>(a.s_out + ((size_t)h * kSD + i_glob) * kSD) + lr;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      finite = finite && isfinite(s[4 * j]) && isfinite(s[4 * j + 1]) && isfinite(s[4 * j + 2]) &&
               isfinite(s[4 * j + 3]);
      dst[8 * j] = make_float4(s[4 * j], s[4 * j + 1], s[4 * j + 2], s[4 * j + 3]);
    }
    if (!finite) raise_flag(a.err, kErrNonFinite);
  }
  __syncthreads();
  // After a timeout, copies still in flight land before the CTA exits: the staging lane waits
  // (bounded) for the last chunk it issued into each buffer.
  if (tid == kScanWarps * 32 && abort_s) {
    for (int c = issued - kBufs < 0 ? 0 : issued - kBufs; c < issued; ++c) {
      const long long c0 = clock64();
      while (!mbar_try_wait(smem_u32(&raw_full[c % kBufs]), (c / kBufs) & 1) && clock64() - c0 < 4000000ll) {
      }
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_scan_dims(const gdn_dims* d) {
  if (d == nullptr || d->T < 0 || d->H < 1) return MOE_ERR_INVALID_ARG;
  if (d->d_k != kSD || d->d_v != kSD || d->H > 65535) return MOE_ERR_UNSUPPORTED;
  if ((long long)d->T * d->H * kSD >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool encode_tokens(CUtensorMap* m, const uint16_t* base, int T, int H, int box_inner) {
  EncodeTiledFn f = encode_fn();
  if (f == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kSD, (cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)kSD * 2, (cuuint64_t)H * kSD * 2};
  const cuuint32_t box[3] = {(cuuint32_t)box_inner, 1, kChunk};
  const cuuint32_t estr[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t gdn_scan_workspace_bytes(const gdn_dims* dims) {
  return check_scan_dims(dims) == MOE_OK ? (size_t)kWsHeadBytes : 0;
}

extern "C" moe_status gdn_scan(const gdn_dims* dims, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const float* g, const float* beta, const float* state_in, float* state_out, float* o,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return gdn_scan_opts(dims, q, k, v, g, beta, state_in, state_out, o, workspace, workspace_bytes, stream, 0u);
}

extern "C" moe_status gdn_scan_opts(const gdn_dims* dims, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    const float* g, const float* beta, const float* state_in, float* state_out,
                                    float* o, void* workspace, size_t workspace_bytes, void* stream,
                                    uint32_t options) {
  if (options & ~(uint32_t)GDN_OPT_STATE_EARLY) return MOE_ERR_INVALID_ARG;
  const int st = check_scan_dims(dims);
  if (st != MOE_OK) return (moe_status)st;
  if (state_in == nullptr || state_out == nullptr || workspace == nullptr) return MOE_ERR_INVALID_ARG;
  if (dims->T > 0 && (q == nullptr || k == nullptr || v == nullptr || g == nullptr || beta == nullptr || o == nullptr))
    return MOE_ERR_INVALID_ARG;
  const void* ps[] = {q, k, v, g, beta, state_in, state_out, o, workspace};
  for (const void* p : ps)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_MISALIGNED;
  if (workspace_bytes < gdn_scan_workspace_bytes(dims)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t state_bytes = (size_t)dims->H * kSD * kSD * sizeof(float);
  if (dims->T == 0) {
    if (state_out == state_in) return MOE_OK;
    return cudaMemcpyAsync(state_out, state_in, state_bytes, cudaMemcpyDeviceToDevice, s) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
  }
  ScanMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (!encode_tokens(&maps.qk[0], q, dims->T, dims->H, kSD) || !encode_tokens(&maps.qk[1], k, dims->T, dims->H, kSD) ||
      !encode_tokens(&maps.v, v, dims->T, dims->H, kRowsPerCta))
    return MOE_ERR_CUDA;
  static bool attr_done = false;   // idempotent: racing first calls set the same value
  if (!attr_done) {
    if (cudaFuncSetAttribute(gdn_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_done = true;
  }
  ScanArgs a;
  a.g = g;
  a.beta = beta;
  a.s_in = state_in;
  a.s_out = state_out;
  a.o = o;
  a.err = static_cast<uint32_t*>(workspace);
  a.T = dims->T;
  a.H = dims->H;
  a.early_state = (options & GDN_OPT_STATE_EARLY) ? 1 : 0;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kSD / kRowsPerCta, dims->H);
  cfg.blockDim = dim3(kThreadsScan);
  cfg.dynamicSmemBytes = kScanSmem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gdn_scan_kernel, maps, a) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
