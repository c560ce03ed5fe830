// Pre-norm block of a stack of MoE layers: residual add, RMSNorm and the router GEMM.
//
// The pages describe the router only as scoring 256 experts per token ("Perplexity ouvre le code
// de Lily...", article body; "Perplexity libera Lily: inferencia en Rust y Metal para Mac", section
// "Tres formas de carga en un mismo modelo").  The stacked-layer workload places it after an
// RMSNorm of the fp32 residual stream: x <- x + y_prev; h = x / sqrt(mean(x^2) + eps) * gamma
// (bf16); logits = h W_r^T with bf16 operands and fp32 accumulation.
//
//   rmsnorm_kernel  one warp per token; fp32 sums; writes x back when a previous output is added.
//   router_kernel   one CTA per (128 experts x 128 tokens) tile: TMA (128-byte swizzle) brings
//                   64-column chunks of W_r and h into a 4-stage ring, one thread issues
//                   tcgen05.mma (kind::f16, bf16 x bf16 -> fp32 in TMEM), four warps read TMEM and
//                   write logits[t][e] (lane = expert, so stores are coalesced).
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) rmsnorm_kernel(NormArgs a) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= a.T) return;
  float4* x4 = reinterpret_cast<float4*>(a.x + (size_t)t * a.d);
  const float4* y4 = a.y_prev ? reinterpret_cast<const float4*>(a.y_prev + (size_t)t * a.d) : nullptr;
  const int n4 = a.d / 4;
  float ss = 0.0f;
  for (int c = lane; c < n4; c += 32) {
    float4 v = x4[c];
    if (y4 != nullptr) {
      const float4 u = __ldg(y4 + c);
      v.x += u.x;
      v.y += u.y;
      v.z += u.z;
      v.w += u.w;
      x4[c] = v;
    }
    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
  const float r = 1.0f / sqrtf(ss / (float)a.d + a.eps);
  __syncwarp();
  uint2* h2 = reinterpret_cast<uint2*>(a.h + (size_t)t * a.d);
  const uint2* g2 = reinterpret_cast<const uint2*>(a.gamma);
  for (int c = lane; c < n4; c += 32) {
    const float4 v = x4[c];
    const uint2 g = __ldg(g2 + c);
    const float gv[4] = {bf16_bits_to_f32(g.x & 0xFFFFu), bf16_bits_to_f32(g.x >> 16), bf16_bits_to_f32(g.y & 0xFFFFu),
                         bf16_bits_to_f32(g.y >> 16)};
    const float vv[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = __bfloat16_as_ushort(__float2bfloat16_rn(vv[i] * r * gv[i]));
    h2[c] = make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
  }
}

constexpr int kStages = 4;
constexpr uint32_t kTile = 128 * 128;   // 128 rows x 64 bf16
constexpr uint32_t kSmem = 2 * kStages * kTile + 1024 + 256;

__device__ __forceinline__ uint32_t idesc_bf16_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__global__ void __launch_bounds__(192, 1) router_kernel(const __grid_constant__ RouterMaps maps, RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t s0 = smem_u32(smem_raw);
  const uint32_t sb = (s0 + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - s0);
  const uint32_t sA = sb, sB = sb + kStages * kTile, sBar = sb + 2 * kStages * kTile;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + 2 * kStages * kTile + 8 * (2 * kStages + 1));
  volatile int* abort_s = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto FULL = [&](int i) { return sBar + 8u * i; };
  auto EMPTY = [&](int i) { return sBar + 8u * (kStages + i); };
  const uint32_t DONE = sBar + 8u * (2 * kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128;   // experts
  const int n0 = blockIdx.y * 128;   // tokens
  const int KC = a.d / 64;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(FULL(i), 1);
      mbar_init(EMPTY(i), 1);
    }
    mbar_init(DONE, 1);
    *abort_s = 0;
    mbar_fence_init();
    prefetch_tmap(&maps.w);
    prefetch_tmap(&maps.h);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      for (int kc = 0; kc < KC; ++kc) {
        const int s = kc % kStages;
        if (!mbar_wait(EMPTY(s), ((kc / kStages) & 1) ^ 1u, abort_s, a.err)) break;
        mbar_arrive_expect_tx(FULL(s), 2 * kTile);
        tma_load_2d(sA + s * kTile, &maps.w, FULL(s), kc * 64, m0);
        tma_load_2d(sB + s * kTile, &maps.h, FULL(s), kc * 64, n0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 128);
      bool ok = true;
      for (int kc = 0; kc < KC; ++kc) {
        const int s = kc % kStages;
        if (!mbar_wait(FULL(s), (kc / kStages) & 1, abort_s, a.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_f16(tmem, smem_desc_sw128(sA + s * kTile + kk * 32), smem_desc_sw128(sB + s * kTile + kk * 32),
                     idesc, (kc | kk) != 0 ? 1u : 0u);
        tc_commit(EMPTY(s));
      }
      if (ok) tc_commit(DONE);
    }
  } else {
    const int q = warp & 3;
    if (mbar_wait_warp(DONE, 0, abort_s, a.err)) {
      tc_fence_after();
      const int e = m0 + q * 32 + lane;
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t v[16];
        tmem_ld16_wait(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = n0 + c0 + i;
          if (t < a.T && e < a.E) a.logits[(size_t)t * a.E + e] = __uint_as_float(v[i]);
        }
      }
    }
  }
  if (threadIdx.x == 0 && *abort_s) {
    const long long t0 = clock64();
    while (clock64() - t0 < 4000000ll) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const NormArgs& a, cudaStream_t st) {
  rmsnorm_kernel<<<(a.T + 7) / 8, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_router(const RouterMaps& maps, const RouterArgs& a, cudaStream_t st) {
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  const dim3 grid((a.E + 127) / 128, (a.T + 127) / 128);
  router_kernel<<<grid, 192, kSmem, st>>>(maps, a);
  return cudaGetLastError();
}

}  // namespace moe
