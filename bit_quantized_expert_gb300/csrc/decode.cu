// Decode (T = 1) MoE layer as two bandwidth-bound dequant-GEMV kernels.
//
// At batch 1 there is almost no weight reuse, so weight bandwidth sets the ceiling ("Perplexity
// libera Lily: inferencia en Rust y Metal para Mac", section "Decode: mover menos bytes por
// token"); the pages also report that removing all arithmetic from the kernels changed speed by
// 0.2% and that matrix ops reached 97.9% of bandwidth ("Perplexity открыла код Lily...",
// section "Спекулятивное декодирование не взлетело").  The design follows from that:
//
//   kernel A  grid (F/32, k + shared): every CTA redoes the top-k of the token's 256 logits
//             (1 KB from L2) instead of waiting for a routing kernel, bulk-copies 32 gate rows and
//             32 up rows of its expert (72 KB at d = 2048) into shared memory with one mbarrier,
//             and computes 32 SwiGLU outputs h in fp32.
//   kernel B  grid (d/16): every CTA redoes the top-k, bulk-copies 16 rows of the down matrix of
//             all k + 1 experts, then (after the programmatic-launch wait for kernel A) computes
//             y[r] = sum_j w_j (W_down[e_j] h_j)[r] + sigmoid(x . w_sg) (W_down_shared h_s)[r].
//   Kernel B is launched as a programmatic dependent of A: its CTAs start while A runs, so its
//   weight copies overlap A's and only the h read waits.  Kernel A issues its own
//   launch_dependents only after its griddepcontrol.wait, so everything B reads before its
//   wait (x, logits, weights) was complete before A started.
//
// Arithmetic: codes become exact fp32 integers via the 2^23 exponent trick, partial dot products
// sum_c q_c x_c accumulate in fp32, then w = q*s + b enters as s * sum(q x) + b * sum(x) per group.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int RF = 32;   // gate/up rows per CTA in kernel A
constexpr int RD = 16;   // down rows per CTA in kernel B
constexpr float kMagic = 8388608.0f;   // 2^23

// Expand nibble n of `w` (or of `w >> 12` for n >= 5) to q * 16^e exactly, e = n < 5 ? n : n - 3.
template <int N>
__device__ __forceinline__ float code_scaled(uint32_t w, uint32_t w12) {
  const uint32_t v = N < 5 ? (w & (0xFu << (4 * N))) : (w12 & (0xFu << (4 * (N - 3))));
  return __uint_as_float(v | 0x4B000000u) - kMagic;
}
// The matching power-of-two pre-scale of the activation: 16^-e.
__host__ __device__ constexpr float act_prescale(int n) {
  return n % 8 == 0 ? 1.0f : n % 8 == 1 ? 0.0625f : n % 8 == 2 ? 0.00390625f : n % 8 == 3 ? 0.000244140625f
       : n % 8 == 4 ? 1.52587890625e-05f : n % 8 == 5 ? 0.00390625f : n % 8 == 6 ? 0.000244140625f
       : 1.52587890625e-05f;
}

// sum over the 8 codes of word w of q_c * xs[c] (xs pre-scaled by act_prescale)
__device__ __forceinline__ float word_dot(uint32_t w, const float* xs, float acc) {
  const uint32_t w12 = w >> 12;
  acc = fmaf(code_scaled<0>(w, w12), xs[0], acc);
  acc = fmaf(code_scaled<1>(w, w12), xs[1], acc);
  acc = fmaf(code_scaled<2>(w, w12), xs[2], acc);
  acc = fmaf(code_scaled<3>(w, w12), xs[3], acc);
  acc = fmaf(code_scaled<4>(w, w12), xs[4], acc);
  acc = fmaf(code_scaled<5>(w, w12), xs[5], acc);
  acc = fmaf(code_scaled<6>(w, w12), xs[6], acc);
  acc = fmaf(code_scaled<7>(w, w12), xs[7], acc);
  return acc;
}

__device__ __forceinline__ int topk_ni(int E) { return (E + 31) / 32; }

// Warp 0 of the CTA: top-k; lane j < k gets (expert, weight).
__device__ __forceinline__ void decode_topk(const float* logits, int E, int k, int* e, float* w) {
  const int ni = topk_ni(E);
  if (ni <= 1) warp_topk_softmax<1>(logits, E, k, e, w);
  else if (ni <= 2) warp_topk_softmax<2>(logits, E, k, e, w);
  else if (ni <= 4) warp_topk_softmax<4>(logits, E, k, e, w);
  else if (ni <= 8) warp_topk_softmax<8>(logits, E, k, e, w);
  else if (ni <= 16) warp_topk_softmax<16>(logits, E, k, e, w);
  else warp_topk_softmax<32>(logits, E, k, e, w);
}

struct SmemA {
  static size_t bytes(int d) {
    const int G = d / 64;
    return (size_t)2 * RF * (d / 2) + (size_t)4 * RF * G * 2 + 64;
  }
};

__global__ void __launch_bounds__(256) decode_gateup_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int d = a.d, G = d / 64;
  const int j = blockIdx.y;                 // 0..k-1 routed, k = shared
  const int f0 = blockIdx.x * RF;
  const bool is_shared = (j == a.k);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint32_t* codes_g = reinterpret_cast<uint32_t*>(sm);
  uint32_t* codes_u = codes_g + RF * (d / 8);
  uint16_t* sc_g = reinterpret_cast<uint16_t*>(codes_u + RF * (d / 8));
  uint16_t* bi_g = sc_g + RF * G;
  uint16_t* sc_u = bi_g + RF * G;
  uint16_t* bi_u = sc_u + RF * G;
  __shared__ __align__(8) uint64_t bar;
  __shared__ int e_s;
  __shared__ int abort_s;
  const uint32_t sbar = smem_u32(&bar);

  if (tid == 0) {
    mbar_init(sbar, 1);
    abort_s = 0;
    mbar_fence_init();
  }
  __syncthreads();

  auto issue = [&](int which, int e) {
    const QPtr& g = a.gate[which];
    const QPtr& u = a.up[which];
    const size_t row0 = (size_t)e * a.F + f0;
    const uint32_t cb = RF * (d / 2), sb = RF * G * 2;
    mbar_arrive_expect_tx(sbar, 2 * cb + 4 * sb);
    bulk_g2s(smem_u32(codes_g), g.codes + row0 * (d / 8), cb, sbar);
    bulk_g2s(smem_u32(codes_u), u.codes + row0 * (d / 8), cb, sbar);
    bulk_g2s(smem_u32(sc_g), g.scales + row0 * G, sb, sbar);
    bulk_g2s(smem_u32(bi_g), g.biases + row0 * G, sb, sbar);
    bulk_g2s(smem_u32(sc_u), u.scales + row0 * G, sb, sbar);
    bulk_g2s(smem_u32(bi_u), u.biases + row0 * G, sb, sbar);
  };

  // The shared expert's rows depend on nothing upstream: start copying before the wait.
  if (is_shared && tid == 0) issue(1, 0);
  pdl_wait();
  if (!is_shared && warp == 0) {
    int e;
    float w;
    decode_topk(a.logits, a.E, a.k, &e, &w);
    if (lane == j) e_s = e;
    __syncwarp();
    if (lane == 0) issue(0, e_s);
  }
  pdl_launch_dependents();

  // Each lane owns groups g = lane, lane + 32, ...; warp w owns rows 4w .. 4w+3 of gate and up.
  float acc[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
  const uint4* xv = reinterpret_cast<const uint4*>(a.x);
  bool waited = false;
  for (int g = lane; g - lane < G; g += 32) {
    const bool active = g < G;
    float xs[64];
    float xsum = 0.0f;
    if (active) {
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const uint4 v = __ldg(xv + g * 8 + c8);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = bf16_bits_to_f32(wv[i] & 0xFFFFu), hi = bf16_bits_to_f32(wv[i] >> 16);
          xsum += lo + hi;
          xs[c8 * 8 + 2 * i] = lo * act_prescale(2 * i);
          xs[c8 * 8 + 2 * i + 1] = hi * act_prescale(2 * i + 1);
        }
      }
    }
    if (!waited) {
      if (!mbar_wait(sbar, 0, &abort_s, a.err)) break;
      waited = true;
    }
    if (active) {
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int row = 4 * warp + (r & 3);
        const uint32_t* cw = (r < 4 ? codes_g : codes_u) + row * (d / 8) + g * 8;
        const uint4 c0 = *reinterpret_cast<const uint4*>(cw);
        const uint4 c1 = *reinterpret_cast<const uint4*>(cw + 4);
        float p = 0.0f;
        p = word_dot(c0.x, xs + 0, p);
        p = word_dot(c0.y, xs + 8, p);
        p = word_dot(c0.z, xs + 16, p);
        p = word_dot(c0.w, xs + 24, p);
        p = word_dot(c1.x, xs + 32, p);
        p = word_dot(c1.y, xs + 40, p);
        p = word_dot(c1.z, xs + 48, p);
        p = word_dot(c1.w, xs + 56, p);
        const float s = bf16_bits_to_f32((r < 4 ? sc_g : sc_u)[row * G + g]);
        const float b = bf16_bits_to_f32((r < 4 ? bi_g : bi_u)[row * G + g]);
        acc[r] = fmaf(s, p, fmaf(b, xsum, acc[r]));
      }
    }
  }
  if (!waited && !abort_s) {
    // lanes with no group still wait so the copies have landed before the CTA exits
    mbar_wait(sbar, 0, &abort_s, a.err);
  }
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xFFFFFFFFu, acc[r], off);
  if (lane < 4 && !abort_s) {
    const float gv = acc[lane], uv = acc[4 + lane];
    const float hv = gv / (1.0f + expf(-gv)) * uv;
    a.h[(size_t)j * a.F + f0 + 4 * warp + lane] = hv;
  }
}

struct SmemB {
  static size_t bytes(int k1, int F) {
    const int GF = F / 64;
    return (size_t)k1 * RD * (F / 2) + (size_t)2 * k1 * RD * GF * 2 + (size_t)k1 * F * 4 + (size_t)k1 * RD * 4 + 64;
  }
};

// EPL: elements of the reduction (F) per lane: max(8, F/32).
template <int EPL>
__global__ void __launch_bounds__(256) decode_down_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int F = a.F, GF = F / 64;
  const int k1 = a.k + (a.has_shared ? 1 : 0);
  const int r0 = blockIdx.x * RD;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint32_t* codes = reinterpret_cast<uint32_t*>(sm);                 // [k1][RD][F/8]
  uint16_t* scl = reinterpret_cast<uint16_t*>(codes + k1 * RD * (F / 8));   // [k1][RD][GF]
  uint16_t* bia = scl + k1 * RD * GF;
  float* hs = reinterpret_cast<float*>(bia + k1 * RD * GF);          // [k1][F]
  float* part = hs + k1 * F;                                          // [k1][RD]
  __shared__ __align__(8) uint64_t bar;
  __shared__ int e_s[32];
  __shared__ float w_s[32];
  __shared__ float gs_s;
  __shared__ int abort_s;
  const uint32_t sbar = smem_u32(&bar);

  if (tid == 0) {
    mbar_init(sbar, 1);
    abort_s = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const uint32_t cb = RD * (F / 2), sb = RD * GF * 2;
  if (tid == 0) mbar_arrive_expect_tx(sbar, (uint32_t)k1 * (cb + 2 * sb));
  auto issue = [&](int slot, int which, int e) {
    const QPtr& q = a.down[which];
    const size_t row0 = (size_t)e * a.d + r0;
    bulk_g2s(smem_u32(codes + slot * RD * (F / 8)), q.codes + row0 * (F / 8), cb, sbar);
    bulk_g2s(smem_u32(scl + slot * RD * GF), q.scales + row0 * GF, sb, sbar);
    bulk_g2s(smem_u32(bia + slot * RD * GF), q.biases + row0 * GF, sb, sbar);
  };
  __syncthreads();   // expect_tx precedes every complete_tx
  if (a.has_shared && tid == 0) issue(a.k, 1, 0);
  if (warp == 0) {
    int e;
    float w;
    decode_topk(a.logits, a.E, a.k, &e, &w);
    if (lane < a.k) {
      e_s[lane] = e;
      w_s[lane] = w;
    }
    __syncwarp();
    if (lane == 0)
      for (int jj = 0; jj < a.k; ++jj) issue(jj, 0, e_s[jj]);
  } else if (warp == 1) {
    float dot = 0.0f;
    if (a.has_shared && a.w_sg != nullptr) {
      for (int c = lane; c < a.d; c += 32) dot = fmaf(bf16_bits_to_f32(a.x[c]), bf16_bits_to_f32(a.w_sg[c]), dot);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
    }
    if (lane == 0) gs_s = 1.0f / (1.0f + expf(-dot));
  }
  pdl_wait();   // h from kernel A is complete and visible past this point
  for (int i = tid; i < k1 * F; i += blockDim.x) hs[i] = a.h[i];
  __syncthreads();

  // Warp w owns expert slots w, w + 8, ...; LPR lanes cover one row, RPW rows at a time.
  constexpr int LPR_MAX = 32;
  const int LPR = F / EPL < LPR_MAX ? F / EPL : LPR_MAX;
  const int RPW = 32 / LPR;
  const int sub = lane / LPR, l = lane % LPR;
  const int c0 = l * EPL;                      // first element of this lane's range
  const int grp = c0 / 64;
  const bool ok = mbar_wait(sbar, 0, &abort_s, a.err);
  for (int jj = warp; jj < k1; jj += (int)(blockDim.x >> 5)) {
    float hv[EPL];
    float hsum = 0.0f;
#pragma unroll
    for (int c = 0; c < EPL; ++c) {
      const float v = hs[jj * F + c0 + c];
      hsum += v;
      hv[c] = v * act_prescale(c);
    }
    for (int rb = 0; rb < RD; rb += RPW) {
      const int r = rb + sub;
      float p = 0.0f, s = 0.0f, b = 0.0f;
      if (ok && r < RD) {
        const uint32_t* cw = codes + (jj * RD + r) * (F / 8) + c0 / 8;
#pragma unroll
        for (int wd = 0; wd < EPL / 8; ++wd) p = word_dot(cw[wd], hv + 8 * wd, p);
        s = bf16_bits_to_f32(scl[(jj * RD + r) * GF + grp]);
        b = bf16_bits_to_f32(bia[(jj * RD + r) * GF + grp]);
      }
      float v = fmaf(s, p, b * hsum);
      for (int off = LPR / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      if (l == 0 && r < RD) part[jj * RD + r] = v;
    }
  }
  __syncthreads();
  if (tid < RD && !abort_s) {
    float y = 0.0f;
    for (int jj = 0; jj < a.k; ++jj) y = fmaf(w_s[jj], part[jj * RD + tid], y);
    if (a.has_shared) y = fmaf(gs_s, part[a.k * RD + tid], y);
    a.y[r0 + tid] = y;
  }
}

}  // namespace

bool decode_supported(int d, int E, int k, int F) {
  const int k1 = k + 1;
  if (k1 > 32 || E > 1024 || F > 2048 || d > 4096) return false;
  // The down kernel gives each lane max(8, F/32) consecutive elements of a row and reduces over
  // F / that many lanes with a butterfly: F must be 128 times a power of two.
  if (F != 128 && F != 256 && F != 512 && F != 1024 && F != 2048) return false;
  return SmemA::bytes(d) <= 200 * 1024 && SmemB::bytes(k1, F) <= 200 * 1024;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st, bool pdl) {
  const int k1 = a.k + (a.has_shared ? 1 : 0);
  const size_t sa = SmemA::bytes(a.d), sb = SmemB::bytes(k1, a.F);
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(decode_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_down_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_down_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_down_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_down_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;

  cudaLaunchConfig_t ca = {};
  ca.gridDim = dim3(a.F / RF, k1);
  ca.blockDim = dim3(256);
  ca.dynamicSmemBytes = sa;
  ca.stream = st;
  ca.attrs = attr;
  ca.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&ca, decode_gateup_kernel, a);
  if (e != cudaSuccess) return e;

  cudaLaunchConfig_t cb = {};
  cb.gridDim = dim3(a.d / RD);
  cb.blockDim = dim3(256);
  cb.dynamicSmemBytes = sb;
  cb.stream = st;
  cb.attrs = attr;
  cb.numAttrs = 1;
  const int epl = a.F / 32 <= 8 ? 8 : a.F / 32;
  if (epl == 8) e = cudaLaunchKernelEx(&cb, decode_down_kernel<8>, a);
  else if (epl == 16) e = cudaLaunchKernelEx(&cb, decode_down_kernel<16>, a);
  else if (epl == 32) e = cudaLaunchKernelEx(&cb, decode_down_kernel<32>, a);
  else e = cudaLaunchKernelEx(&cb, decode_down_kernel<64>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
