// Decode (T = 1) MoE layer as two bandwidth-bound dequant-GEMV kernels.
//
// At batch 1 there is almost no weight reuse, so weight bandwidth sets the ceiling ("Perplexity
// libera Lily: inferencia en Rust y Metal para Mac", section "Decode: mover menos bytes por
// token"); the pages also report that removing all arithmetic from the kernels changed speed by
// 0.2% and that matrix ops reached 97.9% of bandwidth ("Perplexity открыла код Lily...",
// section "Спекулятивное декодирование не взлетело").  The design follows from that:
//
//   kernel A  grid (F/32, k + shared): every CTA redoes the top-k of the token's logits (1 KB
//             from L2) instead of waiting for a routing kernel, bulk-copies 32 gate rows and 32 up
//             rows of its expert (72 KB at d = 2048) into shared memory with one mbarrier, and
//             computes 32 SwiGLU outputs h in fp32.
//   kernel B  grid (d/16): every CTA redoes the top-k, bulk-copies 16 rows of the down matrix of
//             all k + 1 experts, then (after the programmatic-launch wait for kernel A) computes
//             y[r] = sum_j w_j (W_down[e_j] h_j)[r] + sigmoid(x . w_sg) (W_down_shared h_s)[r].
//   Kernel B is launched as a programmatic dependent of A: its CTAs start while A runs, so its
//   weight copies overlap A's and only the h read waits.  Kernel A issues its own
//   launch_dependents only after its griddepcontrol.wait, so everything B reads before its
//   wait (x, logits, weights) was complete before A started.
//
// Both kernels run once per SM per layer with cold instruction caches, so their code is kept
// small: rolled loops over rows and experts, one top-k routine over keys in shared memory with
// redux.sync max/min, no per-size template fan-out except the down kernel's lane width.
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
constexpr int kMaxE = 1024;
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

// One warp: top-k of logits[0..E) (descending, equal logits to the lower index, -0.0 == +0.0,
// NaN lowest) and the softmax of the selected logits.  Keys and values are staged in shared
// memory; each round takes the maximum key with redux.sync max and the lowest index holding it
// with redux.sync min, then clears that key.  Lane j < k returns expert j and its weight.
__device__ __forceinline__ void smem_topk(const float* __restrict__ logits, int E, int k, uint32_t* keys,
                                          float* vals, int* e_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < E; e += 32) {
    const float v = __ldg(logits + e);
    vals[e] = v;
    keys[e] = logit_key(v);
  }
  __syncwarp();
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t best = 0u;
    uint32_t bi = 0xFFFFFFFFu;
    for (int e = lane; e < E; e += 32) {
      const uint32_t kk = keys[e];
      if (kk > best) {   // strict: the first (lowest) index of this lane wins ties
        best = kk;
        bi = (uint32_t)e;
      }
    }
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, best);
    const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, best == m ? bi : 0xFFFFFFFFu);
    if (lane == j) my_e = (int)win;
    if (lane == (int)(win & 31u)) keys[win] = 0u;
    __syncwarp();
  }
  const float v0 = vals[__shfl_sync(0xFFFFFFFFu, my_e, 0)];
  const float ex = (lane < k) ? expf(vals[my_e] - v0) : 0.0f;
  float s = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
  *e_out = my_e;
  *w_out = ex / s;
}

struct SmemA {
  static size_t bytes(int d) {
    const int G = d / 64;
    return (size_t)2 * RF * (d / 2) + (size_t)4 * RF * G * 2 + 64;
  }
};

__global__ void __launch_bounds__(256) decode_gateup_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int d = a.d, G = d / 64;   // G <= 32: one quantisation group per lane
  const int j = blockIdx.y;         // 0..k-1 routed, k = shared
  const int f0 = blockIdx.x * RF;
  const bool is_shared = (j == a.k);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint32_t* codes_g = reinterpret_cast<uint32_t*>(sm);
  uint32_t* codes_u = codes_g + RF * (d / 8);
  uint16_t* sc_g = reinterpret_cast<uint16_t*>(codes_u + RF * (d / 8));
  uint16_t* bi_g = sc_g + RF * G;
  uint16_t* sc_u = bi_g + RF * G;
  uint16_t* bi_u = sc_u + RF * G;
  __shared__ uint32_t keys_s[kMaxE];
  __shared__ float vals_s[kMaxE];
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
    smem_topk(a.logits, a.E, a.k, keys_s, vals_s, &e, &w);
    if (lane == j) e_s = e;
    __syncwarp();
    if (lane == 0) issue(0, e_s);
  }
  pdl_launch_dependents();

  // Lane l owns group l (64 columns) of every row; its activations stay in registers.
  const bool active = lane < G;
  float xs[64];
  float xsum = 0.0f;
  if (active) {
    const uint4* xv = reinterpret_cast<const uint4*>(a.x) + lane * 8;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      const uint4 v = __ldg(xv + c8);
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
  const bool ok = mbar_wait_warp(sbar, 0, &abort_s, a.err);

  // Warp w computes rows 4w .. 4w+3 of gate (slots 0..3) and of up (slots 4..7); lane r keeps
  // the reduced value of slot r.
  float slot = 0.0f;
#pragma unroll 1
  for (int r = 0; r < 8; ++r) {
    const int row = 4 * warp + (r & 3);
    const bool up = r >= 4;
    float v = 0.0f;
    if (active && ok) {
      const uint32_t* cw = (up ? codes_u : codes_g) + row * (d / 8) + lane * 8;
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
      const float s = bf16_bits_to_f32((up ? sc_u : sc_g)[row * G + lane]);
      const float b = bf16_bits_to_f32((up ? bi_u : bi_g)[row * G + lane]);
      v = fmaf(s, p, b * xsum);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    if (lane == r) slot = v;
  }
  const float upv = __shfl_down_sync(0xFFFFFFFFu, slot, 4);
  if (lane < 4 && ok) {
    const float gv = slot;
    a.h[(size_t)j * a.F + f0 + 4 * warp + lane] = gv / (1.0f + expf(-gv)) * upv;
  }
}

struct SmemB {
  static size_t bytes(int k1, int F) {
    const int GF = F / 64;
    return (size_t)k1 * RD * (F / 2) + (size_t)2 * k1 * RD * GF * 2 + (size_t)k1 * F * 4 + 64;
  }
};

// EPL: elements of the reduction (F) per lane, max(8, F/32); LPR = F/EPL lanes cover one row.
template <int EPL>
__global__ void __launch_bounds__(256) decode_down_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int F = a.F, GF = F / 64;
  const int k1 = a.k + (a.has_shared ? 1 : 0);
  const int r0 = blockIdx.x * RD;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint32_t* codes = reinterpret_cast<uint32_t*>(sm);                        // [k1][RD][F/8]
  uint16_t* scl = reinterpret_cast<uint16_t*>(codes + k1 * RD * (F / 8));   // [k1][RD][GF]
  uint16_t* bia = scl + k1 * RD * GF;
  float* hs = reinterpret_cast<float*>(bia + k1 * RD * GF);                 // [k1][F]
  __shared__ uint32_t keys_s[kMaxE];
  __shared__ float vals_s[kMaxE];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int e_s[32];
  __shared__ float w_s[33];   // routing weights, then the shared-expert gate at [k]
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
  if (warp == 0) {
    if (a.has_shared && lane == 0) issue(a.k, 1, 0);
    int e;
    float w;
    smem_topk(a.logits, a.E, a.k, keys_s, vals_s, &e, &w);
    if (lane < a.k) {
      e_s[lane] = e;
      w_s[lane] = w;
    }
    __syncwarp();
    if (lane == 0)
      for (int jj = 0; jj < a.k; ++jj) issue(jj, 0, e_s[jj]);
  } else if (warp == 1 && a.has_shared) {
    float dot = 0.0f;
    const uint4* xv = reinterpret_cast<const uint4*>(a.x);
    const uint4* gv = reinterpret_cast<const uint4*>(a.w_sg);
    for (int c = lane; c < a.d / 8; c += 32) {
      const uint4 xq = __ldg(xv + c), gq = __ldg(gv + c);
      const uint32_t xw[4] = {xq.x, xq.y, xq.z, xq.w}, gw[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dot = fmaf(bf16_bits_to_f32(xw[i] & 0xFFFFu), bf16_bits_to_f32(gw[i] & 0xFFFFu), dot);
        dot = fmaf(bf16_bits_to_f32(xw[i] >> 16), bf16_bits_to_f32(gw[i] >> 16), dot);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
    if (lane == 0) w_s[a.k] = 1.0f / (1.0f + expf(-dot));
  }
  pdl_wait();   // h from kernel A is complete and visible past this point
  {
    const float4* h4 = reinterpret_cast<const float4*>(a.h);
    float4* hs4 = reinterpret_cast<float4*>(hs);
    const int n4 = k1 * F / 4;
#pragma unroll 4
    for (int i = tid; i < n4; i += 256) hs4[i] = h4[i];
  }
  __syncthreads();
  const bool ok = mbar_wait_warp(sbar, 0, &abort_s, a.err);

  // Warp w owns rows 2w and 2w+1 of this CTA's 16; LPR lanes cover a row, RPW rows at a time.
  const int lpr = F / EPL;           // 16 (F = 128) or 32
  const int rpw = 32 / lpr;          // 2 or 1
  const int sub = lane / lpr, l = lane % lpr;
  const int c0 = l * EPL;            // first element of this lane's range
  const int grp = c0 / 64;
  for (int it = 0; it < 2 / rpw; ++it) {
    const int r = 2 * warp + it * rpw + sub;
    float acc = 0.0f;
#pragma unroll 1
    for (int jj = 0; jj < k1; ++jj) {
      float hv[EPL];
      float hsum = 0.0f;
      const float4* hp = reinterpret_cast<const float4*>(hs + jj * F + c0);
#pragma unroll
      for (int c4 = 0; c4 < EPL / 4; ++c4) {
        const float4 v = hp[c4];
        hsum += (v.x + v.y) + (v.z + v.w);
        hv[4 * c4 + 0] = v.x * act_prescale(4 * c4 + 0);
        hv[4 * c4 + 1] = v.y * act_prescale(4 * c4 + 1);
        hv[4 * c4 + 2] = v.z * act_prescale(4 * c4 + 2);
        hv[4 * c4 + 3] = v.w * act_prescale(4 * c4 + 3);
      }
      const uint32_t* cw = codes + (jj * RD + r) * (F / 8) + c0 / 8;
      float p = 0.0f;
#pragma unroll
      for (int wd = 0; wd < EPL / 8; ++wd) p = word_dot(cw[wd], hv + 8 * wd, p);
      const float s = bf16_bits_to_f32(scl[(jj * RD + r) * GF + grp]);
      const float b = bf16_bits_to_f32(bia[(jj * RD + r) * GF + grp]);
      acc = fmaf(w_s[jj], fmaf(s, p, b * hsum), acc);
    }
    for (int off = lpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (l == 0 && ok) a.y[r0 + r] = acc;
  }
}

}  // namespace

bool decode_supported(int d, int E, int k, int F) {
  const int k1 = k + 1;
  // One 64-column group per lane in kernel A: d <= 2048.
  if (k1 > 32 || E > kMaxE || F > 2048 || d > 2048) return false;
  // The down kernel gives each lane max(8, F/32) consecutive elements of a row and reduces over
  // F / that many lanes with a butterfly: F must be 128 times a power of two.
  if (F != 128 && F != 256 && F != 512 && F != 1024 && F != 2048) return false;
  return SmemA::bytes(d) <= 180 * 1024 && SmemB::bytes(k1, F) <= 180 * 1024;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st, bool pdl) {
  const int k1 = a.k + (a.has_shared ? 1 : 0);
  const size_t sa = SmemA::bytes(a.d), sb = SmemB::bytes(k1, a.F);
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    const int lim = 180 * 1024;
    cudaError_t e = cudaFuncSetAttribute(decode_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_down_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_down_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_down_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_down_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
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
