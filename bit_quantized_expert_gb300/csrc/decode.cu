// Decode MoE layer (one token, or a few: T <= 8) as one bandwidth-bound dequant-GEMV kernel.
//
// At batch 1 there is almost no weight reuse, so weight bandwidth sets the ceiling ("Perplexity
// libera Lily: inferencia en Rust y Metal para Mac", section "Decode: mover menos bytes por
// token"); the pages also report that removing all arithmetic from the kernels changed speed by
// 0.2% and that matrix ops reached 97.9% of bandwidth ("Perplexity открыла код Lily...",
// section "Спекулятивное декодирование не взлетело").  On a GB300 one layer's routed weights
// (~16 MB) stream in ~2.3 us, so the layer is as much a latency chain as a bandwidth problem:
// the design keeps that chain short.
//
// One cooperative launch per layer; CTA c (grid = (k+1) F / 32, one per SM, all co-resident)
// owns rows f0 = 32 (c mod F/32) .. f0+31 of expert slot j = c / (F/32) (k = the shared expert):
//   * before the programmatic-launch wait, shared-expert CTAs start their weight copies (weights
//     are never written upstream, so they may be read early);
//   * after it, warp 0 routes the token in registers (top-k of the 1 KB of logits; cheaper than a
//     routing kernel and its launch) and starts the bulk copies of the 32 gate rows and 32 up rows
//     (four quarters, one mbarrier each, so compute starts on the first quarter), while every
//     thread copies the matching 32-column block of the down matrix (all d rows, 16 B each) with
//     cp.async, and one thread bulk-copies the expert's down scales and biases whole (contiguous,
//     so two large requests replace two small ones per row);
//   * the CTA computes its 32 SwiGLU outputs h, then its share of the down projection,
//     part_c[r] = w_j * sum_{f in f0..f0+31} W_down[e_j][r][f] h[f] for every output row r
//     (a split over F: no CTA needs another CTA's h);
//   * every CTA writes part_c and arrives at a grid barrier (one 64-bit word: arrivals in the low
//     half, a generation count in the high half; the last arrival resets the count and bumps the
//     generation), then sums a slice of rows over all CTAs in a fixed order:
//     y[r] = sum_c part_c[r] -- deterministic, no atomics on data.
//
// A few tokens (T > 1, the kernel<true> instantiation): warp t routes token t; every CTA then
// takes its expert slot of token 0, 1, ... in turn, fetching the slot's weights again only when
// its expert changes (the shared expert's stay), and writes part_c per token; one grid barrier
// and one fixed-order reduction serve all tokens, so each token's y is what a one-token launch
// gives, bit for bit.  The one-token launch is the kernel<false> instantiation (T fixed at 1).
//
// Arithmetic: codes become exact fp32 values q * 16^e via the 2^23 exponent trick (the nibble
// stays where it is in the word; the activation carries the matching 16^-e), partial dot
// products sum_c q_c x_c accumulate in fp32 with packed two-lane FMAs, and w = q*s + b enters as
// s * sum(q x) + b * sum(x) per quantisation group (per half group for the down rows).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int RF = 32;   // gate/up rows (and down columns) per CTA
constexpr int kQuarters = 4;
constexpr int kRQ = RF / kQuarters;   // gate/up rows per quarter
constexpr int kMaxE = 1024;
constexpr float kMagic = 8388608.0f;   // 2^23
constexpr int kThreadsDec = 256;

// Activation pre-scale matching the position of code n (0..7) of a word after extraction.
__host__ __device__ constexpr float act_prescale(int n) {
  return n % 8 == 0 ? 1.0f : n % 8 == 1 ? 0.0625f : n % 8 == 2 ? 0.00390625f : n % 8 == 3 ? 0.000244140625f
       : n % 8 == 4 ? 1.52587890625e-05f : n % 8 == 5 ? 0.00390625f : n % 8 == 6 ? 0.000244140625f
       : 1.52587890625e-05f;
}

__device__ __forceinline__ float2 magic_pair(uint32_t a, uint32_t b) {
  return make_float2(__uint_as_float(a | 0x4B000000u), __uint_as_float(b | 0x4B000000u));
}

// acc += sum over the 8 codes of word w of q_c * xs[c] (xs pre-scaled by act_prescale), as four
// packed pairs (codes 0,1 / 2,3 / 4,5 / 6,7).  Codes 5..7 are taken from w >> 12 so that every
// extracted value stays below 2^20 and is exact.
__device__ __forceinline__ float2 word_dot2(uint32_t w, const float2* xs, float2 acc) {
  const uint32_t w12 = w >> 12;
  const float2 m = make_float2(-kMagic, -kMagic);
  acc = __ffma2_rn(__fadd2_rn(magic_pair(w & 0xFu, w & 0xF0u), m), xs[0], acc);
  acc = __ffma2_rn(__fadd2_rn(magic_pair(w & 0xF00u, w & 0xF000u), m), xs[1], acc);
  acc = __ffma2_rn(__fadd2_rn(magic_pair(w & 0xF0000u, w12 & 0xF00u), m), xs[2], acc);
  acc = __ffma2_rn(__fadd2_rn(magic_pair(w12 & 0xF000u, w12 & 0xF0000u), m), xs[3], acc);
  return acc;
}

// Shared-memory plan of one CTA (byte offsets, 16-byte aligned regions).
struct DecPlan {
  int d, F, k1, G, GF, grid;
  bool bulk_sb;   // the down scales and biases of the expert copied whole (two bulk copies)
  uint32_t gu_codes, gu_sb, dn_codes, dn_sb, hbuf, bytes;
  __host__ __device__ DecPlan(int d_, int F_, int k1_) : d(d_), F(F_), k1(k1_) {
    G = d / 64;
    GF = F / 64;
    grid = k1 * (F / RF);
    bulk_sb = 4u * (uint32_t)d * (uint32_t)GF <= 64u * 1024u;
    uint32_t o = 0;
    gu_codes = o;  o += 2u * RF * (d / 2);   // [gate|up][RF][d/8] u32
    gu_sb = o;     o += 4u * RF * G * 2;     // [g.s|g.b|u.s|u.b][RF][G] bf16
    o = (o + 15u) & ~15u;
    dn_codes = o;  o += 16u * d;             // [d][4] u32: code words f0/8 .. f0/8+3 of every row
    dn_sb = o;                               // [s|b][d][GF] bf16 (whole matrices), or
    o += bulk_sb ? 4u * d * GF : 8u * d;     // [s|b][d] u32: the bf16 pair holding group f0/64
    hbuf = o;      o += 4u * RF;             // h of rows f0 .. f0+31, fp32
    bytes = (o + 15u) & ~15u;
  }
};

// Warp-wide top-k of logits[0..E) and the softmax of the selected logits, with the candidates
// held in registers (8 per lane up to E = 256, else 32); lane j < k returns expert j and its
// weight.
__device__ __forceinline__ void reg_topk(const float* __restrict__ logits, int E, int k, int* e_out, float* w_out) {
  if (E <= 256) warp_topk_softmax<8>(logits, E, k, e_out, w_out);
  else warp_topk_softmax<32>(logits, E, k, e_out, w_out);
}

__device__ __forceinline__ unsigned long long atom_add_release(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.release.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// kMulti = false: one token (T fixed at 1, so the token loop and the per-token arrays fold away).
template <bool kMulti>
__global__ void __launch_bounds__(kThreadsDec, 1) decode_layer_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int d = a.d, F = a.F, k = a.k;
  const int k1 = k + (a.has_shared ? 1 : 0);
  const DecPlan P(d, F, k1);
  const int G = P.G, GF = P.GF;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int jobs = F / RF;
  const int j = cta / jobs;            // expert slot: 0..k-1 routed, k shared
  const int f0 = (cta % jobs) * RF;    // first gate/up row = first down column
  const bool shared_cta = (j == k);
  const int wset = shared_cta ? 1 : 0;

  uint32_t* gcodes = reinterpret_cast<uint32_t*>(sm + P.gu_codes);   // gate [RF][d/8], then up
  uint16_t* gsb = reinterpret_cast<uint16_t*>(sm + P.gu_sb);         // [g.s | g.b | u.s | u.b][RF][G]
  uint32_t* dcodes = reinterpret_cast<uint32_t*>(sm + P.dn_codes);   // [d][4]
  uint32_t* dsb = reinterpret_cast<uint32_t*>(sm + P.dn_sb);         // [s | b][d] (pairs), or
  uint16_t* dsb16 = reinterpret_cast<uint16_t*>(sm + P.dn_sb);       // [s | b][d][GF] (whole)
  float* hbuf = reinterpret_cast<float*>(sm + P.hbuf);               // [RF]
  __shared__ __align__(8) uint64_t bars[kQuarters + 1];   // gate/up quarters, then the down scales
  __shared__ int e_s[kDecodeMaxTokens];
  __shared__ float wgt_s[kDecodeMaxTokens];    // w_j (routed) or the shared-expert gate, per token
  __shared__ int abort_s;
  const int T = kMulti ? (a.T > 0 ? a.T : 1) : 1;

  if (tid == 0) {
    for (int i = 0; i <= kQuarters; ++i) mbar_init(smem_u32(&bars[i]), 1);
    abort_s = 0;
    mbar_fence_init();
  }
  __syncthreads();

  // Gate and up rows f0 .. f0+31 of expert e (code words by quarter; scales and biases with the
  // first quarter).
  auto issue_gu = [&](int e) {
    const QPtr& g = a.gate[wset];
    const QPtr& u = a.up[wset];
    const uint32_t cb = kRQ * (d / 2), sb = RF * G * 2;
    const size_t rowb = (size_t)e * F + f0;
    for (int q = 0; q < kQuarters; ++q) {
      const uint32_t bar = smem_u32(&bars[q]);
      const size_t row0 = rowb + q * kRQ;
      mbar_arrive_expect_tx(bar, 2 * cb + (q == 0 ? 4 * sb : 0));
      if (q == 0) {
        bulk_g2s(smem_u32(gsb + 0 * RF * G), g.scales + rowb * G, sb, bar);
        bulk_g2s(smem_u32(gsb + 1 * RF * G), g.biases + rowb * G, sb, bar);
        bulk_g2s(smem_u32(gsb + 2 * RF * G), u.scales + rowb * G, sb, bar);
        bulk_g2s(smem_u32(gsb + 3 * RF * G), u.biases + rowb * G, sb, bar);
      }
      bulk_g2s(smem_u32(gcodes + (q * kRQ) * (d / 8)), g.codes + row0 * (d / 8), cb, bar);
      bulk_g2s(smem_u32(gcodes + (RF + q * kRQ) * (d / 8)), u.codes + row0 * (d / 8), cb, bar);
    }
  };
  // Columns f0 .. f0+31 of every row of the down matrix of expert e: 16 code bytes per row, and
  // the row's scale and bias of group f0/64 -- where they fit, as the expert's whole scale and
  // bias matrices (two contiguous bulk copies instead of two small requests per row), else as the
  // 4-byte aligned bf16 pairs holding the group.
  auto copy_dn = [&](int e) {
    const QPtr& q = a.down[wset];
    if (P.bulk_sb) {
      if (tid == 0) {
        const uint32_t bar = smem_u32(&bars[kQuarters]);
        const uint32_t nb = 2u * d * GF;
        mbar_arrive_expect_tx(bar, 2u * nb);
        bulk_g2s(smem_u32(dsb16), q.scales + (size_t)e * d * GF, nb, bar);
        bulk_g2s(smem_u32(dsb16 + d * GF), q.biases + (size_t)e * d * GF, nb, bar);
      }
    }
    const int g2 = (f0 / 64) & ~1;
    for (int r = tid; r < d; r += kThreadsDec) {
      const size_t row = (size_t)e * d + r;
      cp_async_16(smem_u32(dcodes + 4 * r), q.codes + row * (F / 8) + f0 / 8);
      if (!P.bulk_sb) {
        cp_async_4(smem_u32(dsb + r), q.scales + row * GF + g2);
        cp_async_4(smem_u32(dsb + d + r), q.biases + row * GF + g2);
      }
    }
    cp_async_commit();
  };

  // Weights are never written upstream: the shared expert's copies start before the wait.
  if (shared_cta) {
    if (tid == 0) issue_gu(0);
    copy_dn(0);
  }
  pdl_wait();   // x and logits from upstream kernels are complete and visible past this point

  if (warp < T && !shared_cta) {
    // warp t routes token t; token 0's weights are requested as soon as its expert is known
    int e;
    float w;
    reg_topk(a.logits + (size_t)warp * a.E, a.E, k, &e, &w);
    const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
    const float wj = __shfl_sync(0xFFFFFFFFu, w, j);
    if (lane == 0) {
      e_s[warp] = ej;
      wgt_s[warp] = wj;
      if (warp == 0) issue_gu(ej);
    }
  } else if (shared_cta) {
    // warp w: the shared-expert gates of tokens w, w + 8, ...
    for (int t = warp; t < T; t += kThreadsDec / 32) {
      float dot = 0.0f;
      const uint4* xv = reinterpret_cast<const uint4*>(a.x + (size_t)t * d);
      const uint4* gv = reinterpret_cast<const uint4*>(a.w_sg);
      for (int c = lane; c < d / 8; c += 32) {
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
      if (lane == 0) {
        e_s[t] = 0;
        wgt_s[t] = 1.0f / (1.0f + expf(-dot));
      }
    }
  }
  pdl_launch_dependents();
  __syncthreads();   // e_s and wgt_s
  // Tokens one after another.  The slot's weights stay in shared memory while the slot's expert
  // stays the same (always for the shared expert), and are fetched again when it changes; every
  // fetch is one phase of the copy barriers, so waits use the parity of the fetch count.
  const bool active = lane < G;
  int loads = 1;   // weight fetches so far (token 0's is in flight)
#pragma unroll 1
  for (int t = 0; t < T; ++t) {
    if (t > 0 && abort_s) break;   // uniform: abort_s is only written inside waits, before the barrier below
    const int e_t = e_s[t];
    if (t > 0 && e_t != e_s[t - 1]) ++loads;   // gate/up rows requested during the last down phase
    const uint32_t ph = (uint32_t)(loads - 1) & 1u;
    // x: lane l owns quantisation group l (64 inputs).  For token 0 the loads go out after
    // routing, so the logits are the first reads behind the dependency wait, and before the down
    // copies; the gate/up products wait for the weights, which arrive later.
    uint4 xr[8];
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8)
      xr[c8] = active ? __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * d) + lane * 8 + c8)
                      : make_uint4(0u, 0u, 0u, 0u);
    if ((t == 0 && !shared_cta) || (t > 0 && e_t != e_s[t - 1])) copy_dn(e_t);

    // ---- gate/up: warp w computes gate and up of rows q*8 + w (q = 0..3) as slots s = 2q + mat;
    // a reduce-scatter leaves slot s fully summed in lane 4s.
    float2 xs[32];
    float xsum = 0.0f;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      const uint32_t wv[4] = {xr[c8].x, xr[c8].y, xr[c8].z, xr[c8].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = bf16_bits_to_f32(wv[i] & 0xFFFFu), hi = bf16_bits_to_f32(wv[i] >> 16);
        xsum += lo + hi;
        xs[c8 * 4 + i] = make_float2(lo * act_prescale(2 * i), hi * act_prescale(2 * i + 1));
      }
    }
    float v8[8];
#pragma unroll
    for (int sl = 0; sl < 8; ++sl) v8[sl] = 0.0f;
    bool ok_all = true;
#pragma unroll 1
    for (int q = 0; q < kQuarters; ++q) {
      const bool ok = mbar_wait_warp(smem_u32(&bars[q]), ph, &abort_s, a.err);
      ok_all = ok_all && ok;
#pragma unroll
      for (int mat = 0; mat < 2; ++mat) {
        const int row = q * kRQ + warp;
        float v = 0.0f;
        if (active && ok) {
          const uint32_t* cw = gcodes + (mat * RF + row) * (d / 8) + lane * 8;
          const uint4 c0 = *reinterpret_cast<const uint4*>(cw);
          const uint4 c1 = *reinterpret_cast<const uint4*>(cw + 4);
          float2 p0 = make_float2(0.0f, 0.0f), p1 = make_float2(0.0f, 0.0f);
          p0 = word_dot2(c0.x, xs + 0, p0);
          p1 = word_dot2(c0.y, xs + 4, p1);
          p0 = word_dot2(c0.z, xs + 8, p0);
          p1 = word_dot2(c0.w, xs + 12, p1);
          p0 = word_dot2(c1.x, xs + 16, p0);
          p1 = word_dot2(c1.y, xs + 20, p1);
          p0 = word_dot2(c1.z, xs + 24, p0);
          p1 = word_dot2(c1.w, xs + 28, p1);
          const float p = (p0.x + p0.y) + (p1.x + p1.y);
          const float s = bf16_bits_to_f32(gsb[((2 * mat) * RF + row) * G + lane]);
          const float b = bf16_bits_to_f32(gsb[((2 * mat + 1) * RF + row) * G + lane]);
          v = fmaf(s, p, b * xsum);
        }
        const int sl = 2 * q + mat;
#pragma unroll
        for (int t = 0; t < 8; ++t) v8[t] = (t == sl) ? v : v8[t];
      }
    }
    {
      float t4[4], t2[2];
      const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        t4[i] = (b4 ? v8[i + 4] : v8[i]) + __shfl_xor_sync(0xFFFFFFFFu, b4 ? v8[i] : v8[i + 4], 16);
#pragma unroll
      for (int i = 0; i < 2; ++i)
        t2[i] = (b3 ? t4[i + 2] : t4[i]) + __shfl_xor_sync(0xFFFFFFFFu, b3 ? t4[i] : t4[i + 2], 8);
      float t1 = (b2 ? t2[1] : t2[0]) + __shfl_xor_sync(0xFFFFFFFFu, b2 ? t2[0] : t2[1], 4);
      t1 += __shfl_xor_sync(0xFFFFFFFFu, t1, 2);
      t1 += __shfl_xor_sync(0xFFFFFFFFu, t1, 1);
      const float upv = __shfl_down_sync(0xFFFFFFFFu, t1, 4);   // slot 2q+1 (lane 8q+4) -> lane 8q
      if ((lane & 7) == 0) {
        const float gv = t1;
        hbuf[(lane >> 3) * kRQ + warp] = gv / (1.0f + expf(-gv)) * upv;
      }
    }
    cp_async_wait<0>();
    const bool ok_dn = !P.bulk_sb || mbar_wait_warp(smem_u32(&bars[kQuarters]), ph, &abort_s, a.err);
    __syncthreads();   // h and this thread's down copies -> visible to the whole CTA
    // The gate/up buffers are free from here on (the down share reads h and the down buffers):
    // request the next token's gate/up rows now, so they arrive during this token's down share.
    // abort_s cannot change after the barrier above (no waits follow in this token).
    if (kMulti && tid == 0 && t + 1 < T && e_s[t + 1] != e_t && !abort_s) {
      fence_proxy_async_smem();   // this token's reads of the gate/up buffers are complete
      issue_gu(e_s[t + 1]);
    }

    // ---- down share: part_c[r] = wgt * (s * sum_f q h_f + b * sum_f h_f) over f0 .. f0+31.
    {
      float2 hv[16];
      float hsum = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float hx = hbuf[2 * i], hy = hbuf[2 * i + 1];
        hsum += hx + hy;
        hv[i] = make_float2(hx * act_prescale(2 * i), hy * act_prescale(2 * i + 1));
      }
      const float wgt = wgt_s[t];
      const bool hi_half = ((f0 / 64) & 1) != 0;   // group f0/64 is the upper bf16 of its pair
      const int g = f0 / 64;
      for (int r = tid; r < d && ok_dn; r += kThreadsDec) {
        const uint4 c = *reinterpret_cast<const uint4*>(dcodes + 4 * r);
        float2 p0 = make_float2(0.0f, 0.0f), p1 = make_float2(0.0f, 0.0f);
        p0 = word_dot2(c.x, hv + 0, p0);
        p1 = word_dot2(c.y, hv + 4, p1);
        p0 = word_dot2(c.z, hv + 8, p0);
        p1 = word_dot2(c.w, hv + 12, p1);
        const float p = (p0.x + p0.y) + (p1.x + p1.y);
        float s, b;
        if (P.bulk_sb) {
          s = bf16_bits_to_f32(dsb16[r * GF + g]);
          b = bf16_bits_to_f32(dsb16[(d + r) * GF + g]);
        } else {
          const uint32_t sp = dsb[r], bp = dsb[d + r];
          s = bf16_bits_to_f32(hi_half ? (sp >> 16) : (sp & 0xFFFFu));
          b = bf16_bits_to_f32(hi_half ? (bp >> 16) : (bp & 0xFFFFu));
        }
        a.part[((size_t)t * gridDim.x + cta) * d + r] = wgt * fmaf(s, p, b * hsum);
      }
    }
    __syncthreads();   // this token's reads of the weight buffers and of h are complete
  }

  // ---- grid barrier: every CTA arrives once; the last arrival resets the count and bumps the
  // generation in one atomic.  The partial stores are ordered before the arrival by the block
  // barrier and the fence; the acquire load and fence order the reads below after it.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned long long n = gridDim.x;
    const unsigned long long old = atom_add_release(a.sync, 1ull);
    if ((old & 0xFFFFFFFFull) == n - 1ull) atom_add_release(a.sync, (1ull << 32) - n);
    const unsigned long long g0 = old >> 32;
    const long long t0 = clock64();
    while ((ld_acquire(a.sync) >> 32) == g0) {
      if (clock64() - t0 > kWaitTimeoutCycles) {
        abort_s = 1;
        raise_flag(a.err, kErrWaitTimeout);
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();

  // ---- y rows of this CTA: sum of all CTAs' partials in a fixed order (16 lanes per row, each
  // summing every 16th CTA in increasing order, then a fixed butterfly).  The first ten loads of
  // a lane go out together (one L2 round trip for grids up to 160 CTAs).
  if (!abort_s) {
    const int n = gridDim.x;
    const int rpc = (d + n - 1) / n;
    const int r_lo = cta * rpc, r_hi = min(d, r_lo + rpc);
    const int sub = tid & 15;
#pragma unroll 1
    for (int t = 0; t < T; ++t)
    for (int rb = r_lo; rb < r_hi; rb += kThreadsDec / 16) {
      const float* part = a.part + (size_t)t * n * d;
      const int r = rb + (tid >> 4);
      float acc = 0.0f;
      if (r < r_hi) {
        float v[10];
#pragma unroll
        for (int i = 0; i < 10; ++i) {
          const int c = sub + 16 * i;
          v[i] = c < n ? __ldcg(part + (size_t)c * d + r) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 10; ++i) acc += v[i];
        for (int c = sub + 160; c < n; c += 16) acc += __ldcg(part + (size_t)c * d + r);
      }
      acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 8);
      acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 4);
      acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 2);
      acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
      if (sub == 0 && r < r_hi) a.y[(size_t)t * d + r] = acc;
    }
  }

  // ---- wind down: after a timeout, copies still in flight must land before the CTA exits.
  if (tid == 0 && abort_s) {
    const uint32_t last = (uint32_t)(loads - 1) & 1u;   // parity of the last fetch issued
    for (int i = 0; i <= kQuarters; ++i) {
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(&bars[i]), last) && clock64() - t0 < 4000000ll) {
      }
    }
  }
}

struct DevInfo {
  int sms = 0;
  bool ready = false;
};
constexpr int kMaxDev = 64;
DevInfo g_dev[kMaxDev];
std::mutex g_dev_mu;
constexpr size_t kDecSmemMax = 200 * 1024;

cudaError_t dev_info(DevInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& di = g_dev[dev];
  if (!di.ready) {
    if ((e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_layer_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecSmemMax);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_layer_kernel<false>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_layer_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecSmemMax);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_layer_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    di.ready = true;
  }
  *out = &di;
  return cudaSuccess;
}

}  // namespace

size_t decode_scratch_floats(int d, int k, int F) { return (size_t)(k + 1) * (F / RF) * d; }

bool decode_supported(int d, int E, int k, int F) {
  const int k1 = k + 1;
  // One quantisation group per lane in the gate/up rows: d <= 2048 (and d a multiple of 64).
  // F a multiple of 128: the down columns f0 .. f0+31 of a CTA lie in one bf16 pair of
  // scale (bias) values that starts on a 4-byte boundary (F / 64 even).
  if (k1 > 32 || E > kMaxE || d > 2048 || d % 64 != 0 || F % 128 != 0) return false;
  const DecPlan P(d, F, k1);
  if (P.bytes > kDecSmemMax) return false;
  // Every CTA must be resident at once (one per SM): the grid barrier waits on all of them.
  DevInfo* di = nullptr;
  if (dev_info(&di) != cudaSuccess) return false;
  return P.grid <= di->sms;
}

constexpr int kStageThreads = 256;
constexpr int kStageIn = 4;   // loads in flight per thread per round

__global__ void __launch_bounds__(kStageThreads) stage_in_kernel(const StageArgs a) {
  pdl_wait();   // the previous kernel, the last reader of the destination buffers, is complete
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  for (int base = 0; base < a.x_units; base += kStageThreads * kStageIn) {
    uint4 v[kStageIn];
#pragma unroll
    for (int c = 0; c < kStageIn; ++c) {
      const int i = base + c * kStageThreads + tid;
      if (i < a.x_units) v[c] = a.x_src[i];
    }
#pragma unroll
    for (int c = 0; c < kStageIn; ++c) {
      const int i = base + c * kStageThreads + tid;
      if (i < a.x_units) a.x_dst[i] = v[c];
    }
  }
  for (int base = 0; base < a.lg_n; base += kStageThreads * kStageIn) {
    float v[kStageIn];
#pragma unroll
    for (int c = 0; c < kStageIn; ++c) {
      const int i = base + c * kStageThreads + tid;
      if (i < a.lg_n) v[c] = a.lg_src[i];
    }
#pragma unroll
    for (int c = 0; c < kStageIn; ++c) {
      const int i = base + c * kStageThreads + tid;
      if (i < a.lg_n) a.lg_dst[i] = v[c];
    }
  }
}

cudaError_t launch_stage_in(const StageArgs& a, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kStageThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, stage_in_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

static_assert(kDecodeMaxTokens <= kThreadsDec / 32, "one routing warp per token");
static_assert(kDecodeLayerMaxT <= kDecodeMaxTokens, "the layer path's decode calls fit one launch");

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st, bool pdl) {
  if (a.T > kDecodeMaxTokens) return cudaErrorInvalidValue;
  const int k1 = a.k + (a.has_shared ? 1 : 0);
  DevInfo* di = nullptr;
  cudaError_t e = dev_info(&di);
  if (e != cudaSuccess) return e;
  const DecPlan P(a.d, a.F, k1);
  if (P.grid > di->sms || P.bytes > kDecSmemMax) return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid);
  cfg.blockDim = dim3(kThreadsDec);
  cfg.dynamicSmemBytes = P.bytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  e = a.T > 1 ? cudaLaunchKernelEx(&cfg, decode_layer_kernel<true>, a) : cudaLaunchKernelEx(&cfg, decode_layer_kernel<false>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
