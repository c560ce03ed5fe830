// Decode (T = 1) MoE layer as one bandwidth-bound dequant-GEMV kernel.
//
// At batch 1 there is almost no weight reuse, so weight bandwidth sets the ceiling ("Perplexity
// libera Lily: inferencia en Rust y Metal para Mac", section "Decode: mover menos bytes por
// token"); the pages also report that removing all arithmetic from the kernels changed speed by
// 0.2% and that matrix ops reached 97.9% of bandwidth ("Perplexity открыла код Lily...",
// section "Спекулятивное декодирование не взлетело").  On a GB300 one layer's routed weights
// (~16 MB) stream in ~2.3 us, so the layer is as much a latency chain as a bandwidth problem:
// the design removes every step of that chain that is not a weight byte in flight.
//
// One cooperative launch per layer, one CTA per SM (grid = max(jobs), all CTAs co-resident):
//   * before the programmatic-launch wait, every CTA starts the bulk copies of the shared
//     expert's rows it owns (weights are never written upstream, so they may be read early);
//   * after it, every CTA redoes the top-k of the token's logits in registers (1 KB from L2;
//     cheaper than a routing kernel and its launch) and starts the copies of its routed rows:
//       gate/up job c < (k+1) F / 32: 32 gate rows and the 32 up rows of expert slot c / (F/32),
//         copied in four quarters with one mbarrier each, so compute starts on the first quarter;
//       down job c < d / 16: rows 16c .. 16c+15 of the down matrix of all k + 1 experts;
//   * gate/up jobs write their 32 SwiGLU outputs h (fp32) to global memory, then every CTA
//     arrives at a grid barrier (one 64-bit word: arrivals in the low half, a generation count
//     in the high half; the last arrival resets the count and bumps the generation);
//   * down jobs wait for the generation to move, read all (k + 1) F values of h from L2 into
//     shared memory and compute y[r] = sum_j w_j (W_down[e_j] h_j)[r] + g_s (W_down_s h_s)[r].
//
// Arithmetic: codes become exact fp32 values q * 16^e via the 2^23 exponent trick (the nibble
// stays where it is in the word; the activation carries the matching 16^-e), partial dot
// products sum_c q_c x_c accumulate in fp32 with packed two-lane FMAs, and w = q*s + b enters as
// s * sum(q x) + b * sum(x) per quantisation group.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int RF = 32;   // gate/up rows per job
constexpr int RD = 16;   // down rows per job
constexpr int kQuarters = 4;
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

// Shared-memory plan of one CTA (byte offsets; every region 16-byte aligned).
struct DecPlan {
  int d, F, k1, G, GF, epl, segs;
  uint32_t gu_codes, gu_sb, dn_codes, dn_sb, h, hsum, bytes;
  __host__ __device__ DecPlan(int d_, int F_, int k1_) : d(d_), F(F_), k1(k1_) {
    G = d / 64;
    GF = F / 64;
    epl = F / 32 <= 8 ? 8 : F / 32;   // down-row elements per lane
    segs = F / epl;                   // lanes covering one down row
    uint32_t o = 0;
    gu_codes = o;  o += 2u * RF * (d / 2);                 // [gate|up][RF][d/8] u32
    gu_sb = o;     o += 4u * RF * G * 2;                   // [g.s|g.b|u.s|u.b][RF][G] bf16
    o = (o + 15u) & ~15u;
    dn_codes = o;  o += (uint32_t)k1 * RD * (F / 2);       // [k1][RD][F/8] u32
    dn_sb = o;     o += 2u * k1 * RD * GF * 2;             // [s|b][k1][RD][GF] bf16
    o = (o + 15u) & ~15u;
    h = o;         o += (uint32_t)k1 * segs * (epl + 4) * 4;   // [k1][segs][epl + 4] fp32, padded
    hsum = o;      o += (uint32_t)k1 * segs * 4;               // [k1][segs] fp32
    bytes = (o + 15u) & ~15u;
  }
};

// One warp: top-k of logits[0..E) and the softmax of the selected logits, with the candidates
// held in registers (8 per lane up to E = 256, else 32); lane j < k returns expert j and its weight.
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

// EPL: elements of one down row per lane, max(8, F / 32); F / EPL lanes cover one row.
template <int EPL>
__global__ void __launch_bounds__(kThreadsDec, 1) decode_layer_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int d = a.d, F = a.F, k = a.k;
  const int k1 = k + (a.has_shared ? 1 : 0);
  const DecPlan P(d, F, k1);
  const int G = P.G, GF = P.GF;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int jobs_per_expert = F / RF;
  const bool has_gu = cta < k1 * jobs_per_expert;
  const bool has_dn = cta < d / RD;
  const int j = has_gu ? cta / jobs_per_expert : 0;   // expert slot: 0..k-1 routed, k shared
  const int f0 = has_gu ? (cta % jobs_per_expert) * RF : 0;
  const int r0 = cta * RD;

  uint32_t* gcodes = reinterpret_cast<uint32_t*>(sm + P.gu_codes);   // gate [RF][d/8], then up
  uint16_t* gsb = reinterpret_cast<uint16_t*>(sm + P.gu_sb);         // [g.s | g.b | u.s | u.b][RF][G]
  uint32_t* dcodes = reinterpret_cast<uint32_t*>(sm + P.dn_codes);   // [k1][RD][F/8]
  uint16_t* dsb = reinterpret_cast<uint16_t*>(sm + P.dn_sb);         // [s | b][k1][RD][GF]
  float* hs = reinterpret_cast<float*>(sm + P.h);                    // [k1][segs][EPL + 4]
  float* hsum_s = reinterpret_cast<float*>(sm + P.hsum);             // [k1][segs]
  __shared__ __align__(8) uint64_t bars[kQuarters + 1];
  __shared__ int e_s[32];
  __shared__ float w_s[33];   // routing weights, then the shared-expert gate at [k]
  __shared__ int abort_s;
  __shared__ unsigned long long gen_s;

  if (tid == 0) {
    for (int i = 0; i <= kQuarters; ++i) mbar_init(smem_u32(&bars[i]), 1);
    abort_s = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const uint32_t bar_dn = smem_u32(&bars[kQuarters]);

  // Gate and up rows f0 .. f0+31 of expert e of weight set `which`, in quarters of 8 rows.
  auto issue_gu = [&](int which, int e) {
    const QPtr& g = a.gate[which];
    const QPtr& u = a.up[which];
    constexpr int rq = RF / kQuarters;
    const uint32_t cb = rq * (d / 2), sb = rq * G * 2;
    for (int q = 0; q < kQuarters; ++q) {
      const uint32_t bar = smem_u32(&bars[q]);
      const size_t row0 = (size_t)e * F + f0 + q * rq;
      mbar_arrive_expect_tx(bar, 2 * cb + 4 * sb);
      bulk_g2s(smem_u32(gcodes + (q * rq) * (d / 8)), g.codes + row0 * (d / 8), cb, bar);
      bulk_g2s(smem_u32(gcodes + (RF + q * rq) * (d / 8)), u.codes + row0 * (d / 8), cb, bar);
      bulk_g2s(smem_u32(gsb + (0 * RF + q * rq) * G), g.scales + row0 * G, sb, bar);
      bulk_g2s(smem_u32(gsb + (1 * RF + q * rq) * G), g.biases + row0 * G, sb, bar);
      bulk_g2s(smem_u32(gsb + (2 * RF + q * rq) * G), u.scales + row0 * G, sb, bar);
      bulk_g2s(smem_u32(gsb + (3 * RF + q * rq) * G), u.biases + row0 * G, sb, bar);
    }
  };
  // Down rows r0 .. r0+15 of expert e of weight set `which` into expert slot `slot`.
  auto issue_dn = [&](int slot, int which, int e) {
    const QPtr& q = a.down[which];
    const size_t row0 = (size_t)e * d + r0;
    const uint32_t cb = RD * (F / 2), sb = RD * GF * 2;
    bulk_g2s(smem_u32(dcodes + slot * RD * (F / 8)), q.codes + row0 * (F / 8), cb, bar_dn);
    bulk_g2s(smem_u32(dsb + (slot * RD) * GF), q.scales + row0 * GF, sb, bar_dn);
    bulk_g2s(smem_u32(dsb + ((k1 + slot) * RD) * GF), q.biases + row0 * GF, sb, bar_dn);
  };

  // Weights are never written upstream: the shared expert's copies start before the wait.
  if (tid == 0) {
    if (has_dn) mbar_arrive_expect_tx(bar_dn, (uint32_t)k1 * (RD * (F / 2) + 2 * RD * GF * 2));
    if (a.has_shared) {
      if (has_gu && j == k) issue_gu(1, 0);
      if (has_dn) issue_dn(k, 1, 0);
    }
  }
  pdl_wait();   // x and logits from upstream kernels are complete and visible past this point
  if (warp == 0) {
    int e;
    float w;
    reg_topk(a.logits, a.E, k, &e, &w);
    if (lane < k) {
      e_s[lane] = e;
      w_s[lane] = w;
    }
    __syncwarp();
    if (lane == 0) {
      if (has_gu && j < k) issue_gu(0, e_s[j]);
      if (has_dn)
        for (int jj = 0; jj < k; ++jj) issue_dn(jj, 0, e_s[jj]);
    }
  } else if (warp == 1 && has_dn && a.has_shared) {
    float dot = 0.0f;
    const uint4* xv = reinterpret_cast<const uint4*>(a.x);
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
    if (lane == 0) w_s[k] = 1.0f / (1.0f + expf(-dot));
  }
  pdl_launch_dependents();

  // ---- gate/up job: lane l owns quantisation group l (64 inputs) of every row; warp w computes
  // gate and up of rows q*8 + w (q = 0..3) as slots s = 2q + mat, then a reduce-scatter leaves
  // slot s fully summed in lane 4s.
  if (has_gu) {
    const bool active = lane < G;
    float2 xs[32];
    float xsum = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) xs[i] = make_float2(0.0f, 0.0f);
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
          xs[c8 * 4 + i] = make_float2(lo * act_prescale(2 * i), hi * act_prescale(2 * i + 1));
        }
      }
    }
    float v8[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) v8[s] = 0.0f;
    bool ok_all = true;
#pragma unroll 1
    for (int q = 0; q < kQuarters; ++q) {
      const bool ok = mbar_wait_warp(smem_u32(&bars[q]), 0, &abort_s, a.err);
      ok_all = ok_all && ok;
#pragma unroll
      for (int mat = 0; mat < 2; ++mat) {
        const int row = q * (RF / kQuarters) + warp;
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
#pragma unroll
        for (int s = 0; s < 8; ++s) v8[s] = (s == 2 * q + mat) ? v : v8[s];
      }
    }
    // Reduce-scatter of 8 values over 32 lanes: after the xor-16, -8 and -4 steps lane l holds
    // a partial of slot ((l >> 2) & 7); the xor-2 and -1 steps finish the sum.
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
    if ((lane & 7) == 0 && ok_all) {
      const float gv = t1;
      a.h[(size_t)j * F + f0 + (lane >> 3) * (RF / kQuarters) + warp] = gv / (1.0f + expf(-gv)) * upv;
    }
  }

  // ---- grid barrier: every CTA arrives once; the last arrival resets the count and bumps the
  // generation in one atomic.  The h stores above are ordered before the arrival by the block
  // barrier and the fence.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned long long n = gridDim.x;
    const unsigned long long old = atom_add_release(a.sync, 1ull);
    if ((old & 0xFFFFFFFFull) == n - 1ull) atom_add_release(a.sync, (1ull << 32) - n);
    gen_s = old >> 32;
  }

  // ---- down job: rows r0 .. r0+15; warp w owns rows 2w and 2w+1.
  if (has_dn) {
    if (tid == 0) {
      const unsigned long long g0 = gen_s;
      const long long t0 = clock64();
      while ((ld_acquire(a.sync) >> 32) == g0) {
        if (abort_s || clock64() - t0 > kWaitTimeoutCycles) {
          abort_s = 1;
          raise_flag(a.err, kErrWaitTimeout);
          break;
        }
      }
      __threadfence();
    }
    __syncthreads();
    const int segs = P.segs;   // lanes covering one row (F / EPL)
    if (!abort_s) {
      // h (fp32, from L2) -> shared memory, pre-scaled per code position and padded per lane
      // segment so that the segment loads below are conflict-free; segment sums of unscaled h.
      const float4* h4 = reinterpret_cast<const float4*>(a.h);
      const int n4 = k1 * F / 4;
      for (int base = 0; base < n4; base += kThreadsDec) {
        const int i = base + tid;
        const bool valid = i < n4;
        float4 v = valid ? __ldcg(h4 + i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        float part = (v.x + v.y) + (v.z + v.w);
#pragma unroll
        for (int off = 1; off < EPL / 4; off <<= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
        if (valid) {
          const int e = 4 * i, jj = e / F, c = e % F;
          const int n0 = c & 7;   // 0 or 4
          v.x *= n0 ? act_prescale(4) : act_prescale(0);
          v.y *= n0 ? act_prescale(5) : act_prescale(1);
          v.z *= n0 ? act_prescale(6) : act_prescale(2);
          v.w *= n0 ? act_prescale(7) : act_prescale(3);
          const int sg = jj * segs + c / EPL;
          *reinterpret_cast<float4*>(hs + sg * (EPL + 4) + c % EPL) = v;
          if ((c % EPL) == 0) hsum_s[sg] = part;
        }
      }
    }
    __syncthreads();
    const bool ok = mbar_wait_warp(bar_dn, 0, &abort_s, a.err) && !abort_s;
    constexpr int EPW = EPL / 8;   // code words per lane segment
    const int rpw = 32 / segs;     // rows a warp covers at once (1 or 2)
    const int npass = 2 / rpw;
    const int sub = lane / segs, l = lane % segs;
    const int grp = (l * EPL) / 64;
    float acc[2] = {0.0f, 0.0f};
    if (ok) {
#pragma unroll 1
      for (int jj = 0; jj < k1; ++jj) {
        float2 hv[EPL / 2];
        const float4* hp = reinterpret_cast<const float4*>(hs + (jj * segs + l) * (EPL + 4));
#pragma unroll
        for (int c4 = 0; c4 < EPL / 4; ++c4) {
          const float4 t = hp[c4];
          hv[2 * c4] = make_float2(t.x, t.y);
          hv[2 * c4 + 1] = make_float2(t.z, t.w);
        }
        const float hsm = hsum_s[jj * segs + l];
        const float wj = w_s[jj];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
          if (it < npass) {
            const int r = 2 * warp + it * rpw + sub;
            const uint32_t* cw = dcodes + (jj * RD + r) * (F / 8) + l * EPW;
            uint32_t wd[EPW];
            if (EPW == 1) {
              wd[0] = cw[0];
            } else if (EPW == 2) {
              const uint2 t = *reinterpret_cast<const uint2*>(cw);
              wd[0] = t.x;
              wd[EPW > 1 ? 1 : 0] = t.y;
            } else {
#pragma unroll
              for (int q4 = 0; q4 < EPW / 4; ++q4) {
                const uint4 t = *reinterpret_cast<const uint4*>(cw + 4 * q4);
                wd[(4 * q4) % EPW] = t.x;
                wd[(4 * q4 + 1) % EPW] = t.y;
                wd[(4 * q4 + 2) % EPW] = t.z;
                wd[(4 * q4 + 3) % EPW] = t.w;
              }
            }
            float2 p0 = make_float2(0.0f, 0.0f), p1 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int w8 = 0; w8 < EPW; ++w8) {
              if (w8 & 1) p1 = word_dot2(wd[w8], hv + 4 * w8, p1);
              else p0 = word_dot2(wd[w8], hv + 4 * w8, p0);
            }
            const float p = (p0.x + p0.y) + (p1.x + p1.y);
            const float s = bf16_bits_to_f32(dsb[(jj * RD + r) * GF + grp]);
            const float b = bf16_bits_to_f32(dsb[((k1 + jj) * RD + r) * GF + grp]);
            acc[it] = fmaf(wj, fmaf(s, p, b * hsm), acc[it]);
          }
        }
      }
    }
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      float v = acc[it];
      for (int off = segs / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      if (it < npass && l == 0 && ok) a.y[r0 + 2 * warp + it * rpw + sub] = v;
    }
  }

  // ---- wind down: after a timeout, copies still in flight must land before the CTA exits.
  __syncthreads();
  if (tid == 0 && abort_s) {
    for (int i = 0; i <= kQuarters; ++i) {
      const bool used = (i < kQuarters) ? has_gu : has_dn;
      if (!used) continue;
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(&bars[i]), 0) && clock64() - t0 < 4000000ll) {
      }
    }
  }
}

int dec_epl(int F) { return F / 32 <= 8 ? 8 : F / 32; }
int dec_grid(int d, int k1, int F) { return std::max(k1 * (F / RF), d / RD); }

template <int EPL>
cudaError_t configure(size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(decode_layer_kernel<EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_layer_kernel<EPL>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return e;
}

// Per device: SM count and CTAs per SM of each instantiation at the largest plan (checked at
// every call against the actual plan's grid).
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
    if ((e = configure<8>(kDecSmemMax)) != cudaSuccess) return e;
    if ((e = configure<16>(kDecSmemMax)) != cudaSuccess) return e;
    if ((e = configure<32>(kDecSmemMax)) != cudaSuccess) return e;
    if ((e = configure<64>(kDecSmemMax)) != cudaSuccess) return e;
    di.ready = true;
  }
  *out = &di;
  return cudaSuccess;
}

}  // namespace

bool decode_supported(int d, int E, int k, int F) {
  const int k1 = k + 1;
  // One quantisation group per lane in the gate/up rows: d <= 2048, at most 32 experts per token.
  if (k1 > 32 || E > kMaxE || F > 2048 || d > 2048 || d % RD != 0) return false;
  // A down row is covered by F / max(8, F/32) lanes with a butterfly: F = 128 * 2^n.
  if (F != 128 && F != 256 && F != 512 && F != 1024 && F != 2048) return false;
  if (DecPlan(d, F, k1).bytes > kDecSmemMax) return false;
  // Every CTA must be resident at once (one per SM): the grid barrier waits on all of them.
  DevInfo* di = nullptr;
  if (dev_info(&di) != cudaSuccess) return false;
  return dec_grid(d, k1, F) <= di->sms;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st, bool pdl) {
  const int k1 = a.k + (a.has_shared ? 1 : 0);
  DevInfo* di = nullptr;
  cudaError_t e = dev_info(&di);
  if (e != cudaSuccess) return e;
  const DecPlan P(a.d, a.F, k1);
  const int grid = dec_grid(a.d, k1, a.F);
  if (grid > di->sms || P.bytes > kDecSmemMax) return cudaErrorInvalidConfiguration;

  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreadsDec);
  cfg.dynamicSmemBytes = P.bytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  switch (dec_epl(a.F)) {
    case 8: e = cudaLaunchKernelEx(&cfg, decode_layer_kernel<8>, a); break;
    case 16: e = cudaLaunchKernelEx(&cfg, decode_layer_kernel<16>, a); break;
    case 32: e = cudaLaunchKernelEx(&cfg, decode_layer_kernel<32>, a); break;
    default: e = cudaLaunchKernelEx(&cfg, decode_layer_kernel<64>, a); break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
