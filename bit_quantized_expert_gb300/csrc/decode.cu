// Decode MoE layer (one token, or a few: T <= 8) as one bandwidth-bound dequant-GEMV kernel.
//
// At batch 1 there is almost no weight reuse, so weight bandwidth sets the ceiling ("Perplexity
// libera Lily: inferencia en Rust y Metal para Mac", section "Decode: mover menos bytes por
// token"); the pages also report that removing all arithmetic from the kernels changed speed by
// 0.2% and that matrix ops reached 97.9% of bandwidth ("Perplexity открыла код Lily...",
// section "Спекулятивное декодирование не взлетело").  On a GB300 one layer's routed weights
// (~16 MB) stream in ~2.3 us, so the layer is as much a latency chain as a bandwidth problem:
// the design keeps that chain short and free of grid-wide waits.
//
// Work split.  Expert slot j (0..k-1 routed, k = the shared expert) gets S = F / 32 CTAs; CTA s of
// the slot owns gate/up rows f0 = 32 s .. f0+31.  The S CTAs of a slot form S / 4 thread-block
// clusters of C = 4 CTAs; cluster q covers the F columns KC0 = 128 q .. KC0 + 127 of the down
// projection, and its CTA of rank c owns down rows r0 = c d / 4 .. r0 + d / 4 - 1 over those
// columns.  Clusters of four are what the GPU can co-schedule one CTA per SM across all SMs (larger
// clusters are placed two CTAs to an SM, or wait for a second wave).  Per token:
//   * routing: after the programmatic-launch wait every CTA ranks the 1 KB of logits itself (all
//     eight warps: per-warp candidate ranks by shuffles, then the 8 k survivors ranked in shared
//     memory) -- no routing kernel on the critical path -- and immediately bulk-copies its gate/up
//     rows (four quarters, one mbarrier each, so compute starts on the first quarter) and its down
//     rows (the cluster's 64-byte column block of each row, as one or two 2-D tensor copies) with
//     their scales and biases.  Shared-expert CTAs start their copies before the wait: weights are
//     never written upstream;
//   * each CTA computes its 32 SwiGLU outputs h, turns them into fixed-point byte planes (see
//     Planes) and writes those into the shared memory of every CTA of its cluster (distributed
//     shared memory), then the cluster barrier;
//   * each CTA computes its d / C down rows over the cluster's 32 C columns of h, scaled by the
//     slot's routing weight (or the shared expert's gate), and stores them as one partial of each
//     of its row slices (128 rows);
//   * combine: a second, small kernel (launched with programmatic dependent launch, so its CTAs
//     are resident and waiting when the decode launch ends) sums each row's (k+1) S / C partials
//     in a fixed order and writes y.  Nobody waits on another cluster inside the decode launch;
//     the order of the sum never depends on the order in which CTAs finish.
// Several tokens (the kMulti instantiation): warp t routes token t; every CTA then takes its
// slot of token 0, 1, ... in turn, fetching the slot's weights again only when its expert changes
// (the shared expert's stay), with double-buffered h exchange slots and partials per token, so
// each token's y is what a one-token launch gives, bit for bit.
//
// Arithmetic: w = q*s + b enters as s * sum(q x) + b * sum(x) per quantisation group; sum(q x) is
// an exact integer dot product (dp4a) of the 4-bit codes with the group's activations held as
// 23-bit fixed point relative to the group's largest (Planes below), and everything after it is
// fp32.  Per code word that is two masks and six dp4a, against about twice the issue slots for
// an fp32 dequantise-and-multiply.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int RF = 32;   // gate/up rows per CTA
constexpr int kQuarters = 4;
constexpr int kRQ = RF / kQuarters;   // gate/up rows per quarter
constexpr int kMaxE = 1024;
constexpr int kThreadsDec = 256;
constexpr int kWarpsDec = kThreadsDec / 32;
constexpr int kSliceRows = 128;        // rows of y per combine slice
constexpr int kMaxDecodeD = 2048;      // one quantisation group of the gate/up rows per lane

// ---------------------------------------------------------------- exact integer dot products
// Activations v_c become 23-bit two's-complement fixed point V_c = round(v_c 2^(22-e)), with e the
// smallest exponent such that every |v| of the block is below 2^e, held as three byte planes
// V = hi 2^16 + mid 2^8 + lo (hi signed, mid and lo unsigned: bytes 2, 1, 0 of V).  Byte j of
// plane word [2w + o] is V of column 8w + 2j + o: the byte order in which a 32-bit code word splits
// into its even nibbles (w & 0x0F0F0F0F) and odd nibbles ((w >> 4) & 0x0F0F0F0F).  sum_c q_c v_c
// over a quantisation group (eight code words) is then six dp4a per word, exact in 32-bit integers,
// recombined once in fp32.  The gate/up activations use one exponent per group; h uses one per 32
// columns (the block one CTA produces), so a group has an exponent per half.  Elements more than
// 2^23 below their block's largest are rounded, which keeps a sum within fp32 accumulation error.
struct Planes {
  uint32_t p[3][16];   // [hi | mid | lo][2 w + o], words 0..7 of the group
  float scale[2];      // 2^(e - 22) of code words 0..3 and 4..7
  float sum;           // sum of the group's values (fp32), for the bias term
};

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// e with |v| < 2^e for every v whose magnitude bits are at most mbits (the largest |v| as uint32;
// bit patterns of non-negative floats order like the values), clamped below at -104 so that
// 2^(22 - e) is a normal float; values under 2^-104 then round towards 0.
__device__ __forceinline__ int block_exponent(uint32_t mbits) { return max((int)((mbits >> 23) & 0xFFu) - 126, -104); }
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((127 + k) << 23); }   // -126 <= k <= 127
// round(v * scale) for |v * scale| < 2^22: adding 1.5 * 2^23 leaves the rounded integer in the low bits.
__device__ __forceinline__ int fixed23(float v, float scale) {
  return __float_as_int(fmaf(v, scale, 12582912.0f)) - 0x4B400000;
}
// Planes words of four fixed-point values (columns 8w + o, + 2, + 4, + 6).
__device__ __forceinline__ void pack4(int v0, int v1, int v2, int v3, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  const uint32_t a = __byte_perm(v0, v1, 0x5140), b = __byte_perm(v2, v3, 0x5140);
  lo = __byte_perm(a, b, 0x5410);
  mid = __byte_perm(a, b, 0x7632);
  hi = __byte_perm(__byte_perm(v0, v1, 0x0062), __byte_perm(v2, v3, 0x0062), 0x5410);
}

// The 64 bf16 activations of one quantisation group (eight uint4 = columns 0..63) -> planes with
// one exponent.  Returns false when a value is not finite.
__device__ __forceinline__ bool planes_of_bf16(const uint4 (&xr)[8], Planes& P) {
  uint32_t mb4[4] = {0u, 0u, 0u, 0u};
  float sum4[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // four partial sums: a short dependency chain
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    const uint32_t wv[4] = {xr[c8].x, xr[c8].y, xr[c8].z, xr[c8].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mb4[i] = max(mb4[i], max((wv[i] << 16) & 0x7FFF0000u, wv[i] & 0x7FFF0000u));
      sum4[i] += bf16_bits_to_f32(wv[i] & 0xFFFFu) + bf16_bits_to_f32(wv[i] >> 16);
    }
  }
  const uint32_t mb = max(max(mb4[0], mb4[1]), max(mb4[2], mb4[3]));
  const float sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
  const int e = block_exponent(mb);
  const float sc = pow2i(22 - e);
  P.scale[0] = P.scale[1] = pow2i(e - 22);
  P.sum = sum;
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    const uint32_t wv[4] = {xr[c8].x, xr[c8].y, xr[c8].z, xr[c8].w};
#pragma unroll
    for (int o = 0; o < 2; ++o) {
      int v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = fixed23(bf16_bits_to_f32(o ? (wv[i] >> 16) : (wv[i] & 0xFFFFu)), sc);
      pack4(v[0], v[1], v[2], v[3], P.p[0][2 * c8 + o], P.p[1][2 * c8 + o], P.p[2][2 * c8 + o]);
    }
  }
  return ((mb >> 23) & 0xFFu) != 0xFFu;
}

// sum_c q_c v_c over the 64 columns of eight code words c0, c1 (one quantisation group).
__device__ __forceinline__ float group_dot(const uint4& c0, const uint4& c1, const Planes& P) {
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  int s[2][3] = {{0, 0, 0}, {0, 0, 0}};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t ev = w[j] & 0x0F0F0F0Fu, od = (w[j] >> 4) & 0x0F0F0F0Fu;
    int* a = s[j >> 2];
    a[0] = dp4a_us(ev, P.p[0][2 * j], a[0]);
    a[0] = dp4a_us(od, P.p[0][2 * j + 1], a[0]);
    a[1] = dp4a_uu(ev, P.p[1][2 * j], a[1]);
    a[1] = dp4a_uu(od, P.p[1][2 * j + 1], a[1]);
    a[2] = dp4a_uu(ev, P.p[2][2 * j], a[2]);
    a[2] = dp4a_uu(od, P.p[2][2 * j + 1], a[2]);
  }
  const float t0 = (float)s[0][0] * 65536.0f + (float)s[0][1] * 256.0f + (float)s[0][2];
  const float t1 = (float)s[1][0] * 65536.0f + (float)s[1][1] * 256.0f + (float)s[1][2];
  return fmaf(t0, P.scale[0], t1 * P.scale[1]);
}

// Exchange block of one CTA's 32 h values (their planes, exponent and sum), 32 words.
constexpr int kHBlockWords = 32;

// CTAs per thread-block cluster (S = F / 32 is a multiple of 4).
constexpr int kC = 4;

// Geometry and shared-memory plan of one launch (byte offsets, 16-byte aligned regions).
// Dynamic shared memory of one decode CTA, at most: one token (the kernel also holds ~15 KB of
// static shared memory), several tokens (~21 KB static: the several-token ranking tables).
constexpr uint32_t kDecPlanMax = 200 * 1024;
constexpr uint32_t kDecPlanMaxMulti = 200 * 1024;

struct DecPlan {
  int d, F, k1, G, GF, S, C, NQ, DR, KC, GP, NSC, nslices, NP, grid, box_rows, x_smem;
  uint32_t gu_codes, gu_sb, dn_codes, dn_sb, hclu, xs, bytes;
  // multi: several tokens per launch, nt of them (two h exchange slots, alternating by token; x
  // staging sized for nt)
  __host__ __device__ DecPlan(int d_, int F_, int k1_, bool multi, int nt = kDecodeMaxTokens)
      : d(d_), F(F_), k1(k1_) {
    const uint32_t cap = multi ? kDecPlanMaxMulti : kDecPlanMax;
    G = d / 64;
    GF = F / 64;
    S = F / RF;
    C = kC;
    NQ = S / C;                 // clusters per slot
    DR = d / C;                 // down rows per CTA
    KC = RF * C;                // down columns (F) per cluster
    GP = KC / 64;               // quantisation groups per down row and cluster
    NSC = (DR + kSliceRows - 1) / kSliceRows;   // combine slices per CTA
    nslices = C * NSC;
    NP = k1 * NQ;               // partials per row of y
    grid = k1 * S;
    box_rows = DR <= 256 ? DR : DR / ((DR + 255) / 256);   // rows per 2-D copy of the down codes
    uint32_t o = 0;
    gu_codes = o;  o += 2u * RF * (d / 2);        // [gate|up][RF][d/8] u32
    gu_sb = o;     o += 4u * RF * G * 2;          // [g.s|g.b|u.s|u.b][RF][G] bf16
    o = (o + 127u) & ~127u;
    dn_codes = o;  o += (uint32_t)DR * (KC / 2);  // [DR][KC/8] u32
    dn_sb = o;     o += 4u * DR * GF;             // [s|b][DR][GF] bf16: whole scale and bias rows
    o = (o + 15u) & ~15u;
    hclu = o;      o += (multi ? 2u : 1u) * 4u * KC;   // h of the cluster's columns, fp32, per exchange slot
    if (multi) o = (o + 127u) & ~127u;
    // Several tokens: every token's x row copied in at the start (bf16 [nt][d]) when it fits, so
    // that no token's x load queues behind the weight copies in flight.
    const uint32_t x_bytes = (uint32_t)nt * (uint32_t)d * 2u;
    x_smem = (multi && o + x_bytes <= cap) ? 1 : 0;
    xs = o;
    if (x_smem) o += x_bytes;
    bytes = (o + 15u) & ~15u;
  }
};

// ---------------------------------------------------------------- cluster helpers (PTX ISA)
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address in the shared memory of cluster CTA `rank` matching this CTA's shared address `a`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// ---------------------------------------------------------------- routing of one token
// Softmax of the k selected logits, shared by the one-token and the several-token paths so that
// both give the same weights bit for bit: lane j < k holds the j-th selected logit my_v, vmax is
// the largest; returns lane j's weight.
__device__ __forceinline__ float softmax_tail(float my_v, float vmax, int k, int lane) {
  const float my_ex = lane < k ? expf(my_v - vmax) : 0.0f;
  float s = my_ex;   // lanes >= k hold 0
  if (k > 8) {
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 16);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 8);
  }
  s += __shfl_xor_sync(0xFFFFFFFFu, s, 4);
  s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
  s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
  return my_ex / s;
}

// 64-bit candidate key: the logit's order-preserving key above, the complement of the expert
// index below, so that a larger key is a larger logit or, for equal logits, a lower index; every
// candidate is distinct and 0 marks padding.
__device__ __forceinline__ uint64_t cand_key(float v, int e) {
  return ((uint64_t)logit_key(v) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e);
}
__device__ __forceinline__ int cand_expert(uint64_t c) { return (int)(0xFFFFFFFFu - (uint32_t)c); }

// The k best candidates of a row of E <= 256 * NE logits, by the whole CTA (every thread calls
// it): thread t holds experts t + 256 i; each warp ranks its candidates against the warp's
// (broadcast reads of the warp's keys from shared memory) and keeps its k best in `cand`
// [kWarpsDec][k]; then the first 8 k threads rank those against each other and the k best land in
// sel[0..k-1] in descending order.  `keys` holds kThreadsDec * NE entries.  Two block barriers.
// The same for E <= 256 and k <= 8 with every loop unrolled: thread t holds expert t; it ranks its
// key against its warp's 32 (16-byte broadcast reads), the warp's k best land in cand [8][8]
// (rank order, zero padded); then threads 0..63 rank those 64 against each other and the k best
// land in sel.  keys holds kThreadsDec entries.  Two block barriers.
__device__ __forceinline__ void block_topk_small(const float* __restrict__ row, int E, int k, uint64_t* keys,
                                                 uint64_t* cand, uint64_t* sel) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint64_t key = tid < E ? cand_key(__ldg(row + tid), tid) : 0ull;
  keys[tid] = key;
  if (lane < 8) cand[warp * 8 + lane] = 0ull;
  __syncwarp();
  const ulonglong2* wk = reinterpret_cast<const ulonglong2*>(keys + warp * 32);
  int rank = 0;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const ulonglong2 o = wk[c];
    rank += (o.x > key ? 1 : 0) + (o.y > key ? 1 : 0);
  }
  if (key != 0ull && rank < k) cand[warp * 8 + rank] = key;
  __syncthreads();
  if (tid < kWarpsDec * 8) {
    const uint64_t mine = cand[tid];
    const ulonglong2* ck = reinterpret_cast<const ulonglong2*>(cand);
    int r = 0;
#pragma unroll
    for (int c = 0; c < kWarpsDec * 4; ++c) {
      const ulonglong2 o = ck[c];
      r += (o.x > mine ? 1 : 0) + (o.y > mine ? 1 : 0);
    }
    if (mine != 0ull && r < k) sel[r] = mine;
  }
  __syncthreads();
}

// block_topk_small for T tokens at once (E <= 256, k <= 8, T <= kDecodeMaxTokens): logits [T][E];
// thread t holds expert t of every token, ranks each key against its warp's 32 of the same token,
// and the warp's k best per token land in cand [T][8][8]; then each of the T x 64 candidates is
// ranked against its token's 64 and the k best land in sel [T][8].  keys holds T x kThreadsDec
// entries.  Every token's selection is the one block_topk_small makes.  Two block barriers.
// `between` runs after the logit loads are issued and before their values are used.
template <typename Between>
__device__ __forceinline__ void block_topk_small_tokens(const float* __restrict__ logits, int E, int k, int T,
                                                        uint64_t* keys, uint64_t* cand, uint64_t* sel,
                                                        Between between) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float lv[kDecodeMaxTokens];
#pragma unroll
  for (int t = 0; t < kDecodeMaxTokens; ++t) lv[t] = (t < T && tid < E) ? __ldg(logits + (size_t)t * E + tid) : 0.0f;
  between();
  uint64_t key[kDecodeMaxTokens];
#pragma unroll
  for (int t = 0; t < kDecodeMaxTokens; ++t) {
    key[t] = (t < T && tid < E) ? cand_key(lv[t], tid) : 0ull;
    if (t < T) {
      keys[t * kThreadsDec + tid] = key[t];
      if (lane < 8) cand[(t * kWarpsDec + warp) * 8 + lane] = 0ull;
    }
  }
  __syncwarp();
#pragma unroll
  for (int t = 0; t < kDecodeMaxTokens; ++t) {
    if (t < T) {
      const ulonglong2* wk = reinterpret_cast<const ulonglong2*>(keys + t * kThreadsDec + warp * 32);
      int rank = 0;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const ulonglong2 o = wk[c];
        rank += (o.x > key[t] ? 1 : 0) + (o.y > key[t] ? 1 : 0);
      }
      if (key[t] != 0ull && rank < k) cand[(t * kWarpsDec + warp) * 8 + rank] = key[t];
    }
  }
  __syncthreads();
  for (int i = tid; i < T * kWarpsDec * 8; i += kThreadsDec) {
    const int t = i / (kWarpsDec * 8);
    const uint64_t mine = cand[i];
    const ulonglong2* ck = reinterpret_cast<const ulonglong2*>(cand + t * kWarpsDec * 8);
    int r = 0;
#pragma unroll
    for (int c = 0; c < kWarpsDec * 4; ++c) {
      const ulonglong2 o = ck[c];
      r += (o.x > mine ? 1 : 0) + (o.y > mine ? 1 : 0);
    }
    if (mine != 0ull && r < k) sel[t * 8 + r] = mine;
  }
  __syncthreads();
}

template <int NE>
__device__ __forceinline__ void block_topk(const float* __restrict__ row, int E, int k, uint64_t* keys,
                                           uint64_t* cand, uint64_t* sel) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t key[NE];
  int rank[NE];
#pragma unroll
  for (int i = 0; i < NE; ++i) {
    const int e = tid + kThreadsDec * i;
    key[i] = e < E ? cand_key(__ldg(row + e), e) : 0ull;
    rank[i] = 0;
    keys[(warp * NE + i) * 32 + lane] = key[i];
  }
  for (int i = lane; i < k; i += 32) cand[warp * k + i] = 0ull;
  __syncwarp();
  const uint64_t* wk = keys + warp * NE * 32;
#pragma unroll 8
  for (int c = 0; c < 32 * NE; ++c) {
    const uint64_t o = wk[c];
#pragma unroll
    for (int m = 0; m < NE; ++m) rank[m] += o > key[m] ? 1 : 0;
  }
#pragma unroll
  for (int m = 0; m < NE; ++m)
    if (key[m] != 0ull && rank[m] < k) cand[warp * k + rank[m]] = key[m];
  __syncthreads();
  const int nc = kWarpsDec * k;
  if (tid < nc) {
    const uint64_t mine = cand[tid];
    int r = 0;
#pragma unroll 8
    for (int c = 0; c < nc; ++c) r += cand[c] > mine ? 1 : 0;
    if (mine != 0ull && r < k) sel[r] = mine;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- weight copies of one CTA
// Shared by the layer kernel and its loads-only replica, so both move exactly the same bytes.

// The weight copies of expert e for one CTA, issued by one warp, one copy per lane (an issuing
// thread waits for the copy engine to take each request, so sixteen lanes get sixteen requests out
// in the time of one), in the order the compute needs them: lane 0 first arms every barrier with
// its byte count; then lanes 0, 1 copy the gate and up code rows of quarter 0, lanes 2..5 the
// gate/up scales and biases (with quarter 0), lanes 6..11 the gate (even lane) and up (odd) code
// rows of quarters 1..3, lanes 12..13 the down code boxes (the cluster's 64-byte column block of
// box_rows rows each, by 2-D tensor copy) and lanes 14..15 the down scale and bias rows.
// `which` selects groups of copies: 1 = quarter 0 with the gate/up scales and biases, 4 = quarters
// 1..3, 2 = down (5 = all gate/up, 7 = everything).  bars: shared address of the five barriers
// (gate/up quarters, then down), 8 bytes apart.
__device__ __forceinline__ void issue_copies(const DecPlan& P, const QPtr& g, const QPtr& u, const QPtr& dn,
                                             const CUtensorMap* map, int e, int f0, int r0, int kc0, uint32_t gcodes,
                                             uint32_t gsb, uint32_t dcodes, uint32_t dsb, uint32_t bars, int which,
                                             int lane) {
  const int d = P.d, G = P.G;
  const uint32_t cb = kRQ * (d / 2), sb = RF * G * 2;    // code bytes per quarter and matrix; s/b bytes
  const uint32_t rb = P.KC / 2, sbb = (uint32_t)P.DR * P.GF * 2;
  const size_t rowb = (size_t)e * P.F + f0;
  const size_t drow0 = (size_t)e * d + r0;
  if (lane == 0) {
    if (which & 1) mbar_arrive_expect_tx(bars, 2 * cb + 4 * sb);
    if (which & 4)
      for (int q = 1; q < kQuarters; ++q) mbar_arrive_expect_tx(bars + 8 * q, 2 * cb);
    if (which & 2) mbar_arrive_expect_tx(bars + 8 * kQuarters, (uint32_t)P.DR * rb + 2u * sbb);
  }
  __syncwarp();
  // Each lane's role depends on the lane alone; `which` only switches roles off.
  if (lane < 12) {
    if (which & (lane < 6 ? 1 : 4)) {
      if (lane >= 2 && lane < 6) {
        const int i = lane - 2;
        const uint16_t* src = i == 0 ? g.scales : i == 1 ? g.biases : i == 2 ? u.scales : u.biases;
        bulk_g2s(gsb + i * sb, src + rowb * G, sb, bars);
      } else {
        const int c = lane < 2 ? lane : lane - 4;   // code copy 0..7: quarter c / 2, gate (even) or up (odd)
        const int q = c >> 1, mat = c & 1;
        const QPtr& m = mat ? u : g;
        bulk_g2s(gcodes + (uint32_t)(mat * RF + q * kRQ) * (d / 2), m.codes + (rowb + q * kRQ) * (d / 8), cb,
                 bars + 8 * q);
      }
    }
  } else if (lane < 14) {
    const int r = (lane - 12) * P.box_rows;   // 0 or box_rows
    if ((which & 2) && r < P.DR) tma_load_2d(dcodes + r * rb, map, bars + 8 * kQuarters, kc0 / 8, (int)(drow0 + r));
  } else if (lane < 16) {
    if (which & 2) {
      const uint16_t* src = lane == 14 ? dn.scales : dn.biases;
      bulk_g2s(dsb + (lane - 14) * sbb, src + drow0 * P.GF, sbb, bars + 8 * kQuarters);
    }
  }
}

template <bool kMulti>
__global__ void __launch_bounds__(kThreadsDec, 1)
    decode_layer_kernel(const __grid_constant__ DecodeMaps maps, const DecodeArgs a) {
  constexpr int C = kC;
  extern __shared__ __align__(128) uint8_t sm[];
  const int d = a.d, F = a.F, k = a.k;
  const int k1 = k + (a.has_shared ? 1 : 0);
  const DecPlan P(d, F, k1, kMulti, kMulti ? (a.T > 0 ? a.T : 1) : 1);
  const int G = P.G, GF = P.GF;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int j = cta / P.S;              // expert slot: 0..k-1 routed, k shared
  const int sidx = cta % P.S;
  const int qc = sidx / C;              // cluster of the slot: down columns KC0 .. KC0 + KC - 1
  const int crank = sidx % C;           // rank in the cluster: down rows r0 .. r0 + DR - 1
  const int f0 = sidx * RF;             // first gate/up row
  const int kc0 = qc * P.KC;
  const int r0 = crank * P.DR;
  const bool shared_cta = (j == k);
  const int wset = shared_cta ? 1 : 0;

  uint32_t* dcodes = reinterpret_cast<uint32_t*>(sm + P.dn_codes);   // [DR][KC/8]
  uint16_t* dsb = reinterpret_cast<uint16_t*>(sm + P.dn_sb);         // [s | b][DR][GF]
  float* hclu = reinterpret_cast<float*>(sm + P.hclu);               // [2][KC]
  __shared__ __align__(8) uint64_t bars[kQuarters + 1];   // gate/up quarters, then the down rows
  __shared__ __align__(16) uint64_t cand[kWarpsDec * 32];
  __shared__ __align__(16) uint64_t keys_s[kMulti ? kDecodeMaxTokens * kThreadsDec : kMaxE];
  __shared__ __align__(16) uint64_t cand_t[kMulti ? kDecodeMaxTokens * kWarpsDec * 8 : 1];
  __shared__ uint64_t sel_t[kMulti ? kDecodeMaxTokens * 8 : 1];
  __shared__ uint64_t sel[32];
  __shared__ int e_s[kDecodeMaxTokens];
  __shared__ float wgt_s[kDecodeMaxTokens];    // w_j (routed) or the shared-expert gate, per token
  __shared__ float hloc[RF];   // this CTA's h (rows f0 .. f0+31)
  __shared__ int vloc[RF];     // ... as 23-bit fixed point
  __shared__ int abort_s;
  // One token: x is copied into shared memory as soon as the dependency wait ends, so its latency
  // overlaps the top-k instead of queueing behind the weight copies issued after it.
  __shared__ __align__(16) uint4 xs[kMulti ? 1 : kMaxDecodeD / 8];
  const int T = kMulti ? (a.T > 0 ? a.T : 1) : 1;

  if (tid == 0) {
    for (int i = 0; i <= kQuarters; ++i) mbar_init(smem_u32(&bars[i]), 1);
    abort_s = 0;
    mbar_fence_init();
  }
  __syncthreads();
  cluster_arrive_relaxed();   // this CTA runs: its shared memory may now receive the cluster's h

  // Fetches of the slot's weights, counted by lane 0 of warp 0 (the issuing warp) for the
  // wind-down: gate/up rows and down rows.
  int gu_issued = 0, dn_issued = 0;
  // expert e's copies (which: 5 gate/up, 2 down, 7 both) by the calling warp
  auto issue = [&](int e, int which) {
    issue_copies(P, a.gate[wset], a.up[wset], a.down[wset], &maps.down[wset], e, f0, r0, kc0,
                 smem_u32(sm + P.gu_codes), smem_u32(sm + P.gu_sb), smem_u32(dcodes), smem_u32(dsb),
                 smem_u32(&bars[0]), which, lane);
    if (kMulti && (which & 5)) ++gu_issued;   // one token: one fetch of each, counted below
    if (kMulti && (which & 2)) ++dn_issued;
  };

  // Weights are never written upstream: the shared expert's copies start before the wait.
  if (shared_cta && warp == 0) issue(0, 7);
  if (tid == 32) prefetch_tmap(&maps.down[wset]);
  pdl_wait();   // x and logits from upstream kernels are complete and visible past this point
  if (!kMulti) {   // 16-byte piece i at i ^ ((i / 8) % 8): lane l's eight pieces fall in distinct banks
    for (int i = tid; i < d / 8; i += kThreadsDec) cp_async_16(smem_u32(&xs[i ^ ((i >> 3) & 7)]), a.x + (size_t)i * 8);
    cp_async_commit();
  }
  // Several tokens: every token's row of x, the same layout per token.  On the block-ranking path
  // the copies go out right after the logit loads, so that those do not queue behind them.
  auto stage_x = [&]() {
    uint4* xm = reinterpret_cast<uint4*>(sm + P.xs);
    const int pr = d / 8;
    for (int i = tid; i < T * pr; i += kThreadsDec) {
      const int tk = i / pr, pc = i % pr;
      cp_async_16(smem_u32(&xm[tk * pr + (pc ^ ((pc >> 3) & 7))]), a.x + (size_t)tk * d + (size_t)pc * 8);
    }
    cp_async_commit();
  };
  const bool block_rank = kMulti && !shared_cta && a.E <= kThreadsDec && k <= 8;
  if (kMulti && P.x_smem && !block_rank) stage_x();

  if (!kMulti) {
    if (!shared_cta) {
      if (a.E <= kThreadsDec && k <= 8) block_topk_small(a.logits, a.E, k, keys_s, cand, sel);
      else if (a.E <= kThreadsDec) block_topk<1>(a.logits, a.E, k, keys_s, cand, sel);
      else block_topk<kMaxE / kThreadsDec>(a.logits, a.E, k, keys_s, cand, sel);
      const int ej = cand_expert(sel[j]);
      if (warp == 0) issue(ej, 7);   // all of the slot's weight copies at once
      if (tid == 0) e_s[0] = ej;
      if (warp == 2) {
        const float v = lane < k ? key_logit((uint32_t)(sel[lane] >> 32)) : 0.0f;
        const float w = softmax_tail(v, key_logit((uint32_t)(sel[0] >> 32)), k, lane);
        if (lane == j) wgt_s[0] = w;
      }
    }
  } else if (block_rank) {
    // every token ranked by the whole CTA at once (the one-token ranking, per token); warp t then
    // takes token t's softmax, and token 0's copies go out
    block_topk_small_tokens(a.logits, a.E, k, T, keys_s, cand_t, sel_t, [&]() {
      if (P.x_smem) stage_x();
    });
    if (warp < T) {
      const uint64_t* st = sel_t + warp * 8;
      const float v = lane < k ? key_logit((uint32_t)(st[lane] >> 32)) : 0.0f;
      const float w = softmax_tail(v, key_logit((uint32_t)(st[0] >> 32)), k, lane);
      if (lane == j) {
        e_s[warp] = cand_expert(st[j]);
        wgt_s[warp] = w;
      }
    }
    if (warp == 0) issue(cand_expert(sel_t[j]), 7);
  } else if (warp < T && !shared_cta) {
    // warp t routes token t; token 0's gate/up rows are requested as soon as its expert is known
    int e;
    float w;
    if (a.E <= 256) warp_topk_softmax<8>(a.logits + (size_t)warp * a.E, a.E, k, &e, &w);
    else warp_topk_softmax<32>(a.logits + (size_t)warp * a.E, a.E, k, &e, &w);
    const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
    const float wj = __shfl_sync(0xFFFFFFFFu, w, j);
    if (lane == 0) {
      e_s[warp] = ej;
      wgt_s[warp] = wj;
    }
    if (warp == 0) issue(ej, 7);
  }
  if (shared_cta) {
    // warp w: the shared-expert gates of tokens w, w + 8, ...
    for (int t = warp; t < T; t += kWarpsDec) {
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
  if (!kMulti || P.x_smem) cp_async_wait<0>();
  __syncthreads();   // e_s and wgt_s (and x in shared memory)
  cluster_wait_acquire();   // every CTA of the cluster runs (pairs with the arrive above)

  // Tokens one after another.  Consecutive tokens of the slot with the same expert form a run
  // (always one run for the shared expert); the slot's weights stay in shared memory for a run
  // and are fetched again for the next; every fetch is one phase of the copy barriers, so waits
  // use the parity of the run index.
  const bool active = lane < G;
  const uint32_t* gcodes = reinterpret_cast<const uint32_t*>(sm + P.gu_codes);   // gate [RF][d/8], then up
  const uint16_t* gsb = reinterpret_cast<const uint16_t*>(sm + P.gu_sb);         // [g.s|g.b|u.s|u.b][RF][G]
  int run = 0;
#pragma unroll 1
  for (int t = 0; t < T; ++t) {
    const int e_t = e_s[t];
    if (t > 0 && e_t != e_s[t - 1]) ++run;   // requested during the previous token
    const uint32_t ph = (uint32_t)run & 1u;
    float* hx = hclu + (t & 1) * P.KC;   // this token's exchange slot
    // x: lane l owns quantisation group l (64 inputs)
    uint4 xr[8];
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8)
      xr[c8] = !active ? make_uint4(0u, 0u, 0u, 0u)
               : !kMulti ? xs[(lane * 8 + c8) ^ (lane & 7)]
               : P.x_smem ? reinterpret_cast<const uint4*>(sm + P.xs)[t * (d / 8) + ((lane * 8 + c8) ^ (lane & 7))]
                          : __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * d) + lane * 8 + c8);

    // ---- gate/up: warp w computes gate and up of rows q*8 + w (q = 0..3) as slots s = 2q + mat;
    // a reduce-scatter leaves slot s fully summed in lane 4s.
    Planes xp;
    if (!planes_of_bf16(xr, xp) && active) raise_flag(a.err, kErrNonFinite);
    const float xsum = xp.sum;
    float v8[8];
#pragma unroll
    for (int sl = 0; sl < 8; ++sl) v8[sl] = 0.0f;
#pragma unroll 1
    for (int q = 0; q < kQuarters; ++q) {
      const bool ok = mbar_wait_warp(smem_u32(&bars[q]), ph, &abort_s, a.err);
#pragma unroll
      for (int mat = 0; mat < 2; ++mat) {
        const int row = q * kRQ + warp;
        float v = 0.0f;
        if (active && ok) {
          const uint32_t* cw = gcodes + (mat * RF + row) * (d / 8) + lane * 8;
          const uint4 c0 = *reinterpret_cast<const uint4*>(cw);
          const uint4 c1 = *reinterpret_cast<const uint4*>(cw + 4);
          const float p = group_dot(c0, c1, xp);
          const float s = bf16_bits_to_f32(gsb[((2 * mat) * RF + row) * G + lane]);
          const float b = bf16_bits_to_f32(gsb[((2 * mat + 1) * RF + row) * G + lane]);
          v = fmaf(s, p, b * xsum);
        }
        const int sl = 2 * q + mat;
#pragma unroll
        for (int i = 0; i < 8; ++i) v8[i] = (i == sl) ? v : v8[i];
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
        hloc[(lane >> 3) * kRQ + warp] = gv / (1.0f + expf(-gv)) * upv;   // h of row (lane / 8) * 8 + warp
      }
    }
    __syncthreads();   // the CTA's 32 h values are in hloc; its gate/up reads are done
    if (warp == 0) {
      // The 32 h values (columns 32 crank .. + 31 of the cluster) as one planes block, written into
      // every cluster CTA's exchange slot: lane l holds column l; lanes 0..23 build plane word
      // lane % 8 of plane lane / 8, lane 24 the exponent, lane 25 the sum.
      const float hv = hloc[lane];
      if (!(fabsf(hv) <= 3.402823466e38f)) raise_flag(a.err, kErrNonFinite);
      const uint32_t mb = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(hv) & 0x7FFFFFFFu);
      float hs = hv;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) hs += __shfl_xor_sync(0xFFFFFFFFu, hs, off);
      const int e = block_exponent(mb);
      vloc[lane] = fixed23(hv, pow2i(22 - e));
      __syncwarp();
      uint32_t word = 0;
      if (lane < 24) {
        const int pl = lane >> 3, wi = lane & 7, w = wi >> 1, o = wi & 1;
        uint32_t hi, mid, lo;
        pack4(vloc[8 * w + o], vloc[8 * w + 2 + o], vloc[8 * w + 4 + o], vloc[8 * w + 6 + o], hi, mid, lo);
        word = pl == 0 ? hi : pl == 1 ? mid : lo;
      } else if (lane == 24) {
        word = __float_as_uint(pow2i(e - 22));
      } else if (lane == 25) {
        word = __float_as_uint(hs);
      }
      if (lane < 26) {
        const uint32_t loc = smem_u32(hx + crank * kHBlockWords + lane);
#pragma unroll
        for (int r = 0; r < C; ++r) st_cluster_u32(cluster_map(loc, (uint32_t)r), word);
      }
    }
    cluster_arrive_release();   // this CTA's h block is in every cluster CTA's slot
    // The gate/up buffers are free once the whole CTA is past the gate/up reads: the next token's
    // gate/up rows are requested while this token's down share runs.  abort_s is only written
    // inside waits, so every thread of the CTA reads the same value here after the wait below.
    cluster_wait_acquire();     // every CTA's h has arrived
    if (kMulti && warp == 0 && t + 1 < T && e_s[t + 1] != e_t && !abort_s) {
      // this token ends its run: the gate/up buffers are free
      fence_proxy_async_smem();   // this token's generic reads of the gate/up buffers come first
      issue(e_s[t + 1], 5);
    }

    // ---- down share: rows r0 .. r0+DR-1 over the cluster's columns kc0 .. kc0+KC-1.  GP lanes per
    // row, lane g taking quantisation group g of the columns; GP-lane butterfly; the group-0 lane
    // stores wgt * (sum_g s_g sum q h + b_g sum h) as this CTA's partial of the row.  Two rows per
    // lane and iteration, their shared-memory loads issued together.
    const bool ok_dn = mbar_wait_warp(smem_u32(&bars[kQuarters]), ph, &abort_s, a.err);
    {
      constexpr int GP = kC * RF / 64;
      constexpr int rpp = 32 / GP;   // rows per warp pass
      const int g = lane % GP;
      // group g of the cluster's columns: the h blocks of CTAs 2g (code words 0..3) and 2g + 1 (4..7)
      Planes hp;
      {
        const uint32_t* blk = reinterpret_cast<const uint32_t*>(hx) + 2 * g * kHBlockWords;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t* bh = blk + half * kHBlockWords;
#pragma unroll
          for (int pl = 0; pl < 3; ++pl) {
            const uint4 u0 = *reinterpret_cast<const uint4*>(bh + 8 * pl);
            const uint4 u1 = *reinterpret_cast<const uint4*>(bh + 8 * pl + 4);
            hp.p[pl][8 * half + 0] = u0.x;
            hp.p[pl][8 * half + 1] = u0.y;
            hp.p[pl][8 * half + 2] = u0.z;
            hp.p[pl][8 * half + 3] = u0.w;
            hp.p[pl][8 * half + 4] = u1.x;
            hp.p[pl][8 * half + 5] = u1.y;
            hp.p[pl][8 * half + 6] = u1.z;
            hp.p[pl][8 * half + 7] = u1.w;
          }
          hp.scale[half] = __uint_as_float(bh[24]);
        }
        hp.sum = __uint_as_float(blk[25]) + __uint_as_float(blk[kHBlockWords + 25]);
      }
      const float hsum = hp.sum;
      const float wgt = wgt_s[t];
      const int gcol = kc0 / 64 + g;
      float* part_t = a.part + (size_t)t * P.nslices * P.NP * kSliceRows;
      const int p = j * P.NQ + qc;
#pragma unroll 1
      for (int pass = warp; pass * rpp < P.DR; pass += 2 * kWarpsDec) {
        int r[2];
        uint4 c[2][2];
        float sc[2], bi[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          r[u] = (pass + u * kWarpsDec) * rpp + lane / GP;
          const bool in = r[u] < P.DR && ok_dn;
          const uint32_t* cw = dcodes + (in ? r[u] : 0) * (P.KC / 8) + g * 8;
          c[u][0] = *reinterpret_cast<const uint4*>(cw);
          c[u][1] = *reinterpret_cast<const uint4*>(cw + 4);
          sc[u] = bf16_bits_to_f32(dsb[(in ? r[u] : 0) * GF + gcol]);
          bi[u] = bf16_bits_to_f32(dsb[(P.DR + (in ? r[u] : 0)) * GF + gcol]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float pq = group_dot(c[u][0], c[u][1], hp);
          float v = fmaf(sc[u], pq, bi[u] * hsum);
#pragma unroll
          for (int off = GP >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
          if (g == 0 && r[u] < P.DR) {
            const int sl = crank * P.NSC + r[u] / kSliceRows;
            part_t[((size_t)sl * P.NP + p) * kSliceRows + r[u] % kSliceRows] = wgt * v;
          }
        }
      }
    }
    __syncthreads();   // this token's partials are stored; the down buffers are free
    if (kMulti && warp == 0 && t + 1 < T && e_s[t + 1] != e_t && !abort_s) {
      fence_proxy_async_smem();   // this token's generic reads of the down buffers come first
      issue(e_s[t + 1], 2);
    }

  }

  // ---- wind down: after a timeout, copies still in flight must land before the CTA exits.
  if (tid == 0 && abort_s) {
    // every barrier waits for the parity of its last fetch (thread 0 armed them all)
    for (int i = 0; i <= kQuarters; ++i) {
      const int n = !kMulti ? 1 : i < kQuarters ? gu_issued : dn_issued;
      if (n == 0) continue;
      const uint32_t last = (uint32_t)(n - 1) & 1u;
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(&bars[i]), last) && clock64() - t0 < 4000000ll) {
      }
    }
  }
}

// Loads-only replica of decode_layer_kernel's weight traffic for one token, a measurement aid
// (the bandwidth ceiling of this access pattern): same grid, clusters, shared-memory plan,
// programmatic launch and weight copies, with the experts given instead of routed; it waits for
// every copy to land and does no arithmetic.
__global__ void __launch_bounds__(kThreadsDec, 2)
    decode_stream_kernel(const __grid_constant__ DecodeMaps maps, const StreamArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int k1 = a.k + (a.has_shared ? 1 : 0);
  const DecPlan P(a.d, a.F, k1, false);
  const int tid = threadIdx.x;
  const int cta = blockIdx.x;
  const int j = cta / P.S;
  const int sidx = cta % P.S;
  const int kc0 = (sidx / kC) * P.KC;
  const int r0 = (sidx % kC) * P.DR;
  const int f0 = sidx * RF;
  const bool shared_cta = (j == a.k);
  const int wset = shared_cta ? 1 : 0;
  __shared__ __align__(8) uint64_t bars[kQuarters + 1];
  __shared__ int abort_s;
  if (tid == 0) {
    for (int i = 0; i <= kQuarters; ++i) mbar_init(smem_u32(&bars[i]), 1);
    abort_s = 0;
    mbar_fence_init();
  }
  __syncthreads();
  auto issue = [&](int e) {
    issue_copies(P, a.gate[wset], a.up[wset], a.down[wset], &maps.down[wset], e, f0, r0, kc0,
                 smem_u32(sm + P.gu_codes), smem_u32(sm + P.gu_sb), smem_u32(sm + P.dn_codes),
                 smem_u32(sm + P.dn_sb), smem_u32(&bars[0]), 7, tid & 31);
  };
  if (shared_cta && tid < 32) issue(0);
  pdl_wait();
  if (!shared_cta && tid < 32) issue(__ldg(a.idx + j));   // the same copies as the layer kernel, all at once
  pdl_launch_dependents();
  for (int i = 0; i <= kQuarters; ++i) mbar_wait_warp(smem_u32(&bars[i]), 0, &abort_s, a.err);
  __syncthreads();
  if (tid == 0 && abort_s) {   // copies still in flight land before the CTA exits
    for (int i = 0; i <= kQuarters; ++i) {
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(&bars[i]), 0) && clock64() - t0 < 4000000ll) {
      }
    }
  }
}

// y[t][r] = the sum of the NP partials of row r, one warp per four rows (float4), lane l summing
// partials l, l + 32, ... in order (the first two loads in flight together), then a 32-lane butterfly: every lane ends with the same bits,
// whatever the order in which the decode CTAs finished.  Grid (d / 32, T), 256 threads.
__global__ void __launch_bounds__(256) decode_reduce_kernel(const ReduceArgs a) {
  // The next launch on the stream may start its prologue now: a decode launch reads nothing written
  // here or by the decode launch before its own dependency wait.
  pdl_launch_dependents();
  pdl_wait();   // every partial of the decode launch is stored
  const DecPlan P(a.d, a.F, a.k1, false);
  const int t = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 32 + warp * 4;
  if (r >= a.d) return;
  const int crank = r / P.DR, i = (r % P.DR) / kSliceRows, rr = (r % P.DR) % kSliceRows;
  const int sl = crank * P.NSC + i;
  const float4* base =
      reinterpret_cast<const float4*>(a.part + ((size_t)t * P.nslices + sl) * P.NP * kSliceRows + rr);
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 v0 = lane < P.NP ? __ldcg(base + (size_t)lane * (kSliceRows / 4)) : z;
  const float4 v1 = lane + 32 < P.NP ? __ldcg(base + (size_t)(lane + 32) * (kSliceRows / 4)) : z;
  float4 acc = make_float4(v0.x + v1.x, v0.y + v1.y, v0.z + v1.z, v0.w + v1.w);
  for (int p = lane + 64; p < P.NP; p += 32) {
    const float4 v = __ldcg(base + (size_t)p * (kSliceRows / 4));
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    acc.x += __shfl_xor_sync(0xFFFFFFFFu, acc.x, off);
    acc.y += __shfl_xor_sync(0xFFFFFFFFu, acc.y, off);
    acc.z += __shfl_xor_sync(0xFFFFFFFFu, acc.z, off);
    acc.w += __shfl_xor_sync(0xFFFFFFFFu, acc.w, off);
  }
  if (lane == 0) *reinterpret_cast<float4*>(a.y + (size_t)t * a.d + r) = acc;
}

constexpr int kMaxDev = 64;
bool g_ready[kMaxDev];
std::mutex g_dev_mu;
constexpr size_t kDecSmemMax = kDecPlanMax;

cudaError_t ensure_attrs() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!g_ready[dev]) {
    if ((e = cudaFuncSetAttribute(decode_layer_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kDecPlanMax)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(decode_layer_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kDecPlanMaxMulti)) != cudaSuccess)
      return e;
    for (auto f : {decode_layer_kernel<false>, decode_layer_kernel<true>}) {
      if ((e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100)) != cudaSuccess) return e;
    }
    if ((e = cudaFuncSetAttribute(decode_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kDecSmemMax)) != cudaSuccess)
      return e;
    g_ready[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

size_t decode_scratch_floats(int d, int k, int F) {
  const DecPlan P(d, F, k + 1, false);
  return (size_t)P.nslices * P.NP * kSliceRows;
}

bool decode_supported(int d, int E, int k, int F) {
  const int k1 = k + 1;
  // One quantisation group per lane in the gate/up rows: d <= 2048 (and d a multiple of 64).
  // F a multiple of 128: 32 gate/up rows per CTA and whole quantisation groups per cluster.
  if (k1 > 32 || E > kMaxE || d > 2048 || d % 64 != 0 || F % 128 != 0) return false;
  if (DecPlan(d, F, k1, false).bytes > kDecPlanMax || DecPlan(d, F, k1, true).bytes > kDecPlanMaxMulti) return false;
  return true;
}

constexpr int kStageThreads = 256;
constexpr int kStageIn = 4;   // loads in flight per thread per round

__global__ void __launch_bounds__(kStageThreads) stage_in_kernel(const StageArgs a) {
  // Rounds of kStageIn 16-byte loads of x and kStageIn loads of logits per thread.  The stores go
  // to workspace buffers that the previous kernel may still read, so they follow the dependency
  // wait; with a.early the host inputs are final when the call is made and the first round of
  // reads goes out before the wait (its latency across the CPU-GPU link overlaps that kernel).
  const int tid = threadIdx.x;
  constexpr int kStep = kStageThreads * kStageIn;
  uint4 xv[kStageIn];
  float lv[kStageIn];
  auto load = [&](int base) {
#pragma unroll
    for (int c = 0; c < kStageIn; ++c) {
      const int i = base + c * kStageThreads + tid;
      if (i < a.x_units) xv[c] = a.x_src[i];
      if (i < a.lg_n) lv[c] = a.lg_src[i];
    }
  };
  auto store = [&](int base) {
#pragma unroll
    for (int c = 0; c < kStageIn; ++c) {
      const int i = base + c * kStageThreads + tid;
      if (i < a.x_units) a.x_dst[i] = xv[c];
      if (i < a.lg_n) a.lg_dst[i] = lv[c];
    }
  };
  if (a.early) load(0);
  pdl_wait();   // the previous kernel, the last reader of the destination buffers, is complete
  pdl_launch_dependents();
  if (!a.early) load(0);
  store(0);
  const int n = a.x_units > a.lg_n ? a.x_units : a.lg_n;
  for (int base = kStep; base < n; base += kStep) {
    load(base);
    store(base);
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

static_assert(kDecodeMaxTokens <= kWarpsDec, "one routing warp per token");
static_assert(kC * RF % 64 == 0 && 32 % (kC * RF / 64) == 0, "whole quantisation groups per cluster");
static_assert(kDecodeLayerMaxT <= kDecodeMaxTokens, "the layer path's decode calls fit one launch");

int decode_box_rows(int d, int F) { return DecPlan(d, F, 1, false).box_rows; }

cudaError_t launch_decode(const DecodeMaps& maps, const DecodeArgs& a, cudaStream_t st, bool pdl) {
  if (a.T > kDecodeMaxTokens) return cudaErrorInvalidValue;
  const int k1 = a.k + (a.has_shared ? 1 : 0);
  if (!decode_supported(a.d, a.E, a.k, a.F)) return cudaErrorInvalidConfiguration;
  cudaError_t e = ensure_attrs();
  if (e != cudaSuccess) return e;
  const DecPlan P(a.d, a.F, k1, a.T > 1, a.T > 0 ? a.T : 1);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid);
  cfg.blockDim = dim3(kThreadsDec);
  cfg.dynamicSmemBytes = P.bytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  e = a.T > 1 ? cudaLaunchKernelEx(&cfg, decode_layer_kernel<true>, maps, a)
              : cudaLaunchKernelEx(&cfg, decode_layer_kernel<false>, maps, a);
  if (e != cudaSuccess) return e;
  // The fixed-order sum of the partials, launched to start as soon as the decode launch allows.
  ReduceArgs ra{a.part, a.y, a.d, a.F, k1};
  cudaLaunchConfig_t rc = {};
  rc.gridDim = dim3((unsigned)((a.d + 31) / 32), (unsigned)(a.T > 0 ? a.T : 1));
  rc.blockDim = dim3(256);
  rc.stream = st;
  rc.attrs = &attr[1];
  rc.numAttrs = 1;
  e = cudaLaunchKernelEx(&rc, decode_reduce_kernel, ra);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_decode_stream(const DecodeMaps& maps, const StreamArgs& a, cudaStream_t st) {
  if (!decode_supported(a.d, a.E, a.k, a.F)) return cudaErrorInvalidConfiguration;
  cudaError_t e = ensure_attrs();
  if (e != cudaSuccess) return e;
  const DecPlan P(a.d, a.F, a.k + (a.has_shared ? 1 : 0), false);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid);
  cfg.blockDim = dim3(kThreadsDec);
  cfg.dynamicSmemBytes = P.bytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, decode_stream_kernel, maps, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
