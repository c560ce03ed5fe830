// Warp-wide top-k of one row of fp32 router logits (descending, ties to the lower expert index,
// -0.0 == +0.0, NaN below every number) and the softmax of the selected logits.
#pragma once
#include "common.cuh"

namespace moe {

// Order-preserving 32-bit key of an fp32 logit: larger key = larger logit, -0.0 == +0.0,
// every NaN maps to 1 (below -inf, whose key is 0x007FFFFF); 0 marks padding / taken.
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (v != v) return 1u;
  uint32_t u = (v == 0.0f) ? 0u : __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Lane j < k returns the j-th expert in *e_out and its routing weight in *w_out.
// NI = ceil(E / 32) candidates per lane (compile-time upper bound), lane l holding l + 32 i.
// Each round takes the largest key with redux.sync max and, among the lanes holding it, the
// lowest expert index with redux.sync min; the owning lane then clears that candidate.
template <int NI>
__device__ __forceinline__ void warp_topk_softmax(const float* __restrict__ row, int E, int k, int* e_out,
                                                  float* w_out) {
  const int lane = threadIdx.x & 31;
  uint32_t key[NI];
  float val[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    const float v = e < E ? __ldg(row + e) : 0.0f;
    key[i] = e < E ? logit_key(v) : 0u;
    val[i] = v;
  }
  int my_e = 0;
  float my_v = 0.0f;
  for (int j = 0; j < k; ++j) {
    uint32_t best = 0u, bi = 0xFFFFFFFFu;
    float bestv = 0.0f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      if (key[i] > best) {   // strict: this lane's lowest index wins its ties
        best = key[i];
        bi = (uint32_t)(lane + 32 * i);
        bestv = val[i];
      }
    }
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, best);
    const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, best == m ? bi : 0xFFFFFFFFu);
    const float v_win = __shfl_sync(0xFFFFFFFFu, bestv, (int)(win & 31u));
    const int sel = (lane == (int)(win & 31u)) ? (int)(win >> 5) : -1;
#pragma unroll
    for (int i = 0; i < NI; ++i) key[i] = (i == sel) ? 0u : key[i];
    if (lane == j) {
      my_e = (int)win;
      my_v = v_win;
    }
  }
  const float vmax = __shfl_sync(0xFFFFFFFFu, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - vmax) : 0.0f;
  float s = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
  *e_out = my_e;
  *w_out = ex / s;
}


// E <= 256 and k <= 8, without sequential selection rounds: every lane sorts its 8 candidates
// (Batcher's 19-comparator network), then five butterfly levels merge the lane's sorted top-8
// with that of lane ^ m: the elementwise maximum of one list and the other reversed is a bitonic
// sequence holding the 8 largest of both, which a 12-comparator bitonic merge sorts.  Partners
// compute the same list, so after the last level every lane holds the row's sorted top-8.  A
// candidate is (key << 32 | ~index): equal logits go to the lower expert index, and padding (0)
// sorts below every logit.  Lane j < k returns the j-th expert and its routing weight.
__device__ __forceinline__ void warp_top8_softmax(const float* __restrict__ row, int E, int k, int* e_out,
                                                  float* w_out) {
  const int lane = threadIdx.x & 31;
  uint64_t c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    c[i] = e < E ? ((uint64_t)logit_key(__ldg(row + e)) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e) : 0ull;
  }
  auto cas = [&](int a, int b) {   // c[a] >= c[b] afterwards
    const uint64_t x = c[a], y = c[b];
    const bool sw = x < y;
    c[a] = sw ? y : x;
    c[b] = sw ? x : y;
  };
  cas(0, 1); cas(2, 3); cas(4, 5); cas(6, 7);
  cas(0, 2); cas(1, 3); cas(4, 6); cas(5, 7);
  cas(1, 2); cas(5, 6);
  cas(0, 4); cas(1, 5); cas(2, 6); cas(3, 7);
  cas(2, 4); cas(3, 5);
  cas(1, 2); cas(3, 4); cas(5, 6);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    uint64_t p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = __shfl_xor_sync(0xFFFFFFFFu, c[i], m);
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = c[i] > p[7 - i] ? c[i] : p[7 - i];
    cas(0, 4); cas(1, 5); cas(2, 6); cas(3, 7);
    cas(0, 2); cas(1, 3); cas(4, 6); cas(5, 7);
    cas(0, 1); cas(2, 3); cas(4, 5); cas(6, 7);
  }
  uint64_t mine = 0ull;
#pragma unroll
  for (int i = 0; i < 8; ++i) mine = (lane == i) ? c[i] : mine;
  const int my_e = lane < k ? (int)(0xFFFFFFFFu - (uint32_t)mine) : 0;
  const float my_v = lane < k ? __ldg(row + my_e) : 0.0f;
  const float vmax = __shfl_sync(0xFFFFFFFFu, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - vmax) : 0.0f;
  float s = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
  *e_out = my_e;
  *w_out = ex / s;
}

}  // namespace moe
