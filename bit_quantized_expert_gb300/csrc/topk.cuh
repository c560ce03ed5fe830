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
// NI = ceil(E / 32) candidates per lane (compile-time upper bound).
template <int NI>
__device__ __forceinline__ void warp_topk_softmax(const float* __restrict__ row, int E, int k, int* e_out,
                                                  float* w_out) {
  const int lane = threadIdx.x & 31;
  uint64_t comb[NI];
  float val[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    float v = 0.0f;
    uint64_t c = 0;
    if (e < E) {
      v = __ldg(row + e);
      c = ((uint64_t)logit_key(v) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e);
    }
    comb[i] = c;
    val[i] = v;
  }
  int my_e = 0;
  float my_v = 0.0f;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
    float bestv = 0.0f;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      if (comb[i] > best) {
        best = comb[i];
        bestv = val[i];
        bi = i;
      }
    }
    uint64_t m = best;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, m, off);
      m = o > m ? o : m;
    }
    const int e_win = (int)(0xFFFFFFFFu - (uint32_t)(m & 0xFFFFFFFFu));
    const float v_win = __shfl_sync(0xFFFFFFFFu, bestv, e_win & 31);
    if (best == m && m != 0) {
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (i == bi) comb[i] = 0;
    }
    if (lane == j) {
      my_e = e_win;
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

}  // namespace moe
