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

// Inverse of logit_key for keys of real logits: -0.0 comes back as +0.0 and every NaN as one
// NaN, which leaves the softmax below unchanged.
__device__ __forceinline__ float key_logit(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Lane j < k returns the j-th expert in *e_out and its routing weight in *w_out.
// NI = ceil(E / 32) candidates per lane (compile-time upper bound), lane l holding l + 32 i.
// Each round takes the lane's best candidate by a tree (the lower index wins a tie), the largest
// key over the warp with redux.sync max and, among the lanes holding it, the lowest expert index
// with redux.sync min; the owning lane then clears that candidate.  The winner's logit is the
// inverse of its key (no broadcast); no lane branches inside a round.
template <int NI>
__device__ __forceinline__ void warp_topk_softmax(const float* __restrict__ row, int E, int k, int* e_out,
                                                  float* w_out) {
  const int lane = threadIdx.x & 31;
  uint32_t key[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? logit_key(__ldg(row + e)) : 0u;
  }
  int my_e = 0;
  float my_v = 0.0f, vmax = 0.0f;
  for (int j = 0; j < k; ++j) {
    uint32_t tk[NI], ti[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      tk[i] = key[i];
      ti[i] = (uint32_t)i;
    }
#pragma unroll
    for (int w = 1; w < NI; w <<= 1) {
#pragma unroll
      for (int i = 0; i + w < NI; i += 2 * w) {
        const bool r = tk[i + w] > tk[i];   // strict: the left (lower index) wins a tie
        tk[i] = r ? tk[i + w] : tk[i];
        ti[i] = r ? ti[i + w] : ti[i];
      }
    }
    const uint32_t best = tk[0];
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, best);
    const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, best == m ? (uint32_t)lane + 32u * ti[0] : 0xFFFFFFFFu);
    const int sel = (lane == (int)(win & 31u)) ? (int)(win >> 5) : -1;
#pragma unroll
    for (int i = 0; i < NI; ++i) key[i] = (i == sel) ? 0u : key[i];
    const float v = key_logit(m);
    vmax = j == 0 ? v : vmax;
    my_e = lane == j ? (int)win : my_e;
    my_v = lane == j ? v : my_v;
  }
  const float my_ex = lane < k ? expf(my_v - vmax) : 0.0f;
  float s = my_ex;   // lanes >= k hold 0
  if (k > 8) {
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 16);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 8);
  }
  s += __shfl_xor_sync(0xFFFFFFFFu, s, 4);
  s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
  s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
  *e_out = my_e;
  *w_out = my_ex / s;
}

}  // namespace moe
