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


// E <= 256 variant with shorter rounds: every lane first sorts its 8 candidates (a 19-comparator
// sorting network on (key, lower index first)), so a round only compares the lanes' heads:
// redux.sync max, a ballot for ties (a second reduction, over expert indices, only when several
// lanes hold the maximum) and a shift of the winning lane's list.
__device__ __forceinline__ void warp_topk_softmax_sorted8(const float* __restrict__ row, int E, int k, int* e_out,
                                                          float* w_out) {
  const int lane = threadIdx.x & 31;
  uint64_t rk[8];   // key << 8 | (7 - i): larger first, equal keys -> lower i first
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    const float x = e < E ? __ldg(row + e) : 0.0f;
    rk[i] = ((uint64_t)(e < E ? logit_key(x) : 0u) << 8) | (uint64_t)(7 - i);
    v[i] = x;
  }
  auto cas = [&](int a, int b) {
    const bool sw = rk[a] < rk[b];
    const uint64_t ra = rk[a], rb = rk[b];
    const float va = v[a], vb = v[b];
    rk[a] = sw ? rb : ra;
    rk[b] = sw ? ra : rb;
    v[a] = sw ? vb : va;
    v[b] = sw ? va : vb;
  };
  cas(0, 1); cas(2, 3); cas(4, 5); cas(6, 7);
  cas(0, 2); cas(1, 3); cas(4, 6); cas(5, 7);
  cas(1, 2); cas(5, 6);
  cas(0, 4); cas(1, 5); cas(2, 6); cas(3, 7);
  cas(2, 4); cas(3, 5);
  cas(1, 2); cas(3, 4); cas(5, 6);
  int my_e = 0;
  float my_v = 0.0f;
  for (int j = 0; j < k; ++j) {
    const uint32_t hk = (uint32_t)(rk[0] >> 8);
    const int hidx = lane + 32 * (7 - (int)(rk[0] & 0xFFu));
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, hk);
    const uint32_t tie = __ballot_sync(0xFFFFFFFFu, hk == m);
    int wl;
    if (__popc(tie) == 1) {
      wl = __ffs(tie) - 1;
    } else {
      wl = (int)(__reduce_min_sync(0xFFFFFFFFu, hk == m ? (uint32_t)hidx : 0xFFFFFFFFu) & 31u);
    }
    const int widx = __shfl_sync(0xFFFFFFFFu, hidx, wl);
    const float wv = __shfl_sync(0xFFFFFFFFu, v[0], wl);
    if (lane == j) {
      my_e = widx;
      my_v = wv;
    }
    const bool me = lane == wl;
#pragma unroll
    for (int i = 0; i < 7; ++i) {
      rk[i] = me ? rk[i + 1] : rk[i];
      v[i] = me ? v[i + 1] : v[i];
    }
    rk[7] = me ? 0ull : rk[7];
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
