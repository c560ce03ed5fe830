// GPU-resident routing of the MoE layer: top-k selection and weights per token, then the
// histogram, exclusive scan, scatter (permutation) and block map of the grouped GEMM, all on
// the device with no host synchronisation ("Perplexity libera Lily: inferencia en Rust y Metal
// para Mac", section "Prefill: pesos comprimidos y enrutamiento en la GPU": the routing
// histogram, prefix scan, scatter and block map stay in one GPU command stream).
//
// Kernel 1 (one warp per token): top-k over fp32 logits with ties to the lower expert index,
// softmax over the selected logits, and the shared expert gate sigmoid(x . w_sg).
// Kernel 2 (one CTA): per-expert counts, exclusive offsets, a permutation sorted by
// (expert, token) that depends only on the counts (never on atomic arrival order), its
// inverse and the tile block map.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

template <int NI>
__global__ void __launch_bounds__(256) topk_kernel(RouteArgs a) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= a.T) return;
  int my_e;
  float my_w;
  warp_topk_softmax<NI>(a.logits + (size_t)t * a.E, a.E, a.k, &my_e, &my_w);
  if (lane < a.k) {
    a.idx[(size_t)t * a.k + lane] = my_e;
    a.w[(size_t)t * a.k + lane] = my_w;
  }

  // Shared-expert gate logit x . w_sg (one pass over the token row).
  if (a.x != nullptr && a.gs != nullptr && a.w_sg != nullptr) {
    const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)t * a.d);
    const uint4* wr = reinterpret_cast<const uint4*>(a.w_sg);
    float dot = 0.0f;
    for (int ch = lane; ch < a.d / 8; ch += 32) {
      const uint4 xv = __ldg(xr + ch), wv = __ldg(wr + ch);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dot = fmaf(bf16_bits_to_f32(xw[i] & 0xFFFFu), bf16_bits_to_f32(ww[i] & 0xFFFFu), dot);
        dot = fmaf(bf16_bits_to_f32(xw[i] >> 16), bf16_bits_to_f32(ww[i] >> 16), dot);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
    if (lane == 0) a.gs[t] = 1.0f / (1.0f + expf(-dot));
  }
}

// Exclusive scan over the block (blockDim.x == 1024); every thread passes one value.
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  __syncthreads();
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int wv = warp_tot[lane];
    int wi = wv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, wi, off);
      if (lane >= off) wi += o;
    }
    warp_tot[lane] = wi - wv;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  return incl - v + warp_tot[warp];
}

// Warps that walk the tokens in kernel 2: 32 when their per-warp tables (2 x E ints each) fit
// in 96 KB, fewer for large E.
__host__ __device__ constexpr int tok_warps(int E) { return (96 * 1024) / (8 * E) >= 32 ? 32 : (96 * 1024) / (8 * E); }

// The k expert ids of token t, loaded together (independent loads, one latency); -1 past T or k.
template <int KMAX>
__device__ __forceinline__ void load_token_ids(const int32_t* __restrict__ idx, int t, int T, int k, int E,
                                               int (&ev)[KMAX], uint32_t* err) {
#pragma unroll
  for (int j = 0; j < KMAX; ++j) ev[j] = (j < k && t < T) ? __ldg(idx + (size_t)t * k + j) : -1;
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    if (j < k && t < T && (unsigned)ev[j] >= (unsigned)E) {
      raise_flag(err, kErrBadRouting);
      ev[j] = -1;
    }
}

// KMAX: upper bound on k held in registers per token (8 or 32).
template <int KMAX>
__global__ void __launch_bounds__(1024, 1) tables_kernel(TablesArgs a) {
  extern __shared__ int tsm[];
  const int kTokWarps = tok_warps(a.E);
  int* base = tsm;                                       // [kTokWarps][E]: counts, then running slots
  uint32_t* mask = reinterpret_cast<uint32_t*>(tsm + kTokWarps * a.E);   // [kTokWarps][E]
  __shared__ int warp_tot[32];
  __shared__ int total_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, k = a.k, T = a.T;

  for (int i = tid; i < kTokWarps * E; i += blockDim.x) {
    base[i] = 0;
    mask[i] = 0u;
  }
  __syncthreads();

  const int nchunks = (T + 31) / 32;
  const int c_lo = (int)((long long)warp * nchunks / kTokWarps);
  const int c_hi = (int)((long long)(warp + 1) * nchunks / kTokWarps);

  // Pass A: per-warp histogram of the warp's contiguous token range.
  if (warp < kTokWarps) {
    int* hw = base + warp * E;
    for (int c = c_lo; c < c_hi; ++c) {
      int ev[KMAX];
      load_token_ids<KMAX>(a.idx, c * 32 + lane, T, k, E, ev, a.err);
      // lanes routing to the same expert in round j add their count once (hot experts would
      // otherwise serialise 32 atomics on one word)
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
          const uint32_t m = __match_any_sync(0xFFFFFFFFu, ev[j]);
          if (ev[j] >= 0 && lane == __ffs(m) - 1) atomicAdd(&hw[ev[j]], __popc(m));
        }
      }
    }
  }
  __syncthreads();

  // Pass B: per expert, exclusive prefix over warps (warp order = token order) and the total.
  int cnt = 0;
  if (tid < E) {
    int run = 0;
    for (int w = 0; w < kTokWarps; ++w) {
      const int c = base[w * E + tid];
      base[w * E + tid] = run;
      run += c;
    }
    cnt = run;
    a.counts[tid] = run;
  }
  const int off = block_excl_scan(cnt, warp_tot, &total_s);
  if (tid < E) {
    a.offsets[tid] = off;
    for (int w = 0; w < kTokWarps; ++w) base[w * E + tid] += off;   // absolute first slot
  }
  if (tid == 0) a.offsets[E] = total_s;
  // Block map: ceil(count / tile_n) tiles per non-empty expert, then the shared expert.
  const int nt = (tid < E) ? (cnt + a.tile_n - 1) / a.tile_n : 0;
  const int tile0 = block_excl_scan(nt, warp_tot, &total_s);
  const int routed_tiles = total_s;
  for (int i = 0; i < nt; ++i) {
    int4 r;
    r.x = tid;
    r.y = off + i * a.tile_n;
    r.z = min(a.tile_n, cnt - i * a.tile_n);
    r.w = 0;
    reinterpret_cast<int4*>(a.tiles)[tile0 + i] = r;
  }
  const int shared_tiles = a.has_shared ? (T + a.tile_n - 1) / a.tile_n : 0;
  for (int i = tid; i < shared_tiles; i += blockDim.x) {
    int4 r;
    r.x = E;
    r.y = T * k + i * a.tile_n;
    r.z = min(a.tile_n, T - i * a.tile_n);
    r.w = 0;
    reinterpret_cast<int4*>(a.tiles)[routed_tiles + i] = r;
  }
  if (tid == 0) *a.num_tiles = routed_tiles + shared_tiles;
  __syncthreads();

  // Pass C: slots.  Within a 32-token chunk, a bit mask per expert gives each assignment the
  // number of earlier tokens of the chunk routed to the same expert; the warp's running slot
  // per expert carries the count across chunks.  Every slot follows from the counts alone.
  if (warp < kTokWarps) {
    int* run = base + warp * E;
    uint32_t* mk = mask + warp * E;
    const uint32_t lt = (1u << lane) - 1u;
    for (int c = c_lo; c < c_hi; ++c) {
      const int t = c * 32 + lane;
      int ev[KMAX];
      load_token_ids<KMAX>(a.idx, t, T, k, E, ev, nullptr);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
          const uint32_t m = __match_any_sync(0xFFFFFFFFu, ev[j]);
          if (ev[j] >= 0 && lane == __ffs(m) - 1) atomicOr(&mk[ev[j]], m);
        }
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (ev[j] >= 0) {
          const uint32_t m = mk[ev[j]];
          const int slot = run[ev[j]] + __popc(m & lt);
          a.perm[slot] = t * k + j;
          a.inv[(size_t)t * k + j] = slot;
        }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (ev[j] >= 0) {
          const uint32_t m = mk[ev[j]];
          if (lane == 31 - __clz(m)) run[ev[j]] += __popc(m);   // last token of the chunk for e
        }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (ev[j] >= 0) mk[ev[j]] = 0u;
      __syncwarp();
    }
  }
}

cudaError_t launch_topk(const RouteArgs& a, cudaStream_t st) {
  const int warps = 8;
  const dim3 grid((a.T + warps - 1) / warps), block(32 * warps);
  const int ni = (a.E + 31) / 32;
  if (ni <= 1) topk_kernel<1><<<grid, block, 0, st>>>(a);
  else if (ni <= 2) topk_kernel<2><<<grid, block, 0, st>>>(a);
  else if (ni <= 4) topk_kernel<4><<<grid, block, 0, st>>>(a);
  else if (ni <= 8) topk_kernel<8><<<grid, block, 0, st>>>(a);
  else if (ni <= 16) topk_kernel<16><<<grid, block, 0, st>>>(a);
  else topk_kernel<32><<<grid, block, 0, st>>>(a);
  return cudaGetLastError();
}

size_t tables_smem_bytes(int E) { return (size_t)2 * tok_warps(E) * E * sizeof(int); }

cudaError_t launch_tables(const TablesArgs& a, cudaStream_t st) {
  const size_t smem = tables_smem_bytes(a.E);
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(tables_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(96 * 1024));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tables_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(96 * 1024));
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  if (a.k <= 8) tables_kernel<8><<<1, 1024, smem, st>>>(a);
  else tables_kernel<32><<<1, 1024, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
