// GPU-resident routing of the MoE layer: top-k selection and weights per token, then the
// histogram, exclusive scan, scatter (permutation) and block map of the grouped GEMM, all on
// the device with no host synchronisation ("Perplexity libera Lily: inferencia en Rust y Metal
// para Mac", section "Prefill: pesos comprimidos y enrutamiento en la GPU": the routing
// histogram, prefix scan, scatter and block map stay in one GPU command stream).
//
// Kernel 1 (one warp per token): top-k over fp32 logits with ties to the lower expert index,
// softmax over the selected logits, and the shared expert gate sigmoid(x . w_sg).
// Kernels 2-4 (over 32-token chunks, plus one scan CTA): per-expert counts, exclusive offsets, a
// permutation sorted by (expert, token) that depends only on the counts (never on atomic arrival
// order), its inverse and the tile block map.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

constexpr uint32_t kBf16TwoPowMinus12 = 0x3980u;   // 2^-12 as bf16 bits

constexpr int kGateBatch = 8;   // 16-byte loads of x (and of w_sg) in flight per lane

template <int NI>
__global__ void __launch_bounds__(256) topk_kernel(RouteArgs a) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= a.T) return;
  // Layer path: one pass over the token row gives the shared-expert gate logit x . w_sg and the
  // token's largest |x|.  The row's first kGateBatch loads per lane go out before the top-k, so
  // their latency overlaps the ranking, and every batch is loaded whole before its arithmetic
  // (the sum runs over the row in the same order either way).
  const bool has_x = a.x != nullptr;
  const bool gate = has_x && a.gs != nullptr && a.w_sg != nullptr;
  const int nch = has_x ? a.d / 8 : 0;
  const uint4* xr = has_x ? reinterpret_cast<const uint4*>(a.x + (size_t)t * a.d) : nullptr;
  const uint4* wr = reinterpret_cast<const uint4*>(a.w_sg);
  uint4 xv[kGateBatch], wv[kGateBatch];
  auto load_batch = [&](int ch0) {
#pragma unroll
    for (int i = 0; i < kGateBatch; ++i) {
      const int ch = ch0 + lane + 32 * i;
      xv[i] = ch < nch ? __ldg(xr + ch) : make_uint4(0u, 0u, 0u, 0u);
      wv[i] = gate && ch < nch ? __ldg(wr + ch) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if (has_x) load_batch(0);

  int my_e;
  float my_w;
  warp_topk_softmax<NI>(a.logits + (size_t)t * a.E, a.E, a.k, &my_e, &my_w);
  if (lane < a.k) {
    a.idx[(size_t)t * a.k + lane] = my_e;
    a.w[(size_t)t * a.k + lane] = my_w;
  }

  // The grouped GEMM takes x as fp16 operands: a token whose largest |x| is nonzero but below
  // 2^-12 sits mostly in fp16's subnormal range and loses precision there, so it sets the range
  // flag (values above the fp16 range set it when x is converted).  With bf16 operands x is used
  // as given and there is no such edge.
  if (has_x) {
    float dot = 0.0f;
    uint32_t xmax = 0;   // largest |x| as bf16 magnitude bits
    for (int ch0 = 0; ch0 < nch; ch0 += 32 * kGateBatch) {
      if (ch0 > 0) load_batch(ch0);
#pragma unroll
      for (int b = 0; b < kGateBatch; ++b) {
        const uint32_t xw[4] = {xv[b].x, xv[b].y, xv[b].z, xv[b].w}, ww[4] = {wv[b].x, wv[b].y, wv[b].z, wv[b].w};
        if (ch0 + lane + 32 * b < nch) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            xmax = max(xmax, max(xw[i] & 0x7FFFu, (xw[i] >> 16) & 0x7FFFu));
            dot = fmaf(bf16_bits_to_f32(xw[i] & 0xFFFFu), bf16_bits_to_f32(ww[i] & 0xFFFFu), dot);
            dot = fmaf(bf16_bits_to_f32(xw[i] >> 16), bf16_bits_to_f32(ww[i] >> 16), dot);
          }
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
    xmax = __reduce_max_sync(0xFFFFFFFFu, xmax);
    if (lane == 0 && gate) a.gs[t] = 1.0f / (1.0f + expf(-dot));
    if (lane == 0 && !a.bf16 && xmax != 0u && xmax < kBf16TwoPowMinus12) raise_flag(a.err, kErrFp16Range);
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

// Routing tables in three kernels over 32-token chunks (one warp each), so the token passes use
// the whole GPU:
//   chunk_hist_kernel   per-chunk expert counts -> chunk[c][e];
//   chunk_scan_kernel   one CTA: per expert, exclusive prefix over chunks (in place), counts,
//                       offsets (exclusive scan over experts) and the block map;
//   chunk_scatter_kernel  slot of assignment (t, j) = offsets[e] + chunk[c][e] + (earlier tokens of
//                       the chunk routed to e), from a per-chunk bit mask per expert.
// Slots inside an expert are in token order; they follow from the counts alone.
// KMAX: upper bound on k held in registers per token (8 or 32).
template <int KMAX>
__global__ void __launch_bounds__(256) chunk_hist_kernel(TablesArgs a) {
  extern __shared__ int hsm[];   // [8 warps][E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int E = a.E, k = a.k, T = a.T;
  const int nc = (T + 31) / 32;
  const int c = blockIdx.x * 8 + warp;
  int* hw = hsm + warp * E;
  for (int i = lane; i < E; i += 32) hw[i] = 0;
  __syncwarp();
  if (c < nc) {
    int ev[KMAX];
    load_token_ids<KMAX>(a.idx, c * 32 + lane, T, k, E, ev, a.err);
    // lanes routing to the same expert in round j add their count once
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        const uint32_t m = __match_any_sync(0xFFFFFFFFu, ev[j]);
        if (ev[j] >= 0 && lane == __ffs(m) - 1) atomicAdd(&hw[ev[j]], __popc(m));
      }
    }
    __syncwarp();
    for (int i = lane; i < E; i += 32) a.chunk[(size_t)c * E + i] = hw[i];
  }
}

constexpr int kMaxPartialTiles = 1088;   // one partial tile per expert (E <= 1024) + the shared expert

__global__ void __launch_bounds__(1024, 1) chunk_scan_kernel(TablesArgs a) {
  __shared__ int warp_tot[32];
  __shared__ int total_s;
  __shared__ int part_s[1024];   // [part][expert] chunk sums
  const int tid = threadIdx.x;
  const int E = a.E, k = a.k, T = a.T;
  const int nc = (T + 31) / 32;
  // tpe threads per expert, each owning a contiguous range of chunks; loads go out 16 at a time
  const int tpe = E <= 256 ? 4 : E <= 512 ? 2 : 1;
  const int e = tid % E, p = tid / E;
  const bool owner = tid < E * tpe;
  const int per = (nc + tpe - 1) / tpe;
  const int c_lo = owner ? min(nc, p * per) : 0, c_hi = owner ? min(nc, (p + 1) * per) : 0;
  // The first kScanKeep counts of a thread's range stay in registers between the two passes
  // (every range up to T = 4096 tokens with E <= 256); the rest are read again.
  constexpr int kScanKeep = 32;
  int keep[kScanKeep];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < kScanKeep; ++i) keep[i] = c_lo + i < c_hi ? __ldcg(a.chunk + (size_t)(c_lo + i) * E + e) : 0;
#pragma unroll
  for (int i = 0; i < kScanKeep; ++i) sum += keep[i];
  for (int c0 = c_lo + kScanKeep; c0 < c_hi; c0 += 16) {
    int v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = c0 + i < c_hi ? __ldcg(a.chunk + (size_t)(c0 + i) * E + e) : 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) sum += v[i];
  }
  if (owner) part_s[p * E + e] = sum;
  __syncthreads();
  int run = 0, cnt = 0;
  if (owner) {
    for (int q = 0; q < p; ++q) run += part_s[q * E + e];
#pragma unroll
    for (int i = 0; i < kScanKeep; ++i)
      if (c_lo + i < c_hi) {
        a.chunk[(size_t)(c_lo + i) * E + e] = run;
        run += keep[i];
      }
    for (int c0 = c_lo + kScanKeep; c0 < c_hi; c0 += 16) {
      int v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = c0 + i < c_hi ? __ldcg(a.chunk + (size_t)(c0 + i) * E + e) : 0;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (c0 + i < c_hi) {
          a.chunk[(size_t)(c0 + i) * E + e] = run;
          run += v[i];
        }
    }
  }
  if (tid < E) {
    for (int q = 0; q < tpe; ++q) cnt += part_s[q * E + tid];
    a.counts[tid] = cnt;
  }
  const int off = block_excl_scan(cnt, warp_tot, &total_s);
  if (tid < E) a.offsets[tid] = off;
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

  // The grouped GEMM's walk order, by the rule of schedule_kernel (full tiles in block-map order,
  // then partial tiles by decreasing width, ties in block-map order), from the counts at hand: an
  // expert's full tiles are its first cnt / tile_n, its partial tile (if any) its last.
  if (a.sched != nullptr) {
    __shared__ int pw[kMaxPartialTiles];
    __shared__ int pidx[kMaxPartialTiles];
    const int nfull = (tid < E) ? cnt / a.tile_n : 0;
    const bool part = (tid < E) && (cnt % a.tile_n) != 0;
    const int fpos = block_excl_scan(nfull, warp_tot, &total_s);
    const int routed_full = total_s;
    const int ppos = block_excl_scan(part ? 1 : 0, warp_tot, &total_s);
    const int routed_part = total_s;
    for (int i = 0; i < nfull; ++i) a.sched[fpos + i] = tile0 + i;
    const int sh_full = a.has_shared ? T / a.tile_n : 0;
    const bool sh_part = a.has_shared && (T % a.tile_n) != 0;
    for (int i = tid; i < sh_full; i += blockDim.x) a.sched[routed_full + i] = routed_tiles + i;
    if (part) {
      pw[ppos] = cnt % a.tile_n;
      pidx[ppos] = tile0 + nfull;
    }
    if (tid == 0 && sh_part) {
      pw[routed_part] = T % a.tile_n;
      pidx[routed_part] = routed_tiles + sh_full;
    }
    __syncthreads();
    const int np = routed_part + (sh_part ? 1 : 0);   // <= E + 1 <= kMaxPartialTiles
    const int base = routed_full + sh_full;
    for (int p = tid; p < np; p += blockDim.x) {
      const int w = pw[p];
      int before = 0;
      for (int q = 0; q < np; ++q) before += (pw[q] > w || (pw[q] == w && q < p)) ? 1 : 0;
      a.sched[base + before] = pidx[p];
    }
  }
}

template <int KMAX>
__global__ void __launch_bounds__(256) chunk_scatter_kernel(TablesArgs a) {
  extern __shared__ uint32_t msm[];   // [8 warps][E] bit masks
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int E = a.E, k = a.k, T = a.T;
  const int nc = (T + 31) / 32;
  const int c = blockIdx.x * 8 + warp;
  if (c >= nc) return;   // whole warps leave; no block barrier below
  uint32_t* mk = msm + warp * E;
  for (int i = lane; i < E; i += 32) mk[i] = 0u;
  __syncwarp();
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
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    if (ev[j] >= 0) {
      const int e = ev[j];
      const int slot = __ldg(a.offsets + e) + a.chunk[(size_t)c * E + e] + __popc(mk[e] & lt);
      a.perm[slot] = t * k + j;
      a.inv[(size_t)t * k + j] = slot;
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

// The library's bounded waits, made to run out: thread 0 waits on an mbarrier that nothing
// completes until `limit` cycles pass, gives up, sets the CTA's abort word and the timeout bit of
// the error word; warp 1 then waits on the same barrier collectively and leaves through the abort
// word at once, all lanes with the same outcome.  Nothing else is touched.
__global__ void __launch_bounds__(64) wait_probe_kernel(uint32_t* err, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_s;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_s = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait_for(smem_u32(&bar), 0, &abort_s, err, limit);
  __syncthreads();
  if (threadIdx.x >= 32) (void)mbar_wait_warp_for(smem_u32(&bar), 0, &abort_s, err, limit);
}

cudaError_t launch_wait_probe(uint32_t* err, long long limit, cudaStream_t st) {
  wait_probe_kernel<<<1, 64, 0, st>>>(err, limit);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(1024, 1) schedule_kernel(ScheduleArgs a) {
  __shared__ int pw[kMaxPartialTiles];
  __shared__ int pidx[kMaxPartialTiles];
  __shared__ int warp_tot[32];
  __shared__ int total_s;
  const int tid = threadIdx.x;
  const int n = *a.num_tiles;
  int full_base = 0, part_base = 0;
  for (int i0 = 0; i0 < n; i0 += 1024) {
    const int i = i0 + tid;
    const int w = i < n ? __ldg(a.tiles + 4 * (size_t)i + 2) : 0;
    const bool part = i < n && w < a.tile_n;
    const bool full = i < n && !part;
    const int fpos = block_excl_scan(full ? 1 : 0, warp_tot, &total_s);
    const int ftot = total_s;
    const int ppos = block_excl_scan(part ? 1 : 0, warp_tot, &total_s);
    const int ptot = total_s;
    if (full) a.sched[full_base + fpos] = i;
    if (part) {
      if (part_base + ppos < kMaxPartialTiles) {
        pw[part_base + ppos] = w;
        pidx[part_base + ppos] = i;
      } else {
        raise_flag(a.err, kErrBadRouting);   // more partial tiles than a block map can hold
      }
    }
    full_base += ftot;
    part_base += ptot;
  }
  __syncthreads();
  const int np = min(part_base, kMaxPartialTiles);
  for (int p = tid; p < np; p += 1024) {
    const int w = pw[p];
    int before = 0;
    for (int q = 0; q < np; ++q) before += (pw[q] > w || (pw[q] == w && q < p)) ? 1 : 0;
    a.sched[full_base + before] = pidx[p];
  }
}

cudaError_t launch_schedule(const ScheduleArgs& a, cudaStream_t st) {
  schedule_kernel<<<1, 1024, 0, st>>>(a);
  return cudaGetLastError();
}

size_t tables_scratch_bytes(int T, int E) { return (size_t)((T + 31) / 32) * E * sizeof(int); }

cudaError_t launch_tables(const TablesArgs& a, cudaStream_t st) {
  if (a.T <= 0) {
    // no tokens: empty tables (counts and offsets zero, no tiles)
    chunk_scan_kernel<<<1, 1024, 0, st>>>(a);
    return cudaGetLastError();
  }
  const int nc = (a.T + 31) / 32;
  const int grid = (nc + 7) / 8;
  const size_t smem = (size_t)8 * a.E * sizeof(int);   // <= 32 KB (E <= 1024)
  if (a.k <= 8) chunk_hist_kernel<8><<<grid, 256, smem, st>>>(a);
  else chunk_hist_kernel<32><<<grid, 256, smem, st>>>(a);
  chunk_scan_kernel<<<1, 1024, 0, st>>>(a);
  if (a.k <= 8) chunk_scatter_kernel<8><<<grid, 256, smem, st>>>(a);
  else chunk_scatter_kernel<32><<<grid, 256, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
