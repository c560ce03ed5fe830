// Grouped-query decode attention over a bf16 key/value cache (declarations and contracts in
// include/gqa_attention.h).
//
// The pages' engine shares one thread group among the query heads of a key/value group so that
// each key and value row is loaded once (GQA packing), and cuts long contexts into fixed blocks
// ("Perplexity libera Lily: inferencia en Rust y Metal para Mac", section "Decode: mover menos
// bytes por token").  On GB300 that becomes:
//   * the context is cut into fixed tiles of 64 positions; a key/value tile (16 KB of keys and
//     16 KB of values) arrives in shared memory by four tensor-map copies in the 128-byte swizzle;
//   * one CTA per SM (about), each a contiguous run of tiles of one key/value head, holding ALL
//     query heads of the group (up to eight), so every cached byte is read from HBM exactly once;
//   * one producer warp issues the copies into a six-stage ring; eight consumer warps take
//     alternate tiles (four warps a tile, 16 positions a warp) and compute on the tensor cores
//     with m16n8k16 bf16 MMAs: S = Q K^T with the group's queries as the 16-row A operand
//     (rows 8..15 zero), then O += P V with P as the A operand straight from S's accumulator
//     registers -- rows 0..7 carry bf16(p) and rows 8..15 the rounding remainder
//     bf16(p - bf16(p)), so P enters the product with about 17 significant bits and the two
//     halves of O are added at the end;
//   * each warp keeps a running softmax (max, sum, O) in registers; the CTA merges its warps in
//     a fixed order and writes one partial (max, sum, unnormalised O) per query head;
//   * a second launch (programmatic dependent launch) merges the partials of each head in a
//     fixed order and divides by the sum.
// The work is bound by HBM: 1 KB of cache per position (two heads, keys and values) against
// 32 KFLOP of tensor-core work.

#include <cmath>
#include <cstring>

#include <cuda_bf16.h>

#include "../../include/gqa_attention.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kD = 128;                        // head size
constexpr int kTileN = 64;                     // positions per tile
constexpr int kStages = 6;                     // tiles held per CTA (landed or in flight)
constexpr int kInFlight = 4;                   // tiles in flight per CTA (swept: 1, 2, 3, 4, 6)
static_assert(kInFlight >= 1 && kInFlight <= kStages, "in-flight window");
constexpr int kConsumerWarps = 8;              // two groups of four, alternate tiles
constexpr int kThreadsAttn = (kConsumerWarps + 1) * 32;
constexpr int kBoxBytes = kTileN * 128;        // 64 positions x 64 dims x 2 bytes
constexpr int kStageBytes = 4 * kBoxBytes;     // keys (2 boxes) + values (2 boxes)
constexpr int kMaxGroup = 8;                   // query heads per key/value head
constexpr int kPartFloats = kMaxGroup * kD + 2 * kMaxGroup;   // O rows, then max, then sum
constexpr int kMaxBlocksPerHead = 256;
constexpr int kOStride = kD + 8;               // padded row of the warp-merge buffer (floats)
constexpr size_t kAttnSmem = (size_t)kStages * kStageBytes + 1024;   // + alignment slack
constexpr float kNegBig = -1e30f;              // running max before any position is seen
static_assert(kConsumerWarps * kMaxGroup * kOStride * 4 <= kStages * kStageBytes, "merge buffer");
static_assert(kStages % 2 == 0, "a stage must always belong to the same consumer group");

struct AttnMaps {
  CUtensorMap k, v;   // bf16 {128, N, Hkv}, box {64, 64, 1}, 128-byte swizzle, rows >= N read as zero
};

struct AttnArgs {
  const uint16_t* q;   // bf16 [Hq, 128]
  float* part;         // [Hkv, nblk, kPartFloats]
  uint32_t* err;
  int G;               // query heads per key/value head
  int n_ctx, ntiles, nblk;
  float qk_scale;      // log2(e) / sqrt(128): scores in base-2 units
};

struct MergeArgs {
  const float* part;
  float* o;            // fp32 [Hq, 128]
  uint32_t* err;
  int G, nblk;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// d (+)= A B for one m16n8k16 tile, bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two fp32 values as a bf16 pair (lo in the low half), rounded to nearest.
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// The remainder p - bf16(p) of a pair, as a bf16 pair.
__device__ __forceinline__ uint32_t bf16x2_rem(float lo, float hi, uint32_t top) {
  const __nv_bfloat162 t = *reinterpret_cast<const __nv_bfloat162*>(&top);
  return bf16x2(lo - __low2float(t), hi - __high2float(t));
}

// Byte offset of 16-byte chunk `chunk` (0..15, 8 dims each) of row `pos` (0..63) in a tile of
// two 64-dim boxes written by the tensor map's 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz(int pos, int chunk) {
  return (uint32_t)((chunk >> 3) * kBoxBytes + pos * 128 + (((chunk & 7) ^ (pos & 7)) << 4));
}

__global__ void __launch_bounds__(kThreadsAttn, 1)
    attn_block_kernel(const __grid_constant__ AttnMaps maps, const AttnArgs a) {
  extern __shared__ uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ float m_s[kConsumerWarps][kMaxGroup], l_s[kConsumerWarps][kMaxGroup];
  __shared__ int abort_s;
  const uint32_t raw = smem_u32(sm_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;   // swizzled boxes start on 1024-byte boundaries
  float* merge_s = reinterpret_cast<float*>(sm_raw + (base - raw));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int blk = blockIdx.x, g = blockIdx.y;
  const int t0 = (int)((long long)blk * a.ntiles / a.nblk);
  const int nt = (int)((long long)(blk + 1) * a.ntiles / a.nblk) - t0;   // >= 1 (nblk <= ntiles)

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 4);
    }
    abort_s = 0;
    mbar_fence_init();
  }
  __syncthreads();

  // ---- producer: one lane issues the tile copies into the ring
  const bool producer = (warp == kConsumerWarps && lane == 0);
  int issued = 0;
  auto issue = [&](int i) {
    const uint32_t st = base + (i % kStages) * kStageBytes, bar = smem_u32(&full[i % kStages]);
    const int row = (t0 + i) * kTileN;
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_3d(st, &maps.k, bar, 0, row, g);
    tma_load_3d(st + kBoxBytes, &maps.k, bar, 64, row, g);
    tma_load_3d(st + 2 * kBoxBytes, &maps.v, bar, 0, row, g);
    tma_load_3d(st + 3 * kBoxBytes, &maps.v, bar, 64, row, g);
  };
  // At most kInFlight copies are outstanding: tile i is issued once tile i - kInFlight has landed.
  auto landed = [&](int j) {
    return j < 0 || kInFlight >= kStages ||
           mbar_wait(smem_u32(&full[j % kStages]), (j / kStages) & 1, &abort_s, a.err);
  };
  if (producer) {
    // Cached positions below the last tile are final before this call is enqueued, so their copies
    // start before the preceding kernel in the stream has finished; only q and the tile holding
    // position N-1 (the new token's key and value) may still be in flight from it.
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.v);
    int early = a.ntiles - 1 - t0;
    if (early > nt) early = nt;
    if (early > kStages) early = kStages;
    for (; issued < early; ++issued) {
      if (!landed(issued - kInFlight)) break;
      issue(issued);
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  if (producer) {
    for (; issued < nt; ++issued) {
      const int i = issued;
      if (i >= kStages && !mbar_wait(smem_u32(&empty[i % kStages]), ((i / kStages) - 1) & 1, &abort_s, a.err)) break;
      if (!landed(i - kInFlight)) break;
      issue(i);
    }
    // After a timeout, copies still in flight land before the shared memory is reused or the CTA
    // exits.
    if (abort_s) {
      for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i) {
        const long long c0 = clock64();
        while (!mbar_try_wait(smem_u32(&full[i % kStages]), (i / kStages) & 1) && clock64() - c0 < 4000000ll) {
        }
      }
    }
  }

  float o[16][4];   // O for n-tile j (dims 8j..8j+7): rows r (bf16(p) part) and r + 8 (remainder part)
  float m_run = kNegBig, l_run = 0.f;
  const int r = lane >> 2, c2 = (lane & 3) * 2;
  if (warp < kConsumerWarps) {
    // ---- consumers
    const int wg = warp >> 2, wq = warp & 3;
    uint32_t qa[8][2];   // A fragments of the group's queries, rows r < G (rows 8..15 are zero)
    {
      const bool live = r < a.G;
      const uint32_t* qh = reinterpret_cast<const uint32_t*>(a.q + (size_t)(g * a.G + (live ? r : 0)) * kD + c2);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa[kk][0] = live ? __ldg(qh + 8 * kk) : 0u;
        qa[kk][1] = live ? __ldg(qh + 8 * kk + 4) : 0u;
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    const int lrow = lane & 7, lmat = lane >> 3;
    const int kpos = wq * 16 + 8 * (lmat >> 1) + lrow;   // key row this lane addresses
    const int vpos = wq * 16 + 8 * (lmat & 1) + lrow;    // value row this lane addresses
    for (int i = wg; i < nt; i += 2) {
      const int s = i % kStages;
      if (!mbar_wait_warp(smem_u32(&full[s]), (i / kStages) & 1, &abort_s, a.err)) break;
      const uint32_t st = base + s * kStageBytes;
      // S = Q K^T over this warp's 16 positions: two n-tiles of 8 positions, 8 k-steps of 16 dims.
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(st + swz(kpos, 2 * kk + (lmat & 1)), b0, b1, b2, b3);
        mma_bf16(sc[0], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
        mma_bf16(sc[1], qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
      }
      // Running softmax in base 2 for query row r; positions at or past N do not exist.
      const int p0 = (t0 + i) * kTileN + wq * 16 + c2;
      float s2[2][2];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float v = (p0 + 8 * j + e < a.n_ctx) ? sc[j][e] * a.qk_scale : -INFINITY;
          s2[j][e] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = exp2f(m_run - m_new);
      m_run = m_new;
      float p[2][2];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) p[j][e] = exp2f(s2[j][e] - m_new);
      l_run = l_run * alpha + ((p[0][0] + p[0][1]) + (p[1][0] + p[1][1]));
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= alpha;
        o[j][1] *= alpha;
        o[j][2] *= alpha;
        o[j][3] *= alpha;
      }
      // P as the A operand: k = position within the warp's 16, rows 0..7 bf16(p), rows 8..15 the
      // remainder.
      const uint32_t a0 = bf16x2(p[0][0], p[0][1]);
      const uint32_t a2 = bf16x2(p[1][0], p[1][1]);
      const uint32_t a1 = bf16x2_rem(p[0][0], p[0][1], a0);
      const uint32_t a3 = bf16x2_rem(p[1][0], p[1][1], a2);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(st + 2 * kBoxBytes + swz(vpos, 2 * jj + (lmat >> 1)), b0, b1, b2, b3);
        mma_bf16(o[2 * jj], a0, a1, a2, a3, b0, b1);
        mma_bf16(o[2 * jj + 1], a0, a1, a2, a3, b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 1);
    l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 2);
    if ((lane & 3) == 0) {
      m_s[warp][r] = m_run;
      l_s[warp][r] = l_run;
    }
  }
  __syncthreads();   // every tile consumed and every copy landed: the ring is free
  __shared__ float wt_s[kConsumerWarps][kMaxGroup], mrow_s[kMaxGroup];
  if (warp < kConsumerWarps) {
    float* ow = merge_s + (warp * kMaxGroup + r) * kOStride + c2;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      *reinterpret_cast<float2*>(ow + 8 * j) = make_float2(o[j][0] + o[j][2], o[j][1] + o[j][3]);
  }
  if (tid < kConsumerWarps * kMaxGroup) {   // weight of warp w in row r, relative to the CTA's max
    const int rr = tid & (kMaxGroup - 1), w = tid / kMaxGroup;
    float M = m_s[0][rr];
#pragma unroll
    for (int v = 1; v < kConsumerWarps; ++v) M = fmaxf(M, m_s[v][rr]);
    wt_s[w][rr] = exp2f(m_s[w][rr] - M);
    if (w == 0) mrow_s[rr] = M;
  }
  __syncthreads();
  // ---- merge the eight warps (fixed order) and write this block's partial for each live row:
  // four consecutive dims per thread
  float* out = a.part + ((size_t)g * a.nblk + blk) * kPartFloats;
  for (int e4 = tid; e4 < a.G * (kD / 4); e4 += kThreadsAttn) {
    const int row = e4 / (kD / 4), dim = (e4 % (kD / 4)) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float4 v = *reinterpret_cast<const float4*>(merge_s + (w * kMaxGroup + row) * kOStride + dim);
      const float sw = wt_s[w][row];
      acc.x += v.x * sw;
      acc.y += v.y * sw;
      acc.z += v.z * sw;
      acc.w += v.w * sw;
    }
    *reinterpret_cast<float4*>(out + row * kD + dim) = acc;
  }
  if (tid < a.G) {
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) L += l_s[w][tid] * wt_s[w][tid];
    out[kMaxGroup * kD + tid] = mrow_s[tid];
    out[kMaxGroup * kD + kMaxGroup + tid] = L;
  }
}

// Merge of the blocks of one query head (one CTA per head, 16 warps).  Warp w takes blocks
// w, w + 16, ... with every load of a batch of eight in flight before any is used (one round trip
// to L2 for up to 128 blocks), and keeps a running max, sum and weighted O in block order; the 16
// warps are then combined in order.
constexpr int kMergeWarps = 16;
constexpr int kMergeBatch = 8;

__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(const MergeArgs a) {
  __shared__ float mw_s[kMergeWarps], lw_s[kMergeWarps];
  __shared__ __align__(16) float red[kMergeWarps][kD];
  pdl_wait();
  pdl_launch_dependents();
  const int h = blockIdx.x, g = h / a.G, row = h % a.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* pg = a.part + (size_t)g * a.nblk * kPartFloats;
  float m_t = kNegBig, l_t = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int b0 = warp; b0 < a.nblk; b0 += kMergeWarps * kMergeBatch) {
    float mb[kMergeBatch], lb[kMergeBatch];
    float4 ob[kMergeBatch];
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      const int b = b0 + i * kMergeWarps;
      if (b < a.nblk) {
        const float* pb = pg + (size_t)b * kPartFloats;
        ob[i] = __ldcg(reinterpret_cast<const float4*>(pb + row * kD) + lane);
        mb[i] = __ldcg(pb + kMaxGroup * kD + row);
        lb[i] = __ldcg(pb + kMaxGroup * kD + kMaxGroup + row);
      } else {
        ob[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        mb[i] = kNegBig;
        lb[i] = 0.f;
      }
    }
    float mx = m_t;
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) mx = fmaxf(mx, mb[i]);
    const float sc = exp2f(m_t - mx);
    l_t *= sc;
    acc.x *= sc;
    acc.y *= sc;
    acc.z *= sc;
    acc.w *= sc;
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      const float wb = exp2f(mb[i] - mx);
      l_t += lb[i] * wb;
      acc.x += ob[i].x * wb;
      acc.y += ob[i].y * wb;
      acc.z += ob[i].z * wb;
      acc.w += ob[i].w * wb;
    }
    m_t = mx;
  }
  if (lane == 0) {
    mw_s[warp] = m_t;
    lw_s[warp] = l_t;
  }
  __syncthreads();
  float M = mw_s[0];
#pragma unroll
  for (int w = 1; w < kMergeWarps; ++w) M = fmaxf(M, mw_s[w]);
  const float sw = exp2f(m_t - M);
  *reinterpret_cast<float4*>(&red[warp][4 * lane]) = make_float4(acc.x * sw, acc.y * sw, acc.z * sw, acc.w * sw);
  __syncthreads();
  if (tid < kD) {
    float s = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      s += red[w][tid];
      L += lw_s[w] * exp2f(mw_s[w] - M);
    }
    const float v = s / L;
    a.o[(size_t)h * kD + tid] = v;
    if (!isfinite(v)) raise_flag(a.err, kErrNonFinite);
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_attn_dims(const gqa_dims* d) {
  if (d == nullptr) return MOE_ERR_INVALID_ARG;
  if (d->n_heads < 1 || d->n_kv_heads < 1 || d->n_heads % d->n_kv_heads != 0) return MOE_ERR_INVALID_ARG;
  if (d->n_ctx < 1 || d->capacity < d->n_ctx) return MOE_ERR_INVALID_ARG;
  if (d->head_dim != kD || d->n_heads / d->n_kv_heads > kMaxGroup || d->n_kv_heads > 65535)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int blocks_bound(const gqa_dims* d) {
  const int ntiles = (d->n_ctx + kTileN - 1) / kTileN;
  return ntiles < kMaxBlocksPerHead ? ntiles : kMaxBlocksPerHead;
}

bool encode_cache(CUtensorMap* m, const uint16_t* cache, const gqa_dims* d) {
  EncodeTiledFn f = encode_fn();
  if (f == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)d->n_ctx, (cuuint64_t)d->n_kv_heads};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)d->capacity * kD * 2};
  const cuuint32_t box[3] = {64, kTileN, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(cache), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t gqa_decode_workspace_bytes(const gqa_dims* dims) {
  if (check_attn_dims(dims) != MOE_OK) return 0;
  return (size_t)kWsHeadBytes + (size_t)dims->n_kv_heads * blocks_bound(dims) * kPartFloats * sizeof(float);
}

extern "C" moe_status gqa_decode_attention(const gqa_dims* dims, const uint16_t* q, const uint16_t* k_cache,
                                           const uint16_t* v_cache, float* o, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  const int st = check_attn_dims(dims);
  if (st != MOE_OK) return (moe_status)st;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || o == nullptr || workspace == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(workspace))
    return MOE_ERR_MISALIGNED;
  if (workspace_bytes < gqa_decode_workspace_bytes(dims)) return MOE_ERR_WORKSPACE;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int Hkv = dims->n_kv_heads;
  const int ntiles = (dims->n_ctx + kTileN - 1) / kTileN;
  int nblk = sms / Hkv;
  if (nblk < 1) nblk = 1;
  if (nblk > blocks_bound(dims)) nblk = blocks_bound(dims);

  AttnMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (!encode_cache(&maps.k, k_cache, dims) || !encode_cache(&maps.v, v_cache, dims)) return MOE_ERR_CUDA;

  static bool attr_done = false;   // idempotent: racing first calls set the same value
  if (!attr_done) {
    if (cudaFuncSetAttribute(attn_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttnSmem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    attr_done = true;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  AttnArgs a;
  a.q = q;
  a.part = reinterpret_cast<float*>(ws + kWsHeadBytes);
  a.err = reinterpret_cast<uint32_t*>(ws);
  a.G = dims->n_heads / Hkv;
  a.n_ctx = dims->n_ctx;
  a.ntiles = ntiles;
  a.nblk = nblk;
  a.qk_scale = (float)(1.4426950408889634 / std::sqrt((double)kD));

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nblk, Hkv);
  cfg.blockDim = dim3(kThreadsAttn);
  cfg.dynamicSmemBytes = kAttnSmem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, attn_block_kernel, maps, a) != cudaSuccess) return MOE_ERR_CUDA;

  MergeArgs m;
  m.part = a.part;
  m.o = o;
  m.err = a.err;
  m.G = a.G;
  m.nblk = nblk;
  cfg.gridDim = dim3(dims->n_heads);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  if (cudaLaunchKernelEx(&cfg, attn_merge_kernel, m) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
