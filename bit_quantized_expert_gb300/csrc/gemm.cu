// Fused-dequant grouped GEMM of the MoE experts on sm_103a tensor cores (tcgen05 + TMEM).
//
// The pages describe the prefill expert GEMM as rebuilding the 4-bit weights one tile at a
// time in on-chip memory and accumulating in FP32, so the expanded weights never reach DRAM,
// and report the expert GEMMs as about 90% of prefill time ("Perplexity libera Lily:
// inferencia en Rust y Metal para Mac", section "Prefill: pesos comprimidos y enrutamiento en
// la GPU").  This kernel is that design re-thought for GB300:
//
//   * Swap-AB: the weight rows of one expert form the MMA's M = 128 side, the (few, uneven)
//     tokens routed to the expert form N (16..112, rounded up to 16).  D[m, n] = sum_k W[m, k]
//     X[n, k] lands in TMEM (fp32), lane m, column n.
//   * Work unit = (block-map tile of <= 112 slots of one expert, two 128-row weight tiles),
//     iterated over K in operand stages of two 64-wide chunks (a chunk = one quantisation group):
//     every hand-off between roles happens once per 16 MMAs.  A persistent grid of one CTA per SM
//     walks the units; every role walks the same list.
//   * Warp roles (16 warps): 0 = TMA producer of the activation tiles (x rows in slot order, or
//     h), 1 = MMA issuer (one thread) and TMEM owner, 2 = TMA producer of the packed codes,
//     3 = idle, 4-11 = dequant
//     (one thread per weight row of one of the unit's two tiles: 4-bit codes -> fp16
//     w = q*scale + bias, single rounding; two dequant warps per scheduler so one hides the
//     other's shared-memory and barrier latency),
//     12-15 = epilogue (TMEM -> registers; SwiGLU -> fp16 h, or fp32 expert outputs).
//   * Gate/up mode keeps the gate and up accumulators of the same 128 F-rows side by side in
//     TMEM so the epilogue applies silu(g) * u in registers.  Two accumulator buffers let the
//     epilogue of one unit overlap the MMAs of the next.
//   * Operands are fp16 (the dequantised weights, x and h), accumulation fp32.  Within every
//     8-element K chunk both operands are stored in the order (0,4,1,5,2,6,3,7), which lets the
//     dequant turn one 32-bit code word into four fp16 pairs with one LOP3 each.  An instantiation
//     with bf16 operands (BF) serves callers that ask for them: the same roles and layout, bf16
//     weights w = q*s + b (one rounding), x as given, bf16 h, and bf16 expert outputs.
//   * Every wait is bounded (mbar_wait); on timeout the CTA sets the error word and winds down.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kThreads = 512;
constexpr uint32_t kTileBytes = 128 * 128;   // one 128-row x 64-column fp16 weight tile
constexpr uint32_t kXBytes = kGemmMaxTileN * 128;   // one activation tile: <= 112 rows x 64 columns
constexpr uint32_t kRawBytes = 128 * 64;     // 128 rows x 128 packed 4-bit codes: two K chunks

template <int MODE>
struct Cfg {
  // Two weight tiles per unit: gate and up rows f .. f+127 (gate/up mode), or the down rows of two
  // adjacent 128-row blocks (down mode); both share the unit's activation tile.
  static constexpr int NMAT = 2;
  static constexpr int S_RAW = 2;   // packed-code stages of two K chunks each
  // Operand stages of two K chunks: the W tiles (NMAT x 2 chunks, dequantised) and the X tiles
  // (2 chunks) together, so the MMA thread waits and commits once per 16 MMAs.
  static constexpr int S_W = 2;
  static constexpr int S_X = S_W;
  static constexpr uint32_t W_STAGE = NMAT * 2 * kTileBytes;   // 64 KB
  static constexpr uint32_t X_STAGE = 2 * kXBytes;             // 28 KB
  static constexpr int NBAR = 2 * S_RAW + 2 * S_W + 4;
  static constexpr uint32_t OFF_W = 0;
  static constexpr uint32_t OFF_X = OFF_W + S_W * W_STAGE;
  static constexpr uint32_t OFF_RAW = OFF_X + S_X * X_STAGE;
  static constexpr uint32_t OFF_BAR = OFF_RAW + S_RAW * NMAT * kRawBytes;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t OFF_STG = (OFF_MISC + 16 + 15) & ~15u;   // epilogue staging, 2 KB per warp
  static constexpr uint32_t BYTES = OFF_STG + 4 * 2048 + 1024;        // + alignment slack
  static constexpr uint32_t ACC_COLS = NMAT * 128;          // TMEM columns of one accumulator buffer
  static_assert(BYTES <= 227u * 1024u, "shared memory of one CTA");
  static_assert(kXBytes % 1024 == 0 && X_STAGE % 1024 == 0 && OFF_X % 1024 == 0, "128-byte swizzle atoms");
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Eight bf16 scale (or bias) values of groups g0 .. g0+7 of one weight row.
__device__ __forceinline__ uint4 load_group_block(const uint16_t* row, int g0, int G) {
  if ((G & 7) == 0) return ldg_nc_v4(row + g0);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (g0 + j < G) w[j >> 1] |= (uint32_t)__ldg(row + g0 + j) << (16 * (j & 1));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int J>
__device__ __forceinline__ uint32_t pick_bf16(const uint4& v) {
  const uint32_t w = (J >> 1) == 0 ? v.x : (J >> 1) == 1 ? v.y : (J >> 1) == 2 ? v.z : v.w;
  return (J & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// One packed word (8 codes, logical columns 0..7) -> four fp16x2 words holding
// (w0,w4), (w1,w5), (w2,w6), (w3,w7) with w = q * s + b rounded once to fp16.  A code pair is put
// into the mantissa of 1024.0 (bits 0-3: 1024 + q exactly) or one nibble higher (bits 4-7:
// 1024 + 16 q) and brought back to q exactly, by subtracting 1024 or by (1024 + 16 q) / 16 - 64,
// so only one shift per word is needed.
__device__ __forceinline__ void dequant_word(uint32_t q, __half2 s2, __half2 b2, uint32_t (&o)[4]) {
  const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));    // 1024
  const __half2 k16th = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));    // 1/16
  const __half2 km64 = __halves2half2(__ushort_as_half(0xD400), __ushort_as_half(0xD400));     // -64
  const uint32_t r = q >> 8;
  const uint32_t t[4] = {(q & 0x000F000Fu) | 0x64006400u, (q & 0x00F000F0u) | 0x64006400u,
                         (r & 0x000F000Fu) | 0x64006400u, (r & 0x00F000F0u) | 0x64006400u};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const __half2 h = *reinterpret_cast<const __half2*>(&t[p]);
    __half2 v = (p & 1) ? __hfma2(h, k16th, km64) : __hsub2(h, k1024);   // exact codes
    v = __hfma2(v, s2, b2);
    o[p] = *reinterpret_cast<uint32_t*>(&v);
  }
}

// The same for bf16 operands.  bf16 keeps 7 mantissa bits, so each code is shifted into bits 0-3 of
// 128.0's mantissa (128 + q exactly) on its own and brought back by subtracting 128; then one bf16
// fma gives w = q * s + b with a single rounding.
__device__ __forceinline__ void dequant_word_bf16(uint32_t q, __nv_bfloat162 s2, __nv_bfloat162 b2, uint32_t (&o)[4]) {
  const __nv_bfloat162 k128 = __halves2bfloat162(__ushort_as_bfloat16(0x4300), __ushort_as_bfloat16(0x4300));
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t t = ((q >> (4 * p)) & 0x000F000Fu) | 0x43004300u;   // codes p and p + 4
    __nv_bfloat162 v = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&t), k128);   // exact codes
    v = __hfma2(v, s2, b2);
    o[p] = *reinterpret_cast<uint32_t*>(&v);
  }
}

__device__ __forceinline__ uint16_t f32_to_16(float v, bool bf) {
  return bf ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
}
// Two values rounded to fp16 or bf16 by one packed conversion: a in the low half, b in the high.
__device__ __forceinline__ uint32_t f32x2_to_16x2(float a, float b, bool bf) {
  if (bf) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int MODE, bool BF>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
  using C = Cfg<MODE>;
  constexpr int NMAT = C::NMAT;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t s_raw0 = smem_u32(smem_raw);
  const uint32_t sbase = (s_raw0 + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - s_raw0);
  const uint32_t sW = sbase + C::OFF_W, sX = sbase + C::OFF_X, sRaw = sbase + C::OFF_RAW;
  const uint32_t sBar = sbase + C::OFF_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile int* abort_s = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 4);

  auto RF = [&](int i) { return sBar + 8u * i; };
  auto RE = [&](int i) { return sBar + 8u * (C::S_RAW + i); };
  // Operand stage s holds the dequantised W tile(s) and the activation tile X of one K chunk:
  // WF(s) completes when the 8 dequant warps have arrived and the X bytes have landed; WE(s) when
  // the MMAs reading the stage have completed.
  auto WF = [&](int i) { return sBar + 8u * (2 * C::S_RAW + i); };
  auto WE = [&](int i) { return sBar + 8u * (2 * C::S_RAW + C::S_W + i); };
  auto AF = [&](int i) { return sBar + 8u * (2 * C::S_RAW + 2 * C::S_W + i); };
  auto AE = [&](int i) { return sBar + 8u * (2 * C::S_RAW + 2 * C::S_W + 2 + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::S_RAW; ++i) {
      mbar_init(RF(i), 1);
      mbar_init(RE(i), 8);
    }
    for (int i = 0; i < C::S_W; ++i) {
      mbar_init(WF(i), 8 + 1);   // dequant warps + the producer's expect_tx arrival
      mbar_init(WE(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(AF(i), 1);
      mbar_init(AE(i), 4);
    }
    *abort_s = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.codes[0][0]);
    prefetch_tmap(&maps.codes[0][1]);
    if (NMAT == 2) {
      prefetch_tmap(&maps.codes[1][0]);
      prefetch_tmap(&maps.codes[1][1]);
    }
    if (MODE == 1) {
      prefetch_tmap(&maps.h);
      prefetch_tmap(&maps.h16);
    }
    if (MODE == 0) {
      prefetch_tmap(&maps.x);
      prefetch_tmap(&maps.x16);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int R = MODE == 0 ? a.F : a.d;   // weight rows (output features of this projection)
  const int K = MODE == 0 ? a.d : a.F;   // reduction length
  const int MT = R / (MODE == 0 ? kBM : 2 * kBM);   // units per block-map tile
  const int KC = K / 64;
  const int num_units = (*a.num_tiles) * MT;
  const int4* tiles = reinterpret_cast<const int4*>(a.tiles);
  // Every role walks units blockIdx.x, +gridDim.x, ... of the scheduled tile order (wide tiles
  // first, so the round-robin split is balanced).  A unit's tile is a dependent pair of loads
  // (schedule entry, then block-map row): the walk reads the entry two units ahead and the row one
  // unit ahead, so no role stalls on the pair at a unit boundary.
  const int grid_u = (int)gridDim.x;
  auto sched_at = [&](int u) { return u < num_units ? __ldg(a.sched + u / MT) : 0; };
  auto tile_at = [&](int u, int si) { return u < num_units ? __ldg(tiles + si) : make_int4(0, 0, 0, 0); };
  struct Walk {
    int4 next;   // tile of the next unit
    int s2;      // schedule entry of the unit after it
  };
  auto walk_init = [&](Walk& w) {
    w.next = tile_at((int)blockIdx.x, sched_at((int)blockIdx.x));
    w.s2 = sched_at((int)blockIdx.x + grid_u);
  };
  auto walk_step = [&](Walk& w, int u) {   // returns the tile of unit u
    const int4 cur = w.next;
    w.next = tile_at(u + grid_u, w.s2);
    w.s2 = sched_at(u + 2 * grid_u);
    return cur;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer: activation tiles
    // (x rows in slot order, or h; per K chunk the tile's rows rounded up to 16 -- the MMA's N --
    // by 64 columns: one 112-row box for a full tile, else 16-row boxes, so narrow tiles do not
    // pull unused rows through L2 and shared memory; rows past the tile's end belong to the next
    // tile or lie outside the tensor (zero-filled), and the MMA columns they feed are never
    // stored).  The packed codes have their own producer (warp 2), so their loads run up to
    // S_RAW stages ahead of the dequant instead of waiting behind the operand ring, which only
    // advances as fast as the MMAs retire.
    if (lane == 0) {
      int sx = 0;
      uint32_t phx = 0;
      Walk wk;
      walk_init(wk);
      for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        const int4 tl = walk_step(wk, u);
        const int n16 = (tl.z + 15) >> 4;   // 16-row groups of the tile (1..7)
        bool ok = true;
        for (int kc = 0; kc < KC; kc += 2) {   // K chunks kc and kc+1 (K is a multiple of 128)
          if (!mbar_wait(WE(sx), phx ^ 1u, abort_s, a.err)) { ok = false; break; }
          mbar_arrive_expect_tx(WF(sx), 2u * (uint32_t)n16 * 16u * 128u);
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            const uint32_t dst = sX + sx * C::X_STAGE + (uint32_t)hc * kXBytes;
            if (n16 * 16 == kGemmMaxTileN) {
              tma_load_2d(dst, MODE == 0 ? &maps.x : &maps.h, WF(sx), (kc + hc) * 64, tl.y);
            } else {
              for (int r = 0; r < n16; ++r)
                tma_load_2d(dst + (uint32_t)r * 2048u, MODE == 0 ? &maps.x16 : &maps.h16, WF(sx), (kc + hc) * 64,
                            tl.y + 16 * r);
            }
          }
          if (++sx == C::S_X) { sx = 0; phx ^= 1u; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ TMA producer: packed codes of
    // chunks kc and kc+1 (K is a multiple of 128) of the unit's weight tiles
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      Walk wk;
      walk_init(wk);
      for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        const int4 tl = walk_step(wk, u);
        const int m = u % MT;
        const int which = tl.x == a.E ? 1 : 0;
        const int ec = which ? 0 : tl.x;
        bool ok = true;
        for (int kc = 0; kc < KC; kc += 2) {
          if (!mbar_wait(RE(s), ph ^ 1u, abort_s, a.err)) { ok = false; break; }
          mbar_arrive_expect_tx(RF(s), NMAT * kRawBytes);
#pragma unroll
          for (int mat = 0; mat < NMAT; ++mat)
            tma_load_3d(sRaw + (s * NMAT + mat) * kRawBytes, &maps.codes[MODE == 0 ? mat : 0][which], RF(s), kc * 8,
                        (MODE == 0 ? m : 2 * m + mat) * kBM, ec);
          if (++s == C::S_RAW) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int sw = 0;
      uint32_t phw = 0;
      int li = 0;
      Walk wk;
      walk_init(wk);
      for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++li) {
        const int4 tl = walk_step(wk, u);
        const uint32_t n_inst = (uint32_t)((tl.z + 15) & ~15);
        const int b = li & 1;
        if (!mbar_wait(AE(b), ((li >> 1) & 1) ^ 1u, abort_s, a.err)) break;
        tc_fence_after();
        // A and B formats: fp16 (0) or bf16 (1) in bits 7-9 and 10-12
        const uint32_t idesc = idesc_f16_f32(kBM, n_inst) | (BF ? ((1u << 7) | (1u << 10)) : 0u);
        const uint32_t d0 = tmem + (uint32_t)(b * C::ACC_COLS);
        bool ok = true;
        for (int kc = 0; kc < KC; kc += 2) {
          if (!mbar_wait(WF(sw), phw, abort_s, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Descriptors of the stage's tiles; each 16-element K step advances the start address
          // by 32 bytes (2 in the descriptor's address field, which cannot carry: stages lie
          // below 256 KB).
          static_assert(NMAT == 2, "two weight tiles per unit");
#pragma unroll
          for (int hc = 0; hc < 2; ++hc)
            tc_mma_f16_chunk2(d0, d0 + 128u, smem_desc_sw128(sW + sw * C::W_STAGE + (0 * 2 + hc) * kTileBytes),
                              smem_desc_sw128(sW + sw * C::W_STAGE + (1 * 2 + hc) * kTileBytes),
                              smem_desc_sw128(sX + sw * C::X_STAGE + (uint32_t)hc * kXBytes), idesc,
                              (kc + hc) != 0 ? 1u : 0u);
          tc_commit(WE(sw));
          if (++sw == C::S_W) { sw = 0; phw ^= 1u; }
        }
        if (!ok) break;
        tc_commit(AF(b));
      }
    }
  } else if (warp == 3) {
    // idle (keeps the dequant warps at 4..11 and the epilogue warps at 12..15)
  } else if (warp < 12) {
    // ------------------------------------------------------------ dequant: 8 warps; thread i
    // handles row i % 128 of weight tile i / 128 of every chunk: the gate (0) or up (1) matrix in
    // gate/up mode, the first or second 128-row block of the unit in down mode.
    const int i = (threadIdx.x - 128) & 127;
    const int mat = (threadIdx.x - 128) >> 7;
    constexpr int NW = 8;   // code words per thread per chunk
    const int w0 = 0;
    const uint32_t swz = (uint32_t)(i & 7);
    int s = 0, sw = 0;
    uint32_t ph = 0, phw = 0;
    bool ok = true;
    bool bad = false;
    float wmax = 0.0f;   // upper bound 15 |s| + |b| of this thread's |w| over the unit's row
    const int G = K / 64;
    // Scale and bias rows of this thread's weight row in a unit; the first 8-group block of the
    // next unit is loaded during the last block of the current one.
    auto rows_of = [&](const int4& t, int u, const uint16_t*& sr, const uint16_t*& br) {
      const int which = t.x == a.E ? 1 : 0;
      const int blk = MODE == 0 ? (u % MT) : 2 * (u % MT) + mat;   // 128-row block of the matrix
      const size_t row = (size_t)(which ? 0 : t.x) * R + (size_t)blk * kBM + i;
      const QPtr& qm = a.mat[MODE == 0 ? mat : 0][which];
      sr = qm.scales + row * G;
      br = qm.biases + row * G;
    };
    const uint16_t* srow = nullptr;
    const uint16_t* brow = nullptr;
    uint4 ns = make_uint4(0u, 0u, 0u, 0u), nb = make_uint4(0u, 0u, 0u, 0u);
    Walk wk;
    walk_init(wk);
    if (blockIdx.x < num_units) {
      rows_of(wk.next, blockIdx.x, srow, brow);
      ns = load_group_block(srow, 0, G);
      nb = load_group_block(brow, 0, G);
    }
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      walk_step(wk, u);   // wk.next: the tile of the next unit, needed at this unit's last block
      const uint16_t* srow_n = nullptr;
      const uint16_t* brow_n = nullptr;
      const bool has_next = u + (int)gridDim.x < num_units;
      for (int kb = 0; kb < KC && ok; kb += 8) {
        const uint4 cs = ns, cb = nb;
        if (kb + 8 < KC) {
          ns = load_group_block(srow, kb + 8, G);
          nb = load_group_block(brow, kb + 8, G);
        } else if (has_next) {
          rows_of(wk.next, u + (int)gridDim.x, srow_n, brow_n);
          ns = load_group_block(srow_n, 0, G);
          nb = load_group_block(brow_n, 0, G);
        }
#pragma unroll
        for (int j = 0; j < 8; j += 2) {   // K chunks kb+j and kb+j+1: one operand stage
          if (kb + j >= KC) break;
          const float sf0 = bf16_bits_to_f32(j == 0 ? pick_bf16<0>(cs) : j == 2 ? pick_bf16<2>(cs)
                                             : j == 4 ? pick_bf16<4>(cs) : pick_bf16<6>(cs));
          const float sf1 = bf16_bits_to_f32(j == 0 ? pick_bf16<1>(cs) : j == 2 ? pick_bf16<3>(cs)
                                             : j == 4 ? pick_bf16<5>(cs) : pick_bf16<7>(cs));
          const float bf0 = bf16_bits_to_f32(j == 0 ? pick_bf16<0>(cb) : j == 2 ? pick_bf16<2>(cb)
                                             : j == 4 ? pick_bf16<4>(cb) : pick_bf16<6>(cb));
          const float bf1 = bf16_bits_to_f32(j == 0 ? pick_bf16<1>(cb) : j == 2 ? pick_bf16<3>(cb)
                                             : j == 4 ? pick_bf16<5>(cb) : pick_bf16<7>(cb));
          const float wm0 = fmaf(15.0f, fabsf(sf0), fabsf(bf0)), wm1 = fmaf(15.0f, fabsf(sf1), fabsf(bf1));
          if (!BF) {
            bad = bad || !(wm0 <= 65504.0f) || !(wm1 <= 65504.0f);
            wmax = fmaxf(wmax, fmaxf(wm0, wm1));
          }
          const __half2 s2[2] = {__float2half2_rn(sf0), __float2half2_rn(sf1)};
          const __half2 b2[2] = {__float2half2_rn(bf0), __float2half2_rn(bf1)};
          const __nv_bfloat162 sb2[2] = {__float2bfloat162_rn(sf0), __float2bfloat162_rn(sf1)};   // exact: bf16 given
          const __nv_bfloat162 bb2[2] = {__float2bfloat162_rn(bf0), __float2bfloat162_rn(bf1)};
          // codes of both chunks: the two-chunk stage s.  It holds 64-byte rows in the 64-byte
          // swizzle: 16-byte piece c of row i sits at piece c ^ ((i >> 1) & 3), which keeps the
          // lanes' loads free of bank conflicts; chunk hc is pieces 2 hc and 2 hc + 1.
          if (!mbar_wait(RF(s), ph, abort_s, a.err)) { ok = false; break; }
          const uint32_t row_base = sRaw + (s * NMAT + mat) * kRawBytes + i * 64;
          const uint32_t sx64 = (uint32_t)((i >> 1) & 3);
          uint32_t words[16];
#pragma unroll
          for (int pc = 0; pc < 4; ++pc) {
            const uint4 c4 = ld_shared_v4(row_base + ((((uint32_t)pc) ^ sx64) << 4));
            words[4 * pc] = c4.x; words[4 * pc + 1] = c4.y; words[4 * pc + 2] = c4.z; words[4 * pc + 3] = c4.w;
          }
          const int s_used = s;
          if (++s == C::S_RAW) { s = 0; ph ^= 1u; }
          if (!mbar_wait(WE(sw), phw ^ 1u, abort_s, a.err)) { ok = false; break; }
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            const uint32_t dst = sW + sw * C::W_STAGE + (mat * 2 + hc) * kTileBytes + i * 128;
#pragma unroll
            for (int wd = 0; wd < NW; ++wd) {
              uint32_t o[4];
              if (BF) dequant_word_bf16(words[NW * hc + wd], sb2[hc], bb2[hc], o);
              else dequant_word(words[NW * hc + wd], s2[hc], b2[hc], o);
              st_shared_v4(dst + ((((uint32_t)(w0 + wd)) ^ swz) << 4), o[0], o[1], o[2], o[3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          // The raw stage is released only now: the stores above consumed the codes loaded from
          // it, so every lane's shared-memory read of the stage has completed.  Releasing it right
          // after issuing those reads let the TMA refill land before slow lanes had read it.
          if (lane == 0) {
            mbar_arrive(RE(s_used));
            mbar_arrive(WF(sw));
          }
          if (++sw == C::S_W) { sw = 0; phw ^= 1u; }
        }
      }
      // A weight row whose every |w| is below 2^-12 (but not all zero) lives in fp16's subnormal
      // range and loses precision there: range flag.
      bad = bad || (wmax > 0.0f && wmax < 2.44140625e-4f);
      wmax = 0.0f;
      if (has_next) {
        srow = srow_n;
        brow = brow_n;
      }
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) raise_flag(a.err, kErrFp16Range);
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;   // TMEM lane quarter this warp may access
    const uint32_t stg = sbase + C::OFF_STG + (uint32_t)q * 2048u;
    int li = 0;
    float amax = 0.0f;   // largest |value| rounded to fp16 (above 65504 it does not fit)
    bool tiny = false;   // a token's h all in fp16's subnormal range (gate/up mode)
    Walk wk;
    walk_init(wk);
    for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++li) {
      const int4 tl = walk_step(wk, u);
      const int m = u % MT;
      const int b = li & 1;
      if (!mbar_wait_warp(AF(b), (li >> 1) & 1, abort_s, a.err)) break;
      tc_fence_after();
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * C::ACC_COLS);
      // Per 16-token block: TMEM -> registers -> this warp's staging buffer ([token][32 rows]) ->
      // 16-byte stores of each token's 32 contiguous output columns.
      const int col0 = m * kBM + q * 32;   // gate/up mode: first output column of this warp's rows
      const int nstep = (MODE == 1 && a.y16 != nullptr) ? 32 : 16;   // fp16 down outputs: 32 per round
      for (int n0 = 0; n0 < tl.z; n0 += nstep) {
        uint32_t g[16];
        if (MODE == 0) {
          uint32_t uu[16];
          tmem_ld16x2_wait(tb + n0, tb + 128 + n0, g, uu);
          const int pos = (lane & ~7) | chunk_pos(lane & 7);   // stored operand order of h
          uint32_t big_m = 0u, nz_m = 0u;   // bit i: this lane's h of token n0 + i is >= 2^-12 / nonzero
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float gv = __uint_as_float(g[i]);
            const float hv = gv * __frcp_rn(1.0f + __expf(-gv)) * __uint_as_float(uu[i]);
            if (n0 + i < tl.z) amax = fmaxf(amax, fabsf(hv));
            big_m |= (fabsf(hv) >= 2.44140625e-4f ? 1u : 0u) << i;
            nz_m |= (hv != 0.0f ? 1u : 0u) << i;
            st_shared_u16(stg + (uint32_t)(i * 32 + pos) * 2, f32_to_16(hv, BF));
          }
          if (!BF) {
            // a token whose h over this warp's 32 rows is nonzero but all below 2^-12 sits in fp16's
            // subnormal range (tiny activations): range flag
            const uint32_t big = __reduce_or_sync(0xFFFFFFFFu, big_m), nz = __reduce_or_sync(0xFFFFFFFFu, nz_m);
            const uint32_t live = tl.z - n0 >= 16 ? 0xFFFFu : ((1u << (tl.z - n0)) - 1u);
            tiny = tiny || ((nz & ~big & live) != 0u);
          }
          __syncwarp();
#pragma unroll
          for (int c = lane; c < 64; c += 32) {
            const int n = c >> 2, p = c & 3;
            if (n0 + n < tl.z) {
              const uint4 v = ld_shared_v4(stg + (uint32_t)(n * 32 + p * 8) * 2);
              *reinterpret_cast<uint4*>(a.h + (size_t)(tl.y + n0 + n) * a.F + col0 + p * 8) = v;
            }
          }
          __syncwarp();
        } else {
          // down mode: the unit's two 128-row blocks sit in TMEM columns 0..127 and 128..255
#pragma unroll 1
          for (int mat = 0; mat < 2; ++mat) {
            const int colm = (2 * m + mat) * kBM + q * 32;
            if (a.y16 != nullptr) {
              // 32 tokens: two 16-column loads and one wait, then [token][32 rows] staging (2 KB)
              uint32_t g1[16];
              tmem_ld16x2_wait(tb + (uint32_t)(mat * 128) + n0, tb + (uint32_t)(mat * 128) + n0 + 16, g, g1);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float v0 = __uint_as_float(g[i]), v1 = __uint_as_float(g1[i]);
                if (n0 + i < tl.z) amax = fmaxf(amax, fabsf(v0));
                if (n0 + 16 + i < tl.z) amax = fmaxf(amax, fabsf(v1));
                const uint32_t pk = f32x2_to_16x2(v0, v1, BF);
                st_shared_u16(stg + (uint32_t)(i * 32 + lane) * 2, (uint16_t)(pk & 0xFFFFu));
                st_shared_u16(stg + (uint32_t)((i + 16) * 32 + lane) * 2, (uint16_t)(pk >> 16));
              }
              __syncwarp();
#pragma unroll
              for (int c = lane; c < 128; c += 32) {
                const int n = c >> 2, p = c & 3;
                if (n0 + n < tl.z) {
                  const uint4 v = ld_shared_v4(stg + (uint32_t)(n * 32 + p * 8) * 2);
                  *reinterpret_cast<uint4*>(a.y16 + (size_t)(tl.y + n0 + n) * a.d + colm + p * 8) = v;
                }
              }
            } else {
              tmem_ld16_wait(tb + (uint32_t)(mat * 128) + n0, g);
#pragma unroll
              for (int i = 0; i < 16; ++i) st_shared_u32(stg + (uint32_t)(i * 32 + lane) * 4, g[i]);
              __syncwarp();
#pragma unroll
              for (int c = lane; c < 128; c += 32) {
                const int n = c >> 3, p = c & 7;
                if (n0 + n < tl.z) {
                  const uint4 v = ld_shared_v4(stg + (uint32_t)(n * 32 + p * 4) * 4);
                  *reinterpret_cast<uint4*>(a.y_perm + (size_t)(tl.y + n0 + n) * a.d + colm + p * 4) = v;
                }
              }
            }
            __syncwarp();
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(AE(b));
    }
    if (!BF && __any_sync(0xFFFFFFFFu, !(amax <= 65504.0f) || tiny) && lane == 0) raise_flag(a.err, kErrFp16Range);
  }

  // Wind down.  After a timeout, give copies that may still be in flight time to land before
  // the CTA's shared memory and tensor memory are released.
  if (threadIdx.x == 0 && *abort_s) {
    const long long t0 = clock64();
    while (clock64() - t0 < 4000000ll) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// y[t] = sum_j w[t,j] Y[inv[t,j]] + gs[t] Y[T*k + t], fp32 accumulation in j order.  Y is read as
// fp16 or bf16 (the layer path) or fp32 (expert outputs handed in by a caller), 8 or 4 values per load.
// An fp16 value h, with its magnitude bits moved up by 13 into a float's exponent and mantissa,
// reads as h * 2^-112 exactly (normal and subnormal h alike); the sign moves up by 16.  Scaling the
// weight by 2^112 instead makes fmaf(w * 2^112, that float, acc) the same operation as
// fmaf(w, h, acc): the weights are at most 1, so w * 2^112 is exact.
__device__ __forceinline__ float fp16_bits_scaled(uint32_t h) {
  return __uint_as_float(((h & 0x7FFFu) << 13) | ((h & 0x8000u) << 16));
}

template <bool HALF, bool BF>
__global__ void combine_kernel(CombineArgs a) {
  constexpr int V = HALF ? 8 : 4;
  // fp16 rows: weights scaled by 2^112 (see fp16_bits_scaled)
  const float wscale = (HALF && !BF) ? 5192296858534827628530496329220096.0f : 1.0f;
  const int t = blockIdx.x;
  const int nv = a.d / V;
  for (int c = threadIdx.x; c < nv; c += blockDim.x) {
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.0f;
    auto add_row = [&](size_t row, float wv) {
      float v[V];
      if (HALF) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(a.y16 + row * a.d) + c);
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (BF) {
            v[2 * i] = bf16_bits_to_f32(qw[i] & 0xFFFFu);
            v[2 * i + 1] = bf16_bits_to_f32(qw[i] >> 16);
          } else {
            v[2 * i] = fp16_bits_scaled(qw[i] & 0xFFFFu);
            v[2 * i + 1] = fp16_bits_scaled(qw[i] >> 16);
          }
        }
      } else {
        const float4 q = __ldg(reinterpret_cast<const float4*>(a.y_perm + row * a.d) + c);
        v[0] = q.x;
        v[1] = q.y;
        v[2 % V] = q.z;
        v[3 % V] = q.w;
      }
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(wv, v[i], acc[i]);
    };
    for (int j = 0; j < a.k; ++j)
      add_row((size_t)__ldg(a.inv + (size_t)t * a.k + j), __ldg(a.w + (size_t)t * a.k + j) * wscale);
    if (a.gs != nullptr) add_row((size_t)a.T * a.k + t, __ldg(a.gs + t) * wscale);
    float4* yo = reinterpret_cast<float4*>(a.y + (size_t)t * a.d + (size_t)c * V);
    yo[0] = make_float4(acc[0], acc[1], acc[2 % V], acc[3 % V]);
    if (HALF) yo[1] = make_float4(acc[4 % V], acc[5 % V], acc[6 % V], acc[7 % V]);
  }
}

// Row s of the gate/up activation operand: x of the token routed to slot s (slots below T*k
// through the permutation, the shared expert's slots T*k + t are token t), converted to fp16 (or
// kept in bf16) in the operand chunk order.  Writing the rows in slot order lets the GEMM fetch every activation
// tile with one TMA box load.
constexpr int kPermRows = 8;   // rows per CTA step: eight independent loads in flight per thread

template <bool BF>
__global__ void __launch_bounds__(256) permute_x_kernel(PermuteArgs a) {
  const int nch = a.d / 8;
  const int Tk = a.T * a.k;
  bool bad = false;
  for (int s0 = blockIdx.x * kPermRows; s0 < a.slots; s0 += gridDim.x * kPermRows) {
    int tok[kPermRows];
#pragma unroll
    for (int i = 0; i < kPermRows; ++i) {
      const int s = s0 + i;
      tok[i] = s >= a.slots ? -1 : s < Tk ? __ldg(a.perm + s) / a.k : s - Tk;
    }
    for (int ch = threadIdx.x; ch < nch; ch += blockDim.x) {
      uint4 xv[kPermRows];
#pragma unroll
      for (int i = 0; i < kPermRows; ++i)
        xv[i] = tok[i] >= 0 ? __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)tok[i] * a.d) + ch)
                            : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < kPermRows; ++i) {
        if (tok[i] < 0) continue;
        const uint32_t xw[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
        // stored order (0,4,1,5,2,6,3,7): word p holds logical elements (p, p+4)
        uint32_t o[4];
        if (BF) {   // bf16 bits as given
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const uint32_t lo = (xw[p >> 1] >> (16 * (p & 1))) & 0xFFFFu;
            const uint32_t hi = (xw[(p + 4) >> 1] >> (16 * (p & 1))) & 0xFFFFu;
            o[p] = lo | (hi << 16);
          }
        } else {
          float xf[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            xf[2 * e] = bf16_bits_to_f32(xw[e] & 0xFFFFu);
            xf[2 * e + 1] = bf16_bits_to_f32(xw[e] >> 16);
          }
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            o[p] = f32x2_to_16x2(xf[p], xf[p + 4], false);
            // an infinity in either half: x above fp16's range
            bad = bad || ((o[p] & 0x7FFFu) == 0x7C00u) || ((o[p] & 0x7FFF0000u) == 0x7C000000u);
          }
        }
        reinterpret_cast<uint4*>(a.xperm + (size_t)(s0 + i) * a.d)[ch] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  if (bad) raise_flag(a.err, kErrFp16Range);
}

}  // namespace

size_t gemm_smem_bytes(int mode) { return mode == 0 ? Cfg<0>::BYTES : Cfg<1>::BYTES; }

cudaError_t launch_gemm(int mode, const GemmMaps& maps, const GemmArgs& a, int grid, cudaStream_t st) {
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaSuccess;
    const int b0 = (int)Cfg<0>::BYTES, b1 = (int)Cfg<1>::BYTES;
    if ((e = cudaFuncSetAttribute(gemm_kernel<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, b0)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(gemm_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, b1)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(gemm_kernel<0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, b0)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(gemm_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, b1)) != cudaSuccess)
      return e;
    configured_dev = dev;
  }
  if (a.bf16) {
    if (mode == 0) gemm_kernel<0, true><<<grid, kThreads, Cfg<0>::BYTES, st>>>(maps, a);
    else gemm_kernel<1, true><<<grid, kThreads, Cfg<1>::BYTES, st>>>(maps, a);
  } else {
    if (mode == 0) gemm_kernel<0, false><<<grid, kThreads, Cfg<0>::BYTES, st>>>(maps, a);
    else gemm_kernel<1, false><<<grid, kThreads, Cfg<1>::BYTES, st>>>(maps, a);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
  if (a.y16 == nullptr) combine_kernel<false, false><<<a.T, 256, 0, st>>>(a);
  else if (a.bf16) combine_kernel<true, true><<<a.T, 256, 0, st>>>(a);
  else combine_kernel<true, false><<<a.T, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_permute_x(const PermuteArgs& a, cudaStream_t st) {
  if (a.slots <= 0) return cudaSuccess;
  const int steps = (a.slots + kPermRows - 1) / kPermRows;
  const int grid = steps < 152 * 8 ? steps : 152 * 8;
  if (a.bf16) permute_x_kernel<true><<<grid, 256, 0, st>>>(a);
  else permute_x_kernel<false><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
