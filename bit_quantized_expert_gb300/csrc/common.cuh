// Device helpers shared by the MoE kernels: error flags, bounded mbarrier waits, TMA and
// bulk copies, tcgen05 (TMEM allocation, MMA, commit, loads) and small numeric helpers.
// All inline PTX here is hand-written against the public PTX ISA for sm_100-family targets.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace moe {

// ------------------------------------------------------------------------------------------
// Error flags (one uint32 word at the start of the caller's workspace)
// ------------------------------------------------------------------------------------------
constexpr uint32_t kErrWaitTimeout = 1u;   // a bounded wait gave up; outputs are invalid
constexpr uint32_t kErrFp16Range = 2u;     // a value did not fit the fp16 operand type
constexpr uint32_t kErrBadRouting = 4u;    // routing tables inconsistent with the dims
constexpr uint32_t kErrNonFinite = 8u;     // an activation of the decode path is not finite

// About two seconds at the maximum SM clock: no correct launch waits this long.
constexpr long long kWaitTimeoutCycles = 4000000000ll;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void raise_flag(uint32_t* err, uint32_t f) {
  if (err != nullptr) atomicOr(err, f);
}

// ------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete.  Gives up (returns false) when the CTA-wide
// abort word is set by another role, or after `limit` cycles, in which case it sets the abort
// word and the timeout flag.  No wait in these kernels is unbounded: they all use
// kWaitTimeoutCycles (mbar_wait); only the wait probe passes a shorter limit.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, volatile int* abort_s, uint32_t* err,
                                              long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_s) return false;
    if (clock64() - t0 > limit) {
      *abort_s = 1;
      raise_flag(err, kErrWaitTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_s,
                                          uint32_t* err) {
  return mbar_wait_for(bar, parity, abort_s, err, kWaitTimeoutCycles);
}

// The same wait for a whole warp that next executes warp-collective (.sync.aligned)
// instructions such as tcgen05.ld: mbar_wait is a per-lane polling loop, so lanes may leave it at
// different iterations; the warp is reconverged and agrees on the outcome before returning.
__device__ __forceinline__ bool mbar_wait_warp_for(uint32_t bar, uint32_t parity, volatile int* abort_s,
                                                   uint32_t* err, long long limit) {
  const bool ok = mbar_wait_for(bar, parity, abort_s, err, limit);
  __syncwarp();
  return __all_sync(0xFFFFFFFFu, ok);
}

__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_s,
                                               uint32_t* err) {
  return mbar_wait_warp_for(bar, parity, abort_s, err, kWaitTimeoutCycles);
}

// ------------------------------------------------------------------------------------------
// Bulk and tensor copies (TMA)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 16-byte asynchronous global->shared copy (used for row gathers).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// 4-byte asynchronous global->shared copy (both addresses 4-byte aligned).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later async-proxy reads
// (tensor-core operand fetches).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------------------------------
// Programmatic dependent launch
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both operands K-major 16-bit, fp32 accumulation.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The eight MMAs of one 64-wide K chunk for two weight tiles that share one activation tile:
// for K step kk = 0..3 and tile j = 0..1, D_j (+)= A_j[kk] B[kk], where the operand of step kk
// starts 32 bytes (2 in the descriptor's address field) after that of step kk-1 and the first
// step accumulates only if `accumulate` is non-zero.  One asm statement, so every descriptor is
// in a register before the first MMA and the eight instructions issue back to back: an issuing
// warp that shares its scheduler with busy warps then waits for one issue slot per MMA, not for
// the several an MMA and its descriptor arithmetic would need.
__device__ __forceinline__ void tc_mma_f16_chunk2(uint32_t d0, uint32_t d1, uint64_t a0, uint64_t a1, uint64_t b,
                                                  uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t"
      "setp.ne.b32 p, %15, 0;\n\t"
      "setp.ne.b32 t, %16, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %14, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %6, %10, %14, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %14, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %7, %11, %14, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %14, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %8, %12, %14, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %14, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %9, %13, %14, t;\n\t}" ::"r"(d0),
      "r"(d1), "l"(a0), "l"(a0 + 2u), "l"(a0 + 4u), "l"(a0 + 6u), "l"(a1), "l"(a1 + 2u), "l"(a1 + 4u), "l"(a1 + 6u),
      "l"(b), "l"(b + 2u), "l"(b + 4u), "l"(b + 6u), "r"(idesc), "r"(accumulate), "r"(1u)
      : "memory");
}

// Arrive (once) on an mbarrier when all tcgen05 operations issued so far by this thread complete.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// TMEM -> registers.  tcgen05.ld is asynchronous: its destination registers hold valid data
// only after tcgen05.wait::ld.  Load and wait sit in ONE asm statement, so for the compiler the
// registers are defined only after the wait and no use of them can be scheduled ahead of it.
// Each thread of the warp reads 16 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "{\n\ttcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
      "[%16];\n\ttcgen05.wait::ld.sync.aligned;\n\t}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Two 16-column loads (TMEM addresses ta, tb) and one wait, in one statement.
__device__ __forceinline__ void tmem_ld16x2_wait(uint32_t ta, uint32_t tb, uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile(
      "{\n\ttcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
      "[%32];\n\ttcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,"
      "%29,%30,%31}, [%33];\n\ttcgen05.wait::ld.sync.aligned;\n\t}"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
        "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
        "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
        "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
      : "r"(ta), "r"(tb)
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored in the 128-byte swizzled
// canonical layout: rows of 64 16-bit elements (128 B), 8-row atoms 1024 B apart, the 16-byte
// chunk index of row r XOR-ed with (r & 7).  The tile base must be 1024-byte aligned; the
// start address may advance by 32 B per K=16 step inside the atom.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);           // start address
  d |= (uint64_t)(16u >> 4) << 16;                    // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024u >> 4) << 32;                  // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                             // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                             // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, fp16 x fp16 -> fp32, both K-major, M x N.
__device__ __forceinline__ uint32_t idesc_f16_f32(uint32_t M, uint32_t N) {
  return (1u << 4)                 // D format fp32
         | (0u << 7) | (0u << 10)  // A, B format fp16
         | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// ------------------------------------------------------------------------------------------
// Numerics
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// Position of logical element i (0..7) of an 8-element chunk in the operand layout used by the
// tensor-core path: the chunk is stored as elements (0,4,1,5,2,6,3,7).  Both operands of every
// contraction use the same order, so the dot products are unchanged.
__host__ __device__ __forceinline__ int chunk_pos(int i) { return ((i & 3) << 1) | (i >> 2); }

}  // namespace moe
