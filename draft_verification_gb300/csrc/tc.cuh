// Tensor-core building blocks for sm_103a: tensor memory (TMEM), the
// fifth-generation MMA (tcgen05.mma, kind::f16 with bfloat16 operands and
// float32 accumulators), tensor-map bulk copies (TMA) into 128-byte-swizzled
// shared memory, and the descriptors that tie them together.
//
// Operand tiles are K-major: a tile of `rows` rows and 64 bfloat16 columns
// (128 bytes per row) lands in shared memory through a TMA copy with the
// 128-byte swizzle, i.e. rows are stored one after another, every 8 rows (a
// 1024-byte atom) with their 16-byte chunks permuted by the row index.  The
// shared-memory matrix descriptor of such a tile:
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4 (unused for this layout: 1)
//   bits 32-45  stride-dimension byte offset >> 4 (1024 B between 8-row atoms)
//   bits 46-47  descriptor version (1 on sm_100-class parts)
//   bits 49-51  base offset (0: atoms are 1024-byte aligned)
//   bit  52     leading-dimension offset mode (0)
//   bits 61-63  swizzle mode (2 = 128-byte swizzle)
// A K step of 16 elements (32 bytes) inside the 128-byte row is taken by
// advancing the start address by 32 bytes; the swizzle is a function of the
// address bits, so the hardware finds the permuted chunks.
//
// Instruction descriptor of kind::f16 (dense):
//   bits  4-5   accumulator format (1 = float32)
//   bits  7-9   A format (1 = bfloat16)       bits 10-12  B format (1 = bfloat16)
//   bit  15     A major (0 = K-major)          bit  16     B major (0 = K-major)
//   bits 17-22  N >> 3                         bits 24-28  M >> 4
//
// Every wait here is bounded (the callers record a fault instead of hanging).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// descriptors
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_byte_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_byte_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;                 // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;         // stride byte offset: one 8-row atom
  d |= static_cast<uint64_t>(1u) << 46;                 // version
  d |= static_cast<uint64_t>(2u) << 61;                 // 128-byte swizzle
  return d;
}

__host__ __device__ constexpr uint32_t umma_idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// tensor memory
// ---------------------------------------------------------------------------
// Allocate `ncols` columns (a power of two, >= 32) of this SM's tensor memory
// for the CTA; one whole warp executes it; the base address is written to
// shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, M x N x 16, bfloat16 in, float32 out.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// 32 consecutive float32 columns of this warp's 32 lanes: thread t receives
// lane (lane_base + t), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive float32 columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------
// CTA pairs (cta_group::2): the two CTAs of a cluster of two act as one MMA
// unit.  A of an M = 256 product is split by rows (rows 0-127 in the even
// CTA's shared memory, 128-255 in the odd CTA's, at the same address), B by
// its N rows (the first N/2 in the even CTA, the rest in the odd one), and D
// by rows (each CTA's TMEM lanes 0-127 hold its 128 rows, all N columns).
// Threads of the even CTA issue the MMAs.  Allocation, relinquishing and
// deallocation are collective: one warp of each CTA of the pair executes
// them.  Within a kernel every tcgen05 instruction uses the same group size.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A * B^T over the pair, M = 256, N x 16, bfloat16 in, float32 out.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

// Arrive once, when every pair MMA this thread issued so far has completed,
// on the mbarrier at `bar`'s offset in each CTA of `cta_mask` (cluster ranks).
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(cta_mask)
      : "memory");
}

// Address of `local`'s counterpart in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* local, unsigned rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(local)), "r"(rank));
  return a;
}

// One arrival on an mbarrier of another CTA of the cluster (address from
// cluster_addr), ordered after this thread's earlier memory accesses.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// ---------------------------------------------------------------------------
// tensor-map bulk copies
// ---------------------------------------------------------------------------
// Copy the box at element coordinates (x, y) of the 2-D tensor described by
// `tmap` (a kernel parameter) into shared memory at `dst`, counting its bytes
// on `bar`.  x times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
  // (bf16 tensors: x must be a multiple of 8 elements; the debug build checks)
  if (kDebugChecks && ((x & 7) != 0 || (smem_addr(dst) & 1023u) != 0)) return;
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Bring the box at (x, y) of the 2-D tensor described by `tmap` into L2
// (no shared memory and no barrier are involved).
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(x), "r"(y)
               : "memory");
}

// Pair form of tma_load_2d: the box lands in this CTA's shared memory at
// `dst`, and its bytes are counted on the mbarrier at cluster address
// `cluster_bar`, which may be the peer CTA's (the even CTA of the pair
// counts both CTAs' operand copies).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const void* tmap, int x, int y, uint32_t cluster_bar) {
  if (kDebugChecks && ((x & 7) != 0 || (smem_addr(dst) & 1023u) != 0)) return;
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(cluster_bar)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// One plain arrival on a CTA-local mbarrier.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

}  // namespace sv
