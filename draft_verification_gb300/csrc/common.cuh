// Device helpers shared by the verification kernels (sm_103a).
//
// Numerical conventions used by every kernel, so that the row statistics,
// the accept tests and the sampling passes agree bit for bit:
//   c      = log2(e) / T, rounded once to float on the host
//   M(m)   = __fmul_rn(m, c): the scaled maximum of a row with raw maximum m
//   e(x)   = ex2(fma_rn(x, c, -M)) = 2^(x c - M), the unnormalised weight
//   s      = sum of e(x) over the row
//   p(x)   = e(x) / s
// The unrounded x c - M of one fused multiply-add keeps every weight relative
// to the same shift M, so p(x) computed later from (M, s) is consistent with s.
// The packed (f32x2) forms below round each lane exactly like the scalar
// intrinsics, so packed and scalar code give identical weights.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

// Debug build (SPEC_DEBUG_CHECKS defined; build(debug_checks=True)): the
// vector loads and bulk copies check their alignment preconditions.  A
// misaligned 16-byte load returns NaN bits instead of loading (the row is
// then reported non-finite), and a misaligned bulk copy, L2 prefetch or
// tensor-map copy is not issued (its barrier's bounded wait then gives up
// and the sequence reports SPEC_ERR_INTERNAL), so a broken precondition
// shows up as an error bit instead of a misaligned-address fault.
#ifdef SPEC_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
__device__ __forceinline__ bool misaligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) != 0;
}

constexpr int kStatsThreads = 256;       // row-statistics kernel: small CTAs, many per SM
constexpr int kStatsWarps = kStatsThreads / 32;
constexpr int kVecPerThread = 8;         // 16-byte loads per thread per statistics unit
constexpr int kThreads = 256;            // walk kernels (one CTA of a per-sequence cluster)
constexpr int kWarps = kThreads / 32;
static_assert(kWarps <= 32 && kStatsWarps <= 32, "one warp reduces the per-warp partials");
constexpr int kTileElems = 8 * kThreads; // pass tile: 8 contiguous elements per thread

constexpr float kInf = __builtin_huge_valf();

// bfloat16 is handled as raw 16-bit patterns: the value is the top half of
// a float32 with the same bits.
using bf16_t = uint16_t;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float load_elem(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_elem(const bf16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
}

// 16-byte streaming load that does not allocate in L1 (rows are read once
// by the statistics pass).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  if (kDebugChecks && misaligned16(p)) return make_uint4(0x7fc00000u, 0x7fc00000u, 0x7fc00000u, 0x7fc00000u);
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte load through L2 (the walker re-reads rows the statistics pass
// brought into L2 moments earlier).
__device__ __forceinline__ uint4 ld16(const void* p) {
  if (kDebugChecks && misaligned16(p)) return make_uint4(0x7fc00000u, 0x7fc00000u, 0x7fc00000u, 0x7fc00000u);
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max that returns NaN when either operand is NaN, so that a NaN logit
// poisons the row statistics instead of disappearing.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float y;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

// lane-wise max of two packed bfloat16 pairs, NaN-propagating
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float scaled_max(float m, float c) { return __fmul_rn(m, c); }

// 2^(x c - M): the unnormalised softmax weight of logit x.
__device__ __forceinline__ float weight(float x, float c, float M) {
  return ex2(__fmaf_rn(x, c, -M));
}

// ---------------------------------------------------------------------------
// bulk copies (TMA engine) into shared memory, completed on an mbarrier
// ---------------------------------------------------------------------------
// Bound on an mbarrier wait: kMaxPolls polls, each suspending the thread for
// at most kPollNs nanoseconds (about 65 ms in all) before the wait gives up.
constexpr int kMaxPolls = 1 << 16;
constexpr int kPollNs = 1000;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// Make initialised mbarriers visible to the bulk-copy engine.
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// One arrival that also announces `bytes` of bulk-copy data to come.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  if (kDebugChecks && (misaligned16(dst) || misaligned16(src) || (bytes & 15u))) return;
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "n"(kPollNs)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of `bar` to complete; false if it did not within
// kMaxPolls polls (the caller records a fault instead of hanging).  The
// arrival that completes the phase must already have been issued by a thread
// that is not waiting: a thread issuing copies for a phase that lanes of its
// own warp already wait on could be held back by their suspension.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  for (int i = 0; i < kMaxPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// Bounded wait, with acquire semantics at cluster scope, for phase `parity`
// of a local mbarrier that other CTAs of the cluster send bytes to.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, unsigned parity) {
  for (int i = 0; i < kMaxPolls; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "n"(kPollNs)
        : "memory");
    if (ok) return true;
  }
  return false;
}
// Store v at the address of `local` in cluster CTA `rank`, counting its 4
// bytes on that CTA's mbarrier at the address of `bar` (one network trip:
// the receiver's wait on the barrier makes the value visible).
__device__ __forceinline__ void st_async_cluster(const void* local, unsigned rank, uint32_t v, const uint64_t* bar) {
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_addr(bar)), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(ra), "r"(v), "r"(rb)
               : "memory");
}

// Hint the bulk-copy engine to bring `bytes` (a multiple of 16, 16-byte
// aligned) at `src` into L2.
__device__ __forceinline__ void prefetch_l2(const void* src, unsigned bytes) {
  if (kDebugChecks && (misaligned16(src) || (bytes & 15u))) return;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Order this thread's earlier shared-memory accesses before later bulk copies.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint4 lds16(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

// ---------------------------------------------------------------------------
// double-float numbers: hi + lo with |lo| <= ulp(hi) / 2, about 44 bits of
// precision from float32 arithmetic only (FP64 throughput on GB300 is a small
// fraction of FP32's).  Additions use Knuth's TwoSum, products the fused
// multiply-add error term; every operation is an explicitly rounded
// intrinsic, so the compiler cannot contract or reassociate them.
// ---------------------------------------------------------------------------
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF df_norm(float s, float e) {  // |e| small against s
  const float hi = __fadd_rn(s, e);
  return {hi, __fsub_rn(e, __fsub_rn(hi, s))};
}
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float bb = __fsub_rn(s, a.hi);
  float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  return df_norm(s, e);
}
__device__ __forceinline__ DF df_add_f(DF a, float b) { return df_add(a, DF{b, 0.f}); }
__device__ __forceinline__ DF df_neg(DF a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ DF df_mul_f(DF a, float v) {
  const float p = __fmul_rn(a.hi, v);
  float e = __fmaf_rn(a.hi, v, -p);
  e = __fmaf_rn(a.lo, v, e);
  return df_norm(p, e);
}
__device__ __forceinline__ float df_float(DF a) { return __fadd_rn(a.hi, a.lo); }
__device__ __forceinline__ double df_double(DF a) {
  return static_cast<double>(a.hi) + static_cast<double>(a.lo);
}
__device__ __forceinline__ DF df_shfl_up(DF a, int o) {
  return {__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}

// ---------------------------------------------------------------------------
// (max, sum) pairs of the online softmax
// ---------------------------------------------------------------------------
struct MaxSum {
  float m;  // raw maximum logit (-inf for an empty set)
  float s;  // sum of 2^(x c - M(m))
};

__device__ __forceinline__ MaxSum ms_merge(MaxSum a, MaxSum b, float c) {
  const float m = fmax_nan(a.m, b.m);
  if (m == -kInf) return {m, 0.f};
  const float M = scaled_max(m, c);
  const float ea = ex2(scaled_max(a.m, c) - M);
  const float eb = ex2(scaled_max(b.m, c) - M);
  return {m, __fadd_rn(__fmul_rn(a.s, ea), __fmul_rn(b.s, eb))};
}

// Warp-wide (max, sum): max first, then every lane rescales its sum once and
// the sums are added with a butterfly (fp addition is commutative, so every
// lane ends with the same bits).
__device__ __forceinline__ MaxSum ms_warp_reduce(MaxSum v, float c) {
  float m = v.m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
  if (m != -kInf) s = (v.m == -kInf) ? 0.f : __fmul_rn(v.s, ex2(scaled_max(v.m, c) - scaled_max(m, c)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
  return {m, s};
}

// ---------------------------------------------------------------------------
// (value, index) pairs of the greedy argmax: larger value wins, ties go to
// the lower index; index -1 means "nothing seen".
// ---------------------------------------------------------------------------
struct ArgMax {
  float v;
  int i;
};

__device__ __forceinline__ ArgMax am_merge(ArgMax a, ArgMax b) {
  if (b.i < 0) return a;
  if (a.i < 0) return b;
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}

__device__ __forceinline__ ArgMax am_warp_reduce(ArgMax v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgMax w{__shfl_xor_sync(0xffffffffu, v.v, o), __shfl_xor_sync(0xffffffffu, v.i, o)};
    v = am_merge(v, w);
  }
  return v;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// Allow the next kernel in the stream to be scheduled now.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the previous kernel in the stream has completed and its memory
// is visible (a no-op when this kernel was not launched as a dependent).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// thread-block clusters (one cluster per sequence in the sampling walks)
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_size() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Split cluster barrier.  Every thread of every CTA of the cluster executes
// the same sequence of arrives and waits (the kernels keep the control flow
// around them uniform across the cluster).  Stores to other CTAs' shared
// memory made before an arrive are visible after the matching wait.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}

}  // namespace sv
