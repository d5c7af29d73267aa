// Row statistics: one streaming pass over every logit row of a call.
//
// Sampling mode computes, per 8192-element chunk of a row, the online-softmax
// pair (m, s): m = max logit, s = sum of 2^(x c - M(m)) with c = log2(e)/T
// (the temperature softmax of the verification rule needs exactly these two
// numbers per row).  Greedy mode computes the argmax (lowest index on ties)
// and no exponential.  Chunks are merged later, in a fixed order, by the
// walker kernels, so the result does not depend on scheduling.
//
// Layout and bandwidth: one CTA of 256 threads per (row, chunk); each thread
// issues all of its 16-byte loads (8 bf16 or 4 fp32 logits each) before it
// consumes any, so a CTA keeps 16 KB (bf16) / 32 KB (fp32) in flight.  Loads
// are coalesced (consecutive threads read consecutive 16-byte vectors) and
// bypass L1.  A row whose start is not 16-byte aligned is split into a short
// scalar head, an aligned vector body and a scalar tail.  The CTA order runs
// from the last sequence to the first, so the rows still in L2 when the
// walker starts are those of the first sequences, which the walker's first
// clusters re-read.
#include "common.cuh"
#include "internal.h"

namespace sv {
namespace {

template <typename T>
struct Vec;  // elements per 16-byte vector and their unpacking

template <>
struct Vec<bf16_t> {
  static constexpr int kElems = 8;
  __device__ static void unpack(const uint4& w, float* x) {
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x);
    x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z);
    x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
  }
};

template <>
struct Vec<float> {
  static constexpr int kElems = 4;
  __device__ static void unpack(const uint4& w, float* x) {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
};

// Online (max, sum) state of one thread.
struct SoftmaxAcc {
  float m = -kInf;  // raw max
  float M = -kInf;  // scaled max, __fmul_rn(m, c)
  float s = 0.f;

  template <int N>
  __device__ __forceinline__ void add(const float* x, float c) {
    float vmax = x[0];
#pragma unroll
    for (int e = 1; e < N; ++e) vmax = fmax_nan(vmax, x[e]);
    if (!(vmax <= m)) {  // a larger value, or a NaN on either side
      const float mn = fmax_nan(m, vmax);
      const float Mn = scaled_max(mn, c);
      s = __fmul_rn(s, ex2(M - Mn));
      m = mn;
      M = Mn;
    }
    if (m != -kInf) {
#pragma unroll
      for (int e = 0; e < N; ++e) s = __fadd_rn(s, weight(x[e], c, M));
    }
  }
};

// Argmax state of one thread; elements must arrive in increasing index.
struct ArgMaxAcc {
  float v = -kInf;
  int i = -1;
  bool bad = false;  // a NaN or +inf seen

  template <int N>
  __device__ __forceinline__ void add(const float* x, int first_index) {
#pragma unroll
    for (int e = 0; e < N; ++e) {
      bad |= !(x[e] < kInf);
      if (x[e] > v) {
        v = x[e];
        i = first_index + e;
      }
    }
  }
};

template <typename T, bool kGreedy>
__global__ void __launch_bounds__(kThreads) row_stats_kernel(const StatsParams P) {
  // Let the dependent walker grid be scheduled as soon as this grid's last
  // CTAs are running; it waits for our results with griddepcontrol.wait.
  pdl_launch_dependents();

  constexpr int E = Vec<T>::kElems;
  constexpr int kVecPerChunk = kChunk / E;
  constexpr int kVecPerThread = kVecPerChunk / kThreads;

  const int tid = threadIdx.x;
  const int per_seq = P.rows_per_seq * P.chunks;
  const int unit = blockIdx.x;
  const int b = P.B - 1 - unit / per_seq;
  const int rem = unit - (P.B - 1 - b) * per_seq;
  const int r = rem / P.chunks;
  const int k = rem - r * P.chunks;

  // which tensor holds row r (selects, not an indexed parameter array)
  int i = r;
  const void* base = P.set[0].base;
  int rows = P.set[0].rows;
  if (P.nsets > 1 && i >= rows) {
    i -= rows;
    base = P.set[1].base;
    rows = P.set[1].rows;
    if (P.nsets > 2 && i >= rows) {
      i -= rows;
      base = P.set[2].base;
      rows = P.set[2].rows;
    }
  }
  const T* row = static_cast<const T*>(base) + (static_cast<long long>(b) * rows + i) * P.ld;

  // head: elements before the first 16-byte boundary
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
  int head = static_cast<int>(((16u - (addr & 15u)) & 15u) / sizeof(T));
  if (head > P.V) head = P.V;
  const int nvec = (P.V - head) / E;
  const int tail0 = head + nvec * E;
  const uint4* vrow = reinterpret_cast<const uint4*>(row + head);

  const int v0 = k * kVecPerChunk;
  uint4 buf[kVecPerThread];
#pragma unroll
  for (int j = 0; j < kVecPerThread; ++j) {
    const int vi = v0 + j * kThreads + tid;
    if (vi < nvec) buf[j] = ld_stream16(vrow + vi);
  }

  __shared__ float sh_a[kWarps];
  __shared__ float sh_b[kWarps];
  __shared__ int sh_c[kWarps];
  float2* out = P.partials + (static_cast<long long>(b) * P.rows_per_seq + r) * P.chunks + k;

  if constexpr (kGreedy) {
    ArgMaxAcc acc;
    if (k == 0 && tid < head) {
      float x = load_elem(row + tid);
      acc.add<1>(&x, tid);
    }
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j) {
      const int vi = v0 + j * kThreads + tid;
      if (vi < nvec) {
        float x[E];
        Vec<T>::unpack(buf[j], x);
        acc.add<E>(x, head + vi * E);
      }
    }
    if (k == 0 && tid < P.V - tail0) {
      float x = load_elem(row + tail0 + tid);
      acc.add<1>(&x, tail0 + tid);
    }
    ArgMax am = am_warp_merge(ArgMax{acc.v, acc.i});
    const bool bad = __any_sync(0xffffffffu, acc.bad);
    if ((tid & 31) == 0) {
      sh_a[tid >> 5] = am.v;
      sh_c[tid >> 5] = am.i;
      sh_b[tid >> 5] = bad ? 1.f : 0.f;
    }
    __syncthreads();
    if (tid == 0) {
      ArgMax t{sh_a[0], sh_c[0]};
      bool any_bad = sh_b[0] != 0.f;
      for (int w = 1; w < kWarps; ++w) {
        t = am_merge(t, ArgMax{sh_a[w], sh_c[w]});
        any_bad |= sh_b[w] != 0.f;
      }
      *out = make_float2(any_bad ? __int_as_float(0x7fc00000) : t.v, __int_as_float(t.i));
    }
  } else {
    const float c = P.c;
    SoftmaxAcc acc;
    if (k == 0 && tid < head) {
      float x = load_elem(row + tid);
      acc.add<1>(&x, c);
    }
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j) {
      const int vi = v0 + j * kThreads + tid;
      if (vi < nvec) {
        float x[E];
        Vec<T>::unpack(buf[j], x);
        acc.add<E>(x, c);
      }
    }
    if (k == 0 && tid < P.V - tail0) {
      float x = load_elem(row + tail0 + tid);
      acc.add<1>(&x, c);
    }
    MaxSum ms = ms_warp_merge(MaxSum{acc.m, acc.s}, c);
    if ((tid & 31) == 0) {
      sh_a[tid >> 5] = ms.m;
      sh_b[tid >> 5] = ms.s;
    }
    __syncthreads();
    if (tid == 0) {
      MaxSum t{sh_a[0], sh_b[0]};
      for (int w = 1; w < kWarps; ++w) t = ms_merge(t, MaxSum{sh_a[w], sh_b[w]}, c);
      *out = make_float2(t.m, t.s);
    }
  }
}

}  // namespace

cudaError_t launch_row_stats(const StatsParams& p, bool bf16, bool greedy, cudaStream_t s) {
  const long long units = static_cast<long long>(p.B) * p.rows_per_seq * p.chunks;
  if (units <= 0) return cudaSuccess;
  if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid(static_cast<unsigned>(units)), block(kThreads);
  if (bf16) {
    if (greedy) row_stats_kernel<bf16_t, true><<<grid, block, 0, s>>>(p);
    else row_stats_kernel<bf16_t, false><<<grid, block, 0, s>>>(p);
  } else {
    if (greedy) row_stats_kernel<float, true><<<grid, block, 0, s>>>(p);
    else row_stats_kernel<float, false><<<grid, block, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace sv
