// Row statistics of one chunk of one logit row (one CTA of 256 threads).
//
// The temperature softmax of the verification rule needs two numbers per
// row: m = max logit and s = sum of 2^(x c - M(m)) (c = log2(e)/T).  Greedy
// verification needs the argmax instead (lowest index on ties).  A chunk is
// 256 threads x 8 coalesced 16-byte loads (16384 bf16 or 8192 fp32
// logits); every thread issues its 8 loads before using any, then takes its
// maximum once (packed bfloat16 max) and sums its weights with packed f32x2
// fma/add, so each logit costs about three instructions plus one ex2.
// Elements before the row's first 16-byte boundary (misaligned row strides)
// and after its last full vector are read as scalars by chunk 0.
#pragma once

#include "common.cuh"

namespace sv {

template <typename T>
struct VecTraits;

template <>
struct VecTraits<bf16_t> {
  static constexpr int kElems = 8;
  static constexpr uint32_t kNegInfWord = 0xff80ff80u;  // two bf16 -inf
};

template <>
struct VecTraits<float> {
  static constexpr int kElems = 4;
  static constexpr uint32_t kNegInfWord = 0xff800000u;
};

template <typename T>
constexpr int chunk_elems() {
  return kStatsThreads * kVecPerThread * VecTraits<T>::kElems;
}

struct StatsSmem {
  float a[kStatsWarps];
  float b[kStatsWarps];
  int i[kStatsWarps];
};

// Geometry of a row: scalar head [0, head), vectors, scalar tail [tail0, V).
template <typename T>
struct RowGeom {
  int head, nvec, tail0;
  __device__ __forceinline__ RowGeom(const T* row, int V) {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
    head = static_cast<int>(((16u - (addr & 15u)) & 15u) / sizeof(T));
    if (head > V) head = V;
    nvec = (V - head) / VecTraits<T>::kElems;
    tail0 = head + nvec * VecTraits<T>::kElems;
  }
};

// Writes out[0] = (m, s) (sampling) or (value or NaN if the chunk holds a
// NaN / +inf, index as int bits) (greedy).  Every thread of the CTA calls it.
template <typename T, bool kGreedy>
__device__ __forceinline__ void stats_unit(const T* row, int V, int k, float c, float2* out,
                                           StatsSmem& sm) {
  constexpr int E = VecTraits<T>::kElems;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RowGeom<T> g(row, V);
  const uint4* vrow = reinterpret_cast<const uint4*>(row + g.head);
  const int v0 = k * (kStatsThreads * kVecPerThread);

  uint4 buf[kVecPerThread];
  constexpr uint32_t NI = VecTraits<T>::kNegInfWord;
#pragma unroll
  for (int j = 0; j < kVecPerThread; ++j) {
    const int vi = v0 + j * kStatsThreads + tid;
    buf[j] = (vi < g.nvec) ? ld_stream16(vrow + vi) : make_uint4(NI, NI, NI, NI);
  }
  // scalar head / tail elements, chunk 0 only (at most E - 1 of each)
  const bool has_h = (k == 0) && tid < g.head;
  const bool has_t = (k == 0) && tid < V - g.tail0;
  const float xh = has_h ? load_elem(row + tid) : -kInf;
  const float xt = has_t ? load_elem(row + g.tail0 + tid) : -kInf;

  if constexpr (kGreedy) {
    float best = -kInf;
    int bi = -1;
    bool bad = false;
    auto see = [&](float x, int idx) {
      bad |= !(x < kInf);
      if (x > best) {
        best = x;
        bi = idx;
      }
    };
    if (has_h) see(xh, tid);
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j) {
      const int base = g.head + (v0 + j * kStatsThreads + tid) * E;
      const uint32_t w[4] = {buf[j].x, buf[j].y, buf[j].z, buf[j].w};
      if constexpr (E == 8) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          see(bf16_lo(w[q]), base + 2 * q);
          see(bf16_hi(w[q]), base + 2 * q + 1);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) see(__uint_as_float(w[q]), base + q);
      }
    }
    if (has_t) see(xt, g.tail0 + tid);
    // fill values (-inf) never win: x > best is false for -inf
    ArgMax am = am_warp_reduce(ArgMax{best, bi});
    const bool wbad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      sm.a[warp] = am.v;
      sm.i[warp] = am.i;
      sm.b[warp] = wbad ? 1.f : 0.f;
    }
    __syncthreads();
    if (warp == 0) {
      const bool have = lane < kStatsWarps;
      ArgMax t{have ? sm.a[lane] : -kInf, have ? sm.i[lane] : -1};
      const bool anyb = __any_sync(0xffffffffu, have && sm.b[lane] != 0.f);
      t = am_warp_reduce(t);
      if (lane == 0) *out = make_float2(anyb ? __int_as_float(0x7fc00000) : t.v, __int_as_float(t.i));
    }
  } else {
    // thread maximum
    float m;
    if constexpr (E == 8) {
      uint32_t mx = buf[0].x;
#pragma unroll
      for (int j = 0; j < kVecPerThread; ++j) {
        if (j > 0) mx = bmax2_nan(mx, buf[j].x);
        mx = bmax2_nan(mx, buf[j].y);
        mx = bmax2_nan(mx, buf[j].z);
        mx = bmax2_nan(mx, buf[j].w);
      }
      m = fmax_nan(bf16_lo(mx), bf16_hi(mx));
    } else {
      m = -kInf;
#pragma unroll
      for (int j = 0; j < kVecPerThread; ++j) {
        m = fmax_nan(m, fmax_nan(fmax_nan(__uint_as_float(buf[j].x), __uint_as_float(buf[j].y)),
                                 fmax_nan(__uint_as_float(buf[j].z), __uint_as_float(buf[j].w))));
      }
    }
    m = fmax_nan(m, fmax_nan(xh, xt));
    float s = 0.f;
    if (m != -kInf) {
      const float M = scaled_max(m, c);
      const float2 cc = make_float2(c, c), mm = make_float2(-M, -M);
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < kVecPerThread; ++j) {
        const uint32_t w[4] = {buf[j].x, buf[j].y, buf[j].z, buf[j].w};
#pragma unroll
        for (int q = 0; q < 4; q += (E == 8 ? 1 : 2)) {
          float2 x;
          if constexpr (E == 8) x = make_float2(bf16_lo(w[q]), bf16_hi(w[q]));
          else x = make_float2(__uint_as_float(w[q]), __uint_as_float(w[q + 1]));
          const float2 a = ffma2(x, cc, mm);
          acc = fadd2(acc, make_float2(ex2(a.x), ex2(a.y)));
        }
      }
      acc = fadd2(acc, make_float2(weight(xh, c, M), weight(xt, c, M)));
      s = __fadd_rn(acc.x, acc.y);
    }
    const MaxSum ws = ms_warp_reduce(MaxSum{m, s}, c);
    if (lane == 0) {
      sm.a[warp] = ws.m;
      sm.b[warp] = ws.s;
    }
    __syncthreads();
    if (warp == 0) {
      const bool have = lane < kStatsWarps;
      const MaxSum t = ms_warp_reduce(MaxSum{have ? sm.a[lane] : -kInf, have ? sm.b[lane] : 0.f}, c);
      if (lane == 0) *out = make_float2(t.m, t.s);
    }
  }
}

}  // namespace sv
