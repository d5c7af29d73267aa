// Residual / bonus passes over a (target row, draft row) pair and the
// inverse-CDF draw that follows them.
//
// Weight of element x in a pass (the speculative-sampling residual; the
// PipeSpec review's Circularity Check cites the rule of Leviathan et al.):
//     w(x) = max(0, p(x) - cq * q(x)),   p = target softmax, q = draft softmax
// cq = 0 draws from p itself (the bonus token); cq = 1 is the residual after
// one rejection; larger cq arise after several rejected tree siblings (see
// verify.cu).  The draw returns the first index whose running sum of w, in
// ascending index order, exceeds v * sum(w).
//
// A pass is split into tiles of kTileElems = 8 * kThreads contiguous elements
// (8 per thread).  Any CTA can compute the sums of any range of tiles, so a
// pass is spread over many CTAs (slices), each writing its tiles' sums to
// global memory; the CTA that finishes the last slice draws the token.
//
// Running sums: fp32 within a thread's 8 elements and within a warp (a fixed
// shuffle scan), a fixed sequential fp32 combination of the per-warp totals
// per tile, and fp64 across tiles.  The pass and the draw recompute a tile
// with the same code, so a tile's total is bit-identical in both.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int kMaxTiles = 512;  // V <= 512 * kTileElems

// ---------------------------------------------------------------------------
// the rows and scalars of one pass
// ---------------------------------------------------------------------------
template <typename T>
struct PassSpec {
  const T* P;       // target row
  const T* Q;       // draft row (read only when cq != 0)
  float MP, invSP;  // scaled max and 1/sum of the target row
  float MQ, invSQ;
  float cq;         // coefficient of q
  int pad;
};

// ---------------------------------------------------------------------------
// loading this thread's 8 elements [e0, e0 + 8) of a row
// ---------------------------------------------------------------------------
// Aligned rows: one (bf16) or two (fp32) 16-byte loads; the last partial
// vector of a row and anything past V is read as scalars / -inf.
template <typename T>
struct Load8;

template <>
struct Load8<bf16_t> {
  static constexpr int kRegs = 4;
  __device__ __forceinline__ static void issue(const bf16_t* row, int e0, int V, uint32_t* r) {
    if (e0 + 8 <= V) {
      const uint4 v = ld16(row + e0);
      r[0] = v.x; r[1] = v.y; r[2] = v.z; r[3] = v.w;
    } else {
      uint32_t h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        h[e] = (e0 + e < V) ? static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row + e0 + e)))
                            : 0xff80u;
#pragma unroll
      for (int q = 0; q < 4; ++q) r[q] = h[2 * q] | (h[2 * q + 1] << 16);
    }
  }
  __device__ __forceinline__ static void get(const uint32_t* r, float* x) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      x[2 * q] = bf16_lo(r[q]);
      x[2 * q + 1] = bf16_hi(r[q]);
    }
  }
};

template <>
struct Load8<float> {
  static constexpr int kRegs = 8;
  __device__ __forceinline__ static void issue(const float* row, int e0, int V, uint32_t* r) {
    if (e0 + 8 <= V) {
      const uint4 a = ld16(row + e0), b = ld16(row + e0 + 4);
      r[0] = a.x; r[1] = a.y; r[2] = a.z; r[3] = a.w;
      r[4] = b.x; r[5] = b.y; r[6] = b.z; r[7] = b.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) r[e] = __float_as_uint((e0 + e < V) ? __ldg(row + e0 + e) : -kInf);
    }
  }
  __device__ __forceinline__ static void get(const uint32_t* r, float* x) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(r[e]);
  }
};

// Misaligned rows (row stride not a multiple of 16 bytes): the 8 elements
// come from the aligned 16-byte windows around them.  A window starts inside
// the same row or the previous row of the same array (an array's first row
// is aligned, so never before the array) and, while e0 + 8 + 16 / size <= V,
// ends before the row's end; otherwise scalar loads are used.
template <typename T>
__device__ __forceinline__ void load8_misaligned(const T* row, int e0, int V, float* x) {
  constexpr int kSize = static_cast<int>(sizeof(T));
  if (e0 + 8 + 16 / kSize <= V) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(row + e0);
    const uintptr_t base = a & ~static_cast<uintptr_t>(15);
    const int sh = static_cast<int>(a - base);
    constexpr int kWin = (8 * kSize) / 16 + 1;  // 2 windows (bf16) or 3 (fp32)
    uint32_t win[4 * kWin];
#pragma unroll
    for (int k = 0; k < kWin; ++k) {
      const uint4 v = ld16(reinterpret_cast<const void*>(base + 16 * k));
      win[4 * k] = v.x; win[4 * k + 1] = v.y; win[4 * k + 2] = v.z; win[4 * k + 3] = v.w;
    }
    // the 8 * kSize bytes starting at byte `sh`
    const int q = sh >> 2, bits = (sh & 3) * 8;
    uint32_t o[2 * kSize];
#pragma unroll
    for (int j = 0; j < 2 * kSize; ++j) {
      uint32_t lo = win[j], hi = win[j + 1];
#pragma unroll
      for (int k = 1; k < 4; ++k)  // select win[j + q], win[j + q + 1] without dynamic indexing
        if (q == k) {
          lo = win[j + k];
          hi = win[j + k + 1];
        }
      o[j] = __funnelshift_r(lo, hi, bits);
    }
    if constexpr (kSize == 2) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[2 * k] = bf16_lo(o[k]);
        x[2 * k + 1] = bf16_hi(o[k]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(o[e]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (e0 + e < V) ? load_elem(row + e0 + e) : -kInf;
  }
}

template <typename T>
__device__ __forceinline__ bool row_is_aligned(const T* row) {
  return (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
}

// Weights of 8 elements.
template <typename T>
__device__ __forceinline__ void pass_weights(const PassSpec<T>& S, float c, const float* xp,
                                             const float* xq, float* w) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float p = __fmul_rn(weight(xp[e], c, S.MP), S.invSP);
    if (S.cq != 0.f) {
      const float q = __fmul_rn(weight(xq[e], c, S.MQ), S.invSQ);
      w[e] = fmaxf(__fmaf_rn(-S.cq, q, p), 0.f);
    } else {
      w[e] = p;
    }
  }
}

// Sequential fp32 sum of a thread's 8 weights.
__device__ __forceinline__ float sum8(const float* w) {
  float s = w[0];
#pragma unroll
  for (int e = 1; e < 8; ++e) s = __fadd_rn(s, w[e]);
  return s;
}

__device__ __forceinline__ float warp_incl_scan(float x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = __fadd_rn(x, y);
  }
  return x;
}

// This thread's 8 weights of tile `tile`.
template <typename T>
__device__ __forceinline__ void tile_weights(const PassSpec<T>& S, int V, float c, int tile, float* w) {
  const int e0 = tile * kTileElems + 8 * threadIdx.x;
  float xp[8], xq[8];
  const bool useQ = S.cq != 0.f;
  if (row_is_aligned(S.P)) {
    uint32_t r[Load8<T>::kRegs];
    Load8<T>::issue(S.P, e0, V, r);
    Load8<T>::get(r, xp);
  } else {
    load8_misaligned(S.P, e0, V, xp);
  }
  if (useQ) {
    if (row_is_aligned(S.Q)) {
      uint32_t r[Load8<T>::kRegs];
      Load8<T>::issue(S.Q, e0, V, r);
      Load8<T>::get(r, xq);
    } else {
      load8_misaligned(S.Q, e0, V, xq);
    }
  }
  pass_weights(S, c, xp, xq, w);
}

struct PassSmem {
  float warp_tot[4][kWarps];
  float warp_excl[kWarps];
  float thr_incl[kThreads];
  double tile_excl[kMaxTiles];
  double total;
  double E;
  int tile;
  int thread;
  int last_mode;
  int result;
};

// Sum of a tile's weights from the per-warp totals (fixed sequential order).
__device__ __forceinline__ float tile_total(const float* warp_tot) {
  float s = warp_tot[0];
#pragma unroll 1
  for (int k = 1; k < kWarps; ++k) s = __fadd_rn(s, warp_tot[k]);
  return s;
}

// Sums of tiles [t0, t1) into out[t0 .. t1) (global or shared).  All threads
// call it.  Aligned rows keep 2 tiles (4 rows' loads) in flight per thread.
template <typename T>
__device__ void tile_sums(const PassSpec<T>& S, int V, float c, int t0, int t1, float* out,
                          PassSmem& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool useQ = S.cq != 0.f;
  const bool aligned = row_is_aligned(S.P) && (!useQ || row_is_aligned(S.Q));
  for (int tb = t0; tb < t1; tb += 2) {
    const int nb = min(2, t1 - tb);
    if (aligned) {
      uint32_t rp[2][Load8<T>::kRegs], rq[2][Load8<T>::kRegs];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (j < nb) {
          const int e0 = (tb + j) * kTileElems + 8 * tid;
          Load8<T>::issue(S.P, e0, V, rp[j]);
          if (useQ) Load8<T>::issue(S.Q, e0, V, rq[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (j < nb) {
          float xp[8], xq[8], w[8];
          Load8<T>::get(rp[j], xp);
          if (useQ) Load8<T>::get(rq[j], xq);
          pass_weights(S, c, xp, xq, w);
          const float incl = warp_incl_scan(sum8(w));
          if (lane == 31) sh.warp_tot[j][warp] = incl;
        }
      }
    } else {
#pragma unroll 1
      for (int j = 0; j < nb; ++j) {
        float w[8];
        tile_weights(S, V, c, tb + j, w);
        const float incl = warp_incl_scan(sum8(w));
        if (lane == 31) sh.warp_tot[j][warp] = incl;
      }
    }
    __syncthreads();
    if (tid < nb) out[tb + tid] = tile_total(sh.warp_tot[tid]);
    __syncthreads();
  }
}

// fp64 exclusive prefix of ntiles tile sums (one warp; the sums are read
// through L2 since other CTAs may have written them).  Leaves the prefix in
// sh.tile_excl and returns the total to every thread.
__device__ double tile_prefix(const float* sums, int ntiles, PassSmem& sh) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    const int per = (ntiles + 31) / 32;
    const int j0 = min(ntiles, tid * per), j1 = min(ntiles, j0 + per);
    double run = 0.0;
    for (int j = j0; j < j1; ++j) run += static_cast<double>(__ldcg(sums + j));
    double incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += y;
    }
    double acc = __shfl_up_sync(0xffffffffu, incl, 1);
    if (tid == 0) acc = 0.0;
    for (int j = j0; j < j1; ++j) {
      sh.tile_excl[j] = acc;
      acc += static_cast<double>(__ldcg(sums + j));
    }
    if (tid == 31) sh.total = incl;
  }
  __syncthreads();
  return sh.total;
}

// Inverse-CDF draw over tile sums `sums` (prefix from tile_prefix): the first
// index whose running sum exceeds `target`.  Recomputes the chosen tile with
// the same code as tile_sums.  All threads call it; all get the index.
template <typename T>
__device__ int draw(const PassSpec<T>& S, int V, float c, const float* sums, int ntiles, double target,
                    PassSmem& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 32) {
    // first tile with mass whose end passes the target, else the last with mass
    int first = ntiles, last = -1;
    for (int j = lane; j < ntiles; j += 32) {
      const float s = __ldcg(sums + j);
      if (s > 0.f) {
        if (first == ntiles && sh.tile_excl[j] + static_cast<double>(s) > target) first = j;
        last = j;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
      last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    }
    if (lane == 0) {
      sh.last_mode = first == ntiles;
      sh.tile = first < ntiles ? first : (last >= 0 ? last : 0);
      sh.E = sh.tile_excl[sh.tile];
      sh.thread = sh.last_mode ? -1 : kThreads;
    }
  }
  __syncthreads();
  const int tile = sh.tile;
  float w[8];
  tile_weights(S, V, c, tile, w);
  const float mine = sum8(w);
  const float incl_w = warp_incl_scan(mine);
  if (lane == 31) sh.warp_tot[0][warp] = incl_w;
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
    for (int k = 0; k < kWarps; ++k) {
      sh.warp_excl[k] = s;
      s = (k == 0) ? sh.warp_tot[0][0] : __fadd_rn(s, sh.warp_tot[0][k]);
    }
  }
  __syncthreads();
  const float incl = (warp == 0) ? incl_w : __fadd_rn(sh.warp_excl[warp], incl_w);
  sh.thr_incl[tid] = incl;
  const bool last_mode = sh.last_mode;
  const bool pass_here = mine > 0.f && (last_mode || sh.E + static_cast<double>(incl) > target);
  const unsigned bal = __ballot_sync(0xffffffffu, pass_here);
  if (bal != 0 && lane == 0) {
    if (last_mode) atomicMax(&sh.thread, warp * 32 + 31 - __clz(bal));
    else atomicMin(&sh.thread, warp * 32 + __ffs(bal) - 1);
  }
  __syncthreads();
  int t = sh.thread;
  if (t < 0 || t >= kThreads) t = 0;
  if (tid == t) {
    double run = sh.E + ((t == 0) ? 0.0 : static_cast<double>(sh.thr_incl[t - 1]));
    int y = -1, lastpos = -1;
    for (int e = 0; e < 8; ++e) {
      run += static_cast<double>(w[e]);
      if (w[e] > 0.f) {
        lastpos = e;
        if (!last_mode && y < 0 && run > target) y = e;
      }
    }
    if (y < 0) y = lastpos < 0 ? 0 : lastpos;
    int idx = tile * kTileElems + 8 * t + y;
    if (idx >= V) idx = V - 1;
    sh.result = idx;
  }
  __syncthreads();
  return sh.result;
}

// ---------------------------------------------------------------------------
// scalar probabilities and the accept test (float32 throughout)
// ---------------------------------------------------------------------------
// p(x) for logit x in a row with stats (m, s): 2^(x c - M(m)) / s, with the
// exponent formed exactly as in the passes.
__device__ __forceinline__ float prob(float x, float m, float s, float c) {
  return __fdiv_rn(exp2f(__fmaf_rn(x, c, -scaled_max(m, c))), s);
}

// r = p(x)/q(x) from the token's target logit xp and draft logit xq:
// 2^((xp - xq) c - (M_P - M_Q)) * (s_Q / s_P) with the exponent rounded once.
// q(x) = 0 (xq = -inf) keeps iff p(x) > 0.
__device__ __forceinline__ float ratio(float xp, float mP, float sP, float xq, float mQ, float sQ,
                                       float c) {
  if (xq == -kInf) return xp == -kInf ? 0.f : kInf;
  if (xp == -kInf) return 0.f;
  const float d = __fsub_rn(xp, xq);
  const float D = __fsub_rn(scaled_max(mP, c), scaled_max(mQ, c));
  return __fmul_rn(exp2f(__fmaf_rn(d, c, -D)), __fdiv_rn(sQ, sP));
}

__device__ __forceinline__ bool keeps(float u, float r) { return u < fminf(1.f, r); }

// Merge the chunk partials of one statistics row (one warp; partials were
// written by other CTAs of this grid, so they are read past L1).
__device__ __forceinline__ MaxSum combine_row(const float2* part, int chunks, float c) {
  const int lane = threadIdx.x & 31;
  MaxSum acc{-kInf, 0.f};
  for (int k = lane; k < chunks; k += 32) {
    const float2 p = __ldcg(part + k);
    acc = ms_merge(acc, MaxSum{p.x, p.y}, c);
  }
  return ms_warp_reduce(acc, c);
}

__device__ __forceinline__ ArgMax combine_row_argmax(const float2* part, int chunks, bool& bad) {
  const int lane = threadIdx.x & 31;
  ArgMax acc{-kInf, -1};
  bool b = false;
  for (int k = lane; k < chunks; k += 32) {
    const float2 p = __ldcg(part + k);
    if (p.x != p.x) b = true;
    acc = am_merge(acc, ArgMax{p.x, __float_as_int(p.y)});
  }
  bad = __any_sync(0xffffffffu, b);
  return am_warp_reduce(acc);
}

__device__ __forceinline__ bool row_stats_ok(MaxSum ms) {
  return ms.m > -kInf && ms.m < kInf && ms.s > 0.f && ms.s < kInf;
}

}  // namespace sv
