// Cluster-wide passes over one (target row, draft row) pair and the
// inverse-CDF draw that follows them.  One thread-block cluster serves one
// sequence; its CTAs split the row into 2048-element tiles (8 contiguous
// elements per thread) and exchange their partial sums through distributed
// shared memory.  Every CTA evaluates the same scalar decisions on the same
// data, so control flow stays uniform across the cluster and only hardware
// cluster barriers are used (no flags, no spinning).
//
// Weight of element x in a pass (speculative-sampling residual; the PipeSpec
// review's Circularity Check cites the rule of Leviathan et al.):
//     w(x) = max(0, p(x) - cq * q(x)),   p = target softmax, q = draft softmax
// cq = 0 draws from p itself (bonus token); cq = 1 is the residual after one
// rejection; larger cq arise after several rejected tree siblings (see
// tree.cu).  The draw returns the first index whose running sum of w, in
// ascending index order, exceeds v * sum(w).
//
// Running sums: fp32 within a thread's 8 elements and within a warp (a fixed
// shuffle scan), a fixed sequential fp32 combination of the 8 warp totals per
// tile, and fp64 across tiles and CTAs.  The pass and the later search use the
// same code for the same tile, so a tile's total is bit-identical in both.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace sv {

namespace cg = cooperative_groups;

constexpr int kMaxCluster = 8;
constexpr int kMaxTilesPerCta = 256;  // V <= 8 * 256 * 2048 = 4,194,304
constexpr int kBatchTiles = 4;        // tiles whose loads are in flight together

// ---------------------------------------------------------------------------
// loading 8 contiguous elements [e0, e0 + 8) of a row, as floats
// ---------------------------------------------------------------------------
template <typename T>
struct Raw8;

// bf16: the 8 elements are 16 bytes; a misaligned row needs the two aligned
// 16-byte windows around them.
template <>
struct Raw8<bf16_t> {
  uint4 a, b;
  int mode;  // 0 aligned, 1 realigned (a,b), 2 scalar (a holds the values), 3 empty

  __device__ __forceinline__ void issue(const bf16_t* row, int e0, int V, bool row_aligned) {
    if (e0 >= V) {
      mode = 3;
    } else if (row_aligned && e0 + 8 <= V) {
      mode = 0;
      a = ld16(row + e0);
    } else if (!row_aligned && e0 + 16 <= V) {
      // window [floor16(addr), +32) ends at or before element e0 + 16 < V
      mode = 1;
      const uintptr_t ad = reinterpret_cast<uintptr_t>(row + e0) & ~static_cast<uintptr_t>(15);
      a = ld16(reinterpret_cast<const void*>(ad));
      b = ld16(reinterpret_cast<const void*>(ad + 16));
    } else {
      mode = 2;
      uint32_t h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        h[e] = (e0 + e < V) ? static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row + e0 + e)))
                            : 0xff80u;  // -inf
      a = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
    }
  }

  __device__ __forceinline__ void get(const bf16_t* row, int e0, float* x) const {
    uint4 w = a;
    if (mode == 1) {
      const int sh = static_cast<int>(reinterpret_cast<uintptr_t>(row + e0) & 15u);  // even, 2..14
      const int q = sh >> 2;
      const int bits = (sh & 3) * 8;
      const uint32_t win[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint32_t o[4];
      switch (q) {
        case 0:
#pragma unroll
          for (int j = 0; j < 4; ++j) o[j] = __funnelshift_r(win[j], win[j + 1], bits);
          break;
        case 1:
#pragma unroll
          for (int j = 0; j < 4; ++j) o[j] = __funnelshift_r(win[j + 1], win[j + 2], bits);
          break;
        case 2:
#pragma unroll
          for (int j = 0; j < 4; ++j) o[j] = __funnelshift_r(win[j + 2], win[j + 3], bits);
          break;
        default:
#pragma unroll
          for (int j = 0; j < 4; ++j) o[j] = __funnelshift_r(win[j + 3], win[j + 4], bits);
          break;
      }
      w = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (mode == 3) {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = -kInf;
      return;
    }
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x);
    x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z);
    x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
  }
};

// fp32: the 8 elements are 32 bytes; a misaligned row needs three windows.
template <>
struct Raw8<float> {
  uint4 a, b, c;
  int mode;

  __device__ __forceinline__ void issue(const float* row, int e0, int V, bool row_aligned) {
    if (e0 >= V) {
      mode = 3;
    } else if (row_aligned && e0 + 8 <= V) {
      mode = 0;
      a = ld16(row + e0);
      b = ld16(row + e0 + 4);
    } else if (!row_aligned && e0 + 12 <= V) {
      // window [floor16(addr), +48) ends at or before element e0 + 12 <= V
      mode = 1;
      const uintptr_t ad = reinterpret_cast<uintptr_t>(row + e0) & ~static_cast<uintptr_t>(15);
      a = ld16(reinterpret_cast<const void*>(ad));
      b = ld16(reinterpret_cast<const void*>(ad + 16));
      c = ld16(reinterpret_cast<const void*>(ad + 32));
    } else {
      mode = 2;
      float h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = (e0 + e < V) ? __ldg(row + e0 + e) : -kInf;
      a = make_uint4(__float_as_uint(h[0]), __float_as_uint(h[1]), __float_as_uint(h[2]), __float_as_uint(h[3]));
      b = make_uint4(__float_as_uint(h[4]), __float_as_uint(h[5]), __float_as_uint(h[6]), __float_as_uint(h[7]));
    }
  }

  __device__ __forceinline__ void get(const float* row, int e0, float* x) const {
    if (mode == 3) {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = -kInf;
      return;
    }
    if (mode == 1) {
      const int q = static_cast<int>((reinterpret_cast<uintptr_t>(row + e0) & 15u) >> 2);  // 1..3
      const uint32_t win[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
      switch (q) {
        case 1:
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(win[e + 1]);
          break;
        case 2:
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(win[e + 2]);
          break;
        default:
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(win[e + 3]);
          break;
      }
      return;
    }
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
    x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
  }
};

template <typename T>
__device__ __forceinline__ bool row_is_aligned(const T* row) {
  return (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
}

// ---------------------------------------------------------------------------
// the rows and scalars of one pass
// ---------------------------------------------------------------------------
template <typename T>
struct PassSpec {
  const T* P;      // target row
  const T* Q;      // draft row (read only when cq != 0)
  float MP, invSP; // scaled max and 1/sum of the target row
  float MQ, invSQ;
  float cq;        // coefficient of q
};

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

// ---------------------------------------------------------------------------
// shared state of the walker kernels
// ---------------------------------------------------------------------------
struct PassShared {
  float tile_sum[kMaxTilesPerCta];
  float warp_tot[kBatchTiles][kWarps];
  float warp_excl[kWarps];
  float thr_incl[kThreads];
  double cta_tot[2];            // this CTA's total, double-buffered by pass parity
  double rank_excl[kMaxCluster];
  double rank_tot[kMaxCluster];
  double Z;
  double E;                     // search: running sum before the chosen tile
  int tile;                     // search: chosen tile (local index)
  int thread;                   // search: chosen thread
  int last_mode;                // search: no index exceeded the target; take the last
  int result[2];                // drawn index, double-buffered by search parity
  int parity;
  int sparity;
};

// Tiles of the row owned by this CTA.
__device__ __forceinline__ void cta_tiles(int V, int cs, int rank, int& t0, int& t1) {
  const int ntiles = (V + kTileElems - 1) / kTileElems;
  const int per = (ntiles + cs - 1) / cs;
  t0 = rank * per;
  t1 = min(ntiles, t0 + per);
  if (t0 > t1) t0 = t1;
}

// One pass: sum of w over the whole row, cluster-wide.  Leaves the per-tile
// sums of this CTA and the per-rank totals in shared memory for run_search.
// Must be called by every thread of every CTA of the cluster.
template <typename T>
__device__ double run_pass(const PassSpec<T>& S, int V, float c, PassShared& sh, cg::cluster_group& cl) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cs = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  int t0, t1;
  cta_tiles(V, cs, rank, t0, t1);
  const bool alP = row_is_aligned(S.P);
  const bool useQ = S.cq != 0.f;
  const bool alQ = useQ ? row_is_aligned(S.Q) : true;

  for (int tb = t0; tb < t1; tb += kBatchTiles) {
    const int nb = min(kBatchTiles, t1 - tb);
    Raw8<T> rp[kBatchTiles], rq[kBatchTiles];
#pragma unroll
    for (int j = 0; j < kBatchTiles; ++j) {
      if (j < nb) {
        const int e0 = (tb + j) * kTileElems + 8 * tid;
        rp[j].issue(S.P, e0, V, alP);
        if (useQ) rq[j].issue(S.Q, e0, V, alQ);
      }
    }
#pragma unroll
    for (int j = 0; j < kBatchTiles; ++j) {
      if (j < nb) {
        const int e0 = (tb + j) * kTileElems + 8 * tid;
        float xp[8], xq[8], w[8];
        rp[j].get(S.P, e0, xp);
        if (useQ) rq[j].get(S.Q, e0, xq);
        pass_weights(S, c, xp, xq, w);
        const float incl = warp_incl_scan(sum8(w));
        if (lane == 31) sh.warp_tot[j][warp] = incl;
      }
    }
    __syncthreads();
    if (tid < nb) {
      float s = sh.warp_tot[tid][0];
      for (int w = 1; w < kWarps; ++w) s = __fadd_rn(s, sh.warp_tot[tid][w]);
      sh.tile_sum[tb - t0 + tid] = s;
    }
    __syncthreads();
  }
  if (tid == 0) {
    double tot = 0.0;
    for (int j = 0; j < t1 - t0; ++j) tot += static_cast<double>(sh.tile_sum[j]);
    sh.cta_tot[sh.parity] = tot;
  }
  cl.sync();
  if (tid == 0) {
    double run = 0.0;
    for (int k = 0; k < cs; ++k) {
      const PassShared* other = cl.map_shared_rank(&sh, k);
      const double t = other->cta_tot[sh.parity];
      sh.rank_excl[k] = run;
      sh.rank_tot[k] = t;
      run += t;
    }
    sh.Z = run;
    sh.parity ^= 1;
  }
  __syncthreads();
  return sh.Z;
}

// Inverse-CDF draw over the weights of the last run_pass (same S): the first
// index y whose running sum exceeds `target` (= v * Z).  Every CTA calls it;
// the CTA holding y stores it in its result slot; the return value is the
// rank of that CTA.  Read the index with fetch_result after a cluster sync.
template <typename T>
__device__ int run_search(const PassSpec<T>& S, int V, float c, double target, PassShared& sh,
                          cg::cluster_group& cl) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cs = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());

  // owner CTA: first with a positive total whose range passes the target,
  // else the last with a positive total (target rounded up to Z)
  int owner = -1, last_pos = -1;
  for (int k = 0; k < cs; ++k) {
    if (sh.rank_tot[k] > 0.0) {
      last_pos = k;
      if (owner < 0 && sh.rank_excl[k] + sh.rank_tot[k] > target) owner = k;
    }
  }
  const bool last_mode_cta = owner < 0;
  if (owner < 0) owner = last_pos < 0 ? 0 : last_pos;
  const int sp = sh.sparity;
  if (rank != owner) {
    __syncthreads();
    if (tid == 0) sh.sparity ^= 1;
    __syncthreads();
    return owner;
  }

  int t0, t1;
  cta_tiles(V, cs, rank, t0, t1);
  if (tid == 0) {
    double E = sh.rank_excl[rank];
    int tile = -1, last_tile = -1;
    double E_last = E;
    for (int j = 0; j < t1 - t0; ++j) {
      const double s = static_cast<double>(sh.tile_sum[j]);
      if (s > 0.0) {
        if (!last_mode_cta && E + s > target) {
          tile = j;
          break;
        }
        last_tile = j;
        E_last = E;
      }
      E += s;
    }
    sh.last_mode = (tile < 0);
    sh.tile = tile >= 0 ? tile : (last_tile >= 0 ? last_tile : 0);
    sh.E = tile >= 0 ? E : E_last;
  }
  __syncthreads();

  // recompute the chosen tile exactly as run_pass did
  const int e0 = (t0 + sh.tile) * kTileElems + 8 * tid;
  Raw8<T> rp, rq;
  const bool useQ = S.cq != 0.f;
  rp.issue(S.P, e0, V, row_is_aligned(S.P));
  if (useQ) rq.issue(S.Q, e0, V, row_is_aligned(S.Q));
  float xp[8], xq[8], w[8];
  rp.get(S.P, e0, xp);
  if (useQ) rq.get(S.Q, e0, xq);
  pass_weights(S, c, xp, xq, w);
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
  const bool pass_here = mine > 0.f && (sh.last_mode ? true : (sh.E + static_cast<double>(incl) > target));
  // first thread that passes the target (last thread with mass in last mode)
  const unsigned bal = __ballot_sync(0xffffffffu, pass_here);
  if (tid == 0) sh.thread = sh.last_mode ? -1 : kThreads;
  __syncthreads();
  if (bal != 0 && lane == 0) {
    if (sh.last_mode) atomicMax(&sh.thread, warp * 32 + 31 - __clz(bal));
    else atomicMin(&sh.thread, warp * 32 + __ffs(bal) - 1);
  }
  __syncthreads();
  int t = sh.thread;
  if (t < 0 || t >= kThreads) t = 0;
  if (tid == t) {
    const double base = sh.E + ((t == 0) ? 0.0 : static_cast<double>(sh.thr_incl[t - 1]));
    double run = base;
    int y = -1, last = -1;
    for (int e = 0; e < 8; ++e) {
      run += static_cast<double>(w[e]);
      if (w[e] > 0.f) {
        last = e;
        if (!sh.last_mode && y < 0 && run > target) y = e;
      }
    }
    if (y < 0) y = last < 0 ? 0 : last;
    int idx = e0 + y;
    if (idx >= V) idx = V - 1;
    sh.result[sp] = idx;
  }
  __syncthreads();
  if (tid == 0) sh.sparity ^= 1;
  __syncthreads();
  return owner;
}

// The index drawn by the last run_search, read from the owner CTA.  Call
// after a cluster sync that follows run_search.
__device__ __forceinline__ int fetch_result(PassShared& sh, int owner, cg::cluster_group& cl) {
  const PassShared* o = cl.map_shared_rank(&sh, owner);
  return o->result[sh.sparity ^ 1];
}

// log2 of the softmax probability of logit x in a row with stats (m, s),
// computed in double from the same scaled quantities as the passes.
__device__ __forceinline__ double log2_prob(float x, float m, float s, float c) {
  if (x == -kInf) return -INFINITY;
  const double M = static_cast<double>(scaled_max(m, c));
  return static_cast<double>(x) * static_cast<double>(c) - M - log2(static_cast<double>(s));
}

// Accept-test ratio p/q from log2 p and log2 q (q = 0 keeps iff p > 0).
__device__ __forceinline__ double accept_ratio(double lp, double lq) {
  if (lq == -INFINITY) return lp == -INFINITY ? 0.0 : INFINITY;
  return exp2(lp - lq);
}

__device__ __forceinline__ bool keeps(float u, double ratio) {
  return static_cast<double>(u) < (ratio < 1.0 ? ratio : 1.0);
}

// Merge the chunk partials of one statistics row (one warp).
__device__ __forceinline__ MaxSum combine_row(const float2* part, int chunks, float c) {
  const int lane = threadIdx.x & 31;
  MaxSum acc{-kInf, 0.f};
  for (int k = lane; k < chunks; k += 32) {
    const float2 p = part[k];
    acc = ms_merge(acc, MaxSum{p.x, p.y}, c);
  }
  return ms_warp_merge(acc, c);
}

__device__ __forceinline__ ArgMax combine_row_argmax(const float2* part, int chunks, bool& bad) {
  const int lane = threadIdx.x & 31;
  ArgMax acc{-kInf, -1};
  bool b = false;
  for (int k = lane; k < chunks; k += 32) {
    const float2 p = part[k];
    if (p.x != p.x) b = true;
    acc = am_merge(acc, ArgMax{p.x, __float_as_int(p.y)});
  }
  bad = __any_sync(0xffffffffu, b);
  return am_warp_merge(acc);
}

__device__ __forceinline__ bool row_stats_ok(MaxSum ms) {
  return ms.m > -kInf && ms.m < kInf && ms.s > 0.f && ms.s < kInf;
}

}  // namespace sv
