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
// (8 per thread).  The CTAs of one thread-block cluster (one cluster per
// sequence) each sum a slice of the tiles and store the sums into the shared
// memory of every CTA of the cluster; after one cluster barrier every CTA
// holds the whole row's tile sums, so the total and the tile of the draw are
// found without another trip through global memory.
//
// Running sums: fp32 within a thread's 8 elements and within a warp (a fixed
// shuffle scan), a fixed sequential fp32 combination of the per-warp totals
// per tile, and double-float (two fp32 numbers) across tiles.  The pass and
// the draw recompute a tile with the same code, so a tile's total is
// bit-identical in both.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int kMaxTiles = 1024;  // V <= kMaxTiles * kTileElems = 2,097,152

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
  unsigned extra_tx;  // bytes each bulk-copy wait (a ring stage or a resident
                      // slice) expects beyond its copies: 0, or 16 under the
                      // copy-timeout test hook
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

// Weights of 8 elements, two at a time in packed f32x2 arithmetic (each lane
// rounds exactly like the scalar intrinsics: fma, ex2, mul, fma, max).
template <typename T>
__device__ __forceinline__ void pass_weights(const PassSpec<T>& S, float c, const float* xp,
                                             const float* xq, float* w) {
  const float2 cc = make_float2(c, c);
  const float2 mp = make_float2(-S.MP, -S.MP), ip = make_float2(S.invSP, S.invSP);
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const float2 ap = ffma2(make_float2(xp[e], xp[e + 1]), cc, mp);
    const float2 p = fmul2(make_float2(ex2(ap.x), ex2(ap.y)), ip);
    if (S.cq != 0.f) {
      const float2 mq = make_float2(-S.MQ, -S.MQ), iq = make_float2(S.invSQ, S.invSQ);
      const float2 ncq = make_float2(-S.cq, -S.cq);
      const float2 aq = ffma2(make_float2(xq[e], xq[e + 1]), cc, mq);
      const float2 q = fmul2(make_float2(ex2(aq.x), ex2(aq.y)), iq);
      const float2 d = ffma2(ncq, q, p);
      w[e] = fmaxf(d.x, 0.f);
      w[e + 1] = fmaxf(d.y, 0.f);
    } else {
      w[e] = p.x;
      w[e + 1] = p.y;
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

// Tiles a thread keeps in flight on the register path of tile_sums (two
// 16-byte loads, target and draft row, per bf16 tile; four per float32
// tile), kept small: the register path only serves misaligned rows and a
// row's last partial tile.
template <typename T>
struct PassBatch {
  static constexpr int k = 2;
};
template <>
struct PassBatch<float> {
  static constexpr int k = 1;
};
constexpr int kMaxBatch = 2;

// Bulk-copy pipeline of the staged path: kStages buffers, each holding
// kStageRowBytes of the target row and as much of the draft row.  They are
// the first kStageBytes of the walk kernels' dynamic shared memory.
constexpr int kStageRowBytes = 8192;
constexpr int kStages = 2;
constexpr int kStageBytes = kStages * 2 * kStageRowBytes;
constexpr int kMaxCluster = 8;
constexpr int kResidentTiles = 16;  // tiles of a resident slice (two bf16 rows of 16 tiles: 128 KB)
extern __shared__ __align__(128) unsigned char dyn_smem[];

struct PassSmem {
  float warp_tot[2][kMaxBatch][kWarps];  // ring of per-warp tile totals
  float res_tot[kResidentTiles][kWarps]; // per-warp totals of the resident tiles
  float warp_excl[kWarps];
  float thr_incl[kThreads];
  float all[2][kMaxTiles];  // tile sums of a whole pass, double-buffered
  uint64_t bar[kStages];    // one mbarrier per stage buffer
  uint64_t xbar[2];         // tile-sum exchange between the CTAs of the cluster
  uint64_t lbar;            // loads of a resident slice
  int loads;                // resident slices loaded so far (phase of lbar)
  int staged;               // stages issued by earlier passes of this kernel
  int exchanges;            // exchanges completed by earlier passes
  int flt[kMaxCluster];     // fault state of each CTA of the cluster
  float xv[2][kMaxCluster][4];  // per-CTA values shared across the cluster (double-buffered)
  float red[2][kWarps][2];      // per-warp (max, sum) of two rows (block reductions)
  int fault;                // a bulk copy here or in a peer did not complete
  float rf;                 // target minus the prefix before the drawn tile
  int owner;                // CTA whose slice holds the drawn tile
  int tile;
  int thread;
  int last_mode;
  int result;
};

// Before the first pass (thread 0; the kernel synchronises before any pass,
// and peers write flt[] only after the cluster entry barrier).  The stage
// mbarriers are initialised once per kernel: every pass continues their
// phases (stage number `staged + k` uses buffer (staged + k) % kStages in
// its ((staged + k) / kStages)-th phase).
// The exchange barriers complete when the CTA itself has armed them with the
// bytes its peers will send for the pass and all those bytes have landed;
// pass number x uses xbar[x & 1] in its (x >> 1)-th phase.
__device__ __forceinline__ void pass_begin(PassSmem& sh) {
  if (threadIdx.x == 0) {
    sh.fault = 0;
    sh.staged = 0;
    sh.exchanges = 0;
    sh.loads = 0;
    for (int r = 0; r < kMaxCluster; ++r) sh.flt[r] = 0;
    for (int s = 0; s < kStages; ++s) mbar_init(&sh.bar[s], 1);
    mbar_init(&sh.lbar, 1);
    mbar_init(&sh.xbar[0], 1);
    mbar_init(&sh.xbar[1], 1);
    mbar_fence_init();
  }
}

// Sum of a tile's weights from the per-warp totals (fixed sequential order).
__device__ __forceinline__ float tile_total(const float* warp_tot) {
  float s = warp_tot[0];
#pragma unroll 1
  for (int k = 1; k < kWarps; ++k) s = __fadd_rn(s, warp_tot[k]);
  return s;
}

// This thread's 8 elements of tile j of a staged row.
template <typename T>
__device__ __forceinline__ void stage_load8(const unsigned char* row, int j, uint32_t* r) {
  const unsigned char* p = row + static_cast<size_t>(j * kTileElems + 8 * threadIdx.x) * sizeof(T);
  const uint4 a = lds16(p);
  r[0] = a.x; r[1] = a.y; r[2] = a.z; r[3] = a.w;
  if constexpr (sizeof(T) == 4) {
    const uint4 b = lds16(p + 16);
    r[4] = b.x; r[5] = b.y; r[6] = b.z; r[7] = b.w;
  }
}

// Elements [0, Vv) of a row come in whole 16-byte vectors: what a bulk copy
// of an aligned row can bring; elements [Vv, V) are read one by one.
template <typename T>
__device__ __forceinline__ int vector_end(int V) {
  constexpr int E = 16 / static_cast<int>(sizeof(T));
  return V / E * E;
}

// This thread's 8 elements of tile `tile` of a staged row whose copy in
// `row` (local tile j) holds its elements below vector_end(V): elements in
// [Vv, V) are loaded from the row in global memory `g`, elements >= V are
// -inf.  Used for a row's last, partial tile.
template <typename T>
__device__ __forceinline__ void stage_load8_tail(const unsigned char* row, int j, const T* g, int tile, int V,
                                                 float* x) {
  const int Vv = vector_end<T>(V);
  const int e0 = tile * kTileElems + 8 * threadIdx.x;
  const T* s = reinterpret_cast<const T*>(row) + j * kTileElems + 8 * threadIdx.x;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int idx = e0 + e;
    float v = -kInf;
    if (idx < Vv) {
      if constexpr (sizeof(T) == 2) v = __uint_as_float(static_cast<uint32_t>(s[e]) << 16);
      else v = s[e];
    } else if (idx < V) {
      v = load_elem(g + idx);
    }
    x[e] = v;
  }
}

// Staged path: tiles [t0, t1) of rows whose addresses are 16-byte aligned,
// the row's last tile included even when it is partial (its whole vectors
// come by bulk copy, the rest by plain loads).  Thread 0 streams the tiles
// through kStages shared-memory buffers with bulk copies (one mbarrier per
// buffer, up to kStages in flight) while all threads compute the tiles
// already landed.  A buffer is refilled only after the barrier that ends the
// computation on it.
template <typename T>
__device__ void staged_sums(const PassSpec<T>& S, int V, float c, int t0, int t1, float* out, PassSmem& sh) {
  constexpr int TPS = kStageRowBytes / (kTileElems * static_cast<int>(sizeof(T)));  // tiles per stage
  static_assert(TPS >= 1 && TPS <= kMaxBatch, "stage geometry");
  constexpr int R = Load8<T>::kRegs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool useQ = S.cq != 0.f;
  const int nst = (t1 - t0 + TPS - 1) / TPS;
  const int g0 = sh.staged;  // global number of this pass's first stage
  const int Vv = vector_end<T>(V);
  auto issue = [&](int k) {  // thread 0
    const int ta = t0 + k * TPS, te = min(t1, ta + TPS);
    // whole vectors of tiles [ta, te): a multiple of 16 bytes, possibly 0
    const unsigned bytes = static_cast<unsigned>((min(te * kTileElems, Vv) - ta * kTileElems) * sizeof(T));
    const int b = (g0 + k) % kStages;
    unsigned char* buf = dyn_smem + b * 2 * kStageRowBytes;
    mbar_expect_tx(&sh.bar[b], (useQ ? 2 * bytes : bytes) + S.extra_tx);
    if (bytes == 0) return;  // the arrival alone completes the phase
    bulk_load(buf, S.P + static_cast<long long>(ta) * kTileElems, bytes, &sh.bar[b]);
    if (useQ) bulk_load(buf + kStageRowBytes, S.Q + static_cast<long long>(ta) * kTileElems, bytes, &sh.bar[b]);
  };
  if (tid == 0) {
    fence_proxy_async();  // the buffers were last read by ordinary loads
    for (int k = 0; k < min(kStages, nst); ++k) issue(k);
  }
  // Nobody waits before the first stages are issued (thread 0 shares a warp
  // with waiting threads); later stages are issued after the barrier that
  // ends a stage, long before anyone waits on them.
  __syncthreads();
  bool fault = false;
  int slot = 0;
  for (int k = 0; k < nst; ++k, slot ^= 1) {
    const int ta = t0 + k * TPS, nb = min(TPS, t1 - ta);
    const int b = (g0 + k) % kStages;
    const unsigned char* buf = dyn_smem + b * 2 * kStageRowBytes;
    if (!mbar_wait(&sh.bar[b], ((g0 + k) / kStages) & 1)) fault = true;
#pragma unroll
    for (int j = 0; j < TPS; ++j) {
      if (j < nb) {
        float xp[8], xq[8], w[8];
        if ((ta + j + 1) * kTileElems <= Vv) {
          uint32_t rp[R], rq[R];
          stage_load8<T>(buf, j, rp);
          Load8<T>::get(rp, xp);
          if (useQ) {
            stage_load8<T>(buf + kStageRowBytes, j, rq);
            Load8<T>::get(rq, xq);
          }
        } else {  // the row's last tile, partial
          stage_load8_tail<T>(buf, j, S.P, ta + j, V, xp);
          if (useQ) stage_load8_tail<T>(buf + kStageRowBytes, j, S.Q, ta + j, V, xq);
        }
        pass_weights(S, c, xp, xq, w);
        const float incl = warp_incl_scan(sum8(w));
        if (lane == 31) sh.warp_tot[slot][j][warp] = incl;
      }
    }
    __syncthreads();  // buffer b is free; the warp totals are complete
    if (tid < nb) out[ta + tid] = tile_total(sh.warp_tot[slot][tid]);
    if (tid == 0 && k + kStages < nst) {
      fence_proxy_async();
      issue(k + kStages);
    }
  }
  if (fault) {
    // a copy that did not land in time may still be in flight: wait for the
    // last use of every buffer once more (bounded) before it is reused
    for (int k = max(0, nst - kStages); k < nst; ++k)
      mbar_wait(&sh.bar[(g0 + k) % kStages], ((g0 + k) / kStages) & 1);
    sh.fault = 1;
  }
  if (tid == 0) sh.staged = g0 + nst;  // read by the next pass after tile_sums' barrier
}

// Register path: tiles [t0, t1) loaded straight from global memory, NB
// tiles per thread in flight (misaligned rows, and a row's last partial tile).
template <typename T>
__device__ void direct_sums(const PassSpec<T>& S, int V, float c, int t0, int t1, float* out, PassSmem& sh) {
  constexpr int NB = PassBatch<T>::k;
  constexpr int R = Load8<T>::kRegs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool useQ = S.cq != 0.f;
  const bool aligned = row_is_aligned(S.P) && (!useQ || row_is_aligned(S.Q));
  int slot = 0;
  for (int tb = t0; tb < t1; tb += NB, slot ^= 1) {
    const int nb = min(NB, t1 - tb);
    if (aligned) {
      uint32_t rp[NB][R], rq[NB][R];
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        if (j < nb) {
          const int e0 = (tb + j) * kTileElems + 8 * tid;
          Load8<T>::issue(S.P, e0, V, rp[j]);
          if (useQ) Load8<T>::issue(S.Q, e0, V, rq[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        if (j < nb) {
          float xp[8], xq[8], w[8];
          Load8<T>::get(rp[j], xp);
          if (useQ) Load8<T>::get(rq[j], xq);
          pass_weights(S, c, xp, xq, w);
          const float incl = warp_incl_scan(sum8(w));
          if (lane == 31) sh.warp_tot[slot][j][warp] = incl;
        }
      }
    } else {
#pragma unroll 1
      for (int j = 0; j < nb; ++j) {
        float w[8];
        tile_weights(S, V, c, tb + j, w);
        const float incl = warp_incl_scan(sum8(w));
        if (lane == 31) sh.warp_tot[slot][j][warp] = incl;
      }
    }
    __syncthreads();
    // the ring slot written next is the other one, so no second barrier
    if (tid < nb) out[tb + tid] = tile_total(sh.warp_tot[slot][tid]);
  }
}

// ---------------------------------------------------------------------------
// resident slices: a CTA's tiles [t0, t1) of a (target, draft) row pair kept
// in the stage region of shared memory, so that several passes over the same
// rows (the sibling passes at one tree node) read the logits once
// ---------------------------------------------------------------------------
// Bytes of a resident slice of `nt` tiles of both rows.
template <typename T>
__host__ __device__ constexpr size_t slice_bytes(int nt) {
  return 2 * static_cast<size_t>(nt) * kTileElems * sizeof(T);
}

// Whether `nt` tiles of both rows fit in `region` bytes of dynamic shared
// memory (by default the stage region every walk kernel has).
template <typename T>
__device__ __forceinline__ bool slice_fits(int nt, size_t region = kStageBytes) {
  return nt <= kResidentTiles && slice_bytes<T>(nt) <= region;
}

// This thread's 8 elements of local tile j of a resident row as floats.
template <typename T>
__device__ __forceinline__ void slice_get8(const unsigned char* buf, int j, float* x) {
  uint32_t r[Load8<T>::kRegs];
  stage_load8<T>(buf, j, r);
  Load8<T>::get(r, x);
}

// Store 8 floats that are values of T into local tile j of a resident row.
template <typename T>
__device__ __forceinline__ void slice_put8(unsigned char* buf, int j, const float* x) {
  T* p = reinterpret_cast<T*>(buf) + j * kTileElems + 8 * threadIdx.x;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if constexpr (sizeof(T) == 2) p[e] = static_cast<bf16_t>(__float_as_uint(x[e]) >> 16);
    else p[e] = x[e];
  }
}

// Tiles [t0, t1) of `row` into buf (local tile 0 = t0).  Full tiles of a
// 16-byte-aligned row by bulk copy, issued by thread 0 on `bar` (the byte
// count is returned); the rest (misaligned rows, a row's last partial tile)
// by plain loads, with -inf past V.
template <typename T>
__device__ unsigned slice_issue(const T* row, int V, int t0, int t1, unsigned char* buf, uint64_t* bar) {
  const int tf = row_is_aligned(row) ? max(t0, min(t1, V / kTileElems)) : t0;
  unsigned bytes = 0;
  if (tf > t0) {
    bytes = static_cast<unsigned>((tf - t0) * kTileElems * sizeof(T));
    if (threadIdx.x == 0) bulk_load(buf, row + static_cast<long long>(t0) * kTileElems, bytes, bar);
  }
  for (int t = tf; t < t1; ++t) {
    float x[8];
    const int e0 = t * kTileElems + 8 * threadIdx.x;
    if (row_is_aligned(row)) {
      uint32_t r[Load8<T>::kRegs];
      Load8<T>::issue(row, e0, V, r);
      Load8<T>::get(r, x);
    } else {
      load8_misaligned(row, e0, V, x);
    }
    slice_put8<T>(buf, t - t0, x);
  }
  return bytes;
}

// Load this CTA's slice of the pass's rows (the draft row only when
// `with_q`) into the stage region; every thread returns after the data is
// in place.  A load that does not complete in time sets the fault state.
template <typename T>
__device__ void slice_load(const PassSpec<T>& S, bool with_q, int V, int t0, int t1, PassSmem& sh) {
  const int tpc = t1 - t0;
  unsigned char* pbuf = dyn_smem;
  unsigned char* qbuf = dyn_smem + static_cast<size_t>(tpc) * kTileElems * sizeof(T);
  __syncthreads();  // earlier passes have finished with the stage region
  if (threadIdx.x == 0) fence_proxy_async();
  unsigned bytes = slice_issue(S.P, V, t0, t1, pbuf, &sh.lbar);
  if (with_q) bytes += slice_issue(S.Q, V, t0, t1, qbuf, &sh.lbar);
  const int phase = sh.loads;
  if (threadIdx.x == 0) mbar_expect_tx(&sh.lbar, bytes + S.extra_tx);
  __syncthreads();  // armed and issued before anyone waits; plain stores visible
  if (!mbar_wait(&sh.lbar, phase & 1)) sh.fault = 1;
  __syncthreads();
  if (threadIdx.x == 0) sh.loads = phase + 1;
}

// Sums of the resident tiles (local 0 .. t1 - t0) into out[t0 .. t1), with
// the same arithmetic as the other paths.  Every tile's per-warp totals are
// formed before one barrier; then one thread per tile adds them.
template <typename T>
__device__ void resident_sums(const PassSpec<T>& S, float c, int t0, int t1, float* out, PassSmem& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tpc = t1 - t0;
  const unsigned char* pbuf = dyn_smem;
  const unsigned char* qbuf = dyn_smem + static_cast<size_t>(tpc) * kTileElems * sizeof(T);
  const bool useQ = S.cq != 0.f;
  for (int j = 0; j < tpc; ++j) {
    float xp[8], xq[8], w[8];
    slice_get8<T>(pbuf, j, xp);
    if (useQ) slice_get8<T>(qbuf, j, xq);
    pass_weights(S, c, xp, xq, w);
    const float incl = warp_incl_scan(sum8(w));
    if (lane == 31) sh.res_tot[j][warp] = incl;
  }
  __syncthreads();
  if (tid < tpc) out[t0 + tid] = tile_total(sh.res_tot[tid]);
  __syncthreads();
}

// Sums of tiles [t0, t1) into out[t0 .. t1) (shared memory).  All threads
// call it; out[] is complete when it returns.  Tiles of aligned rows go
// through the staged path, tiles of misaligned rows through the register
// path.
template <typename T>
__device__ void tile_sums(const PassSpec<T>& S, int V, float c, int t0, int t1, float* out, PassSmem& sh) {
  const bool useQ = S.cq != 0.f;
  const bool aligned = row_is_aligned(S.P) && (!useQ || row_is_aligned(S.Q));
  if (t1 <= t0) {
  } else if (aligned) {
    staged_sums(S, V, c, t0, t1, out, sh);
  } else {
    direct_sums(S, V, c, t0, t1, out, sh);
  }
  __syncthreads();
}

// Contiguous block of tiles handled by one lane of the prefix.
__device__ __forceinline__ void lane_block(int ntiles, int lane, int& j0, int& j1) {
  const int per = (ntiles + 31) / 32;
  j0 = min(ntiles, lane * per);
  j1 = min(ntiles, j0 + per);
}

// Inclusive double-float scan of the tile sums all[0 .. ntiles) by one warp:
// lane l adds the tiles of its block [j0, j1) in order, the block sums are
// scanned across the lanes by shuffles (a fixed order), and each lane gets
// the prefix before its block in *excl.  Returns the total to every lane.
// Every warp that runs it on the same tile sums gets the same bits.
__device__ DF warp_tile_scan(const float* all, int ntiles, DF* excl) {
  const int lane = threadIdx.x & 31;
  int j0, j1;
  lane_block(ntiles, lane, j0, j1);
  DF blk{0.f, 0.f};
  for (int j = j0; j < j1; ++j) blk = df_add_f(blk, all[j]);
  DF incl = blk;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF y = df_shfl_up(incl, o);
    if (lane >= o) incl = df_add(y, incl);
  }
  const DF prev = df_shfl_up(incl, 1);
  *excl = lane == 0 ? DF{0.f, 0.f} : prev;
  return {__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
}

// One pass split over the CTAs of the cluster (from the resident slice when
// `resident`, which then holds this CTA's tiles of the pass's rows).  CTA
// `rank` sums its slice of the tiles into sh.all[buf] and sends the sums to
// every other CTA of the cluster by asynchronous stores that count on the
// receiver's exchange barrier (warp 0); once its own barrier has every
// peer's bytes, each CTA holds every tile sum.
// Returns the pass total, the warp_tile_scan total of all tile sums (the
// same bits in every warp of every CTA).  Every CTA of the cluster calls it
// with the same pass.  Consecutive passes alternate `buf` and the exchange
// barrier: a CTA can send into a peer's buffer or barrier again only after
// it has received that peer's data for the next pass, which the peer sends
// after it has finished reading this one (fault states are not
// double-buffered: they only go from 0 to 1, so reading a later one is
// harmless).  A wait that gives up sets the fault state instead of hanging.
template <typename T>
__device__ DF cluster_pass(const PassSpec<T>& S, int V, float c, int ntiles, int buf, PassSmem& sh,
                           bool resident = false) {
  const int tid = threadIdx.x;
  const int rank = static_cast<int>(cluster_rank()), n = static_cast<int>(cluster_size());
  const int tpc = (ntiles + n - 1) / n;
  const int t0 = min(ntiles, rank * tpc), t1 = min(ntiles, t0 + tpc);
  float* all = sh.all[buf];
  if (resident) resident_sums(S, c, t0, t1, all, sh);
  else tile_sums(S, V, c, t0, t1, all, sh);
  if (n > 1) {
    int x = 0;  // exchanges completed before this one (thread 0 keeps the count)
    if (tid < 32) {
      x = __shfl_sync(0xffffffffu, sh.exchanges, 0);
      // every peer's tile sums and fault state arrive by asynchronous stores
      // counted on this CTA's exchange barrier
      uint64_t* xb = &sh.xbar[x & 1];
      if (tid == 0) {
        unsigned expect = 0;
        for (int d = 0; d < n; ++d)
          if (d != rank) expect += 4u * static_cast<unsigned>(min(ntiles, d * tpc + tpc) - min(ntiles, d * tpc)) + 4u;
        mbar_expect_tx(xb, expect);
        sh.flt[rank] = sh.fault;
      }
      const int nt = t1 - t0;
      for (int i = tid; i < nt * (n - 1); i += 32) {
        int d = i / nt;
        const int k = i - d * nt;
        if (d >= rank) ++d;
        st_async_cluster(all + t0 + k, static_cast<unsigned>(d), __float_as_uint(all[t0 + k]), xb);
      }
      if (tid < n && tid != rank)
        st_async_cluster(&sh.flt[rank], static_cast<unsigned>(tid), static_cast<uint32_t>(sh.fault), xb);
      if (!mbar_wait_cluster(xb, (x >> 1) & 1)) sh.fault = 1;
    }
    __syncthreads();
    if (tid == 0) {
      int f = sh.fault;
      for (int r = 0; r < n; ++r) f |= sh.flt[r];
      sh.fault = f;
      sh.exchanges = x + 1;
    }
  }
  DF excl;
  return warp_tile_scan(all, ntiles, &excl);
}

__device__ __forceinline__ bool pass_ok(DF z) { return z.hi > 0.f && z.hi < kInf; }

// Inverse-CDF draw from a pass given as tile sums `all` (ntiles, shared
// memory): the first index whose running sum exceeds `target`.  With E_j
// the prefix before tile j (warp_tile_scan's block prefix plus the tile
// sums before j in the block, double-float) and r_j = target - E_j rounded
// to float, the drawn tile is the first tile with mass whose sum exceeds r_j
// (else the last tile with mass), and inside the tile the first element
// whose float running sum exceeds r_j (else its last element with mass).
//
// locate_tile finds the tile (warp 0; every CTA gets the same result) and
// the CTA of the cluster (of n) whose slice holds it; draw_in_tile
// recomputes that tile with the same code as the pass and returns the index
// to all threads.
__device__ void locate_tile(const float* all, int n, int ntiles, DF target, PassSmem& sh) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid < 32) {
    DF e;
    warp_tile_scan(all, ntiles, &e);
    int j0, j1;
    lane_block(ntiles, lane, j0, j1);
    int first = 0x7fffffff, last = -1;
    float rf_first = 0.f, rf_last = 0.f;
    for (int j = j0; j < j1; ++j) {
      const float s = all[j];
      if (s > 0.f) {
        const float rf = df_float(df_add(target, df_neg(e)));
        if (first == 0x7fffffff && s > rf) {
          first = j;
          rf_first = rf;
        }
        last = j;
        rf_last = rf;
      }
      e = df_add_f(e, s);
    }
    const int fmin = __reduce_min_sync(0xffffffffu, first);
    const int lmax = __reduce_max_sync(0xffffffffu, last);
    if (fmin != 0x7fffffff) {
      if (first == fmin) {
        sh.tile = first;
        sh.rf = rf_first;
        sh.last_mode = 0;
        sh.thread = kThreads;
      }
    } else if (lmax >= 0) {
      if (last == lmax) {
        sh.tile = last;
        sh.rf = rf_last;
        sh.last_mode = 1;
        sh.thread = -1;
      }
    } else if (lane == 0) {  // no mass at all (the callers rule this out)
      sh.tile = 0;
      sh.rf = 0.f;
      sh.last_mode = 1;
      sh.thread = -1;
    }
    __syncwarp();
    if (lane == 0) sh.owner = sh.tile / ((ntiles + n - 1) / n);
  }
  __syncthreads();
}

// With `res_t0` >= 0 the drawing CTA's resident slice (first tile res_t0,
// res_nt tiles, laid out as slice_load leaves it) holds the tile, and its
// elements come from shared memory instead of global memory.
template <typename T>
__device__ int draw_in_tile(const PassSpec<T>& S, int V, float c, PassSmem& sh, int res_t0 = -1, int res_nt = 0) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = sh.tile;
  float w[8];
  if (res_t0 >= 0) {
    float xp[8], xq[8];
    const int j = tile - res_t0;
    slice_get8<T>(dyn_smem, j, xp);
    if (S.cq != 0.f) slice_get8<T>(dyn_smem + static_cast<size_t>(res_nt) * kTileElems * sizeof(T), j, xq);
    pass_weights(S, c, xp, xq, w);
  } else {
    tile_weights(S, V, c, tile, w);
  }
  const float mine = sum8(w);
  const float incl_w = warp_incl_scan(mine);
  if (lane == 31) sh.warp_tot[0][0][warp] = incl_w;
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
    for (int k = 0; k < kWarps; ++k) {
      sh.warp_excl[k] = s;
      s = (k == 0) ? sh.warp_tot[0][0][0] : __fadd_rn(s, sh.warp_tot[0][0][k]);
    }
  }
  __syncthreads();
  const float incl = (warp == 0) ? incl_w : __fadd_rn(sh.warp_excl[warp], incl_w);
  sh.thr_incl[tid] = incl;
  const bool last_mode = sh.last_mode;
  const float rf = sh.rf;
  const bool pass_here = mine > 0.f && (last_mode || incl > rf);
  const unsigned bal = __ballot_sync(0xffffffffu, pass_here);
  if (bal != 0 && lane == 0) {
    if (last_mode) atomicMax(&sh.thread, warp * 32 + 31 - __clz(bal));
    else atomicMin(&sh.thread, warp * 32 + __ffs(bal) - 1);
  }
  __syncthreads();
  int t = sh.thread;
  if (t < 0 || t >= kThreads) t = 0;
  if (tid == t) {
    float run = (t == 0) ? 0.f : sh.thr_incl[t - 1];
    int y = -1, lastpos = -1;
    for (int e = 0; e < 8; ++e) {
      run = __fadd_rn(run, w[e]);
      if (w[e] > 0.f) {
        lastpos = e;
        if (!last_mode && y < 0 && run > rf) y = e;
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

// The draw from a cluster pass (the tile sums in sh.all[buf]): every CTA
// locates the tile; the CTA owning its slice, or every CTA when all_ctas is
// set, recomputes the tile and returns the index; the others return -1.
template <typename T>
__device__ int cluster_draw(const PassSpec<T>& S, int V, float c, int ntiles, int buf, DF target,
                            bool all_ctas, PassSmem& sh, bool resident = false) {
  const int n = static_cast<int>(cluster_size()), rank = static_cast<int>(cluster_rank());
  locate_tile(sh.all[buf], n, ntiles, target, sh);
  if (!all_ctas && sh.owner != rank) return -1;
  if (resident && sh.owner == rank) {
    const int tpc = (ntiles + n - 1) / n;
    const int t0 = min(ntiles, rank * tpc), t1 = min(ntiles, t0 + tpc);
    return draw_in_tile(S, V, c, sh, t0, t1 - t0);
  }
  return draw_in_tile(S, V, c, sh);
}

// ---------------------------------------------------------------------------
// row statistics computed by the walk itself (consulted-only mode): each CTA
// of the cluster reduces its slice of a row pair to (max, sum of
// 2^(x c - M)) or, greedy, to (max, first index); the cluster shares the
// partials and merges them in rank order, so every CTA holds the same bits
// ---------------------------------------------------------------------------
// Fold 8 logits into a running (max, sum): the sum is rescaled to the new
// maximum once per 8 elements.  NaN propagates into the maximum and +inf
// makes it infinite, so such a row fails row_stats_ok.
__device__ __forceinline__ void online8(const float* x, float c, float& m, float& s) {
  float cm = x[0];
#pragma unroll
  for (int e = 1; e < 8; ++e) cm = fmax_nan(cm, x[e]);
  const float mn = fmax_nan(m, cm);
  if (mn == -kInf) return;
  const float M = scaled_max(mn, c);
  float acc = (m == -kInf) ? 0.f : __fmul_rn(s, ex2(scaled_max(m, c) - M));
#pragma unroll
  for (int e = 0; e < 8; ++e) acc = __fadd_rn(acc, weight(x[e], c, M));
  s = acc;
  m = mn;
}

// Greedy counterpart: the first index of the maximum (-inf never wins) and
// whether a NaN or +inf was seen.
__device__ __forceinline__ void argmax8(const float* x, int e0, float& best, int& bi, bool& bad) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    bad |= !(x[e] < kInf);
    if (x[e] > best) {
      best = x[e];
      bi = e0 + e;
    }
  }
}

// Block reduction of per-thread (max, sum) of two rows into out[0..1] (all
// threads get the result).
__device__ __forceinline__ void block_ms2(MaxSum a, MaxSum b, float c, PassSmem& sh, MaxSum* out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = ms_warp_reduce(a, c);
  b = ms_warp_reduce(b, c);
  if (lane == 0) {
    sh.red[0][warp][0] = a.m;
    sh.red[0][warp][1] = a.s;
    sh.red[1][warp][0] = b.m;
    sh.red[1][warp][1] = b.s;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    MaxSum t{-kInf, 0.f};
    for (int w = 0; w < kWarps; ++w) t = ms_merge(t, MaxSum{sh.red[r][w][0], sh.red[r][w][1]}, c);
    out[r] = t;
  }
  __syncthreads();
}

// Block argmax (lowest index on ties) of one row; bad if any thread saw a
// NaN or +inf.  out = (value, index), index -1 for a row without a finite
// maximum.
__device__ __forceinline__ ArgMax block_argmax(float best, int bi, bool bad, PassSmem& sh, bool* any_bad) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ArgMax t = am_warp_reduce(ArgMax{best, bi});
  const bool wb = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    sh.red[0][warp][0] = t.v;
    sh.red[0][warp][1] = __int_as_float(t.i);
    sh.red[1][warp][0] = wb ? 1.f : 0.f;
  }
  __syncthreads();
  ArgMax r{-kInf, -1};
  bool b = false;
  for (int w = 0; w < kWarps; ++w) {
    r = am_merge(r, ArgMax{sh.red[0][w][0], __float_as_int(sh.red[0][w][1])});
    b |= sh.red[1][w][0] != 0.f;
  }
  __syncthreads();
  *any_bad = b;
  return r;
}

// This CTA's (max, sum) of tiles [t0, t1) of rows P and Q (Q may be null)
// from its resident slice (slice_load's layout, nt = t1 - t0 tiles).
template <typename T>
__device__ void resident_row_stats(bool with_q, int nt, float c, PassSmem& sh, MaxSum* out) {
  const unsigned char* qbuf = dyn_smem + static_cast<size_t>(nt) * kTileElems * sizeof(T);
  float mp = -kInf, sp = 0.f, mq = -kInf, sq = 0.f;
  for (int j = 0; j < nt; ++j) {
    float x[8];
    slice_get8<T>(dyn_smem, j, x);
    online8(x, c, mp, sp);
    if (with_q) {
      slice_get8<T>(qbuf, j, x);
      online8(x, c, mq, sq);
    }
  }
  block_ms2(MaxSum{mp, sp}, MaxSum{mq, sq}, c, sh, out);
}

// Greedy counterpart over the resident target slice (first tile t0).
template <typename T>
__device__ ArgMax resident_row_argmax(int t0, int nt, PassSmem& sh, bool* bad) {
  float best = -kInf;
  int bi = -1;
  bool b = false;
  for (int j = 0; j < nt; ++j) {
    float x[8];
    slice_get8<T>(dyn_smem, j, x);
    argmax8(x, (t0 + j) * kTileElems + 8 * static_cast<int>(threadIdx.x), best, bi, b);
  }
  return block_argmax(best, bi, b, sh, bad);
}

// This CTA's (max, sum) of tiles [t0, t1) of rows P and Q (Q may be null)
// streamed from global memory through the stage ring (aligned rows) or by
// plain loads (misaligned rows); the same stage counters as the passes.
template <typename T>
__device__ void streamed_row_stats(const T* P, const T* Q, int V, float c, int t0, int t1, PassSmem& sh,
                                   MaxSum* out) {
  constexpr int TPS = kStageRowBytes / (kTileElems * static_cast<int>(sizeof(T)));
  constexpr int R = Load8<T>::kRegs;
  const int tid = threadIdx.x;
  const bool useQ = Q != nullptr;
  float mp = -kInf, sp = 0.f, mq = -kInf, sq = 0.f;
  const bool aligned = row_is_aligned(P) && (!useQ || row_is_aligned(Q));
  if (!aligned) {
    for (int t = t0; t < t1; ++t) {
      float x[8];
      const int e0 = t * kTileElems + 8 * tid;
      load8_misaligned(P, e0, V, x);
      online8(x, c, mp, sp);
      if (useQ) {
        load8_misaligned(Q, e0, V, x);
        online8(x, c, mq, sq);
      }
    }
    block_ms2(MaxSum{mp, sp}, MaxSum{mq, sq}, c, sh, out);
    return;
  }
  const int nst = (t1 - t0 + TPS - 1) / TPS;
  const int g0 = sh.staged;
  const int Vv = vector_end<T>(V);
  auto issue = [&](int k) {  // thread 0
    const int ta = t0 + k * TPS, te = min(t1, ta + TPS);
    const unsigned bytes = static_cast<unsigned>((min(te * kTileElems, Vv) - ta * kTileElems) * sizeof(T));
    const int b = (g0 + k) % kStages;
    unsigned char* buf = dyn_smem + b * 2 * kStageRowBytes;
    mbar_expect_tx(&sh.bar[b], useQ ? 2 * bytes : bytes);
    if (bytes == 0) return;
    bulk_load(buf, P + static_cast<long long>(ta) * kTileElems, bytes, &sh.bar[b]);
    if (useQ) bulk_load(buf + kStageRowBytes, Q + static_cast<long long>(ta) * kTileElems, bytes, &sh.bar[b]);
  };
  __syncthreads();  // earlier users of the stage region are done with it
  if (tid == 0) {
    fence_proxy_async();
    for (int k = 0; k < min(kStages, nst); ++k) issue(k);
  }
  __syncthreads();
  bool fault = false;
  for (int k = 0; k < nst; ++k) {
    const int ta = t0 + k * TPS, nb = min(TPS, t1 - ta);
    const int b = (g0 + k) % kStages;
    const unsigned char* buf = dyn_smem + b * 2 * kStageRowBytes;
    if (!mbar_wait(&sh.bar[b], ((g0 + k) / kStages) & 1)) fault = true;
#pragma unroll
    for (int j = 0; j < TPS; ++j) {
      if (j < nb) {
        float x[8];
        if ((ta + j + 1) * kTileElems <= Vv) {
          uint32_t r[R];
          stage_load8<T>(buf, j, r);
          Load8<T>::get(r, x);
          online8(x, c, mp, sp);
          if (useQ) {
            stage_load8<T>(buf + kStageRowBytes, j, r);
            Load8<T>::get(r, x);
            online8(x, c, mq, sq);
          }
        } else {
          stage_load8_tail<T>(buf, j, P, ta + j, V, x);
          online8(x, c, mp, sp);
          if (useQ) {
            stage_load8_tail<T>(buf + kStageRowBytes, j, Q, ta + j, V, x);
            online8(x, c, mq, sq);
          }
        }
      }
    }
    __syncthreads();  // buffer b is free
    if (tid == 0 && k + kStages < nst) {
      fence_proxy_async();
      issue(k + kStages);
    }
  }
  if (fault) {
    for (int k = max(0, nst - kStages); k < nst; ++k)
      mbar_wait(&sh.bar[(g0 + k) % kStages], ((g0 + k) / kStages) & 1);
    sh.fault = 1;
  }
  if (tid == 0) sh.staged = g0 + nst;
  block_ms2(MaxSum{mp, sp}, MaxSum{mq, sq}, c, sh, out);
}

// Share four floats per CTA across the cluster (asynchronous stores counted
// on the receivers' exchange barriers, like a pass's tile sums).  Returns the
// buffer of sh.xv that holds every CTA's values, indexed by rank.  Every CTA
// of the cluster calls it, in the same sequence of exchanges as its passes.
__device__ __forceinline__ int cluster_share4(float v0, float v1, float v2, float v3, PassSmem& sh) {
  const int tid = threadIdx.x;
  const int rank = static_cast<int>(cluster_rank()), n = static_cast<int>(cluster_size());
  __syncthreads();  // sh.exchanges is current
  const int x = sh.exchanges;
  const int xb_i = x & 1;
  if (tid == 0) {
    sh.xv[xb_i][rank][0] = v0;
    sh.xv[xb_i][rank][1] = v1;
    sh.xv[xb_i][rank][2] = v2;
    sh.xv[xb_i][rank][3] = v3;
  }
  if (n > 1) {
    if (tid < 32) {
      uint64_t* xb = &sh.xbar[xb_i];
      if (tid == 0) {
        mbar_expect_tx(xb, 20u * static_cast<unsigned>(n - 1));
        sh.flt[rank] = sh.fault;
      }
      __syncwarp();
      if (tid < n && tid != rank) {
        const unsigned d = static_cast<unsigned>(tid);
        st_async_cluster(&sh.xv[xb_i][rank][0], d, __float_as_uint(v0), xb);
        st_async_cluster(&sh.xv[xb_i][rank][1], d, __float_as_uint(v1), xb);
        st_async_cluster(&sh.xv[xb_i][rank][2], d, __float_as_uint(v2), xb);
        st_async_cluster(&sh.xv[xb_i][rank][3], d, __float_as_uint(v3), xb);
        st_async_cluster(&sh.flt[rank], d, static_cast<uint32_t>(sh.fault), xb);
      }
      if (!mbar_wait_cluster(xb, (x >> 1) & 1)) sh.fault = 1;
    }
    __syncthreads();
    if (tid == 0) {
      int f = sh.fault;
      for (int r = 0; r < n; ++r) f |= sh.flt[r];
      sh.fault = f;
      sh.exchanges = x + 1;
    }
  }
  __syncthreads();
  return xb_i;
}

// Merge the shared (max, sum) pairs of rows 0 and 1 in rank order.
__device__ __forceinline__ void merge_shared_ms2(int xb_i, float c, PassSmem& sh, MaxSum* out) {
  const int n = static_cast<int>(cluster_size());
  MaxSum a{-kInf, 0.f}, b{-kInf, 0.f};
  for (int r = 0; r < n; ++r) {
    a = ms_merge(a, MaxSum{sh.xv[xb_i][r][0], sh.xv[xb_i][r][1]}, c);
    b = ms_merge(b, MaxSum{sh.xv[xb_i][r][2], sh.xv[xb_i][r][3]}, c);
  }
  out[0] = a;
  out[1] = b;
}

// Merge shared (value, index bits, bad flag) triples in rank order (lowest
// index on ties).
__device__ __forceinline__ ArgMax merge_shared_argmax(int xb_i, const PassSmem& sh, bool* bad) {
  const int n = static_cast<int>(cluster_size());
  ArgMax r{-kInf, -1};
  bool b = false;
  for (int k = 0; k < n; ++k) {
    r = am_merge(r, ArgMax{sh.xv[xb_i][k][0], __float_as_int(sh.xv[xb_i][k][1])});
    b |= sh.xv[xb_i][k][2] != 0.f;
  }
  *bad = b;
  return r;
}

// Greedy: this CTA's argmax of tiles [t0, t1) of row P by plain loads.
template <typename T>
__device__ ArgMax direct_row_argmax(const T* P, int V, int t0, int t1, PassSmem& sh, bool* bad) {
  float best = -kInf;
  int bi = -1;
  bool b = false;
  for (int t = t0; t < t1; ++t) {
    float x[8];
    const int e0 = t * kTileElems + 8 * static_cast<int>(threadIdx.x);
    if (row_is_aligned(P)) {
      uint32_t r[Load8<T>::kRegs];
      Load8<T>::issue(P, e0, V, r);
      Load8<T>::get(r, x);
    } else {
      load8_misaligned(P, e0, V, x);
    }
    argmax8(x, e0, best, bi, b);
  }
  return block_argmax(best, bi, b, sh, bad);
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

// Merge the chunk partials of one statistics row in chunk order (one
// thread; `part` points into shared memory, where the partials were staged).
__device__ __forceinline__ MaxSum combine_row(const float2* part, int chunks, float c) {
  MaxSum acc{-kInf, 0.f};
  for (int k = 0; k < chunks; ++k) {
    const float2 p = part[k];
    acc = ms_merge(acc, MaxSum{p.x, p.y}, c);
  }
  return acc;
}

// Argmax over the chunk partials of one row (one thread); `bad` is set when
// a chunk saw a NaN or +inf.
__device__ __forceinline__ ArgMax combine_row_argmax(const float2* part, int chunks, bool& bad) {
  ArgMax acc{-kInf, -1};
  bad = false;
  for (int k = 0; k < chunks; ++k) {
    const float2 p = part[k];
    if (p.x != p.x) bad = true;
    acc = am_merge(acc, ArgMax{p.x, __float_as_int(p.y)});
  }
  return acc;
}

__device__ __forceinline__ bool row_stats_ok(MaxSum ms) {
  return ms.m > -kInf && ms.m < kInf && ms.s > 0.f && ms.s < kInf;
}

}  // namespace sv
