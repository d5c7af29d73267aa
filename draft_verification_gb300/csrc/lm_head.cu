// Chain verification from the models' final hidden states: the LM head and
// the row statistics in one tensor-core kernel per head, then the chain walk.
//
// Source: "Accelerating LLM Inference with Staged Speculative Decoding"
// (arXiv 2308.04623), abstract: small-batch inference has low arithmetic
// intensity, so the step is bound by the bytes it moves, and the logits the
// verification reads are what the LM head writes just before it.  Folding
// the row statistics into the head's epilogue removes the statistics pass
// over the vocabulary-wide rows.  The rule applied afterwards is the one of
// spec_verify_chain (PipeSpec review, Circularity Check).
//
// lm_head_kernel: logits L = X W^T for one head, X [R, d] (bfloat16 hidden
// states, one row per position), W [V, d] (bfloat16 LM-head weights), float32
// accumulation in tensor memory.  One persistent CTA per SM owns a
// contiguous slab of N-entry vocabulary tiles (N chosen per call).  Per tile
// and per block of at most 512 hidden rows, the CTA streams K in 64-element
// steps:
//   warp 8  (one thread)  TMA copies of the W tile [N x 64] and the X tiles
//                         [128 x 64] of the row block into a ring of stages;
//   warps 9-11 (one thread each)  tcgen05.mma, M = 128 rows, N vocabulary
//                         entries, K = 16, one accumulator of N columns per
//                         row tile (at most 4 tiles within the 512 TMEM
//                         columns); warp 9 + i issues the row tiles t with
//                         t % 3 == i, so three instruction streams feed the
//                         tensor pipe; each issuer's commits free the stages
//                         and hand the tile's accumulators to the epilogue;
//   warps 0-7             the epilogue: thread t of warps w and w + 4 owns
//                         TMEM lane 32 w + t, i.e. one hidden row of every
//                         row tile; warp w takes the first half of the tile's
//                         16-column chunks, warp w + 4 the second half; each
//                         folds its logits into the row's running
//                         (max, sum of 2^(x c - M)) (sampling) or (max, first
//                         index) (greedy), in ascending vocabulary order, and
//                         in sampling mode stores the float32 logits for the
//                         walk's residual or bonus draw.
// At the end of a row block the two halves' states are merged and the CTA
// writes one partial per row in the statistics
// kernel's format, so the chain walk merges them exactly like the partials of
// stored logits.  Greedy calls store no logits at all: the walk needs only
// the argmaxes.
//
// lm_head_pair_kernel (described at its definition): the same product and
// partials on clusters of two CTAs issuing cta_group::2 products over
// 256-entry vocabulary tiles, which halves each CTA's tensor-pipe operand
// reads.  The host picks it when the target head has at least 256 rows and
// its tiles balance better over the pairs than the single-CTA tiles over the
// SMs; both heads of a call then use it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "spec_verify.h"
#include "tc.cuh"

namespace sv {
namespace {

constexpr int kBK = 64;            // K elements per stage: one 128-byte swizzled row
constexpr int kBR = 128;           // hidden rows per row tile (MMA M)
constexpr int kMaxRowTiles = 4;    // 4 accumulators of 128 float32 columns: all of TMEM
constexpr int kRowBlock = kBR * kMaxRowTiles;
constexpr int kTileBytes = kBR * kBK * 2;  // 16 KB: one hidden-state tile
constexpr int kMaxStages = 6;
constexpr int kSmemBudget = 208 * 1024;
constexpr int kEpiWarps = 8;       // two epilogue warps per TMEM lane quarter, each half of a tile's columns
constexpr int kProdWarp = kEpiWarps;
constexpr int kIssuer0 = kEpiWarps + 1;
constexpr int kLmThreads = 32 * (kEpiWarps + 4);
constexpr int kIssuers = 3;        // MMA-issuing warps (9, 10, 11): one thread's issue rate was the limit
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxChunks = 256;    // partial columns per row (persistent CTAs)
constexpr int kPrefetchSteps = 8;  // shallow rings: weight tiles brought into L2 this many K steps ahead

struct LmParams {
  int R, V, d;
  int bv;             // vocabulary entries per tile (MMA N): a multiple of 16, 64..256
  int ntv;            // vocabulary tiles
  int nkb;            // K steps of 64
  int rt_max;         // row tiles of the largest row block
  int stages;
  int prefetch;       // K steps of weight tiles requested into L2 ahead of the ring (0: none)
  int per;            // hidden rows per sequence of this head
  int rows_seq;       // statistics rows per sequence
  int row_off;        // this head's first statistics row
  int chunks;         // CTAs of the launch
  int greedy;
  float c;            // log2(e) / T (sampling)
  float2* partials;   // [B][rows_seq][chunks]
  float* logits;      // [R][ldl] (sampling) or null
  long long ldl;
  int* error_word;    // optional: SPEC_ERR_INTERNAL when a wait gives up
};

// 8 floats to global memory in one 32-byte store (dst 32-byte aligned): a
// whole sector per store, so the rows' scattered writes need no merging
__device__ __forceinline__ void st_global_v8(float* dst, const float* v) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "f"(v[0]), "f"(v[1]),
               "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}

// Test hook (spec_test_inject_head_copy_timeout): nonzero makes every stage
// of both head kernels expect 16 bytes that never come (on the even CTA's
// barrier for a pair), so that the MMA issuers' bounded waits give up.  Zero
// in normal operation.
__device__ int g_lm_copy_timeout_test = 0;

__device__ __forceinline__ bool lm_wait(uint64_t* bar, unsigned parity, volatile int* fault) {
  for (int i = 0; i < kMaxPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*fault) return false;
  }
  *fault = 1;
  return false;
}

__global__ void __launch_bounds__(kLmThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                   const LmParams P) {
  extern __shared__ __align__(1024) unsigned char lm_dyn[];
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages], tfull, tempty, drain;
  __shared__ uint32_t tmem_s;
  __shared__ int fault_s;
  __shared__ int issued_s;  // stages the producer issued
  __shared__ float2 xch[kMaxRowTiles][kBR];          // second-half epilogue states, handed over per row block
  __shared__ unsigned char xbad[kMaxRowTiles][kBR];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* ring = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(lm_dyn) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  const int wbytes = P.bv * kBK * 2;  // a weight tile
  const int stage_bytes = wbytes + kTileBytes * P.rt_max;
  const int G = P.chunks, cta = blockIdx.x;
  const int v_t0 = static_cast<int>((static_cast<long long>(cta) * P.ntv) / G);
  const int v_t1 = static_cast<int>((static_cast<long long>(cta + 1) * P.ntv) / G);
  const int nrb = (P.R + kRowBlock - 1) / kRowBlock;
  volatile int* fault = &fault_s;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kIssuers);
    }
    mbar_init(&tfull, kIssuers);
    mbar_init(&tempty, kEpiWarps);
    mbar_init(&drain, kIssuers);
    fault_s = 0;
    issued_s = 0;
    mbar_fence_init();
  }
  if (warp == kIssuer0) {
    tmem_alloc(&tmem_s, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_s;

  if (warp == kProdWarp) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_w);
      const unsigned extra_tx = g_lm_copy_timeout_test ? 16u : 0u;
      int it = 0;
      const int slab_steps = (v_t1 - v_t0) * P.nkb;
      for (int rb = 0; rb < nrb && !*fault; ++rb) {
        const int rows = min(kRowBlock, P.R - rb * kRowBlock);
        const int rt = (rows + kBR - 1) / kBR;
        // a ring of two stages does not cover the weights' HBM latency: then
        // the first weight tiles are requested into L2 now and every later
        // one P.prefetch K steps before its copy
        for (int j = 0; j < min(P.prefetch, slab_steps); ++j)
          tma_prefetch_l2_2d(&tm_w, (j % P.nkb) * kBK, (v_t0 + j / P.nkb) * P.bv);
        for (int vt = v_t0; vt < v_t1 && !*fault; ++vt) {
          for (int kb = 0; kb < P.nkb; ++kb, ++it) {
            const int j = (vt - v_t0) * P.nkb + kb + P.prefetch;
            if (P.prefetch > 0 && j < slab_steps)
              tma_prefetch_l2_2d(&tm_w, (j % P.nkb) * kBK, (v_t0 + j / P.nkb) * P.bv);
            const int s = it % P.stages;
            const unsigned ph = static_cast<unsigned>(it / P.stages) & 1u;
            if (!lm_wait(&empty[s], ph ^ 1u, fault)) break;
            unsigned char* st = ring + static_cast<size_t>(s) * stage_bytes;
            mbar_expect_tx(&full[s], static_cast<unsigned>(wbytes + kTileBytes * rt) + extra_tx);
            tma_load_2d(st, &tm_w, kb * kBK, vt * P.bv, &full[s]);
            for (int t = 0; t < rt; ++t)
              tma_load_2d(st + wbytes + kTileBytes * t, &tm_x, kb * kBK, rb * kRowBlock + t * kBR, &full[s]);
            issued_s = it + 1;
          }
        }
      }
    }
  } else if (warp >= kIssuer0 && warp < kIssuer0 + kIssuers) {
    // ---------------- MMA issuers: row tiles t with t % kIssuers == warp - kIssuer0 ----------------
    const int me = warp - kIssuer0;
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16_f32(kBR, P.bv);
      int it = 0, acc = 0;
      for (int rb = 0; rb < nrb && !*fault; ++rb) {
        const int rows = min(kRowBlock, P.R - rb * kRowBlock);
        const int rt = (rows + kBR - 1) / kBR;
        for (int vt = v_t0; vt < v_t1 && !*fault; ++vt, ++acc) {
          if (!lm_wait(&tempty, (static_cast<unsigned>(acc) & 1u) ^ 1u, fault)) break;
          tc_fence_after();
          for (int kb = 0; kb < P.nkb; ++kb, ++it) {
            const int s = it % P.stages;
            const unsigned ph = static_cast<unsigned>(it / P.stages) & 1u;
            if (!lm_wait(&full[s], ph, fault)) break;
            tc_fence_after();
            const uint32_t st = smem_addr(ring + static_cast<size_t>(s) * stage_bytes);
            // descriptors of the stage's tiles, built once: a K step of 16
            // elements adds 32 bytes (2 in the start-address field), a row
            // tile 16 KB (1024)
            const uint64_t dw = umma_desc_sw128(st);
            const uint64_t dx = umma_desc_sw128(st + wbytes);
#pragma unroll
            for (int t = 0; t < kMaxRowTiles; ++t) {
              if (t < rt && t % kIssuers == me) {
                const uint64_t dxt = dx + static_cast<uint64_t>(t * (kTileBytes >> 4));
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                  umma_bf16(tmem + static_cast<uint32_t>(t * P.bv), dxt + 2u * k, dw + 2u * k, idesc, kb > 0 || k > 0);
              }
            }
            umma_commit(&empty[s]);  // the stage is free once these MMAs are done
          }
          if (*fault) break;
          umma_commit(&tfull);  // the tile's accumulators are complete
        }
      }
      // every MMA issued has completed before TMEM is released
      umma_commit(&drain);
      mbar_wait(&drain, 0);
    }
  } else {
    // ---------------- epilogue (warps 0-3) ----------------
    const float c = P.c;
    int acc = 0;
    for (int rb = 0; rb < nrb; ++rb) {
      const int rows = min(kRowBlock, P.R - rb * kRowBlock);
      const int rt = (rows + kBR - 1) / kBR;
      float m[kMaxRowTiles], s[kMaxRowTiles];
      int bi[kMaxRowTiles];
      bool bad[kMaxRowTiles];
#pragma unroll
      for (int t = 0; t < kMaxRowTiles; ++t) {
        m[t] = -kInf;
        s[t] = 0.f;
        bi[t] = -1;
        bad[t] = false;
      }
      const int q = warp & 3, h = warp >> 2;  // TMEM lane quarter, column half
      const int nch16 = P.bv / 16;
      const int c_lo = h ? (nch16 + 1) / 2 : 0, c_hi = h ? nch16 : (nch16 + 1) / 2;
      for (int vt = v_t0; vt < v_t1; ++vt, ++acc) {
        // the warp decides together: the TMEM loads below are warp-wide
        const bool ready = __all_sync(0xffffffffu, lm_wait(&tfull, static_cast<unsigned>(acc) & 1u, fault));
        if (!ready) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < kMaxRowTiles; ++t) {
          if (t >= rt) break;
          const int row = rb * kRowBlock + t * kBR + q * 32 + lane;
          float* dst = (P.logits && row < P.R) ? P.logits + static_cast<long long>(row) * P.ldl : nullptr;
#pragma unroll 1
          for (int cc = c_lo; cc < c_hi; ++cc) {
            float v[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(t * P.bv + cc * 16),
                      v);
            const int v0 = vt * P.bv + cc * 16;
            if (v0 >= P.V) break;  // past the vocabulary in its last, partial tile
            const int nv = min(16, P.V - v0);
            if (P.greedy) {
              // the chunk's maximum, NaN-propagating in two independent
              // halves: a NaN or +inf anywhere marks the row bad (its
              // argmax is then not used); otherwise a chunk maximum strictly
              // above the running one moves the argmax to its first index, so
              // ties keep the lowest index and -inf never wins (a row of -inf
              // has no argmax)
              float ca = -kInf, cb = -kInf;
#pragma unroll
              for (int j = 0; j < 16; j += 2) {
                if (j < nv) ca = fmax_nan(ca, v[j]);
                if (j + 1 < nv) cb = fmax_nan(cb, v[j + 1]);
              }
              const float cm = fmax_nan(ca, cb);
              bad[t] |= !(cm < kInf);
              if (cm > m[t] && cm < kInf) {
                int first = 0;
#pragma unroll
                for (int j = 15; j >= 0; --j)
                  if (j < nv && v[j] == cm) first = j;
                m[t] = cm;
                bi[t] = v0 + first;
              }
            } else {
              // two independent chains (even and odd entries) halve the
              // dependent latency of the max and of the sum
              float ca = -kInf, cb = -kInf;
#pragma unroll
              for (int j = 0; j < 16; j += 2) {
                if (j < nv) ca = fmax_nan(ca, v[j]);
                if (j + 1 < nv) cb = fmax_nan(cb, v[j + 1]);
              }
              const float mn = fmax_nan(m[t], fmax_nan(ca, cb));
              if (mn != -kInf) {
                const float Mn = scaled_max(mn, c);
                const float scale = (m[t] == -kInf) ? 0.f : ex2(scaled_max(m[t], c) - Mn);
                float sa = 0.f, sb = 0.f;
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                  if (j < nv) sa = __fadd_rn(sa, weight(v[j], c, Mn));
                  if (j + 1 < nv) sb = __fadd_rn(sb, weight(v[j + 1], c, Mn));
                }
                s[t] = __fadd_rn(__fmul_rn(s[t], scale), __fadd_rn(sa, sb));
                m[t] = mn;
              }
              if (dst) {
                if (nv == 16) {
                  st_global_v8(dst + v0, v);
                  st_global_v8(dst + v0 + 8, v + 8);
                } else {
#pragma unroll
                  for (int j = 0; j < 16; ++j)
                    if (j < nv) dst[v0 + j] = v[j];
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty);
      }
      // the second half's warps hand their state to the first half's, which
      // merge it (larger maximum wins, ties to the lower index) and write one
      // partial per row of the block for this CTA's slab
      if (h) {
#pragma unroll
        for (int t = 0; t < kMaxRowTiles; ++t) {
          if (t >= rt) break;
          xch[t][q * 32 + lane] = P.greedy ? make_float2(m[t], __int_as_float(bi[t])) : make_float2(m[t], s[t]);
          xbad[t][q * 32 + lane] = bad[t] ? 1 : 0;
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
      if (!h) {
#pragma unroll
        for (int t = 0; t < kMaxRowTiles; ++t) {
          if (t >= rt) break;
          const int row = rb * kRowBlock + t * kBR + q * 32 + lane;
          if (row >= P.R) continue;
          const long long prow = static_cast<long long>(row / P.per) * P.rows_seq + P.row_off + row % P.per;
          const float2 o = xch[t][q * 32 + lane];
          float2 out;
          if (P.greedy) {
            const int oi = __float_as_int(o.y);
            if (oi >= 0 && (bi[t] < 0 || o.x > m[t] || (o.x == m[t] && oi < bi[t]))) {
              m[t] = o.x;
              bi[t] = oi;
            }
            const bool b = bad[t] || xbad[t][q * 32 + lane];
            out = make_float2(b ? __int_as_float(0x7fc00000) : m[t], __int_as_float(bi[t]));
          } else {
            const MaxSum ms = ms_merge(MaxSum{m[t], s[t]}, MaxSum{o.x, o.y}, c);
            out = make_float2(ms.m, ms.s);
          }
          if (*fault) out = make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
          P.partials[prow * P.chunks + cta] = out;
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
    }
  }

  __syncthreads();
  if (*fault && threadIdx.x == 0) {
    // copies still in flight land before the CTA exits: wait (bounded) for
    // the last phase of every stage the producer issued
    const int issued = issued_s;
    for (int k = max(0, issued - P.stages); k < issued; ++k)
      mbar_wait(&full[k % P.stages], static_cast<unsigned>(k / P.stages) & 1u);
    if (P.error_word) atomicOr(P.error_word, SPEC_ERR_INTERNAL);
  }
  __syncthreads();
  if (warp == kIssuer0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// lm_head_pair_kernel: the same product and partials on CTA pairs.  A
// cluster of two CTAs owns a slab of 256-entry vocabulary tiles; per tile,
// row block and 64-element K step the pair issues M = 256 products with the
// weights as A (the even CTA holds vocabulary rows 0-127 of the tile, the
// odd CTA rows 128-255) and the hidden rows as B, in one or two chunks of
// Nc <= 256 rows (the even CTA holds the first Nc/2 rows of each chunk, the
// odd CTA the rest).  Each CTA therefore copies 16 KB of weights and half of
// the hidden rows per stage, and its tensor pipe reads half of B.  Warps 17
// and 18 of the even CTA each issue one chunk's products.  The accumulators
// land with one vocabulary entry per TMEM lane and one hidden row per
// column; the epilogue (warps 0-15 of each CTA, four per TMEM lane quarter)
// transposes each 32-entry x 16-row block through shared memory, so that
// lanes l and l + 16 hold 16 entries each of one row, fold them and combine
// by one shuffle into the quarter's running state of the row; at the end of
// a row block the four quarters' states are merged into one partial per row
// and CTA.
// ---------------------------------------------------------------------------
constexpr int kPairM = 256;              // vocabulary entries per pair tile
constexpr int kPairMaxRows = 512;        // hidden rows per row block (TMEM columns)
constexpr int kPairRing = 188 * 1024;    // ring budget per CTA
constexpr int kPairMaxStages = 12;
// CTA pairs only for calls whose target head has at least this many rows
// (the products dominate; smaller calls stream the weights faster on single
// CTAs: B = 4 and 16 at V = 128256 15-20 %), and only when the pairs' coarser
// 256-entry tiles do not balance worse than the single-CTA tiles (below)
constexpr int kPairMinRows = 256;
constexpr int kPairWBytes = 128 * kBK * 2;  // a CTA's weight tile: 16 KB
constexpr int kPairIssuers = 2;          // warps 17 and 18 of the even CTA: one chunk each
constexpr int kPairEpi = 16;             // epilogue warps: four per TMEM lane quarter
constexpr int kPairProd = kPairEpi;      // the TMA producer warp
constexpr int kPairIss0 = kPairEpi + 1;  // the first MMA-issuing warp
constexpr int kPairThreads = 32 * (kPairEpi + 1 + kPairIssuers);
constexpr int kPairScrLd = 36;           // floats per row of a warp's transpose block (32 entries, padded)
constexpr int kPairScr = 16 * kPairScrLd;  // floats of one warp's transpose block (16 rows x 32 entries)
constexpr int kPairExtra = kPairEpi * kPairScr * 4;  // the epilogue warps' transpose blocks
// a row block's quarter states and bad-row flags reuse the transpose blocks
static_assert(4 * kPairMaxRows * 8 + 4 * kPairMaxRows <= kPairExtra, "quarter states fit the transpose blocks");

struct LmPairParams {
  int R, V, d, nkb;
  int nc;             // hidden rows per chunk (MMA N): a multiple of 16, <= 256
  int nch;            // chunks per full row block (1 or 2)
  int ntv;            // 256-entry vocabulary tiles
  int stages;
  int per, rows_seq, row_off;
  int chunks;         // CTAs of the launch: one partial column each
  int greedy;
  float c;
  float2* partials;
  float* logits;
  long long ldl;
  int* error_word;
};

// Folds of one lane's 16 consecutive logits of a row, of which the first nl
// are inside the vocabulary; kFull: all 16 are (no per-entry tests).
// NaN-propagating maximum, in two independent chains.
template <bool kFull>
__device__ __forceinline__ float max16(const float* y, int nl) {
  float ca = -kInf, cb = -kInf;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    if (kFull || i < nl) ca = fmax_nan(ca, y[i]);
    if (kFull || i + 1 < nl) cb = fmax_nan(cb, y[i + 1]);
  }
  return fmax_nan(ca, cb);
}
// Sum of 2^(y c - Mn), in two independent chains.
template <bool kFull>
__device__ __forceinline__ float sum16(const float* y, int nl, float c, float Mn) {
  float sa = 0.f, sb = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    if (kFull || i < nl) sa = __fadd_rn(sa, weight(y[i], c, Mn));
    if (kFull || i + 1 < nl) sb = __fadd_rn(sb, weight(y[i + 1], c, Mn));
  }
  return __fadd_rn(sa, sb);
}
// The first i with y[i] == m, or 16.
template <bool kFull>
__device__ __forceinline__ int first16(const float* y, int nl, float m) {
  int f = 16;
#pragma unroll
  for (int i = 15; i >= 0; --i)
    if ((kFull || i < nl) && y[i] == m) f = i;
  return f;
}

// Bounded wait with acquire semantics at cluster scope (arrivals come from
// the peer CTA).
__device__ __forceinline__ bool lm_wait_cluster(uint64_t* bar, unsigned parity, volatile int* fault) {
  for (int i = 0; i < kMaxPolls; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "n"(kPollNs)
        : "memory");
    if (ok) return true;
    if (*fault) return false;
  }
  *fault = 1;
  return false;
}

__global__ void __launch_bounds__(kPairThreads, 1)
    lm_head_pair_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                        const LmPairParams P) {
  extern __shared__ __align__(1024) unsigned char lp_dyn[];
  __shared__ uint64_t full[kPairMaxStages], empty[kPairMaxStages], tfull, tempty, drain;
  __shared__ uint32_t tmem_s;
  __shared__ int fault_s;
  __shared__ int issued_s;       // stages this CTA's producer issued
  __shared__ int peer_issued_s;  // (even CTA) stages the odd CTA's producer issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_rank());
  const bool lead = rank == 0;
  unsigned char* ring = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(lp_dyn) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  const int xhalf = P.nc / 2 * kBK * 2;  // one CTA's half of a chunk of hidden rows, one K step
  const int stage_bytes = kPairWBytes + P.nch * xhalf;
  float* scratch = reinterpret_cast<float*>(ring + static_cast<size_t>(P.stages) * stage_bytes);
  // at the end of a row block, once every epilogue warp is past its
  // transposes, the same bytes hold the quarter states and bad-row flags
  float2* state = reinterpret_cast<float2*>(scratch);
  unsigned char* sbad = reinterpret_cast<unsigned char*>(state + 4 * kPairMaxRows);
  const int pairs = static_cast<int>(gridDim.x) / 2, pair = static_cast<int>(blockIdx.x) / 2;
  const int v_t0 = static_cast<int>((static_cast<long long>(pair) * P.ntv) / pairs);
  const int v_t1 = static_cast<int>((static_cast<long long>(pair + 1) * P.ntv) / pairs);
  const int rbrows = P.nc * P.nch;
  const int nrb = (P.R + rbrows - 1) / rbrows;
  volatile int* fault = &fault_s;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kPairIssuers);
    }
    mbar_init(&tfull, kPairIssuers);
    mbar_init(&tempty, 2 * kPairEpi);  // the epilogue warps of both CTAs of the pair
    mbar_init(&drain, kPairIssuers);
    fault_s = 0;
    issued_s = 0;
    peer_issued_s = 0;
    mbar_fence_init();
  }
  if (warp == kPairIss0) {
    tmem_alloc_pair(&tmem_s, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_arrive();  // both CTAs' barriers are initialised before either signals the other's
  cluster_wait();
  tc_fence_after();
  const uint32_t tmem = tmem_s;

  if (warp == kPairProd) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_w);
      const unsigned extra_tx = g_lm_copy_timeout_test ? 16u : 0u;
      int it = 0;
      for (int rb = 0; rb < nrb && !*fault; ++rb) {
        const int rows = min(rbrows, P.R - rb * rbrows);
        const int nch = (rows + P.nc - 1) / P.nc;
        for (int vt = v_t0; vt < v_t1 && !*fault; ++vt) {
          for (int kb = 0; kb < P.nkb; ++kb, ++it) {
            const int s = it % P.stages;
            const unsigned ph = static_cast<unsigned>(it / P.stages) & 1u;
            if (!lm_wait(&empty[s], ph ^ 1u, fault)) break;
            unsigned char* st = ring + static_cast<size_t>(s) * stage_bytes;
            const uint32_t fb = cluster_addr(&full[s], 0);
            // the even CTA's barrier counts both CTAs' bytes
            if (lead) mbar_expect_tx(&full[s], 2u * static_cast<unsigned>(kPairWBytes + nch * xhalf) + extra_tx);
            tma_load_2d_pair(st, &tm_w, kb * kBK, vt * kPairM + rank * 128, fb);
            for (int j = 0; j < nch; ++j)
              tma_load_2d_pair(st + kPairWBytes + j * xhalf, &tm_x, kb * kBK, rb * rbrows + j * P.nc + rank * (P.nc / 2),
                               fb);
            issued_s = it + 1;
          }
        }
      }
    }
  } else if (warp >= kPairIss0) {
    // ---------------- MMA issuers (even CTA): chunk j = warp - kPairIss0 ----------------
    const int j = warp - kPairIss0;
    if (lead && lane == 0) {
      const uint32_t idesc = umma_idesc_bf16_f32(kPairM, P.nc);
      int it = 0, acc = 0;
      for (int rb = 0; rb < nrb && !*fault; ++rb) {
        const int rows = min(rbrows, P.R - rb * rbrows);
        const bool mine = j < (rows + P.nc - 1) / P.nc;
        for (int vt = v_t0; vt < v_t1 && !*fault; ++vt, ++acc) {
          // both CTAs' epilogues have read the previous tile's accumulators
          if (!lm_wait_cluster(&tempty, (static_cast<unsigned>(acc) & 1u) ^ 1u, fault)) break;
          tc_fence_after();
          for (int kb = 0; kb < P.nkb; ++kb, ++it) {
            const int s = it % P.stages;
            const unsigned ph = static_cast<unsigned>(it / P.stages) & 1u;
            if (!lm_wait(&full[s], ph, fault)) break;
            tc_fence_after();
            if (mine) {
              // descriptors built once per stage: a K step adds 2 to the
              // start-address field
              const uint32_t st = smem_addr(ring + static_cast<size_t>(s) * stage_bytes);
              const uint64_t dw = umma_desc_sw128(st);
              const uint64_t dx = umma_desc_sw128(st + kPairWBytes + j * xhalf);
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                umma_bf16_pair(tmem + static_cast<uint32_t>(j * P.nc), dw + 2u * k, dx + 2u * k, idesc,
                               kb > 0 || k > 0);
            }
            umma_commit_pair(&empty[s], 3);  // the stage is free in both CTAs once these products are done
          }
          if (*fault) break;
          umma_commit_pair(&tfull, 3);  // the tile's accumulators are complete in both CTAs
        }
      }
      umma_commit_pair(&drain, 3);
    }
    if (lane == 0) mbar_wait(&drain, 0);  // no product of the pair still reads or writes this CTA's memory
  } else {
    // ---------------- epilogue (warps 0-15, both CTAs) ----------------
    // warps q, q + 4, q + 8 and q + 12 read TMEM lane quarter q; warp
    // q + 4h takes the 32-row groups g with g % 4 == h
    const float c = P.c;
    const int q = warp & 3, h = warp >> 2;
    constexpr int kPerQ = kPairEpi / 4;
    constexpr int kGrpW = kPairMaxRows / 32 / kPerQ;  // 32-row groups per warp and row block, at most
    float2* my = state + q * kPairMaxRows;  // the quarter's state of every row of the block, at its end
    unsigned char* mybad = sbad + q * kPairMaxRows;
    float* scr = scratch + warp * kPairScr;
    const int rr = lane & 15, eh = lane >> 4;  // after the transpose: row rr of a half group, entries 16 eh ..
    int acc = 0;
    for (int rb = 0; rb < nrb; ++rb) {
      const int rows = min(rbrows, P.R - rb * rbrows);
      const int ngrp = (rows + 31) / 32;
      // the running states of this lane's rows (group h + kPerQ k, half hh,
      // row rr), the same bits in lanes l and l ^ 16; bit 2k + hh of bad
      // marks a row that saw a NaN or +inf
      float2 st[kGrpW][2];
      unsigned bad = 0;
#pragma unroll
      for (int k = 0; k < kGrpW; ++k)
        st[k][0] = st[k][1] = P.greedy ? make_float2(-kInf, __int_as_float(-1)) : make_float2(-kInf, 0.f);
      for (int vt = v_t0; vt < v_t1; ++vt, ++acc) {
        // the warp decides together: the TMEM loads below are warp-wide
        const bool ready = __all_sync(0xffffffffu, lm_wait(&tfull, static_cast<unsigned>(acc) & 1u, fault));
        if (!ready) break;
        tc_fence_after();
        const int vw = vt * kPairM + rank * 128 + q * 32;  // the quarter's first vocabulary entry
        const int nv = max(0, min(32, P.V - vw));            // of its 32 entries, those below V
        const int e0 = eh * 16;                              // this lane's first entry after the transpose
        const int nl = max(0, min(16, nv - e0));             // of its 16 entries, those below V
#pragma unroll
        for (int k = 0; k < kGrpW; ++k) {
          const int g = h + kPerQ * k;
          if (g >= ngrp) break;
          float x[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(g * 32), x);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            // transpose the quarter's 32 entries x 16 rows: lane l writes
            // its entry of every row, then reads entries e0 .. e0 + 15 of
            // row rr of the half group (four 16-byte loads; the padded rows
            // keep both sides free of bank conflicts)
#pragma unroll
            for (int j = 0; j < 16; ++j) scr[j * kPairScrLd + lane] = x[hh * 16 + j];
            __syncwarp();
            float y[16];
#pragma unroll
            for (int f = 0; f < 4; ++f) {
              const float4 v = *reinterpret_cast<const float4*>(scr + rr * kPairScrLd + e0 + 4 * f);
              y[4 * f] = v.x;
              y[4 * f + 1] = v.y;
              y[4 * f + 2] = v.z;
              y[4 * f + 3] = v.w;
            }
            __syncwarp();
            const int row = rb * rbrows + g * 32 + hh * 16 + rr;  // the lane's hidden row
            if (P.logits && row < P.R) {
              // 16 consecutive float32 logits: whole 32-byte sectors
              float* dst = P.logits + static_cast<long long>(row) * P.ldl + vw + e0;
              if (nl == 16) {
                st_global_v8(dst, y);
                st_global_v8(dst + 8, y + 8);
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  if (i < nl) dst[i] = y[i];
              }
            }
            const float2 cur = st[k][hh];
            // the row's maximum over its 32 entries, NaN-propagating: each
            // lane's 16, then the lane pair (l, l ^ 16)
            float cm = nl == 16 ? max16<true>(y, nl) : max16<false>(y, nl);
            cm = fmax_nan(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
            if (P.greedy) {
              // NaN or +inf marks the row bad; a maximum strictly above the
              // running one moves the argmax to its first entry (ties keep
              // the lowest index)
              if (!(cm < kInf)) bad |= 1u << (2 * k + hh);
              const bool up = cm > cur.x && cm < kInf;
              int first = 32;
              if (up) {
                const int f = nl == 16 ? first16<true>(y, nl, cm) : first16<false>(y, nl, cm);
                if (f < 16) first = e0 + f;
              }
              first = min(first, __shfl_xor_sync(0xffffffffu, first, 16));
              if (up) st[k][hh] = make_float2(cm, __int_as_float(vw + first));
            } else {
              const float mn = fmax_nan(cur.x, cm);
              const float Mn = (mn == -kInf) ? 0.f : scaled_max(mn, c);
              float sp = nl == 16 ? sum16<true>(y, nl, c, Mn) : sum16<false>(y, nl, c, Mn);
              sp = __fadd_rn(sp, __shfl_xor_sync(0xffffffffu, sp, 16));  // the same bits in both lanes
              if (mn != -kInf) {
                const float scale = (cur.x == -kInf) ? 0.f : ex2(scaled_max(cur.x, c) - Mn);
                st[k][hh] = make_float2(mn, __fadd_rn(__fmul_rn(cur.y, scale), sp));
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (lead) mbar_arrive(&tempty);
          else mbar_arrive_remote(cluster_addr(&tempty, 0));
        }
      }
      // this warp's rows into the quarter's states (lanes 0-15 of the pairs),
      // which overlay the transpose blocks: every warp is past its last
      // transpose of the block first
      asm volatile("bar.sync 1, %0;" ::"n"(kPairEpi * 32) : "memory");
      if (eh == 0) {
#pragma unroll
        for (int k = 0; k < kGrpW; ++k) {
          const int g = h + kPerQ * k;
          if (g >= ngrp) break;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            my[g * 32 + hh * 16 + rr] = st[k][hh];
            mybad[g * 32 + hh * 16 + rr] = (bad >> (2 * k + hh)) & 1u;
          }
        }
      }
      // merge the four quarters' states of each row, in quarter order, into this
      // CTA's partial (one column per CTA of the launch)
      asm volatile("bar.sync 1, %0;" ::"n"(kPairEpi * 32) : "memory");
      for (int r = static_cast<int>(threadIdx.x); r < rows; r += kPairEpi * 32) {
        const int row = rb * rbrows + r;
        const long long prow = static_cast<long long>(row / P.per) * P.rows_seq + P.row_off + row % P.per;
        float2 out;
        if (P.greedy) {
          ArgMax m2{-kInf, -1};
          bool rbad = false;
          for (int w = 0; w < 4; ++w) {
            const float2 sw = state[w * kPairMaxRows + r];
            m2 = am_merge(m2, ArgMax{sw.x, __float_as_int(sw.y)});
            rbad |= sbad[w * kPairMaxRows + r] != 0;
          }
          out = make_float2(rbad ? __int_as_float(0x7fc00000) : m2.v, __int_as_float(m2.i));
        } else {
          MaxSum m2{-kInf, 0.f};
          for (int w = 0; w < 4; ++w) {
            const float2 sw = state[w * kPairMaxRows + r];
            m2 = ms_merge(m2, MaxSum{sw.x, sw.y}, c);
          }
          out = make_float2(m2.m, m2.s);
        }
        if (*fault) out = make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
        P.partials[prow * P.chunks + blockIdx.x] = out;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kPairEpi * 32) : "memory");
    }
  }

  __syncthreads();
  if (!lead && threadIdx.x == 0) {
    // tell the even CTA how many stages this CTA's producer issued: their
    // copies count on its barriers
    const uint32_t dst = cluster_addr(&peer_issued_s, 0);
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(dst), "r"(issued_s) : "memory");
  }
  cluster_arrive();
  cluster_wait();
  if (*fault && lead && threadIdx.x == 0) {
    // copies still in flight (this CTA's or the odd CTA's) land before
    // either CTA exits: wait (bounded) for the last phase of every stage
    const int issued = max(issued_s, peer_issued_s);
    for (int k = max(0, issued - P.stages); k < issued; ++k)
      mbar_wait(&full[k % P.stages], static_cast<unsigned>(k / P.stages) & 1u);
  }
  if (*fault && threadIdx.x == 0 && P.error_word) atomicOr(P.error_word, SPEC_ERR_INTERNAL);
  __syncthreads();
  cluster_arrive();  // neither CTA leaves while the other may still signal or read it
  cluster_wait();
  if (warp == kPairIss0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// Tensor map of a row-major bfloat16 matrix [rows, cols] (cols contiguous,
// row stride cols elements): boxes of box_rows rows x 64 columns, 128-byte
// swizzle, out-of-range elements read as zero.
bool make_map(CUtensorMap* map, const void* base, long long rows, int cols, int box_rows) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {kBK, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cache[dev] = n;
  return n;
}

// The kernel's dynamic shared memory limit, raised once per device.
cudaError_t smem_attribute() {
  static std::mutex mu;
  static std::map<int, bool> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count(dev)) return cudaSuccess;
  e = cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget + 1024);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

// Partial columns the workspace is sized for: two per 256-entry tile (a CTA
// pair's; at least one per 128-entry tile) and at most kMaxChunks.
int lm_chunks(int V) {
  const int n = 2 * ((V + kPairM - 1) / kPairM);
  return n < kMaxChunks ? n : kMaxChunks;
}

// Row tiles of the largest row block of a head with R rows.
int row_tiles(long long R) {
  const long long t = (R + kBR - 1) / kBR;
  return static_cast<int>(t < kMaxRowTiles ? t : kMaxRowTiles);
}

// The vocabulary tile N (MMA N, a multiple of 16).  Its accumulators for
// all row tiles must fit in the 512 TMEM columns.  The busiest CTA works
// through ceil(ceil(V / N) / G) tiles and copies N * 128 + rt * 16384 bytes
// per tile and K step (a weight tile and the hidden-state tiles), so N is the
// width, from 64 up to that limit, that minimises the busiest CTA's bytes
// (ties: the wider).  Wider tiles feed more products per hidden-state byte;
// narrower ones can balance the tiles over the CTAs better.
int vocab_tile(int rt, int V, int G) {
  const int most = min(256, 512 / rt / 16 * 16);
  int best = most;
  long long best_bytes = -1;
  for (int n = most; n >= 64; n -= 16) {
    const long long tiles = (V + n - 1) / n;
    const long long bytes = (tiles + G - 1) / G * (static_cast<long long>(n) * kBK * 2 + rt * kTileBytes);
    if (best_bytes < 0 || bytes < best_bytes) {
      best_bytes = bytes;
      best = n;
    }
  }
  return best;
}

// rows start on 32-byte boundaries: the epilogue stores 8 floats at a time
long long logit_ld(int V) { return (static_cast<long long>(V) + 7) / 8 * 8; }

struct LmLayout {
  size_t partials, tlogits, dlogits, total;
};

LmLayout lm_layout(int B, int gamma, int V, bool greedy) {
  LmLayout L{};
  const int rows = greedy ? gamma + 1 : 2 * gamma + 1;
  L.partials = align256(static_cast<size_t>(B) * rows * lm_chunks(V) * sizeof(float2));
  if (!greedy) {
    L.tlogits = align256(static_cast<size_t>(B) * (gamma + 1) * logit_ld(V) * sizeof(float));
    L.dlogits = align256(static_cast<size_t>(B) * gamma * logit_ld(V) * sizeof(float));
  }
  L.total = L.partials + L.tlogits + L.dlogits;
  return L;
}

cudaError_t launch_head(const void* x, long long R, int d, const void* w, int V, int bv, const LmParams& proto,
                        cudaStream_t s) {
  LmParams P = proto;
  P.R = static_cast<int>(R);
  P.V = V;
  P.d = d;
  P.rt_max = row_tiles(R);
  P.bv = bv;
  P.ntv = (V + P.bv - 1) / P.bv;
  P.nkb = (d + kBK - 1) / kBK;
  CUtensorMap tx, tw;
  if (!make_map(&tx, x, R, d, kBR) || !make_map(&tw, w, V, d, P.bv)) return cudaErrorInvalidValue;
  const int stage_bytes = P.bv * kBK * 2 + kTileBytes * P.rt_max;
  P.stages = min(kMaxStages, kSmemBudget / stage_bytes);
  // measured: with 3 or more stages the L2 requests only add traffic (B = 4
  // to 64 at V = 128256 slower); with 2 stages (512-row blocks) they pay
  P.prefetch = P.stages <= 2 ? kPrefetchSteps : 0;
  const int dyn = P.stages * stage_bytes + 1024;
  cudaError_t e = smem_attribute();
  if (e != cudaSuccess) return e;
  lm_head_kernel<<<P.chunks, kLmThreads, dyn, s>>>(tx, tw, P);
  return cudaGetLastError();
}

// CTA pairs of lm_head_pair_kernel that can be resident at once (a pair
// must fit in one GPC), cached per device.
cudaError_t pair_slots(int* out) {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  const int dyn = kPairRing + kPairExtra + 1024;
  e = cudaFuncSetAttribute(lm_head_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = dyn;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, lm_head_pair_kernel, &cfg);
  if (e != cudaSuccess) return e;
  cache[dev] = n;
  *out = n;
  return cudaSuccess;
}

// One head on `pairs` CTA pairs.  Rows are taken in blocks of up to 512 (two
// chunks of up to 256 when a block holds more than 256 rows); the chunk width
// is the block's rows split evenly, rounded up to a multiple of 16.
cudaError_t launch_head_pair(const void* x, long long R, int d, const void* w, int V, int pairs,
                             const LmPairParams& proto, cudaStream_t s) {
  LmPairParams P = proto;
  P.R = static_cast<int>(R);
  P.V = V;
  P.d = d;
  P.nkb = (d + kBK - 1) / kBK;
  const int rb = static_cast<int>(R < kPairMaxRows ? R : kPairMaxRows);
  P.nch = rb > 256 ? 2 : 1;
  P.nc = ((rb + P.nch - 1) / P.nch + 15) / 16 * 16;
  P.ntv = (V + kPairM - 1) / kPairM;
  CUtensorMap tx, tw;
  if (!make_map(&tx, x, R, d, P.nc / 2) || !make_map(&tw, w, V, d, 128)) return cudaErrorInvalidValue;
  const int stage_bytes = kPairWBytes + P.nch * (P.nc / 2) * kBK * 2;
  P.stages = min(kPairMaxStages, kPairRing / stage_bytes);
  const int dyn = P.stages * stage_bytes + kPairExtra + 1024;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lm_head_pair_kernel, tx, tw, P);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace sv

extern "C" spec_status spec_test_inject_head_copy_timeout(int enable) {
  const int v = enable ? 1 : 0;
  return cudaMemcpyToSymbol(sv::g_lm_copy_timeout_test, &v, sizeof(v)) == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

extern "C" size_t spec_lm_head_chain_workspace_size(int B, int gamma, int V, spec_mode mode) {
  if (B < 1 || gamma < 0 || gamma > 32 || V < 1) return 0;
  return sv::lm_layout(B, gamma, V, mode == SPEC_GREEDY).total;
}

extern "C" spec_status spec_verify_chain_lm_head(const spec_lm_head_chain_args* a, cudaStream_t stream) {
  using namespace sv;
  NvtxRange nvtx_range("spec_verify_chain_lm_head");
  if (a == nullptr) return SPEC_EINVAL;
  if (a->mode != SPEC_GREEDY && a->mode != SPEC_SAMPLE) return SPEC_EDTYPE;
  const bool greedy = a->mode == SPEC_GREEDY;
  if (a->B < 1 || a->B > kMaxSeq || a->gamma < 0 || a->gamma > 32) return SPEC_EINVAL;
  if (a->V < 1 || a->V > 2097152) return SPEC_EINVAL;
  if (a->d_target < 8 || a->d_target > 65536 || a->d_target % 8) return SPEC_EINVAL;
  if (!greedy && a->gamma > 0 && (a->d_draft < 8 || a->d_draft > 65536 || a->d_draft % 8)) return SPEC_EINVAL;
  if (!greedy && !(a->temperature > 0.f && std::isfinite(a->temperature))) return SPEC_EINVAL;
  if (!a->h_target || !a->w_target || !a->accept_len || !a->out_token) return SPEC_EINVAL;
  if (a->gamma > 0 && !a->draft_tokens) return SPEC_EINVAL;
  if (!greedy && (!a->v || (a->gamma > 0 && (!a->h_draft || !a->w_draft || !a->u)))) return SPEC_EINVAL;
  if (!aligned16(a->h_target) || !aligned16(a->w_target)) return SPEC_EALIGN;
  if (!greedy && a->gamma > 0 && (!aligned16(a->h_draft) || !aligned16(a->w_draft))) return SPEC_EALIGN;
  const LmLayout L = lm_layout(a->B, a->gamma, a->V, greedy);
  if (!a->workspace || a->workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(a->workspace) & 255u))
    return SPEC_EWORKSPACE;
  const int nsm = sm_count();
  if (nsm < 1) return SPEC_ECUDA;

  char* ws = static_cast<char*>(a->workspace);
  const int gamma = a->gamma;
  const int rows_seq = greedy ? gamma + 1 : 2 * gamma + 1;
  // one partial column per CTA; both heads use the same count (the smaller
  // vocabulary-tile count of the two, at most one CTA per SM)
  const long long rows_t = static_cast<long long>(a->B) * (gamma + 1);
  const long long rows_d = static_cast<long long>(a->B) * gamma;
  const int slots = min(lm_chunks(a->V), nsm);
  const int bv_t = vocab_tile(row_tiles(rows_t), a->V, slots);
  const int bv_d = vocab_tile(row_tiles(rows_d > 0 ? rows_d : 1), a->V, slots);
  int chunks = min(slots, (a->V + bv_t - 1) / bv_t);
  if (!greedy && gamma > 0) chunks = min(chunks, (a->V + bv_d - 1) / bv_d);
  int pairs = 0;
  bool use_pair = rows_t >= kPairMinRows;
  if (use_pair) {
    cudaError_t pe = pair_slots(&pairs);
    if (pe != cudaSuccess || pairs < 1) return SPEC_ECUDA;
    pairs = min(pairs, (a->V + kPairM - 1) / kPairM);
    // the busier of the two launches' slowest unit: a pair's 256-entry
    // tile takes about 36 us at 384 rows, a CTA's tile about 46 us per 144
    // entries (measured); the pairs' coarser tiles can balance worse
    const int ntv_pair = (a->V + kPairM - 1) / kPairM;
    const double t_pair = 36.0 * static_cast<double>((ntv_pair + pairs - 1) / pairs);
    const double t_single = 46.0 / 144.0 * bv_t * static_cast<double>(((a->V + bv_t - 1) / bv_t + chunks - 1) / chunks);
    use_pair = t_pair < t_single;
  }
  if (use_pair) chunks = 2 * pairs;
  const long long ldl = logit_ld(a->V);
  float* tlog = greedy ? nullptr : reinterpret_cast<float*>(ws + L.partials);
  float* dlog = greedy ? nullptr : reinterpret_cast<float*>(ws + L.partials + L.tlogits);

  LmParams proto{};
  proto.rows_seq = rows_seq;
  proto.chunks = chunks;
  proto.greedy = greedy ? 1 : 0;
  proto.c = greedy ? 1.f : static_cast<float>(1.4426950408889634073599 / static_cast<double>(a->temperature));
  proto.partials = reinterpret_cast<float2*>(ws);
  proto.ldl = ldl;
  proto.error_word = a->error_word;

  // target head: rows (b, i), i <= gamma, statistics rows 0 .. gamma
  LmPairParams pp{};
  pp.rows_seq = rows_seq;
  pp.chunks = chunks;
  pp.greedy = proto.greedy;
  pp.c = proto.c;
  pp.partials = proto.partials;
  pp.ldl = ldl;
  pp.error_word = a->error_word;
  LmParams pt = proto;
  pt.per = gamma + 1;
  pt.row_off = 0;
  pt.logits = tlog;
  LmPairParams ppt = pp;
  ppt.per = gamma + 1;
  ppt.row_off = 0;
  ppt.logits = tlog;
  cudaError_t e = use_pair
                      ? launch_head_pair(a->h_target, rows_t, a->d_target, a->w_target, a->V, pairs, ppt, stream)
                      : launch_head(a->h_target, rows_t, a->d_target, a->w_target, a->V, bv_t, pt, stream);
  if (e != cudaSuccess) return e == cudaErrorInvalidValue ? SPEC_EINVAL : SPEC_ECUDA;
  if (!greedy && gamma > 0) {
    // draft head: rows (b, i), i < gamma, statistics rows gamma + 1 ..
    LmParams pd = proto;
    pd.per = gamma;
    pd.row_off = gamma + 1;
    pd.logits = dlog;
    LmPairParams ppd = pp;
    ppd.per = gamma;
    ppd.row_off = gamma + 1;
    ppd.logits = dlog;
    e = use_pair ? launch_head_pair(a->h_draft, rows_d, a->d_draft, a->w_draft, a->V, pairs, ppd, stream)
                     : launch_head(a->h_draft, rows_d, a->d_draft, a->w_draft, a->V, bv_d, pd, stream);
    if (e != cudaSuccess) return e == cudaErrorInvalidValue ? SPEC_EINVAL : SPEC_ECUDA;
  }

  // the chain walk over the partials (and, sampling, the stored logits)
  StatsParams sp{};
  sp.set[0] = RowSet{tlog, gamma + 1};
  sp.set[1] = RowSet{dlog, gamma};
  sp.nsets = (greedy || gamma == 0) ? 1 : 2;
  sp.rows_per_seq = rows_seq;
  sp.B = a->B;
  sp.V = a->V;
  sp.ld = ldl;
  sp.chunks = chunks;
  sp.ntiles = pass_tiles(a->V);
  sp.c = proto.c;
  sp.partials = proto.partials;
  ChainParams cp{};
  cp.B = a->B;
  cp.gamma = gamma;
  cp.V = a->V;
  cp.ld = ldl;
  cp.target = tlog;
  cp.draft = dlog;
  cp.tokens = a->draft_tokens;
  cp.u = a->u;
  cp.v = a->v;
  cp.prefix = a->prefix_len;
  cp.accept_len = a->accept_len;
  cp.out_token = a->out_token;
  cp.rollback = a->rollback_idx;
  cp.p_at = a->p_at_draft;
  cp.q_at = a->q_at_draft;
  cp.resid = a->resid_mass;
  cp.seq_error = a->seq_error;
  cp.error_word = a->error_word;
  return launch_chain_walk_f32(sp, cp, greedy, stream) == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}
