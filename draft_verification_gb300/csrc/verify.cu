// Batched draft verification kernels and their launch sequence.
//
// A call is two kernels on the caller's stream; the second is launched
// with programmatic dependent launch, so it is resident and has read its own
// inputs by the time the first finishes:
//
//   1. stats_kernel  one CTA per (sequence, row, 16384-element chunk): the
//                    online-softmax (max, sum) or the argmax of the chunk
//                    (stats.cuh).  This streams every logit once; it is
//                    the bandwidth-bound kernel.
//   2. walk kernel   sampling: one thread-block cluster of up to 8 CTAs per
//                    sequence.  Every CTA merges the sequence's statistics
//                    and evaluates the accept tests itself (a few hundred
//                    bytes), then the cluster sums the residual / bonus
//                    weights of the chosen row pair, each CTA a slice of
//                    its tiles, exchanging the tile sums through distributed
//                    shared memory (walk.cuh); the CTA holding the drawn
//                    index's tile writes the result.  Greedy calls use one
//                    CTA per sequence.  The cascade runs both of its stages
//                    in the same cluster, the k-model pipeline its k - 1
//                    stages; a tree runs its serial walk in every CTA of its
//                    cluster and splits each pass.
//
// Variants: large sampling chains run as batch groups (several statistics
// and walk launches on forked library streams); the consulted-only chain
// mode is one kernel, chain_consulted_kernel, whose clusters compute the
// statistics of each position's rows themselves, in position order, and stop
// at the first rejection.
//
// Rules (pages: the Pith review of PipeSpec, "What carries the argument" and
// the acceptance rule of Leviathan et al. its Circularity Check cites; Staged
// Speculative Decoding, abstract):
//  * chain: keep drafts while u < min(1, p/q); draw from max(0, p - q) at the
//    first rejection, from the bonus row when all are kept; greedy keeps
//    drafts equal to the target argmax;
//  * cascade: stage 1 (M_1 verifies M_0's drafts), then stage 2 (M_2 verifies
//    the first tokens of stage 1's output); the pipeline generalises it to k
//    models with an optional final-stage bonus;
//  * tree: a serial walk from the root (each rejected sibling changes the
//    distribution the next sibling is tested against).
//
// Cluster discipline: all CTAs of a cluster read the same inputs and run the
// same code on them, so they take the same branches; every cluster barrier
// is therefore reached by all of them or by none.
#include <array>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "common.cuh"
#include "internal.h"
#include "spec_verify.h"
#include "stats.cuh"
#include "walk.cuh"

namespace sv {
namespace {

constexpr int kMaxGamma = 32;


// Test hook (spec_test_inject_copy_timeout): nonzero makes every bulk-copy
// wait of a residual or bonus pass (ring stage or resident slice) expect 16
// bytes that never come, so that its bounded wait gives up.  Zero in normal
// operation.
__device__ int g_copy_timeout_test = 0;
constexpr int kStage = 4 * kThreads;  // chunk partials staged per round (8 KB)
static_assert(kMaxTiles * kTileElems >= 2097152, "tile sums of the largest row fit in shared memory");

template <typename T>
__device__ __forceinline__ const T* stats_row(const StatsParams& G, int b, int r) {
  // the set holding statistics row r of a sequence, and r's row within it
  int i = r, k = 0;
  while (k + 1 < G.nsets && i >= G.set[k].rows) {
    i -= G.set[k].rows;
    ++k;
  }
  return static_cast<const T*>(G.set[k].base) + (static_cast<long long>(b) * G.set[k].rows + i) * G.ld;
}

// Row statistics of sequence b.  The chunk partials of a group of rows are
// loaded at once (at most 4 per thread) into `stage`; then each row is
// merged in a fixed order, so every CTA of a cluster gets the same bits.
// kWide false: one thread per row, in chunk order (the statistics kernel's
// few chunks per row; a shuffle tree is no faster there).  kWide true: one
// warp per row, each lane merging its chunks k, k + 32, ... in order and the
// warp combining them with shuffles (the LM head's up to 256 partials per
// row).  One thread per row calls emit(row, stats, ok): stats is (max, sum),
// or (unused, argmax bits) in greedy mode; ok is false for a row with a NaN
// or +inf, or without a finite entry.
template <bool kGreedy, bool kWide, typename Emit>
__device__ void merge_stats(const StatsParams& G, int b, float2* stage, Emit emit) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = G.chunks, R = G.rows_per_seq;
  const int rpg = max(1, kStage / C);
  const float2* part = G.partials + static_cast<long long>(b) * R * C;
  for (int r0 = 0; r0 < R; r0 += rpg) {
    const int nr = min(rpg, R - r0);
    const int n = nr * C;
    const float2* src = part + static_cast<long long>(r0) * C;
    float2 v[kStage / kThreads];
#pragma unroll
    for (int q = 0; q < kStage / kThreads; ++q) {
      const int i = q * kThreads + tid;
      if (i < n) v[q] = __ldcg(src + i);
    }
#pragma unroll
    for (int q = 0; q < kStage / kThreads; ++q) {
      const int i = q * kThreads + tid;
      if (i < n) stage[i] = v[q];
    }
    __syncthreads();
    if constexpr (!kWide) {
      for (int r = tid; r < nr; r += kThreads) {
        if constexpr (kGreedy) {
          bool bad;
          const ArgMax am = combine_row_argmax(stage + r * C, C, bad);
          emit(r0 + r, make_float2(0.f, __int_as_float(am.i)), !bad && am.i >= 0);
        } else {
          const MaxSum ms = combine_row(stage + r * C, C, G.c);
          emit(r0 + r, make_float2(ms.m, ms.s), row_stats_ok(ms));
        }
      }
    } else {
      for (int r = warp; r < nr; r += kThreads / 32) {  // warp-uniform
        const float2* pr = stage + r * C;
        if constexpr (kGreedy) {
          ArgMax acc{-kInf, -1};
          bool bad = false;
          for (int k = lane; k < C; k += 32) {
            if (pr[k].x != pr[k].x) bad = true;
            acc = am_merge(acc, ArgMax{pr[k].x, __float_as_int(pr[k].y)});
          }
          acc = am_warp_reduce(acc);
          bad = __any_sync(0xffffffffu, bad);
          if (lane == 0) emit(r0 + r, make_float2(0.f, __int_as_float(acc.i)), !bad && acc.i >= 0);
        } else {
          MaxSum acc{-kInf, 0.f};
          for (int k = lane; k < C; k += 32) acc = ms_merge(acc, MaxSum{pr[k].x, pr[k].y}, G.c);
          acc = ms_warp_reduce(acc, G.c);
          if (lane == 0) emit(r0 + r, make_float2(acc.m, acc.s), row_stats_ok(acc));
        }
      }
    }
    __syncthreads();
  }
}

// Statistics into separate arrays; returns the error bits (or'ed into *err_s).
template <bool kGreedy, bool kWide = false>
__device__ int gather_stats(const StatsParams& G, int b, float* st_m, float* st_s, int* st_arg, int* err_s,
                            float2* stage) {
  merge_stats<kGreedy, kWide>(G, b, stage, [&](int r, float2 v, bool ok) {
    if (kGreedy) {
      st_arg[r] = __float_as_int(v.y);
    } else {
      st_m[r] = v.x;
      st_s[r] = v.y;
    }
    if (!ok) atomicOr(err_s, SPEC_ERR_NONFINITE);
  });
  return *err_s;
}

// Cluster entry and readiness: every CTA arrives when it starts (after
// initialising its pass state) and waits before it first writes another
// CTA's shared memory (or exits), so no CTA touches a peer that has not
// started.
__device__ __forceinline__ void cluster_enter() {
  if (cluster_size() > 1) cluster_arrive();
}
__device__ __forceinline__ void cluster_ready() {
  if (cluster_size() > 1) cluster_wait();
}

template <typename T>
__device__ __forceinline__ PassSpec<T> make_spec(const T* P, float mP, float sP, const T* Q, float mQ, float sQ,
                                                 float cq, float c) {
  PassSpec<T> S;
  S.P = P;
  S.MP = scaled_max(mP, c);
  S.invSP = __fdiv_rn(1.f, sP);
  S.Q = Q;
  S.MQ = Q ? scaled_max(mQ, c) : 0.f;
  S.invSQ = Q ? __fdiv_rn(1.f, sQ) : 0.f;
  S.cq = Q ? cq : 0.f;
  S.extra_tx = g_copy_timeout_test ? 16u : 0u;
  return S;
}

// A pass over the cluster with the zero-mass fallback: if the residual has
// no (finite) mass, the pass is redone on the target row alone (cq = 0) and
// *flag gets SPEC_ERR_ZERO_MASS.  *buf is the buffer of the first pass on
// entry and of the pass to draw from on return.
template <typename T>
__device__ DF pass_or_fallback(PassSpec<T>& S, int V, float c, int ntiles, int* buf, int* flag, PassSmem& ps) {
  DF z = cluster_pass(S, V, c, ntiles, *buf, ps);
  if (!pass_ok(z)) {
    *flag |= SPEC_ERR_ZERO_MASS;
    S.cq = 0.f;
    S.Q = nullptr;
    *buf ^= 1;
    z = cluster_pass(S, V, c, ntiles, *buf, ps);
  }
  return z;
}

// ===========================================================================
// 1. statistics
// ===========================================================================
template <typename T, bool kGreedy>
__global__ void __launch_bounds__(kStatsThreads, 5) stats_kernel(const StatsParams G) {
  pdl_launch_dependents();
  __shared__ StatsSmem sm;
  const int k = blockIdx.x, r = blockIdx.y, b = blockIdx.z;
  float2* out = G.partials + (static_cast<long long>(b) * G.rows_per_seq + r) * G.chunks + k;
  stats_unit<T, kGreedy>(stats_row<T>(G, b, r), G.V, k, G.c, out, sm);
}

// ===========================================================================
// 2a. chain
// ===========================================================================
struct ChainSmem {
  float st_m[2 * kMaxGamma + 1], st_s[2 * kMaxGamma + 1];
  int st_arg[kMaxGamma + 1];
  int tok[kMaxGamma];
  float gp[kMaxGamma], gq[kMaxGamma];
  float u[kMaxGamma], v;  // the call's uniforms (sampling)
  int err, a;
};

// Tokens, the logits at the drafted tokens and the uniforms (inputs only:
// safe before the statistics are complete).
template <typename T>
__device__ void chain_inputs(const ChainParams& P, int b, ChainSmem& cs, bool sampling) {
  const int g = P.gamma, tid = threadIdx.x;
  if (tid == 0) cs.err = 0;
  __syncthreads();
  if (sampling && tid == kThreads - 1) cs.v = P.v[b];
  if (tid < g) {
    const long long d0 = static_cast<long long>(b) * g;
    const long long t0 = static_cast<long long>(b) * (g + 1);
    if (sampling) cs.u[tid] = P.u[d0 + tid];
    const int t = P.tokens[d0 + tid];
    cs.tok[tid] = t;
    if (t < 0 || t >= P.V) {
      atomicOr(&cs.err, SPEC_ERR_TOKEN);
    } else if (sampling) {
      cs.gp[tid] = load_elem(static_cast<const T*>(P.target) + (t0 + tid) * P.ld + t);
      cs.gq[tid] = load_elem(static_cast<const T*>(P.draft) + (d0 + tid) * P.ld + t);
    }
  }
}

__device__ void chain_error_out(const ChainParams& P, int b, int err) {
  const int tid = threadIdx.x, g = P.gamma;
  if (tid == 0) {
    P.accept_len[b] = 0;
    P.out_token[b] = -1;
    if (P.rollback) P.rollback[b] = P.prefix ? P.prefix[b] : 0;
    if (P.resid) P.resid[b] = 0.f;
    if (P.seq_error) P.seq_error[b] = err;
    if (P.error_word) atomicOr(P.error_word, err);
  }
  if (tid < g) {
    if (P.p_at) P.p_at[static_cast<long long>(b) * g + tid] = 0.f;
    if (P.q_at) P.q_at[static_cast<long long>(b) * g + tid] = 0.f;
  }
}

// kWide: the row partials come from the LM head (many chunks per row).
template <typename T, bool kWide = false>
__global__ void __launch_bounds__(kThreads) chain_greedy_kernel(const StatsParams G, const ChainParams P) {
  __shared__ ChainSmem cs;
  __shared__ float2 stage[kStage];
  const int b = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = P.gamma;
  chain_inputs<T>(P, b, cs, false);
  pdl_wait();
  const int err = gather_stats<true, kWide>(G, b, cs.st_m, cs.st_s, cs.st_arg, &cs.err, stage);
  if (err) {
    chain_error_out(P, b, err);
    return;
  }
  if (warp == 0) {
    const unsigned rej = __ballot_sync(0xffffffffu, lane < g && cs.tok[lane] != cs.st_arg[lane]);
    const int a = rej ? __ffs(rej) - 1 : g;
    if (lane == 0) {
      P.accept_len[b] = a;
      P.out_token[b] = cs.st_arg[a];
      if (P.rollback) P.rollback[b] = (P.prefix ? P.prefix[b] : 0) + a;
      if (P.resid) P.resid[b] = 0.f;
      if (P.seq_error) P.seq_error[b] = 0;
    }
    if (lane < g) {
      if (P.p_at) P.p_at[static_cast<long long>(b) * g + lane] = 0.f;
      if (P.q_at) P.q_at[static_cast<long long>(b) * g + lane] = 0.f;
    }
  }
}

// Sampling chain: one cluster per sequence (grid (S, B), cluster (S, 1, 1)).
// kResident: every CTA loads its whole slice of the chosen row pair into
// dynamic shared memory at once (one bulk-copy round trip instead of a ring
// of stages) and the drawing CTA finds the element there; used where the
// walk runs after the statistics have been read (the last batch group), so
// its larger shared memory does not crowd the statistics kernel.  kWide:
// the row partials come from the LM head (many chunks per row).
template <typename T, bool kResident, bool kWide = false>
__global__ void __launch_bounds__(kThreads, 4) chain_walk_kernel(const StatsParams G, const ChainParams P) {
  __shared__ ChainSmem cs;
  __shared__ PassSmem ps;
  __shared__ float2 stage[kStage];
  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = P.gamma;
  const float c = G.c;
  const bool lead = cluster_rank() == 0;
  const T* target = static_cast<const T*>(P.target);
  const T* draft = static_cast<const T*>(P.draft);
  const long long trow0 = static_cast<long long>(b) * (g + 1);
  const long long drow0 = static_cast<long long>(b) * g;

  pass_begin(ps);
  cluster_enter();
  chain_inputs<T>(P, b, cs, true);
  pdl_wait();  // the statistics are complete and visible from here on
  const int err = gather_stats<false, kWide>(G, b, cs.st_m, cs.st_s, cs.st_arg, &cs.err, stage);
  cluster_ready();
  if (err) {  // every CTA of the cluster sees the same error; the lead reports it
    if (lead) chain_error_out(P, b, err);
    return;
  }
  if (warp == 0) {
    bool keep = true;
    if (lane < g) {
      const float mq = cs.st_m[g + 1 + lane], sq = cs.st_s[g + 1 + lane];
      keep = keeps(cs.u[lane], ratio(cs.gp[lane], cs.st_m[lane], cs.st_s[lane], cs.gq[lane], mq, sq, c));
      if (lead) {
        if (P.p_at) P.p_at[drow0 + lane] = prob(cs.gp[lane], cs.st_m[lane], cs.st_s[lane], c);
        if (P.q_at) P.q_at[drow0 + lane] = prob(cs.gq[lane], mq, sq, c);
      }
    }
    const unsigned rej = __ballot_sync(0xffffffffu, lane < g && !keep);
    if (lane == 0) cs.a = rej ? __ffs(rej) - 1 : g;
  }
  __syncthreads();
  const int a = cs.a;
  // residual max(0, p_a - q_a) after a rejection, the bonus row p_gamma otherwise
  PassSpec<T> S = make_spec(target + (trow0 + a) * P.ld, cs.st_m[a], cs.st_s[a],
                            a < g ? draft + (drow0 + a) * P.ld : nullptr, a < g ? cs.st_m[g + 1 + a] : 0.f,
                            a < g ? cs.st_s[g + 1 + a] : 1.f, 1.f, c);
  int buf = 0, flag = 0;
  DF Z;
  int y;
  if constexpr (kResident) {
    const int ncl = static_cast<int>(cluster_size());
    const int tpc = (G.ntiles + ncl - 1) / ncl;
    const int t0 = min(G.ntiles, static_cast<int>(cluster_rank()) * tpc), t1 = min(G.ntiles, t0 + tpc);
    slice_load(S, a < g, G.V, t0, t1, ps);
    Z = cluster_pass(S, G.V, c, G.ntiles, buf, ps, true);
    if (!pass_ok(Z)) {  // reading R3: the target row alone, already resident
      flag |= SPEC_ERR_ZERO_MASS;
      S.cq = 0.f;
      S.Q = nullptr;
      buf ^= 1;
      Z = cluster_pass(S, G.V, c, G.ntiles, buf, ps, true);
    }
    y = cluster_draw(S, G.V, c, G.ntiles, buf, df_mul_f(Z, cs.v), false, ps, true);
  } else {
    Z = pass_or_fallback(S, G.V, c, G.ntiles, &buf, &flag, ps);
    y = cluster_draw(S, G.V, c, G.ntiles, buf, df_mul_f(Z, cs.v), false, ps);
  }
  if (y < 0) return;  // another CTA of the cluster holds the drawn tile
  if (ps.fault) {  // a bounded wait gave up: the draw is not trusted
    flag |= SPEC_ERR_INTERNAL;
    if (tid == 0) {
      P.accept_len[b] = 0;
      P.out_token[b] = -1;
      if (P.rollback) P.rollback[b] = P.prefix ? P.prefix[b] : 0;
      if (P.resid) P.resid[b] = 0.f;
      if (P.seq_error) P.seq_error[b] = flag;
      if (P.error_word) atomicOr(P.error_word, flag);
    }
    return;
  }
  if (tid == 0) {
    P.accept_len[b] = a;
    P.out_token[b] = y;
    if (P.rollback) P.rollback[b] = (P.prefix ? P.prefix[b] : 0) + a;
    if (P.resid) P.resid[b] = df_float(Z);
    if (P.seq_error) P.seq_error[b] = flag;
    if (flag && P.error_word) atomicOr(P.error_word, flag);
  }
}

// Consulted-only sampling chain (PipeSpec review, "What carries the
// argument": the tokens after the first mismatch are rolled back unused):
// one cluster per sequence walks the positions in order and computes each
// position's row statistics itself, so rows after the first rejection are
// never read.  At position i every CTA streams its slice of target row i and
// draft row i, the cluster shares the (max, sum) partials and merges them in
// rank order, and the accept test runs on the merged statistics; a
// rejection is followed by the residual pass over the same two rows and the
// draw; when every draft is kept, the bonus row gamma gets its statistics
// and the draw.  No statistics kernel and no workspace.  Grid (S, B).
template <typename T>
__global__ void __launch_bounds__(kThreads, 4) chain_consulted_kernel(const StatsParams G, const ChainParams P) {
  __shared__ ChainSmem cs;
  __shared__ PassSmem ps;
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  const int g = P.gamma;
  const float c = G.c;
  const bool lead = cluster_rank() == 0;
  const T* target = static_cast<const T*>(P.target);
  const T* draft = static_cast<const T*>(P.draft);
  const long long trow0 = static_cast<long long>(b) * (g + 1);
  const long long drow0 = static_cast<long long>(b) * g;
  const int ncl = static_cast<int>(cluster_size());
  const int tpc = (G.ntiles + ncl - 1) / ncl;
  const int t0 = min(G.ntiles, static_cast<int>(cluster_rank()) * tpc), t1 = min(G.ntiles, t0 + tpc);

  pass_begin(ps);
  cluster_enter();
  chain_inputs<T>(P, b, cs, true);
  cluster_ready();
  __syncthreads();
  if (cs.err) {  // a drafted token out of range: nothing is consulted
    if (lead) chain_error_out(P, b, cs.err);
    return;
  }
  for (int i = 0;; ++i) {
    const bool bonus = i == g;
    const T* prow = target + (trow0 + i) * P.ld;
    const T* qrow = bonus ? nullptr : draft + (drow0 + i) * P.ld;
    MaxSum part[2];
    streamed_row_stats<T>(prow, qrow, G.V, c, t0, t1, ps, part);
    const int xb = cluster_share4(part[0].m, part[0].s, part[1].m, part[1].s, ps);
    MaxSum st[2];
    merge_shared_ms2(xb, c, ps, st);
    const bool bad = !row_stats_ok(st[0]) || (!bonus && !row_stats_ok(st[1]));
    if (bad) {
      if (lead) chain_error_out(P, b, SPEC_ERR_NONFINITE);
      return;
    }
    bool keep = true;
    if (!bonus) {
      keep = keeps(cs.u[i], ratio(cs.gp[i], st[0].m, st[0].s, cs.gq[i], st[1].m, st[1].s, c));
      if (lead && tid == 0) {
        if (P.p_at) P.p_at[drow0 + i] = prob(cs.gp[i], st[0].m, st[0].s, c);
        if (P.q_at) P.q_at[drow0 + i] = prob(cs.gq[i], st[1].m, st[1].s, c);
      }
    }
    if (!bonus && keep) continue;
    // position i: the residual after a rejection, or the bonus row
    const int a = i;
    if (lead && tid < g && tid > a) {  // positions never consulted
      if (P.p_at) P.p_at[drow0 + tid] = __int_as_float(0x7fc00000);
      if (P.q_at) P.q_at[drow0 + tid] = __int_as_float(0x7fc00000);
    }
    PassSpec<T> S = make_spec(prow, st[0].m, st[0].s, qrow, bonus ? 0.f : st[1].m, bonus ? 1.f : st[1].s, 1.f, c);
    int buf = 0, flag = 0;
    const DF Z = pass_or_fallback(S, G.V, c, G.ntiles, &buf, &flag, ps);
    const int y = cluster_draw(S, G.V, c, G.ntiles, buf, df_mul_f(Z, cs.v), false, ps);
    if (y < 0) return;  // another CTA of the cluster holds the drawn tile
    if (ps.fault) flag |= SPEC_ERR_INTERNAL;
    if (tid == 0) {
      const bool ok = !(flag & SPEC_ERR_INTERNAL);
      P.accept_len[b] = ok ? a : 0;
      P.out_token[b] = ok ? y : -1;
      if (P.rollback) P.rollback[b] = (P.prefix ? P.prefix[b] : 0) + (ok ? a : 0);
      if (P.resid) P.resid[b] = ok ? df_float(Z) : 0.f;
      if (P.seq_error) P.seq_error[b] = flag;
      if (flag && P.error_word) atomicOr(P.error_word, flag);
    }
    return;
  }
}

// ===========================================================================
// 2b. cascade
// Statistics rows: sampling: M_0 [0, g1), M_1 [g1, 2 g1 + 1), M_2 after;
// greedy (M_0 not read): M_1 [0, g1 + 1), M_2 [g1 + 1, ...).
// ===========================================================================
struct CascadeSmem {
  float st_m[3 * kMaxGamma + 1], st_s[3 * kMaxGamma + 1];
  int st_arg[3 * kMaxGamma + 1];
  int tok[kMaxGamma];
  float g1p[kMaxGamma], g1q[kMaxGamma];
  float g2p[kMaxGamma], g2q[kMaxGamma];  // M_2 and M_1 logits at drafted token i (i < min(g1, g2))
  float u1[kMaxGamma], u2[kMaxGamma], v1, v2;  // the call's uniforms (sampling)
  int err, a1, a2;
};

struct CascadeOut {
  const CascadeParams& P;
  int b;
  __device__ void write(int a1, int t1, int a2, int w2, int t2, int t2v, int flag) const {
    if (flag & SPEC_ERR_INTERNAL) {  // a bounded wait gave up: empty outputs
      a1 = 0;
      t1 = -1;
      a2 = 0;
      w2 = 0;
      t2 = -1;
      t2v = 0;
    }
    const bool rej = a2 < w2;
    const int base0 = P.base0 ? P.base0[b] : 0;
    const int base1 = P.base1 ? P.base1[b] : 0;
    P.a1[b] = a1;
    P.t1[b] = t1;
    P.a2[b] = a2;
    P.w2[b] = w2;
    P.t2[b] = t2;
    P.t2_valid[b] = t2v;
    P.r0[b] = base0 + (rej ? min(a1, a2) : a1);
    P.r1[b] = base1 + (rej ? a2 : w2);
    P.committed[b] = a2 + t2v;
    if (P.seq_error) P.seq_error[b] = flag;
    if (flag && P.error_word) atomicOr(P.error_word, flag);
  }
};

template <typename T>
__device__ void cascade_inputs(const CascadeParams& P, int b, CascadeSmem& cs, bool sampling) {
  const int g1 = P.g1, g2 = P.g2, tid = threadIdx.x;
  if (tid == 0) cs.err = 0;
  __syncthreads();
  if (sampling && tid == kThreads - 1) {
    cs.v1 = P.v1[b];
    cs.v2 = P.v2[b];
  }
  if (sampling && tid < g2) cs.u2[tid] = P.u2[static_cast<long long>(b) * g2 + tid];
  if (tid < g1) {
    const long long b0 = static_cast<long long>(b) * g1, b1 = static_cast<long long>(b) * (g1 + 1);
    const long long b2 = static_cast<long long>(b) * g2;
    if (sampling) cs.u1[tid] = P.u1[b0 + tid];
    const int t = P.tokens[b0 + tid];
    cs.tok[tid] = t;
    if (t < 0 || t >= P.V) {
      atomicOr(&cs.err, SPEC_ERR_TOKEN);
    } else if (sampling) {
      cs.g1p[tid] = load_elem(static_cast<const T*>(P.l1) + (b1 + tid) * P.ld + t);
      cs.g1q[tid] = load_elem(static_cast<const T*>(P.l0) + (b0 + tid) * P.ld + t);
      if (tid < g2) {  // stage 2 tests drafted token i at position i while i < a1
        cs.g2p[tid] = load_elem(static_cast<const T*>(P.l2) + (b2 + tid) * P.ld + t);
        cs.g2q[tid] = cs.g1p[tid];
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) cascade_greedy_kernel(const StatsParams G, const CascadeParams P) {
  __shared__ CascadeSmem cs;
  __shared__ float2 stage[kStage];
  const int b = blockIdx.x;
  const int g1 = P.g1, g2 = P.g2;
  cascade_inputs<T>(P, b, cs, false);
  pdl_wait();
  const int err = gather_stats<true>(G, b, cs.st_m, cs.st_s, cs.st_arg, &cs.err, stage);
  if (threadIdx.x != 0) return;
  const CascadeOut out{P, b};
  if (err) {
    out.write(0, -1, 0, 0, -1, 0, err);
    return;
  }
  const int r1 = 0, r2 = g1 + 1;
  int a1 = g1;
  for (int q = 0; q < g1; ++q)
    if (cs.tok[q] != cs.st_arg[r1 + q]) {
      a1 = q;
      break;
    }
  const int t1 = cs.st_arg[r1 + a1];
  const int w2 = min(g2, a1 + 1);
  int a2 = w2;
  for (int q = 0; q < w2; ++q) {
    const int o = q < a1 ? cs.tok[q] : t1;
    if (o != cs.st_arg[r2 + q]) {
      a2 = q;
      break;
    }
  }
  out.write(a1, t1, a2, w2, a2 < w2 ? cs.st_arg[r2 + a2] : -1, a2 < w2 ? 1 : 0, 0);
}

// Sampling cascade, both stages in one cluster per sequence.  Every CTA
// draws t1 (the stage-2 tests need it); the CTA holding t2's tile writes.
template <typename T>
__global__ void __launch_bounds__(kThreads, 4) cascade_walk_kernel(const StatsParams G, const CascadeParams P) {
  __shared__ CascadeSmem cs;
  __shared__ PassSmem ps;
  __shared__ float2 stage[kStage];
  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g1 = P.g1, g2 = P.g2;
  const float c = G.c;
  const int r1 = g1, r2 = 2 * g1 + 1;
  const bool lead = cluster_rank() == 0;
  const T* L0 = static_cast<const T*>(P.l0);
  const T* L1 = static_cast<const T*>(P.l1);
  const T* L2 = static_cast<const T*>(P.l2);
  const long long b0 = static_cast<long long>(b) * g1;
  const long long b1 = static_cast<long long>(b) * (g1 + 1);
  const long long b2 = static_cast<long long>(b) * g2;
  const CascadeOut out{P, b};

  pass_begin(ps);
  cluster_enter();
  cascade_inputs<T>(P, b, cs, true);
  pdl_wait();
  const int err = gather_stats<false>(G, b, cs.st_m, cs.st_s, cs.st_arg, &cs.err, stage);
  cluster_ready();
  if (err) {
    if (lead && tid == 0) out.write(0, -1, 0, 0, -1, 0, err);
    return;
  }
  // stage 1: M_1 verifies O_0 against M_0
  if (warp == 0) {
    bool keep = true;
    if (lane < g1)
      keep = keeps(cs.u1[lane], ratio(cs.g1p[lane], cs.st_m[r1 + lane], cs.st_s[r1 + lane], cs.g1q[lane],
                                         cs.st_m[lane], cs.st_s[lane], c));
    const unsigned rej = __ballot_sync(0xffffffffu, lane < g1 && !keep);
    if (lane == 0) cs.a1 = rej ? __ffs(rej) - 1 : g1;
  }
  __syncthreads();
  const int a1 = cs.a1;
  PassSpec<T> S1 = make_spec(L1 + (b1 + a1) * P.ld, cs.st_m[r1 + a1], cs.st_s[r1 + a1],
                             a1 < g1 ? L0 + (b0 + a1) * P.ld : nullptr, a1 < g1 ? cs.st_m[a1] : 0.f,
                             a1 < g1 ? cs.st_s[a1] : 1.f, 1.f, c);
  int buf = 0, flag = 0;
  const DF Z1 = pass_or_fallback(S1, G.V, c, G.ntiles, &buf, &flag, ps);
  const int t1 = cluster_draw(S1, G.V, c, G.ntiles, buf, df_mul_f(Z1, cs.v1), true, ps);

  // stage 2: M_2 verifies the first w2 tokens of O_1 = d[0, a1) ++ t1 against M_1
  const int w2 = min(g2, a1 + 1);
  if (warp == 0) {
    bool keep = true;
    if (lane < w2) {
      // drafted tokens' logits were loaded with the inputs; only t1's is new
      const float xp = lane < a1 ? cs.g2p[lane] : load_elem(L2 + (b2 + lane) * P.ld + t1);
      const float xq = lane < a1 ? cs.g2q[lane] : load_elem(L1 + (b1 + lane) * P.ld + t1);
      keep = keeps(cs.u2[lane],
                   ratio(xp, cs.st_m[r2 + lane], cs.st_s[r2 + lane], xq, cs.st_m[r1 + lane], cs.st_s[r1 + lane], c));
    }
    const unsigned rej = __ballot_sync(0xffffffffu, lane < w2 && !keep);
    if (lane == 0) cs.a2 = rej ? __ffs(rej) - 1 : w2;
  }
  __syncthreads();
  const int a2 = cs.a2;
  if (a2 == w2) {  // all w2 kept: no stage-2 draw
    if (lead && tid == 0) out.write(a1, t1, a2, w2, -1, 0, flag | (ps.fault ? SPEC_ERR_INTERNAL : 0));
    return;
  }
  // the residual max(0, p2 - p1) at position a2
  PassSpec<T> S2 = make_spec(L2 + (b2 + a2) * P.ld, cs.st_m[r2 + a2], cs.st_s[r2 + a2], L1 + (b1 + a2) * P.ld,
                             cs.st_m[r1 + a2], cs.st_s[r1 + a2], 1.f, c);
  buf ^= 1;
  const DF Z2 = pass_or_fallback(S2, G.V, c, G.ntiles, &buf, &flag, ps);
  const int t2 = cluster_draw(S2, G.V, c, G.ntiles, buf, df_mul_f(Z2, cs.v2), false, ps);
  if (t2 < 0) return;
  if (tid == 0) out.write(a1, t1, a2, w2, t2, 1, flag | (ps.fault ? SPEC_ERR_INTERNAL : 0));
}

// ===========================================================================
// 2b'. k-model pipeline (PipeSpec review, "What carries the argument")
// Statistics rows: model s's rows start at P.rowoff[s] (sampling: M_0 first;
// greedy: M_0 not read).
// ===========================================================================
constexpr int kMaxPipeRows = kMaxGamma + (kMaxSets - 1) * (kMaxGamma + 1);

struct PipeSmem {
  float st_m[kMaxPipeRows], st_s[kMaxPipeRows];
  int st_arg[kMaxPipeRows];
  int buf[kMaxGamma + 1];  // the buffer the current stage verifies
  float u[kMaxSets - 1][kMaxGamma], v[kMaxSets - 1];
  int a[kMaxSets - 1], w[kMaxSets - 1], t[kMaxSets - 1], tv[kMaxSets - 1];
  int err, len, ra;
};

// Tokens and uniforms (inputs only: safe before the statistics are complete).
__device__ void pipe_inputs(const PipelineParams& P, int b, PipeSmem& cs, bool sampling) {
  const int g1 = P.window[0], tid = threadIdx.x;
  if (tid == 0) cs.err = 0;
  __syncthreads();
  if (tid < g1) {
    const int t = P.tokens[static_cast<long long>(b) * g1 + tid];
    cs.buf[tid] = t;
    if (t < 0 || t >= P.V) atomicOr(&cs.err, SPEC_ERR_TOKEN);
  }
  if (sampling) {
    for (int i = tid; i < (P.k - 1) * kMaxGamma; i += kThreads) {
      const int s = i / kMaxGamma, j = i - s * kMaxGamma;
      if (j < P.window[s]) cs.u[s][j] = P.u[s][static_cast<long long>(b) * P.window[s] + j];
    }
    if (tid < P.k - 1) cs.v[tid] = P.v[tid][b];
  }
}

// The outputs of sequence b (one thread).  Rollback: buffer O_j keeps
// min(L_j, a_s of every rejecting stage s > j), L_0 = a_1, L_j = w_{j+1}.
__device__ void pipe_write(const PipelineParams& P, int b, const PipeSmem& cs, int flag, bool error) {
  const int k1 = P.k - 1;
  const long long o = static_cast<long long>(b) * k1;
  for (int s = 0; s < k1; ++s) {
    P.a[o + s] = error ? 0 : cs.a[s];
    P.w[o + s] = error ? 0 : cs.w[s];
    P.t[o + s] = error ? -1 : cs.t[s];
    P.t_valid[o + s] = error ? 0 : cs.tv[s];
  }
  for (int j = 0; j < k1; ++j) {
    int keep = 0;
    if (!error) {
      keep = j == 0 ? cs.a[0] : cs.w[j];
      for (int s = j; s < k1; ++s)  // stage s + 1 > j
        if (cs.a[s] < cs.w[s]) keep = min(keep, cs.a[s]);
    }
    P.r[o + j] = (P.base ? P.base[static_cast<long long>(j) * P.B + b] : 0) + keep;
  }
  P.committed[b] = error ? 0 : cs.len;
  if (P.seq_error) P.seq_error[b] = flag;
  if (flag && P.error_word) atomicOr(P.error_word, flag);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) pipeline_greedy_kernel(const StatsParams G, const PipelineParams P) {
  __shared__ PipeSmem cs;
  __shared__ float2 stage[kStage];
  const int b = blockIdx.x, k = P.k;
  pipe_inputs(P, b, cs, false);
  pdl_wait();
  const int err = gather_stats<true>(G, b, cs.st_m, cs.st_s, cs.st_arg, &cs.err, stage);
  if (threadIdx.x != 0) return;
  if (err) {
    pipe_write(P, b, cs, err, true);
    return;
  }
  int len = P.window[0];
  for (int s = 1; s < k; ++s) {
    const int* arg = cs.st_arg + P.rowoff[s];
    const int w = s == 1 ? P.window[0] : min(P.window[s - 1], len);
    int a = w;
    for (int j = 0; j < w; ++j)
      if (cs.buf[j] != arg[j]) {
        a = j;
        break;
      }
    const bool bonus = s == 1 || (P.final_bonus && s == k - 1);
    int tok = -1, valid = 0;
    if (a < w || bonus) {
      tok = arg[a];  // a == w for the bonus: the row after the window
      valid = 1;
      cs.buf[a] = tok;
      len = a + 1;
    } else {
      len = w;
    }
    cs.a[s - 1] = a;
    cs.w[s - 1] = w;
    cs.t[s - 1] = tok;
    cs.tv[s - 1] = valid;
  }
  cs.len = len;
  pipe_write(P, b, cs, 0, false);
}

// Sampling pipeline, every stage in one cluster per sequence.  Every CTA
// draws every emitted token (the next stage tests it); the lead CTA writes.
template <typename T>
__global__ void __launch_bounds__(kThreads, 4) pipeline_walk_kernel(const StatsParams G, const PipelineParams P) {
  __shared__ PipeSmem cs;
  __shared__ PassSmem ps;
  __shared__ float2 stage[kStage];
  const int b = blockIdx.y, k = P.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float c = G.c;
  const bool lead = cluster_rank() == 0;

  pass_begin(ps);
  cluster_enter();
  pipe_inputs(P, b, cs, true);
  pdl_wait();
  const int err = gather_stats<false>(G, b, cs.st_m, cs.st_s, cs.st_arg, &cs.err, stage);
  cluster_ready();
  if (err) {
    if (lead && tid == 0) pipe_write(P, b, cs, err, true);
    return;
  }
  if (tid == 0) cs.len = P.window[0];
  __syncthreads();
  int pbuf = 1, flag = 0;
  for (int s = 1; s < k; ++s) {
    const T* Ms = static_cast<const T*>(P.logits[s]) + static_cast<long long>(b) * P.rows[s] * P.ld;
    const T* Mq = static_cast<const T*>(P.logits[s - 1]) + static_cast<long long>(b) * P.rows[s - 1] * P.ld;
    const int ros = P.rowoff[s], roq = P.rowoff[s - 1];
    const int w = s == 1 ? P.window[0] : min(P.window[s - 1], cs.len);
    if (warp == 0) {
      bool keep = true;
      if (lane < w) {
        const int o = cs.buf[lane];
        const float xp = load_elem(Ms + lane * P.ld + o), xq = load_elem(Mq + lane * P.ld + o);
        keep = keeps(cs.u[s - 1][lane],
                     ratio(xp, cs.st_m[ros + lane], cs.st_s[ros + lane], xq, cs.st_m[roq + lane], cs.st_s[roq + lane], c));
      }
      const unsigned rej = __ballot_sync(0xffffffffu, lane < w && !keep);
      if (lane == 0) cs.ra = rej ? __ffs(rej) - 1 : w;
    }
    __syncthreads();
    const int a = cs.ra;
    const bool bonus = s == 1 || (P.final_bonus && s == k - 1);
    int tok = -1;
    if (a < w || bonus) {
      // the residual max(0, p_s - p_{s-1}) at position a, or M_s's row w for the bonus
      PassSpec<T> S = make_spec(Ms + a * P.ld, cs.st_m[ros + a], cs.st_s[ros + a], a < w ? Mq + a * P.ld : nullptr,
                                a < w ? cs.st_m[roq + a] : 0.f, a < w ? cs.st_s[roq + a] : 1.f, 1.f, c);
      pbuf ^= 1;
      const DF Z = pass_or_fallback(S, G.V, c, G.ntiles, &pbuf, &flag, ps);
      tok = cluster_draw(S, G.V, c, G.ntiles, pbuf, df_mul_f(Z, cs.v[s - 1]), true, ps);
    }
    if (tid == 0) {
      cs.a[s - 1] = a;
      cs.w[s - 1] = w;
      cs.t[s - 1] = tok;
      cs.tv[s - 1] = tok >= 0 ? 1 : 0;
      if (tok >= 0) {
        cs.buf[a] = tok;
        cs.len = a + 1;
      } else {
        cs.len = w;
      }
    }
    __syncthreads();
  }
  if (lead && tid == 0) pipe_write(P, b, cs, flag | (ps.fault ? SPEC_ERR_INTERNAL : 0), ps.fault != 0);
}

// ===========================================================================
// 2c. tree (one cluster per tree in sampling mode, one CTA in greedy mode)
//
// After k rejected siblings at one node the current distribution is
//     p_k = max(0, p - c_k q) / W_k,   c_0 = 0, W_0 = 1,
//     c_{k+1} = c_k + W_k,             W_{k+1} = sum_x max(0, p - c_{k+1} q),
// since max(0, max(0, p - c_k q)/W_k - q) = max(0, p - (c_k + W_k) q)/W_k
// where the inner term is positive, and both sides are 0 elsewhere.  So each
// rejection costs one pass with the scalar cq = c_{k+1}, and a final draw
// searches the last pass with target v * W_k: the iterated renormalisation
// of the rule, written in closed form.
// ===========================================================================
struct TreeSmem {
  float2* st;  // [2N] (max, sum) of target rows then draft rows; greedy: argmax in .y
  int* par;    // [N]
  int* tk;     // [N]
  float* gp;   // [N] target logit of node i's token in its parent's row
  float* gq;   // [N] draft logit of the same
  int* scr_a;  // [N] depth pointer jumping, then the children of the current node
  int* scr_b;  // [N] depth pointer jumping, then the kept path
  float* u;    // [N] node i's accept uniform
};
constexpr int kTreeSmemPerNode = 44;
constexpr int kMaxNodes = 1024;

__device__ __forceinline__ TreeSmem tree_smem(char* base, int N) {
  TreeSmem t;
  t.st = reinterpret_cast<float2*>(base);
  t.par = reinterpret_cast<int*>(base + 16 * N);
  t.tk = t.par + N;
  t.gp = reinterpret_cast<float*>(t.tk + N);
  t.gq = t.gp + N;
  t.scr_a = reinterpret_cast<int*>(t.gq + N);
  t.scr_b = t.scr_a + N;
  t.u = reinterpret_cast<float*>(t.scr_b + N);
  return t;
}

// Children of `node`, ascending, into kids[] (warp 0); count for all threads.
__device__ int list_children(const int* par, int N, int node, int* kids, int* count_s) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid < 32) {
    int count = 0;
    for (int base = node + 1; base < N; base += 32) {
      const int i = base + lane;
      const bool ch = i < N && par[i] == node;
      const unsigned m = __ballot_sync(0xffffffffu, ch);
      if (ch) kids[count + __popc(m & ((1u << lane) - 1u))] = i;
      count += __popc(m);
    }
    if (lane == 0) *count_s = count;
  }
  __syncthreads();
  return *count_s;
}

// kConsulted (Staged Speculative Decoding, abstract: the walk keeps one
// child per level; PipeSpec review, "What carries the argument": tokens after
// the first mismatch are never used): no statistics kernel; the cluster
// computes the statistics of node n's rows when the walk stands at n (the
// target row, and in sampling mode the draft row when n has children), so
// rows of nodes off the walked path are never read.  Sampling and greedy
// both run as clusters with the stage region.
template <typename T, bool kGreedy, bool kConsulted>
__global__ void __launch_bounds__(kThreads) tree_kernel(const StatsParams G, const TreeParams P) {
  __shared__ PassSmem ps;
  __shared__ float2 stage[kConsulted ? 1 : kStage];
  __shared__ int err_s, nk_s, keep_s;
  __shared__ float v_s;
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  const int N = P.N;
  const float c = G.c;
  const bool lead = cluster_rank() == 0;
  constexpr bool kStageRegion = !kGreedy || kConsulted;
  TreeSmem ts = tree_smem(reinterpret_cast<char*>(dyn_smem + (kStageRegion ? kStageBytes : 0)), N);
  const long long row0 = static_cast<long long>(b) * N;

  pass_begin(ps);
  cluster_enter();
  // tree shape and tokens (inputs: read while the statistics finish)
  if (tid == 0) err_s = 0;
  for (int i = tid; i < N; i += kThreads) {
    ts.par[i] = P.parent[row0 + i];
    ts.tk[i] = P.tokens[row0 + i];
  }
  __syncthreads();
  for (int i = tid; i < N; i += kThreads) {
    const int p = ts.par[i];
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) atomicOr(&err_s, SPEC_ERR_PARENT);
    if (i > 0 && (ts.tk[i] < 0 || ts.tk[i] >= P.V)) atomicOr(&err_s, SPEC_ERR_TOKEN);
  }
  __syncthreads();
  if (!(err_s & SPEC_ERR_PARENT)) {
    // depth by pointer jumping (N <= kMaxNodes): D[i] += D[A[i]], A[i] = A[A[i]]
    constexpr int kPer = kMaxNodes / kThreads;
    for (int i = tid; i < N; i += kThreads) {
      ts.scr_a[i] = i == 0 ? 0 : ts.par[i];
      ts.scr_b[i] = i == 0 ? 0 : 1;
    }
    __syncthreads();
    for (int span = 1; span < N; span <<= 1) {
      int na[kPer], nd[kPer];
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const int i = tid + q * kThreads;
        if (i < N) {
          const int a = ts.scr_a[i];
          nd[q] = ts.scr_b[i] + ts.scr_b[a];
          na[q] = ts.scr_a[a];
        }
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const int i = tid + q * kThreads;
        if (i < N) {
          ts.scr_a[i] = na[q];
          ts.scr_b[i] = nd[q];
        }
      }
      __syncthreads();
    }
    for (int i = tid; i < N; i += kThreads)
      if (ts.scr_b[i] > P.max_depth) atomicOr(&err_s, SPEC_ERR_PARENT);
    __syncthreads();
    if (!kGreedy && err_s == 0) {
      for (int i = tid + 1; i < N; i += kThreads) {
        const long long off = (row0 + ts.par[i]) * P.ld + ts.tk[i];
        ts.u[i] = P.u[row0 + i];
        ts.gp[i] = load_elem(static_cast<const T*>(P.target) + off);
        ts.gq[i] = load_elem(static_cast<const T*>(P.draft) + off);
      }
      if (tid == 0) v_s = P.v[b];
    }
  }
  if constexpr (!kConsulted) {
    pdl_wait();
    merge_stats<kGreedy, false>(G, b, stage, [&](int r, float2 v, bool ok) {
      ts.st[r] = v;
      if (!ok) atomicOr(&err_s, SPEC_ERR_NONFINITE);
    });
  } else {
    (void)stage;
    __syncthreads();
  }
  cluster_ready();

  const int err = err_s;
  const int prefix = P.prefix ? P.prefix[b] : 0;
  const int pn = P.max_depth + 1;
  int* pnodes = P.path_nodes + static_cast<long long>(b) * pn;
  if (err) {
    if (lead) {
      if (tid == 0) {
        P.path_len[b] = 0;
        P.out_token[b] = -1;
        if (P.rollback) P.rollback[b] = prefix;
        if (P.seq_error) P.seq_error[b] = err;
        if (P.error_word) atomicOr(P.error_word, err);
      }
      for (int q = tid; q < pn; q += kThreads) pnodes[q] = -1;
    }
    return;
  }

  const T* target = static_cast<const T*>(P.target);
  const T* draft = static_cast<const T*>(P.draft);
  int* kids = ts.scr_a;
  int* path = ts.scr_b;
  int node = 0, plen = 0, flag = 0, token = -1, buf = 0;
  bool writer = lead;
  // this CTA's tiles; when they fit, a node's rows are loaded into shared
  // memory once and every pass at the node reads them there
  const int ncl = static_cast<int>(cluster_size());
  const int tpc = (G.ntiles + ncl - 1) / ncl;
  const int t0 = min(G.ntiles, static_cast<int>(cluster_rank()) * tpc), t1 = min(G.ntiles, t0 + tpc);
  const bool res_ok = !kGreedy && slice_fits<T>(tpc);
  // greedy consulted: the target row alone is resident when it fits
  const bool res_one = kGreedy && kConsulted && static_cast<size_t>(tpc) * kTileElems * sizeof(T) <= kStageBytes &&
                       tpc <= kResidentTiles;
  while (true) {
    const int nk = list_children(ts.par, N, node, kids, &nk_s);
    // the statistics of node's rows: from the statistics kernel, or computed
    // here (consulted-only) for the rows the walk reads at this node
    float2 sp_node{0.f, 0.f}, sq_node{0.f, 0.f};
    int best_node = -1;
    bool resident_entry = false;
    if constexpr (kConsulted) {
      const T* prow = static_cast<const T*>(P.target) + (row0 + node) * P.ld;
      const T* qrow = static_cast<const T*>(P.draft) + (row0 + node) * P.ld;
      bool bad = false;
      if constexpr (kGreedy) {
        ArgMax am;
        bool lbad = false;
        if (res_one) {
          PassSpec<T> L = make_spec(prow, 0.f, 1.f, static_cast<const T*>(nullptr), 0.f, 1.f, 0.f, 1.f);
          slice_load(L, false, P.V, t0, t1, ps);
          am = resident_row_argmax<T>(t0, t1 - t0, ps, &lbad);
        } else {
          am = direct_row_argmax<T>(prow, P.V, t0, t1, ps, &lbad);
        }
        const int xb = cluster_share4(am.v, __int_as_float(am.i), lbad ? 1.f : 0.f, 0.f, ps);
        const ArgMax all = merge_shared_argmax(xb, ps, &bad);
        bad |= all.i < 0;
        best_node = all.i;
      } else {
        const bool with_q = nk > 0;
        MaxSum part[2];
        if (res_ok) {
          PassSpec<T> L = make_spec(prow, 0.f, 1.f, with_q ? qrow : static_cast<const T*>(nullptr), 0.f, 1.f, 1.f, c);
          slice_load(L, with_q, P.V, t0, t1, ps);
          resident_entry = true;
          resident_row_stats<T>(with_q, t1 - t0, c, ps, part);
        } else {
          streamed_row_stats<T>(prow, with_q ? qrow : nullptr, P.V, c, t0, t1, ps, part);
        }
        const int xb = cluster_share4(part[0].m, part[0].s, part[1].m, part[1].s, ps);
        MaxSum st2[2];
        merge_shared_ms2(xb, c, ps, st2);
        bad = !row_stats_ok(st2[0]) || (with_q && !row_stats_ok(st2[1]));
        sp_node = make_float2(st2[0].m, st2[0].s);
        sq_node = make_float2(st2[1].m, st2[1].s);
      }
      if (bad) {  // a row the walk reads is not finite: empty outputs
        if (lead) {
          if (tid == 0) {
            P.path_len[b] = 0;
            P.out_token[b] = -1;
            if (P.rollback) P.rollback[b] = prefix;
            if (P.seq_error) P.seq_error[b] = SPEC_ERR_NONFINITE;
            if (P.error_word) atomicOr(P.error_word, SPEC_ERR_NONFINITE);
          }
          for (int q = tid; q < pn; q += kThreads) pnodes[q] = -1;
        }
        return;
      }
    } else {
      sp_node = ts.st[node];
      sq_node = ts.st[N + node];
      best_node = __float_as_int(ts.st[node].y);
    }
    if (!kGreedy && !kConsulted && res_ok && tid < nk) {
      // whichever child is kept next, its rows' slice of this CTA will come
      // from L2: hint the bulk-copy engine to bring every child's in now
      // (not in consulted-only mode, which reads no row off the path)
      const int ch = kids[tid];
      const T* cp = target + (row0 + ch) * P.ld;
      const T* cq = draft + (row0 + ch) * P.ld;
      const int tf = min(t1, P.V / kTileElems);
      if (tf > t0 && row_is_aligned(cp) && row_is_aligned(cq)) {
        const unsigned bytes = static_cast<unsigned>((tf - t0) * kTileElems * sizeof(T));
        prefetch_l2(cp + static_cast<long long>(t0) * kTileElems, bytes);
        prefetch_l2(cq + static_cast<long long>(t0) * kTileElems, bytes);
      }
    }
    if constexpr (kGreedy) {
      const int best = best_node;
      int kept = -1;
      for (int q = 0; q < nk; ++q)
        if (ts.tk[kids[q]] == best) {
          kept = kids[q];
          break;
        }
      __syncthreads();  // kids[] is rewritten by the next list_children
      if (kept < 0) {
        token = best;
        break;
      }
      if (tid == 0) path[plen] = kept;
      ++plen;
      node = kept;
    } else {
      const float2 sp = sp_node;
      const float2 sq = sq_node;
      PassSpec<T> S = make_spec(target + (row0 + node) * P.ld, sp.x, sp.y, draft + (row0 + node) * P.ld, sq.x,
                                sq.y, 1.f, c);
      S.cq = 0.f;
      double cc = 0.0, W = 1.0;
      DF Wdf{1.f, 0.f};
      int kept = -1;
      bool zero_mass = false, resident = resident_entry;
      for (int q = 0; q < nk; ++q) {
        const int ch = kids[q];
        if (tid == 0) {
          // sibling test u < min(1, r) with r = max(0, p - c_k q) / (W_k q) at
          // the child's token; since u < 1 it is u W_k q < max(0, p - c_k q),
          // which needs no division and keeps exactly when p - c_k q > 0 if
          // q = 0
          const double pt = prob(ts.gp[ch], sp.x, sp.y, c);
          const double qt = prob(ts.gq[ch], sq.x, sq.y, c);
          const double num = fmax(0.0, pt - cc * qt);
          keep_s = static_cast<double>(ts.u[ch]) * W * qt < num;
        }
        __syncthreads();
        if (keep_s) {
          kept = ch;
          break;
        }
        const double cn = cc + W;
        S.cq = static_cast<float>(cn);
        buf ^= 1;
        if (res_ok && !resident) {
          slice_load(S, true, P.V, t0, t1, ps);
          resident = true;
        }
        const DF Wn = cluster_pass(S, P.V, c, G.ntiles, buf, ps, res_ok);
        if (!pass_ok(Wn)) {
          zero_mass = true;
          break;
        }
        cc = cn;
        W = df_double(Wn);
        Wdf = Wn;
      }
      __syncthreads();  // kids[] is rewritten by the next list_children
      if (kept >= 0) {
        if (tid == 0) path[plen] = kept;
        ++plen;
        node = kept;
        continue;
      }
      DF Z = Wdf;
      if (zero_mass || nk == 0) {
        if (zero_mass) flag = SPEC_ERR_ZERO_MASS;
        S.cq = 0.f;  // draw from the node's own target distribution
        buf ^= 1;
        if (res_ok && !resident) {
          slice_load(S, false, P.V, t0, t1, ps);
          resident = true;
        }
        Z = cluster_pass(S, P.V, c, G.ntiles, buf, ps, res_ok);
      }
      token = cluster_draw(S, P.V, c, G.ntiles, buf, df_mul_f(Z, v_s), false, ps, res_ok);
      writer = token >= 0;
      break;
    }
  }
  __syncthreads();
  if (!writer) return;
  if (ps.fault) {  // a bounded wait gave up: empty outputs
    flag |= SPEC_ERR_INTERNAL;
    token = -1;
    plen = 0;
  }
  if (tid == 0) {
    P.out_token[b] = token;
    P.path_len[b] = plen;
    if (P.rollback) P.rollback[b] = prefix + plen;
    if (P.seq_error) P.seq_error[b] = flag;
    if (flag && P.error_word) atomicOr(P.error_word, flag);
  }
  for (int q = tid; q < pn; q += kThreads)
    pnodes[q] = ps.fault ? -1 : (q == 0 ? 0 : (q <= plen ? path[q - 1] : -1));
}

// ---------------------------------------------------------------------------
// launches
// ---------------------------------------------------------------------------
// Scheduling priority of rank r (0 = most urgent): the device's greatest
// priority for r = 0, one level less per rank, never below the least.
int launch_priority(int r) {
  static int least = 0, greatest = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) least = greatest = 0;
  });
  return min(least, greatest + r);
}

template <typename K>
cudaError_t launch_stats(K kernel, const StatsParams& G, cudaStream_t s, int rank = -1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G.chunks, G.rows_per_seq, G.B);
  cfg.blockDim = dim3(kStatsThreads);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  if (rank >= 0) {
    at[0].id = cudaLaunchAttributePriority;
    at[0].val.priority = launch_priority(rank);
    cfg.attrs = at;
    cfg.numAttrs = 1;
  }
  void* argv[] = {const_cast<StatsParams*>(&G)};
  return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kernel), argv);
}

// Clusters of 1, 2, 4 and 8 CTAs of `fn` that can be resident at once on the
// current device, cached per (kernel, device).
cudaError_t resident_clusters(const void* fn, size_t dyn, std::array<int, 4>* out) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, std::array<int, 4>> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find({fn, dev});
  if (it != cache.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  std::array<int, 4> n{};
  for (int i = 0; i < 4; ++i) {
    const int S = 1 << i;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = dyn;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int count = 0;
    if (cudaOccupancyMaxActiveClusters(&count, fn, &cfg) != cudaSuccess) {
      cudaGetLastError();  // a size the device cannot co-schedule: not used
      count = 0;
    }
    n[i] = count;
  }
  cache[{fn, dev}] = n;
  *out = n;
  return cudaSuccess;
}

// Largest cluster (at most 8 CTAs, at most one per tile) for which all B
// sequences' clusters fit in 7/8 of the clusters the occupancy query reports
// resident at once; 1 when even single CTAs need more than one wave.  The
// margin is for placement: a cluster must fit inside one GPC, and the walk
// is placed while the statistics kernel still drains, so the clusters that
// really fit are fewer than on an empty GPU (a second wave of a few
// clusters costs a whole walk).
int cluster_for(const std::array<int, 4>& resident, int B, int ntiles) {
  for (int i = 3; i >= 1; --i) {
    const int S = 1 << i;
    if (S <= ntiles && 8 * B <= 7 * resident[i]) return S;
  }
  return 1;
}

// A dependent kernel: programmatic stream serialisation lets it start while
// its predecessor drains; it reads the predecessor's results only after
// griddepcontrol.wait.  cluster > 0 launches clusters of that many CTAs
// along x.
// With pdl false the kernel is launched in plain stream order instead (its
// predecessor's results are then visible from its first instruction).
template <typename K, typename A>
cudaError_t launch_dependent(K kernel, dim3 grid, int cluster, size_t dyn, const StatsParams& G, const A& args,
                             cudaStream_t s, int rank = -1, bool pdl = true) {
  const void* fn = reinterpret_cast<const void*>(kernel);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = s;
  cudaLaunchAttribute at[3];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  int na = 1;
  if (cluster > 0) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = cluster;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  if (rank >= 0) {
    at[na].id = cudaLaunchAttributePriority;
    at[na].val.priority = launch_priority(rank);
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  void* argv[] = {const_cast<StatsParams*>(&G), const_cast<A*>(&args)};
  return cudaLaunchKernelExC(&cfg, fn, argv);
}

// Raise a kernel's dynamic shared memory limit to `bytes`, once per
// (kernel, device).
cudaError_t smem_limit(const void* fn, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find({fn, dev});
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[{fn, dev}] = bytes;
  return e;
}

// A sampling walk kernel with one cluster per sequence; `occupancy_dyn` is
// the dynamic shared memory the cluster size is chosen for (at least dyn).
template <typename K, typename A>
cudaError_t launch_walk(K kernel, size_t dyn, size_t occupancy_dyn, const StatsParams& G, const A& args,
                        cudaStream_t s, int rank = -1, bool pdl = true) {
  const void* fn = reinterpret_cast<const void*>(kernel);
  cudaError_t e = smem_limit(fn, static_cast<int>(occupancy_dyn));
  if (e != cudaSuccess) return e;
  std::array<int, 4> resident;
  e = resident_clusters(fn, occupancy_dyn, &resident);
  if (e != cudaSuccess) return e;
  const int S = cluster_for(resident, G.B, G.ntiles);
  return launch_dependent(kernel, dim3(S, G.B), S, dyn, G, args, s, rank, pdl);
}

// The resident-slice chain walk, used when the cluster the staged walk would
// get (same occupancy rule, same dynamic shared memory) holds its slices in
// the stage region; otherwise the staged walk.  A larger resident region was
// measured: alone, a 64 KB slice per CTA (V = 128256, clusters of 8) made the
// walk faster (18.3 against 21.6 us), but as the last of four batch groups
// the call took 54.7 instead of 44.6 us: clusters of CTAs that large are
// placed late beside the other groups' statistics and walks.

template <typename T>
cudaError_t launch_chain_walk_resident(const StatsParams& G, const ChainParams& args, cudaStream_t s, int rank) {
  const void* fn = reinterpret_cast<const void*>(chain_walk_kernel<T, true>);
  cudaError_t e = smem_limit(fn, kStageBytes);
  if (e != cudaSuccess) return e;
  std::array<int, 4> resident;
  e = resident_clusters(fn, kStageBytes, &resident);
  if (e != cudaSuccess) return e;
  const int S = cluster_for(resident, G.B, G.ntiles);
  if (slice_bytes<T>((G.ntiles + S - 1) / S) <= static_cast<size_t>(kStageBytes) &&
      (G.ntiles + S - 1) / S <= kResidentTiles)
    return launch_dependent(chain_walk_kernel<T, true>, dim3(S, G.B), S, kStageBytes, G, args, s, rank);
  return launch_walk(chain_walk_kernel<T, false>, kStageBytes, kStageBytes, G, args, s, rank);
}

// ---------------------------------------------------------------------------
// batch groups: large calls are split into up to kMaxGroups groups of
// sequences, each verified by its own statistics kernel and walk on a
// library-owned stream forked from (and joined back into) the caller's
// stream.  The statistics kernels of all groups stream back to back, and
// each group's walk runs as soon as that group's statistics are complete,
// alongside the statistics of the later groups; only the last group's walk
// is left after the logits have been read.  A group is a smaller batch:
// its pointers are offsets into the caller's arrays and its partials a
// disjoint part of the workspace.
// ---------------------------------------------------------------------------
constexpr int kMaxGroups = 4;
constexpr double kGroupBytes = 40e6;  // logits per group at least
constexpr int kGroupSeqs = 16;        // sequences per group at least
constexpr int kTreeGroupSeqs = 4;     // trees per group at least (a tree holds 2N rows)

struct Groups {
  int n;
  int b0[kMaxGroups + 1];
};

Groups plan_groups(int B, double bytes, int min_seqs = kGroupSeqs) {
  Groups g{};
  int n = min(kMaxGroups, B / min_seqs);
  n = min(n, static_cast<int>(bytes / kGroupBytes));
  g.n = max(n, 1);
  for (int i = 0; i <= g.n; ++i) g.b0[i] = static_cast<int>((static_cast<long long>(B) * i) / g.n);
  return g;
}

// Library streams and events of the calling host thread on the current
// device: one side stream per group, the fork event and one join event per
// group.  They are created on the thread's first grouped call on the device
// and reused by its later calls, so a call creates nothing; keeping them per
// thread means that calls from different host threads never share a side
// stream (one thread capturing a call into a graph cannot pull another
// thread's eager call into its capture).  They are released when the thread
// exits.
struct GroupResources {
  cudaStream_t side[kMaxGroups];
  cudaEvent_t fork;
  cudaEvent_t join[kMaxGroups];
};

struct ThreadGroupResources {
  std::map<int, GroupResources> per_device;
  ~ThreadGroupResources() {
    for (auto& kv : per_device) {
      int cur = 0;
      if (cudaGetDevice(&cur) != cudaSuccess) return;  // the runtime is already gone
      if (cudaSetDevice(kv.first) != cudaSuccess) continue;
      for (int i = 0; i < kMaxGroups; ++i) {
        cudaStreamDestroy(kv.second.side[i]);
        cudaEventDestroy(kv.second.join[i]);
      }
      cudaEventDestroy(kv.second.fork);
      cudaSetDevice(cur);
    }
  }
};

cudaError_t group_resources(GroupResources** out) {
  thread_local ThreadGroupResources mine;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  auto it = mine.per_device.find(dev);
  if (it == mine.per_device.end()) {
    GroupResources r{};
    for (int i = 0; i < kMaxGroups && e == cudaSuccess; ++i) {
      e = cudaStreamCreateWithFlags(&r.side[i], cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.join[i], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.fork, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;  // (a partial set is not kept)
    it = mine.per_device.emplace(dev, r).first;
  }
  *out = &it->second;
  return cudaSuccess;
}

// Fork the caller's stream into one library stream per group, run
// launch_group(i, stream) on each, and join them back.  The join is recorded
// even when a launch fails, so the caller's stream never runs ahead of work
// that was enqueued.
template <typename F>
cudaError_t run_groups(const Groups& gr, cudaStream_t s, F launch_group) {
  GroupResources* r = nullptr;
  cudaError_t e = group_resources(&r);
  if (e != cudaSuccess) return e;
  e = cudaEventRecord(r->fork, s);
  cudaError_t first = e;
  for (int i = 0; i < gr.n && first == cudaSuccess; ++i) {
    e = cudaStreamWaitEvent(r->side[i], r->fork, 0);
    if (e == cudaSuccess) e = launch_group(i, r->side[i]);
    if (e != cudaSuccess) first = e;
    if (cudaEventRecord(r->join[i], r->side[i]) == cudaSuccess) {
      e = cudaStreamWaitEvent(s, r->join[i], 0);
      if (e != cudaSuccess && first == cudaSuccess) first = e;
    }
  }
  return first;
}

template <typename T>
StatsParams stats_group(const StatsParams& G, int b0, int nb) {
  StatsParams g = G;
  g.B = nb;
  for (int k = 0; k < G.nsets; ++k)
    g.set[k].base = static_cast<const T*>(G.set[k].base) + static_cast<long long>(b0) * G.set[k].rows * G.ld;
  g.partials = G.partials + static_cast<long long>(b0) * G.rows_per_seq * G.chunks;
  return g;
}

template <typename X>
X* at_seq(X* p, int b0, long long per) {
  return p ? p + static_cast<long long>(b0) * per : nullptr;
}

template <typename T>
ChainParams chain_group(const ChainParams& p, int b0, int nb) {
  ChainParams g = p;
  const long long gam = p.gamma;
  g.B = nb;
  g.target = static_cast<const T*>(p.target) + static_cast<long long>(b0) * (gam + 1) * p.ld;
  g.draft = p.draft ? static_cast<const T*>(p.draft) + static_cast<long long>(b0) * gam * p.ld : nullptr;
  g.tokens = at_seq(p.tokens, b0, gam);
  g.u = at_seq(p.u, b0, gam);
  g.v = at_seq(p.v, b0, 1);
  g.prefix = at_seq(p.prefix, b0, 1);
  g.accept_len = at_seq(p.accept_len, b0, 1);
  g.out_token = at_seq(p.out_token, b0, 1);
  g.rollback = at_seq(p.rollback, b0, 1);
  g.p_at = at_seq(p.p_at, b0, gam);
  g.q_at = at_seq(p.q_at, b0, gam);
  g.resid = at_seq(p.resid, b0, 1);
  g.seq_error = at_seq(p.seq_error, b0, 1);
  return g;
}

template <typename T>
TreeParams tree_group(const TreeParams& p, int b0, int nb) {
  TreeParams g = p;
  const long long n = p.N;
  g.B = nb;
  g.target = static_cast<const T*>(p.target) + static_cast<long long>(b0) * n * p.ld;
  g.draft = p.draft ? static_cast<const T*>(p.draft) + static_cast<long long>(b0) * n * p.ld : nullptr;
  g.parent = at_seq(p.parent, b0, n);
  g.tokens = at_seq(p.tokens, b0, n);
  g.u = at_seq(p.u, b0, n);
  g.v = at_seq(p.v, b0, 1);
  g.prefix = at_seq(p.prefix, b0, 1);
  g.path_len = at_seq(p.path_len, b0, 1);
  g.path_nodes = at_seq(p.path_nodes, b0, p.max_depth + 1);
  g.out_token = at_seq(p.out_token, b0, 1);
  g.rollback = at_seq(p.rollback, b0, 1);
  g.seq_error = at_seq(p.seq_error, b0, 1);
  return g;
}

double logit_bytes(const StatsParams& G, size_t elt) {
  return static_cast<double>(G.B) * G.rows_per_seq * G.V * static_cast<double>(elt);
}

// One group: its statistics, then its walk.  With group >= 0 the launches
// carry priorities: every walk above every statistics kernel, and the
// statistics of earlier groups above later ones, so that groups finish
// their statistics in order and each walk starts as soon as it can.
// `last`: no statistics kernel of this call runs after this group's, so its
// walk takes the resident-slice form.
template <typename T>
cudaError_t chain_one(const StatsParams& G, const ChainParams& p, bool greedy, cudaStream_t s, int group,
                      bool last) {
  const int sr = group < 0 ? -1 : 1 + group, wr = group < 0 ? -1 : 0;
  cudaError_t e = greedy ? launch_stats(stats_kernel<T, true>, G, s, sr) : launch_stats(stats_kernel<T, false>, G, s, sr);
  if (e != cudaSuccess) return e;
  if (greedy) return launch_dependent(chain_greedy_kernel<T>, dim3(G.B), 0, 0, G, p, s, wr);
  if (last) return launch_chain_walk_resident<T>(G, p, s, wr);
  return launch_walk(chain_walk_kernel<T, false>, kStageBytes, kStageBytes, G, p, s, wr);
}

template <typename T>
cudaError_t chain_consulted(const StatsParams& G, const ChainParams& p, cudaStream_t s) {
  return launch_walk(chain_consulted_kernel<T>, kStageBytes, kStageBytes, G, p, s);
}

template <typename T>
cudaError_t chain_impl(const StatsParams& G, const ChainParams& p, bool greedy, bool grouped, bool consulted,
                       cudaStream_t s) {
  if (consulted) return chain_consulted<T>(G, p, s);
  const Groups gr = plan_groups(G.B, logit_bytes(G, sizeof(T)));
  if (!grouped || gr.n == 1) return chain_one<T>(G, p, greedy, s, -1, true);
  return run_groups(gr, s, [&](int i, cudaStream_t si) {
    const int b0 = gr.b0[i], nb = gr.b0[i + 1] - b0;
    return chain_one<T>(stats_group<T>(G, b0, nb), chain_group<T>(p, b0, nb), greedy, si, i, i == gr.n - 1);
  });
}

// One group of trees: its statistics, then its walk (priorities as for the
// chain's groups).
template <typename T>
cudaError_t tree_one(const StatsParams& G, const TreeParams& p, bool greedy, cudaStream_t s, int group) {
  const int sr = group < 0 ? -1 : 1 + group, wr = group < 0 ? -1 : 0;
  const size_t nodes = static_cast<size_t>(kTreeSmemPerNode) * p.N;
  const size_t most = static_cast<size_t>(kStageBytes) + static_cast<size_t>(kTreeSmemPerNode) * kMaxNodes;
  cudaError_t e = greedy ? launch_stats(stats_kernel<T, true>, G, s, sr) : launch_stats(stats_kernel<T, false>, G, s, sr);
  if (e != cudaSuccess) return e;
  if (greedy) {
    e = smem_limit(reinterpret_cast<const void*>(tree_kernel<T, true, false>), kTreeSmemPerNode * kMaxNodes);
    if (e != cudaSuccess) return e;
    return launch_dependent(tree_kernel<T, true, false>, dim3(1, G.B), 0, nodes, G, p, s, wr);
  }
  return launch_walk(tree_kernel<T, false, false>, kStageBytes + nodes, most, G, p, s, wr);
}

template <typename T>
cudaError_t tree_impl(const StatsParams& G, const TreeParams& p, bool greedy, bool consulted, cudaStream_t s) {
  const size_t nodes = static_cast<size_t>(kTreeSmemPerNode) * p.N;
  // occupancy is evaluated once, at the largest tree's shared memory
  const size_t most = static_cast<size_t>(kStageBytes) + static_cast<size_t>(kTreeSmemPerNode) * kMaxNodes;
  if (consulted) {  // one kernel: the walk computes the statistics it reads
    if (greedy) return launch_walk(tree_kernel<T, true, true>, kStageBytes + nodes, most, G, p, s);
    return launch_walk(tree_kernel<T, false, true>, kStageBytes + nodes, most, G, p, s);
  }
  const Groups gr = plan_groups(G.B, logit_bytes(G, sizeof(T)), kTreeGroupSeqs);
  if (gr.n == 1) return tree_one<T>(G, p, greedy, s, -1);
  return run_groups(gr, s, [&](int i, cudaStream_t si) {
    const int b0 = gr.b0[i], nb = gr.b0[i + 1] - b0;
    return tree_one<T>(stats_group<T>(G, b0, nb), tree_group<T>(p, b0, nb), greedy, si, i);
  });
}

template <typename T>
cudaError_t cascade_one(const StatsParams& G, const CascadeParams& p, bool greedy, cudaStream_t s, int group) {
  const int sr = group < 0 ? -1 : 1 + group, wr = group < 0 ? -1 : 0;
  cudaError_t e = greedy ? launch_stats(stats_kernel<T, true>, G, s, sr) : launch_stats(stats_kernel<T, false>, G, s, sr);
  if (e != cudaSuccess) return e;
  if (greedy) return launch_dependent(cascade_greedy_kernel<T>, dim3(G.B), 0, 0, G, p, s, wr);
  return launch_walk(cascade_walk_kernel<T>, kStageBytes, kStageBytes, G, p, s, wr);
}

// The cascade is not split into groups: its walk (two passes per sequence)
// holds the SMs long enough that running it beside later groups'
// statistics costs more than it hides.
template <typename T>
cudaError_t cascade_impl(const StatsParams& G, const CascadeParams& p, bool greedy, cudaStream_t s) {
  return cascade_one<T>(G, p, greedy, s, -1);
}

template <typename T>
cudaError_t pipeline_impl(const StatsParams& G, const PipelineParams& p, bool greedy, cudaStream_t s) {
  cudaError_t e = greedy ? launch_stats(stats_kernel<T, true>, G, s) : launch_stats(stats_kernel<T, false>, G, s);
  if (e != cudaSuccess) return e;
  if (greedy) return launch_dependent(pipeline_greedy_kernel<T>, dim3(G.B), 0, 0, G, p, s);
  return launch_walk(pipeline_walk_kernel<T>, kStageBytes, kStageBytes, G, p, s);
}

}  // namespace

cudaError_t launch_pipeline(const StatsParams& G, const PipelineParams& p, bool bf16, bool greedy, cudaStream_t s) {
  return bf16 ? pipeline_impl<bf16_t>(G, p, greedy, s) : pipeline_impl<float>(G, p, greedy, s);
}

int stats_chunks(int V, bool bf16) {
  const int ce = bf16 ? chunk_elems<bf16_t>() : chunk_elems<float>();
  return (V + ce - 1) / ce;
}

int pass_tiles(int V) { return (V + kTileElems - 1) / kTileElems; }

cudaError_t launch_chain(const StatsParams& G, const ChainParams& p, bool bf16, bool greedy, bool grouped,
                         bool consulted, cudaStream_t s) {
  return bf16 ? chain_impl<bf16_t>(G, p, greedy, grouped, consulted, s)
              : chain_impl<float>(G, p, greedy, grouped, consulted, s);
}

cudaError_t launch_tree(const StatsParams& G, const TreeParams& p, bool bf16, bool greedy, bool consulted,
                        cudaStream_t s) {
  return bf16 ? tree_impl<bf16_t>(G, p, greedy, consulted, s) : tree_impl<float>(G, p, greedy, consulted, s);
}

cudaError_t launch_cascade(const StatsParams& G, const CascadeParams& p, bool bf16, bool greedy, cudaStream_t s) {
  return bf16 ? cascade_impl<bf16_t>(G, p, greedy, s) : cascade_impl<float>(G, p, greedy, s);
}

cudaError_t launch_chain_walk_f32(const StatsParams& G, const ChainParams& p, bool greedy, cudaStream_t s) {
  // plain stream order: the walk reads the logits at the drafted tokens
  // before it waits, and here those logits come from the preceding kernel
  if (greedy) return launch_dependent(chain_greedy_kernel<float, true>, dim3(G.B), 0, 0, G, p, s, -1, false);
  return launch_walk(chain_walk_kernel<float, false, true>, kStageBytes, kStageBytes, G, p, s, -1, false);
}

}  // namespace sv

extern "C" spec_status spec_test_inject_copy_timeout(int enable) {
  const int v = enable ? 1 : 0;
  return cudaMemcpyToSymbol(sv::g_copy_timeout_test, &v, sizeof(v)) == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}
