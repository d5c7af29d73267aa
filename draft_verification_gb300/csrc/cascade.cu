// PipeSpec 3-model cascade, one synchronous snapshot of the pipeline.
//
// Pith review of PipeSpec (2505.01572), "What carries the argument": model
// M_i reads buffer O_{i-1}, verifies it against its own prediction, appends
// the longest matching prefix to O_i and, on a mismatch, makes the earlier
// stages roll back to the last verified token.  Staged Speculative Decoding
// (2308.04623), abstract: a second speculative stage.
//
// Stage 1: M_1 verifies the gamma1 tokens of O_0 with the chain rule
// (p = M_1, q = M_0): a1 kept, t1 = the correction or the bonus from M_1's
// row gamma1; O_1 = d[0..a1) ++ t1.  Stage 2: M_2 verifies the first
// w2 = min(gamma2, a1 + 1) tokens of O_1 (p = M_2, q = M_1): a2 kept; a
// rejection draws t2 from max(0, p2 - p1); keeping all w2 draws nothing
// (M_2's next row would be conditioned on tokens it has not seen).  A
// final-stage rejection rolls O_0 back to min(a1, a2).
//
// Rows per sequence in the statistics workspace: sampling: M_0 rows
// [0, g1), M_1 rows [g1, 2 g1 + 1), M_2 rows [2 g1 + 1, 2 g1 + 1 + g2);
// greedy (M_0 is not read): M_1 rows [0, g1 + 1), M_2 rows [g1 + 1, ...).
#include "common.cuh"
#include "internal.h"
#include "spec_verify.h"
#include "walk.cuh"

namespace sv {
namespace {

constexpr int kMaxG = 32;
constexpr int kMaxRows = 3 * kMaxG + 1;

template <typename T, bool kGreedy>
__global__ void __launch_bounds__(kThreads) cascade_walk_kernel(const CascadeParams P) {
  cg::cluster_group cl = cg::this_cluster();
  const int cs = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / cs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g1 = P.g1, g2 = P.g2;
  const float c = P.c;
  // statistics row of M_0 row j / M_1 row j / M_2 row j
  const int r1 = kGreedy ? 0 : g1;
  const int r2 = r1 + g1 + 1;

  __shared__ PassShared sh;
  __shared__ float2 st[kMaxRows];
  __shared__ int tok[kMaxG];
  __shared__ int o1[kMaxG + 1];
  __shared__ int err_s, a1_s, a2_s;
  if (tid == 0) {
    sh.parity = 0;
    sh.sparity = 0;
    err_s = 0;
  }
  __syncthreads();
  pdl_wait();

  if (tid < g1) {
    const int t = P.tokens[static_cast<long long>(b) * g1 + tid];
    tok[tid] = t;
    if (t < 0 || t >= P.V) atomicOr(&err_s, SPEC_ERR_TOKEN);
  }
  const float2* part = P.partials + static_cast<long long>(b) * P.rows_per_seq * P.chunks;
  for (int r = warp; r < P.rows_per_seq; r += kWarps) {
    if constexpr (kGreedy) {
      bool bad;
      const ArgMax am = combine_row_argmax(part + static_cast<long long>(r) * P.chunks, P.chunks, bad);
      if (lane == 0) {
        st[r] = make_float2(0.f, __int_as_float(am.i));
        if (bad || am.i < 0) atomicOr(&err_s, SPEC_ERR_NONFINITE);
      }
    } else {
      const MaxSum ms = combine_row(part + static_cast<long long>(r) * P.chunks, P.chunks, c);
      if (lane == 0) {
        st[r] = make_float2(ms.m, ms.s);
        if (!row_stats_ok(ms)) atomicOr(&err_s, SPEC_ERR_NONFINITE);
      }
    }
  }
  __syncthreads();

  const int err = err_s;
  const int base0 = P.base0 ? P.base0[b] : 0;
  const int base1 = P.base1 ? P.base1[b] : 0;
  auto write_out = [&](int a1, int t1, int a2, int w2, int t2, int t2v, int flag) {
    const bool rej = a2 < w2;
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
  };
  if (err) {
    if (rank == 0 && tid == 0) write_out(0, -1, 0, 0, -1, 0, err);
    return;
  }

  if constexpr (kGreedy) {
    if (tid == 0 && rank == 0) {
      int a1 = g1;
      for (int j = 0; j < g1; ++j)
        if (tok[j] != __float_as_int(st[r1 + j].y)) {
          a1 = j;
          break;
        }
      const int t1 = __float_as_int(st[r1 + a1].y);
      const int w2 = min(g2, a1 + 1);
      int a2 = w2;
      for (int j = 0; j < w2; ++j) {
        const int o = j < a1 ? tok[j] : t1;
        if (o != __float_as_int(st[r2 + j].y)) {
          a2 = j;
          break;
        }
      }
      const int t2 = a2 < w2 ? __float_as_int(st[r2 + a2].y) : -1;
      write_out(a1, t1, a2, w2, t2, a2 < w2 ? 1 : 0, 0);
    }
    return;
  } else {
    const T* L0 = static_cast<const T*>(P.l0);
    const T* L1 = static_cast<const T*>(P.l1);
    const T* L2 = static_cast<const T*>(P.l2);
    const long long b0 = static_cast<long long>(b) * g1;        // first M_0 row of b
    const long long b1 = static_cast<long long>(b) * (g1 + 1);  // first M_1 row
    const long long b2 = static_cast<long long>(b) * g2;        // first M_2 row
    int flag = 0;

    // stage 1: M_1 verifies O_0 against M_0
    if (warp == 0) {
      bool keep = true;
      if (lane < g1) {
        const int d = tok[lane];
        const float xp = load_elem(L1 + (b1 + lane) * P.ld + d);
        const float xq = load_elem(L0 + (b0 + lane) * P.ld + d);
        const double lp = log2_prob(xp, st[r1 + lane].x, st[r1 + lane].y, c);
        const double lq = log2_prob(xq, st[lane].x, st[lane].y, c);
        keep = keeps(P.u1[b0 + lane], accept_ratio(lp, lq));
      }
      const unsigned rej = __ballot_sync(0xffffffffu, lane < g1 && !keep);
      if (lane == 0) a1_s = rej ? __ffs(rej) - 1 : g1;
    }
    __syncthreads();
    const int a1 = a1_s;
    PassSpec<T> S;
    S.P = L1 + (b1 + a1) * P.ld;
    S.MP = scaled_max(st[r1 + a1].x, c);
    S.invSP = __fdiv_rn(1.f, st[r1 + a1].y);
    if (a1 < g1) {
      S.Q = L0 + (b0 + a1) * P.ld;
      S.MQ = scaled_max(st[a1].x, c);
      S.invSQ = __fdiv_rn(1.f, st[a1].y);
      S.cq = 1.f;
    } else {
      S.Q = nullptr;
      S.MQ = S.invSQ = 0.f;
      S.cq = 0.f;
    }
    double Z = run_pass(S, P.V, c, sh, cl);
    if (!(Z > 0.0) || !(Z < INFINITY)) {
      flag = SPEC_ERR_ZERO_MASS;
      S.cq = 0.f;
      Z = run_pass(S, P.V, c, sh, cl);
    }
    int owner = run_search(S, P.V, c, static_cast<double>(P.v1[b]) * Z, sh, cl);
    cl.sync();
    const int t1 = fetch_result(sh, owner, cl);

    // stage 2: M_2 verifies the first w2 tokens of O_1 against M_1
    const int w2 = min(g2, a1 + 1);
    if (tid <= a1 && tid < kMaxG + 1) o1[tid] = tid < a1 ? tok[tid] : t1;
    __syncthreads();
    if (warp == 0) {
      bool keep = true;
      if (lane < w2) {
        const int o = o1[lane];
        const float xp = load_elem(L2 + (b2 + lane) * P.ld + o);
        const float xq = load_elem(L1 + (b1 + lane) * P.ld + o);
        const double lp = log2_prob(xp, st[r2 + lane].x, st[r2 + lane].y, c);
        const double lq = log2_prob(xq, st[r1 + lane].x, st[r1 + lane].y, c);
        keep = keeps(P.u2[static_cast<long long>(b) * g2 + lane], accept_ratio(lp, lq));
      }
      const unsigned rej = __ballot_sync(0xffffffffu, lane < w2 && !keep);
      if (lane == 0) a2_s = rej ? __ffs(rej) - 1 : w2;
    }
    __syncthreads();
    const int a2 = a2_s;
    int t2 = -1, t2v = 0;
    owner = -1;
    if (a2 < w2) {
      PassSpec<T> S2;
      S2.P = L2 + (b2 + a2) * P.ld;
      S2.MP = scaled_max(st[r2 + a2].x, c);
      S2.invSP = __fdiv_rn(1.f, st[r2 + a2].y);
      S2.Q = L1 + (b1 + a2) * P.ld;
      S2.MQ = scaled_max(st[r1 + a2].x, c);
      S2.invSQ = __fdiv_rn(1.f, st[r1 + a2].y);
      S2.cq = 1.f;
      double Z2 = run_pass(S2, P.V, c, sh, cl);
      if (!(Z2 > 0.0) || !(Z2 < INFINITY)) {
        flag = SPEC_ERR_ZERO_MASS;
        S2.cq = 0.f;
        Z2 = run_pass(S2, P.V, c, sh, cl);
      }
      owner = run_search(S2, P.V, c, static_cast<double>(P.v2[b]) * Z2, sh, cl);
      t2v = 1;
    }
    cl.sync();
    if (owner >= 0) t2 = fetch_result(sh, owner, cl);
    if (rank == 0 && tid == 0) write_out(a1, t1, a2, w2, t2, t2v, flag);
    cl.sync();  // remote readers are done before any CTA exits
  }
}

}  // namespace

cudaError_t launch_cascade_walk(const CascadeParams& p, bool bf16, bool greedy, cudaStream_t s) {
  void* args[] = {const_cast<CascadeParams*>(&p)};
  const void* k;
  if (bf16) k = greedy ? reinterpret_cast<const void*>(&cascade_walk_kernel<bf16_t, true>)
                       : reinterpret_cast<const void*>(&cascade_walk_kernel<bf16_t, false>);
  else k = greedy ? reinterpret_cast<const void*>(&cascade_walk_kernel<float, true>)
                  : reinterpret_cast<const void*>(&cascade_walk_kernel<float, false>);
  return launch_walker(k, args, p.B, greedy ? 1 : p.cluster, 0, s);
}

}  // namespace sv
