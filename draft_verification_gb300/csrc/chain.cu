// Chain verification: decide, per sequence, how many of the gamma drafted
// tokens are kept and draw the correction or bonus token.
//
// PipeSpec review (pith.science 2505.01572), "What carries the argument":
// keep the longest prefix that matches, roll back to the last verified
// token.  The accept test and residual are the speculative-sampling rule of
// Leviathan et al. that its Circularity Check cites: keep draft d_i while
// u_i < min(1, p_i(d_i)/q_i(d_i)); at the first rejection a draw from
// max(0, p_a - q_a); if all are kept, a draw from the bonus row p_gamma.
// Greedy (the review's "Reading between the lines": temperature 0): keep
// while d_i equals the target argmax, emit the argmax where the chain stops.
//
// One cluster per sequence.  Every CTA merges the row statistics of its
// sequence and evaluates the gamma accept tests (a ballot finds the first
// rejection); the cluster then runs one pass over the selected row pair and
// the inverse-CDF draw (walk.cuh).
#include "common.cuh"
#include "internal.h"
#include "spec_verify.h"
#include "walk.cuh"

namespace sv {
namespace {

constexpr int kMaxGamma = 32;

template <typename T, bool kGreedy>
__global__ void __launch_bounds__(kThreads) chain_walk_kernel(const ChainParams P) {
  cg::cluster_group cl = cg::this_cluster();
  const int cs = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / cs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = P.gamma;
  const float c = P.c;

  __shared__ PassShared sh;
  __shared__ float st_m[2 * kMaxGamma + 1];
  __shared__ float st_s[2 * kMaxGamma + 1];
  __shared__ int st_arg[kMaxGamma + 1];
  __shared__ int tok[kMaxGamma];
  __shared__ int err_s;
  __shared__ int a_s;
  if (tid == 0) {
    sh.parity = 0;
    sh.sparity = 0;
    err_s = 0;
  }
  __syncthreads();

  pdl_wait();  // the statistics grid has finished and its writes are visible

  if (tid < g) {
    const int t = P.tokens[static_cast<long long>(b) * g + tid];
    tok[tid] = t;
    if (t < 0 || t >= P.V) atomicOr(&err_s, SPEC_ERR_TOKEN);
  }
  const float2* part = P.partials + static_cast<long long>(b) * P.rows_per_seq * P.chunks;
  for (int r = warp; r < P.rows_per_seq; r += kWarps) {
    if constexpr (kGreedy) {
      bool bad;
      const ArgMax am = combine_row_argmax(part + static_cast<long long>(r) * P.chunks, P.chunks, bad);
      if (lane == 0) {
        st_arg[r] = am.i;
        if (bad || am.i < 0) atomicOr(&err_s, SPEC_ERR_NONFINITE);
      }
    } else {
      const MaxSum ms = combine_row(part + static_cast<long long>(r) * P.chunks, P.chunks, c);
      if (lane == 0) {
        st_m[r] = ms.m;
        st_s[r] = ms.s;
        if (!row_stats_ok(ms)) atomicOr(&err_s, SPEC_ERR_NONFINITE);
      }
    }
  }
  __syncthreads();

  const int err = err_s;
  const int prefix = P.prefix ? P.prefix[b] : 0;
  if (err) {  // data error: empty outputs, no draw
    if (rank == 0) {
      if (tid == 0) {
        P.accept_len[b] = 0;
        P.out_token[b] = -1;
        if (P.rollback) P.rollback[b] = prefix;
        if (P.resid) P.resid[b] = 0.f;
        if (P.seq_error) P.seq_error[b] = err;
        if (P.error_word) atomicOr(P.error_word, err);
      }
      if (tid < g) {
        if (P.p_at) P.p_at[static_cast<long long>(b) * g + tid] = 0.f;
        if (P.q_at) P.q_at[static_cast<long long>(b) * g + tid] = 0.f;
      }
    }
    return;  // no distributed shared memory was touched
  }

  if constexpr (kGreedy) {
    if (warp == 0) {
      const bool miss = lane < g && tok[lane] != st_arg[lane];
      const unsigned rej = __ballot_sync(0xffffffffu, miss);
      const int a = rej ? __ffs(rej) - 1 : g;
      if (rank == 0) {
        if (lane == 0) {
          P.accept_len[b] = a;
          P.out_token[b] = st_arg[a];
          if (P.rollback) P.rollback[b] = prefix + a;
          if (P.resid) P.resid[b] = 0.f;
          if (P.seq_error) P.seq_error[b] = 0;
        }
        if (lane < g) {
          if (P.p_at) P.p_at[static_cast<long long>(b) * g + lane] = 0.f;
          if (P.q_at) P.q_at[static_cast<long long>(b) * g + lane] = 0.f;
        }
      }
    }
    return;
  } else {
    const T* target = static_cast<const T*>(P.target);
    const T* draft = static_cast<const T*>(P.draft);
    const long long trow0 = static_cast<long long>(b) * (g + 1);
    const long long drow0 = static_cast<long long>(b) * g;

    // accept tests, one lane per drafted position
    if (warp == 0) {
      bool keep = true;
      if (lane < g) {
        const int d = tok[lane];
        const float xp = load_elem(target + (trow0 + lane) * P.ld + d);
        const float xq = load_elem(draft + (drow0 + lane) * P.ld + d);
        const double lp = log2_prob(xp, st_m[lane], st_s[lane], c);
        const double lq = log2_prob(xq, st_m[g + 1 + lane], st_s[g + 1 + lane], c);
        keep = keeps(P.u[drow0 + lane], accept_ratio(lp, lq));
        if (rank == 0) {
          if (P.p_at) P.p_at[drow0 + lane] = static_cast<float>(exp2(lp));
          if (P.q_at) P.q_at[drow0 + lane] = static_cast<float>(exp2(lq));
        }
      }
      const unsigned rej = __ballot_sync(0xffffffffu, lane < g && !keep);
      if (lane == 0) a_s = rej ? __ffs(rej) - 1 : g;
    }
    __syncthreads();
    const int a = a_s;

    // residual max(0, p_a - q_a) after a rejection, the bonus row otherwise
    PassSpec<T> S;
    S.P = target + (trow0 + a) * P.ld;
    S.MP = scaled_max(st_m[a], c);
    S.invSP = __fdiv_rn(1.f, st_s[a]);
    if (a < g) {
      S.Q = draft + (drow0 + a) * P.ld;
      S.MQ = scaled_max(st_m[g + 1 + a], c);
      S.invSQ = __fdiv_rn(1.f, st_s[g + 1 + a]);
      S.cq = 1.f;
    } else {
      S.Q = nullptr;
      S.MQ = 0.f;
      S.invSQ = 0.f;
      S.cq = 0.f;
    }
    double Z = run_pass(S, P.V, c, sh, cl);
    int flag = 0;
    if (!(Z > 0.0) || !(Z < INFINITY)) {  // p == q numerically: draw from p
      flag = SPEC_ERR_ZERO_MASS;
      S.cq = 0.f;
      Z = run_pass(S, P.V, c, sh, cl);
    }
    const int owner = run_search(S, P.V, c, static_cast<double>(P.v[b]) * Z, sh, cl);
    if (rank == owner && tid == 0) P.out_token[b] = sh.result[sh.sparity ^ 1];
    if (rank == 0 && tid == 0) {
      P.accept_len[b] = a;
      if (P.rollback) P.rollback[b] = prefix + a;
      if (P.resid) P.resid[b] = static_cast<float>(Z);
      if (P.seq_error) P.seq_error[b] = flag;
      if (flag && P.error_word) atomicOr(P.error_word, flag);
    }
    cl.sync();  // no CTA leaves while another may still read its shared memory
  }
}

}  // namespace

cudaError_t launch_chain_walk(const ChainParams& p, bool bf16, bool greedy, cudaStream_t s) {
  void* args[] = {const_cast<ChainParams*>(&p)};
  const void* k;
  if (bf16) k = greedy ? reinterpret_cast<const void*>(&chain_walk_kernel<bf16_t, true>)
                       : reinterpret_cast<const void*>(&chain_walk_kernel<bf16_t, false>);
  else k = greedy ? reinterpret_cast<const void*>(&chain_walk_kernel<float, true>)
                  : reinterpret_cast<const void*>(&chain_walk_kernel<float, false>);
  return launch_walker(k, args, p.B, greedy ? 1 : p.cluster, 0, s);
}

}  // namespace sv
