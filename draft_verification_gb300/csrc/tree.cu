// Tree verification: walk each sequence's draft tree from the root.
//
// "Accelerating LLM Inference with Staged Speculative Decoding", abstract:
// the speculative batch is restructured as a tree.  Row n of the logit arrays
// is the distribution over the children of node n.  At a node, the children
// are tried in ascending index; a kept child becomes the next node; a
// rejected child turns the current target distribution p into
// norm(max(0, p - q)) (q unchanged) before the next sibling is tried; when no
// child is kept the token is drawn from the current p (from the node's own
// target row at a leaf).  Greedy keeps the first child whose token is the
// target argmax and otherwise emits the argmax.
//
// Repeated residuals without repeated normalisation.  After k rejections at
// one node the current distribution is
//     p_k = max(0, p - c_k q) / W_k,  c_0 = 0, W_0 = 1,
//     c_{k+1} = c_k + W_k,            W_{k+1} = sum_x max(0, p - c_{k+1} q),
// because max(0, max(0, p - c_k q)/W_k - q) = max(0, p - (c_k + W_k) q)/W_k
// wherever the inner term is positive, and both sides are 0 elsewhere.  So
// each rejection costs one pass with the scalar cq = c_{k+1}, and the final
// draw searches the last pass (target v * W_k).  This is the iterated
// renormalisation written in closed form; the result is the same.
//
// One cluster per sequence; every CTA repeats the (cheap) tree bookkeeping so
// that all decisions are taken identically everywhere.
#include "common.cuh"
#include "internal.h"
#include "spec_verify.h"
#include "walk.cuh"

namespace sv {
namespace {

// Dynamic shared memory: 40 bytes per node (see tree_smem_bytes).
struct TreeSmem {
  float2* st;   // [2N] (max, sum) of target rows then draft rows; greedy: .x unused, argmax in .y
  int* par;     // [N]
  int* tk;      // [N]
  float* gp;    // [N] target logit of node i's token in its parent's row
  float* gq;    // [N] draft logit of the same
  int* scr_a;   // [N] depth pointer jumping, then the children of the current node
  int* scr_b;   // [N] depth pointer jumping, then the kept path
};

__device__ __forceinline__ TreeSmem tree_smem(char* base, int N) {
  TreeSmem t;
  t.st = reinterpret_cast<float2*>(base);
  t.par = reinterpret_cast<int*>(base + 16 * N);
  t.tk = t.par + N;
  t.gp = reinterpret_cast<float*>(t.tk + N);
  t.gq = t.gp + N;
  t.scr_a = reinterpret_cast<int*>(t.gq + N);
  t.scr_b = t.scr_a + N;
  return t;
}

// Children of `node`, ascending, into kids[]; returns their number (warp 0
// computes, result valid for the whole CTA after the barrier).
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

template <typename T, bool kGreedy>
__global__ void __launch_bounds__(kThreads) tree_walk_kernel(const TreeParams P) {
  extern __shared__ __align__(16) char dyn[];
  cg::cluster_group cl = cg::this_cluster();
  const int cs = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / cs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = P.N;
  const float c = P.c;
  TreeSmem ts = tree_smem(dyn, N);

  __shared__ PassShared sh;
  __shared__ int err_s, nk_s, accepted_s;
  if (tid == 0) {
    sh.parity = 0;
    sh.sparity = 0;
    err_s = 0;
  }
  const long long row0 = static_cast<long long>(b) * N;
  for (int i = tid; i < N; i += kThreads) {
    const int p = P.parent[row0 + i];
    const int t = P.tokens[row0 + i];
    ts.par[i] = p;
    ts.tk[i] = t;
  }
  __syncthreads();
  // well-formed parents and tokens
  for (int i = tid; i < N; i += kThreads) {
    const int p = ts.par[i];
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) atomicOr(&err_s, SPEC_ERR_PARENT);
    if (i > 0 && (ts.tk[i] < 0 || ts.tk[i] >= P.V)) atomicOr(&err_s, SPEC_ERR_TOKEN);
  }
  __syncthreads();
  if (!(err_s & SPEC_ERR_PARENT)) {
    // depth by pointer jumping: D[i] += D[A[i]], A[i] = A[A[i]]
    constexpr int kPer = 1024 / kThreads;
    for (int i = tid; i < N; i += kThreads) {
      ts.scr_a[i] = i == 0 ? 0 : ts.par[i];
      ts.scr_b[i] = i == 0 ? 0 : 1;
    }
    __syncthreads();
    for (int span = 1; span < N; span <<= 1) {
      int na[kPer], nd[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = tid + j * kThreads;
        if (i < N) {
          const int a = ts.scr_a[i];
          nd[j] = ts.scr_b[i] + ts.scr_b[a];
          na[j] = ts.scr_a[a];
        }
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = tid + j * kThreads;
        if (i < N) {
          ts.scr_a[i] = na[j];
          ts.scr_b[i] = nd[j];
        }
      }
      __syncthreads();
    }
    for (int i = tid; i < N; i += kThreads)
      if (ts.scr_b[i] > P.max_depth) atomicOr(&err_s, SPEC_ERR_PARENT);
  }

  pdl_wait();  // statistics are complete from here on

  const float2* part = P.partials + static_cast<long long>(b) * P.rows_per_seq * P.chunks;
  for (int r = warp; r < P.rows_per_seq; r += kWarps) {
    if constexpr (kGreedy) {
      bool bad;
      const ArgMax am = combine_row_argmax(part + static_cast<long long>(r) * P.chunks, P.chunks, bad);
      if (lane == 0) {
        ts.st[r] = make_float2(0.f, __int_as_float(am.i));
        if (bad || am.i < 0) atomicOr(&err_s, SPEC_ERR_NONFINITE);
      }
    } else {
      const MaxSum ms = combine_row(part + static_cast<long long>(r) * P.chunks, P.chunks, c);
      if (lane == 0) {
        ts.st[r] = make_float2(ms.m, ms.s);
        if (!row_stats_ok(ms)) atomicOr(&err_s, SPEC_ERR_NONFINITE);
      }
    }
  }
  __syncthreads();

  const int err = err_s;
  const int prefix = P.prefix ? P.prefix[b] : 0;
  const int pn = P.max_depth + 1;
  if (err) {
    if (rank == 0) {
      if (tid == 0) {
        P.path_len[b] = 0;
        P.out_token[b] = -1;
        if (P.rollback) P.rollback[b] = prefix;
        if (P.seq_error) P.seq_error[b] = err;
        if (P.error_word) atomicOr(P.error_word, err);
      }
      for (int j = tid; j < pn; j += kThreads) P.path_nodes[static_cast<long long>(b) * pn + j] = -1;
    }
    return;
  }

  const T* target = static_cast<const T*>(P.target);
  const T* draft = static_cast<const T*>(P.draft);
  if constexpr (!kGreedy) {
    for (int i = tid + 1; i < N; i += kThreads) {
      const long long off = (row0 + ts.par[i]) * P.ld + ts.tk[i];
      ts.gp[i] = load_elem(target + off);
      ts.gq[i] = load_elem(draft + off);
    }
  }
  __syncthreads();

  int* kids = ts.scr_a;
  int* path = ts.scr_b;
  int node = 0, plen = 0, flag = 0, token = -1, owner = -1;
  while (true) {
    const int nk = list_children(ts.par, N, node, kids, &nk_s);
    if constexpr (kGreedy) {
      const int best = __float_as_int(ts.st[node].y);
      int kept = -1;
      for (int j = 0; j < nk; ++j)
        if (ts.tk[kids[j]] == best) {
          kept = kids[j];
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
      const float2 sp = ts.st[node];
      const float2 sq = ts.st[N + node];
      PassSpec<T> S;
      S.P = target + (row0 + node) * P.ld;
      S.Q = draft + (row0 + node) * P.ld;
      S.MP = scaled_max(sp.x, c);
      S.invSP = __fdiv_rn(1.f, sp.y);
      S.MQ = scaled_max(sq.x, c);
      S.invSQ = __fdiv_rn(1.f, sq.y);
      S.cq = 0.f;
      double cc = 0.0, W = 1.0;
      if (tid == 0) accepted_s = -1;
      __syncthreads();
      int kept = -1;
      bool zero_mass = false;
      for (int j = 0; j < nk; ++j) {
        const int ch = kids[j];
        const double lp = log2_prob(ts.gp[ch], sp.x, sp.y, c);
        const double lq = log2_prob(ts.gq[ch], sq.x, sq.y, c);
        const double pt = exp2(lp), qt = exp2(lq);
        const double pk = fmax(0.0, pt - cc * qt) / W;
        double ratio;
        if (qt > 0.0) ratio = pk / qt;
        else ratio = pk > 0.0 ? INFINITY : 0.0;
        if (keeps(P.u[row0 + ch], ratio)) {
          kept = ch;
          break;
        }
        const double cn = cc + W;
        S.cq = static_cast<float>(cn);
        const double Wn = run_pass(S, P.V, c, sh, cl);
        if (!(Wn > 0.0) || !(Wn < INFINITY)) {
          zero_mass = true;
          break;
        }
        cc = cn;
        W = Wn;
      }
      __syncthreads();
      if (kept >= 0) {
        if (tid == 0) path[plen] = kept;
        ++plen;
        node = kept;
        continue;
      }
      double Z = W;
      if (zero_mass || nk == 0) {
        if (zero_mass) flag = SPEC_ERR_ZERO_MASS;
        S.cq = 0.f;  // draw from the node's own target distribution
        Z = run_pass(S, P.V, c, sh, cl);
      }
      owner = run_search(S, P.V, c, static_cast<double>(P.v[b]) * Z, sh, cl);
      break;
    }
  }
  __syncthreads();

  if constexpr (!kGreedy) {
    if (rank == owner && tid == 0) P.out_token[b] = sh.result[sh.sparity ^ 1];
  }
  if (rank == 0) {
    if (tid == 0) {
      if constexpr (kGreedy) P.out_token[b] = token;
      P.path_len[b] = plen;
      if (P.rollback) P.rollback[b] = prefix + plen;
      if (P.seq_error) P.seq_error[b] = flag;
      if (flag && P.error_word) atomicOr(P.error_word, flag);
    }
    int* pnodes = P.path_nodes + static_cast<long long>(b) * pn;
    for (int j = tid; j < pn; j += kThreads) pnodes[j] = j == 0 ? 0 : (j <= plen ? path[j - 1] : -1);
  }
  if constexpr (!kGreedy) cl.sync();  // keep shared memory alive for remote readers
}

size_t tree_smem_bytes(int N) { return static_cast<size_t>(40) * N; }

}  // namespace

cudaError_t launch_tree_walk(const TreeParams& p, bool bf16, bool greedy, cudaStream_t s) {
  void* args[] = {const_cast<TreeParams*>(&p)};
  const void* k;
  if (bf16) k = greedy ? reinterpret_cast<const void*>(&tree_walk_kernel<bf16_t, true>)
                       : reinterpret_cast<const void*>(&tree_walk_kernel<bf16_t, false>);
  else k = greedy ? reinterpret_cast<const void*>(&tree_walk_kernel<float, true>)
                  : reinterpret_cast<const void*>(&tree_walk_kernel<float, false>);
  const size_t smem = tree_smem_bytes(p.N);
  if (smem > 40 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_walker(k, args, p.B, greedy ? 1 : p.cluster, smem, s);
}

}  // namespace sv
