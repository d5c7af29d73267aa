// C ABI of the verification library: argument checks, workspace sizing and
// the one launch of every call.  Nothing here allocates or synchronises.
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "spec_verify.h"

namespace sv {

namespace {

constexpr int kMaxV = 2097152;  // tile sums of a whole row fit in shared memory (walk.cuh)
constexpr int kMaxB = kMaxSeq;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

spec_status check_common(int B, int V, long long ld, spec_dtype dtype, spec_mode mode,
                         float temperature) {
  if (B < 1 || B > kMaxB) return SPEC_EINVAL;
  if (V < 1 || V > kMaxV) return SPEC_EINVAL;
  if (ld < V || ld > (1LL << 40)) return SPEC_EINVAL;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_EDTYPE;
  if (mode != SPEC_GREEDY && mode != SPEC_SAMPLE) return SPEC_EDTYPE;
  if (mode == SPEC_SAMPLE && !(temperature > 0.f && std::isfinite(temperature))) return SPEC_EINVAL;
  return SPEC_OK;
}

// log2(e) / T, rounded once to float: the scale applied to every logit.
float logit_scale(float temperature) {
  return static_cast<float>(1.4426950408889634073599 / static_cast<double>(temperature));
}

spec_status run(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA; }

// Statistics geometry and workspace pointers shared by the three entry points.
bool stats_params(StatsParams& sp, int B, int V, long long ld, bool bf16, bool greedy, float temperature,
                  int rows, void* workspace) {
  sp = StatsParams{};
  sp.rows_per_seq = rows;
  sp.B = B;
  sp.V = V;
  sp.ld = ld;
  sp.chunks = stats_chunks(V, bf16);
  sp.ntiles = pass_tiles(V);
  sp.c = greedy ? 1.f : logit_scale(temperature);
  sp.partials = static_cast<float2*>(workspace);
  return rows <= 65535 && sp.chunks <= 0x7fffffff;
}

}  // namespace
}  // namespace sv

using namespace sv;

spec_status sv::verify_chain(const spec_chain_args* a, cudaStream_t stream, bool grouped) {
  if (a == nullptr) return SPEC_EINVAL;
  spec_status st = check_common(a->B, a->V, a->ld, a->dtype, a->mode, a->temperature);
  if (st != SPEC_OK) return st;
  const bool greedy = a->mode == SPEC_GREEDY;
  const bool bf16 = a->dtype == SPEC_BF16;
  if (a->gamma < 0 || a->gamma > 32) return SPEC_EINVAL;
  if (!a->target_logits || !a->accept_len || !a->out_token) return SPEC_EINVAL;
  if (a->gamma > 0 && !a->draft_tokens) return SPEC_EINVAL;
  if (!greedy && (!a->v || (a->gamma > 0 && (!a->draft_logits || !a->u)))) return SPEC_EINVAL;
  if (!aligned16(a->target_logits) || (!greedy && a->gamma > 0 && !aligned16(a->draft_logits)))
    return SPEC_EALIGN;
  // sampling reads the draft rows too; greedy reads the target rows only
  const int rows = greedy ? a->gamma + 1 : 2 * a->gamma + 1;
  const bool consulted = a->consulted_only != 0;
  if (consulted && (greedy || a->gamma < 1)) return SPEC_EINVAL;
  if (!a->workspace || a->workspace_bytes < chain_workspace_bytes(a->B, a->gamma, rows, a->V) ||
      !aligned16(a->workspace))
    return SPEC_EWORKSPACE;

  StatsParams sp;
  if (!stats_params(sp, a->B, a->V, a->ld, bf16, greedy, a->temperature, rows, a->workspace))
    return SPEC_EINVAL;
  sp.set[0] = RowSet{a->target_logits, a->gamma + 1};
  sp.set[1] = RowSet{a->draft_logits, a->gamma};
  sp.nsets = (greedy || a->gamma == 0) ? 1 : 2;

  ChainParams cp = {};
  cp.B = a->B;
  cp.gamma = a->gamma;
  cp.V = a->V;
  cp.ld = a->ld;
  cp.target = a->target_logits;
  cp.draft = a->draft_logits;
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
  return run(launch_chain(sp, cp, bf16, greedy, grouped, consulted, stream));
}

extern "C" {

const char* spec_status_string(spec_status status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_EINVAL: return "invalid argument";
    case SPEC_EDTYPE: return "unknown dtype or mode";
    case SPEC_EALIGN: return "logit base address not 16-byte aligned";
    case SPEC_EWORKSPACE: return "workspace missing or too small";
    case SPEC_ECUDA: return "CUDA launch failed";
  }
  return "unknown status";
}

size_t spec_chain_workspace_size(int B, int gamma, int V) {
  if (B < 1 || gamma < 0 || V < 1) return 0;
  return chain_workspace_bytes(B, gamma, 2 * gamma + 1, V);
}

size_t spec_tree_workspace_size(int B, int N, int V) {
  if (B < 1 || N < 1 || V < 1) return 0;
  return workspace_bytes(B, 2 * N, V);
}

size_t spec_cascade_workspace_size(int B, int gamma1, int gamma2, int V) {
  if (B < 1 || gamma1 < 1 || gamma2 < 1 || V < 1) return 0;
  return workspace_bytes(B, 2 * gamma1 + 1 + gamma2, V);
}

spec_status spec_verify_chain(const spec_chain_args* a, cudaStream_t stream) {
  sv::NvtxRange nvtx_range("spec_verify_chain");
  return sv::verify_chain(a, stream, true);
}

spec_status spec_verify_tree(const spec_tree_args* a, cudaStream_t stream) {
  sv::NvtxRange nvtx_range("spec_verify_tree");
  if (a == nullptr) return SPEC_EINVAL;
  spec_status st = check_common(a->B, a->V, a->ld, a->dtype, a->mode, a->temperature);
  if (st != SPEC_OK) return st;
  const bool greedy = a->mode == SPEC_GREEDY;
  const bool bf16 = a->dtype == SPEC_BF16;
  if (a->N < 1 || a->N > 1024) return SPEC_EINVAL;
  if (a->max_depth < 0 || a->max_depth > a->N - 1) return SPEC_EINVAL;
  if (!a->parent || !a->node_tokens || !a->target_logits || !a->path_len || !a->path_nodes ||
      !a->out_token)
    return SPEC_EINVAL;
  if (!greedy && (!a->draft_logits || !a->u || !a->v)) return SPEC_EINVAL;
  if (!aligned16(a->target_logits) || (!greedy && !aligned16(a->draft_logits))) return SPEC_EALIGN;
  const int rows = greedy ? a->N : 2 * a->N;
  if (!a->workspace || a->workspace_bytes < workspace_bytes(a->B, rows, a->V) ||
      !aligned16(a->workspace))
    return SPEC_EWORKSPACE;

  StatsParams sp;
  if (!stats_params(sp, a->B, a->V, a->ld, bf16, greedy, a->temperature, rows, a->workspace))
    return SPEC_EINVAL;
  sp.set[0] = RowSet{a->target_logits, a->N};
  sp.set[1] = RowSet{a->draft_logits, a->N};
  sp.nsets = greedy ? 1 : 2;

  TreeParams tp = {};
  tp.B = a->B;
  tp.N = a->N;
  tp.max_depth = a->max_depth;
  tp.V = a->V;
  tp.ld = a->ld;
  tp.parent = a->parent;
  tp.tokens = a->node_tokens;
  tp.target = a->target_logits;
  tp.draft = a->draft_logits;
  tp.u = a->u;
  tp.v = a->v;
  tp.prefix = a->prefix_len;
  tp.path_len = a->path_len;
  tp.path_nodes = a->path_nodes;
  tp.out_token = a->out_token;
  tp.rollback = a->rollback_idx;
  tp.seq_error = a->seq_error;
  tp.error_word = a->error_word;
  return run(launch_tree(sp, tp, bf16, greedy, a->consulted_only != 0, stream));
}

spec_status spec_verify_cascade(const spec_cascade_args* a, cudaStream_t stream) {
  sv::NvtxRange nvtx_range("spec_verify_cascade");
  if (a == nullptr) return SPEC_EINVAL;
  spec_status st = check_common(a->B, a->V, a->ld, a->dtype, a->mode, a->temperature);
  if (st != SPEC_OK) return st;
  const bool greedy = a->mode == SPEC_GREEDY;
  const bool bf16 = a->dtype == SPEC_BF16;
  if (a->gamma1 < 1 || a->gamma1 > 32) return SPEC_EINVAL;
  if (a->gamma2 < 1 || a->gamma2 > 32 || a->gamma2 > a->gamma1 + 1) return SPEC_EINVAL;
  if (!a->l1 || !a->l2 || !a->draft_tokens) return SPEC_EINVAL;
  if (!a->a1 || !a->t1 || !a->a2 || !a->w2 || !a->t2 || !a->t2_valid || !a->r0 || !a->r1 ||
      !a->committed)
    return SPEC_EINVAL;
  if (!greedy && (!a->l0 || !a->u1 || !a->v1 || !a->u2 || !a->v2)) return SPEC_EINVAL;
  if (!aligned16(a->l1) || !aligned16(a->l2) || (!greedy && !aligned16(a->l0))) return SPEC_EALIGN;
  const int rows = greedy ? a->gamma1 + 1 + a->gamma2 : 2 * a->gamma1 + 1 + a->gamma2;
  if (!a->workspace || a->workspace_bytes < workspace_bytes(a->B, rows, a->V) ||
      !aligned16(a->workspace))
    return SPEC_EWORKSPACE;

  StatsParams sp;
  if (!stats_params(sp, a->B, a->V, a->ld, bf16, greedy, a->temperature, rows, a->workspace))
    return SPEC_EINVAL;
  if (greedy) {
    sp.set[0] = RowSet{a->l1, a->gamma1 + 1};
    sp.set[1] = RowSet{a->l2, a->gamma2};
    sp.nsets = 2;
  } else {
    sp.set[0] = RowSet{a->l0, a->gamma1};
    sp.set[1] = RowSet{a->l1, a->gamma1 + 1};
    sp.set[2] = RowSet{a->l2, a->gamma2};
    sp.nsets = 3;
  }

  CascadeParams cp = {};
  cp.B = a->B;
  cp.g1 = a->gamma1;
  cp.g2 = a->gamma2;
  cp.V = a->V;
  cp.ld = a->ld;
  cp.l0 = a->l0;
  cp.l1 = a->l1;
  cp.l2 = a->l2;
  cp.tokens = a->draft_tokens;
  cp.u1 = a->u1;
  cp.v1 = a->v1;
  cp.u2 = a->u2;
  cp.v2 = a->v2;
  cp.base0 = a->base0;
  cp.base1 = a->base1;
  cp.a1 = a->a1;
  cp.t1 = a->t1;
  cp.a2 = a->a2;
  cp.w2 = a->w2;
  cp.t2 = a->t2;
  cp.t2_valid = a->t2_valid;
  cp.r0 = a->r0;
  cp.r1 = a->r1;
  cp.committed = a->committed;
  cp.seq_error = a->seq_error;
  cp.error_word = a->error_word;
  return run(launch_cascade(sp, cp, bf16, greedy, stream));
}

}  // extern "C"

namespace {

// Rows per sequence of each model of a pipeline (model s at index s), their
// total over the models the statistics read, or -1 for a bad window.
int pipeline_rows(int k, const int* window, bool final_bonus, bool greedy, int* rows) {
  if (k < 2 || k > kMaxSets) return -1;
  for (int s = 0; s < k - 1; ++s)
    if (window[s] < 1 || window[s] > 32) return -1;
  rows[0] = window[0];
  rows[1] = window[0] + 1;
  for (int s = 2; s < k; ++s) rows[s] = window[s - 1] + ((final_bonus && s == k - 1) ? 1 : 0);
  if (k == 2 && final_bonus) rows[1] = window[0] + 1;  // stage 1 always has its bonus row
  int total = 0;
  for (int s = greedy ? 1 : 0; s < k; ++s) total += rows[s];
  return total;
}

}  // namespace

extern "C" size_t spec_pipeline_workspace_size(int B, int k, const int* window, int final_bonus, int V) {
  if (B < 1 || V < 1 || window == nullptr) return 0;
  int rows[kMaxSets];
  const int total = pipeline_rows(k, window, final_bonus != 0, false, rows);
  if (total < 0) return 0;
  return workspace_bytes(B, total, V);
}

extern "C" spec_status spec_verify_pipeline(const spec_pipeline_args* a, cudaStream_t stream) {
  sv::NvtxRange nvtx_range("spec_verify_pipeline");
  if (a == nullptr) return SPEC_EINVAL;
  spec_status st = check_common(a->B, a->V, a->ld, a->dtype, a->mode, a->temperature);
  if (st != SPEC_OK) return st;
  const bool greedy = a->mode == SPEC_GREEDY;
  const bool bf16 = a->dtype == SPEC_BF16;
  const int k = a->k;
  int rows[kMaxSets];
  const int total = pipeline_rows(k, a->window, a->final_bonus != 0, greedy, rows);
  if (total < 0) return SPEC_EINVAL;
  if (!a->draft_tokens || !a->a || !a->w || !a->t || !a->t_valid || !a->r || !a->committed) return SPEC_EINVAL;
  for (int s = greedy ? 1 : 0; s < k; ++s) {
    if (!a->logits[s]) return SPEC_EINVAL;
    if (!aligned16(a->logits[s])) return SPEC_EALIGN;
  }
  if (!greedy)
    for (int s = 0; s < k - 1; ++s)
      if (!a->u[s] || !a->v[s]) return SPEC_EINVAL;
  if (!a->workspace || a->workspace_bytes < workspace_bytes(a->B, total, a->V) || !aligned16(a->workspace))
    return SPEC_EWORKSPACE;

  StatsParams sp;
  if (!stats_params(sp, a->B, a->V, a->ld, bf16, greedy, a->temperature, total, a->workspace)) return SPEC_EINVAL;
  PipelineParams pp = {};
  pp.B = a->B;
  pp.k = k;
  pp.V = a->V;
  pp.ld = a->ld;
  pp.final_bonus = a->final_bonus != 0;
  int off = 0;
  sp.nsets = 0;
  for (int s = 0; s < k; ++s) {
    pp.rows[s] = rows[s];
    pp.logits[s] = a->logits[s];
    if (greedy && s == 0) {
      pp.rowoff[0] = 0;
      continue;
    }
    pp.rowoff[s] = off;
    off += rows[s];
    sp.set[sp.nsets++] = RowSet{a->logits[s], rows[s]};
  }
  for (int s = 0; s < k - 1; ++s) {
    pp.window[s] = a->window[s];
    pp.u[s] = greedy ? nullptr : a->u[s];
    pp.v[s] = greedy ? nullptr : a->v[s];
  }
  pp.tokens = a->draft_tokens;
  pp.base = a->base;
  pp.a = a->a;
  pp.w = a->w;
  pp.t = a->t;
  pp.t_valid = a->t_valid;
  pp.r = a->r;
  pp.committed = a->committed;
  pp.seq_error = a->seq_error;
  pp.error_word = a->error_word;
  return run(launch_pipeline(sp, pp, bf16, greedy, stream));
}
