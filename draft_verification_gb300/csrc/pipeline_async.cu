// PipeSpec stages at independent buffer offsets: one asynchronous snapshot.
//
// Source: Pith review of "PipeSpec: Breaking Stage Dependencies in
// Hierarchical LLM Decoding" (arXiv 2505.01572), "What carries the
// argument": the models run without global synchronisation; each M_s
// verifies the buffer O_{s-1} below it, appends the longest matching prefix
// to O_s, and a mismatch rolls every earlier buffer back to the last
// verified token.
//
// The stages of an asynchronous snapshot do not feed one another: stage s
// reads the window O_{s-1}[l_s, l_s + w_s) that was in place before the
// snapshot.  So each stage is one chain verification of its own window (the
// same statistics and walk kernels as spec_verify_chain, with no prefix: the
// chain reports only the stage's accept length a_s, token and error bits),
// and the stages run one after another on the caller's stream sharing one
// workspace.  pipeline_async_combine_kernel then forms each rejection
// position P_s = l_s + a_s from the buffer lengths and applies the emission
// and rollback rules per sequence:
//   - a window that does not fit (l_{s-1} < l_s + w_s) or a negative length
//     makes the sequence malformed (SPEC_ERR_WINDOW, empty outputs);
//   - a rejection emits the correction and cuts every earlier buffer to at
//     most P_s = l_s + a_s;
//   - with every token kept, stage 1 and (with the final bonus) the last
//     stage emit the bonus only if position l_s + w_s is still empty in the
//     buffer below after that buffer's own appends (stages resolved in
//     ascending order); middle stages emit nothing;
//   - O_s grows to l_s + a_s (+1 when it emits); r_j = min(that, P_s of
//     every rejecting stage s > j).
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "spec_verify.h"

namespace sv {
namespace {

constexpr int kMaxStages = SPEC_MAX_MODELS - 1;
constexpr int kMaxVocab = 2097152;  // the chain call's limit
constexpr int kCombineThreads = 128;
constexpr int kHardErrors = SPEC_ERR_TOKEN | SPEC_ERR_NONFINITE | SPEC_ERR_INTERNAL | SPEC_ERR_WINDOW;

struct AsyncParams {
  int B, k, final_bonus;
  int window[kMaxStages];
  const int* length;     // [k][B]
  const int* accept;     // [k-1][B]: the stages' chain outputs
  const int* token;      // [k-1][B]
  const int* stage_err;  // [k-1][B]
  int* a;                // [B][k-1]
  int* t;
  int* t_valid;
  int* r;                // [B][k-1]
  int* committed;        // [B]
  int* seq_error;        // [B] or null
  int* error_word;       // or null
};

__global__ void __launch_bounds__(kCombineThreads) pipeline_async_combine_kernel(AsyncParams p) {
  const int b = blockIdx.x * kCombineThreads + threadIdx.x;
  if (b >= p.B) return;
  const int k = p.k, B = p.B, S = k - 1;
  int l[kMaxStages + 1];
  for (int j = 0; j < k; ++j) l[j] = p.length[static_cast<size_t>(j) * B + b];
  int err = 0;
  for (int j = 0; j < k; ++j)
    if (l[j] < 0) err |= SPEC_ERR_WINDOW;
  for (int s = 1; s < k; ++s)
    if (static_cast<long long>(l[s - 1]) < static_cast<long long>(l[s]) + p.window[s - 1]) err |= SPEC_ERR_WINDOW;
  for (int s = 1; s < k; ++s) err |= p.stage_err[static_cast<size_t>(s - 1) * B + b];

  int* a_out = p.a + static_cast<size_t>(b) * S;
  int* t_out = p.t + static_cast<size_t>(b) * S;
  int* v_out = p.t_valid + static_cast<size_t>(b) * S;
  int* r_out = p.r + static_cast<size_t>(b) * S;
  if (p.seq_error) p.seq_error[b] = err;
  // the stages' own bits were OR-ed into the error word by their chains
  if (p.error_word && (err & SPEC_ERR_WINDOW)) atomicOr(p.error_word, SPEC_ERR_WINDOW);
  if (err & kHardErrors) {
    for (int s = 0; s < S; ++s) {
      a_out[s] = 0;
      t_out[s] = -1;
      v_out[s] = 0;
      r_out[s] = l[s];
    }
    p.committed[b] = l[k - 1];
    return;
  }
  int grown[kMaxStages + 1];  // new length of each buffer before the cuts
  int cut[kMaxStages + 1];    // P_s of a rejecting stage s, else INT_MAX
  grown[0] = l[0];
  cut[0] = INT_MAX;
  for (int s = 1; s < k; ++s) {
    const int w = p.window[s - 1];
    const int acc = p.accept[static_cast<size_t>(s - 1) * B + b];
    const bool rejected = acc < w;
    const bool bonus = (s == 1 || (p.final_bonus && s == k - 1)) && grown[s - 1] == l[s] + w;
    const bool emits = rejected || bonus;
    a_out[s - 1] = acc;
    t_out[s - 1] = emits ? p.token[static_cast<size_t>(s - 1) * B + b] : -1;
    v_out[s - 1] = emits ? 1 : 0;
    grown[s] = l[s] + acc + (emits ? 1 : 0);
    cut[s] = rejected ? l[s] + acc : INT_MAX;
  }
  // r_j = min(grown_j, cut_s for s > j): a suffix minimum over the stages
  int below = INT_MAX;
  int rj[kMaxStages + 1];
  for (int j = k - 1; j >= 0; --j) {
    rj[j] = min(grown[j], below);
    below = min(below, cut[j]);
  }
  for (int j = 0; j < S; ++j) r_out[j] = rj[j];
  p.committed[b] = rj[k - 1];
}

struct AsyncLayout {
  size_t chain, scratch, total;
};

bool async_layout(int B, int k, const int* window, int V, AsyncLayout* out) {
  if (B < 1 || B > kMaxSeq || k < 2 || k > SPEC_MAX_MODELS || window == nullptr || V < 1) return false;
  size_t chain = 0;
  for (int s = 0; s < k - 1; ++s) {
    if (window[s] < 1 || window[s] > 32) return false;
    chain = std::max(chain, chain_workspace_bytes(B, window[s], 2 * window[s] + 1, V));
  }
  out->chain = align256(chain);
  out->scratch = align256(static_cast<size_t>(3) * (k - 1) * B * sizeof(int));
  out->total = out->chain + out->scratch;
  return true;
}

bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

}  // namespace
}  // namespace sv

extern "C" size_t spec_pipeline_async_workspace_size(int B, int k, const int* window, int V) {
  sv::AsyncLayout w;
  return sv::async_layout(B, k, window, V, &w) ? w.total : 0;
}

extern "C" spec_status spec_verify_pipeline_async(const spec_pipeline_async_args* a, cudaStream_t stream) {
  sv::NvtxRange nvtx_range("spec_verify_pipeline_async");
  using namespace sv;
  if (a == nullptr) return SPEC_EINVAL;
  AsyncLayout w;
  if (!async_layout(a->B, a->k, a->window, a->V, &w)) return SPEC_EINVAL;
  if (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16) return SPEC_EDTYPE;
  if (a->mode != SPEC_GREEDY && a->mode != SPEC_SAMPLE) return SPEC_EDTYPE;
  const bool greedy = a->mode == SPEC_GREEDY;
  // every check a stage's chain call makes is made here first, so that an
  // argument error is reported before any stage has been launched
  if (a->V > kMaxVocab || a->ld < a->V || a->ld > (1LL << 40)) return SPEC_EINVAL;
  if (!greedy && !(a->temperature > 0.f && std::isfinite(a->temperature))) return SPEC_EINVAL;
  if (!a->length || !a->a || !a->t || !a->t_valid || !a->r || !a->committed) return SPEC_EINVAL;
  const int S = a->k - 1;
  for (int s = 0; s < S; ++s) {
    if (!a->target[s] || !a->tokens[s]) return SPEC_EINVAL;
    if (!greedy && (!a->draft[s] || !a->u[s] || !a->v[s])) return SPEC_EINVAL;
  }
  for (int s = 0; s < S; ++s)
    if (!aligned16(a->target[s]) || (!greedy && !aligned16(a->draft[s]))) return SPEC_EALIGN;
  if (!a->workspace || a->workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(a->workspace) & 15u))
    return SPEC_EWORKSPACE;
  char* ws = static_cast<char*>(a->workspace);
  int* accept = reinterpret_cast<int*>(ws + w.chain);
  int* token = accept + static_cast<size_t>(S) * a->B;
  int* stage_err = token + static_cast<size_t>(S) * a->B;

  // one chain verification per stage; the chain's rollback index (prefix +
  // accept length) is not needed, the combine recomputes the cuts
  for (int s = 0; s < S; ++s) {
    spec_chain_args c{};
    c.B = a->B;
    c.gamma = a->window[s];
    c.V = a->V;
    c.ld = a->ld;
    c.dtype = a->dtype;
    c.mode = a->mode;
    c.temperature = a->temperature;
    c.target_logits = a->target[s];
    c.draft_logits = greedy ? nullptr : a->draft[s];
    c.draft_tokens = a->tokens[s];
    c.u = greedy ? nullptr : a->u[s];
    c.v = greedy ? nullptr : a->v[s];
    c.prefix_len = nullptr;
    c.accept_len = accept + static_cast<size_t>(s) * a->B;
    c.out_token = token + static_cast<size_t>(s) * a->B;
    c.seq_error = stage_err + static_cast<size_t>(s) * a->B;
    c.error_word = a->error_word;
    c.workspace = a->workspace;
    c.workspace_bytes = w.chain;
    const spec_status st = verify_chain(&c, stream, true);
    if (st != SPEC_OK) return st;
  }
  AsyncParams p{};
  p.B = a->B;
  p.k = a->k;
  p.final_bonus = a->final_bonus != 0;
  for (int s = 0; s < S; ++s) p.window[s] = a->window[s];
  p.length = a->length;
  p.accept = accept;
  p.token = token;
  p.stage_err = stage_err;
  p.a = a->a;
  p.t = a->t;
  p.t_valid = a->t_valid;
  p.r = a->r;
  p.committed = a->committed;
  p.seq_error = a->seq_error;
  p.error_word = a->error_word;
  pipeline_async_combine_kernel<<<(a->B + kCombineThreads - 1) / kCombineThreads, kCombineThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}
