// Host-side declarations shared by the translation units of the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "spec_verify.h"

#include <nvtx3/nvToolsExt.h>

namespace sv {

// NVTX range around one entry-point call (the call's launches nest inside
// it on a profiler's timeline; costs nothing when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Logit rows of one tensor: row (b, i) starts at base + (b * rows + i) * ld.
struct RowSet {
  const void* base;
  int rows;
};

// Row sets of one call: up to one per model of a k-model pipeline.
constexpr int kMaxSets = 8;

// Everything the kernels need besides the kind-specific arguments.
struct StatsParams {
  RowSet set[kMaxSets];
  int nsets;
  int rows_per_seq;     // sum of set[k].rows
  int B;
  int V;
  long long ld;
  int chunks;           // statistics CTAs per row
  int ntiles;           // pass tiles per row
  float c;              // log2(e) / T (sampling); unused in greedy mode
  float2* partials;     // [B][rows_per_seq][chunks]: (max, sum) or (value, index)
};

// Chunks per row for the dtype; the workspace is sized for the larger
// (float32) count so one size serves both dtypes.
int stats_chunks(int V, bool bf16);
int pass_tiles(int V);

constexpr int kMaxSeq = 65535;  // statistics grid z extent

// Workspace: the chunk partials of the statistics kernel, 8 bytes per
// (sequence, row, chunk), written by the first kernel of a call and read by
// the second; nothing in it outlives a call, so it needs no initialisation.
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline size_t workspace_bytes(int B, int rows_per_seq, int V) {
  return align256(static_cast<size_t>(B) * rows_per_seq * stats_chunks(V, false) * 8);
}
// Chain workspace: the partials (the consulted-only mode uses none).
inline size_t chain_workspace_bytes(int B, int gamma, int rows_per_seq, int V) {
  (void)gamma;
  return workspace_bytes(B, rows_per_seq, V);
}


struct ChainParams {
  int B, gamma, V;
  long long ld;
  const void* target;
  const void* draft;
  const int* tokens;
  const float* u;
  const float* v;
  const int* prefix;
  int* accept_len;
  int* out_token;
  int* rollback;
  float* p_at;
  float* q_at;
  float* resid;
  int* seq_error;
  int* error_word;
};

struct TreeParams {
  int B, N, max_depth, V;
  long long ld;
  const int* parent;
  const int* tokens;
  const void* target;
  const void* draft;
  const float* u;
  const float* v;
  const int* prefix;
  int* path_len;
  int* path_nodes;
  int* out_token;
  int* rollback;
  int* seq_error;
  int* error_word;
};

struct CascadeParams {
  int B, g1, g2, V;
  long long ld;
  const void* l0;
  const void* l1;
  const void* l2;
  const int* tokens;
  const float* u1;
  const float* v1;
  const float* u2;
  const float* v2;
  const int* base0;
  const int* base1;
  int* a1;
  int* t1;
  int* a2;
  int* w2;
  int* t2;
  int* t2_valid;
  int* r0;
  int* r1;
  int* committed;
  int* seq_error;
  int* error_word;
};

// k-model pipeline.  Model s's rows of a sequence: window[0] (M_0),
// window[0] + 1 (M_1), window[s-1] (+1 for the last model with the bonus);
// rowoff[s] is the first statistics row of model s (greedy calls have no
// M_0 rows: rowoff[0] is unused there).
struct PipelineParams {
  int B, k, V, final_bonus;
  long long ld;
  int window[kMaxSets - 1];
  int rows[kMaxSets];
  int rowoff[kMaxSets];
  const void* logits[kMaxSets];
  const int* tokens;
  const float* u[kMaxSets - 1];
  const float* v[kMaxSets - 1];
  const int* base;
  int* a;
  int* w;
  int* t;
  int* t_valid;
  int* r;
  int* committed;
  int* seq_error;
  int* error_word;
};

cudaError_t launch_pipeline(const StatsParams& g, const PipelineParams& p, bool bf16, bool greedy,
                            cudaStream_t s);

// `grouped` allows a large call to be split into batch groups on library
// streams (forked from and joined into s); false keeps every launch on s.
// `consulted` runs the consulted-only walk (no statistics kernel).
cudaError_t launch_chain(const StatsParams& g, const ChainParams& p, bool bf16, bool greedy, bool grouped,
                         bool consulted, cudaStream_t s);
// `consulted` runs the consulted-only tree walk (no statistics kernel).
cudaError_t launch_tree(const StatsParams& g, const TreeParams& p, bool bf16, bool greedy, bool consulted,
                        cudaStream_t s);
cudaError_t launch_cascade(const StatsParams& g, const CascadeParams& p, bool bf16, bool greedy,
                           cudaStream_t s);
// The chain walk alone over float32 logit rows whose chunk partials a
// preceding kernel on s wrote (the LM-head path); plain stream order.
cudaError_t launch_chain_walk_f32(const StatsParams& g, const ChainParams& p, bool greedy, cudaStream_t s);

}  // namespace sv

namespace sv {
// spec_verify_chain with batch groups allowed or not (the no-allocation
// entry point runs everything on the caller's stream).
spec_status verify_chain(const spec_chain_args* a, cudaStream_t stream, bool grouped);
}  // namespace sv
