// Host-side declarations shared by the translation units of the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

// Logit rows of one tensor: row (b, i) starts at base + (b * rows + i) * ld.
struct RowSet {
  const void* base;
  int rows;
};

// One launch of the row-statistics kernel over up to three tensors.  The
// rows of a sequence are numbered set by set: set 0's rows first.
struct StatsParams {
  RowSet set[3];
  int nsets;
  int rows_per_seq;   // sum of set[k].rows
  int B;
  int V;
  long long ld;
  int chunks;         // row-statistics CTAs per row
  float c;            // log2(e) / T (sampling); unused in greedy mode
  float2* partials;   // [B][rows_per_seq][chunks]: (max, sum) or (value, index)
};

inline int stats_chunks(int V) { return (V + 8191) / 8192; }

// Workspace bytes for `rows_per_seq` statistics rows per sequence.
inline size_t stats_workspace_bytes(int B, int rows_per_seq, int V) {
  return static_cast<size_t>(B) * rows_per_seq * stats_chunks(V) * sizeof(float2);
}

cudaError_t launch_row_stats(const StatsParams& p, bool bf16, bool greedy, cudaStream_t s);

// Cluster size of the walker kernels: enough CTAs that each covers about
// four 2048-element tiles of a row, at most 8 (the portable cluster size).
inline int walker_cluster(int V) {
  int tiles = (V + 2047) / 2048;
  int cs = (tiles + 3) / 4;
  return cs < 1 ? 1 : (cs > 8 ? 8 : cs);
}

struct ChainParams {
  int B, gamma, V;
  long long ld;
  float c;                  // log2(e) / T
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
  const float2* partials;
  int chunks;
  int rows_per_seq;
  int cluster;
};
cudaError_t launch_chain_walk(const ChainParams& p, bool bf16, bool greedy, cudaStream_t s);

struct TreeParams {
  int B, N, max_depth, V;
  long long ld;
  float c;
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
  const float2* partials;
  int chunks;
  int rows_per_seq;
  int cluster;
};
cudaError_t launch_tree_walk(const TreeParams& p, bool bf16, bool greedy, cudaStream_t s);

struct CascadeParams {
  int B, g1, g2, V;
  long long ld;
  float c;
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
  const float2* partials;
  int chunks;
  int rows_per_seq;
  int cluster;
};
cudaError_t launch_cascade_walk(const CascadeParams& p, bool bf16, bool greedy, cudaStream_t s);

// Launch helper: `cluster` CTAs per sequence, with programmatic dependent
// launch so the walker's CTAs are scheduled while the statistics kernel
// drains.
cudaError_t launch_walker(const void* kernel, void** args, int B, int cluster,
                          size_t dyn_smem, cudaStream_t s);

}  // namespace sv
