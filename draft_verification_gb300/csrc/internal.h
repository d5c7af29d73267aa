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

// Everything the kernels need besides the kind-specific arguments.
struct StatsParams {
  RowSet set[3];
  int nsets;
  int rows_per_seq;     // sum of set[k].rows
  int B;
  int V;
  long long ld;
  int chunks;           // statistics CTAs per row
  int ntiles;           // pass tiles per row
  int tps;              // pass tiles per slice CTA
  float c;              // log2(e) / T (sampling); unused in greedy mode
  void* state;          // [kMaxSeq] per-sequence counters, zero between calls
  void* specs;          // [B] cascade: the stage-2 pass
  void* mid;            // [B] cascade: stage-1 flags
  float* sums;          // [B][2][ntiles] pass tile sums
  float2* partials;     // [B][rows_per_seq][chunks]: (max, sum) or (value, index)
};

// Chunks per row for the dtype; the workspace is sized for the larger
// (float32) count so one size serves both dtypes.
int stats_chunks(int V, bool bf16);
int pass_tiles(int V);
constexpr int kTilesPerSlice = 4;

// Workspace layout.  A fixed head, zeroed once by the caller and left zero by
// every call: 256 reserved bytes and one 32-byte record per possible sequence
// index, so that calls of any batch size, mode or kind share it.  Then
// per-call scratch, fully written before it is read.
constexpr int kMaxSeq = 65535;
constexpr size_t kSeqStateBytes = 32;
constexpr size_t kSpecBytes = 48;
constexpr size_t kHeadBytes = 256 + 65536 * kSeqStateBytes;
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Layout {
  size_t specs, mid, sums, partials, total;
};
inline Layout workspace_layout(int B, int rows_per_seq, int V) {
  Layout L;
  size_t off = kHeadBytes;
  L.specs = off;
  off = align256(off + static_cast<size_t>(B) * kSpecBytes);
  L.mid = off;
  off = align256(off + static_cast<size_t>(B) * 16);
  L.sums = off;
  off = align256(off + static_cast<size_t>(B) * 2 * pass_tiles(V) * 4);
  L.partials = off;
  off = align256(off + static_cast<size_t>(B) * rows_per_seq * stats_chunks(V, false) * 8);
  L.total = off;
  return L;
}
inline size_t workspace_bytes(int B, int rows_per_seq, int V) {
  return workspace_layout(B, rows_per_seq, V).total;
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

cudaError_t launch_chain(const StatsParams& g, const ChainParams& p, bool bf16, bool greedy, cudaStream_t s);
cudaError_t launch_tree(const StatsParams& g, const TreeParams& p, bool bf16, bool greedy, cudaStream_t s);
cudaError_t launch_cascade(const StatsParams& g, const CascadeParams& p, bool bf16, bool greedy,
                           cudaStream_t s);

}  // namespace sv
