// Cache compaction after a tree verification (spec_compact_tree_path).
//
// Staged Speculative Decoding, abstract: the speculative batch is a tree;
// PipeSpec review, "What carries the argument": a buffer keeps the verified
// prefix and is rolled back to the last verified token.  The verify pass
// wrote one row of W bytes per tree node; the rows of the kept root path move
// to contiguous cache positions prefix_len, prefix_len + 1, ...
//
// One kernel: CTA (x, i, b) moves chunk x (kChunkBytes) of the row at path
// position i of sequence b.  Every CTA checks its sequence's path itself (a
// few int loads by one warp), so no CTA depends on another; CTA (0, 0, b)
// reports the sequence's error bits.  The copy is HBM-bound: each thread
// keeps four 16-byte loads in flight before it stores.
#include <cstdint>

#include "internal.h"
#include "spec_verify.h"

namespace sv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyVecs = 4;  // 16-byte vectors per thread per chunk
constexpr long long kChunkBytes = static_cast<long long>(kCopyThreads) * kCopyVecs * 16;

struct CompactParams {
  int B, N, D1, C;
  long long W, tree_ld, cache_ld;
  const unsigned char* tree;
  unsigned char* cache;
  const int* path_nodes;
  const int* path_len;
  const int* prefix;
  int* seq_error;
  int* error_word;
};

__device__ __forceinline__ uint4 ld_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <bool kVec>
__global__ void __launch_bounds__(kCopyThreads) compact_kernel(const CompactParams P) {
  __shared__ int s_status, s_node, s_base, s_rows;
  const int b = blockIdx.z, i = blockIdx.y, tid = threadIdx.x;
  if (tid < 32) {
    // the sequence's path: 0 = copy, 1 = skip (verifier error), 2 = malformed
    const int* nodes = P.path_nodes + static_cast<long long>(b) * P.D1;
    const int first = nodes[0];
    const int rows = P.path_len[b] + 1;
    const int base = P.prefix ? P.prefix[b] : 0;
    bool bad = rows < 1 || rows > P.D1 || base < 0 || base > P.C - rows;
    if (!bad)
      for (int j = tid; j < rows; j += 32) bad |= nodes[j] < 0 || nodes[j] >= P.N;
    bad = __any_sync(0xffffffffu, bad);
    if (tid == 0) {
      s_status = first < 0 ? 1 : (bad ? 2 : 0);
      s_rows = rows;
      s_base = base;
      s_node = (!bad && i < rows) ? nodes[i] : -1;
    }
  }
  __syncthreads();
  const int status = s_status;
  if (blockIdx.x == 0 && i == 0 && tid == 0) {
    const int err = status == 2 ? SPEC_ERR_PARENT : 0;
    if (P.seq_error) P.seq_error[b] = err;
    if (err && P.error_word) atomicOr(P.error_word, err);
  }
  if (status != 0 || i >= s_rows) return;
  const long long off = static_cast<long long>(blockIdx.x) * kChunkBytes;
  const long long n = P.W - off < kChunkBytes ? P.W - off : kChunkBytes;
  const unsigned char* src =
      P.tree + (static_cast<long long>(b) * P.N + s_node) * P.tree_ld + off;
  unsigned char* dst = P.cache + (static_cast<long long>(b) * P.C + s_base + i) * P.cache_ld + off;
  if constexpr (kVec) {
    uint4 v[kCopyVecs];
#pragma unroll
    for (int k = 0; k < kCopyVecs; ++k) {
      const long long o = (static_cast<long long>(k) * kCopyThreads + tid) * 16;
      if (o < n) v[k] = ld_nc16(src + o);
    }
#pragma unroll
    for (int k = 0; k < kCopyVecs; ++k) {
      const long long o = (static_cast<long long>(k) * kCopyThreads + tid) * 16;
      if (o < n) *reinterpret_cast<uint4*>(dst + o) = v[k];
    }
  } else {
    for (long long o = tid; o < n; o += kCopyThreads) dst[o] = src[o];
  }
}

bool multiple16(long long x) { return (x & 15) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" spec_status spec_compact_tree_path(const spec_compact_args* a, cudaStream_t stream) {
  sv::NvtxRange nvtx_range("spec_compact_tree_path");
  if (a == nullptr) return SPEC_EINVAL;
  if (a->B < 1 || a->B > 65535 || a->N < 1 || a->max_depth < 0 || a->max_depth > 65534 || a->cache_rows < 1)
    return SPEC_EINVAL;
  if (a->row_bytes < 1 || a->tree_ld < a->row_bytes || a->cache_ld < a->row_bytes) return SPEC_EINVAL;
  if (!a->tree_rows || !a->cache || !a->path_nodes || !a->path_len) return SPEC_EINVAL;
  const long long chunks = (a->row_bytes + kChunkBytes - 1) / kChunkBytes;
  if (chunks > 0x7fffffffLL) return SPEC_EINVAL;
  CompactParams p;
  p.B = a->B;
  p.N = a->N;
  p.D1 = a->max_depth + 1;
  p.C = a->cache_rows;
  p.W = a->row_bytes;
  p.tree_ld = a->tree_ld;
  p.cache_ld = a->cache_ld;
  p.tree = static_cast<const unsigned char*>(a->tree_rows);
  p.cache = static_cast<unsigned char*>(a->cache);
  p.path_nodes = a->path_nodes;
  p.path_len = a->path_len;
  p.prefix = a->prefix_len;
  p.seq_error = a->seq_error;
  p.error_word = a->error_word;
  const bool vec = multiple16(p.W) && multiple16(p.tree_ld) && multiple16(p.cache_ld) && aligned16(a->tree_rows) &&
                   aligned16(a->cache);
  const dim3 grid(static_cast<unsigned>(chunks), static_cast<unsigned>(p.D1), static_cast<unsigned>(p.B));
  if (vec) compact_kernel<true><<<grid, kCopyThreads, 0, stream>>>(p);
  else compact_kernel<false><<<grid, kCopyThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}
