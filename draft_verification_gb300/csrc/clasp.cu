// CLaSp layer selection: the skip-set dynamic program over hidden states.
//
// Source: Pith review of "CLaSp: In-Context Layer Skip for Self-Speculative
// Decoding" (arXiv 2505.24196), "What carries the argument": g(i, j) is the
// best hidden state reachable by skipping j of the first i layers, scored by
// cosine similarity to the full model's state h_i; a backtracking pass
// recovers the skip set.  Referee report, minor comments 1 and 4: the
// transition D(i, j) = max{cos(h_i, g(i-1, j-1)), cos(h_i, f_{i-1}(g(i-1, j)))}.
//
// The layer functions are residual linear maps f_l(x) = x + W_l x with
// bfloat16 weights W_l [d, d] (out, in) and the product at full input
// precision: each float32 state is split into two bfloat16 terms, x = hi +
// lo with hi = bf16(x) and lo = bf16(x - hi) (x - hi is exact in float32),
// and W_l x = W_l hi + W_l lo on the tensor cores with float32 accumulation.
// The split carries about 16 significant bits of x, so the product does not
// depend on which way x rounds to bfloat16 (rounding x itself made float32
// and float64 runs of the same path drift apart by 5e-3 over 32 layers).
// A tie keeps the layer; backtracking follows the stored decisions.
//
// One call, per layer i = 1 .. L (the layer applied is l = i - 1):
//   1. the products Y = W_l [hi lo] for every state that can still reach
//      (L, M) and may keep layer l: one cuBLAS bf16 GEMM (m = d, n = 2 x B x
//      states, k = d) that streams W_l from HBM once for the whole batch;
//   2. clasp_step_kernel, one CTA per (sequence, state j), launched with
//      programmatic dependent launch so that its launch overlaps the GEMM's
//      tail (every memory access waits for the GEMM): the cosines of both
//      candidates with h_i (float32 sums), the decision, and the chosen state
//      written as the next g(i, j) in float32 and as its two bfloat16 terms.
// Then clasp_backtrack_kernel, one warp per sequence, stages the sequence's
// decisions in shared memory and walks them back from (L, M).
//
// Only states with max(0, M - (L - i)) <= j <= min(i, M) are evaluated: a
// state with fewer skips can no longer reach M skips by layer L, so it never
// feeds g(L, M).  This changes no decision that the backtracking visits.
//
// Precision: the sums of the five products are float32 (per-thread partials
// of at most d / 2048 float4 groups, then shuffle trees), relative error
// about 1e-6 at d = 4096, far inside the margin a decision needs to be
// reproducible against a float64 evaluation (1e-5 and more on the cosines).
//
// Workspace (every part 256-byte aligned):
//   G0, G1  float32 [M+1][B][d]        states g(i-1, .) and g(i, .), ping-pong
//   X       bfloat16 [M+1][2][B][d]    the states' hi and lo terms
//   Y       float32 [M+1][2][B][d]     W_l X
//   table   uint8 [B][L][M+1]          decisions (1 = skip)
//   blas    32 MiB                     cuBLAS workspace (no cuBLAS allocation)
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>

#include "internal.h"
#include "spec_verify.h"

namespace sv {
namespace {

constexpr int kStepThreads = 512;
constexpr int kStepWarps = kStepThreads / 32;
constexpr int kCached = 2;                            // float4 groups per thread kept in registers
constexpr size_t kBlasWorkspace = size_t(32) << 20;
constexpr int kMaxLayers = 4096;
constexpr int kMaxWidth = 65536;
constexpr int kBacktrackSmem = 48 * 1024;             // decisions staged per sequence

struct ClaspParams {
  int B, L, d, M;
  const float* h;              // [B][L+1][d]
  float* G[2];                 // [M+1][B][d]
  __nv_bfloat16* X;            // [M+1][2][B][d]
  const float* Y;              // [M+1][2][B][d]
  unsigned char* table;        // [B][L][M+1]
  int* mask;                   // [B][L]
  float* score;                // [B]
  unsigned char* choice;       // [B][L][M+1] or null
};

// States of layer i that can still reach (L, M).
__host__ __device__ inline int state_lo(int i, int L, int M) { return max(0, M - (L - i)); }
__host__ __device__ inline int state_hi(int i, int M) { return min(i, M); }

__device__ inline float dot4(float4 a, float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

__device__ inline float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

__device__ inline unsigned pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<unsigned*>(&v);
}

__device__ inline float2 unpack_bf16x2(unsigned u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

// Four state values as their hi terms (at hi) and lo terms (at lo).
__device__ inline void store_split4(__nv_bfloat16* hi, __nv_bfloat16* lo, float4 v) {
  uint2 h;
  h.x = pack_bf16x2(v.x, v.y);
  h.y = pack_bf16x2(v.z, v.w);
  const float2 h01 = unpack_bf16x2(h.x), h23 = unpack_bf16x2(h.y);
  uint2 l;
  l.x = pack_bf16x2(v.x - h01.x, v.y - h01.y);
  l.y = pack_bf16x2(v.z - h23.x, v.w - h23.y);
  *reinterpret_cast<uint2*>(hi) = h;
  *reinterpret_cast<uint2*>(lo) = l;
}

// g(0, 0) = h_0 for every sequence, and its two bfloat16 terms.
__global__ void __launch_bounds__(kStepThreads) clasp_init_kernel(ClaspParams p) {
  const int b = blockIdx.x;
  const size_t d = p.d;
  const float4* src = reinterpret_cast<const float4*>(p.h + static_cast<size_t>(b) * (p.L + 1) * d);
  float4* g = reinterpret_cast<float4*>(p.G[0] + static_cast<size_t>(b) * d);
  __nv_bfloat16* xh = p.X + static_cast<size_t>(b) * d;       // state 0, hi
  __nv_bfloat16* xl = xh + static_cast<size_t>(p.B) * d;       // state 0, lo
  for (int e = threadIdx.x; e < p.d / 4; e += kStepThreads) {
    const float4 v = src[e];
    g[e] = v;
    store_split4(xh + 4 * e, xl + 4 * e, v);
  }
}

// The five partial sums of one float4 group (see clasp_step_kernel).
struct Sums {
  float hh = 0.f, hk = 0.f, kk = 0.f, hs = 0.f, ss = 0.f;
};

// One DP step: state (layer i, j) of sequence b, j = state_lo(i) + blockIdx.y.
__global__ void __launch_bounds__(kStepThreads) clasp_step_kernel(ClaspParams p, int i, int prev) {
  const int b = blockIdx.x;
  const int j = state_lo(i, p.L, p.M) + blockIdx.y;
  const int B = p.B;
  const size_t d = p.d;
  const int n4 = p.d / 4;
  const bool can_keep = j <= i - 1;  // g(i-1, j) exists
  const bool can_skip = j >= 1;      // g(i-1, j-1) exists
  const float* Gp = p.G[prev];
  const float4* hv = reinterpret_cast<const float4*>(p.h + (static_cast<size_t>(b) * (p.L + 1) + i) * d);
  const float4* gk = reinterpret_cast<const float4*>(Gp + (static_cast<size_t>(j) * B + b) * d);
  const float4* yh = reinterpret_cast<const float4*>(p.Y + (static_cast<size_t>(j) * 2 * B + b) * d);
  const float4* yl = yh + static_cast<size_t>(B) * d / 4;
  const float4* gs = can_skip ? reinterpret_cast<const float4*>(Gp + (static_cast<size_t>(j - 1) * B + b) * d)
                              : nullptr;
  // the products of this layer (and, through stream order, everything
  // before them) are complete past this point
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // <h, h>, <h, k>, <k, k>, <h, s>, <s, s> with k = g(i-1, j) + W g(i-1, j)
  // the kept candidate and s = g(i-1, j-1) the skipped one; the first
  // kCached groups of each candidate stay in registers for the write-back
  Sums t;
  float4 kc[kCached], sc[kCached];
#pragma unroll
  for (int c = 0; c < kCached; ++c) {
    const int e = threadIdx.x + c * kStepThreads;
    kc[c] = sc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e < n4) {
      const float4 x = hv[e];
      t.hh = dot4(x, x, t.hh);
      if (can_keep) {
        kc[c] = add4(gk[e], add4(yh[e], yl[e]));
        t.hk = dot4(x, kc[c], t.hk);
        t.kk = dot4(kc[c], kc[c], t.kk);
      }
      if (can_skip) {
        sc[c] = gs[e];
        t.hs = dot4(x, sc[c], t.hs);
        t.ss = dot4(sc[c], sc[c], t.ss);
      }
    }
  }
  for (int e = threadIdx.x + kCached * kStepThreads; e < n4; e += kStepThreads) {
    const float4 x = hv[e];
    t.hh = dot4(x, x, t.hh);
    if (can_keep) {
      const float4 k = add4(gk[e], add4(yh[e], yl[e]));
      t.hk = dot4(x, k, t.hk);
      t.kk = dot4(k, k, t.kk);
    }
    if (can_skip) {
      const float4 s = gs[e];
      t.hs = dot4(x, s, t.hs);
      t.ss = dot4(s, s, t.ss);
    }
  }
  float v[5] = {t.hh, t.hk, t.kk, t.hs, t.ss};
#pragma unroll
  for (int q = 0; q < 5; ++q)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v[q] += __shfl_xor_sync(0xffffffffu, v[q], off);
  __shared__ float red[5][kStepWarps];
  __shared__ int decided;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
#pragma unroll
    for (int q = 0; q < 5; ++q) red[q][warp] = v[q];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int q = 0; q < 5; ++q) {
      float a = lane < kStepWarps ? red[q][lane] : 0.f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
      v[q] = a;
    }
    if (lane == 0) {
      const float nh = sqrtf(v[0]);
      const float cos_keep = v[1] / (nh * sqrtf(v[2]));
      const float cos_skip = v[3] / (nh * sqrtf(v[4]));
      // the larger cosine wins; a tie (or a NaN comparison) keeps the layer
      const bool skip = !can_keep || (can_skip && cos_skip > cos_keep);
      decided = skip;
      p.table[(static_cast<size_t>(b) * p.L + (i - 1)) * (p.M + 1) + j] = skip ? 1 : 0;
      if (i == p.L) p.score[b] = skip ? cos_skip : cos_keep;
    }
  }
  if (i == p.L) return;  // g(L, M) itself is not needed, only its score
  __syncthreads();
  const bool skip = decided;

  float4* gc = reinterpret_cast<float4*>(p.G[prev ^ 1] + (static_cast<size_t>(j) * B + b) * d);
  __nv_bfloat16* xh = p.X + (static_cast<size_t>(j) * 2 * B + b) * d;
  __nv_bfloat16* xl = xh + static_cast<size_t>(B) * d;
#pragma unroll
  for (int c = 0; c < kCached; ++c) {
    const int e = threadIdx.x + c * kStepThreads;
    if (e < n4) {
      const float4 w = skip ? sc[c] : kc[c];
      gc[e] = w;
      store_split4(xh + 4 * e, xl + 4 * e, w);
    }
  }
  for (int e = threadIdx.x + kCached * kStepThreads; e < n4; e += kStepThreads) {
    const float4 w = skip ? gs[e] : add4(gk[e], add4(yh[e], yl[e]));
    gc[e] = w;
    store_split4(xh + 4 * e, xl + 4 * e, w);
  }
}

// Backtracking from (L, M) over the stored decisions: one warp per sequence;
// the sequence's decisions are staged in shared memory when they fit.
__global__ void __launch_bounds__(32) clasp_backtrack_kernel(ClaspParams p) {
  extern __shared__ unsigned char staged[];
  const int b = blockIdx.x, lane = threadIdx.x;
  const int L = p.L, M = p.M;
  const size_t n = static_cast<size_t>(L) * (M + 1);
  const unsigned char* src = p.table + static_cast<size_t>(b) * n;
  const bool in_smem = n <= static_cast<size_t>(kBacktrackSmem);
  if (in_smem)
    for (size_t e = lane; e < n; e += 32) staged[e] = src[e];
  __syncwarp();
  const unsigned char* t = in_smem ? staged : src;
  if (lane == 0) {
    int j = M;
    for (int i = L; i >= 1; --i) {
      const int c = t[static_cast<size_t>(i - 1) * (M + 1) + j];
      p.mask[static_cast<size_t>(b) * L + (i - 1)] = c;
      j -= c;
    }
  }
  if (p.choice == nullptr) return;
  for (size_t e = lane; e < n; e += 32) {
    const int i = static_cast<int>(e / (M + 1)) + 1, jj = static_cast<int>(e % (M + 1));
    p.choice[static_cast<size_t>(b) * n + e] = (jj >= state_lo(i, L, M) && jj <= state_hi(i, M)) ? t[e] : 255;
  }
}

// One cuBLAS handle per device, created by the first call on the device and
// kept for the life of the process.  The handle's stream and workspace are
// set on every call, so the enqueue of a whole call holds the lock.
std::mutex g_blas_mutex;
std::map<int, cublasHandle_t> g_blas;

cublasHandle_t blas_handle_locked() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  auto it = g_blas.find(dev);
  if (it != g_blas.end()) return it->second;
  cublasHandle_t h = nullptr;
  if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return nullptr;
  g_blas.emplace(dev, h);
  return h;
}

struct Layout {
  size_t states, x, y, table, total;
};

Layout layout(int B, int L, int d, int M) {
  const size_t cells = static_cast<size_t>(M + 1) * B * d;
  Layout w;
  w.states = align256(cells * sizeof(float));
  w.x = align256(2 * cells * sizeof(__nv_bfloat16));
  w.y = align256(2 * cells * sizeof(float));
  w.table = align256(static_cast<size_t>(L) * (M + 1) * B);
  w.total = 2 * w.states + w.x + w.y + w.table + kBlasWorkspace;
  return w;
}

bool sizes_ok(int B, int L, int d, int M) {
  return B >= 1 && B <= kMaxSeq && L >= 1 && L <= kMaxLayers && d >= 8 && d <= kMaxWidth && d % 8 == 0 &&
         M >= 0 && M <= L;
}

// The step kernel of layer i, launched so that it may start while the
// layer's GEMM drains (it waits for the GEMM before any memory access).
cudaError_t launch_step(const ClaspParams& p, int i, int prev, cudaStream_t s) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.B, state_hi(i, p.M) - state_lo(i, p.L, p.M) + 1);
  cfg.blockDim = dim3(kStepThreads);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, clasp_step_kernel, p, i, prev);
}

cudaError_t launch_clasp(const ClaspParams& p, const __nv_bfloat16* W, cublasHandle_t blas, void* blas_ws,
                         cudaStream_t s) {
  if (cublasSetStream(blas, s) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  if (cublasSetWorkspace(blas, blas_ws, kBlasWorkspace) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  clasp_init_kernel<<<p.B, kStepThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const float one = 1.f, zero = 0.f;
  const size_t d = p.d;
  int prev = 0;
  for (int i = 1; i <= p.L; ++i) {
    const int lo = state_lo(i, p.L, p.M);
    const int last_keep = state_hi(i - 1, p.M);  // states of layer i-1 that may keep layer i-1
    if (lo <= last_keep) {
      const size_t off = static_cast<size_t>(lo) * 2 * p.B * d;
      const int n = (last_keep - lo + 1) * 2 * p.B;
      // Y[:, cols] = W_{i-1} X[:, cols] (hi and lo columns of each state);
      // column-major views: W_{i-1} stored [out][in] row-major is its
      // transpose with leading dimension d
      if (cublasGemmEx(blas, CUBLAS_OP_T, CUBLAS_OP_N, p.d, n, p.d, &one, W + static_cast<size_t>(i - 1) * d * d,
                       CUDA_R_16BF, p.d, p.X + off, CUDA_R_16BF, p.d, &zero, const_cast<float*>(p.Y) + off,
                       CUDA_R_32F, p.d, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
        return cudaErrorUnknown;
    }
    e = launch_step(p, i, prev, s);
    if (e != cudaSuccess) return e;
    prev ^= 1;
  }
  const size_t n = static_cast<size_t>(p.L) * (p.M + 1);
  const int smem = n <= static_cast<size_t>(kBacktrackSmem) ? static_cast<int>(n) : 0;
  clasp_backtrack_kernel<<<p.B, 32, smem, s>>>(p);
  return cudaGetLastError();
}

bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

}  // namespace
}  // namespace sv

extern "C" size_t spec_clasp_workspace_size(int B, int L, int d, int M) {
  if (!sv::sizes_ok(B, L, d, M)) return 0;
  return sv::layout(B, L, d, M).total;
}

extern "C" spec_status spec_clasp_layer_select(const spec_clasp_args* a, cudaStream_t stream) {
  sv::NvtxRange nvtx_range("spec_clasp_layer_select");
  using namespace sv;
  if (a == nullptr) return SPEC_EINVAL;
  if (!sizes_ok(a->B, a->L, a->d, a->M)) return SPEC_EINVAL;
  if (a->hidden == nullptr || a->weights == nullptr || a->skip_mask == nullptr || a->score == nullptr)
    return SPEC_EINVAL;
  if (!aligned16(a->hidden) || !aligned16(a->weights)) return SPEC_EALIGN;
  const Layout w = layout(a->B, a->L, a->d, a->M);
  if (a->workspace == nullptr || a->workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(a->workspace) & 255u))
    return SPEC_EWORKSPACE;
  char* ws = static_cast<char*>(a->workspace);
  ClaspParams p{};
  p.B = a->B;
  p.L = a->L;
  p.d = a->d;
  p.M = a->M;
  p.h = a->hidden;
  p.G[0] = reinterpret_cast<float*>(ws);
  p.G[1] = reinterpret_cast<float*>(ws + w.states);
  p.X = reinterpret_cast<__nv_bfloat16*>(ws + 2 * w.states);
  p.Y = reinterpret_cast<const float*>(ws + 2 * w.states + w.x);
  p.table = reinterpret_cast<unsigned char*>(ws + 2 * w.states + w.x + w.y);
  void* blas_ws = ws + 2 * w.states + w.x + w.y + w.table;
  p.mask = a->skip_mask;
  p.score = a->score;
  p.choice = a->choice;
  std::lock_guard<std::mutex> lock(g_blas_mutex);
  cublasHandle_t blas = blas_handle_locked();
  if (blas == nullptr) return SPEC_ECUDA;
  return launch_clasp(p, static_cast<const __nv_bfloat16*>(a->weights), blas, blas_ws, stream) == cudaSuccess
             ? SPEC_OK
             : SPEC_ECUDA;
}
