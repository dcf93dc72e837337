// libvc_accept: lowest-index argmax over the verify logits, first mismatch
// with the drafts, accepted length and bonus / correction token.
//
// VeriCache (gist.science/paper/2605.17613), Technical Summary, Core
// Algorithm, Acceptance: drafts are kept up to the first disagreement with
// the full-KV prediction; when all agree one more (bonus) token is kept.
// This library emits the full-KV prediction at the first disagreement in
// every case (bonus when n = k, correction otherwise).
//
// One launch.  Grid (S splits, B*(k+1) rows): each CTA scans 1/S of a row
// with 16-byte loads and writes its (max, lowest index) to the workspace;
// the last CTA of a request (per-request arrival counter, reset by that CTA)
// folds the partials in split order, so ties resolve to the lowest index,
// and writes n_acc / next_tok / argmax.  HBM-bound: B*(k+1)*V*4 bytes read.
#include <cfloat>

#include "vc_internal.h"

namespace {

constexpr int kThreads = 256;

struct Best {
  float v;
  int i;
};

// a beats b: larger value, or equal value at a lower index (IEEE ==, so
// -0.0 and +0.0 tie).
__device__ __forceinline__ bool beats(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

__host__ __device__ inline int accept_splits(int rows, int V) {
  int by_grid = (1216 + rows - 1) / rows;
  int by_len = (V + 2047) / 2048;
  int s = by_grid < by_len ? by_grid : by_len;
  return s < 1 ? 1 : s;
}

__global__ void __launch_bounds__(kThreads) accept_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ draft, int k, int V, int S,
    float* __restrict__ part_v, int* __restrict__ part_i, unsigned int* __restrict__ counter,
    int32_t* __restrict__ n_acc, int32_t* __restrict__ next_tok, int32_t* __restrict__ argmax_out) {
  const int split = blockIdx.x;
  const int row = blockIdx.y;             // b * (k+1) + i
  const int R = k + 1;
  const int b = row / R;
  const int span = (V + S - 1) / S;
  const int span4 = (span + 3) & ~3;      // keep split starts 16-byte aligned
  const int lo = split * span4;
  const int hi = min(V, lo + span4);
  const float* x = logits + static_cast<size_t>(row) * V;

  float bv = -INFINITY;
  int bi = INT_MAX;
  if (lo < hi) {
    if ((V & 3) == 0) {
      const float4* x4 = reinterpret_cast<const float4*>(x + lo);
      const int n4 = (hi - lo) >> 2;
      // 4 independent 16-byte loads in flight per thread
      int j = threadIdx.x;
      for (; j + 3 * kThreads < n4; j += 4 * kThreads) {
        float4 a0 = __ldcs(x4 + j), a1 = __ldcs(x4 + j + kThreads);
        float4 a2 = __ldcs(x4 + j + 2 * kThreads), a3 = __ldcs(x4 + j + 3 * kThreads);
        const float4 arr[4] = {a0, a1, a2, a3};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int base = lo + 4 * (j + u * kThreads);
          if (beats(arr[u].x, base + 0, bv, bi)) { bv = arr[u].x; bi = base + 0; }
          if (beats(arr[u].y, base + 1, bv, bi)) { bv = arr[u].y; bi = base + 1; }
          if (beats(arr[u].z, base + 2, bv, bi)) { bv = arr[u].z; bi = base + 2; }
          if (beats(arr[u].w, base + 3, bv, bi)) { bv = arr[u].w; bi = base + 3; }
        }
      }
      for (; j < n4; j += kThreads) {
        float4 a = __ldcs(x4 + j);
        const int base = lo + 4 * j;
        if (beats(a.x, base + 0, bv, bi)) { bv = a.x; bi = base + 0; }
        if (beats(a.y, base + 1, bv, bi)) { bv = a.y; bi = base + 1; }
        if (beats(a.z, base + 2, bv, bi)) { bv = a.z; bi = base + 2; }
        if (beats(a.w, base + 3, bv, bi)) { bv = a.w; bi = base + 3; }
      }
    } else {
      for (int j = lo + threadIdx.x; j < hi; j += kThreads) {
        float a = x[j];
        if (beats(a, j, bv, bi)) { bv = a; bi = j; }
      }
    }
  }
  // warp then block reduction with the same tie rule
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, bv, off);
    int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    if (beats(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  __shared__ float sv[kThreads / 32];
  __shared__ int si[kThreads / 32];
  __shared__ bool last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w)
      if (beats(sv[w], si[w], bv, bi)) { bv = sv[w]; bi = si[w]; }
    part_v[static_cast<size_t>(row) * S + split] = bv;
    part_i[static_cast<size_t>(row) * S + split] = bi;
    __threadfence();
    const unsigned int arrived = atomicAdd(counter + b, 1u);
    last = (arrived == static_cast<unsigned int>(S * R - 1));
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  // The last CTA of request b: fold partials per row (threads = rows).
  __shared__ int amax[64];
  for (int i = threadIdx.x; i < R; i += kThreads) {
    const size_t base = static_cast<size_t>(b * R + i) * S;
    float v = __ldcg(part_v + base);
    int id = __ldcg(part_i + base);
    for (int s = 1; s < S; ++s) {
      float ov = __ldcg(part_v + base + s);
      int oi = __ldcg(part_i + base + s);
      if (beats(ov, oi, v, id)) { v = ov; id = oi; }
    }
    amax[i] = id;
    if (argmax_out) argmax_out[b * R + i] = id;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = k;
    for (int i = 0; i < k; ++i)
      if (amax[i] != draft[b * k + i]) { n = i; break; }
    n_acc[b] = n;
    next_tok[b] = amax[n];
    counter[b] = 0u;    // leave the workspace zero-filled for the next call
  }
}

// Workspace: the B arrival counters first (their place does not depend on k
// or V, so one zero-filled workspace serves calls with any k and V for the
// same B), then the partial maxima and their indices.
size_t counter_bytes(int B) { return (static_cast<size_t>(B) * sizeof(unsigned int) + 255) & ~size_t(255); }

size_t ws_bytes(int B, int k, int V) {
  const int rows = B * (k + 1);
  const int S = accept_splits(rows, V);
  size_t part = static_cast<size_t>(rows) * S;
  size_t bytes = counter_bytes(B) + part * sizeof(float);
  bytes = (bytes + 255) & ~size_t(255);
  bytes += part * sizeof(int);
  return bytes;
}

}  // namespace

extern "C" vc_status_t vc_accept_workspace_size(int32_t B, int32_t k, int32_t V, size_t* bytes) {
  VC_REQUIRE(bytes != nullptr, "bytes is NULL");
  VC_REQUIRE(B >= 1 && k >= 0 && V >= 1, "need B >= 1, k >= 0, V >= 1 (got %d, %d, %d)", B, k, V);
  VC_REQUIRE(k + 1 <= 64, "k + 1 <= 64 rows per request (got k = %d)", k);
  *bytes = ws_bytes(B, k, V);
  return VC_OK;
}

extern "C" vc_status_t vc_accept(int32_t B, int32_t k, int32_t V, const float* logits,
                                 const int32_t* draft, int32_t* n_acc, int32_t* next_tok,
                                 int32_t* argmax, void* workspace, size_t workspace_bytes,
                                 vc_stream_t stream) {
  VC_REQUIRE(B >= 1 && k >= 0 && V >= 1, "need B >= 1, k >= 0, V >= 1 (got %d, %d, %d)", B, k, V);
  VC_REQUIRE(k + 1 <= 64, "k + 1 <= 64 rows per request (got k = %d)", k);
  VC_REQUIRE(logits && n_acc && next_tok, "logits, n_acc and next_tok must not be NULL");
  VC_REQUIRE(k == 0 || draft, "draft must not be NULL when k > 0");
  VC_REQUIRE(vc_aligned16(logits), "logits must be 16-byte aligned");
  VC_REQUIRE(static_cast<int64_t>(B) * (k + 1) <= 65535, "B*(k+1) <= 65535");
  const size_t need = ws_bytes(B, k, V);
  if (!workspace || workspace_bytes < need)
    VC_FAIL(VC_ERR_WORKSPACE, "accept workspace needs %zu bytes (got %zu)", need, workspace_bytes);
  VC_REQUIRE(vc_aligned16(workspace), "workspace must be 16-byte aligned");
  const int rows = B * (k + 1);
  const int S = accept_splits(rows, V);
  char* ws = static_cast<char*>(workspace);
  unsigned int* counter = reinterpret_cast<unsigned int*>(ws);
  size_t off = counter_bytes(B);
  float* part_v = reinterpret_cast<float*>(ws + off);
  off = (off + static_cast<size_t>(rows) * S * sizeof(float) + 255) & ~size_t(255);
  int* part_i = reinterpret_cast<int*>(ws + off);
  dim3 grid(S, rows);
  accept_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      logits, draft, k, V, S, part_v, part_i, counter, n_acc, next_tok, argmax);
  VC_LAUNCH_CHECK("accept_kernel");
  return VC_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant.
//
// Some callers of this library cannot allocate device memory at all: a plugin
// that a serving framework hands only its input and output buffers (the
// framework owns every byte of device memory and its budget), or a
// latency-critical loop where a cudaMalloc (which may synchronise the device)
// is not allowed.  For them vc_accept_noalloc keeps its scratch (the per-split
// partial maxima and the per-request arrival counters) in a fixed array that
// lives in the library's own device memory, loaded with the library.
//
// Limits: B * (k + 1) * S <= kNoAllocParts partials, where S is the number of
// splits per row (see accept_splits), and B <= kNoAllocRequests.  Every GPU
// that loads this library holds the 64 KiB array until the process exits.
// All calls share the array: two calls that overlap on the GPU (different
// streams, or different threads) race and give wrong results.
namespace {
constexpr int kNoAllocParts = 6144;
constexpr int kNoAllocRequests = 4096;
struct NoAllocScratch {
  float part_v[kNoAllocParts];
  int part_i[kNoAllocParts];
  unsigned int counter[kNoAllocRequests];
};
static __device__ __align__(256) NoAllocScratch g_accept_scratch;

// Device address of g_accept_scratch on the current device, looked up on
// every call (a host-side query, no allocation and no synchronisation), so
// that a new context after a device reset gets its own address.
vc_status_t scratch_address(NoAllocScratch** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_accept_scratch);
  if (e != cudaSuccess) VC_FAIL(VC_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  *out = static_cast<NoAllocScratch*>(p);
  return VC_OK;
}
}  // namespace

extern "C" vc_status_t vc_accept_noalloc(int32_t B, int32_t k, int32_t V, const float* logits,
                                         const int32_t* draft, int32_t* n_acc, int32_t* next_tok,
                                         int32_t* argmax, vc_stream_t stream) {
  VC_REQUIRE(B >= 1 && k >= 0 && V >= 1, "need B >= 1, k >= 0, V >= 1 (got %d, %d, %d)", B, k, V);
  VC_REQUIRE(k + 1 <= 64, "k + 1 <= 64 rows per request (got k = %d)", k);
  VC_REQUIRE(logits && n_acc && next_tok, "logits, n_acc and next_tok must not be NULL");
  VC_REQUIRE(k == 0 || draft, "draft must not be NULL when k > 0");
  VC_REQUIRE(vc_aligned16(logits), "logits must be 16-byte aligned");
  const int rows = B * (k + 1);
  const int S = accept_splits(rows, V);
  if (B > kNoAllocRequests)
    VC_FAIL(VC_ERR_CAPACITY, "vc_accept_noalloc: B = %d exceeds the fixed scratch limit of %d requests", B,
            kNoAllocRequests);
  if (static_cast<int64_t>(rows) * S > kNoAllocParts)
    VC_FAIL(VC_ERR_CAPACITY,
            "vc_accept_noalloc: B*(k+1)*splits = %d*%d exceeds the fixed scratch limit of %d partials "
            "(use vc_accept with a caller-provided workspace)",
            rows, S, kNoAllocParts);
  NoAllocScratch* sp = nullptr;
  vc_status_t st = scratch_address(&sp);
  if (st != VC_OK) return st;
  auto cs = reinterpret_cast<cudaStream_t>(stream);
  // the arrival counters must start at zero for every call
  VC_CUDA_CHECK(cudaMemsetAsync(sp->counter, 0, sizeof(unsigned int) * B, cs));
  dim3 grid(S, rows);
  accept_kernel<<<grid, kThreads, 0, cs>>>(logits, draft, k, V, S, sp->part_v, sp->part_i, sp->counter, n_acc,
                                           next_tok, argmax);
  VC_LAUNCH_CHECK("accept_kernel (no-alloc)");
  return VC_OK;
}
