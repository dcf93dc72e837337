// Internal helpers of the vc_* libraries: argument checks, error reporting,
// small device utilities (bf16/fp16 bit conversions, mbarrier and bulk-copy
// PTX).  Not part of the public ABI.
#ifndef VC_INTERNAL_H_
#define VC_INTERNAL_H_

#include <stddef.h>
#include <stdint.h>

#include "vc.h"

#ifdef __cplusplus
extern "C" {
#endif
/* Record a printf-style reason for the calling thread and return s. */
vc_status_t vc_internal_fail(vc_status_t s, const char* fmt, ...);
void vc_internal_clear(void);
#ifdef __cplusplus
}
#endif

#ifdef __CUDACC__
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#define VC_FAIL(st, ...) return vc_internal_fail((st), __VA_ARGS__)
#define VC_REQUIRE(cond, ...)                                   \
  do {                                                          \
    if (!(cond)) return vc_internal_fail(VC_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)
#define VC_CUDA_CHECK(expr)                                                     \
  do {                                                                          \
    cudaError_t e_ = (expr);                                                    \
    if (e_ != cudaSuccess)                                                      \
      return vc_internal_fail(VC_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)
// After a launch: report a launch-configuration error synchronously.
#define VC_LAUNCH_CHECK(name)                                                   \
  do {                                                                          \
    cudaError_t e_ = cudaGetLastError();                                        \
    if (e_ != cudaSuccess)                                                      \
      return vc_internal_fail(VC_ERR_CUDA, "%s launch: %s", name, cudaGetErrorString(e_)); \
  } while (0)

static inline bool vc_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device status flags (each library keeps its own word, see *_device_status).
enum : uint32_t {
  VC_DEV_BARRIER_TIMEOUT = 1u,
  VC_DEV_CAPACITY = 2u,
  VC_DEV_BAD_INDEX = 4u,
};

// ---------------------------------------------------------------- numbers
__device__ __forceinline__ float vc_bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t vc_f32_to_bf16_rn(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float vc_f16_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ uint16_t vc_f32_to_f16_rn(float x) { return __half_as_ushort(__float2half_rn(x)); }

// ---------------------------------------------------------------- PTX: mbarrier + bulk copy
__device__ __forceinline__ uint32_t vc_smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void vc_mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(vc_smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void vc_fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void vc_mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(vc_smem_addr(bar)), "r"(bytes)
               : "memory");
}
// One non-blocking probe of phase `parity`; true once that phase completed.
__device__ __forceinline__ bool vc_mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(vc_smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: gives up after ~`limit_cycles` SM clocks and returns false.
__device__ __forceinline__ bool vc_mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit_cycles) {
  if (vc_mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!vc_mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit_cycles) return false;
  }
  return true;
}
// Plain arrival (no transaction bytes) on an mbarrier.
__device__ __forceinline__ void vc_mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(vc_smem_addr(bar)) : "memory");
}
// Bounded wait that also gives up as soon as *abort is non-zero (another warp
// already gave up); on its own timeout it sets *abort.  Returns true once
// phase `parity` completed.
__device__ __forceinline__ bool vc_mbar_wait_or_abort(uint64_t* bar, uint32_t parity, volatile uint32_t* abort,
                                                      long long limit_cycles) {
  if (vc_mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!vc_mbar_try_wait(bar, parity)) {
    if (*abort != 0u) return false;
    if (clock64() - t0 > limit_cycles) {
      *abort = 1u;
      return false;
    }
  }
  return true;
}
// Barrier over the first `count` threads of the CTA (named barrier `id`, 1..15).
__device__ __forceinline__ void vc_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Barrier over the first `count` threads returning the OR of `pred` over them.
__device__ __forceinline__ bool vc_bar_red_or(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n"
      " setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
// Order this thread's earlier generic-proxy shared-memory accesses before its
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void vc_fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk (non-tensor) async copy global -> this CTA's shared memory; completion
// is signalled on `bar` as transaction bytes.  dst, src 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void vc_bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(vc_smem_addr(dst)), "l"(src), "r"(bytes), "r"(vc_smem_addr(bar))
      : "memory");
}
#endif  // __CUDACC__

#endif  // VC_INTERNAL_H_
