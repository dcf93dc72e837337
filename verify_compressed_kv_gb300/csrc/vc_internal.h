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
#include <cuda.h>
#include <cudaTypedefs.h>
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
// As vc_mbar_wait_or_abort, but each probe lets the thread sleep up to
// `sleep_ns` nanoseconds for the phase (mbarrier.try_wait with a suspend-time
// hint) instead of spinning: a waiting warp takes no issue slots.
__device__ __forceinline__ bool vc_mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t sleep_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(vc_smem_addr(bar)), "r"(parity), "r"(sleep_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool vc_mbar_wait_sleep_or_abort(uint64_t* bar, uint32_t parity, volatile uint32_t* abort,
                                                            long long limit_cycles, uint32_t sleep_ns = 20000u) {
  if (vc_mbar_try_wait_sleep(bar, parity, sleep_ns)) return true;
  const long long t0 = clock64();
  while (!vc_mbar_try_wait_sleep(bar, parity, sleep_ns)) {
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

// TMA tensor copy (2-D tile at coordinates x (innermost), y) into this CTA's
// shared memory, completion as transaction bytes on `bar`.  x times the element
// size must be a multiple of 16 bytes.
__device__ __forceinline__ void vc_tma2(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(vc_smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(vc_smem_addr(bar))
      : "memory");
}
// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to
// the driver library); null when the driver does not provide it.
static inline PFN_cuTensorMapEncodeTiled_v12000 vc_tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// ---------------------------------------------------------------- PTX: tcgen05 (tensor cores with TMEM accumulators)
// Operand tiles live in shared memory as K-major core matrices without
// swizzle: a core matrix is 8 rows x 16 bytes (8 bf16 of the K axis), 128
// contiguous bytes; `lbo` is the byte distance between core matrices that
// are neighbours along K, `sbo` the distance between neighbouring 8-row
// groups.  Descriptor fields: start address >> 4 (bits 0-13), lbo >> 4
// (16-29), sbo >> 4 (32-45), descriptor version 1 (bit 46), no swizzle.
__device__ __forceinline__ uint64_t vc_tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Descriptor of a K-major operand in the 128-byte-swizzled layout: rows of
// 64 bf16 (128 B), 8-row atoms of 1024 B (1024-byte aligned) in which the
// 16-byte chunk c of row r sits at chunk c ^ (r % 8), the layout a TMA copy
// with 128-byte swizzle writes.  lbo = 16 (unused within a row), sbo = 1024,
// swizzle code 2 (bits 61-63).  A 16-channel step inside the row is +32 bytes
// on the start address.
__device__ __forceinline__ uint64_t vc_tc_desc_sw128(uint32_t saddr) {
  return vc_tc_desc(saddr, 16, 1024) | (2ull << 61);
}
// Instruction descriptor of an M x N x 16 kind::f16 product: bf16 A and B,
// fp32 D, both operands K-major (D format bit 4, A / B formats bits 7 / 10,
// N >> 3 at bit 17, M >> 4 at bit 24).  M = 128: N a multiple of 16 in
// [16, 256]; D row i is TMEM lane i, column j is TMEM column j.
__host__ __device__ constexpr uint32_t vc_tc_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// Instruction descriptor of an M x N x 16 kind::f16 product with fp16 A and B
// and fp32 D (A/B format fields 0).  A is K-major (or in TMEM); B is K-major,
// or MN-major when b_mn (bit 16).  M = 128: N a multiple of 16 in [16, 256].
__host__ __device__ constexpr uint32_t vc_tc_idesc_f16(int M, int N, bool b_mn) {
  return (1u << 4) | (b_mn ? (1u << 16) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// TMEM allocation of `ncols` columns (a power of two >= 32) by one whole
// warp; the base address is written to *slot (shared memory).
__device__ __forceinline__ void vc_tc_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(vc_smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void vc_tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (TMEM) = A . B^T (+ D if acc), issued by one thread.
__device__ __forceinline__ void vc_tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}
// D (TMEM) = A . B^T (+ D if acc) with A in TMEM: lane m holds row m, a 32-bit
// column holds two consecutive K elements (16-bit types), so one K = 16 step
// spans 8 columns from a_tmem.  Issued by one thread.
__device__ __forceinline__ void vc_tc_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}
// 16 consecutive 32-bit columns of the warp's 32 TMEM lanes from registers:
// thread i writes lane 32 (warp % 4) + i.  Asynchronous: tcgen05.wait::st
// (vc_tc_wait_st) before the values are relied on.
__device__ __forceinline__ void vc_tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void vc_tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Arrive once on `bar` when every earlier tcgen05.mma of this thread completed.
__device__ __forceinline__ void vc_tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   vc_smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void vc_tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void vc_tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 8 / 16 / 32 consecutive fp32 columns of the warp's 32 TMEM lanes (lane quarter
// warp % 4): thread i gets lane 32 (warp % 4) + i.  Load and wait in one
// statement, so no use of the values can move above the wait.
__device__ __forceinline__ void vc_tc_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void vc_tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void vc_tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// Several TMEM loads and one wait in a single statement: columns [0, N) from
// taddr (x64 = one load of 64 columns; the others combine 32-, 16- and 8-column
// loads), or two 32-column runs from taddr_a and taddr_b.

__device__ __forceinline__ void vc_tc_ld24(uint32_t taddr, float (&v)[24]) {
  uint32_t r[24];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%24];\n"
      "{\n .reg .b32 ta;\n add.u32 ta, %24, 16;\n tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [ta];\n}\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 24; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void vc_tc_ld40(uint32_t taddr, float (&v)[40]) {
  uint32_t r[40];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%40];\n"
      "{\n .reg .b32 ta;\n add.u32 ta, %40, 32;\n tcgen05.ld.sync.aligned.32x32b.x8.b32 {%32,%33,%34,%35,%36,%37,%38,%39}, [ta];\n}\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 40; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void vc_tc_ld48(uint32_t taddr, float (&v)[48]) {
  uint32_t r[48];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%48];\n"
      "{\n .reg .b32 ta;\n add.u32 ta, %48, 32;\n tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [ta];\n}\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 48; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void vc_tc_ld56(uint32_t taddr, float (&v)[56]) {
  uint32_t r[56];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%56];\n"
      "{\n .reg .b32 ta;\n add.u32 ta, %56, 32;\n tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [ta];\n}\n"
      "{\n .reg .b32 ta;\n add.u32 ta, %56, 48;\n tcgen05.ld.sync.aligned.32x32b.x8.b32 {%48,%49,%50,%51,%52,%53,%54,%55}, [ta];\n}\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 56; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void vc_tc_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void vc_tc_ld32x2(uint32_t taddr_a, uint32_t taddr_b, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr_a), "r"(taddr_b)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
#endif  // __CUDACC__

#endif  // VC_INTERNAL_H_
