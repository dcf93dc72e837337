// libvc_verify_attn: verify attention over the full KV, streamed from pinned
// host memory, and the commit of accepted tokens to that store.
//
// VeriCache (gist.science/paper/2605.17613), Technical Summary:
//   * Core Algorithm, Verification: one forward pass over the full KV checks
//     all k drafted tokens at once -> k + 1 causal query rows per request;
//   * Key System Innovations (1): verification is bound by the CPU-GPU
//     interconnect (loading the full KV) and by compute;
//   * Architecture Support, long-context decoding: the full KV sits in CPU
//     memory and is loaded to the GPU for verification.
//
// Data path: the host store is chunk-major, [chunk][K|V][B][Hkv][C][d] bf16,
// so each chunk is one contiguous copy.  The copy stream moves chunk c into
// ring slot c % S and records `copied[slot]`; the compute stream waits for it,
// runs the chunk kernel and records `consumed[slot]`, which the copy stream
// waits for before reusing the slot.  No host waits.
//
// Chunk kernel: grid (parts, row blocks, B*Hkv).  Each CTA owns up to 128
// query rows of one KV head ((k+1)*G rows: all verify positions x the G
// query heads sharing that KV head) and 1/parts of the chunk's tokens.  QK^T
// and PV run on the tcgen05 tensor cores with fp32 accumulators in TMEM, K/V
// tiles of 64 tokens arrive by TMA (two stages), the online softmax runs one
// row per thread out of TMEM.  The part's (max, sum, unnormalised output) is
// merged into a per-part running state in the workspace with the log-sum-exp
// rule, so any number of chunks needs only `parts` states.  The finish kernel
// (mma.sync m16n8k16: a few rows of new tokens) adds the causal block of the
// k+1 new tokens and merges everything into bf16 output.
#include <algorithm>
#include <cfloat>
#include <cstdlib>
#include <string>
#include <vector>

#include "vc_internal.h"

namespace {

__device__ uint32_t g_verify_status = 0;

constexpr int kTile = 64;              // tokens per K/V tile
constexpr int kMaxWarps = 8;           // 16 query rows per warp
// Launch bound of the attention kernels: 384 threads caps registers at 168, so three
// warps fit per scheduler and two CTAs of up to 6 warps share an SM (they launch
// with at most kMaxWarps warps)
constexpr int kBoundThreads = 384;
constexpr int kMaxPlannedParts = 16;   // vc_verify_attn_parts searches 1 .. 16
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = vc_smem_addr(smem);
  const int n = valid ? 16 : 0;        // src-size 0: fill with zeros, read nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(vc_smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(vc_smem_addr(p)));
}
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D (fp32)
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// 2^x (ex2.approx.ftz: relative error ~2^-22; results below 2^-126 flush to
// 0, far below what a bf16 softmax weight next to the row's max can hold)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 lanes in one 64-bit register pair (fma/add .f32x2, sm_100 and later).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// ------------------------------------------------------------------ kernel args
struct VerifyArgs {
  const uint16_t* q;          // [B, R, Hq, D]
  const uint16_t* k_src;      // chunk: [B, Hkv, C, D] (slot K half); new: [B, R, Hkv, D]
  const uint16_t* v_src;
  int B, Hq, Hkv, R, G, M;    // R = k + 1, M = R * G rows per KV head
  int C, chunk_start;         // chunk geometry (chunk kernel)
  const int32_t* prefix_len;  // [B]
  int parts, part_tokens;
  int first;                  // chunk kernel: overwrite the running state
  int any_chunk;              // finish kernel: merge the running state
  float scale_log2;
  float* st_o;                // [parts, B*Hkv, M, D] running unnormalised output
  float* st_ml;               // [parts, B*Hkv, M, 2] running (max, sum), log2 units
  uint16_t* out;              // [B, R, Hq, D]
};

template <int D>
struct Cfg {
  static constexpr int LD = D + 8;                  // padded smem row (bf16): conflict-free ldmatrix
  static constexpr int KSTEPS = D / 16;
  static constexpr int NT_O = D / 8;                // output n-tiles
};

template <int D>
size_t smem_bytes(int nw) {
  return (static_cast<size_t>(nw) * 16 + 4 * kTile) * Cfg<D>::LD * sizeof(uint16_t);
}

// Load a 64-token K or V tile (token rows [t0, t0 + 64) of `src`, row stride
// `rstride` elements, rows >= n_valid zero-filled) into smem [64][LD].
template <int D>
__device__ __forceinline__ void load_kv_tile(uint16_t* dst, const uint16_t* src, size_t rstride, int t0,
                                             int n_valid) {
  constexpr int VEC = D / 8;
  for (int i = threadIdx.x; i < kTile * VEC; i += blockDim.x) {
    const int t = i / VEC, v = i % VEC;
    const bool ok = (t0 + t) < n_valid;
    const uint16_t* g = src + (ok ? (static_cast<size_t>(t0 + t) * rstride + v * 8) : 0);
    cp_async16(dst + t * Cfg<D>::LD + v * 8, g, ok);
  }
}

// The attention core shared by the chunk and the finish kernels.  Computes,
// for the warp's 16 rows, the online-softmax state over tokens [t_lo, t_hi)
// of a source with `rstride`-element rows; `causal` masks token u for row r
// when u > r / G (new-token block).
template <int D>
__device__ void attend_range(const uint16_t* q_s, uint16_t* k_s, uint16_t* v_s, const uint16_t* ksrc,
                             const uint16_t* vsrc, size_t rstride, int t_lo, int t_hi, bool causal, int G,
                             int row0, float scale_log2, float (&acc)[Cfg<D>::NT_O][4], float (&m)[2],
                             float (&l)[2]) {
  constexpr int LD = Cfg<D>::LD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Q fragments of the warp's 16 rows, kept in registers
  uint32_t qa[Cfg<D>::KSTEPS][4];
#pragma unroll
  for (int ks = 0; ks < Cfg<D>::KSTEPS; ++ks) {
    const uint16_t* p = q_s + (warp * 16 + (lane & 15)) * LD + ks * 16 + (lane >> 4) * 8;
    ldsm_x4(qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], p);
  }
  const int n_tiles = (t_hi - t_lo + kTile - 1) / kTile;
  if (n_tiles <= 0) return;
  // prologue: tile 0 into buffer 0
  load_kv_tile<D>(k_s, ksrc, rstride, t_lo, t_hi);
  load_kv_tile<D>(v_s, vsrc, rstride, t_lo, t_hi);
  cp_async_commit();
  const int r_a = row0 + warp * 16 + (lane >> 2);   // this thread's rows: r_a, r_a + 8
  for (int it = 0; it < n_tiles; ++it) {
    const int buf = it & 1;
    if (it + 1 < n_tiles) {
      const int nb = buf ^ 1;
      load_kv_tile<D>(k_s + nb * kTile * LD, ksrc, rstride, t_lo + (it + 1) * kTile, t_hi);
      load_kv_tile<D>(v_s + nb * kTile * LD, vsrc, rstride, t_lo + (it + 1) * kTile, t_hi);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint16_t* kt = k_s + buf * kTile * LD;
    const uint16_t* vt = v_s + buf * kTile * LD;
    const int tok0 = t_lo + it * kTile;
    // S = Q K^T (16 x 64 per warp)
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < Cfg<D>::KSTEPS; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {              // pairs of n-tiles (16 tokens)
        uint32_t b0, b1, b2, b3;
        const uint16_t* p = kt + (np * 16 + (lane & 7) + ((lane >> 4) << 3)) * LD + ks * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x4(b0, b1, b2, b3, p);
        mma_bf16(s[2 * np], qa[ks], b0, b1);
        mma_bf16(s[2 * np + 1], qa[ks], b2, b3);
      }
    }
    // scale, mask, online softmax
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int u = tok0 + nt * 8 + (lane & 3) * 2 + (e & 1);
        const int r = r_a + (e >> 1) * 8;
        bool ok = u < t_hi;
        if (causal) ok = ok && (u <= r / G);
        s[nt][e] = ok ? s[nt][e] * scale_log2 : -INFINITY;
        mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
      }
    }
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float mn = fmaxf(m[h], mx[h]);
      alpha[h] = (mn == -INFINITY) ? 1.0f : exp2f(m[h] - mn);
      m[h] = mn;
      l[h] *= alpha[h];                              // rescale the running sum first
    }
    uint32_t pa[4][4];                               // P as A fragments (4 k-steps of 16 tokens)
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mm = m[e >> 1];
        p[e] = (mm == -INFINITY) ? 0.0f : exp2f(s[nt][e] - mm);
        l[e >> 1] += p[e];
      }
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p[0], p[1]);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p[2], p[3]);
    }
#pragma unroll
    for (int nt = 0; nt < Cfg<D>::NT_O; ++nt) {
      acc[nt][0] *= alpha[0];
      acc[nt][1] *= alpha[0];
      acc[nt][2] *= alpha[1];
      acc[nt][3] *= alpha[1];
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int np = 0; np < Cfg<D>::NT_O / 2; ++np) {
        uint32_t b0, b1, b2, b3;
        const uint16_t* p = vt + (kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3)) * LD + np * 16 + (lane >> 4) * 8;
        ldsm_x4_t(b0, b1, b2, b3, p);
        mma_bf16(acc[2 * np], pa[kk], b0, b1);
        mma_bf16(acc[2 * np + 1], pa[kk], b2, b3);
      }
    }
    __syncthreads();                                 // buffer `buf` is refilled next iteration
  }
}

// Load the CTA's query rows [row0, row0 + 16*nw) of KV head kvh into smem.
template <int D>
__device__ void load_q_rows(uint16_t* q_s, const VerifyArgs& a, int b, int kvh, int row0, int nw) {
  constexpr int VEC = D / 8;
  for (int i = threadIdx.x; i < nw * 16 * VEC; i += blockDim.x) {
    const int rr = i / VEC, v = i % VEC;
    const int r = row0 + rr;
    const bool ok = r < a.M;
    const int j = ok ? r / a.G : 0, g = ok ? r % a.G : 0;
    const uint16_t* src = a.q + ((static_cast<size_t>(b) * a.R + j) * a.Hq + kvh * a.G + g) * D + v * 8;
    cp_async16(q_s + rr * Cfg<D>::LD + v * 8, ok ? src : a.q, ok);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
}

// Thread-local l -> row sums over the quad of lanes that share a row.
__device__ __forceinline__ void finish_l(float (&l)[2]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
  }
}

// New-token causal block + merge of every part state -> bf16 output.
// grid (row blocks, B*Hkv).
template <int D>
__global__ void __launch_bounds__(kBoundThreads) verify_finish_kernel(VerifyArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr int LD = Cfg<D>::LD;
  const int nw = blockDim.x >> 5;
  uint16_t* q_s = reinterpret_cast<uint16_t*>(smem);
  uint16_t* k_s = q_s + nw * 16 * LD;
  uint16_t* v_s = k_s + 2 * kTile * LD;
  const int rb = blockIdx.x, bh = blockIdx.y;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int row0 = rb * nw * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc[Cfg<D>::NT_O][4];
#pragma unroll
  for (int nt = 0; nt < Cfg<D>::NT_O; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
  load_q_rows<D>(q_s, a, b, kvh, row0, nw);
  // new tokens of request b, KV head kvh: rows of [R, Hkv, D] with stride Hkv*D
  const size_t base = (static_cast<size_t>(b) * a.R * a.Hkv + kvh) * D;
  attend_range<D>(q_s, k_s, v_s, a.k_src + base, a.v_src + base, static_cast<size_t>(a.Hkv) * D, 0, a.R, true,
                  a.G, row0, a.scale_log2, acc, m, l);
  finish_l(l);
  const int r_a = row0 + warp * 16 + (lane >> 2);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = r_a + h * 8;
    if (r >= a.M) continue;
    // merge the part states (log-sum-exp), then normalise
    float M = m[h];
    if (a.any_chunk)
      for (int p = 0; p < a.parts; ++p) {
        const size_t row = (static_cast<size_t>(p) * a.B * a.Hkv + bh) * a.M + r;
        M = fmaxf(M, reinterpret_cast<const float2*>(a.st_ml)[row].x);
      }
    const float wn = exp2f(m[h] - M);            // m[h] is finite: token j sees itself
    float L = l[h] * wn;
    float o[Cfg<D>::NT_O][2];
#pragma unroll
    for (int nt = 0; nt < Cfg<D>::NT_O; ++nt) {
      o[nt][0] = acc[nt][h * 2] * wn;
      o[nt][1] = acc[nt][h * 2 + 1] * wn;
    }
    if (a.any_chunk)
      for (int p = 0; p < a.parts; ++p) {
        const size_t row = (static_cast<size_t>(p) * a.B * a.Hkv + bh) * a.M + r;
        const float2 ml = reinterpret_cast<const float2*>(a.st_ml)[row];
        if (ml.x == -INFINITY) continue;
        const float wp = exp2f(ml.x - M);
        L = fmaf(ml.y, wp, L);
        const float* so = a.st_o + row * D;
#pragma unroll
        for (int nt = 0; nt < Cfg<D>::NT_O; ++nt) {
          const float2 v = *reinterpret_cast<const float2*>(so + nt * 8 + (lane & 3) * 2);
          o[nt][0] = fmaf(v.x, wp, o[nt][0]);
          o[nt][1] = fmaf(v.y, wp, o[nt][1]);
        }
      }
    const float inv = 1.0f / L;
    const int j = r / a.G, g = r % a.G;
    uint16_t* dst = a.out + ((static_cast<size_t>(b) * a.R + j) * a.Hq + kvh * a.G + g) * D;
#pragma unroll
    for (int nt = 0; nt < Cfg<D>::NT_O; ++nt) {
      const uint32_t pk = pack_bf16(o[nt][0] * inv, o[nt][1] * inv);
      *reinterpret_cast<uint32_t*>(dst + nt * 8 + (lane & 3) * 2) = pk;
    }
  }
}

// ------------------------------------------------------------------ chunk kernel on tcgen05
// grid (parts, ceil(M / 128), B*Hkv); 6 warps:
//   * warps 0-3: one query row per thread (row = TMEM lane): load the CTA's
//     128 rows of Q into shared memory, then per tile read the row's scores S
//     from TMEM, keep the online softmax (max raised only past max + 2^8, the
//     row's O in TMEM rescaled when it is), write P as bf16 over the row's
//     scores, and at the end merge the row's (max, sum, O) into the part's
//     running state;
//   * warp 4, one thread: K and V tiles of 64 tokens by TMA (128-byte swizzle,
//     two stages);
//   * warp 5, one thread: S = Q . K^T (M = 128 rows, N = 64 tokens, K = d;
//     Q and K K-major in shared memory) and O += P . V (M = 128 rows, N = d,
//     K = 64 tokens; P from TMEM, V MN-major in shared memory), bf16 operands,
//     fp32 accumulators in TMEM.  Products of one thread run in issue order,
//     so S of tile i + 2 is written only after P of tile i has been read.
constexpr int kTcRows = 128;
constexpr int kTcTok = 64;
constexpr int kTcStages = 2;
constexpr int kTcThreads = 192;
constexpr long long kTcWait = 4000000000LL;   // ~2 s
constexpr float kTcLazy = 8.0f;

template <int D>
struct TcPlan {
  static constexpr int H = D / 64;                           // 64-channel (128-byte) column halves
  static constexpr uint32_t q_bytes = H * kTcRows * 128;
  static constexpr uint32_t kv_bytes = H * kTcTok * 128;     // one K or V tile
  static constexpr uint32_t stage = 2 * kv_bytes;
  static constexpr uint32_t off_st = q_bytes;
  static constexpr uint32_t off_bar = off_st + kTcStages * stage;
  // full_k[S], full_v[S], empty_k[S], empty_v[S], q_ready, s_full[2], p_ready[2], o_done[2], done
  static constexpr int n_bars = 4 * kTcStages + 8;
  static constexpr uint32_t off_misc = off_bar + n_bars * 8;   // TMEM base, abort flag
  static constexpr uint32_t total = off_misc + 16 + 1024;      // + room to align the base to 1024
  static constexpr uint32_t col_s = 0, col_o = 2 * kTcTok;    // TMEM: S[2] (P written over S), O
  static constexpr uint32_t alloc = col_o + D <= 256 ? 256 : 512;
};

template <int D>
__global__ void __launch_bounds__(kTcThreads) verify_chunk_tc(VerifyArgs a, const __grid_constant__ CUtensorMap tkv) {
  using P = TcPlan<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (vc_smem_addr(smem_raw) & 1023u)) & 1023u);   // swizzle atoms: 1024-aligned
  const int part = blockIdx.x, rb = blockIdx.y, bh = blockIdx.z;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int n_valid = min(max(a.prefix_len[b] - a.chunk_start, 0), a.C);
  const int t_lo = part * a.part_tokens;
  const int t_hi = min(n_valid, t_lo + a.part_tokens);
  const int n_tiles = t_hi > t_lo ? (t_hi - t_lo + kTcTok - 1) / kTcTok : 0;
  if (n_tiles == 0 && !a.first) return;                      // nothing to merge (uniform over the CTA)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P::off_bar);
  uint64_t* full_k = bars;
  uint64_t* full_v = bars + kTcStages;
  uint64_t* empty_k = bars + 2 * kTcStages;
  uint64_t* empty_v = bars + 3 * kTcStages;
  uint64_t* q_ready = bars + 4 * kTcStages;
  uint64_t* s_full = q_ready + 1;
  uint64_t* p_ready = s_full + 2;
  uint64_t* o_done = p_ready + 2;
  uint64_t* done = o_done + 2;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + P::off_misc);
  volatile uint32_t* abort = misc + 1;
  if (warp == 0) vc_tc_alloc(misc, P::alloc);
  if (threadIdx.x == 32) {
    for (int i = 0; i < 4 * kTcStages; ++i) vc_mbar_init(bars + i, 1);
    vc_mbar_init(q_ready, 4);
    for (int i = 0; i < 2; ++i) {
      vc_mbar_init(s_full + i, 1);
      vc_mbar_init(p_ready + i, 4);
      vc_mbar_init(o_done + i, 1);
    }
    vc_mbar_init(done, 1);
    *abort = 0u;
    vc_fence_mbar_init();
  }
  vc_tc_fence_before();
  __syncthreads();
  vc_tc_fence_after();
  const uint32_t tmem = misc[0];
  auto wait = [&](uint64_t* bar, uint32_t parity) { return vc_mbar_wait_sleep_or_abort(bar, parity, abort, kTcWait); };

  if (warp < 4) {
    // ---------------- one query row per thread
    const int rl = warp * 32 + lane, r = rb * kTcRows + rl;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bool ok = true;
    if (n_tiles > 0) {
      const bool rv = r < a.M;
      const int j = rv ? r / a.G : 0, g = rv ? r % a.G : 0;
      const uint16_t* src = a.q + ((static_cast<size_t>(b) * a.R + j) * a.Hq + kvh * a.G + g) * D;
#pragma unroll
      for (int c8 = 0; c8 < D / 8; ++c8) {                   // 128-byte swizzle: chunk c of row rl at c ^ (rl % 8)
        const uint4 v = rv ? *reinterpret_cast<const uint4*>(src + 8 * c8) : make_uint4(0u, 0u, 0u, 0u);
        const int h = c8 / 8, c = c8 % 8;
        *reinterpret_cast<uint4*>(smem + h * (kTcRows * 128) + (rl / 8) * 1024 + (rl % 8) * 128 + ((c ^ (rl % 8)) * 16)) = v;
      }
      vc_fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) vc_mbar_arrive(q_ready);
    }
    float m = -INFINITY, l = 0.0f;
    for (int i = 0; i < n_tiles; ++i) {
      const int bb = i & 1;
      ok = __all_sync(0xffffffffu, ok && wait(s_full + bb, static_cast<uint32_t>((i >> 1) & 1)));
      vc_tc_fence_after();
      float sv[kTcTok];
      __syncwarp();
      vc_tc_ld64(t_lane + P::col_s + bb * kTcTok, sv);
      // raw scores: the max commutes with the (positive) scale, which enters
      // once per tile here and once per score inside the exponent below
      const int t0 = t_lo + i * kTcTok;
      if (t0 + kTcTok > t_hi) {                              // a part's last tile: mask past t_hi
#pragma unroll
        for (int x = 0; x < kTcTok; ++x) sv[x] = (t0 + x < t_hi) ? sv[x] : -INFINITY;
      }
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int x = 0; x < kTcTok; x += 2) mq[(x >> 1) & 3] = fmax3(mq[(x >> 1) & 3], sv[x], sv[x + 1]);
      const float mx = fmax3(fmaxf(mq[0], mq[1]), mq[2], mq[3]) * a.scale_log2;
      // Raise the running max of the rows that outgrew it by more than kTcLazy
      // (log2 units; rare after the first tile).  The decision is per warp:
      // TMEM loads and stores are warp-collective, so every lane takes part and
      // the lanes that keep their max rescale by 1.
      const bool raise = mx > m + kTcLazy;
      if (__any_sync(0xffffffffu, raise)) {
        const float mn = raise ? mx : m;                     // finite: every tile holds a valid token
        const float alpha = fast_exp2(m - mn);               // m = -inf: 0
        if (i > 0 && ok) {                                   // O holds tiles 0 .. i-1: rescale it in TMEM
          ok = __all_sync(0xffffffffu, wait(o_done + ((i - 1) & 1), static_cast<uint32_t>(((i - 1) >> 1) & 1)));
          vc_tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            float ov[32];
            vc_tc_ld32(t_lane + P::col_o + c0, ov);
            uint32_t w0[16], w1[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
              w0[x] = __float_as_uint(ov[x] * alpha);
              w1[x] = __float_as_uint(ov[16 + x] * alpha);
            }
            vc_tc_st16(t_lane + P::col_o + c0, w0);
            vc_tc_st16(t_lane + P::col_o + c0 + 16, w1);
          }
          vc_tc_wait_st();
        }
        l *= alpha;
        m = mn;
      }
      // weights 2^(s * scale - m) two lanes per instruction; the sum in two
      // lane pairs
      uint32_t pk[kTcTok / 2];
      const uint64_t c2 = f2_pack(a.scale_log2, a.scale_log2), nm2 = f2_pack(-m, -m);
      uint64_t ps2[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
#pragma unroll
      for (int x = 0; x < kTcTok / 2; ++x) {
        float e0, e1;
        f2_unpack(f2_fma(f2_pack(sv[2 * x], sv[2 * x + 1]), c2, nm2), e0, e1);
        const float p0 = fast_exp2(e0), p1 = fast_exp2(e1);
        ps2[x & 1] = f2_add(ps2[x & 1], f2_pack(p0, p1));
        pk[x] = pack_bf16(p0, p1);
      }
      float q0, q1, q2, q3;
      f2_unpack(ps2[0], q0, q1);
      f2_unpack(ps2[1], q2, q3);
      l += (q0 + q1) + (q2 + q3);
      // P (bf16 pairs) over the first kTcTok / 2 columns of this tile's S
      __syncwarp();
      vc_tc_st16(t_lane + P::col_s + bb * kTcTok, *reinterpret_cast<const uint32_t(*)[16]>(pk));
      vc_tc_st16(t_lane + P::col_s + bb * kTcTok + 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + 16));
      vc_tc_wait_st();
      vc_tc_fence_before();
      __syncwarp();
      if (lane == 0) vc_mbar_arrive(p_ready + bb);
    }
    // ---------------- merge the row into the part's running state
    if (n_tiles > 0) {
      ok = ok && wait(o_done + ((n_tiles - 1) & 1), static_cast<uint32_t>(((n_tiles - 1) >> 1) & 1));
      vc_tc_fence_after();
    }
    ok = __all_sync(0xffffffffu, ok);
    const bool rv = r < a.M;
    // warp-uniform: the TMEM loads below are warp-collective, rows past M only skip the stores
    if (ok && __any_sync(0xffffffffu, rv)) {
      const size_t row = (static_cast<size_t>(part) * a.B * a.Hkv + bh) * a.M + (rv ? r : 0);
      float* so = a.st_o + row * D;
      float2* sml = reinterpret_cast<float2*>(a.st_ml) + row;
      float sa = 1.0f, sb = 0.0f, mo = m, lo = l;
      if (!a.first && rv) {
        const float2 old = *sml;
        const float mn = fmaxf(old.x, m);
        if (mn != -INFINITY) {
          sb = exp2f(old.x - mn);
          sa = exp2f(m - mn);
        }
        mo = mn;
        lo = old.y * sb + l * sa;
      }
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float ov[32];
        __syncwarp();
        if (n_tiles > 0) {
          vc_tc_ld32(t_lane + P::col_o + c0, ov);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) ov[x] = 0.0f;
        }
        if (rv) {
#pragma unroll
          for (int x = 0; x < 32; x += 4) {
            float4 v = make_float4(ov[x] * sa, ov[x + 1] * sa, ov[x + 2] * sa, ov[x + 3] * sa);
            if (!a.first) {
              const float4 o4 = *reinterpret_cast<const float4*>(so + c0 + x);
              v.x = fmaf(o4.x, sb, v.x);
              v.y = fmaf(o4.y, sb, v.y);
              v.z = fmaf(o4.z, sb, v.z);
              v.w = fmaf(o4.w, sb, v.w);
            }
            *reinterpret_cast<float4*>(so + c0 + x) = v;
          }
        }
      }
      if (rv) *sml = make_float2(mo, lo);
    }
  } else if (warp == 4) {
    // ---------------- K / V tiles by TMA, each ring refilled as soon as its own
    // consumer (S = Q.K^T for K, O += P.V for V) has completed on that stage
    if (lane == 0 && n_tiles > 0) {
      const int krow0 = (b * a.Hkv + kvh) * a.C;
      const int vrow0 = a.B * a.Hkv * a.C + krow0;
      int ik = 0, iv = 0;                                    // next K / V tile to issue
      long long t_last = clock64();
      while (ik < n_tiles || iv < n_tiles) {
        bool moved = false;
        if (ik < n_tiles && (ik < kTcStages ||
                             vc_mbar_try_wait(empty_k + ik % kTcStages, static_cast<uint32_t>(((ik / kTcStages) - 1) & 1)))) {
          uint8_t* st = smem + P::off_st + (ik % kTcStages) * P::stage;
          vc_mbar_arrive_expect_tx(full_k + ik % kTcStages, P::kv_bytes);
#pragma unroll
          for (int h = 0; h < P::H; ++h)
            vc_tma2(st + h * (kTcTok * 128), &tkv, 64 * h, krow0 + t_lo + ik * kTcTok, full_k + ik % kTcStages);
          ++ik;
          moved = true;
        }
        if (iv < n_tiles && (iv < kTcStages ||
                             vc_mbar_try_wait(empty_v + iv % kTcStages, static_cast<uint32_t>(((iv / kTcStages) - 1) & 1)))) {
          uint8_t* st = smem + P::off_st + (iv % kTcStages) * P::stage + P::kv_bytes;
          vc_mbar_arrive_expect_tx(full_v + iv % kTcStages, P::kv_bytes);
#pragma unroll
          for (int h = 0; h < P::H; ++h)
            vc_tma2(st + h * (kTcTok * 128), &tkv, 64 * h, vrow0 + t_lo + iv * kTcTok, full_v + iv % kTcStages);
          ++iv;
          moved = true;
        }
        if (moved) {
          t_last = clock64();
        } else {
          if (*abort != 0u) break;
          if (clock64() - t_last > kTcWait) {
            *abort = 1u;
            break;
          }
          __nanosleep(64);
        }
      }
      // every tile issued has landed before the CTA may exit
      for (int i = ik - kTcStages < 0 ? 0 : ik - kTcStages; i < ik; ++i)
        vc_mbar_wait_bounded(full_k + i % kTcStages, static_cast<uint32_t>((i / kTcStages) & 1), kTcWait);
      for (int i = iv - kTcStages < 0 ? 0 : iv - kTcStages; i < iv; ++i)
        vc_mbar_wait_bounded(full_v + i % kTcStages, static_cast<uint32_t>((i / kTcStages) & 1), kTcWait);
    }
  } else {
    // ---------------- products (one thread)
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t id_qk = vc_tc_idesc_bf16(128, kTcTok);
      constexpr uint32_t id_pv = vc_tc_idesc_bf16(128, D) | (1u << 16);    // V: MN-major B
      const uint32_t q_addr = vc_smem_addr(smem), st_addr = vc_smem_addr(smem + P::off_st);
      bool ok = wait(q_ready, 0);
      auto pv = [&](int t) {
        const int s = t % kTcStages, bb = t & 1;
        if (!wait(p_ready + bb, static_cast<uint32_t>((t >> 1) & 1))) return false;
        if (!wait(full_v + s, static_cast<uint32_t>((t / kTcStages) & 1))) return false;
        vc_tc_fence_after();
        const uint32_t v_addr = st_addr + s * P::stage + P::kv_bytes;
#pragma unroll
        for (int ks = 0; ks < kTcTok / 16; ++ks)
          vc_tc_mma_ta(tmem + P::col_o, tmem + P::col_s + bb * kTcTok + ks * 8,
                       vc_tc_desc(v_addr + ks * 2048, kTcTok * 128, 1024) | (2ull << 61), id_pv, t > 0 || ks > 0);
        vc_tc_commit(o_done + bb);
        vc_tc_commit(empty_v + s);
        return true;
      };
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int s = i % kTcStages, bb = i & 1;
        if (!wait(full_k + s, static_cast<uint32_t>((i / kTcStages) & 1))) {
          ok = false;
          break;
        }
        vc_tc_fence_after();
        const uint32_t k_addr = st_addr + s * P::stage;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          vc_tc_mma(tmem + P::col_s + bb * kTcTok,
                    vc_tc_desc_sw128(q_addr + (ks / 4) * (kTcRows * 128) + (ks % 4) * 32),
                    vc_tc_desc_sw128(k_addr + (ks / 4) * (kTcTok * 128) + (ks % 4) * 32), id_qk, ks > 0);
        vc_tc_commit(s_full + bb);
        vc_tc_commit(empty_k + s);                            // the K stage is free once S is computed
        if (i > 0) ok = pv(i - 1);
      }
      if (ok) ok = pv(n_tiles - 1);
      // every product issued has completed before TMEM is freed
      vc_tc_commit(done);
      vc_mbar_wait_bounded(done, 0, kTcWait);
      if (!ok) *abort = 1u;
    }
  }
  vc_tc_fence_before();
  __syncthreads();
  vc_tc_fence_after();
  if (threadIdx.x == 0 && *abort != 0u) atomicOr(&g_verify_status, VC_DEV_BARRIER_TIMEOUT);
  if (warp == 0) vc_tc_dealloc(tmem, P::alloc);
}

// Commit: grid (2 * Hkv, B), one CTA per (K|V, KV head, request).  Writes rows
// 0..n of k_new / v_new into the host store (mapped pinned memory) at the
// request's prefix length; commit_lengths_kernel advances the lengths after.
__global__ void commit_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                              const int32_t* __restrict__ n_acc, const int32_t* prefix_len, uint16_t* host_kv, int B,
                              int R, int Hkv, int D, int C, int T_cap) {
  const int kv = blockIdx.x / Hkv, h = blockIdx.x % Hkv, b = blockIdx.y;
  const int n = n_acc ? n_acc[b] : R - 1;
  const int len = prefix_len[b];
  if (n < 0 || n >= R || len < 0 || len + n + 1 > T_cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(&g_verify_status, VC_DEV_CAPACITY);
    return;
  }
  const int vec = D / 8;
  const uint16_t* base = kv ? v_new : k_new;
  for (int i = threadIdx.x; i < (n + 1) * vec; i += blockDim.x) {
    const int v = i % vec, r = i / vec;
    const int pos = len + r;
    const int chunk = pos / C, t = pos % C;
    const uint16_t* src = base + ((static_cast<size_t>(b) * R + r) * Hkv + h) * D + v * 8;
    uint16_t* dst = host_kv + ((((static_cast<size_t>(chunk) * 2 + kv) * B + b) * Hkv + h) * C + t) * D + v * 8;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

__global__ void commit_lengths_kernel(const int32_t* __restrict__ n_acc, int32_t* prefix_len, int B, int R, int T_cap) {
  __threadfence_system();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int n = n_acc ? n_acc[b] : R - 1;
    const int len = prefix_len[b];
    if (n < 0 || n >= R || len < 0 || len + n + 1 > T_cap) continue;
    prefix_len[b] = len + n + 1;
  }
}

// ------------------------------------------------------------------ host side
vc_status_t check(const vc_shape_t* s) {
  VC_REQUIRE(s != nullptr, "shape is NULL");
  VC_REQUIRE(s->B >= 1 && s->Hkv >= 1 && s->Hq >= s->Hkv && s->Hq % s->Hkv == 0, "bad B/Hq/Hkv");
  if (s->d != 64 && s->d != 128) VC_FAIL(VC_ERR_UNSUPPORTED, "head dim %d not in {64, 128}", s->d);
  VC_REQUIRE(s->k >= 0, "k >= 0");
  const int M = (s->k + 1) * (s->Hq / s->Hkv);
  if (M > 512) VC_FAIL(VC_ERR_UNSUPPORTED, "(k+1)*G = %d rows per KV head > 512", M);
  VC_REQUIRE(static_cast<int64_t>(s->B) * s->Hkv <= 65535, "B*Hkv <= 65535");
  return VC_OK;
}

struct Geometry {
  int M, nw, row_blocks;
};
Geometry geometry(const vc_shape_t* s) {
  Geometry g;
  g.M = (s->k + 1) * (s->Hq / s->Hkv);
  const int tiles = (g.M + 15) / 16;
  g.row_blocks = (tiles + kMaxWarps - 1) / kMaxWarps;
  g.nw = (tiles + g.row_blocks - 1) / g.row_blocks;     // balance warps over row blocks
  return g;
}

size_t ws_bytes(const vc_shape_t* s, int parts) {
  const size_t rows = static_cast<size_t>(parts) * s->B * s->Hkv * ((s->k + 1) * (s->Hq / s->Hkv));
  size_t o = rows * s->d * sizeof(float);
  o = (o + 255) & ~size_t(255);
  return o + rows * 2 * sizeof(float);
}

void fill_args(VerifyArgs& a, const vc_shape_t* s, int parts, void* ws) {
  a.B = s->B; a.Hq = s->Hq; a.Hkv = s->Hkv; a.R = s->k + 1; a.G = s->Hq / s->Hkv; a.M = a.R * a.G;
  a.parts = parts;
  a.scale_log2 = s->softmax_scale * kLog2e;
  const size_t rows = static_cast<size_t>(parts) * s->B * s->Hkv * a.M;
  a.st_o = static_cast<float*>(ws);
  a.st_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + ((rows * s->d * sizeof(float) + 255) & ~size_t(255)));
}

// Row blocks of the tcgen05 chunk kernel: 128 rows each.
int tc_row_blocks(const vc_shape_t* s) { return ((s->k + 1) * (s->Hq / s->Hkv) + kTcRows - 1) / kTcRows; }

template <int D>
vc_status_t tc_setup() {
  VC_CUDA_CHECK(cudaFuncSetAttribute(verify_chunk_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(TcPlan<D>::total)));
  VC_CUDA_CHECK(cudaFuncSetAttribute(verify_chunk_tc<D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared));   // two CTAs per SM
  return VC_OK;
}

// A chunk slot [K|V][B][Hkv][C][d] as one 2-D tensor of 2*B*Hkv*C rows of d
// bf16, in boxes of 64 channels x 64 tokens with the 128-byte swizzle (zero past the end).
template <int D>
vc_status_t launch_chunk(const VerifyArgs& a, const vc_shape_t* s, cudaStream_t cs) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = vc_tensor_map_encoder();
  if (!encode) VC_FAIL(VC_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  CUtensorMap tkv;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), 2ull * a.B * a.Hkv * a.C};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kTcTok)}, es[2] = {1, 1};
  const CUresult r = encode(&tkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.k_src), dims, strides,
                            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) VC_FAIL(VC_ERR_CUDA, "chunk tensor map: error %d", static_cast<int>(r));
  vc_status_t st = tc_setup<D>();
  if (st != VC_OK) return st;
  verify_chunk_tc<D><<<dim3(a.parts, tc_row_blocks(s), a.B * a.Hkv), kTcThreads, TcPlan<D>::total, cs>>>(a, tkv);
  VC_LAUNCH_CHECK("verify_chunk_tc");
  return VC_OK;
}

template <int D>
vc_status_t launch_finish(const VerifyArgs& a, const Geometry& g, cudaStream_t cs) {
  const size_t sm = smem_bytes<D>(g.nw);
  VC_CUDA_CHECK(cudaFuncSetAttribute(verify_finish_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm));
  verify_finish_kernel<D><<<dim3(g.row_blocks, a.B * a.Hkv), g.nw * 32, sm, cs>>>(a);
  VC_LAUNCH_CHECK("verify_finish_kernel");
  return VC_OK;
}

vc_status_t chunk_impl(const vc_shape_t* s, const uint16_t* q, const uint16_t* kv_slot, int C, int chunk_start,
                       const int32_t* prefix_len, int parts, int first, void* ws, cudaStream_t cs) {
  VerifyArgs a{};
  fill_args(a, s, parts, ws);
  a.q = q;
  a.k_src = kv_slot;
  a.v_src = kv_slot + static_cast<size_t>(s->B) * s->Hkv * C * s->d;
  a.C = C;
  a.chunk_start = chunk_start;
  a.prefix_len = prefix_len;
  a.part_tokens = ((C + parts - 1) / parts + kTcTok - 1) / kTcTok * kTcTok;
  a.first = first;
  return s->d == 128 ? launch_chunk<128>(a, s, cs) : launch_chunk<64>(a, s, cs);
}

vc_status_t finish_impl(const vc_shape_t* s, const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                        int parts, int any_chunk, uint16_t* out, void* ws, cudaStream_t cs) {
  VerifyArgs a{};
  fill_args(a, s, parts, ws);
  a.q = q;
  a.k_src = k_new;
  a.v_src = v_new;
  a.any_chunk = any_chunk;
  a.out = out;
  const Geometry g = geometry(s);
  return s->d == 128 ? launch_finish<128>(a, g, cs) : launch_finish<64>(a, g, cs);
}

vc_status_t check_pinned(const void* p) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    VC_FAIL(VC_ERR_INVALID_ARG, "host_kv: cudaPointerGetAttributes failed (%s)", cudaGetErrorString(e));
  }
  if (at.type != cudaMemoryTypeHost)
    VC_FAIL(VC_ERR_INVALID_ARG, "host_kv must be pinned host memory (cudaHostAlloc / pin_memory)");
  return VC_OK;
}

}  // namespace

// Ring of device slots and the events that order copies and kernels.
struct vc_verify_pipeline {
  int n_slots = 0;
  std::vector<cudaEvent_t> copied, consumed;
  std::vector<char> consumed_recorded;
  int issued = 0;        // chunks of the current pass already issued on the copy stream
};

namespace {
// Issue host->device copies of chunks [p->issued, upto) into their slots.
vc_status_t issue_copies(vc_verify_pipeline* p, const vc_shape_t* s, const uint16_t* host_kv, int C, int max_prefix,
                         uint16_t* dev_slots, int upto, cudaStream_t copy) {
  const size_t row_elems = static_cast<size_t>(C) * s->d;           // one (K|V, b, h) row of a chunk
  const size_t rows = 2 * static_cast<size_t>(s->B) * s->Hkv;
  const size_t chunk_elems = rows * row_elems;
  for (int c = p->issued; c < upto; ++c) {
    const int slot = c % p->n_slots;
    if (p->consumed_recorded[slot]) VC_CUDA_CHECK(cudaStreamWaitEvent(copy, p->consumed[slot], 0));
    const int n_tok = max_prefix - c * C < C ? max_prefix - c * C : C;
    uint16_t* dst = dev_slots + static_cast<size_t>(slot) * chunk_elems;
    const uint16_t* src = host_kv + static_cast<size_t>(c) * chunk_elems;
    if (n_tok == C) {
      VC_CUDA_CHECK(cudaMemcpyAsync(dst, src, chunk_elems * sizeof(uint16_t), cudaMemcpyHostToDevice, copy));
    } else {
      VC_CUDA_CHECK(cudaMemcpy2DAsync(dst, row_elems * sizeof(uint16_t), src, row_elems * sizeof(uint16_t),
                                      static_cast<size_t>(n_tok) * s->d * sizeof(uint16_t), rows,
                                      cudaMemcpyHostToDevice, copy));
    }
    VC_CUDA_CHECK(cudaEventRecord(p->copied[slot], copy));
  }
  if (upto > p->issued) p->issued = upto;
  return VC_OK;
}
}  // namespace

extern "C" vc_status_t vc_verify_attn_workspace_size(const vc_shape_t* s, int32_t parts_per_chunk, size_t* bytes) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE(bytes, "bytes is NULL");
  VC_REQUIRE(parts_per_chunk >= 1 && parts_per_chunk <= 64, "1 <= parts_per_chunk <= 64");
  *bytes = ws_bytes(s, parts_per_chunk);
  return VC_OK;
}

// Parts per chunk for a chunk launch: the most that keep all B * Hkv * row
// blocks * parts CTAs in one wave of the CTAs that fit at once (per SM from
// the kernel's registers, shared memory and TMEM columns, x SMs).  Each CTA
// walks ceil(tiles / parts) 64-token tiles and then merges its state.
namespace {
template <int D>
vc_status_t plan_parts(const vc_shape_t* s, int C, int* parts) {
  vc_status_t st = tc_setup<D>();
  if (st != VC_OK) return st;
  // CTAs resident per SM from the kernel's own limits: registers, shared memory
  // and TMEM columns (512 per SM)
  int dev = 0, sms = 0, smem_sm = 0, smem_rsv = 0;
  VC_CUDA_CHECK(cudaGetDevice(&dev));
  VC_CUDA_CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  VC_CUDA_CHECK(cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev));
  VC_CUDA_CHECK(cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev));
  cudaFuncAttributes fa{};
  VC_CUDA_CHECK(cudaFuncGetAttributes(&fa, verify_chunk_tc<D>));
  const int by_regs = 65536 / (((fa.numRegs + 7) / 8) * 8 * kTcThreads);
  const int by_smem = smem_sm / (static_cast<int>(TcPlan<D>::total) + smem_rsv);
  const int by_tmem = 512 / static_cast<int>(TcPlan<D>::alloc);
  const int per_sm = std::max(1, std::min(by_regs, std::min(by_smem, by_tmem)));
  const int64_t slots = static_cast<int64_t>(per_sm) * sms;
  const int64_t units = static_cast<int64_t>(s->B) * s->Hkv * tc_row_blocks(s);
  const int tiles = (C + kTcTok - 1) / kTcTok;
  // as many parts as keep every CTA in one wave: a second wave (or a CTA that
  // waits for a slot) costs more than the longer tile loop of fewer parts
  int64_t best = slots / std::max<int64_t>(1, units);
  best = std::max<int64_t>(1, std::min<int64_t>(best, std::min(tiles, kMaxPlannedParts)));
  *parts = static_cast<int>(best);
  return VC_OK;
}
}  // namespace

extern "C" vc_status_t vc_verify_attn_parts(const vc_shape_t* s, int32_t C, int32_t* parts) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE(C >= 1 && parts, "need C >= 1 and parts != NULL");
  int p = 1;
  st = s->d == 128 ? plan_parts<128>(s, C, &p) : plan_parts<64>(s, C, &p);
  if (st != VC_OK) return st;
  *parts = p;
  return VC_OK;
}

extern "C" vc_status_t vc_verify_attn_chunk(const vc_shape_t* s, const uint16_t* q, const uint16_t* kv_slot,
                                            int32_t C, int32_t chunk_start, const int32_t* prefix_len,
                                            int32_t parts_per_chunk, int32_t first, void* workspace,
                                            size_t workspace_bytes, vc_stream_t stream) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE(q && kv_slot && prefix_len, "NULL pointer");
  VC_REQUIRE(C >= 1 && chunk_start >= 0, "need C >= 1 and chunk_start >= 0");
  VC_REQUIRE(parts_per_chunk >= 1 && parts_per_chunk <= 64, "1 <= parts_per_chunk <= 64");
  VC_REQUIRE(vc_aligned16(q) && vc_aligned16(kv_slot), "pointers must be 16-byte aligned");
  const size_t need = ws_bytes(s, parts_per_chunk);
  if (!workspace || workspace_bytes < need)
    VC_FAIL(VC_ERR_WORKSPACE, "verify workspace needs %zu bytes (got %zu)", need, workspace_bytes);
  return chunk_impl(s, q, kv_slot, C, chunk_start, prefix_len, parts_per_chunk, first, workspace,
                    reinterpret_cast<cudaStream_t>(stream));
}

extern "C" vc_status_t vc_verify_attn_finish(const vc_shape_t* s, const uint16_t* q, const uint16_t* k_new,
                                             const uint16_t* v_new, int32_t parts_per_chunk, int32_t any_chunk,
                                             uint16_t* out, void* workspace, size_t workspace_bytes,
                                             vc_stream_t stream) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE(q && k_new && v_new && out, "NULL pointer");
  VC_REQUIRE(parts_per_chunk >= 1 && parts_per_chunk <= 64, "1 <= parts_per_chunk <= 64");
  VC_REQUIRE(vc_aligned16(q) && vc_aligned16(k_new) && vc_aligned16(v_new) && vc_aligned16(out),
             "pointers must be 16-byte aligned");
  const size_t need = ws_bytes(s, parts_per_chunk);
  if (!workspace || workspace_bytes < need)
    VC_FAIL(VC_ERR_WORKSPACE, "verify workspace needs %zu bytes (got %zu)", need, workspace_bytes);
  return finish_impl(s, q, k_new, v_new, parts_per_chunk, any_chunk, out, workspace,
                     reinterpret_cast<cudaStream_t>(stream));
}

extern "C" vc_status_t vc_verify_pipeline_create(int32_t n_slots, vc_verify_pipeline_t* out) {
  VC_REQUIRE(out, "out is NULL");
  VC_REQUIRE(n_slots >= 1 && n_slots <= 256, "1 <= n_slots <= 256");
  auto* p = new (std::nothrow) vc_verify_pipeline;
  if (!p) VC_FAIL(VC_ERR_CAPACITY, "out of host memory");
  p->n_slots = n_slots;
  p->copied.resize(n_slots);
  p->consumed.resize(n_slots);
  p->consumed_recorded.assign(n_slots, 0);
  for (int i = 0; i < n_slots; ++i) {
    cudaError_t e1 = cudaEventCreateWithFlags(&p->copied[i], cudaEventDisableTiming);
    cudaError_t e2 = cudaEventCreateWithFlags(&p->consumed[i], cudaEventDisableTiming);
    if (e1 != cudaSuccess || e2 != cudaSuccess) {
      for (int j = 0; j <= i; ++j) {
        if (p->copied[j]) cudaEventDestroy(p->copied[j]);
        if (p->consumed[j]) cudaEventDestroy(p->consumed[j]);
      }
      delete p;
      VC_FAIL(VC_ERR_CUDA, "cudaEventCreate: %s", cudaGetErrorString(e1 != cudaSuccess ? e1 : e2));
    }
  }
  *out = p;
  return VC_OK;
}

extern "C" vc_status_t vc_verify_pipeline_destroy(vc_verify_pipeline_t p) {
  if (!p) return VC_OK;
  for (int i = 0; i < p->n_slots; ++i) {
    cudaEventDestroy(p->copied[i]);
    cudaEventDestroy(p->consumed[i]);
  }
  delete p;
  return VC_OK;
}

extern "C" vc_status_t vc_verify_prefetch(vc_verify_pipeline_t p, const vc_shape_t* s, const uint16_t* host_kv,
                                          int32_t C, int32_t max_prefix, int32_t T_cap, uint16_t* dev_slots,
                                          vc_stream_t copy_stream) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE(p && host_kv && dev_slots, "NULL pointer");
  VC_REQUIRE(C >= 1 && T_cap >= 0 && T_cap % C == 0, "need C >= 1 and T_cap a multiple of C");
  VC_REQUIRE(max_prefix >= 0 && max_prefix <= T_cap, "max_prefix %d outside the store's 0 .. %d tokens", max_prefix,
             T_cap);
  if ((st = check_pinned(host_kv)) != VC_OK) return st;
  const int n_chunks = (max_prefix + C - 1) / C;
  const int upto = n_chunks < p->n_slots ? n_chunks : p->n_slots;
  return issue_copies(p, s, host_kv, C, max_prefix, dev_slots, upto, reinterpret_cast<cudaStream_t>(copy_stream));
}

extern "C" vc_status_t vc_verify_attn_streamed(vc_verify_pipeline_t p, const vc_shape_t* s, const uint16_t* q,
                                               const uint16_t* host_kv, int32_t C, int32_t max_prefix,
                                               int32_t T_cap, const int32_t* prefix_len, uint16_t* dev_slots,
                                               const uint16_t* k_new, const uint16_t* v_new, uint16_t* out,
                                               int32_t parts_per_chunk, void* workspace, size_t workspace_bytes,
                                               vc_stream_t compute_stream, vc_stream_t copy_stream) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE(p && q && host_kv && prefix_len && dev_slots && k_new && v_new && out, "NULL pointer");
  VC_REQUIRE(C >= 1 && T_cap >= 0 && T_cap % C == 0, "need C >= 1 and T_cap a multiple of C");
  VC_REQUIRE(max_prefix >= 0 && max_prefix <= T_cap, "max_prefix %d outside the store's 0 .. %d tokens", max_prefix,
             T_cap);
  VC_REQUIRE(parts_per_chunk >= 1 && parts_per_chunk <= 64, "1 <= parts_per_chunk <= 64");
  const size_t need = ws_bytes(s, parts_per_chunk);
  if (!workspace || workspace_bytes < need)
    VC_FAIL(VC_ERR_WORKSPACE, "verify workspace needs %zu bytes (got %zu)", need, workspace_bytes);
  // host-side fault injection for tests: fail before touching CUDA
  if (const char* f = std::getenv("VC_FAULT")) {
    if (std::string(f) == "h2d_fail") VC_FAIL(VC_ERR_CUDA, "injected host-to-device failure (VC_FAULT=h2d_fail)");
  }
  if ((st = check_pinned(host_kv)) != VC_OK) return st;
  auto cs = reinterpret_cast<cudaStream_t>(compute_stream);
  auto xs = reinterpret_cast<cudaStream_t>(copy_stream);
  const int n_chunks = (max_prefix + C - 1) / C;
  for (int c = 0; c < n_chunks; ++c) {
    const int upto = c + p->n_slots < n_chunks ? c + p->n_slots : n_chunks;
    if ((st = issue_copies(p, s, host_kv, C, max_prefix, dev_slots, upto, xs)) != VC_OK) return st;
    const int slot = c % p->n_slots;
    VC_CUDA_CHECK(cudaStreamWaitEvent(cs, p->copied[slot], 0));
    const uint16_t* slot_ptr = dev_slots + static_cast<size_t>(slot) * 2 * s->B * s->Hkv * C * s->d;
    if ((st = chunk_impl(s, q, slot_ptr, C, c * C, prefix_len, parts_per_chunk, c == 0, workspace, cs)) != VC_OK)
      return st;
    VC_CUDA_CHECK(cudaEventRecord(p->consumed[slot], cs));
    p->consumed_recorded[slot] = 1;
  }
  p->issued = 0;        // the next pass starts at chunk 0
  return finish_impl(s, q, k_new, v_new, parts_per_chunk, n_chunks > 0, out, workspace, cs);
}

extern "C" vc_status_t vc_verify_commit(const vc_shape_t* s, const uint16_t* k_new, const uint16_t* v_new,
                                        const int32_t* n_acc, int32_t* prefix_len, uint16_t* host_kv, int32_t C,
                                        int32_t T_cap, vc_stream_t stream) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE(k_new && v_new && prefix_len && host_kv, "NULL pointer");
  VC_REQUIRE(C >= 1 && T_cap >= 0 && T_cap % C == 0, "need C >= 1 and T_cap a multiple of C");
  VC_REQUIRE(vc_aligned16(k_new) && vc_aligned16(v_new) && vc_aligned16(host_kv), "pointers must be 16-byte aligned");
  if ((st = check_pinned(host_kv)) != VC_OK) return st;
  void* dptr = nullptr;
  VC_CUDA_CHECK(cudaHostGetDevicePointer(&dptr, const_cast<uint16_t*>(host_kv), 0));
  auto cs = reinterpret_cast<cudaStream_t>(stream);
  commit_kernel<<<dim3(2 * s->Hkv, s->B), 128, 0, cs>>>(k_new, v_new, n_acc, prefix_len, static_cast<uint16_t*>(dptr),
                                                        s->B, s->k + 1, s->Hkv, s->d, C, T_cap);
  VC_LAUNCH_CHECK("commit_kernel");
  commit_lengths_kernel<<<1, 256, 0, cs>>>(n_acc, prefix_len, s->B, s->k + 1, T_cap);
  VC_LAUNCH_CHECK("commit_lengths_kernel");
  return VC_OK;
}

extern "C" vc_status_t vc_verify_attn_device_status(uint32_t* status) {
  VC_REQUIRE(status, "status is NULL");
  VC_CUDA_CHECK(cudaDeviceSynchronize());
  uint32_t v = 0, zero = 0;
  VC_CUDA_CHECK(cudaMemcpyFromSymbol(&v, g_verify_status, sizeof(v)));
  VC_CUDA_CHECK(cudaMemcpyToSymbol(g_verify_status, &zero, sizeof(zero)));
  *status = v;
  return VC_OK;
}
