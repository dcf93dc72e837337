// libvc_draft_attn: decode attention over the KIVI-packed draft cache.
//
// VeriCache (gist.science/paper/2605.17613), Technical Summary, Core
// Algorithm (Drafting: candidate tokens come from the compressed KV) and Key
// System Innovations (drafting is bound by HBM bandwidth, reading the
// compressed KV).  One query token per request per step; all G query heads
// of a KV head share every byte read.
//
// Split-KV.  Grid (n_splits + 1, B*Hkv).  CTA x < n_splits owns 32-token
// groups [x*NGS, (x+1)*NGS) of the packed prefix of one (request, KV head):
//   1. one thread issues bulk async copies (cp.async.bulk, mbarrier
//      transaction count) of the split's K codes, K scale/zero, V codes and
//      V scale/zero into shared memory -- four contiguous ranges, since the
//      packed layout is group-major;
//   2. QK: lane (w, ts) of a warp holds word column w (32/bits channels) of
//      W tokens of a group, dequantises x^ = fma(code, s, z) exactly as the
//      quantiser defines it, multiplies by the lane's slice of q for all G
//      heads, and the W lanes of a token row are folded by recursive halving
//      (shuffles), leaving one token's G scores per lane;
//   3. exact softmax statistics of the split (max, sum of exp2) per head;
//   4. PV with the same lane mapping and per-token value scale/zero;
//   5. per-head partial output (normalised) and log2-sum-exp to workspace.
// CTA x == n_splits handles the bf16 tail (tokens committed since the last
// full group, plus earlier draft steps) and the current token, and stores
// the current token's K/V into the tail for the next steps.
// A second kernel merges the partials of every (request, query head).
#include <cfloat>

#include "vc_internal.h"

namespace {

__device__ uint32_t g_draft_status = 0;

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kGroup = 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitCycles = 4000000000LL;   // ~2 s at 2 GHz

struct DraftArgs {
  const uint16_t* q;        // [B, Hq, D]
  const uint16_t* k_cur;    // [B, Hkv, D] or null
  const uint16_t* v_cur;
  const uint32_t* kc;       // [B, Hkv, NG, W, 32]
  const uint16_t* ksz;      // [B, Hkv, NG, D, 2]
  const uint32_t* vc;
  const uint16_t* vsz;      // [B, Hkv, NG, D/32, 32, 2]
  const int32_t* packed_len;
  uint16_t* tail_k;         // [B, Hkv, tail_cap, D]
  uint16_t* tail_v;
  const int32_t* tail_len;
  int tail_cap, step;
  int Hq, Hkv, NG;          // NG = T_cap / 32
  int n_splits, NGS;        // packed splits per (b, h), groups per split
  float scale_log2;
  float* part_o;            // [B*Hq, n_splits + 1, D]
  float* part_lse;          // [B*Hq, n_splits + 1]
};

// Shared-memory carve-up (bytes), identical on host and device.
struct Smem {
  size_t kc, ksz, vc, vsz, q, sc, stat, bar, red, total;
};
__host__ __device__ inline size_t up16(size_t x) { return (x + 15) & ~size_t(15); }
__host__ __device__ inline Smem smem_plan(int D, int BITS, int G, int NGS, int tail_cap) {
  const int W = D * BITS / 32;
  const int toks = NGS * kGroup > tail_cap + 1 ? NGS * kGroup : tail_cap + 1;
  Smem s;
  size_t o = 0;
  s.kc = o;   o = up16(o + static_cast<size_t>(NGS) * W * kGroup * 4);
  s.ksz = o;  o = up16(o + static_cast<size_t>(NGS) * D * 4);
  s.vc = o;   o = up16(o + static_cast<size_t>(NGS) * W * kGroup * 4);
  s.vsz = o;  o = up16(o + static_cast<size_t>(NGS) * D * 4);
  s.q = o;    o = up16(o + static_cast<size_t>(G) * D * 4);
  s.sc = o;   o = up16(o + static_cast<size_t>(G) * toks * 4);
  s.stat = o; o = up16(o + 2 * 8 * 4);
  s.bar = o;  o = up16(o + 8);
  // the cross-warp output reduction (kWarps * G * D floats) reuses the key
  // staging [kc, vc), dead by then, when it fits
  const size_t red = static_cast<size_t>(kWarps) * G * D * 4;
  if (red <= s.vc) {
    s.red = s.kc;
  } else {
    s.red = o;
    o = up16(o + red);
  }
  s.total = o;
  return s;
}

template <int G>
__device__ __forceinline__ void load_q(const DraftArgs& a, int b, int kvh, float* q_s, int D) {
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    q_s[i] = vc_bf16_to_f32(a.q[(static_cast<size_t>(b) * a.Hq + kvh * G + h) * D + c]) * a.scale_log2;
  }
}

// Softmax statistics of `n` scores per head in sc_s[h * stride + t]: max m_h,
// p = exp2(s - m_h) written back, l_h = sum p.  One warp per head.
template <int G>
__device__ void softmax_stats(float* sc_s, int stride, int n, float* m_s, float* l_s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int h = warp; h < G; h += kWarps) {
    float* s = sc_s + h * stride;
    float m = -INFINITY;
    for (int t = lane; t < n; t += 32) m = fmaxf(m, s[t]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float l = 0.0f;
    for (int t = lane; t < n; t += 32) {
      const float p = exp2f(s[t] - m);
      s[t] = p;
      l += p;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane == 0) { m_s[h] = m; l_s[h] = l; }
  }
}

template <int D, int BITS, int G>
__global__ void __launch_bounds__(kThreads) draft_split_kernel(DraftArgs a) {
  constexpr int W = D * BITS / 32;         // words per token
  constexpr int CPW = 32 / BITS;           // channels per word
  constexpr int TS = 32 / W;               // token rows per warp
  constexpr int TPL = W;                   // tokens per lane per group
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  constexpr int NC = D / kGroup;           // value channel groups
  // accumulator channel block for PV: keep G * CB <= 64 registers
  constexpr int CB = (G * CPW <= 64) ? CPW : ((64 / G) >= 8 ? 8 : 4);
  static_assert(CPW % CB == 0 && CB % 4 == 0, "channel block");

  extern __shared__ __align__(16) uint8_t smem[];
  const Smem P = smem_plan(D, BITS, G, a.NGS, a.tail_cap);
  uint32_t* kc_s = reinterpret_cast<uint32_t*>(smem + P.kc);
  const uint16_t* ksz_s = reinterpret_cast<const uint16_t*>(smem + P.ksz);
  uint32_t* vc_s = reinterpret_cast<uint32_t*>(smem + P.vc);
  const uint16_t* vsz_s = reinterpret_cast<const uint16_t*>(smem + P.vsz);
  float* q_s = reinterpret_cast<float*>(smem + P.q);
  float* sc_s = reinterpret_cast<float*>(smem + P.sc);
  float* m_s = reinterpret_cast<float*>(smem + P.stat);
  float* l_s = m_s + 8;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + P.bar);
  float* red_s = reinterpret_cast<float*>(smem + P.red);

  const int split = blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int n_parts = a.n_splits + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = lane % W, ts = lane / W;

  const int ng_req = a.packed_len[b] / kGroup;
  const int g0 = split * a.NGS;
  const int ng = min(a.NGS, ng_req - g0);
  if (ng <= 0) {                           // nothing of this request in this split
    for (int h = threadIdx.x; h < G; h += blockDim.x)
      a.part_lse[static_cast<size_t>(b * a.Hq + kvh * G + h) * n_parts + split] = -INFINITY;
    return;
  }
  // ---- 1. stage the split's packed bytes with bulk async copies
  if (threadIdx.x == 0) {
    vc_mbar_init(bar, 1);
    vc_fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const size_t gbase = static_cast<size_t>(bh) * a.NG + g0;
    const uint32_t code_bytes = static_cast<uint32_t>(ng) * W * kGroup * 4;
    const uint32_t meta_bytes = static_cast<uint32_t>(ng) * D * 4;
    vc_mbar_arrive_expect_tx(bar, 2 * code_bytes + 2 * meta_bytes);
    vc_bulk_g2s(kc_s, a.kc + gbase * W * kGroup, code_bytes, bar);
    vc_bulk_g2s(smem + P.ksz, a.ksz + gbase * D * 2, meta_bytes, bar);
    vc_bulk_g2s(vc_s, a.vc + gbase * W * kGroup, code_bytes, bar);
    vc_bulk_g2s(smem + P.vsz, a.vsz + gbase * D * 2, meta_bytes, bar);
  }
  load_q<G>(a, b, kvh, q_s, D);
  __syncthreads();
  if (!vc_mbar_wait_bounded(bar, 0, kWaitCycles)) {
    if (threadIdx.x == 0) atomicOr(&g_draft_status, VC_DEV_BARRIER_TIMEOUT);
    for (int h = threadIdx.x; h < G; h += blockDim.x)
      a.part_lse[static_cast<size_t>(b * a.Hq + kvh * G + h) * n_parts + split] = -INFINITY;
    return;
  }
  const int n_tok = ng * kGroup;
  const int stride = a.NGS * kGroup;

  // ---- 2. QK^T with fused dequantisation
  for (int g = warp; g < ng; g += kWarps) {
    uint32_t words[TPL];
#pragma unroll
    for (int tl = 0; tl < TPL; tl += 4) {
      const uint4 v4 = *reinterpret_cast<const uint4*>(kc_s + (g * W + w) * kGroup + ts * TPL + tl);
      words[tl] = v4.x; words[tl + 1] = v4.y; words[tl + 2] = v4.z; words[tl + 3] = v4.w;
    }
    float part[G][TPL];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int tl = 0; tl < TPL; ++tl) part[h][tl] = 0.0f;
#pragma unroll
    for (int cb = 0; cb < CPW / 4; ++cb) {
      const int c0 = w * CPW + cb * 4;
      const uint4 mz = *reinterpret_cast<const uint4*>(ksz_s + (g * D + c0) * 2);   // 4 x (s, z)
      const __half2* sz = reinterpret_cast<const __half2*>(&mz);
      float s[4], z[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float2 f = __half22float2(sz[jj]);
        s[jj] = f.x;
        z[jj] = f.y;
      }
      float qv[G][4];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float4 q4 = *reinterpret_cast<const float4*>(q_s + h * D + c0);
        qv[h][0] = q4.x; qv[h][1] = q4.y; qv[h][2] = q4.z; qv[h][3] = q4.w;
      }
#pragma unroll
      for (int tl = 0; tl < TPL; ++tl) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const float code = static_cast<float>((words[tl] >> (BITS * (cb * 4 + jj))) & MASK);
          const float kh = fmaf(code, s[jj], z[jj]);
#pragma unroll
          for (int h = 0; h < G; ++h) part[h][tl] = fmaf(qv[h][jj], kh, part[h][tl]);
        }
      }
    }
    // fold the W lanes of this token row; afterwards part[h][0] = token (ts*W + w)
#pragma unroll
    for (int o = W / 2; o >= 1; o >>= 1) {
      const bool up = (w & o) != 0;
#pragma unroll
      for (int i = 0; i < o; ++i) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float send = up ? part[h][i] : part[h][i + o];
          const float keep = up ? part[h][i + o] : part[h][i];
          part[h][i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) sc_s[h * stride + g * kGroup + ts * TPL + w] = part[h][0];
  }
  __syncthreads();
  // ---- 3. softmax statistics of the split
  softmax_stats<G>(sc_s, stride, n_tok, m_s, l_s);
  __syncthreads();
  // ---- 4. PV with per-token value scale / zero
  const int cgrp = (w * CPW) / kGroup;        // the lane's value channel group
#pragma unroll 1
  for (int cbk = 0; cbk < CPW / CB; ++cbk) {
    float acc[G][CB];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int jj = 0; jj < CB; ++jj) acc[h][jj] = 0.0f;
    for (int g = warp; g < ng; g += kWarps) {
      uint32_t words[TPL];
#pragma unroll
      for (int tl = 0; tl < TPL; tl += 4) {
        const uint4 v4 = *reinterpret_cast<const uint4*>(vc_s + (g * W + w) * kGroup + ts * TPL + tl);
        words[tl] = v4.x; words[tl + 1] = v4.y; words[tl + 2] = v4.z; words[tl + 3] = v4.w;
      }
#pragma unroll
      for (int tl = 0; tl < TPL; ++tl) {
        const int t = g * kGroup + ts * TPL + tl;
        const __half2 szh = *reinterpret_cast<const __half2*>(vsz_s + ((g * NC + cgrp) * kGroup + ts * TPL + tl) * 2);
        const float2 sz = __half22float2(szh);
        float p[G];
#pragma unroll
        for (int h = 0; h < G; ++h) p[h] = sc_s[h * stride + t];
#pragma unroll
        for (int jj = 0; jj < CB; ++jj) {
          const float code = static_cast<float>((words[tl] >> (BITS * (cbk * CB + jj))) & MASK);
          const float vh = fmaf(code, sz.x, sz.y);
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h][jj] = fmaf(p[h], vh, acc[h][jj]);
        }
      }
    }
    // fold the TS token rows (lanes w, w+W, ...)
#pragma unroll
    for (int o = W; o < 32; o <<= 1)
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int jj = 0; jj < CB; ++jj) acc[h][jj] += __shfl_xor_sync(0xffffffffu, acc[h][jj], o);
    if (cbk == 0) __syncthreads();          // K staging is dead from here: reuse it
    if (ts == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int jj = 0; jj < CB; ++jj) red_s[(warp * G + h) * D + w * CPW + cbk * CB + jj] = acc[h][jj];
    }
  }
  __syncthreads();
  // ---- 5. partial output of the split
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    float o = 0.0f;
#pragma unroll
    for (int x = 0; x < kWarps; ++x) o += red_s[(x * G + h) * D + c];
    const size_t row = static_cast<size_t>(b * a.Hq + kvh * G + h) * n_parts + split;
    a.part_o[row * D + c] = o / l_s[h];
    if (c == 0) a.part_lse[row] = m_s[h] + log2f(l_s[h]);
  }
}

// The bf16 tail (+ the current token): grid (1, B*Hkv) launched as part of
// the same kernel family; simple warp-per-token dots.
template <int D, int G>
__global__ void __launch_bounds__(kThreads) draft_tail_kernel(DraftArgs a, int BITS) {
  extern __shared__ __align__(16) uint8_t smem[];
  const Smem P = smem_plan(D, BITS, G, a.NGS, a.tail_cap);
  float* q_s = reinterpret_cast<float*>(smem + P.q);
  float* sc_s = reinterpret_cast<float*>(smem + P.sc);
  float* m_s = reinterpret_cast<float*>(smem + P.stat);
  float* l_s = m_s + 8;
  const int bh = blockIdx.y;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int n_parts = a.n_splits + 1;
  const int split = a.n_splits;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tail = a.tail_len[b] + a.step;
  const bool has_cur = a.k_cur != nullptr;
  const int n_tok = n_tail + (has_cur ? 1 : 0);
  const size_t tbase = static_cast<size_t>(bh) * a.tail_cap * D;
  if (n_tail < 0 || n_tok > a.tail_cap + 1 || (has_cur && n_tail >= a.tail_cap)) {
    if (threadIdx.x == 0) atomicOr(&g_draft_status, VC_DEV_CAPACITY);
    for (int h = threadIdx.x; h < G; h += blockDim.x)
      a.part_lse[static_cast<size_t>(b * a.Hq + kvh * G + h) * n_parts + split] = -INFINITY;
    return;
  }
  if (n_tok == 0) {
    for (int h = threadIdx.x; h < G; h += blockDim.x)
      a.part_lse[static_cast<size_t>(b * a.Hq + kvh * G + h) * n_parts + split] = -INFINITY;
    return;
  }
  load_q<G>(a, b, kvh, q_s, D);
  __syncthreads();
  const int stride = a.tail_cap + 1;
  // scores: warp per token, lanes over channels
  for (int t = warp; t < n_tok; t += kWarps) {
    const uint16_t* kr = (t < n_tail) ? a.tail_k + tbase + static_cast<size_t>(t) * D
                                      : a.k_cur + static_cast<size_t>(bh) * D;
    float part[G];
#pragma unroll
    for (int h = 0; h < G; ++h) part[h] = 0.0f;
    for (int c = lane; c < D; c += 32) {
      const float kv = vc_bf16_to_f32(kr[c]);
#pragma unroll
      for (int h = 0; h < G; ++h) part[h] = fmaf(q_s[h * D + c], kv, part[h]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) part[h] += __shfl_xor_sync(0xffffffffu, part[h], off);
      if (lane == 0) sc_s[h * stride + t] = part[h];
    }
  }
  __syncthreads();
  softmax_stats<G>(sc_s, stride, n_tok, m_s, l_s);
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    float o = 0.0f;
    for (int t = 0; t < n_tok; ++t) {
      const uint16_t* vr = (t < n_tail) ? a.tail_v + tbase + static_cast<size_t>(t) * D
                                        : a.v_cur + static_cast<size_t>(bh) * D;
      o = fmaf(sc_s[h * stride + t], vc_bf16_to_f32(vr[c]), o);
    }
    const size_t row = static_cast<size_t>(b * a.Hq + kvh * G + h) * n_parts + split;
    a.part_o[row * D + c] = o / l_s[h];
    if (c == 0) a.part_lse[row] = m_s[h] + log2f(l_s[h]);
  }
  // keep the current token for the following draft steps
  if (has_cur) {
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
      a.tail_k[tbase + static_cast<size_t>(n_tail) * D + c] = a.k_cur[static_cast<size_t>(bh) * D + c];
      a.tail_v[tbase + static_cast<size_t>(n_tail) * D + c] = a.v_cur[static_cast<size_t>(bh) * D + c];
    }
  }
}

// out[b, h, :] = sum_x 2^(lse_x - M) o_x / sum_x 2^(lse_x - M); grid B*Hq.
__global__ void combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse, int n_parts,
                               int D, uint16_t* __restrict__ out) {
  const int row = blockIdx.x;
  const float* lse = part_lse + static_cast<size_t>(row) * n_parts;
  float M = -INFINITY;
  for (int x = 0; x < n_parts; ++x) M = fmaxf(M, lse[x]);
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float num = 0.0f, den = 0.0f;
    if (M != -INFINITY) {
      for (int x = 0; x < n_parts; ++x) {
        if (lse[x] == -INFINITY) continue;
        const float wgt = exp2f(lse[x] - M);
        num = fmaf(wgt, part_o[(static_cast<size_t>(row) * n_parts + x) * D + c], num);
        den += wgt;
      }
    }
    out[static_cast<size_t>(row) * D + c] = vc_f32_to_bf16_rn(den > 0.0f ? num / den : 0.0f);
  }
}

int groups_per_split(int bits) { return bits == 2 ? 16 : 8; }

vc_status_t check(const vc_shape_t* s) {
  VC_REQUIRE(s != nullptr, "shape is NULL");
  VC_REQUIRE(s->B >= 1 && s->Hkv >= 1 && s->Hq >= s->Hkv && s->Hq % s->Hkv == 0, "bad B/Hq/Hkv");
  if (s->d != 64 && s->d != 128) VC_FAIL(VC_ERR_UNSUPPORTED, "head dim %d not in {64, 128}", s->d);
  if (s->bits != 2 && s->bits != 4) VC_FAIL(VC_ERR_UNSUPPORTED, "bits %d not in {2, 4}", s->bits);
  const int G = s->Hq / s->Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 5 && G != 8) VC_FAIL(VC_ERR_UNSUPPORTED, "G = %d not in {1,2,4,5,8}", G);
  return VC_OK;
}

size_t ws_bytes(const vc_shape_t* s, int max_packed) {
  const int NGS = groups_per_split(s->bits);
  const int n_splits = (max_packed / kGroup + NGS - 1) / NGS;
  const size_t rows = static_cast<size_t>(s->B) * s->Hq * (n_splits + 1);
  size_t bytes = rows * s->d * sizeof(float);
  bytes = (bytes + 255) & ~size_t(255);
  return bytes + rows * sizeof(float);
}

template <int D, int BITS, int G>
vc_status_t launch(const DraftArgs& a, int B, int Hkv, cudaStream_t cs) {
  const Smem P = smem_plan(D, BITS, G, a.NGS, a.tail_cap);
  if (P.total > 200 * 1024) VC_FAIL(VC_ERR_UNSUPPORTED, "shared memory plan %zu bytes too large", P.total);
  VC_CUDA_CHECK(cudaFuncSetAttribute(draft_split_kernel<D, BITS, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(P.total)));
  VC_CUDA_CHECK(cudaFuncSetAttribute(draft_tail_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(P.total)));
  if (a.n_splits > 0) {
    draft_split_kernel<D, BITS, G><<<dim3(a.n_splits, B * Hkv), kThreads, P.total, cs>>>(a);
    VC_LAUNCH_CHECK("draft_split_kernel");
  }
  draft_tail_kernel<D, G><<<dim3(1, B * Hkv), kThreads, P.total, cs>>>(a, BITS);
  VC_LAUNCH_CHECK("draft_tail_kernel");
  return VC_OK;
}

template <int D, int BITS>
vc_status_t launch_g(const DraftArgs& a, int G, int B, int Hkv, cudaStream_t cs) {
  switch (G) {
    case 1: return launch<D, BITS, 1>(a, B, Hkv, cs);
    case 2: return launch<D, BITS, 2>(a, B, Hkv, cs);
    case 4: return launch<D, BITS, 4>(a, B, Hkv, cs);
    case 5: return launch<D, BITS, 5>(a, B, Hkv, cs);
    case 8: return launch<D, BITS, 8>(a, B, Hkv, cs);
  }
  VC_FAIL(VC_ERR_UNSUPPORTED, "G = %d", G);
}

}  // namespace

extern "C" vc_status_t vc_draft_attn_workspace_size(const vc_shape_t* s, int32_t max_packed, size_t* bytes) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE(bytes, "bytes is NULL");
  VC_REQUIRE(max_packed >= 0 && max_packed % kGroup == 0, "max_packed must be a non-negative multiple of 32");
  *bytes = ws_bytes(s, max_packed);
  return VC_OK;
}

extern "C" vc_status_t vc_draft_attn(const vc_shape_t* s, const uint16_t* q, const uint16_t* k_cur,
                                     const uint16_t* v_cur, const uint32_t* kc, const uint16_t* ksz,
                                     const uint32_t* vc, const uint16_t* vsz, const int32_t* packed_len,
                                     int32_t max_packed, int32_t T_cap, uint16_t* tail_k, uint16_t* tail_v,
                                     const int32_t* tail_len, int32_t tail_cap, int32_t step, uint16_t* out,
                                     void* workspace, size_t workspace_bytes, vc_stream_t stream) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE(max_packed >= 0 && max_packed % kGroup == 0 && max_packed <= T_cap && T_cap % kGroup == 0,
             "need 0 <= max_packed <= T_cap, multiples of 32 (max_packed=%d, T_cap=%d)", max_packed, T_cap);
  VC_REQUIRE(q && out && packed_len && tail_len && tail_k && tail_v, "NULL pointer");
  VC_REQUIRE((k_cur == nullptr) == (v_cur == nullptr), "k_cur and v_cur must both be given or both NULL");
  VC_REQUIRE(max_packed == 0 || (kc && ksz && vc && vsz), "packed cache pointers are NULL");
  VC_REQUIRE(tail_cap >= 1 && tail_cap <= 1024 && step >= 0, "need 1 <= tail_cap <= 1024 and step >= 0");
  VC_REQUIRE(vc_aligned16(kc) && vc_aligned16(ksz) && vc_aligned16(vc) && vc_aligned16(vsz) && vc_aligned16(q),
             "pointers must be 16-byte aligned");
  VC_REQUIRE(static_cast<int64_t>(s->B) * s->Hkv <= 65535, "B*Hkv <= 65535");
  const size_t need = ws_bytes(s, max_packed);
  if (!workspace || workspace_bytes < need)
    VC_FAIL(VC_ERR_WORKSPACE, "draft workspace needs %zu bytes (got %zu)", need, workspace_bytes);
  DraftArgs a;
  a.q = q; a.k_cur = k_cur; a.v_cur = v_cur;
  a.kc = kc; a.ksz = ksz; a.vc = vc; a.vsz = vsz;
  a.packed_len = packed_len; a.tail_k = tail_k; a.tail_v = tail_v; a.tail_len = tail_len;
  a.tail_cap = tail_cap; a.step = step;
  a.Hq = s->Hq; a.Hkv = s->Hkv; a.NG = T_cap / kGroup;
  a.NGS = groups_per_split(s->bits);
  a.n_splits = (max_packed / kGroup + a.NGS - 1) / a.NGS;
  a.scale_log2 = s->softmax_scale * kLog2e;
  const size_t rows = static_cast<size_t>(s->B) * s->Hq * (a.n_splits + 1);
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        ((rows * s->d * sizeof(float) + 255) & ~size_t(255)));
  auto cs = reinterpret_cast<cudaStream_t>(stream);
  const int G = s->Hq / s->Hkv;
  if (s->d == 128)
    st = s->bits == 2 ? launch_g<128, 2>(a, G, s->B, s->Hkv, cs) : launch_g<128, 4>(a, G, s->B, s->Hkv, cs);
  else
    st = s->bits == 2 ? launch_g<64, 2>(a, G, s->B, s->Hkv, cs) : launch_g<64, 4>(a, G, s->B, s->Hkv, cs);
  if (st != VC_OK) return st;
  combine_kernel<<<s->B * s->Hq, 128, 0, cs>>>(a.part_o, a.part_lse, a.n_splits + 1, s->d, out);
  VC_LAUNCH_CHECK("combine_kernel");
  return VC_OK;
}

extern "C" vc_status_t vc_draft_attn_device_status(uint32_t* status) {
  VC_REQUIRE(status, "status is NULL");
  VC_CUDA_CHECK(cudaDeviceSynchronize());
  uint32_t v = 0, zero = 0;
  VC_CUDA_CHECK(cudaMemcpyFromSymbol(&v, g_draft_status, sizeof(v)));
  VC_CUDA_CHECK(cudaMemcpyToSymbol(g_draft_status, &zero, sizeof(zero)));
  *status = v;
  return VC_OK;
}
