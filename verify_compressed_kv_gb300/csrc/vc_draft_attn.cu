// libvc_draft_attn: decode attention over the KIVI-packed draft cache.
//
// VeriCache (gist.science/paper/2605.17613), Technical Summary, Core
// Algorithm (Drafting: candidate tokens come from the compressed KV) and Key
// System Innovations (drafting is bound by HBM bandwidth, reading the
// compressed KV).  One query token per request per step; all G query heads
// of a KV head share every byte read.
//
// One launch per draft step.  Grid = B*Hkv tail CTAs followed by a persistent
// set of stream CTAs (occupancy x SM count):
//   * stream-K partition: the packed groups of every (request, KV head) are
//     laid end to end and each stream CTA takes an equal contiguous range, so
//     the work is balanced whatever B*Hkv is; a range may span two heads
//     (segments);
//   * a segment is streamed through a ring of shared-memory stages (8 groups
//     of 32 tokens each: K codes, K scale/zero, V codes, V scale/zero), filled
//     by bulk async copies (cp.async.bulk + mbarrier transaction counts, bounded
//     waits) while the 8 warps compute on earlier stages;
//   * each warp owns one group per stage and keeps its own online-softmax
//     state (max, sum) and output accumulators; QK dequantises exactly
//     (fma(code, s, z), the quantiser's definition) with f32x2 FMAs; PV folds
//     the per-token value scale into the softmax weight;
//   * at the end of a segment the warps are merged (log-sum-exp) into one
//     partial per query head; the last CTA to finish a (request, KV head)
//     (arrival counter in the workspace, reset by that CTA) merges all its
//     partials and writes the bf16 output.
// The tail CTAs handle the bf16 tail (tokens committed since the last full
// group plus earlier draft steps) and the current token, and store the
// current token's K/V into the tail for the following steps.
#include <cfloat>

#include "vc_internal.h"

namespace {

__device__ uint32_t g_draft_status = 0;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kGroup = 32;
// Head split: with many heads per KV head (G = 8) two warps share a group,
// each taking G/2 heads, so a warp's registers stay those of the G = 4 case.
template <int G>
struct HeadSplit {
  static constexpr int HS = G >= 8 ? 2 : 1;   // warps per group
  static constexpr int GW = G / HS;           // heads per warp
  static constexpr int SG = kWarps / HS;      // groups per stage
};
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitCycles = 4000000000LL;   // ~2 s at 2 GHz
#ifndef VC_DRAFT_QK_TB
#define VC_DRAFT_QK_TB 8                           // QK tokens per lane per pass
#endif

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }
// 2^-e as an exact float constant (0 <= e <= 30)
__host__ __device__ constexpr float pow2neg(int e) { return 1.0f / static_cast<float>(1u << e); }

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
  int B, Hq, Hkv;
  int NG;                   // layout stride: T_cap / 32 groups per (b, h)
  int NGmax;                // groups per (b, h) covered by the partition
  int n_stream;             // stream CTAs
  long long total;          // B * Hkv * NGmax
  int max_parts;            // partial slots per (b, h): stream CTAs + the tail
  float scale_log2;
  float* part_o;            // [B*Hq, max_parts, D]   normalised partial outputs
  float* part_lse;          // [B*Hq, max_parts]      log2-sum-exp of each partial
  unsigned int* counter;    // [B*Hkv] arrivals (zero between calls)
  uint16_t* out;            // [B, Hq, D]
};

// ------------------------------------------------------------------ partition
__host__ __device__ inline long long range_lo(long long c, long long total, long long n) { return c * total / n; }

// Stream CTAs overlapping the groups of (b, h) index bh: [first, last].
__host__ __device__ inline void ctas_of(int bh, const DraftArgs& a, int& first, int& last) {
  if (a.n_stream <= 0 || a.NGmax <= 0) {
    first = 0;
    last = -1;
    return;
  }
  const long long s = static_cast<long long>(bh) * a.NGmax, e = s + a.NGmax;
  long long c = s * a.n_stream / a.total;
  while (c + 1 < a.n_stream && range_lo(c + 1, a.total, a.n_stream) <= s) ++c;
  while (c > 0 && range_lo(c, a.total, a.n_stream) > s) --c;
  first = static_cast<int>(c);
  long long d = (e * a.n_stream + a.total - 1) / a.total;
  if (d > a.n_stream - 1) d = a.n_stream - 1;
  while (d > 0 && range_lo(d, a.total, a.n_stream) >= e) --d;
  while (d + 1 < a.n_stream && range_lo(d + 1, a.total, a.n_stream) < e) ++d;
  last = static_cast<int>(d);
}

// ------------------------------------------------------------------ shared memory plan
template <int D, int BITS, int G>
struct Plan {
  static constexpr int W = D * BITS / 32;
  static constexpr int GW = HeadSplit<G>::GW, SG = HeadSplit<G>::SG;
  static constexpr size_t kc = static_cast<size_t>(SG) * W * kGroup * 4;
  static constexpr size_t meta = static_cast<size_t>(SG) * D * 4;
  static constexpr size_t stage = 2 * kc + 2 * meta;             // K codes, K meta, V codes, V meta
  // ring depth: about 72 KB of stages in flight, at least double buffering
  static constexpr int NS = (72 * 1024 / stage) < 2 ? 2 : ((72 * 1024 / stage) > 6 ? 6 : static_cast<int>(72 * 1024 / stage));
  static constexpr size_t ring = stage * NS;
  static constexpr size_t red = static_cast<size_t>(kWarps) * GW * D * 4;  // warp merge (aliases the ring)
  static constexpr size_t body = ring > red ? ring : red;
  static constexpr size_t sc = static_cast<size_t>(kWarps) * GW * kGroup * 4;  // per-warp scores
  static constexpr size_t q = static_cast<size_t>(G) * D * 4;
  static constexpr size_t wstat = static_cast<size_t>(kWarps) * (GW > 8 ? GW : 8) * 2 * 4;  // per-warp (max, sum)
  static constexpr size_t off_sc = body;
  static constexpr size_t off_q = off_sc + sc;
  static constexpr size_t off_wstat = off_q + q;
  static constexpr size_t off_bar = (off_wstat + wstat + 15) & ~size_t(15);
  static constexpr size_t off_flag = off_bar + 8 * NS;
  static constexpr size_t total = off_flag + 16;
};

// Shared memory the tail CTA needs inside the same allocation (rows of the tail
// K/V plus its scores); checked on the host against Plan::total.
template <int D, int G>
__host__ __device__ inline size_t tail_smem(int tail_cap) {
  return 2 * static_cast<size_t>(tail_cap + 1) * D * 2 + static_cast<size_t>(G) * (tail_cap + 1) * 4 + 64;
}

template <int D, int G>
__device__ __forceinline__ void load_q(const DraftArgs& a, int b, int kvh, float* q_s) {
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    q_s[i] = vc_bf16_to_f32(a.q[(static_cast<size_t>(b) * a.Hq + kvh * G + h) * D + c]) * a.scale_log2;
  }
}

// Issue the bulk copies of one stage (groups [g, g + n) of slice bh) into `buf`.
template <int D, int BITS, int G>
__device__ __forceinline__ void issue_stage(const DraftArgs& a, uint8_t* buf, uint64_t* bar, int bh, int g, int n) {
  using P = Plan<D, BITS, G>;
  constexpr int W = P::W;
  const size_t gb = static_cast<size_t>(bh) * a.NG + g;
  const uint32_t code_bytes = static_cast<uint32_t>(n) * W * kGroup * 4;
  const uint32_t meta_bytes = static_cast<uint32_t>(n) * D * 4;
  vc_mbar_arrive_expect_tx(bar, 2 * code_bytes + 2 * meta_bytes);
  vc_bulk_g2s(buf, a.kc + gb * W * kGroup, code_bytes, bar);
  vc_bulk_g2s(buf + P::kc, a.ksz + gb * D * 2, meta_bytes, bar);
  vc_bulk_g2s(buf + P::kc + P::meta, a.vc + gb * W * kGroup, code_bytes, bar);
  vc_bulk_g2s(buf + 2 * P::kc + P::meta, a.vsz + gb * D * 2, meta_bytes, bar);
}

// ------------------------------------------------------------------ one group, one warp
// Load N consecutive 32-bit words (N % 4 == 0) starting at `src` into out[],
// issuing the 16-byte chunks in an order rotated by `rot`.  A word column is
// 128 bytes, so lanes of a quarter-warp that sit in different columns would
// otherwise hit the same bank slot; rotating by the column index spreads them.
template <int N>
__device__ __forceinline__ void load_words_rotated(const uint32_t* src, int rot, uint32_t (&out)[N]) {
  constexpr int NCH = N / 4;
  uint4 tmp[NCH];
#pragma unroll
  for (int k = 0; k < NCH; ++k) tmp[k] = *reinterpret_cast<const uint4*>(src + ((k + rot) % NCH) * 4);
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    uint4 v = tmp[0];
#pragma unroll
    for (int k = 1; k < NCH; ++k)
      if ((k + rot) % NCH == c) v = tmp[k];
    out[4 * c] = v.x; out[4 * c + 1] = v.y; out[4 * c + 2] = v.z; out[4 * c + 3] = v.w;
  }
}

// Lane layout for QK: lane = w * TS + ts holds word column w (CPW channels) of
// TPL = W tokens (rows ts * W .. ts * W + W - 1 of the group), TS = 32 / W.
//
// Code j of a word sits at bits [BITS*j, BITS*j + BITS); channels j < HALF
// come from the low 16 bits, the rest from the high 16 bits.  OR-ing the
// masked code (still at position BITS*jj) into the mantissa of 2^23 and
// subtracting 2^23 gives code * 2^(BITS*jj) exactly; folding 2^(-BITS*jj) into
// the channel's fp32 scale makes fma(code * 2^(BITS*jj), s * 2^(-BITS*jj), z)
// bit-identical to fma(code, s, z).  Channel pairs go through f32x2 FMAs.
template <int D, int BITS, int G>
__device__ __forceinline__ void qk_group(const uint32_t* kc_g, const uint16_t* ksz_g, const float* q_s,
                                         float* sc, int lane) {
  constexpr int W = D * BITS / 32, CPW = 32 / BITS, HALF = CPW / 2, TPL = W;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  constexpr int TB = TPL < VC_DRAFT_QK_TB ? TPL : VC_DRAFT_QK_TB, NTB = TPL / TB;
  constexpr int LOGW = ilog2(W), LOGTB = ilog2(TB);
  constexpr int HB = (2 * G * TB <= 80) ? G : (G + 1) / 2;     // heads per pass (register budget)
  constexpr int NHB = (G + HB - 1) / HB;
  static_assert(LOGTB <= LOGW, "token block wider than the word row");
  constexpr int TS = 32 / W;
  const int w = lane / TS, ts = lane % TS;
  uint32_t lo[TPL], hi[TPL];
  load_words_rotated<TPL>(kc_g + w * kGroup + ts * TPL, w, lo);
#pragma unroll
  for (int tl = 0; tl < TPL; ++tl) hi[tl] = lo[tl] >> 16;
  const uint16_t* kmeta = ksz_g + w * CPW * 2;                    // the lane's CPW (s, z) pairs
#pragma unroll
  for (int tb = 0; tb < NTB; ++tb) {
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
      float2 acc[HB][TB];
#pragma unroll
      for (int h = 0; h < HB; ++h)
#pragma unroll
        for (int tl = 0; tl < TB; ++tl) acc[h][tl] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int cp = 0; cp < CPW / 2; ++cp) {
        const int j0 = 2 * cp;
        const bool upper = j0 >= HALF;
        const int jj = j0 % HALF;
        const uint32_t m0 = MASK << (BITS * jj), m1 = MASK << (BITS * (jj + 1));
        const uint2 raw = *reinterpret_cast<const uint2*>(kmeta + j0 * 2);
        const float2 sz0 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 sz1 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        const float2 s2 = make_float2(sz0.x * pow2neg(BITS * jj), sz1.x * pow2neg(BITS * (jj + 1)));
        const float2 z2 = make_float2(sz0.y, sz1.y);
        float2 q2[HB];
#pragma unroll
        for (int h = 0; h < HB; ++h)
          q2[h] = (hb * HB + h < G) ? *reinterpret_cast<const float2*>(q_s + (hb * HB + h) * D + w * CPW + j0)
                                    : make_float2(0.0f, 0.0f);
#pragma unroll
        for (int tl = 0; tl < TB; ++tl) {
          const uint32_t src = upper ? hi[tb * TB + tl] : lo[tb * TB + tl];
          float2 f = make_float2(__uint_as_float(0x4B000000u | (src & m0)),
                                 __uint_as_float(0x4B000000u | (src & m1)));
          f = __fadd2_rn(f, make_float2(-8388608.0f, -8388608.0f));
          const float2 k2 = __ffma2_rn(f, s2, z2);
#pragma unroll
          for (int h = 0; h < HB; ++h) acc[h][tl] = __ffma2_rn(q2[h], k2, acc[h][tl]);
        }
      }
      float part[HB][TB];
#pragma unroll
      for (int h = 0; h < HB; ++h)
#pragma unroll
        for (int tl = 0; tl < TB; ++tl) part[h][tl] = acc[h][tl].x + acc[h][tl].y;
      // fold the W lanes of the token row: recursive halving over the TB token
      // slots, then an all-reduce over the remaining lane bits
#pragma unroll
      for (int step = 0; step < LOGW; ++step) {
        const int o = W >> (step + 1);                    // bit of w; lanes differ by o * TS
        if (step < LOGTB) {
          const int half = TB >> (step + 1);
          const bool up = (w & o) != 0;
#pragma unroll
          for (int i = 0; i < TB / 2; ++i) {
            if (i < half) {
#pragma unroll
              for (int h = 0; h < HB; ++h) {
                const float send = up ? part[h][i] : part[h][i + half];
                const float keep = up ? part[h][i + half] : part[h][i];
                part[h][i] = keep + __shfl_xor_sync(0xffffffffu, send, o * TS);
              }
            }
          }
        } else {
#pragma unroll
          for (int h = 0; h < HB; ++h) part[h][0] += __shfl_xor_sync(0xffffffffu, part[h][0], o * TS);
        }
      }
      if ((w & ((1 << (LOGW - LOGTB)) - 1)) == 0) {
        const int t = ts * TPL + tb * TB + (w >> (LOGW - LOGTB));
#pragma unroll
        for (int h = 0; h < HB; ++h)
          if (hb * HB + h < G) sc[(hb * HB + h) * kGroup + t] = part[h][0];
      }
    }
  }
}

// Warp-level online softmax over one group's 32 scores per head (sc[h][t],
// log2 units): running max m (warp-uniform), per-lane partial sums l, the
// rescale factor of the earlier accumulators, and p written back over sc.
template <int G>
__device__ __forceinline__ bool softmax_group(float* sc, float (&m)[G], float (&l)[G], float (&alpha)[G], int lane) {
  bool rescale = false;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float s = sc[h * kGroup + lane];
    float gm = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, off));
    const float mn = fmaxf(m[h], gm);
    alpha[h] = exp2f(m[h] - mn);          // m = -inf at the start: alpha = 0, nothing to keep
    rescale |= (alpha[h] != 1.0f);
    const float p = exp2f(s - mn);
    sc[h * kGroup + lane] = p;
    l[h] = fmaf(l[h], alpha[h], p);
    m[h] = mn;
  }
  return rescale;
}

// PV lane layout: SUB lanes share a word (SUB = 2 halves the per-lane channels
// when G is large); lane = wr * TSR + tsr with WR = W * SUB lanes per token row.
template <int D, int BITS, int G>
struct PvLayout {
  static constexpr int W = D * BITS / 32, CPW = 32 / BITS, HALF = CPW / 2;
  static constexpr int SUB = (G * CPW > 64) ? 2 : 1;
  static constexpr int CPL = CPW / SUB;        // channels per lane
  static constexpr int WR = W * SUB;           // lanes per token row
  static constexpr int TSR = 32 / WR;          // token rows per warp
  static constexpr int TPLR = WR;              // tokens per lane per group
  static_assert(SUB == 1 || CPL == HALF, "a lane's channels lie in one half word");
  static_assert(TSR >= 1 && TPLR % 4 == 0, "lane layout");
};

// sum_t p_t (c_t s_t + z_t) = sum_t (p_t s_t) c_t + sum_t p_t z_t: raw codes
// (times 2^(BITS*jj), undone at the end) accumulate against p_t s_t.
template <int D, int BITS, int G>
__device__ __forceinline__ void pv_group(const uint32_t* vc_g, const uint16_t* vsz_g, const float* sc,
                                         float2 (&acc)[G][PvLayout<D, BITS, G>::CPL / 2], float (&zacc)[G],
                                         int lane) {
  using L = PvLayout<D, BITS, G>;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  const int wr = lane / L::TSR, tsr = lane % L::TSR;
  const int w = wr / L::SUB, sub = wr % L::SUB;
  const int cgrp = (w * L::CPW) / kGroup;
  uint32_t wv[L::TPLR];
  load_words_rotated<L::TPLR>(vc_g + w * kGroup + tsr * L::TPLR, w, wv);
#pragma unroll
  for (int tl = 0; tl < L::TPLR; ++tl) {
    const int t = tsr * L::TPLR + tl;
    const float2 sz = __half22float2(*reinterpret_cast<const __half2*>(vsz_g + (cgrp * kGroup + t) * 2));
    float2 w2[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float p = sc[h * kGroup + t];
      const float wgt = p * sz.x;
      w2[h] = make_float2(wgt, wgt);
      zacc[h] = fmaf(p, sz.y, zacc[h]);
    }
    const uint32_t lo = wv[tl], hi = lo >> 16;
#pragma unroll
    for (int jp = 0; jp < L::CPL / 2; ++jp) {
      // lane channel j = sub * CPL + 2 jp (+1); with SUB == 2 a lane owns one half word
      const int jl = 2 * jp;
      uint32_t src;
      int jj;
      if (L::SUB == 1) {
        src = (jl >= L::HALF) ? hi : lo;
        jj = jl % L::HALF;
      } else {
        src = sub ? hi : lo;
        jj = jl;
      }
      float2 f = make_float2(__uint_as_float(0x4B000000u | (src & (MASK << (BITS * jj)))),
                             __uint_as_float(0x4B000000u | (src & (MASK << (BITS * (jj + 1))))));
      f = __fadd2_rn(f, make_float2(-8388608.0f, -8388608.0f));
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h][jp] = __ffma2_rn(w2[h], f, acc[h][jp]);
    }
  }
}

// ------------------------------------------------------------------ merge / arrive / combine
// Partial of this CTA for slice bh: merge the warps' (max, sum, output) in
// shared memory and write one normalised partial + log2-sum-exp per head.
template <int D, int BITS, int G>
__device__ void write_partial(const DraftArgs& a, uint8_t* smem, int bh, int slot,
                              float (&m)[HeadSplit<G>::GW], float (&l)[HeadSplit<G>::GW],
                              float2 (&acc)[HeadSplit<G>::GW][PvLayout<D, BITS, HeadSplit<G>::GW>::CPL / 2],
                              float (&zacc)[HeadSplit<G>::GW]) {
  using P = Plan<D, BITS, G>;
  constexpr int GW = HeadSplit<G>::GW, HS = HeadSplit<G>::HS;
  using L = PvLayout<D, BITS, GW>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* red = reinterpret_cast<float*>(smem);                          // [warp][GW][D], aliases the ring
  float* wstat = reinterpret_cast<float*>(smem + P::off_wstat);         // [warp][GW][2]
  const int wr = lane / L::TSR, tsr = lane % L::TSR;
  const int w = wr / L::SUB, sub = wr % L::SUB;
  // fold the token rows of the PV layout (the low lane bits)
#pragma unroll
  for (int o = 1; o < L::TSR; o <<= 1)
#pragma unroll
    for (int h = 0; h < GW; ++h) {
      zacc[h] += __shfl_xor_sync(0xffffffffu, zacc[h], o);
#pragma unroll
      for (int jp = 0; jp < L::CPL / 2; ++jp) {
        acc[h][jp].x += __shfl_xor_sync(0xffffffffu, acc[h][jp].x, o);
        acc[h][jp].y += __shfl_xor_sync(0xffffffffu, acc[h][jp].y, o);
      }
    }
#pragma unroll
  for (int h = 0; h < GW; ++h) {
    float s = l[h];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    l[h] = s;
  }
  __syncthreads();                                 // every warp is done with the ring
  if (tsr == 0) {
#pragma unroll
    for (int h = 0; h < GW; ++h)
#pragma unroll
      for (int jp = 0; jp < L::CPL / 2; ++jp) {
        const int jl = 2 * jp;
        const int jj = (L::SUB == 1) ? (jl % L::HALF) : jl;
        float* dst = red + (warp * GW + h) * D + w * L::CPW + sub * L::CPL + jl;
        dst[0] = fmaf(acc[h][jp].x, pow2neg(BITS * jj), zacc[h]);
        dst[1] = fmaf(acc[h][jp].y, pow2neg(BITS * (jj + 1)), zacc[h]);
      }
  }
  if (lane == 0)
#pragma unroll
    for (int h = 0; h < GW; ++h) {
      wstat[(warp * GW + h) * 2] = m[h];
      wstat[(warp * GW + h) * 2 + 1] = l[h];
    }
  __syncthreads();
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    const int half = h / GW, hl = h % GW;             // warps x with x % HS == half hold head h
    float M = -INFINITY;
#pragma unroll
    for (int x = half; x < kWarps; x += HS) M = fmaxf(M, wstat[(x * GW + hl) * 2]);
    const size_t row = static_cast<size_t>(b * a.Hq + kvh * G + h) * a.max_parts + slot;
    if (M == -INFINITY) {
      if (c == 0) a.part_lse[row] = -INFINITY;
      continue;
    }
    float o = 0.0f, Ls = 0.0f;
#pragma unroll
    for (int x = half; x < kWarps; x += HS) {
      const float mx = wstat[(x * GW + hl) * 2];
      if (mx == -INFINITY) continue;
      const float wgt = exp2f(mx - M);
      o = fmaf(wgt, red[(x * GW + hl) * D + c], o);
      Ls = fmaf(wgt, wstat[(x * GW + hl) * 2 + 1], Ls);
    }
    a.part_o[row * D + c] = o / Ls;
    if (c == 0) a.part_lse[row] = M + log2f(Ls);
  }
}

// Count this CTA's partial for slice bh; the last of the n_parts arrivals
// merges all partials of the slice and writes its bf16 output.
template <int G, int D>
__device__ void arrive_and_combine(const DraftArgs& a, unsigned int* flag, int bh, int n_parts) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int prev = atomicAdd(a.counter + bh, 1u);
    *flag = (prev + 1 == static_cast<unsigned int>(n_parts)) ? 1u : 0u;
  }
  __syncthreads();
  if (*flag == 0u) return;
  __threadfence();
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    const size_t row = static_cast<size_t>(b * a.Hq + kvh * G + h) * a.max_parts;
    float M = -INFINITY;
    for (int x = 0; x < n_parts; ++x) M = fmaxf(M, __ldcg(a.part_lse + row + x));
    float num = 0.0f, den = 0.0f;
    if (M != -INFINITY) {
      for (int x = 0; x < n_parts; ++x) {
        const float lse = __ldcg(a.part_lse + row + x);
        if (lse == -INFINITY) continue;
        const float wgt = exp2f(lse - M);
        num = fmaf(wgt, __ldcg(a.part_o + (row + x) * D + c), num);
        den += wgt;
      }
    }
    a.out[(static_cast<size_t>(b) * a.Hq + kvh * G + h) * D + c] = vc_f32_to_bf16_rn(den > 0.0f ? num / den : 0.0f);
  }
  if (threadIdx.x == 0) a.counter[bh] = 0u;          // zero again for the next call
}

// ------------------------------------------------------------------ stream CTA
template <int D, int BITS, int G>
__device__ void stream_cta(const DraftArgs& a, uint8_t* smem, int c) {
  using P = Plan<D, BITS, G>;
  constexpr int GW = HeadSplit<G>::GW, HS = HeadSplit<G>::HS, SG = HeadSplit<G>::SG;
  using L = PvLayout<D, BITS, GW>;
  constexpr int W = P::W, NS = P::NS, NC = D / kGroup;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sc = reinterpret_cast<float*>(smem + P::off_sc) + warp * GW * kGroup;
  float* q_s = reinterpret_cast<float*>(smem + P::off_q);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P::off_bar);
  unsigned int* flag = reinterpret_cast<unsigned int*>(smem + P::off_flag);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) vc_mbar_init(bars + i, 1);
    vc_fence_mbar_init();
  }
  __syncthreads();
  long long gstage = 0;                        // stages consumed by this CTA (ring position, phase)
  const long long hi = range_lo(c + 1, a.total, a.n_stream);
  long long pos = range_lo(c, a.total, a.n_stream);
  while (pos < hi) {
    const int bh = static_cast<int>(pos / a.NGmax);
    const int gs = static_cast<int>(pos % a.NGmax);
    const int ge = static_cast<int>(min(static_cast<long long>(a.NGmax), gs + (hi - pos)));
    pos += ge - gs;
    const int b = bh / a.Hkv, kvh = bh % a.Hkv;
    int ng_req = a.packed_len[b] / kGroup;
    if (ng_req > a.NGmax) {
      if (threadIdx.x == 0) atomicOr(&g_draft_status, VC_DEV_CAPACITY);
      ng_req = a.NGmax;
    }
    const int n_valid = max(0, min(ge, ng_req) - gs);
    const int n_st = (n_valid + SG - 1) / SG;
    int first, last;
    ctas_of(bh, a, first, last);
    // ---- prologue: fill the ring (the proxy fence orders earlier generic
    // writes to the ring, the previous segment's warp merge, before the copies)
    if (threadIdx.x == 0) vc_fence_proxy_async_smem();
    if (threadIdx.x == 0)
      for (int i = 0; i < NS && i < n_st; ++i) {
        const int buf = static_cast<int>((gstage + i) % NS);
        issue_stage<D, BITS, G>(a, smem + buf * P::stage, bars + buf, bh, gs + i * SG,
                                min(SG, n_valid - i * SG));
      }
    load_q<D, G>(a, b, kvh, q_s);
    __syncthreads();
    float m[GW], l[GW], zacc[GW];
    float2 acc[GW][L::CPL / 2];
#pragma unroll
    for (int h = 0; h < GW; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.0f;
      zacc[h] = 0.0f;
#pragma unroll
      for (int jp = 0; jp < L::CPL / 2; ++jp) acc[h][jp] = make_float2(0.0f, 0.0f);
    }
    bool ok = true;
    for (int st = 0; st < n_st; ++st) {
      const int buf = static_cast<int>((gstage + st) % NS);
      const uint32_t parity = static_cast<uint32_t>(((gstage + st) / NS) & 1);
      const bool mine = vc_mbar_wait_bounded(bars + buf, parity, kWaitCycles);
      ok = __syncthreads_and(mine) != 0;
      if (!ok) break;
      const uint8_t* base = smem + buf * P::stage;
      const int gl = warp / HS;                              // this warp's group in the stage
      const float* q_w = q_s + (warp % HS) * GW * D;         // ... and its heads
      if (st * SG + gl < n_valid) {
        const uint32_t* kc_g = reinterpret_cast<const uint32_t*>(base) + gl * W * kGroup;
        const uint16_t* ksz_g = reinterpret_cast<const uint16_t*>(base + P::kc) + gl * D * 2;
        const uint32_t* vc_g = reinterpret_cast<const uint32_t*>(base + P::kc + P::meta) + gl * W * kGroup;
        const uint16_t* vsz_g = reinterpret_cast<const uint16_t*>(base + 2 * P::kc + P::meta) + gl * NC * kGroup * 2;
        qk_group<D, BITS, GW>(kc_g, ksz_g, q_w, sc, lane);
        __syncwarp();
        float alpha[GW];
        if (softmax_group<GW>(sc, m, l, alpha, lane)) {
#pragma unroll
          for (int h = 0; h < GW; ++h) {
            zacc[h] *= alpha[h];
#pragma unroll
            for (int jp = 0; jp < L::CPL / 2; ++jp) acc[h][jp] = __fmul2_rn(acc[h][jp], make_float2(alpha[h], alpha[h]));
          }
        }
        __syncwarp();
        pv_group<D, BITS, GW>(vc_g, vsz_g, sc, acc, zacc, lane);
        __syncwarp();
      }
      __syncthreads();                                      // stage `buf` fully consumed
      if (threadIdx.x == 0 && st + NS < n_st)
        issue_stage<D, BITS, G>(a, smem + buf * P::stage, bars + buf, bh, gs + (st + NS) * SG,
                                min(SG, n_valid - (st + NS) * SG));
    }
    gstage += n_st;
    if (!ok) {
      if (threadIdx.x == 0) atomicOr(&g_draft_status, VC_DEV_BARRIER_TIMEOUT);
      return;                                               // outputs of this call are invalid
    }
    write_partial<D, BITS, G>(a, smem, bh, c - first, m, l, acc, zacc);
    arrive_and_combine<G, D>(a, flag, bh, last - first + 2);
    __syncthreads();                                        // smem (red / q) reused by the next segment
  }
}

// ------------------------------------------------------------------ tail CTA
// bf16 tail tokens 0 .. tail_len + step - 1 and the current token of slice bh.
template <int D, int BITS, int G>
__device__ void tail_cta(const DraftArgs& a, uint8_t* smem, int bh) {
  using P = Plan<D, BITS, G>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* q_s = reinterpret_cast<float*>(smem + P::off_q);
  unsigned int* flag = reinterpret_cast<unsigned int*>(smem + P::off_flag);
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  int first, last;
  ctas_of(bh, a, first, last);
  const int n_c = last - first + 1;
  const int slot = n_c;                                  // the tail's partial follows the stream CTAs'
  const int n_tail = a.tail_len[b] + a.step;
  const bool has_cur = a.k_cur != nullptr;
  const int n_tok = n_tail + (has_cur ? 1 : 0);
  const size_t tbase = static_cast<size_t>(bh) * a.tail_cap * D;
  const bool bad = n_tail < 0 || n_tail > a.tail_cap || (has_cur && n_tail >= a.tail_cap);
  if (bad && threadIdx.x == 0) atomicOr(&g_draft_status, VC_DEV_CAPACITY);
  if (bad || n_tok == 0) {
    for (int h = threadIdx.x; h < G; h += blockDim.x)
      a.part_lse[static_cast<size_t>(b * a.Hq + kvh * G + h) * a.max_parts + slot] = -INFINITY;
    arrive_and_combine<G, D>(a, flag, bh, n_c + 1);
    return;
  }
  uint16_t* krow = reinterpret_cast<uint16_t*>(smem);                      // [n_tok][D]
  uint16_t* vrow = krow + static_cast<size_t>(a.tail_cap + 1) * D;
  float* sc = reinterpret_cast<float*>(vrow + static_cast<size_t>(a.tail_cap + 1) * D);   // [G][n_tok]
  float* ml = reinterpret_cast<float*>(smem + P::off_wstat);               // [G][2]
  constexpr int VEC = D / 8;
  for (int i = threadIdx.x; i < n_tok * VEC; i += blockDim.x) {
    const int t = i / VEC, v = i % VEC;
    const uint16_t* ks = (t < n_tail) ? a.tail_k + tbase + static_cast<size_t>(t) * D : a.k_cur + static_cast<size_t>(bh) * D;
    const uint16_t* vs = (t < n_tail) ? a.tail_v + tbase + static_cast<size_t>(t) * D : a.v_cur + static_cast<size_t>(bh) * D;
    *reinterpret_cast<uint4*>(krow + t * D + v * 8) = *reinterpret_cast<const uint4*>(ks + v * 8);
    *reinterpret_cast<uint4*>(vrow + t * D + v * 8) = *reinterpret_cast<const uint4*>(vs + v * 8);
  }
  load_q<D, G>(a, b, kvh, q_s);
  __syncthreads();
  // scores: warp per token, lanes over channel pairs
  for (int t = warp; t < n_tok; t += kWarps) {
    float part[G];
#pragma unroll
    for (int h = 0; h < G; ++h) part[h] = 0.0f;
    for (int c = 2 * lane; c < D; c += 64) {
      const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(krow + t * D + c));
#pragma unroll
      for (int h = 0; h < G; ++h) part[h] = fmaf(q_s[h * D + c], kv.x, fmaf(q_s[h * D + c + 1], kv.y, part[h]));
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) part[h] += __shfl_xor_sync(0xffffffffu, part[h], off);
      if (lane == 0) sc[h * n_tok + t] = part[h];
    }
  }
  __syncthreads();
  for (int h = warp; h < G; h += kWarps) {
    float mx = -INFINITY;
    for (int t = lane; t < n_tok; t += 32) mx = fmaxf(mx, sc[h * n_tok + t]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float sum = 0.0f;
    for (int t = lane; t < n_tok; t += 32) {
      const float p = exp2f(sc[h * n_tok + t] - mx);
      sc[h * n_tok + t] = p;
      sum += p;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) { ml[2 * h] = mx; ml[2 * h + 1] = sum; }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D / 2; i += blockDim.x) {
    const int h = i / (D / 2), c = 2 * (i % (D / 2));
    float ox = 0.0f, oy = 0.0f;
    for (int t = 0; t < n_tok; ++t) {
      const float p = sc[h * n_tok + t];
      const float2 vv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vrow + t * D + c));
      ox = fmaf(p, vv.x, ox);
      oy = fmaf(p, vv.y, oy);
    }
    const size_t row = static_cast<size_t>(b * a.Hq + kvh * G + h) * a.max_parts + slot;
    const float inv = 1.0f / ml[2 * h + 1];
    a.part_o[row * D + c] = ox * inv;
    a.part_o[row * D + c + 1] = oy * inv;
    if (c == 0) a.part_lse[row] = ml[2 * h] + log2f(ml[2 * h + 1]);
  }
  if (has_cur) {                                   // keep the current token for the next steps
    for (int i = threadIdx.x; i < VEC; i += blockDim.x) {
      *reinterpret_cast<uint4*>(a.tail_k + tbase + static_cast<size_t>(n_tail) * D + i * 8) =
          *reinterpret_cast<const uint4*>(krow + n_tail * D + i * 8);
      *reinterpret_cast<uint4*>(a.tail_v + tbase + static_cast<size_t>(n_tail) * D + i * 8) =
          *reinterpret_cast<const uint4*>(vrow + n_tail * D + i * 8);
    }
  }
  arrive_and_combine<G, D>(a, flag, bh, n_c + 1);
}

template <int D, int BITS, int G, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) draft_kernel(DraftArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int nbh = a.B * a.Hkv;
  if (static_cast<int>(blockIdx.x) < nbh)
    tail_cta<D, BITS, G>(a, smem, blockIdx.x);
  else
    stream_cta<D, BITS, G>(a, smem, blockIdx.x - nbh);
}

// ------------------------------------------------------------------ host side
vc_status_t check(const vc_shape_t* s) {
  VC_REQUIRE(s != nullptr, "shape is NULL");
  VC_REQUIRE(s->B >= 1 && s->Hkv >= 1 && s->Hq >= s->Hkv && s->Hq % s->Hkv == 0, "bad B/Hq/Hkv");
  if (s->d != 64 && s->d != 128) VC_FAIL(VC_ERR_UNSUPPORTED, "head dim %d not in {64, 128}", s->d);
  if (s->bits != 2 && s->bits != 4) VC_FAIL(VC_ERR_UNSUPPORTED, "bits %d not in {2, 4}", s->bits);
  const int G = s->Hq / s->Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 5 && G != 8) VC_FAIL(VC_ERR_UNSUPPORTED, "G = %d not in {1,2,4,5,8}", G);
  return VC_OK;
}

#ifndef VC_DRAFT_MINB
#define VC_DRAFT_MINB 1
#endif
template <int G>
struct MinBlocks {
  // CTAs per SM the register allocation targets (2 caps registers at 128)
  static constexpr int value = G <= 5 ? VC_DRAFT_MINB : 1;
};

struct LaunchPlan {
  int n_stream = 0, max_parts = 1;
  long long total = 0;
  size_t smem = 0;
};

template <int D, int BITS, int G>
vc_status_t plan_t(const vc_shape_t* s, int max_packed, LaunchPlan* lp) {
  using P = Plan<D, BITS, G>;
  auto fn = draft_kernel<D, BITS, G, MinBlocks<G>::value>;
  VC_CUDA_CHECK(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(P::total)));
  int dev = 0, sms = 0, occ = 0;
  VC_CUDA_CHECK(cudaGetDevice(&dev));
  VC_CUDA_CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  VC_CUDA_CHECK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kThreads, P::total));
  if (occ < 1) VC_FAIL(VC_ERR_UNSUPPORTED, "draft kernel does not fit on an SM");
  const long long NGmax = max_packed / kGroup;
  lp->total = static_cast<long long>(s->B) * s->Hkv * NGmax;
  long long n = static_cast<long long>(occ) * sms;
  const long long by_work = lp->total / HeadSplit<G>::SG;      // at least one stage per CTA
  if (n > by_work) n = by_work;
  if (n < 1 && lp->total > 0) n = 1;
  lp->n_stream = static_cast<int>(lp->total > 0 ? n : 0);
  if (lp->n_stream > 0) {
    const long long per = lp->total / lp->n_stream;               // >= 1 group per CTA
    lp->max_parts = static_cast<int>((NGmax + per - 1) / per + 1) + 1;
  } else {
    lp->max_parts = 1;
  }
  lp->smem = P::total;
  return VC_OK;
}

vc_status_t plan(const vc_shape_t* s, int max_packed, LaunchPlan* lp) {
  const int G = s->Hq / s->Hkv;
#define VC_PLAN(D_, B_, G_) \
  if (s->d == D_ && s->bits == B_ && G == G_) return plan_t<D_, B_, G_>(s, max_packed, lp);
#define VC_PLAN_G(D_, B_) VC_PLAN(D_, B_, 1) VC_PLAN(D_, B_, 2) VC_PLAN(D_, B_, 4) VC_PLAN(D_, B_, 5) VC_PLAN(D_, B_, 8)
  VC_PLAN_G(128, 2) VC_PLAN_G(128, 4) VC_PLAN_G(64, 2) VC_PLAN_G(64, 4)
#undef VC_PLAN_G
#undef VC_PLAN
  VC_FAIL(VC_ERR_UNSUPPORTED, "no kernel for d=%d bits=%d G=%d", s->d, s->bits, G);
}

size_t ws_bytes(const vc_shape_t* s, const LaunchPlan& lp) {
  const size_t rows = static_cast<size_t>(s->B) * s->Hq * lp.max_parts;
  size_t o = (rows * s->d * sizeof(float) + 255) & ~size_t(255);
  o += (rows * sizeof(float) + 255) & ~size_t(255);
  return o + static_cast<size_t>(s->B) * s->Hkv * sizeof(unsigned int);
}

template <int D, int BITS, int G>
vc_status_t launch_t(const DraftArgs& a, const LaunchPlan& lp, cudaStream_t cs) {
  if (tail_smem<D, G>(a.tail_cap) > Plan<D, BITS, G>::off_sc)
    VC_FAIL(VC_ERR_UNSUPPORTED, "tail_cap %d too large for the shared-memory plan", a.tail_cap);
  const int grid = a.B * a.Hkv + lp.n_stream;
  draft_kernel<D, BITS, G, MinBlocks<G>::value><<<grid, kThreads, lp.smem, cs>>>(a);
  VC_LAUNCH_CHECK("draft_kernel");
  return VC_OK;
}

vc_status_t launch(const vc_shape_t* s, const DraftArgs& a, const LaunchPlan& lp, cudaStream_t cs) {
  const int G = s->Hq / s->Hkv;
#define VC_L(D_, B_, G_) \
  if (s->d == D_ && s->bits == B_ && G == G_) return launch_t<D_, B_, G_>(a, lp, cs);
#define VC_L_G(D_, B_) VC_L(D_, B_, 1) VC_L(D_, B_, 2) VC_L(D_, B_, 4) VC_L(D_, B_, 5) VC_L(D_, B_, 8)
  VC_L_G(128, 2) VC_L_G(128, 4) VC_L_G(64, 2) VC_L_G(64, 4)
#undef VC_L_G
#undef VC_L
  VC_FAIL(VC_ERR_UNSUPPORTED, "no kernel for d=%d bits=%d G=%d", s->d, s->bits, G);
}

}  // namespace

extern "C" vc_status_t vc_draft_attn_workspace_size(const vc_shape_t* s, int32_t max_packed, size_t* bytes) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE(bytes, "bytes is NULL");
  VC_REQUIRE(max_packed >= 0 && max_packed % kGroup == 0, "max_packed must be a non-negative multiple of 32");
  LaunchPlan lp;
  if ((st = plan(s, max_packed, &lp)) != VC_OK) return st;
  *bytes = ws_bytes(s, lp);
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
  VC_REQUIRE(tail_cap >= 1 && step >= 0, "need tail_cap >= 1 and step >= 0");
  VC_REQUIRE(vc_aligned16(kc) && vc_aligned16(ksz) && vc_aligned16(vc) && vc_aligned16(vsz) && vc_aligned16(q) &&
                 vc_aligned16(tail_k) && vc_aligned16(tail_v) && (!k_cur || (vc_aligned16(k_cur) && vc_aligned16(v_cur))),
             "pointers must be 16-byte aligned");
  LaunchPlan lp;
  if ((st = plan(s, max_packed, &lp)) != VC_OK) return st;
  const size_t need = ws_bytes(s, lp);
  if (!workspace || workspace_bytes < need)
    VC_FAIL(VC_ERR_WORKSPACE, "draft workspace needs %zu bytes (got %zu)", need, workspace_bytes);
  VC_REQUIRE(vc_aligned16(workspace), "workspace must be 16-byte aligned");
  DraftArgs a{};
  a.q = q; a.k_cur = k_cur; a.v_cur = v_cur;
  a.kc = kc; a.ksz = ksz; a.vc = vc; a.vsz = vsz;
  a.packed_len = packed_len; a.tail_k = tail_k; a.tail_v = tail_v; a.tail_len = tail_len;
  a.tail_cap = tail_cap; a.step = step;
  a.B = s->B; a.Hq = s->Hq; a.Hkv = s->Hkv;
  a.NG = T_cap / kGroup;
  a.NGmax = max_packed / kGroup;
  a.n_stream = lp.n_stream;
  a.total = lp.total;
  a.max_parts = lp.max_parts;
  a.scale_log2 = s->softmax_scale * kLog2e;
  const size_t rows = static_cast<size_t>(s->B) * s->Hq * lp.max_parts;
  char* ws = static_cast<char*>(workspace);
  a.part_o = reinterpret_cast<float*>(ws);
  size_t off = (rows * s->d * sizeof(float) + 255) & ~size_t(255);
  a.part_lse = reinterpret_cast<float*>(ws + off);
  off += (rows * sizeof(float) + 255) & ~size_t(255);
  a.counter = reinterpret_cast<unsigned int*>(ws + off);
  a.out = out;
  return launch(s, a, lp, reinterpret_cast<cudaStream_t>(stream));
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
