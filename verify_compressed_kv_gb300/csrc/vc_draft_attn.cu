// libvc_draft_attn: decode attention over the KIVI-packed draft cache, on the
// tcgen05 tensor cores.
//
// VeriCache (gist.science/paper/2605.17613), Technical Summary, Core
// Algorithm (Drafting: candidate tokens come from the compressed KV) and Key
// System Innovations (drafting is bound by HBM bandwidth, reading the
// compressed KV).  One query token per request per step; all G query heads
// of a KV head share every byte read.
//
// One launch per draft step.  Grid = B*Hkv tail CTAs followed by a persistent
// set of stream CTAs (one per SM):
//   * stream-K partition: the packed groups of every (request, KV head) are
//     laid end to end and each stream CTA takes an equal contiguous range, so
//     the work is balanced whatever B*Hkv is; a range may span slices
//     (segments);
//   * a segment is cut into tiles of 4 groups (128 tokens); a producer thread
//     fills a ring of tile stages (K codes, K scale/zero, V codes, V
//     scale/zero) with bulk async copies;
//   * 4 token warps (one 32-token group each: TMEM lane quarter = group)
//     dequantise their tokens' K rows into TMEM as fp16, and D/32 channel
//     warps dequantise the tile's V rows (TMEM lane = channel, tokens along
//     the row): the code field OR-ed into the mantissa of 1.0 gives
//     y = 1 + code/f exactly, and x^ = fma(y - 1, f s, z) is the correctly
//     rounded fp16 of code s + z, two elements per instruction;
//   * one thread issues S = K^ . Q^T (M = 128 tokens, N = 16 columns for the
//     G heads, K = d; A in TMEM, Q in shared memory) and O^T = V^T . P^T
//     (M = channels, N = 16, K = the tile's 128 tokens; A in TMEM, P in
//     shared memory), fp16 operands, fp32 accumulators in TMEM;
//   * the token warps turn S into softmax weights against a running maximum
//     that is raised only when a score exceeds it by more than 2^3 (the four
//     warps agree once per tile on one barrier), write P as fp16 and keep the
//     weight sums; the channel warps fold each tile's O into registers,
//     rescaling when the maximum rose;
//   * at the end of a segment the sums and outputs give one normalised
//     partial + log2-sum-exp per head; the last CTA to finish a (request, KV
//     head) (arrival counter in the workspace, reset by that CTA) merges all
//     its partials and writes the bf16 output.
// The tail CTAs handle the bf16 tail (tokens committed since the last full
// group plus earlier draft steps) and the current token, and store the
// current token's K/V into the tail for the following steps.
// Every wait is bounded (~2 s); a wait that runs out sets the device status
// flag, the CTA drains its copies and products, frees its TMEM and returns,
// and the call's outputs are invalid (vc_draft_attn_device_status).
#include <cfloat>

#include "vc_internal.h"

namespace {

__device__ uint32_t g_draft_status = 0;

constexpr int kGroup = 32;
constexpr int kTileGroups = 4;                    // a tile: 4 groups = 128 tokens = the products' M
constexpr int kTile = kTileGroups * kGroup;
constexpr int kTokWarps = 4;                      // token warp q: group q of a tile, TMEM lanes 32q..
constexpr int kN = 16;                            // N of both products: the G <= 16 heads, zero-padded
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitCycles = 4000000000LL;   // ~2 s at 2 GHz
constexpr float kLazy = 3.0f;                     // running max raised only past max + 2^3

struct DraftArgs {
  const uint16_t* q;        // [B, Hq, D]
  const uint16_t* k_cur;    // [B, Hkv, D] or null
  const uint16_t* v_cur;
  const uint32_t* kc;       // [B, Hkv, NG, D*BITS] words
  const uint16_t* ksz;      // [B, Hkv, NG, 2, D]
  const uint32_t* vc;       // [B, Hkv, NG, D*BITS] words
  const uint16_t* vsz;      // [B, Hkv, NG, D/32, 2, 32]
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

// Segments of stream CTA c: consecutive calls walk [range_lo(c), range_lo(c+1)).
struct Segment {
  int bh, gs, n_valid, n_tiles;
};
__device__ __forceinline__ bool next_segment(const DraftArgs& a, long long& pos, long long hi, Segment& sg,
                                             bool& over_capacity) {
  if (pos >= hi) return false;
  sg.bh = static_cast<int>(pos / a.NGmax);
  sg.gs = static_cast<int>(pos % a.NGmax);
  const int ge = static_cast<int>(min(static_cast<long long>(a.NGmax), sg.gs + (hi - pos)));
  pos += ge - sg.gs;
  int ng_req = a.packed_len[sg.bh / a.Hkv] / kGroup;
  over_capacity = ng_req > a.NGmax;
  if (over_capacity) ng_req = a.NGmax;
  sg.n_valid = max(0, min(ge, ng_req) - sg.gs);
  sg.n_tiles = (sg.n_valid + kTileGroups - 1) / kTileGroups;
  return true;
}

// ------------------------------------------------------------------ roles and shared memory
template <int D>
struct Roles {
  static constexpr int chan_warps = D / 32;                   // channel warp c: channels 32c.., TMEM lanes 32c..
  static constexpr int compute_warps = kTokWarps + chan_warps;
  static constexpr int compute_threads = 32 * compute_warps;
  static constexpr int producer_warp = compute_warps;    // then the products' warp
  static constexpr int threads = 32 * (compute_warps + 2);
};

template <int D, int BITS>
struct Plan {
  static constexpr uint32_t kcb = D * BITS * 4;               // one group's K codes (bytes)
  static constexpr uint32_t kmb = D * 4;                      // one group's K scale/zero
  static constexpr uint32_t vcb = D * BITS * 4;
  static constexpr uint32_t vmb = D * 4;
  static constexpr uint32_t off_kc = 0;
  static constexpr uint32_t off_km = off_kc + kTileGroups * kcb;
  static constexpr uint32_t off_vc = off_km + kTileGroups * kmb;
  static constexpr uint32_t off_vm = off_vc + kTileGroups * vcb;
  static constexpr uint32_t stage = off_vm + kTileGroups * vmb;
  static constexpr int NS = (96 * 1024 / stage) < 2 ? 2 : ((96 * 1024 / stage) > 8 ? 8 : static_cast<int>(96 * 1024 / stage));
  static constexpr uint32_t ring = stage * NS;
  // B operands: Q [16 heads x D] K-major core matrices (8 rows x 16 B; K step
  // 128 B, 8-row step 16 D B), P [128 tokens x 16 heads] MN-major (8 tokens x
  // 8 heads per 128 B core matrix; head step 128 B, token step 256 B)
  static constexpr uint32_t q_bytes = kN * D * 2;
  static constexpr uint32_t p_bytes = kTile * kN * 2;
  static constexpr uint32_t off_q = ring;                     // [2] by segment parity
  static constexpr uint32_t off_p = off_q + 2 * q_bytes;      // [2] by tile parity
  static constexpr uint32_t off_mt = off_p + 2 * p_bytes;                   // max of a tile [2][kN]
  static constexpr uint32_t off_red = off_mt + 2 * kN * 4;                   // [4][kN] exchange
  static constexpr uint32_t off_bar = off_red + kTokWarps * kN * 4;
  // full[NS], empty[NS], then [2] each of: ak, sf, av, pr, of, ofree, mr; done
  static constexpr int n_bars = 2 * NS + 15;
  static constexpr uint32_t off_misc = off_bar + n_bars * 8;  // TMEM base, combine flag, abort flag
  static constexpr uint32_t total = off_misc + 16;
  static_assert(stage % 16 == 0 && off_bar % 8 == 0, "alignment");
  static_assert(total <= 227 * 1024, "shared memory");
};

// TMEM columns: A_K[2] (D/2 each), A_V[2] (64 each), S[2], O[2] (16 each).
template <int D>
struct Cols {
  static constexpr uint32_t ak = 0, av = D, s = D + 2 * (kTile / 2), o = s + 2 * kN;
  static constexpr uint32_t used = o + 2 * kN;
  static constexpr uint32_t alloc = used <= 256 ? 256 : 512;
};

// Shared memory the tail CTA uses (rows of the tail K/V, scores, fp32 queries,
// per-head (max, sum), combine flag); checked on the host against Plan::total.
template <int D, int G>
struct TailPlan {
  __host__ __device__ static size_t rows(int cap) { return 2 * static_cast<size_t>(cap + 1) * D * 2; }
  __host__ __device__ static size_t off_sc(int cap) { return rows(cap); }
  __host__ __device__ static size_t off_q(int cap) { return (off_sc(cap) + static_cast<size_t>(G) * (cap + 1) * 4 + 15) & ~size_t(15); }
  __host__ __device__ static size_t off_ml(int cap) { return off_q(cap) + static_cast<size_t>(G) * D * 4; }
  __host__ __device__ static size_t off_flag(int cap) { return off_ml(cap) + static_cast<size_t>(G) * 2 * 4; }
  __host__ __device__ static size_t total(int cap) { return off_flag(cap) + 16; }
};

// ------------------------------------------------------------------ small device pieces
__device__ __forceinline__ float fast_exp2(float x) {   // ex2.approx.ftz: relative error ~2^-22
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
// Operand pair of field k of packed word w: the field of both half-words moved
// into the top mantissa bits of the fp16 pattern of f, giving y = f + code
// exactly.  b = 2: field k at bit 2k; one shift puts the odd field of a nibble
// at bits 8-9 (f = 4) and the even one at bits 6-7 (f = 16).  b = 4: bits 6-9
// (f = 16).  b = 8: bits 2-9 (f = 256).
template <int BITS>
__device__ __forceinline__ uint32_t pair_operand(uint32_t w, int k) {
  if (BITS == 2) {
    const int u = k >> 1;
    const uint32_t x = u == 0 ? (w << 6) : u == 1 ? (w << 2) : u == 2 ? (w >> 2) : (w >> 6);
    return (k & 1) ? ((x & 0x03000300u) | 0x44004400u) : ((x & 0x00C000C0u) | 0x4C004C00u);
  } else if (BITS == 4) {
    const uint32_t x = k == 0 ? (w << 6) : k == 1 ? (w << 2) : k == 2 ? (w >> 2) : (w >> 6);
    return (x & 0x03C003C0u) | 0x4C004C00u;
  } else {
    const uint32_t x = k == 0 ? (w << 2) : (w >> 6);
    return (x & 0x03FC03FCu) | 0x5C005C00u;
  }
}
// f of field k (the fp16 pattern pair_operand ORs the field into).
template <int BITS>
__host__ __device__ constexpr float field_f(int k) {
  return BITS == 2 ? ((k & 1) ? 4.0f : 16.0f) : (BITS == 4 ? 16.0f : 256.0f);
}
// x^ = fma(y - f, s, z) for an operand pair y = f + code: y - f = code is exact,
// so x^ is the correctly rounded fp16 of code s + z (two elements at once).
template <int BITS>
__device__ __forceinline__ uint32_t dequant2(uint32_t y, int k, uint32_t s, uint32_t z) {
  return h2u(__hfma2(__hsub2(u2h(y), __float2half2_rn(field_f<BITS>(k))), u2h(s), u2h(z)));
}

// ------------------------------------------------------------------ token warp: K rows
// Dequantise token t's K row into the warp's TMEM lanes of A_K at column ta
// (pair m = channels 2m, 2m+1 at column m).  kc_g: the group's K codes, 32
// token rows of W = D*BITS/32 words stored in chunks of 4 words (word w of
// token t at ((w/4)*32 + t)*4 + w%4, so the warp's 16-byte loads cover
// contiguous 512 bytes); km: the group's scales then zeros, fp16 pairs.
template <int D, int BITS>
__device__ __forceinline__ void dequant_k_row(const uint32_t* kc_g, const uint32_t* km, int t, uint32_t ta) {
  constexpr int W = D * BITS / 32;
  constexpr int PH = 16 / BITS;                  // pairs per word
  uint32_t wv[W];
#pragma unroll
  for (int ch = 0; ch < W / 4; ++ch) {
    const uint4 v = *reinterpret_cast<const uint4*>(kc_g + (ch * 32 + t) * 4);
    wv[4 * ch] = v.x; wv[4 * ch + 1] = v.y; wv[4 * ch + 2] = v.z; wv[4 * ch + 3] = v.w;
  }
  uint32_t r[16];
#pragma unroll
  for (int m0 = 0; m0 < D / 2; m0 += 4) {        // 4 pairs: one 16-byte load of scales, one of zeros
    const uint4 s4 = *reinterpret_cast<const uint4*>(km + m0);
    const uint4 z4 = *reinterpret_cast<const uint4*>(km + D / 2 + m0);
    const uint32_t sv[4] = {s4.x, s4.y, s4.z, s4.w}, zv[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = m0 + i, k = m % PH;
      r[m & 15] = dequant2<BITS>(pair_operand<BITS>(wv[m / PH], k), k, sv[i], zv[i]);
    }
    if (((m0 + 3) & 15) == 15) vc_tc_st16(ta + (m0 + 3 - 15), r);
  }
}

// ------------------------------------------------------------------ channel warp: V rows
// Dequantise channel ch's V row of one group (its 32 tokens: pair m = tokens
// 2m, 2m+1) into the warp's TMEM lanes at column ta .. ta + 15.  vc_g: the
// group's V codes, D channel rows of BITS words in chunks of min(BITS, 4)
// words; vm: the scales then zeros of the channel's 32-channel group, fp16 pairs.
template <int D, int BITS>
__device__ __forceinline__ void dequant_v_row(const uint32_t* vc_g, const uint32_t* vm, int ch, uint32_t ta) {
  constexpr int PH = 16 / BITS;
  uint32_t wv[BITS];
  if (BITS == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(vc_g + ch * 2);
    wv[0] = v.x;
    wv[1] = v.y;
  } else {
#pragma unroll
    for (int c4 = 0; c4 < BITS / 4; ++c4) {
      const uint4 v = *reinterpret_cast<const uint4*>(vc_g + (c4 * D + ch) * 4);
      wv[4 * c4] = v.x; wv[4 * c4 + 1] = v.y; wv[4 * c4 + 2] = v.z; wv[4 * c4 + 3] = v.w;
    }
  }
  uint32_t r[16];
#pragma unroll
  for (int m0 = 0; m0 < 16; m0 += 4) {
    const uint4 s4 = *reinterpret_cast<const uint4*>(vm + m0);
    const uint4 z4 = *reinterpret_cast<const uint4*>(vm + 16 + m0);
    const uint32_t sv[4] = {s4.x, s4.y, s4.z, s4.w}, zv[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = m0 + i, k = m % PH;
      r[m] = dequant2<BITS>(pair_operand<BITS>(wv[m / PH], k), k, sv[i], zv[i]);
    }
  }
  vc_tc_st16(ta, r);
}

// ------------------------------------------------------------------ merge / arrive / combine
// Barrier over `nthr` threads: the whole tail CTA, or the compute warps of a
// stream CTA (named barrier 2).
__device__ __forceinline__ void sync_part(int nthr) {
  if (nthr == static_cast<int>(blockDim.x)) __syncthreads(); else vc_bar_sync(2, nthr);
}

// Count this CTA's partial for slice bh; the last of the n_parts arrivals
// merges all partials of the slice and writes its bf16 output.
template <int G, int D>
__device__ void arrive_and_combine(const DraftArgs& a, unsigned int* flag, int bh, int n_parts, int nthr) {
  __threadfence();
  sync_part(nthr);
  if (threadIdx.x == 0) {
    const unsigned int prev = atomicAdd(a.counter + bh, 1u);
    *flag = (prev + 1 == static_cast<unsigned int>(n_parts)) ? 1u : 0u;
  }
  sync_part(nthr);
  if (*flag == 0u) return;
  __threadfence();
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  for (int i = threadIdx.x; i < G * D; i += nthr) {
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
struct Stream {
  using P = Plan<D, BITS>;
  using R = Roles<D>;
  using C = Cols<D>;
  static constexpr int NL = G <= 8 ? 8 : 16;       // TMEM columns a thread reads per row

  uint8_t* smem;
  uint64_t* full;
  uint64_t* empty;
  uint64_t *ak, *sf, *av, *pr, *of, *ofree, *mr, *done;
  uint32_t tmem;
  unsigned int* flag;
  volatile uint32_t* abort;

  __device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity) {
    return vc_mbar_wait_or_abort(bar, parity, abort, kWaitCycles);
  }
};

// Producer (one thread): the tile stages of every segment, in order.
template <int D, int BITS, int G>
__device__ void produce(const DraftArgs& a, Stream<D, BITS, G>& S, int c) {
  using P = Plan<D, BITS>;
  const long long hi = range_lo(c + 1, a.total, a.n_stream);
  long long pos = range_lo(c, a.total, a.n_stream);
  Segment sg{};
  bool over, ok = true;
  long long gt = 0;                           // global tile index (tiles issued so far)
  while (ok && next_segment(a, pos, hi, sg, over)) {
    for (int j = 0; j < sg.n_tiles; ++j, ++gt) {
      const int s = static_cast<int>(gt % P::NS);
      if (gt >= P::NS && !S.wait(S.empty + s, static_cast<uint32_t>((gt / P::NS - 1) & 1))) {
        ok = false;
        break;
      }
      const int n = min(kTileGroups, sg.n_valid - j * kTileGroups);
      const size_t g0 = static_cast<size_t>(sg.bh) * a.NG + sg.gs + j * kTileGroups;
      uint8_t* st = S.smem + s * P::stage;
      vc_mbar_arrive_expect_tx(S.full + s, n * (P::kcb + P::kmb + P::vcb + P::vmb));
      vc_bulk_g2s(st + P::off_kc, a.kc + g0 * (P::kcb / 4), n * P::kcb, S.full + s);
      vc_bulk_g2s(st + P::off_km, a.ksz + g0 * (P::kmb / 2), n * P::kmb, S.full + s);
      vc_bulk_g2s(st + P::off_vc, a.vc + g0 * (P::vcb / 4), n * P::vcb, S.full + s);
      vc_bulk_g2s(st + P::off_vm, a.vsz + g0 * (P::vmb / 2), n * P::vmb, S.full + s);
    }
  }
  // drain: every stage issued has landed before the CTA may exit
  for (long long x = gt - P::NS < 0 ? 0 : gt - P::NS; x < gt; ++x)
    vc_mbar_wait_bounded(S.full + x % P::NS, static_cast<uint32_t>((x / P::NS) & 1), kWaitCycles);
}

// Products (one thread): per tile S = K^ . Q^T, then O^T = V^T . P^T.
template <int D, int BITS, int G>
__device__ void issue(const DraftArgs& a, Stream<D, BITS, G>& S, int c) {
  using P = Plan<D, BITS>;
  using C = Cols<D>;
  constexpr uint32_t id_qk = vc_tc_idesc_f16(128, kN, false), id_pv = vc_tc_idesc_f16(128, kN, true);
  const uint32_t q0 = vc_smem_addr(S.smem + P::off_q), p0 = vc_smem_addr(S.smem + P::off_p);
  const long long hi = range_lo(c + 1, a.total, a.n_stream);
  long long pos = range_lo(c, a.total, a.n_stream);
  Segment sg{};
  bool over, ok = true, any = false;
  long long gt = 0;
  int seg = 0;
  auto qk = [&](long long t, int sb) {
    const int b = static_cast<int>(t & 1);
    if (!S.wait(S.ak + b, static_cast<uint32_t>((t >> 1) & 1))) return false;
    vc_tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
      vc_tc_mma_ta(S.tmem + C::s + b * kN, S.tmem + C::ak + b * (D / 2) + ks * 8,
                   vc_tc_desc(q0 + sb * P::q_bytes + ks * 256, 128, 16 * D), id_qk, ks > 0);
    vc_tc_commit(S.sf + b);
    return true;
  };
  auto pv = [&](long long t) {
    const int b = static_cast<int>(t & 1);
    if (!S.wait(S.pr + b, static_cast<uint32_t>((t >> 1) & 1))) return false;
    if (!S.wait(S.av + b, static_cast<uint32_t>((t >> 1) & 1))) return false;
    if (t >= 2 && !S.wait(S.ofree + b, static_cast<uint32_t>(((t >> 1) + 1) & 1))) return false;
    vc_tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < kTile / 16; ++ks)
      vc_tc_mma_ta(S.tmem + C::o + b * kN, S.tmem + C::av + b * (kTile / 2) + ks * 8,
                   vc_tc_desc(p0 + b * P::p_bytes + ks * 512, 256, 128), id_pv, ks > 0);
    vc_tc_commit(S.of + b);
    return true;
  };
  while (ok && next_segment(a, pos, hi, sg, over)) {
    const int sb = seg & 1;
    if (sg.n_tiles > 0) {
      any = true;
      ok = qk(gt, sb);
      for (int j = 0; ok && j < sg.n_tiles; ++j) {
        if (j + 1 < sg.n_tiles) ok = qk(gt + j + 1, sb);
        if (ok) ok = pv(gt + j);
      }
      gt += sg.n_tiles;
    }
    ++seg;
  }
  // every product issued has completed before TMEM is freed
  if (any) {
    vc_tc_commit(S.done);
    vc_mbar_wait_bounded(S.done, 0, kWaitCycles);
  }
}

// Q of slice bh (G heads) into the K-major operand buffer sb: fp16 q * scale * log2(e).
template <int D, int BITS, int G>
__device__ __forceinline__ void write_q(const DraftArgs& a, Stream<D, BITS, G>& S, int bh, int sb) {
  using P = Plan<D, BITS>;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  uint8_t* qs = S.smem + P::off_q + sb * P::q_bytes;
  for (int i = threadIdx.x; i < G * D / 8; i += 32 * kTokWarps) {
    const int h = i / (D / 8), kc = i % (D / 8);
    const uint4 raw = *reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(b) * a.Hq + kvh * G + h) * D + 8 * kc);
    const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = h2u(__floats2half2_rn(vc_bf16_to_f32(static_cast<uint16_t>(rw[j])) * a.scale_log2,
                                   vc_bf16_to_f32(static_cast<uint16_t>(rw[j] >> 16)) * a.scale_log2));
    *reinterpret_cast<uint4*>(qs + (h / 8) * (16 * D) + kc * 128 + (h % 8) * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  vc_fence_proxy_async_smem();
}

// Token warp q.
template <int D, int BITS, int G>
__device__ void token_warp(const DraftArgs& a, Stream<D, BITS, G>& S, int c) {
  using P = Plan<D, BITS>;
  using R = Roles<D>;
  using C = Cols<D>;
  constexpr int NL = Stream<D, BITS, G>::NL;
  const int q = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t t_lane = S.tmem + (static_cast<uint32_t>(q * 32) << 16);
  float* red = reinterpret_cast<float*>(S.smem + P::off_red);
  float* mt = reinterpret_cast<float*>(S.smem + P::off_mt);
  const long long hi = range_lo(c + 1, a.total, a.n_stream);
  long long pos = range_lo(c, a.total, a.n_stream);
  Segment sg{};
  bool over;
  long long gt = 0;
  int seg = 0;
  float m[G], l[G];

  // tile t of the CTA (j-th of the segment): K rows of group q into A_K[t & 1]
  auto extract = [&](long long t, int j, int sb) {
    const int s = static_cast<int>(t % P::NS);
    bool ok = S.wait(S.full + s, static_cast<uint32_t>((t / P::NS) & 1));
    ok = __all_sync(0xffffffffu, ok);
    if (j == 0) write_q(a, S, sg.bh, sb);        // this segment's queries (first tile)
    const int n = min(kTileGroups, sg.n_valid - j * kTileGroups);
    if (ok && q < n) {
      const uint8_t* st = S.smem + s * P::stage;
      dequant_k_row<D, BITS>(reinterpret_cast<const uint32_t*>(st + P::off_kc + q * P::kcb),
                             reinterpret_cast<const uint32_t*>(st + P::off_km + q * P::kmb), lane,
                             t_lane + C::ak + static_cast<uint32_t>(t & 1) * (D / 2));
      vc_tc_wait_st();
    }
    vc_tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      vc_mbar_arrive(S.ak + (t & 1));
      vc_mbar_arrive(S.empty + s);
    }
  };

  // softmax of tile t: weights of group q's tokens into P[t & 1]
  auto softmax = [&](long long t, int j) {
    const int b = static_cast<int>(t & 1);
    const int n = min(kTileGroups, sg.n_valid - j * kTileGroups);
    const bool valid = q < n;
    bool ok = S.wait(S.sf + b, static_cast<uint32_t>((t >> 1) & 1));
    ok = __all_sync(0xffffffffu, ok);
    vc_tc_fence_after();
    float sc[NL];
    if constexpr (NL == 8) vc_tc_ld8(t_lane + C::s + b * kN, sc);
    else vc_tc_ld16(t_lane + C::s + b * kN, sc);
    const bool live = ok && valid;
    bool need = false;
#pragma unroll
    for (int h = 0; h < G; ++h) need |= live && !(sc[h] <= m[h] + kLazy);
    if (vc_bar_red_or(1, 32 * kTokWarps, need)) {            // raise the running max (same in every token warp)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float x = live ? sc[h] : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        if (lane == 0) red[q * kN + h] = x;
      }
      vc_bar_sync(1, 32 * kTokWarps);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mx = fmaxf(fmaxf(red[h], red[kN + h]), fmaxf(red[2 * kN + h], red[3 * kN + h]));
        const float mn = fmaxf(m[h], mx);
        if (mn != -INFINITY) {
          l[h] *= fast_exp2(m[h] - mn);                       // m = -inf at the start: 0
          m[h] = mn;
        }
      }
      vc_bar_sync(1, 32 * kTokWarps);
    }
    float p[kN];
#pragma unroll
    for (int h = 0; h < kN; ++h) {
      p[h] = 0.0f;
      if (h < G && live) {
        p[h] = fast_exp2(sc[h] - m[h]);
        l[h] += p[h];
      }
    }
    vc_tc_fence_before();                                     // S read out before the buffer is refilled
    // P[b] and the tile max: their previous readers (tile t - 2) are done
    if (t >= 2) {
      ok = S.wait(S.ofree + b, static_cast<uint32_t>(((t >> 1) + 1) & 1));
      ok = __all_sync(0xffffffffu, ok);
    }
    uint8_t* pb = S.smem + P::off_p + b * P::p_bytes;
    const int pt = q * 32 + lane;                              // the token's position in the tile
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = h2u(__floats2half2_rn(p[2 * i], p[2 * i + 1]));
    *reinterpret_cast<uint4*>(pb + (pt / 8) * 256 + (pt % 8) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    if (G > 8) *reinterpret_cast<uint4*>(pb + (pt / 8) * 256 + 128 + (pt % 8) * 16) = make_uint4(w[4], w[5], w[6], w[7]);
    vc_fence_proxy_async_smem();
    if (q == 0 && lane == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) mt[b * kN + h] = m[h];
    }
    __syncwarp();
    if (lane == 0) {
      vc_mbar_arrive(S.pr + b);
      if (q == 0) vc_mbar_arrive(S.mr + b);
    }
  };

  while (next_segment(a, pos, hi, sg, over)) {
    if (over && threadIdx.x == 0) atomicOr(&g_draft_status, VC_DEV_CAPACITY);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.0f;
    }
    const int sb = seg & 1;
    if (sg.n_tiles > 0) extract(gt, 0, sb);
    for (int j = 0; j < sg.n_tiles; ++j) {
      if (j + 1 < sg.n_tiles) extract(gt + j + 1, j + 1, sb);
      softmax(gt + j, j);
    }
    gt += sg.n_tiles;
    ++seg;
    // segment end: the weight sums of the 128 token rows, per head, for the channel warps
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float x = l[h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if (lane == 0) red[q * kN + h] = x;
    }
    vc_bar_sync(2, R::compute_threads);                        // sums in red; channel warps write the partial
    int first, last;
    ctas_of(sg.bh, a, first, last);
    arrive_and_combine<G, D>(a, S.flag, sg.bh, last - first + 2, R::compute_threads);
    vc_bar_sync(2, R::compute_threads);                        // red / flag reused by the next segment
  }
}

// Channel warp cw (warp kTokWarps + cw): channels 32 cw .. 32 cw + 31.
template <int D, int BITS, int G>
__device__ void channel_warp(const DraftArgs& a, Stream<D, BITS, G>& S, int c) {
  using P = Plan<D, BITS>;
  using R = Roles<D>;
  using C = Cols<D>;
  constexpr int NL = Stream<D, BITS, G>::NL;
  const int cw = (threadIdx.x >> 5) - kTokWarps, lane = threadIdx.x & 31;
  const int ch = 32 * cw + lane;
  const uint32_t t_lane = S.tmem + (static_cast<uint32_t>(cw * 32) << 16);   // warp % 4 == cw
  const float* red = reinterpret_cast<const float*>(S.smem + P::off_red);
  const float* mt = reinterpret_cast<const float*>(S.smem + P::off_mt);
  const long long hi = range_lo(c + 1, a.total, a.n_stream);
  long long pos = range_lo(c, a.total, a.n_stream);
  Segment sg{};
  bool over;
  long long gt = 0;
  float o[G], mc[G];

  // tile t: V rows of this warp's channels into A_V[t & 1] (zeros past the valid groups)
  auto extract = [&](long long t, int j) {
    const int s = static_cast<int>(t % P::NS);
    bool ok = S.wait(S.full + s, static_cast<uint32_t>((t / P::NS) & 1));
    ok = __all_sync(0xffffffffu, ok);
    const int n = min(kTileGroups, sg.n_valid - j * kTileGroups);
    const uint8_t* st = S.smem + s * P::stage;
    const uint32_t ta = t_lane + C::av + static_cast<uint32_t>(t & 1) * (kTile / 2);
#pragma unroll
    for (int g = 0; g < kTileGroups; ++g) {
      if (ok && g < n) {
        dequant_v_row<D, BITS>(reinterpret_cast<const uint32_t*>(st + P::off_vc + g * P::vcb),
                               reinterpret_cast<const uint32_t*>(st + P::off_vm + g * P::vmb) + cw * 32, ch,
                               ta + g * 16);
      } else {
        const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        vc_tc_st16(ta + g * 16, z);
      }
    }
    vc_tc_wait_st();
    vc_tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      vc_mbar_arrive(S.av + (t & 1));
      vc_mbar_arrive(S.empty + s);
    }
  };

  // tile t's O^T rows of this warp's channels into the running outputs
  auto merge = [&](long long t) {
    const int b = static_cast<int>(t & 1);
    bool ok = S.wait(S.of + b, static_cast<uint32_t>((t >> 1) & 1));
    ok = ok && S.wait(S.mr + b, static_cast<uint32_t>((t >> 1) & 1));
    ok = __all_sync(0xffffffffu, ok);
    vc_tc_fence_after();
    float ot[NL];
    if constexpr (NL == 8) vc_tc_ld8(t_lane + C::o + b * kN, ot);
    else vc_tc_ld16(t_lane + C::o + b * kN, ot);
    if (ok) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mtile = mt[b * kN + h];
        if (mtile > mc[h]) {
          o[h] *= fast_exp2(mc[h] - mtile);                   // mc = -inf at the start: 0
          mc[h] = mtile;
        }
        o[h] += ot[h];
      }
    }
    vc_tc_fence_before();
    __syncwarp();
    if (lane == 0) vc_mbar_arrive(S.ofree + b);
  };

  while (next_segment(a, pos, hi, sg, over)) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      o[h] = 0.0f;
      mc[h] = -INFINITY;
    }
    if (sg.n_tiles > 0) extract(gt, 0);
    for (int j = 0; j < sg.n_tiles; ++j) {
      if (j + 1 < sg.n_tiles) extract(gt + j + 1, j + 1);
      merge(gt + j);
    }
    gt += sg.n_tiles;
    vc_bar_sync(2, R::compute_threads);                        // the token warps' sums are in red
    int first, last;
    ctas_of(sg.bh, a, first, last);
    const int b = sg.bh / a.Hkv, kvh = sg.bh % a.Hkv;
    const int slot = c - first;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float lh = red[h] + red[kN + h] + red[2 * kN + h] + red[3 * kN + h];
      const size_t row = static_cast<size_t>(b * a.Hq + kvh * G + h) * a.max_parts + slot;
      a.part_o[row * D + ch] = lh > 0.0f ? o[h] / lh : 0.0f;
      if (ch == 0) a.part_lse[row] = lh > 0.0f ? mc[h] + log2f(lh) : -INFINITY;
    }
    arrive_and_combine<G, D>(a, S.flag, sg.bh, last - first + 2, R::compute_threads);
    vc_bar_sync(2, R::compute_threads);
  }
}

template <int D, int BITS, int G>
__device__ void stream_cta(const DraftArgs& a, uint8_t* smem, int c) {
  using P = Plan<D, BITS>;
  using R = Roles<D>;
  using C = Cols<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Stream<D, BITS, G> S;
  S.smem = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P::off_bar);
  S.full = bars;
  S.empty = bars + P::NS;
  S.ak = bars + 2 * P::NS;
  S.sf = S.ak + 2;
  S.av = S.sf + 2;
  S.pr = S.av + 2;
  S.of = S.pr + 2;
  S.ofree = S.of + 2;
  S.mr = S.ofree + 2;
  S.done = S.mr + 2;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + P::off_misc);
  S.flag = misc + 1;
  S.abort = misc + 2;
  if (warp == 0) vc_tc_alloc(misc, C::alloc);
  if (threadIdx.x == 32) {
    for (int i = 0; i < P::NS; ++i) {
      vc_mbar_init(S.full + i, 1);
      vc_mbar_init(S.empty + i, R::compute_warps);
    }
    for (int b = 0; b < 2; ++b) {
      vc_mbar_init(S.ak + b, kTokWarps);
      vc_mbar_init(S.sf + b, 1);
      vc_mbar_init(S.av + b, R::chan_warps);
      vc_mbar_init(S.pr + b, kTokWarps);
      vc_mbar_init(S.of + b, 1);
      vc_mbar_init(S.ofree + b, R::chan_warps);
      vc_mbar_init(S.mr + b, 1);
    }
    vc_mbar_init(S.done, 1);
    *S.abort = 0u;
    vc_fence_mbar_init();
  }
  // zero the operand buffers once: the padded heads of Q and P stay zero
  for (int i = threadIdx.x; i < static_cast<int>(2 * (P::q_bytes + P::p_bytes) / 16); i += blockDim.x)
    reinterpret_cast<uint4*>(smem + P::off_q)[i] = make_uint4(0u, 0u, 0u, 0u);
  vc_fence_proxy_async_smem();
  vc_tc_fence_before();
  __syncthreads();
  vc_tc_fence_after();
  S.tmem = misc[0];

  if (warp < kTokWarps) {
    token_warp<D, BITS, G>(a, S, c);
  } else if (warp < R::compute_warps) {
    channel_warp<D, BITS, G>(a, S, c);
  } else if (warp == R::producer_warp) {
    if (lane == 0) produce<D, BITS, G>(a, S, c);
  } else if (lane == 0) {
    issue<D, BITS, G>(a, S, c);
  }
  vc_tc_fence_before();
  __syncthreads();
  vc_tc_fence_after();
  if (threadIdx.x == 0 && *S.abort != 0u) atomicOr(&g_draft_status, VC_DEV_BARRIER_TIMEOUT);
  if (warp == 0) vc_tc_dealloc(S.tmem, C::alloc);
}

// ------------------------------------------------------------------ tail CTA
// bf16 tail tokens 0 .. tail_len + step - 1 and the current token of slice bh.
template <int D, int BITS, int G>
__device__ void tail_cta(const DraftArgs& a, uint8_t* smem, int bh) {
  using T = TailPlan<D, G>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cap = a.tail_cap;
  float* q_s = reinterpret_cast<float*>(smem + T::off_q(cap));
  unsigned int* flag = reinterpret_cast<unsigned int*>(smem + T::off_flag(cap));
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
    arrive_and_combine<G, D>(a, flag, bh, n_c + 1, blockDim.x);
    return;
  }
  uint16_t* krow = reinterpret_cast<uint16_t*>(smem);                      // [n_tok][D]
  uint16_t* vrow = krow + static_cast<size_t>(cap + 1) * D;
  float* sc = reinterpret_cast<float*>(smem + T::off_sc(cap));             // [G][n_tok]
  float* ml = reinterpret_cast<float*>(smem + T::off_ml(cap));             // [G][2]
  constexpr int VEC = D / 8;
  for (int i = threadIdx.x; i < n_tok * VEC; i += blockDim.x) {
    const int t = i / VEC, v = i % VEC;
    const uint16_t* ks = (t < n_tail) ? a.tail_k + tbase + static_cast<size_t>(t) * D : a.k_cur + static_cast<size_t>(bh) * D;
    const uint16_t* vs = (t < n_tail) ? a.tail_v + tbase + static_cast<size_t>(t) * D : a.v_cur + static_cast<size_t>(bh) * D;
    *reinterpret_cast<uint4*>(krow + t * D + v * 8) = *reinterpret_cast<const uint4*>(ks + v * 8);
    *reinterpret_cast<uint4*>(vrow + t * D + v * 8) = *reinterpret_cast<const uint4*>(vs + v * 8);
  }
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    q_s[i] = vc_bf16_to_f32(a.q[(static_cast<size_t>(b) * a.Hq + kvh * G + h) * D + c]) * a.scale_log2;
  }
  __syncthreads();
  // scores: warp per token, lanes over channel pairs
  const int nw = blockDim.x / 32;
  for (int t = warp; t < n_tok; t += nw) {
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
  for (int h = warp; h < G; h += nw) {
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
  arrive_and_combine<G, D>(a, flag, bh, n_c + 1, blockDim.x);
}

template <int D, int BITS, int G>
__global__ void __launch_bounds__(Roles<D>::threads, 1) draft_kernel(DraftArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
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
  if (s->bits != 2 && s->bits != 4 && s->bits != 8) VC_FAIL(VC_ERR_UNSUPPORTED, "bits %d not in {2, 4, 8}", s->bits);
  const int G = s->Hq / s->Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 5 && G != 8) VC_FAIL(VC_ERR_UNSUPPORTED, "G = %d not in {1,2,4,5,8}", G);
  VC_REQUIRE(s->softmax_scale > 0.0f, "softmax_scale must be positive");
  return VC_OK;
}

struct LaunchPlan {
  int n_stream = 0, max_parts = 1, threads = 0;
  long long total = 0;
  size_t smem = 0;
};

template <int D, int BITS, int G>
vc_status_t plan_t(const vc_shape_t* s, int max_packed, LaunchPlan* lp) {
  using P = Plan<D, BITS>;
  auto fn = draft_kernel<D, BITS, G>;
  VC_CUDA_CHECK(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(P::total)));
  int dev = 0, sms = 0, occ = 0;
  VC_CUDA_CHECK(cudaGetDevice(&dev));
  VC_CUDA_CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  VC_CUDA_CHECK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, Roles<D>::threads, P::total));
  if (occ < 1) VC_FAIL(VC_ERR_UNSUPPORTED, "draft kernel does not fit on an SM");
  const long long NGmax = max_packed / kGroup;
  lp->total = static_cast<long long>(s->B) * s->Hkv * NGmax;
  long long n = sms;                                            // one CTA per SM (TMEM and shared memory)
  const long long by_work = lp->total / kTileGroups;            // at least one tile per CTA
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
  lp->threads = Roles<D>::threads;
  return VC_OK;
}

vc_status_t plan(const vc_shape_t* s, int max_packed, LaunchPlan* lp) {
  const int G = s->Hq / s->Hkv;
#define VC_PLAN(D_, B_, G_) \
  if (s->d == D_ && s->bits == B_ && G == G_) return plan_t<D_, B_, G_>(s, max_packed, lp);
#define VC_PLAN_G(D_, B_) VC_PLAN(D_, B_, 1) VC_PLAN(D_, B_, 2) VC_PLAN(D_, B_, 4) VC_PLAN(D_, B_, 5) VC_PLAN(D_, B_, 8)
  VC_PLAN_G(128, 2) VC_PLAN_G(128, 4) VC_PLAN_G(128, 8) VC_PLAN_G(64, 2) VC_PLAN_G(64, 4) VC_PLAN_G(64, 8)
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
  if (TailPlan<D, G>::total(a.tail_cap) > Plan<D, BITS>::total)
    VC_FAIL(VC_ERR_UNSUPPORTED, "tail_cap %d too large for the shared-memory plan", a.tail_cap);
  const int grid = a.B * a.Hkv + lp.n_stream;
  draft_kernel<D, BITS, G><<<grid, lp.threads, lp.smem, cs>>>(a);
  VC_LAUNCH_CHECK("draft_kernel");
  return VC_OK;
}

vc_status_t launch(const vc_shape_t* s, const DraftArgs& a, const LaunchPlan& lp, cudaStream_t cs) {
  const int G = s->Hq / s->Hkv;
#define VC_L(D_, B_, G_) \
  if (s->d == D_ && s->bits == B_ && G == G_) return launch_t<D_, B_, G_>(a, lp, cs);
#define VC_L_G(D_, B_) VC_L(D_, B_, 1) VC_L(D_, B_, 2) VC_L(D_, B_, 4) VC_L(D_, B_, 5) VC_L(D_, B_, 8)
  VC_L_G(128, 2) VC_L_G(128, 4) VC_L_G(128, 8) VC_L_G(64, 2) VC_L_G(64, 4) VC_L_G(64, 8)
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
