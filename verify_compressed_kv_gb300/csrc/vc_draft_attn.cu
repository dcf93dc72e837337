// libvc_draft_attn: decode attention over the KIVI-packed draft cache.
//
// VeriCache (gist.science/paper/2605.17613), Technical Summary, Core
// Algorithm (Drafting: candidate tokens come from the compressed KV) and Key
// System Innovations (drafting is bound by HBM bandwidth, reading the
// compressed KV).  One query token per request per step; all G query heads
// of a KV head share every byte read.
//
// One launch per draft step: one wave of persistent stream CTAs (occupancy x
// SM count):
//   * stream-K partition: the packed groups of every (request, KV head) are
//     laid end to end and each stream CTA takes a contiguous range, so the
//     work is balanced whatever B*Hkv is; a range may span several heads
//     (segments).  The ranges are balanced by cost, not by groups: a head
//     switch inside a range and a bf16 tail pass (below) are each charged as
//     a number of groups, measured on per-CTA timestamps;
//   * a segment is streamed through a ring of shared-memory stages (11 groups
//     of 32 tokens each: K codes, K scale/zero, V codes, V scale/zero), filled
//     by bulk async copies (cp.async.bulk + mbarrier transaction counts, bounded
//     waits) while the 11 consumer warps compute on earlier stages;
//   * each warp owns one group per stage and keeps its own online-softmax
//     state (max, sums) and output accumulators for all G heads of the KV
//     head, on 16x8x16 fp16 tensor-core products with the codes as the A
//     operand and the heads as the 8 columns (group_mma): a packed code field,
//     masked in place, is itself an fp16 subnormal, code * 2^(p - 24), so an
//     operand register of two codes costs one AND; the key scales and the
//     codes' powers of two fold into the query, the value scales into the
//     softmax weights, and the zero points enter through two narrow products
//     (q . z per head; weights . z per channel group).  The folded operands
//     are single fp16 values: the draft is lossy by design, and their
//     rounding sits far below the codes' own error;
//   * at the end of a segment the warps are merged (log-sum-exp) into one
//     partial per query head; the last CTA to finish a (request, KV head)
//     (arrival counter in the workspace, reset by that CTA) merges all its
//     partials and writes the bf16 output.
// The bf16 tails (tokens committed since the last full group, earlier draft
// steps, the current token) are taken by the stream CTAs before their ranges
// (the ring fills meanwhile), each slice's by a fixed CTA, which also stores
// the current token's K/V into the tail for the following steps.  Without packed groups, tail CTAs alone
// take them.
#include <algorithm>
#include <cfloat>
#include <climits>
#include <mutex>
#include <vector>

#include "vc_internal.h"

namespace {

__device__ uint32_t g_draft_status = 0;

// 11 consumer warps + 1 producer: three warps per scheduler, the same
// register budget (168) as 8 + 1.
constexpr int kWarps = 11;                      // consumer warps of a stream CTA (one group each per stage)
constexpr int kConsumers = kWarps * 32;
constexpr int kThreads = kConsumers + 32;        // + one producer warp
constexpr int kGroup = 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxStream = 512;                 // stream CTAs one launch can describe (partition table)
// Costs charged in the partition, in 32-token groups of 3072 bytes (d = 128,
// int2), scaled by 3072 / (bytes of a group) for other shapes.  Per-CTA
// timestamps: such a group streams in ~0.1 us; a head switch inside a range
// costs 6-8 us (flush, the next head's queries, ring refill); a tail pass
// ~5 us (a chain of dependent global round trips under full HBM load).
constexpr long long kSwitchGroups = 72;
constexpr long long kTailGroups = 50;
constexpr long long kRefGroupBytes = 3072;
constexpr long long kWaitCycles = 4000000000LL;   // default wait bound: ~2 s at 2 GHz
// Test hooks (vc_draft_attn_test_hooks): the wait bound and a withheld first
// stage, so that a test can make the bounded waits run out.  Host side only.
long long g_wait_cycles = kWaitCycles;
int g_withhold_first = 0;
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
  int n_stream;             // stream CTAs (0: no packed groups)
  int n_cta;                // CTAs launched: n_stream stream CTAs, or tail CTAs alone
  long long total;          // B * Hkv * NGmax
  int max_parts;            // partial slots per (b, h): stream CTAs + the tail
  float scale_log2;
  long long wait_cycles;    // bound of every mbarrier wait (clock64 cycles)
  int withhold_first;       // test only: the producers issue nothing for their first stage
  float* part_o;            // [B*Hq, max_parts, D]   normalised partial outputs
  float* part_lse;          // [B*Hq, max_parts]      log2-sum-exp of each partial
  unsigned int* counter;    // [B*Hkv] arrivals (zero between calls)
  uint16_t* out;            // [B, Hq, D]
  int lo_tab[kMaxStream + 1];  // stream CTA c takes groups [lo_tab[c], lo_tab[c + 1]) (slice-major)
};

// Programmatic dependent launch.  Every CTA lets the next grid on the stream
// launch as soon as it starts; that grid's CTAs then take SMs as this one's
// finish.  Every CTA's consumer threads wait for the previous grid before
// their first read of anything but the packed cache, so a grid completes only
// after its predecessor did, and each grid sees all earlier grids' writes.
// Both instructions are no-ops for a launch without the programmatic
// serialisation attribute.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ partition
// Start of stream CTA c's groups in the stream-K order.
__host__ __device__ inline long long range_lo(long long c, const DraftArgs& a) {
  return c >= a.n_stream ? a.total : a.lo_tab[c];
}

// The stream CTA whose range holds position x: the largest c < n with
// lo[c] <= x (lo[0] = 0 and the ranges are non-empty up to the last group).
__host__ __device__ inline int cta_at(long long x, const int* lo, int n) {
  int l = 0, h = n - 1;
  while (l < h) {
    const int m = (l + h + 1) >> 1;
    if (lo[m] <= x) l = m; else h = m - 1;
  }
  return l;
}

// Stream CTAs overlapping the groups of (b, h) index bh: [first, last].
__host__ __device__ inline void ctas_of(int bh, const DraftArgs& a, int& first, int& last) {
  if (a.n_stream <= 0 || a.NGmax <= 0) {
    first = 0;
    last = -1;
    return;
  }
  const long long s = static_cast<long long>(bh) * a.NGmax;
  first = cta_at(s, a.lo_tab, a.n_stream);
  last = cta_at(s + a.NGmax - 1, a.lo_tab, a.n_stream);
}

// Slices whose bf16 tail stream CTA c runs after its range: bh with
// floor(bh * n / nbh) = c, i.e. [tail_lo(c), tail_lo(c + 1)).
__host__ __device__ inline long long tail_lo(long long c, long long n, long long nbh) {
  return (c * nbh + n - 1) / n;
}

// ------------------------------------------------------------------ shared memory plan
template <int D, int BITS, int G>
struct Plan {
  static constexpr size_t codes = static_cast<size_t>(D) * BITS * 4;   // bytes of one group's K (or V) codes
  static constexpr size_t meta = static_cast<size_t>(D) * 4;           // bytes of one group's K (or V) meta
  static constexpr size_t kc = kWarps * codes;                         // a stage holds kWarps groups
  static constexpr size_t mt = kWarps * meta;
  static constexpr size_t stage = 2 * kc + 2 * mt;                      // K codes, K meta, V codes, V meta
  // ring depth: about 100 KB of stages in flight, at least double buffering
  static constexpr int NS = (100 * 1024 / stage) < 2 ? 2 : ((100 * 1024 / stage) > 6 ? 6 : static_cast<int>(100 * 1024 / stage));
  static constexpr size_t ring = stage * NS;
  static constexpr size_t red = static_cast<size_t>(kWarps) * G * D * 4;   // warp merge
  static constexpr size_t off_red = ring;
  static constexpr size_t body = ring + red;
  static constexpr size_t wstat = static_cast<size_t>(kWarps) * 8 * 2 * 4;  // per-warp (max, sum) per head
  static constexpr size_t off_wstat = body;
  static constexpr size_t off_bar = (off_wstat + wstat + 15) & ~size_t(15);   // full[NS], empty[NS]
  static constexpr size_t off_flag = off_bar + 16 * NS;                      // combine flag, abort flag
  static constexpr size_t total = off_flag + 16;
};

// Issue the bulk copies of one stage (groups [g, g + n) of slice bh) into `buf`.
template <int D, int BITS, int G>
__device__ __forceinline__ void issue_stage(const DraftArgs& a, uint8_t* buf, uint64_t* bar, int bh, int g, int n) {
  using P = Plan<D, BITS, G>;
  const size_t gb = static_cast<size_t>(bh) * a.NG + g;
  const uint32_t code_bytes = static_cast<uint32_t>(n * P::codes);
  const uint32_t meta_bytes = static_cast<uint32_t>(n * P::meta);
  vc_mbar_arrive_expect_tx(bar, 2 * code_bytes + 2 * meta_bytes);
  vc_bulk_g2s(buf, a.kc + gb * D * BITS, code_bytes, bar);
  vc_bulk_g2s(buf + P::kc, a.ksz + gb * 2 * D, meta_bytes, bar);
  vc_bulk_g2s(buf + P::kc + P::mt, a.vc + gb * D * BITS, code_bytes, bar);
  vc_bulk_g2s(buf + 2 * P::kc + P::mt, a.vsz + gb * 2 * D, meta_bytes, bar);
}

// ------------------------------------------------------------------ tensor-core pieces
// 16x8x16 products, fp16 operands, fp32 accumulators.  Lane = 4*gid + tig.
// A rows: gid = head gid (leading part), gid + 8 = the same head (remainder
// part), so that hi + lo carry ~22 significant bits of a product that fp16
// alone would round to 11.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x (ex2.approx.ftz: relative error ~2^-22; results below 2^-126 flush to 0)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Code operands.  A packed code field becomes a tensor-core operand with no
// arithmetic: masked in place inside the mantissa of an fp16 whose exponent
// bits are zero, the field IS the subnormal number code * 2^(p - 24), p its
// lowest bit.  One AND (one immediate) per operand register, two codes, one
// per 16-bit half; the fields that lie above bit 9 are first brought down by
// one shift of the whole word, shared by every field of that word.  The power
// 2^(p - 24) is folded into the other operand (the query, per k-step and
// register, for keys; the weights per register and a per-channel output factor
// for values) and into the softmax scale.  Field positions (include/vc.h):
//   b = 2: slot (u, r) at 16e + 4u + 2(1 - r); u = 2, 3 from the word shifted
//          right by 6, so p = R(u) + C(r), R = {0, 4, 2, 6}, C(r) = 2(1 - r);
//   b = 4: slot u at 16e + 4u; u = 2, 3 from the word shifted right by 8, so
//          p = 4 (u & 1), which is 4r for keys and values alike;
//   b = 8: slot u at 16e + 8u; u = 1 from the word shifted right by 8; p = 0.
template <int BITS>
__host__ __device__ constexpr int pos_row(int u) {
  return BITS == 2 ? 4 * (u & 1) + 2 * (u >> 1) : 0;
}
template <int BITS>
__host__ __device__ constexpr int pos_col(int r) {
  return BITS == 2 ? 2 * (1 - r) : (BITS == 4 ? 4 * r : 0);
}
// Key operands carry slot u = ks % 4 in k-step ks (b = 2), so the field
// position of register r of k-step ks is:
template <int BITS>
__host__ __device__ constexpr int pos_key(int ks, int r) {
  return pos_row<BITS>(ks % 4) + pos_col<BITS>(r);
}
// The folded operands keep the codes' powers of two at most 2^kFold, as the
// weights (<= 2^kLazy) and the folded query must stay inside the fp16 range:
// keys Q' = q s 2^(kFold - p) (scores come out times 2^(kFold - 24)), values
// P' = p s 2^(kFold - C(r)) (outputs times 2^(kFold - 24 + R(u))).
constexpr int kFold = 4;
// fp16 2^k in both halves of a register (|k| <= 14).
__host__ __device__ constexpr uint32_t pow2_h2(int k) {
  return (static_cast<uint32_t>(k + 15) << 10) * 0x10001u;
}

// Operand registers (r = 0, 1) of fragment index i — the field rules of the
// packed words (include/vc.h): b = 2: word i/4, slot u = i%4; b = 4: i2 = 2i + r,
// word i2/4, slot u = i2%4; b = 8: word (2i + r)/2 = i, slot u = r.
template <int BITS, int WPL>
__device__ __forceinline__ void code_operands(const uint32_t (&w)[WPL], int i, uint32_t& b0, uint32_t& b1) {
  if (BITS == 2) {
    const int u = i % 4;
    const uint32_t x = u < 2 ? w[i / 4] : (w[i / 4] >> 6);
    b0 = x & (0x00030003u << (pos_row<2>(u) + pos_col<2>(0)));
    b1 = x & (0x00030003u << (pos_row<2>(u) + pos_col<2>(1)));
  } else if (BITS == 4) {
    const int i0 = 2 * i, i1 = 2 * i + 1;
    b0 = ((i0 % 4) < 2 ? w[i0 / 4] : (w[i0 / 4] >> 8)) & 0x000F000Fu;
    b1 = ((i1 % 4) < 2 ? w[i1 / 4] : (w[i1 / 4] >> 8)) & 0x00F000F0u;
  } else {
    b0 = w[i] & 0x00FF00FFu;
    b1 = (w[i] >> 8) & 0x00FF00FFu;
  }
}

// The lane's words of one group: word w at (w/4)*128 + 4*lane + w%4.
template <int WPL>
__device__ __forceinline__ void load_lane_words(const uint32_t* g, int lane, uint32_t (&w)[WPL]) {
#pragma unroll
  for (int c = 0; c < WPL / 4; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(g + c * 128 + 4 * lane);
    w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
  }
}

// Rescale threshold (log2 units): the running max is raised only when a group's
// max exceeds it by more than this, so weights stay <= 2^kLazy * 16.
constexpr float kLazy = 3.0f;

// ------------------------------------------------------------------ group product
// One group of 32 tokens for all G heads of the warp's KV head, on tensor
// cores with the codes as the A operand and the heads as the 8 columns:
//   S^T = codes . Q'^T (16 tokens per m-tile, k = channels), and
//   O^T += V^T . P'^T  (16 channels per m-tile, k = tokens),
// 16 QK + 16 PV products per group (d = 128).  With
//   score(t) = sum_c q_c (s_c code_tc + z_c) = sum_c Q'_c code_tc 2^(p_c - 24) 2^(24 - kFold) + sum_c q_c z_c
// the first sum is the QK product (code operands as above, Q' = q s 2^(kFold - p)
// per k-step and register) and the second, the bias, one narrow product per
// k-step with A = q and B = the zeros.  Likewise
//   out_h(c) = sum_t p_t (sv_t code_tc + zv_t)
// is the PV product (P' = p sv 2^(kFold - C(r))) times the channel's output
// factor, plus one correction product per k-step with A = the weights and B =
// the zeros of each channel group.  The packed words need no change: the B
// fragment of n-tile j is the top (b0) / bottom (b1) register pair of an A
// fragment whose rows are the tokens of n-tiles j and j' (a0 = b0 of j, a1 =
// b0 of j', a2 = b1 of j, a3 = b1 of j').  The QK accumulator block of tokens
// 4 gid + j (j = 2 mt + half), transposed in registers (movmatrix), is the PV
// B fragment of k-step s = j / 2, register r = j % 2.  G = 4 fills columns
// 4-7 with the same 4 heads at zero weight (each lane then holds whole heads).

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Per-warp running state of one segment: the lane's heads are h0 = 2 (tig & 1)
// (G = 4) or 2 tig, and h0 + 1.
template <int D>
struct WarpState {
  static constexpr int MT = D / 16;
  float o[MT][4];       // O^T: rows = channels 16 mt + gid (+ 8), cols 2 tig (+1) = heads h0 (+1)
  float oz[4];          // correction: rows = P' columns (head gid; G = 4: gid & 3), cols = channel group tig (zeros)
  float l0[2], l1[2];   // per head: sums of the weights of r = 0 / r = 1 tokens (times 2^(kFold - C(r)))
  float m[2];           // per head: running max (log2 units)
};

template <int D>
__device__ __forceinline__ void init_state(WarpState<D>& st) {
#pragma unroll
  for (int m = 0; m < D / 16; ++m) st.o[m][0] = st.o[m][1] = st.o[m][2] = st.o[m][3] = 0.0f;
  st.oz[0] = st.oz[1] = st.oz[2] = st.oz[3] = 0.0f;
  st.l0[0] = st.l0[1] = st.l1[0] = st.l1[1] = 0.0f;
  st.m[0] = st.m[1] = -INFINITY;
}

// cs = softmax scale in log2 units; cs_code = cs * 2^(24 - kFold) for the
// code products.
template <int D, int BITS, int G>
__device__ __forceinline__ void group_mma(const uint32_t* kc_g, const uint16_t* ksz_g, const uint32_t* vc_g,
                                          const uint16_t* vsz_g, const uint32_t (&qf)[D / 16][2],
                                          uint32_t zcol_mul0, uint32_t zcol_mul1, int zcol_off, float cs,
                                          float cs_code, WarpState<D>& st, int lane) {
  constexpr int KS = D / 16, NT = D / 8, NCG = D / 32, WPL = D * BITS / 32;
  const int gid = lane >> 2, tig = lane & 3;
  const bool lo_p = G == 4 && tig >= 2;         // G = 4: columns 4-7 (zero weight)
  const int h0 = G == 4 ? 2 * (tig & 1) : 2 * tig;
  // ---------------- S^T = codes . Q'^T
  uint32_t kw[WPL];
  load_lane_words<WPL>(kc_g, lane, kw);
  const uint32_t* srow = reinterpret_cast<const uint32_t*>(ksz_g) + (D / 8) * tig;
  // bias columns: gid 0 and 1 feed the zeros (of the even / odd k-step of a pair)
  const uint32_t* zrow = reinterpret_cast<const uint32_t*>(ksz_g) + (gid <= 1 ? D / 2 : 0) + (D / 8) * tig;
  float c[2][2][4];                              // [m-tile][k-step parity]: two short chains each
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) c[mt][h][0] = c[mt][h][1] = c[mt][h][2] = c[mt][h][3] = 0.0f;
  float cb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int kq = 0; kq < KS / 2; ++kq) {
    const uint4 s4 = *reinterpret_cast<const uint4*>(srow + 4 * kq);
    const uint4 z4 = *reinterpret_cast<const uint4*>(zrow + 4 * kq);
    const uint32_t sv[4] = {s4.x, s4.y, s4.z, s4.w};
    const uint32_t zv[4] = {z4.x, z4.y, z4.z, z4.w};
    // bias q . z of k-steps 2 kq and 2 kq + 1 in one product: A rows 0-7 = q of the
    // even k-step, rows 8-15 = q of the odd one; B column 0 = zeros of the even,
    // column 1 = zeros of the odd k-step (q itself: the power of two undone exactly)
    uint32_t qz[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int e = pos_key<BITS>(2 * kq + h, r) - kFold;
        qz[h][r] = e == 0 ? qf[2 * kq + h][r] : h2u(__hmul2(u2h(qf[2 * kq + h][r]), u2h(pow2_h2(e))));
      }
    mma16816(cb, qz[0][0], qz[1][0], qz[0][1], qz[1][1], gid == 1 ? zv[2] : zv[0], gid == 1 ? zv[3] : zv[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int ks = 2 * kq + h;
      // Q'^T column n carries head n (G = 4: head n & 3): fp16 q s 2^(kFold - p)
      const uint32_t qb0 = h2u(__hmul2(u2h(qf[ks][0]), u2h(sv[2 * h])));
      const uint32_t qb1 = h2u(__hmul2(u2h(qf[ks][1]), u2h(sv[2 * h + 1])));
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        uint32_t a0, a1, a2, a3;
        code_operands<BITS, WPL>(kw, (2 * mt) * KS + ks, a0, a2);
        code_operands<BITS, WPL>(kw, (2 * mt + 1) * KS + ks, a1, a3);
        mma16816(c[mt][h], a0, a1, a2, a3, qb0, qb1);
      }
    }
  }
  // bias of head h: row h, column 0 plus row h + 8, column 1 (lane 4 h)
  const float cbs = cb[0] + cb[3];
  const float bias[2] = {__shfl_sync(0xffffffffu, cbs, 4 * h0), __shfl_sync(0xffffffffu, cbs, 4 * h0 + 4)};
  // y[mt][2 half + hh] = code part of the score of token 4 gid + 2 mt + half, head
  // h0 + hh, times 2^(kFold - 24) (columns 2 tig, 2 tig + 1 hold heads h0, h0 + 1)
  float y[2][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int k = 0; k < 4; ++k) y[mt][k] = c[mt][0][k] + c[mt][1][k];
  // ---------------- online softmax, one state per head
  // The running max is raised only past max + kLazy: a lane-local check of its own
  // 4 tokens per head, and the exact group max (8 lanes) only when some lane needs it.
  float my[2];
  bool need_l = false;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    my[hh] = fmaxf(fmaxf(y[0][hh], y[0][2 + hh]), fmaxf(y[1][hh], y[1][2 + hh]));
    need_l = need_l || !(fmaf(my[hh], cs_code, bias[hh] * cs) <= st.m[hh] + kLazy);
  }
  if (__any_sync(0xffffffffu, need_l)) {
    float alpha[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float g = my[hh];
      g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, 4));
      g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, 8));
      g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, 16));
      const float mx = fmaf(g, cs_code, bias[hh] * cs);
      const float mn = mx <= st.m[hh] + kLazy ? st.m[hh] : mx;
      alpha[hh] = fast_exp2(st.m[hh] - mn);     // m = -inf at the start: alpha = 0
      st.l0[hh] *= alpha[hh];
      st.l1[hh] *= alpha[hh];
      st.m[hh] = mn;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      st.o[mt][0] *= alpha[0];
      st.o[mt][1] *= alpha[1];
      st.o[mt][2] *= alpha[0];
      st.o[mt][3] *= alpha[1];
    }
    // correction row gid belongs to head gid (gid & 3 for G = 4): its factor sits in
    // the lane of that row whose columns hold the head
    const float a_g = (gid & 1) ? alpha[1] : alpha[0];
    const float a_oz = __shfl_sync(0xffffffffu, a_g, 4 * gid + (G == 4 ? ((gid & 3) >> 1) : (gid >> 1)));
#pragma unroll
    for (int k = 0; k < 4; ++k) st.oz[k] *= a_oz;
  }
  const float kk[2] = {fmaf(bias[0], cs, -st.m[0]), fmaf(bias[1], cs, -st.m[1])};
  // weights times 2^(kFold - C(r)) (r = token parity = half) in fp16; block j = 2 mt + half
  uint32_t ph[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int mt = j >> 1, half = j & 1;
    const float lf = static_cast<float>(kFold - pos_col<BITS>(half));
    const float p0 = fast_exp2(fmaf(y[mt][2 * half], cs_code, kk[0] + lf));
    const float p1 = fast_exp2(fmaf(y[mt][2 * half + 1], cs_code, kk[1] + lf));
    if (half) {
      st.l1[0] += p0;
      st.l1[1] += p1;
    } else {
      st.l0[0] += p0;
      st.l0[1] += p1;
    }
    ph[j] = h2u(__floats2half2_rn(p0, p1));
  }
  // ---------------- correction: A = P' blocks transposed (rows = P' columns; rows 8-15 zero), B = zero columns
  // pu[j], lane (gid, tig): head gid (G = 4: gid & 3), tokens 8 tig + j and 8 tig + 4 + j
  uint32_t pu[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) pu[j] = movmatrix_t(lo_p ? 0u : ph[j]);
  {
    const uint4 r4 = *reinterpret_cast<const uint4*>(vsz_g + zcol_off + 8 * tig);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t b0 = h2u(__hmul2(u2h(s ? r4.z : r4.x), u2h(zcol_mul0)));
      const uint32_t b1 = h2u(__hmul2(u2h(s ? r4.w : r4.y), u2h(zcol_mul1)));
      mma16816(st.oz, pu[2 * s], 0u, pu[2 * s + 1], 0u, b0, b1);
    }
  }
  // ---------------- O^T += V^T . P'^T, one P'^T per channel group (the value scales of its tokens)
  uint32_t vw[WPL];
  load_lane_words<WPL>(vc_g, lane, vw);
#pragma unroll
  for (int g = 0; g < NCG; ++g) {
    // scales of tokens 8 tig + j, 8 tig + 4 + j: word 4 tig + j of the group's
    // scale row (the value meta layout pairs exactly these tokens)
    const uint4 s4 = *reinterpret_cast<const uint4*>(vsz_g + g * 64 + 8 * tig);
    const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w};
    uint32_t pb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) pb[j] = h2u(__hmul2(u2h(pu[j]), u2h(sw[j])));
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int m = 2 * g + u;                  // channels 16 m .. 16 m + 15 = n-tiles 2 m, 2 m + 1
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        uint32_t a0, a1, a2, a3;
        code_operands<BITS, WPL>(vw, s * NT + 2 * m, a0, a2);
        code_operands<BITS, WPL>(vw, s * NT + 2 * m + 1, a1, a3);
        mma16816(st.o[m], a0, a1, a2, a3, pb[2 * s], pb[2 * s + 1]);
      }
    }
  }
}

// ------------------------------------------------------------------ merge / arrive / combine
template <int D, int BITS, int G>
__device__ void merge_partials(const DraftArgs& a, uint8_t* smem, int bh, int slot);

// The warps' (max, sum, output) of slice bh, left in `red` / `wstat` by the
// consumer warps (after a consumer barrier), merged into one normalised
// partial + log2-sum-exp per head.
template <int D, int BITS, int G>
__device__ void merge_partials(const DraftArgs& a, uint8_t* smem, int bh, int slot) {
  using P = Plan<D, BITS, G>;
  const float* red = reinterpret_cast<const float*>(smem + P::off_red);
  const float* wstat = reinterpret_cast<const float*>(smem + P::off_wstat);
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  for (int i = threadIdx.x; i < G * D; i += kConsumers) {
    const int h = i / D, c = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int x = 0; x < kWarps; ++x) M = fmaxf(M, wstat[(x * 8 + h) * 2]);
    const size_t row = static_cast<size_t>(b * a.Hq + kvh * G + h) * a.max_parts + slot;
    if (M == -INFINITY) {
      if (c == 0) a.part_lse[row] = -INFINITY;
      continue;
    }
    float o = 0.0f, Ls = 0.0f;
#pragma unroll
    for (int x = 0; x < kWarps; ++x) {
      const float mx = wstat[(x * 8 + h) * 2];
      if (mx == -INFINITY) continue;
      const float wgt = exp2f(mx - M);
      o = fmaf(wgt, red[(x * G + h) * D + c], o);
      Ls = fmaf(wgt, wstat[(x * 8 + h) * 2 + 1], Ls);
    }
    a.part_o[row * D + c] = o / Ls;
    if (c == 0) a.part_lse[row] = M + log2f(Ls);
  }
}

// Partial of this CTA for slice bh: each warp leaves per head its output
// (G = 4: the column and its zero-weight repeat added; the code part times the
// channel's output factor 2^(24 - kFold - R(u)), plus the correction of the
// channel group) and its (max, softmax sum) in shared memory; then the warps
// are merged into one normalised partial + log2-sum-exp per head.
template <int D, int BITS, int G>
__device__ void write_partial(const DraftArgs& a, uint8_t* smem, int bh, int slot, WarpState<D>& st) {
  using P = Plan<D, BITS, G>;
  static_assert(G <= 8, "the group product carries at most 8 heads");
  constexpr int MT = D / 16, NCG = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int h0 = G == 4 ? 2 * (tig & 1) : 2 * tig;
  float* red = reinterpret_cast<float*>(smem + P::off_red);             // [warp][G][D]
  float* wstat = reinterpret_cast<float*>(smem + P::off_wstat);         // [warp][8][2]
  // correction of (head of row gid, channel group tig); G = 4: rows gid and gid ^ 4 hold the same head
  float cz = st.oz[0] + st.oz[1] + st.oz[2] + st.oz[3];
  if (G == 4) cz += __shfl_xor_sync(0xffffffffu, cz, 16);
  float corr[2][NCG];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int g = 0; g < NCG; ++g) corr[hh][g] = __shfl_sync(0xffffffffu, cz, 4 * (h0 + hh) + g);
  float l[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float x = st.l0[hh] * exp2f(static_cast<float>(pos_col<BITS>(0) - kFold)) +
              st.l1[hh] * exp2f(static_cast<float>(pos_col<BITS>(1) - kFold));
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    x += __shfl_xor_sync(0xffffffffu, x, 16);
    l[hh] = x;
  }
  float v[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      v[m][e] = G == 4 ? st.o[m][e] + __shfl_xor_sync(0xffffffffu, st.o[m][e], 2) : st.o[m][e];
  if (G != 4 || tig < 2) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const int c0 = 16 * m + gid, g = m / 2;
      // rows gid / gid + 8 of m-tile m: n-tiles 2 m / 2 m + 1, slots (2 m) % 4 / (2 m + 1) % 4
      const float f_lo = exp2f(static_cast<float>(24 - kFold - pos_row<BITS>((2 * m) % 4)));
      const float f_hi = exp2f(static_cast<float>(24 - kFold - pos_row<BITS>((2 * m + 1) % 4)));
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (h0 + hh >= G) continue;
        red[(warp * G + h0 + hh) * D + c0] = fmaf(v[m][hh], f_lo, corr[hh][g]);
        red[(warp * G + h0 + hh) * D + c0 + 8] = fmaf(v[m][2 + hh], f_hi, corr[hh][g]);
      }
    }
    if (gid == 0) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (h0 + hh >= G) continue;
        wstat[(warp * 8 + h0 + hh) * 2] = st.m[hh];
        wstat[(warp * 8 + h0 + hh) * 2 + 1] = l[hh];
      }
    }
  }
  vc_bar_sync(1, kConsumers);
  merge_partials<D, BITS, G>(a, smem, bh, slot);
}

// Count this CTA's partial for slice bh; the last of the n_parts arrivals
// merges all partials of the slice and writes its bf16 output.  The consumer
// warps of the CTA take part (named barrier 1; the producer warp does not).
__device__ __forceinline__ void sync_part(int nthr) { vc_bar_sync(1, nthr); }

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
    // parts 8 at a time, all loads of a chunk in flight together; the running
    // (max, numerator, denominator) is rescaled when a chunk raises the max
    float M = -INFINITY, num = 0.0f, den = 0.0f;
    for (int x0 = 0; x0 < n_parts; x0 += 8) {
      float lse[8], ov[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const bool in = x0 + u < n_parts;
        lse[u] = in ? __ldcg(a.part_lse + row + x0 + u) : -INFINITY;
        ov[u] = in ? __ldcg(a.part_o + (row + x0 + u) * D + c) : 0.0f;
      }
      float cm = M;
#pragma unroll
      for (int u = 0; u < 8; ++u) cm = fmaxf(cm, lse[u]);
      if (cm == -INFINITY) continue;
      const float r = exp2f(M - cm);             // M = -inf: 0
      num *= r;
      den *= r;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (lse[u] == -INFINITY) continue;         // an empty part: its output is not read
        const float wgt = exp2f(lse[u] - cm);
        num = fmaf(wgt, ov[u], num);
        den += wgt;
      }
      M = cm;
    }
    a.out[(static_cast<size_t>(b) * a.Hq + kvh * G + h) * D + c] = vc_f32_to_bf16_rn(den > 0.0f ? num / den : 0.0f);
  }
  if (threadIdx.x == 0) a.counter[bh] = 0u;          // zero again for the next call
}

// ------------------------------------------------------------------ bf16 tail
// The bf16 tail tokens 0 .. tail_len + step - 1 and the current token of slice
// bh, taken by the consumer warps of the stream CTA the slice's tail is
// assigned to (of a tail CTA when there are no packed groups).  Warp w takes the tokens t = w
// (mod kWarps), 8 in flight, K and V rows straight from global memory (each
// lane D/32 channels), with an online-softmax state per head in registers;
// the warps' (max, sum, output) go to the warp-merge region and
// merge_partials writes the tail's partial (the slot after the stream CTAs'
// of the slice).  The current token's K/V are kept in the tail for the
// following steps.
template <int D, int BITS, int G>
__device__ void tail_part(const DraftArgs& a, uint8_t* smem, int bh) {
  using P = Plan<D, BITS, G>;
  constexpr int CPL = D / 32;                  // channels per lane
  constexpr int U = 8;                         // tokens per warp in flight
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* red = reinterpret_cast<float*>(smem + P::off_red);
  float* wstat = reinterpret_cast<float*>(smem + P::off_wstat);
  unsigned int* flag = reinterpret_cast<unsigned int*>(smem + P::off_flag);
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  int first, last;
  ctas_of(bh, a, first, last);
  const int n_c = last - first + 1;
  const int slot = n_c;                        // the tail's partial follows the stream CTAs'
  const int n_tail = a.tail_len[b] + a.step;
  const bool has_cur = a.k_cur != nullptr;
  const int n_tok = n_tail + (has_cur ? 1 : 0);
  const size_t tbase = static_cast<size_t>(bh) * a.tail_cap * D;
  const bool bad = n_tail < 0 || n_tail > a.tail_cap || (has_cur && n_tail >= a.tail_cap);
  if (bad && threadIdx.x == 0) atomicOr(&g_draft_status, VC_DEV_CAPACITY);
  if (bad || n_tok == 0) {
    for (int h = threadIdx.x; h < G; h += kConsumers)
      a.part_lse[static_cast<size_t>(b * a.Hq + kvh * G + h) * a.max_parts + slot] = -INFINITY;
    arrive_and_combine<G, D>(a, flag, bh, n_c + 1, kConsumers);
    return;
  }
  float m[G], l[G], o[G][CPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) o[h][j] = 0.0f;
  }
  float qv[G][CPL];
  for (int t0 = warp; t0 < n_tok; t0 += kWarps * U) {
    uint32_t kr[U][CPL / 2], vr[U][CPL / 2];   // bf16 pairs of the lane's channels
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = t0 + u * kWarps;
      const uint16_t* kp = t < n_tail ? a.tail_k + tbase + static_cast<size_t>(t) * D : a.k_cur + static_cast<size_t>(bh) * D;
      const uint16_t* vp = t < n_tail ? a.tail_v + tbase + static_cast<size_t>(t) * D : a.v_cur + static_cast<size_t>(bh) * D;
#pragma unroll
      for (int j = 0; j < CPL / 2; ++j) {
        kr[u][j] = t < n_tok ? reinterpret_cast<const uint32_t*>(kp + CPL * lane)[j] : 0u;
        vr[u][j] = t < n_tok ? reinterpret_cast<const uint32_t*>(vp + CPL * lane)[j] : 0u;
      }
    }
    if (t0 == warp) {                          // the queries, once the first rows are in flight
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const uint32_t* qp = reinterpret_cast<const uint32_t*>(a.q + (static_cast<size_t>(b) * a.Hq + kvh * G + h) * D + CPL * lane);
#pragma unroll
        for (int j = 0; j < CPL / 2; ++j) {
          const uint32_t x = qp[j];
          qv[h][2 * j] = __uint_as_float(x << 16) * a.scale_log2;
          qv[h][2 * j + 1] = __uint_as_float(x & 0xFFFF0000u) * a.scale_log2;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (t0 + u * kWarps >= n_tok) break;     // uniform over the warp
      float kf[CPL], vf[CPL];
#pragma unroll
      for (int j = 0; j < CPL / 2; ++j) {
        kf[2 * j] = __uint_as_float(kr[u][j] << 16);
        kf[2 * j + 1] = __uint_as_float(kr[u][j] & 0xFFFF0000u);
        vf[2 * j] = __uint_as_float(vr[u][j] << 16);
        vf[2 * j + 1] = __uint_as_float(vr[u][j] & 0xFFFF0000u);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < CPL; ++j) s = fmaf(qv[h][j], kf[j], s);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        const float mn = fmaxf(m[h], s);
        const float alpha = exp2f(m[h] - mn);  // m = -inf at the first token: 0
        const float p = exp2f(s - mn);
        l[h] = fmaf(l[h], alpha, p);
#pragma unroll
        for (int j = 0; j < CPL; ++j) o[h][j] = fmaf(o[h][j], alpha, p * vf[j]);
        m[h] = mn;
      }
    }
  }
  // the warp's (max, sum, output) per head (a warp without tokens leaves max = -inf)
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) red[(warp * G + h) * D + CPL * lane + j] = o[h][j];
    if (lane == 0) {
      wstat[(warp * 8 + h) * 2] = m[h];
      wstat[(warp * 8 + h) * 2 + 1] = l[h];
    }
  }
  vc_bar_sync(1, kConsumers);
  merge_partials<D, BITS, G>(a, smem, bh, slot);
  if (has_cur) {                               // keep the current token for the next steps
    for (int i = threadIdx.x; i < D / 8; i += kConsumers) {
      reinterpret_cast<uint4*>(a.tail_k + tbase + static_cast<size_t>(n_tail) * D)[i] =
          reinterpret_cast<const uint4*>(a.k_cur + static_cast<size_t>(bh) * D)[i];
      reinterpret_cast<uint4*>(a.tail_v + tbase + static_cast<size_t>(n_tail) * D)[i] =
          reinterpret_cast<const uint4*>(a.v_cur + static_cast<size_t>(bh) * D)[i];
    }
  }
  arrive_and_combine<G, D>(a, flag, bh, n_c + 1, kConsumers);
}

// ------------------------------------------------------------------ stream CTA
// Segments of stream CTA c: consecutive calls walk [range_lo(c), range_lo(c+1)).
struct Segment {
  int bh, gs, n_valid, n_st;
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
  sg.n_st = (sg.n_valid + kWarps - 1) / kWarps;
  return true;
}

// Producer warp (lane 0): fills the ring stage by stage, across segments,
// each stage once all consumer warps released its previous use.  It stops
// issuing once the CTA's abort flag is up, and before returning waits (bounded)
// for the copies of its last stages, so that no copy lands after the CTA ends.
template <int D, int BITS, int G>
__device__ void produce(const DraftArgs& a, uint8_t* smem, int c, uint64_t* full, uint64_t* empty,
                        volatile uint32_t* abort) {
  using P = Plan<D, BITS, G>;
  int buf = 0;                                  // ring position of the next stage use
  uint32_t phase = 0;                           // completed wraps of the ring, mod 2
  bool wrapped = false;                         // every buffer used at least once
  uint32_t in_flight = 0;                       // bit i: buffer i holds an issued copy not yet drained
  uint32_t in_phase = 0;                        // bit i: its phase
  const long long hi = range_lo(c + 1, a);
  long long pos = range_lo(c, a);
  Segment sg;
  bool over;
  bool stop = false;
  while (!stop && next_segment(a, pos, hi, sg, over)) {
    for (int s = 0; s < sg.n_st; ++s) {
      // the previous use of `buf` (one wrap earlier) must have been released
      if ((wrapped && !vc_mbar_wait_or_abort(empty + buf, phase ^ 1u, abort, a.wait_cycles)) || *abort != 0u) {
        stop = true;
        break;
      }
      // (test only) the first stage withheld: its consumers' waits run out
      if (!(a.withhold_first && !wrapped && buf == 0)) {
        issue_stage<D, BITS, G>(a, smem + buf * P::stage, full + buf, sg.bh, sg.gs + s * kWarps,
                                min(kWarps, sg.n_valid - s * kWarps));
        in_flight |= 1u << buf;
        in_phase = (in_phase & ~(1u << buf)) | (phase << buf);
      } else {
        in_flight &= ~(1u << buf);
      }
      if (++buf == P::NS) {
        buf = 0;
        phase ^= 1u;
        wrapped = true;
      }
    }
  }
  // the copies of the last use of every buffer have landed (consumed ones return at once)
  for (int i = 0; i < P::NS; ++i)
    if (in_flight & (1u << i)) vc_mbar_wait_bounded(full + i, (in_phase >> i) & 1u, a.wait_cycles);
}

template <int D, int BITS, int G>
__device__ void stream_cta(const DraftArgs& a, uint8_t* smem, int c) {
  using P = Plan<D, BITS, G>;
  constexpr int NS = P::NS, KS = D / 16, NCG = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P::off_bar);
  uint64_t* empty = full + NS;
  unsigned int* flag = reinterpret_cast<unsigned int*>(smem + P::off_flag);
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(flag + 1);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      vc_mbar_init(full + i, 1);
      vc_mbar_init(empty + i, kWarps);
    }
    *abort = 0u;
    vc_fence_mbar_init();
  }
  __syncthreads();
  if (warp == kWarps) {                         // producer warp
    if (lane == 0) produce<D, BITS, G>(a, smem, c, full, empty, abort);
    return;
  }
  // the first segment from packed_len (packed-cache data); a chained call:
  // everything past the wait (queries, tails, partials, counters, output)
  // waits for the previous grid on the stream; only packed-cache reads run
  // ahead of it
  const long long hi = range_lo(c + 1, a);
  long long pos = range_lo(c, a);
  Segment sg;
  bool over;
  bool more = next_segment(a, pos, hi, sg, over);
  grid_dependency_wait();
  // the bf16 tails of the slices assigned to this CTA, first: the ring is
  // already filled, and a tail partial arrives long before the stream
  // partials of its slice and leaves the merge to the last of them
  {
    const long long nbh = static_cast<long long>(a.B) * a.Hkv;
    for (long long bh = tail_lo(c, a.n_stream, nbh); bh < tail_lo(c + 1, a.n_stream, nbh); ++bh)
      tail_part<D, BITS, G>(a, smem, static_cast<int>(bh));
    vc_bar_sync(1, kConsumers);                             // red / flag reused by the segments
  }
  // lane constants: correction columns (gid = 2g: the zeros of channel group
  // g, over the weights' factor 2^(kFold - C(r)); odd gid: zero columns; a V
  // meta row pair holds the scales first, then the zeros)
  const bool zc = gid < 2 * NCG && (gid & 1) == 0;
  const uint32_t zcol_mul0 = zc ? pow2_h2(pos_col<BITS>(0) - kFold) : 0u;
  const uint32_t zcol_mul1 = zc ? pow2_h2(pos_col<BITS>(1) - kFold) : 0u;
  const int zcol_off = zc ? 32 * (gid + 1) : 0;
  const float cs_code = a.scale_log2 * exp2f(static_cast<float>(24 - kFold));
  int buf = 0;                                  // ring position and phase of the next stage use
  uint32_t phase = 0;
  for (; more; more = next_segment(a, pos, hi, sg, over)) {
    if (over && threadIdx.x == 0) atomicOr(&g_draft_status, VC_DEV_CAPACITY);
    const int b = sg.bh / a.Hkv, kvh = sg.bh % a.Hkv;
    int first, last;
    ctas_of(sg.bh, a, first, last);
    // query fragments of head gid times 2^(kFold - p) of their k-step and register:
    // channels (D/4) tig + 4ks + 2r + {0, 1} (G = 4: lanes gid and gid + 4 both hold head gid & 3)
    uint32_t qf[KS][2];
    {
      constexpr bool kT = G == 4;                // heads repeated in columns 4-7
      const int head = kT ? (gid & 3) : (gid < G ? gid : 0);
      const uint16_t* qrow = a.q + (static_cast<size_t>(b) * a.Hq + kvh * G + head) * D + (D / 4) * tig;
      const float on = (kT || gid < G) ? 1.0f : 0.0f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint2 raw = *reinterpret_cast<const uint2*>(qrow + 4 * ks);
        const float q0 = vc_bf16_to_f32(static_cast<uint16_t>(raw.x)), q1 = vc_bf16_to_f32(static_cast<uint16_t>(raw.x >> 16));
        const float q2 = vc_bf16_to_f32(static_cast<uint16_t>(raw.y)), q3 = vc_bf16_to_f32(static_cast<uint16_t>(raw.y >> 16));
        const float f0 = on * exp2f(static_cast<float>(kFold - pos_key<BITS>(ks, 0)));
        const float f1 = on * exp2f(static_cast<float>(kFold - pos_key<BITS>(ks, 1)));
        qf[ks][0] = h2u(__floats2half2_rn(q0 * f0, q1 * f0));
        qf[ks][1] = h2u(__floats2half2_rn(q2 * f1, q3 * f1));
      }
    }
    WarpState<D> st;
    init_state(st);
    for (int s = 0; s < sg.n_st; ++s) {
      const bool ok = __all_sync(0xffffffffu, vc_mbar_wait_or_abort(full + buf, phase, abort, a.wait_cycles));
      if (ok && s * kWarps + warp < sg.n_valid) {
        const uint8_t* base = smem + buf * P::stage;
        const uint32_t* kc_g = reinterpret_cast<const uint32_t*>(base + warp * P::codes);
        const uint16_t* ksz_g = reinterpret_cast<const uint16_t*>(base + P::kc + warp * P::meta);
        const uint32_t* vc_g = reinterpret_cast<const uint32_t*>(base + P::kc + P::mt + warp * P::codes);
        const uint16_t* vsz_g = reinterpret_cast<const uint16_t*>(base + 2 * P::kc + P::mt + warp * P::meta);
        group_mma<D, BITS, G>(kc_g, ksz_g, vc_g, vsz_g, qf, zcol_mul0, zcol_mul1, zcol_off, a.scale_log2, cs_code,
                              st, lane);
      }
      __syncwarp();
      if (lane == 0) vc_mbar_arrive(empty + buf);          // this warp is done with the stage
      if (++buf == NS) {
        buf = 0;
        phase ^= 1u;
      }
    }
    // every consumer thread takes the same branch: the OR of the abort flag
    if (vc_bar_red_or(1, kConsumers, *abort != 0u)) {
      if (threadIdx.x == 0) atomicOr(&g_draft_status, VC_DEV_BARRIER_TIMEOUT);
      return;                                               // outputs of this call are invalid
    }
    write_partial<D, BITS, G>(a, smem, sg.bh, c - first, st);
    arrive_and_combine<G, D>(a, flag, sg.bh, last - first + 2, kConsumers);
    vc_bar_sync(1, kConsumers);                             // red / flag reused by the next segment
  }
}

template <int D, int BITS, int G, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) draft_kernel(const __grid_constant__ DraftArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int c = blockIdx.x;
  grid_launch_dependents();
  if (a.n_stream > 0) {
    stream_cta<D, BITS, G>(a, smem, c);
  } else if ((threadIdx.x >> 5) < kWarps) {     // no packed groups: tail CTA c takes slices c, c + n_cta, ...
    grid_dependency_wait();                     // the tail rows come from earlier calls
    for (int bh = c; bh < a.B * a.Hkv; bh += a.n_cta) tail_part<D, BITS, G>(a, smem, bh);
  }
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

// One CTA of kThreads (11 consumer warps + the producer) per SM: the warps keep
// the output accumulators and the query fragments in registers.
template <int G>
struct MinBlocks {
  static constexpr int value = 1;
};

struct LaunchPlan {
  int n_stream = 0, n_cta = 0, max_parts = 1;
  long long total = 0;
  size_t smem = 0;
  std::vector<int> lo;                          // n_stream + 1 range starts
};

// Cost-balanced stream-K partition of the slice-major groups [0, total)
// (slice boundaries every NG groups) over n CTAs.  A CTA's cost is its
// groups, plus `sw` per slice boundary strictly inside its range, plus `tl`
// per bf16 tail it runs.  Each CTA in turn takes the longest range whose
// cost stays within T, but at least `min_range` groups (so that a slice
// meets a bounded number of CTAs); T is the smallest budget that covers
// every group, by bisection.
struct Partition {
  long long total, NG, sw, tl;
  int n;
  long long nbh, min_range;
  long long crossings(long long p, long long e) const { return e > p + 1 ? (e - 1) / NG - p / NG : 0; }
  long long end_of(int c, long long p, long long T) const {
    long long budget = T - tl * (tail_lo(c + 1, n, nbh) - tail_lo(c, n, nbh));
    if (budget < 1) budget = 1;
    long long best = std::min(total, p + min_range);
    for (long long k = 0;; ++k) {               // ends between boundaries, crossing at most k
      const long long e = std::min(total, p + budget - sw * k);
      if (e <= p) break;
      if (crossings(p, e) <= k) {
        best = std::max(best, e);
        break;
      }
    }
    for (long long j = 1;; ++j) {               // ends on the j-th boundary after p
      const long long b = (p / NG + j) * NG;
      if (b > total || b - p + sw * (j - 1) > budget) break;
      best = std::max(best, b);
    }
    return best;
  }
  bool covers(long long T) const {
    long long p = 0;
    for (int c = 0; c < n && p < total; ++c) p = end_of(c, p, T);
    return p >= total;
  }
  void fill(std::vector<int>& lo) const {
    long long T_hi = std::max<long long>(1, (total + n - 1) / n);
    while (!covers(T_hi)) T_hi *= 2;
    long long T_lo = 0;                         // not covering
    while (T_hi - T_lo > 1) {
      const long long m = T_lo + (T_hi - T_lo) / 2;
      if (covers(m)) T_hi = m; else T_lo = m;
    }
    lo.assign(static_cast<size_t>(n) + 1, static_cast<int>(total));
    long long p = 0;
    for (int c = 0; c < n; ++c) {
      lo[c] = static_cast<int>(p);
      if (p < total) p = end_of(c, p, T_hi);
    }
  }
};

// The stream CTAs, partition table and partial slots of a launch over
// `slices` slices of NGmax groups, with `slots` launch slots (occupancy x
// SMs); host only.  group_bytes: the packed bytes of one group (K and V
// codes, K and V scale/zero), which scale the partition's charges.
vc_status_t partition_plan(long long slices, long long NGmax, long long slots, long long group_bytes, LaunchPlan* lp) {
  lp->total = slices * NGmax;
  if (lp->total > INT_MAX) VC_FAIL(VC_ERR_UNSUPPORTED, "B * Hkv * max_packed / 32 = %lld groups exceeds 2^31 - 1", lp->total);
  const long long n_max = std::min<long long>(slots, kMaxStream);
  long long n = n_max;
  const long long by_work = lp->total / kWarps;                 // at least one stage per CTA
  if (n > by_work) n = by_work;
  if (n < 1 && lp->total > 0) n = 1;
  lp->n_stream = static_cast<int>(lp->total > 0 ? n : 0);
  if (lp->n_stream == 0) {                                      // tail CTAs alone
    lp->n_cta = static_cast<int>(std::min(slices, slots));
    lp->max_parts = 1;
    lp->lo.assign(1, 0);
    return VC_OK;
  }
  lp->n_cta = lp->n_stream;
  // partial slots of a slice: at most `stream_parts` stream CTAs, a bound set
  // by the device and B * Hkv alone (so that a workspace sized for one
  // max_packed serves every max_packed), then the tail.  Each range inside a
  // slice holds >= min_range groups, so at most stream_parts - 2 of them fit.
  const long long stream_parts = std::min(n_max, 2 * ((n_max + slices - 1) / slices) + 2);
  const long long min_range = stream_parts >= n ? 1 : (NGmax + stream_parts - 3) / (stream_parts - 2);
  lp->max_parts = static_cast<int>(stream_parts) + 1;
  const Partition part{lp->total, NGmax, kSwitchGroups * kRefGroupBytes / group_bytes,
                       kTailGroups * kRefGroupBytes / group_bytes, lp->n_stream, slices, min_range};
  part.fill(lp->lo);
  for (long long bh = 0; bh < slices; ++bh) {
    const int first = cta_at(bh * NGmax, lp->lo.data(), lp->n_stream);
    const int last = cta_at(bh * NGmax + NGmax - 1, lp->lo.data(), lp->n_stream);
    if (last - first + 2 > lp->max_parts)
      VC_FAIL(VC_ERR_UNSUPPORTED, "partition: slice %lld meets %d CTAs (bound %d)", bh, last - first + 1,
              lp->max_parts - 1);
  }
  return VC_OK;
}

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
  lp->smem = P::total;
  return partition_plan(static_cast<long long>(s->B) * s->Hkv, max_packed / kGroup, static_cast<long long>(occ) * sms,
                        2 * static_cast<long long>(P::codes + P::meta), lp);
}

// Plans by (device, shape, max_packed): the partition costs a bisection, and
// the draft steps of a decode loop repeat a handful of shapes.
struct PlanKey {
  int dev, d, bits, G, B, Hkv, max_packed;
  bool operator==(const PlanKey& o) const {
    return dev == o.dev && d == o.d && bits == o.bits && G == o.G && B == o.B && Hkv == o.Hkv && max_packed == o.max_packed;
  }
};
constexpr int kPlanCache = 16;
std::mutex g_plan_mu;
PlanKey g_plan_key[kPlanCache];
LaunchPlan g_plan_val[kPlanCache];
int g_plan_n = 0, g_plan_next = 0;

vc_status_t plan_uncached(const vc_shape_t* s, int max_packed, LaunchPlan* lp);

vc_status_t plan(const vc_shape_t* s, int max_packed, LaunchPlan* lp) {
  int dev = 0;
  VC_CUDA_CHECK(cudaGetDevice(&dev));
  const PlanKey key{dev, s->d, s->bits, s->Hq / s->Hkv, s->B, s->Hkv, max_packed};
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    for (int i = 0; i < g_plan_n; ++i)
      if (g_plan_key[i] == key) {
        *lp = g_plan_val[i];
        return VC_OK;
      }
  }
  const vc_status_t st = plan_uncached(s, max_packed, lp);
  if (st != VC_OK) return st;
  std::lock_guard<std::mutex> lock(g_plan_mu);
  g_plan_key[g_plan_next] = key;
  g_plan_val[g_plan_next] = *lp;
  g_plan_next = (g_plan_next + 1) % kPlanCache;
  g_plan_n = std::min(g_plan_n + 1, kPlanCache);
  return VC_OK;
}

vc_status_t plan_uncached(const vc_shape_t* s, int max_packed, LaunchPlan* lp) {
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

// chained: launched with programmatic stream serialisation, so that it may
// start while the previous kernel on the stream (a draft call) finishes.
template <int D, int BITS, int G>
vc_status_t launch_t(const DraftArgs& a, const LaunchPlan& lp, cudaStream_t cs, bool chained) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(lp.n_cta));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = lp.smem;
  cfg.stream = cs;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = chained ? 1 : 0;
  VC_CUDA_CHECK(cudaLaunchKernelEx(&cfg, draft_kernel<D, BITS, G, MinBlocks<G>::value>, a));
  VC_LAUNCH_CHECK("draft_kernel");
  return VC_OK;
}

vc_status_t launch(const vc_shape_t* s, const DraftArgs& a, const LaunchPlan& lp, cudaStream_t cs, bool chained) {
  const int G = s->Hq / s->Hkv;
#define VC_L(D_, B_, G_) \
  if (s->d == D_ && s->bits == B_ && G == G_) return launch_t<D_, B_, G_>(a, lp, cs, chained);
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
                                     void* workspace, size_t workspace_bytes, uint32_t flags, vc_stream_t stream) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE((flags & ~VC_DRAFT_CHAINED) == 0u, "unknown flags 0x%x", flags);
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
  a.n_cta = lp.n_cta;
  a.total = lp.total;
  a.max_parts = lp.max_parts;
  a.scale_log2 = s->softmax_scale * kLog2e;
  a.wait_cycles = g_wait_cycles;
  a.withhold_first = g_withhold_first;
  for (int c = 0; c <= lp.n_stream; ++c) a.lo_tab[c] = lp.lo[c];
  const size_t rows = static_cast<size_t>(s->B) * s->Hq * lp.max_parts;
  char* ws = static_cast<char*>(workspace);
  a.part_o = reinterpret_cast<float*>(ws);
  size_t off = (rows * s->d * sizeof(float) + 255) & ~size_t(255);
  a.part_lse = reinterpret_cast<float*>(ws + off);
  off += (rows * sizeof(float) + 255) & ~size_t(255);
  a.counter = reinterpret_cast<unsigned int*>(ws + off);
  a.out = out;
  return launch(s, a, lp, reinterpret_cast<cudaStream_t>(stream), (flags & VC_DRAFT_CHAINED) != 0u);
}

extern "C" vc_status_t vc_draft_attn_partition(const vc_shape_t* s, int32_t max_packed, int32_t slots,
                                               int32_t* n_stream, int32_t* lo, int32_t lo_len, int32_t* max_parts) {
  vc_status_t st = check(s);
  if (st != VC_OK) return st;
  VC_REQUIRE(n_stream && lo && max_parts, "NULL pointer");
  VC_REQUIRE(max_packed >= 0 && max_packed % kGroup == 0, "max_packed must be a non-negative multiple of 32");
  VC_REQUIRE(slots >= 1, "slots must be >= 1");
  LaunchPlan lp;
  const long long group_bytes = 8LL * s->d * (s->bits + 1);    // K and V codes, K and V scale/zero
  if ((st = partition_plan(static_cast<long long>(s->B) * s->Hkv, max_packed / kGroup, slots, group_bytes, &lp)) != VC_OK)
    return st;
  VC_REQUIRE(lo_len >= lp.n_stream + 1, "lo holds %d entries, the partition needs %d", lo_len, lp.n_stream + 1);
  for (int c = 0; c <= lp.n_stream; ++c) lo[c] = lp.lo[c];
  *n_stream = lp.n_stream;
  *max_parts = lp.max_parts;
  return VC_OK;
}

extern "C" vc_status_t vc_draft_attn_test_hooks(int64_t wait_cycles, int32_t withhold_first_stage) {
  VC_REQUIRE(wait_cycles == 0 || wait_cycles >= 1000, "wait_cycles must be 0 (default) or >= 1000");
  VC_REQUIRE(withhold_first_stage == 0 || withhold_first_stage == 1, "withhold_first_stage must be 0 or 1");
  g_wait_cycles = wait_cycles == 0 ? kWaitCycles : wait_cycles;
  g_withhold_first = withhold_first_stage;
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
