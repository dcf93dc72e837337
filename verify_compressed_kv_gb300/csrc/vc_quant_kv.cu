// libvc_quant_kv: the draft-cache compressors behind VeriCache's uniform
// compressor interface (gist.science/paper/2605.17613, Technical Summary,
// Architecture Support: token-dropping and quantisation methods, e.g. KIVI
// and SnapKV, plug in without touching scheduling or verification).
//
//   * KIVI-style quantiser: int2/int4/int8 codes, keys per channel over 32 tokens,
//     values per token over 32 channels, fp16 scale/zero from min/max,
//     round-half-even.  pack (prefill), append (commit of accepted tokens +
//     packing of full tail groups), unpack (tests).
//   * SnapKV-style token dropping: score (attention mass from the last n_obs
//     prompt queries, causal), select (7-wide max-pool, top-k + last tokens,
//     ascending), gather.
//
// The quantiser's arithmetic is the exact fp32 sequence of the recipe
// (separate correctly rounded subtract and divide, rintf, fp16 RNE), so the
// codes are reproducible bit for bit.  Packed layout: include/vc.h.
#include <cfloat>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "vc_internal.h"

namespace {

__device__ uint32_t g_quant_status = 0;

constexpr int kGroup = 32;

// ------------------------------------------------------------------ quantiser

// ------------------------------------------------------------------ packed layout
// Field rules of the packed words (the library's format; include/vc.h): per
// group, 32 lanes x d*b/32 words; word w of lane L at (w/4)*128 + 4L + w%4.
// b = 2: slot (u, r, e) starts at bit 16e + 4u + 2(1 - r);
// b = 4: slot (u, e) starts at 16e + 4u; b = 8: at 16e + 8u.  No field crosses bit 31.
__device__ __forceinline__ int field_pos(int bits, int u, int r, int e) {
  return bits == 2 ? (16 * e + 4 * u + 2 * (1 - r)) : (16 * e + bits * u);
}

// Word `idx` of a group's K codes (V codes when IS_V) from a code tile
// codes[t * ld + c].  K: lane L = 4a + c holds tokens 4a + j, channels
// (d/4) c + 4k + 2r + e, fragment i = j*(d/16) + k.  V: tokens 8c + 4e + 2s + r,
// channels 8n + a, fragment i = s*(d/8) + n.  b = 2: word i/4, u = i%4;
// b = 4, 8: i2 = 2i + r, SPW = 16/b slots per word, word i2/SPW, u = i2%SPW.
template <int BITS, bool IS_V, int D>
__device__ __forceinline__ uint32_t build_word(const uint8_t* codes, int ld, int idx) {
  const int L = (idx % 128) / 4, w = (idx / 128) * 4 + idx % 4;
  const int a = L / 4, c = L % 4;
  constexpr int per = IS_V ? D / 8 : D / 16;      // fragments per j (K) or per s (V)
  constexpr int SPW = BITS == 2 ? 4 : 16 / BITS;   // slots per word
  uint32_t word = 0;
#pragma unroll
  for (int u = 0; u < SPW; ++u)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      int i;
      if (BITS == 2) {
        i = 4 * w + u;
      } else {
        if ((u & 1) != r) continue;               // b = 4, 8: slot u carries r = u % 2 (SPW even)
        i = (SPW * w + u) >> 1;
      }
      const int hi = i / per, lo = i % per;         // (j, k) for K, (s, n) for V
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        int t, ch;
        if (IS_V) {
          t = 8 * c + 4 * e + 2 * hi + r;
          ch = 8 * lo + a;
        } else {
          t = 4 * a + hi;
          ch = (D / 4) * c + 4 * lo + 2 * r + e;
        }
        const uint32_t code = codes[t * ld + ch];
        word += code << field_pos(BITS, u, r, e);      // disjoint fields: + == |
      }
    }
  return word;
}

// Entry of a V meta row (32 entries, one per token) that holds token t:
// entry 8c + 4s + 2r + e holds token 8c + 4e + 2s + r.
__device__ __forceinline__ int vmeta_entry(int t) {
  return (t & ~7) | (((t >> 1) & 1) << 2) | ((t & 1) << 1) | ((t >> 2) & 1);
}

// Quantisation parameters of one group (KIVI recipe): scale s = fp16((max - min) / qmax),
// zero z = fp16(min), both applied in fp32.
struct QParams {
  float s, z;
  float y;        // RN(1/s) for a fast group (see qparams), else 0: every code exact
  uint16_t s16, z16;
};

// A group is fast when s > 0 and finite, z finite, and every q = RN(RN(x - z) y)
// of its elements lies in (-1/4, qmax + 1/4): q is monotone in x (each step rounds
// monotonically and y > 0), so the group's min and max bound it.  Then
// rint(q) is already in [0, qmax] and no element needs the clamp.
template <int QMAX>
__device__ __forceinline__ QParams qparams(float mn, float mx) {
  QParams p;
  p.s16 = vc_f32_to_f16_rn(__fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(QMAX)));
  p.z16 = vc_f32_to_f16_rn(mn);
  p.s = vc_f16_to_f32(p.s16);
  p.z = vc_f16_to_f32(p.z16);
  p.y = 0.0f;
  if (p.s > 0.0f && isfinite(p.s) && isfinite(p.z)) {
    const float y = __frcp_rn(p.s);
    const float qlo = __fmul_rn(__fsub_rn(mn, p.z), y), qhi = __fmul_rn(__fsub_rn(mx, p.z), y);
    if (qlo > -0.25f && qhi < static_cast<float>(QMAX) + 0.25f) p.y = y;
  }
  return p;
}

// QParams travel between lanes as (s16 | z16 << 16, y).
__device__ __forceinline__ uint32_t share_sz(const QParams& p) {
  return p.s16 | (static_cast<uint32_t>(p.z16) << 16);
}
__device__ __forceinline__ QParams unshare(uint32_t sz, float y) {
  QParams p;
  p.s16 = static_cast<uint16_t>(sz & 0xFFFFu);
  p.z16 = static_cast<uint16_t>(sz >> 16);
  p.s = vc_f16_to_f32(p.s16);
  p.z = vc_f16_to_f32(p.z16);
  p.y = y;
  return p;
}

// The recipe's code: clamp(rint((x - z) / s), 0, qmax), correctly rounded subtract
// and divide; 0 when s = 0.
template <int QMAX>
__device__ __forceinline__ uint32_t code_exact(float x, float s, float z) {
  if (s == 0.0f) return 0u;
  float r = rintf(__fdiv_rn(__fsub_rn(x, z), s));
  r = fminf(fmaxf(r, 0.0f), static_cast<float>(QMAX));
  return static_cast<uint32_t>(r);
}

// Two fp32 values in one 64-bit register; add / sub / mul act on both lanes with
// IEEE round-to-nearest (sm_100 family f32x2 instructions).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float f2lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Paired bf16 min / max (a NaN operand yields the other) and byte permute.
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Codes are decided exactly unless c = rint-candidate lies within this distance of
// a half-integer.  A code depends only on where q sits against 1/2 .. qmax - 1/2,
// so only |q| < 2^b matters; there q = RN((x - z) y) is within |a/s| (2^-23 + 2^-47)
// of a/s (a = x - z, y = RN(1/s)) and RN(a/s) within |a/s| 2^-24, so the two are
// less than 2^(b-22) apart and round to the same integer outside the window.
template <int QMAX>
__device__ __forceinline__ constexpr float tie_window() { return static_cast<float>(QMAX + 1) * 0x1p-21f; }

// The codes of two elements of fast groups (y > 0) without a division.  2^23 + q
// rounds q in (-1/4, 2^22) to an integer, ties to even, in the low bits, and
// q - rint(q) is exact.  A near-tie (or a NaN) sets `tie`; the caller redoes the
// pair's elements with code_recheck.  Returns code(x.lo) | code(x.hi) << 8 in the
// low half (the high half is unspecified).
template <int QMAX>
__device__ __forceinline__ uint32_t code_pair(uint64_t x, uint64_t z, uint64_t y, bool& tie) {
  const uint64_t big = f2(0x1p23f, 0x1p23f);
  const uint64_t q = f2_mul(f2_sub(x, z), y);
  const uint64_t m = f2_add(q, big);
  const uint64_t frac = f2_sub(q, f2_sub(m, big));
  tie |= !(fabsf(f2lo(frac)) < 0.5f - tie_window<QMAX>()) | !(fabsf(f2hi(frac)) < 0.5f - tie_window<QMAX>());
  return prmt(static_cast<uint32_t>(m), static_cast<uint32_t>(m >> 32), 0x0040u);
}

// One element's exact code by the cheapest sure route: the reciprocal product when
// its group is fast and it is not near a tie (clamped, so it also serves groups
// whose range test failed), else the division.
template <int QMAX>
__device__ __forceinline__ uint32_t code_recheck(float x, float s, float z, float y) {
  if (y > 0.0f) {
    const float q = __fmul_rn(__fsub_rn(x, z), y);
    const float c = fminf(fmaxf(q, 0.0f), static_cast<float>(QMAX));
    const float r = __fsub_rn(__fadd_rn(c, 0x1p23f), 0x1p23f);
    if (fabsf(__fsub_rn(c, r)) < 0.5f - tie_window<QMAX>()) return static_cast<uint32_t>(r);
  }
  return code_exact<QMAX>(x, s, z);
}

// Codes of one thread's key elements (channels 2cp, 2cp + 1, tokens t0 .. t0 + TPT
// - 1) re-read from global memory: the rare path after code_pair flagged one, or
// for a group that is not fast.
template <int QMAX, int D, int TPT>
__device__ __noinline__ void k_codes_exact(const uint16_t* Kg, int t0, int cp, QParams p0, QParams p1,
                                           uint8_t* kcodes) {
  for (int j = 0; j < TPT; ++j) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(Kg + (t0 + j) * D + 2 * cp);
    const uint32_t c = code_recheck<QMAX>(bf16_lo(w), p0.s, p0.z, p0.y) |
                       (code_recheck<QMAX>(bf16_hi(w), p1.s, p1.z, p1.y) << 8);
    *reinterpret_cast<uint16_t*>(kcodes + (t0 + j) * (D + 4) + 2 * cp) = static_cast<uint16_t>(c);
  }
}

// Codes of 4 value elements (one lane's piece of a token row), the same way.
template <int QMAX>
__device__ __noinline__ uint32_t v_codes_exact(uint2 w, QParams p) {
  return code_recheck<QMAX>(bf16_lo(w.x), p.s, p.z, p.y) | (code_recheck<QMAX>(bf16_hi(w.x), p.s, p.z, p.y) << 8) |
         (code_recheck<QMAX>(bf16_lo(w.y), p.s, p.z, p.y) << 16) |
         (code_recheck<QMAX>(bf16_hi(w.y), p.s, p.z, p.y) << 24);
}

constexpr int kPackThreads = 128;

// Quantise one 32-token group: Kg, Vg point at its 32 rows of d bf16 (row stride
// D) in global memory.  Writes the group's words and metadata into group `g` of the
// (b, h) slice of the packed arrays.  All kPackThreads threads of the CTA call it;
// codes_s is 2 x [32][D + 4] bytes of shared memory.
//   keys:   thread = (channel pair, slice of 32/TQ tokens); the TQ slices of a pair
//           sit in one warp and combine min/max by shuffles.
//   values: a lane holds 4 channels of one token row; 8 lanes = one 32-channel group.
// All loads of the group are issued before the first use.  Min and max are taken
// on the bf16 inputs themselves (exact).
template <int BITS, int D>
__device__ __forceinline__ void quantize_group(const uint16_t* Kg, const uint16_t* Vg, uint8_t* codes_s, int g,
                                               uint32_t* kc, uint16_t* ksz, uint32_t* vc, uint16_t* vsz) {
  static_assert(D == 64 || D == 128, "head dim");
  constexpr int QMAX = (1 << BITS) - 1;
  constexpr int CLD = D + 4;                         // code tile row stride (bytes)
  constexpr int TQ = 2 * kPackThreads / D;           // token slices per channel pair
  constexpr int TPT = kGroup / TQ;                   // tokens per slice
  constexpr int PPW = 32 / TQ;                       // channel pairs per warp
  constexpr int LPR = D / 4;                         // lanes per V row
  constexpr int NPI = kGroup * LPR / kPackThreads;   // V row pieces per thread
  constexpr int NC = D / kGroup;                     // V channel groups per token
  uint8_t* kcodes = codes_s;
  uint8_t* vcodes = codes_s + kGroup * CLD;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cp = warp * PPW + lane % PPW, sl = lane / PPW;

  uint32_t kx[TPT];
#pragma unroll
  for (int j = 0; j < TPT; ++j) kx[j] = *reinterpret_cast<const uint32_t*>(Kg + (sl * TPT + j) * D + 2 * cp);
  uint2 vx[NPI];
#pragma unroll
  for (int it = 0; it < NPI; ++it) {
    const int pi = it * kPackThreads + tid;
    vx[it] = *reinterpret_cast<const uint2*>(Vg + (pi / LPR) * D + 4 * (pi % LPR));
  }

  // ---- keys: channels 2cp, 2cp + 1 over the group's 32 tokens
  {
    uint32_t kmn = kx[0], kmx = kx[0];
#pragma unroll
    for (int j = 1; j < TPT; ++j) {
      kmn = bmin2(kmn, kx[j]);
      kmx = bmax2(kmx, kx[j]);
    }
#pragma unroll
    for (int o = PPW; o < 32; o <<= 1) {
      kmn = bmin2(kmn, __shfl_xor_sync(0xFFFFFFFFu, kmn, o));
      kmx = bmax2(kmx, __shfl_xor_sync(0xFFFFFFFFu, kmx, o));
    }
    // odd slices derive channel 2cp + 1's parameters, even ones 2cp's; swap across slices
    const bool odd = sl & 1;
    const QParams mine = odd ? qparams<QMAX>(bf16_hi(kmn), bf16_hi(kmx)) : qparams<QMAX>(bf16_lo(kmn), bf16_lo(kmx));
    const QParams other = unshare(__shfl_xor_sync(0xFFFFFFFFu, share_sz(mine), PPW),
                                  __shfl_xor_sync(0xFFFFFFFFu, mine.y, PPW));
    const QParams p0 = odd ? other : mine, p1 = odd ? mine : other;
    if (sl == 0) {                                   // scales row, then zeros row
      uint32_t* m = reinterpret_cast<uint32_t*>(ksz + static_cast<size_t>(g) * 2 * D);
      m[cp] = p0.s16 | (static_cast<uint32_t>(p1.s16) << 16);
      m[D / 2 + cp] = p0.z16 | (static_cast<uint32_t>(p1.z16) << 16);
    }
    bool tie = !(p0.y > 0.0f) | !(p1.y > 0.0f);
    const uint64_t z2 = f2(p0.z, p1.z), y2 = f2(p0.y, p1.y);
#pragma unroll
    for (int j = 0; j < TPT; ++j) {
      const uint32_t c = code_pair<QMAX>(f2(bf16_lo(kx[j]), bf16_hi(kx[j])), z2, y2, tie);
      *reinterpret_cast<uint16_t*>(kcodes + (sl * TPT + j) * CLD + 2 * cp) = static_cast<uint16_t>(c);
    }
    if (tie) k_codes_exact<QMAX, D, TPT>(Kg, sl * TPT, cp, p0, p1, kcodes);
  }
  // ---- values: 4 channels of token t per lane.  Each piece's partial (min, -max)
  // travels as one bf16 pair; the 8 lanes of a 32-channel group reduce-scatter
  // their NPI pairs, so each lane derives the parameters of one (piece, group) and
  // the group's lanes fetch them by shuffle.
  {
    constexpr int LOG_NPI = NPI == 8 ? 3 : 2;
    uint32_t pr[NPI];
#pragma unroll
    for (int it = 0; it < NPI; ++it) {
      const uint32_t a = bmin2(vx[it].x, vx[it].y), b = bmax2(vx[it].x, vx[it].y) ^ 0x80008000u;
      pr[it] = bmin2(prmt(a, b, 0x5410u), prmt(a, b, 0x7632u));     // (min, -max)
    }
    // halving exchanges at lane offsets 4, 2, 1: a lane with the offset bit set keeps
    // the upper half; once one value is left, the remaining stages are all-reduces
#pragma unroll
    for (int st = 0, n = NPI; st < 3; ++st) {
      const int o = 4 >> st;
      const bool up = lane & o;
      if (n > 1) {
        const int half = n / 2;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const uint32_t send = up ? pr[i] : pr[i + half], keep = up ? pr[i + half] : pr[i];
          pr[i] = bmin2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, o));
        }
        n = half;
      } else {
        pr[0] = bmin2(pr[0], __shfl_xor_sync(0xFFFFFFFFu, pr[0], o));
      }
    }
    const int own = (lane & 7) >> (3 - LOG_NPI);     // the piece this lane's parameters belong to
    const QParams po = qparams<QMAX>(bf16_lo(pr[0]), -bf16_hi(pr[0]));
    {
      const int pi = own * kPackThreads + tid, t = pi / LPR, q4 = pi % LPR;
      if (((lane & 7) & ((8 >> LOG_NPI) - 1)) == 0) {
        const size_t m = ((static_cast<size_t>(g) * NC + q4 / 8) * 2) * kGroup + vmeta_entry(t);
        vsz[m] = po.s16;
        vsz[m + kGroup] = po.z16;
      }
    }
    const uint32_t sz_own = share_sz(po);
#pragma unroll
    for (int it = 0; it < NPI; ++it) {
      const int src = (lane & ~7) | (it << (3 - LOG_NPI));
      const QParams p = unshare(__shfl_sync(0xFFFFFFFFu, sz_own, src), __shfl_sync(0xFFFFFFFFu, po.y, src));
      const int pi = it * kPackThreads + tid, t = pi / LPR, q4 = pi % LPR;
      bool tie = !(p.y > 0.0f);
      const uint64_t z2 = f2(p.z, p.z), y2 = f2(p.y, p.y);
      uint32_t packed = prmt(code_pair<QMAX>(f2(bf16_lo(vx[it].x), bf16_hi(vx[it].x)), z2, y2, tie),
                             code_pair<QMAX>(f2(bf16_lo(vx[it].y), bf16_hi(vx[it].y)), z2, y2, tie), 0x5410u);
      if (tie) packed = v_codes_exact<QMAX>(vx[it], p);
      *reinterpret_cast<uint32_t*>(vcodes + t * CLD + 4 * q4) = packed;
    }
  }
  __syncthreads();
  // ---- words: consecutive threads -> consecutive words
  constexpr int n_words = D * BITS;
#pragma unroll
  for (int idx = tid; idx < n_words; idx += kPackThreads) {
    kc[static_cast<size_t>(g) * n_words + idx] = build_word<BITS, false, D>(kcodes, CLD, idx);
    vc[static_cast<size_t>(g) * n_words + idx] = build_word<BITS, true, D>(vcodes, CLD, idx);
  }
  __syncthreads();
}

struct Packed {
  uint32_t* kc;
  uint16_t* ksz;
  uint32_t* vc;
  uint16_t* vsz;
};

// Offsets of (b, h)'s slice in each packed array.
__host__ __device__ inline Packed slice(Packed p, int bh, int T_cap, int d, int bits) {
  const int NG = T_cap / kGroup;
  const int W = d * bits / 32;
  Packed r;
  r.kc = p.kc + static_cast<size_t>(bh) * NG * W * kGroup;
  r.vc = p.vc + static_cast<size_t>(bh) * NG * W * kGroup;
  r.ksz = p.ksz + static_cast<size_t>(bh) * NG * d * 2;
  r.vsz = p.vsz + static_cast<size_t>(bh) * NG * d * 2;
  return r;
}

// grid (T/32, B*Hkv): one 32-token group of one (b, h) per CTA.
template <int BITS, int D>
__global__ void __launch_bounds__(kPackThreads, 8) pack_kernel(const uint16_t* __restrict__ K,
                                                            const uint16_t* __restrict__ V, int T,
                                                            int T_cap, Packed p) {
  __shared__ __align__(16) uint8_t codes_s[2 * kGroup * (D + 4)];
  const int g = blockIdx.x, bh = blockIdx.y;
  const size_t base = (static_cast<size_t>(bh) * T + static_cast<size_t>(g) * kGroup) * D;
  Packed s = slice(p, bh, T_cap, D, BITS);
  quantize_group<BITS, D>(K + base, V + base, codes_s, g, s.kc, s.ksz, s.vc, s.vsz);
}

// append_kernel's shared memory: two bf16 [32][d + 2] staging tiles for the tail
// shift, then the code tiles.
size_t append_smem(int d) { return 2 * kGroup * (d + 2) * sizeof(uint16_t) + 2 * kGroup * (d + 4); }

// The commit of one request's accepted tokens for one KV head (grid (Hkv, B)):
// append rows 0..n of k_new/v_new to the tail, pack whole groups from the
// tail's front, shift the rest down.  Lengths are read here and written by
// append_lengths_kernel afterwards, so no CTA sees another's update.
template <int BITS, int D>
__global__ void __launch_bounds__(kPackThreads) append_kernel(
    const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
    const int32_t* __restrict__ n_acc, int k, int Hkv, uint16_t* tail_k, uint16_t* tail_v,
    const int32_t* tail_len, int tail_cap, Packed p, const int32_t* packed_len, int T_cap) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr int d = D;
  constexpr int ld = d + 2;
  uint16_t* k_s = reinterpret_cast<uint16_t*>(smem);
  uint16_t* v_s = k_s + kGroup * ld;
  uint8_t* codes_s = reinterpret_cast<uint8_t*>(v_s + kGroup * ld);
  const int h = blockIdx.x, b = blockIdx.y;
  const int n = n_acc ? n_acc[b] : k;
  const int len = tail_len[b];
  const int plen = packed_len[b];
  const int add = n + 1;
  if (n < 0 || n > k || len < 0 || len + add > tail_cap) {
    if (threadIdx.x == 0) atomicOr(&g_quant_status, VC_DEV_CAPACITY);
    return;
  }
  const int total = len + add;
  const int n_pack = total / kGroup;
  if (plen + n_pack * kGroup > T_cap) {
    if (threadIdx.x == 0) atomicOr(&g_quant_status, VC_DEV_CAPACITY);
    return;
  }
  const int vec = d / 8;
  const size_t tb = (static_cast<size_t>(b) * Hkv + h) * tail_cap * d;
  // 1. append: tail[b, h, len + r] = new[b, r, h] for r <= n
  for (int i = threadIdx.x; i < add * vec; i += blockDim.x) {
    const int v = i % vec, r = i / vec;
    const size_t src = ((static_cast<size_t>(b) * (k + 1) + r) * Hkv + h) * d + v * 8;
    const size_t dst = tb + static_cast<size_t>(len + r) * d + v * 8;
    *reinterpret_cast<uint4*>(tail_k + dst) = *reinterpret_cast<const uint4*>(k_new + src);
    *reinterpret_cast<uint4*>(tail_v + dst) = *reinterpret_cast<const uint4*>(v_new + src);
  }
  __syncthreads();
  // 2. pack whole groups from the front of the tail
  Packed s = slice(p, b * Hkv + h, T_cap, d, BITS);
  for (int grp = 0; grp < n_pack; ++grp)
    quantize_group<BITS, D>(tail_k + tb + static_cast<size_t>(grp) * kGroup * d,
                            tail_v + tb + static_cast<size_t>(grp) * kGroup * d, codes_s, plen / kGroup + grp, s.kc,
                            s.ksz, s.vc, s.vsz);
  // 3. shift the remaining (total - 32*n_pack < 32) tail tokens to the front
  const int shift = n_pack * kGroup;
  const int rest = total - shift;
  if (shift > 0 && rest > 0) {
    // stage through smem: the source and destination rows may overlap
    for (int i = threadIdx.x; i < rest * vec; i += blockDim.x) {
      const int t = i / vec, v = i % vec;
      const uint4 a = *reinterpret_cast<const uint4*>(tail_k + tb + static_cast<size_t>(shift + t) * d + v * 8);
      const uint4 c = *reinterpret_cast<const uint4*>(tail_v + tb + static_cast<size_t>(shift + t) * d + v * 8);
      uint32_t* ok = reinterpret_cast<uint32_t*>(k_s + t * ld + v * 8);
      uint32_t* ov = reinterpret_cast<uint32_t*>(v_s + t * ld + v * 8);
      ok[0] = a.x; ok[1] = a.y; ok[2] = a.z; ok[3] = a.w;
      ov[0] = c.x; ov[1] = c.y; ov[2] = c.z; ov[3] = c.w;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < rest * vec; i += blockDim.x) {
      const int t = i / vec, v = i % vec;
      const uint32_t* ik = reinterpret_cast<const uint32_t*>(k_s + t * ld + v * 8);
      const uint32_t* iv = reinterpret_cast<const uint32_t*>(v_s + t * ld + v * 8);
      *reinterpret_cast<uint4*>(tail_k + tb + static_cast<size_t>(t) * d + v * 8) = make_uint4(ik[0], ik[1], ik[2], ik[3]);
      *reinterpret_cast<uint4*>(tail_v + tb + static_cast<size_t>(t) * d + v * 8) = make_uint4(iv[0], iv[1], iv[2], iv[3]);
    }
  }
}

// New lengths after append_kernel (same checks, so a rejected request keeps its lengths).
__global__ void append_lengths_kernel(const int32_t* __restrict__ n_acc, int B, int k, int32_t* tail_len,
                                      int tail_cap, int32_t* packed_len, int T_cap) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int n = n_acc ? n_acc[b] : k;
    const int len = tail_len[b], plen = packed_len[b];
    if (n < 0 || n > k || len < 0 || len + n + 1 > tail_cap) continue;
    const int total = len + n + 1;
    const int shift = (total / kGroup) * kGroup;
    if (plen + shift > T_cap) continue;
    tail_len[b] = total - shift;
    packed_len[b] = plen + shift;
  }
}

// Position of code (t, ch) of a group: word index and field start.
template <int BITS, bool IS_V>
__device__ __forceinline__ void locate(int t, int ch, int d, int& idx, int& pos) {
  int L, i, r, e;
  if (IS_V) {
    const int c = t / 8, s = (t >> 1) & 1;
    e = (t >> 2) & 1;
    r = t & 1;
    const int a = ch % 8, n = ch / 8;
    L = 4 * a + c;
    i = s * (d / 8) + n;
  } else {
    const int a = t / 4, j = t % 4;
    const int c = ch / (d / 4), rem = ch % (d / 4);
    const int k = rem / 4;
    r = (rem >> 1) & 1;
    e = rem & 1;
    L = 4 * a + c;
    i = j * (d / 16) + k;
  }
  int w, u;
  if (BITS == 2) {
    w = i / 4;
    u = i % 4;
  } else {
    constexpr int SPW = 16 / BITS;
    const int i2 = 2 * i + r;
    w = i2 / SPW;
    u = i2 % SPW;
  }
  idx = (w / 4) * 128 + 4 * L + w % 4;
  pos = field_pos(BITS, u, r, e);
}

// grid (T/32, B*Hkv), thread per (token, channel) pairs.
template <int BITS>
__global__ void unpack_kernel(int T, int T_cap, int d, Packed p, float* K_hat, float* V_hat) {
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  const int g = blockIdx.x, bh = blockIdx.y;
  Packed s = slice(p, bh, T_cap, d, BITS);
  const int n_words = d * BITS;
  for (int i = threadIdx.x; i < kGroup * d; i += blockDim.x) {
    const int t = i / d, c = i % d;
    int ki, kp, vi, vp;
    locate<BITS, false>(t, c, d, ki, kp);
    locate<BITS, true>(t, c, d, vi, vp);
    const uint32_t kw = s.kc[static_cast<size_t>(g) * n_words + ki];
    const uint32_t vw = s.vc[static_cast<size_t>(g) * n_words + vi];
    const float kcode = static_cast<float>((kw >> kp) & MASK);
    const float vcode = static_cast<float>((vw >> vp) & MASK);
    const size_t km = static_cast<size_t>(g) * 2 * d + c;
    const size_t vm = ((static_cast<size_t>(g) * (d / kGroup) + c / kGroup) * 2) * kGroup + vmeta_entry(t);
    const size_t o = (static_cast<size_t>(bh) * T + static_cast<size_t>(g) * kGroup + t) * d + c;
    K_hat[o] = fmaf(kcode, vc_f16_to_f32(s.ksz[km]), vc_f16_to_f32(s.ksz[km + d]));
    V_hat[o] = fmaf(vcode, vc_f16_to_f32(s.vsz[vm]), vc_f16_to_f32(s.vsz[vm + kGroup]));
  }
}

// ------------------------------------------------------------------ token score
//
// S = q_obs . K^T per KV head on the tcgen05 tensor cores: bf16 operands in
// shared memory, fp32 accumulators in TMEM (the products of bf16 values are
// exact), log2 softmax scale applied to the fp32 sums.  The work is a list of
// items, one per (b, KV head) and kScoreRange = 1024-token range; a
// persistent CTA per SM takes a contiguous run of items and walks their
// 128-token K tiles as one sequence.  Warp roles:
//   * lane 0 of the last warp loads K tiles (and q when the KV head changes)
//     with TMA tensor copies into a kScoreStages ring and issues each tile's
//     products into one of two TMEM buffers;
//   * 16 epilogue warps read a buffer (warp w: TMEM lane quarter w % 4) while
//     the tensor cores fill the other.
// They meet only on mbarriers: stage full (TMA bytes), stage empty and buffer
// full (tcgen05.commit), buffer empty (16 warp arrivals); with up to four
// TMEM buffers the products run up to three tiles ahead of the epilogue.  Both
// operands are K-major tiles in the 128-byte-swizzled layout (vc_tc_desc_sw128)
// written by TMA boxes of 64 channels x all rows: region h of a tile holds
// channels 64 h .. 64 h + 63, 128 bytes per row.
//   pass 1: D = Q . K_tile^T (rows in TMEM lanes): each thread folds (max,
//           sum exp2) of one row over 32 tokens of every tile; per item the
//           4 partials of every row are merged into the range's statistics.
//           Rows 0-127 are one M = 128 product; for NR > 128 a second one
//           takes rows NR - 128 .. NR - 1, so its new rows (128 and up) sit in
//           the highest lane quarters, away from the issuing thread's
//           scheduler (quarter 0), and no row past NR is read;
//   merge:  per row, the threshold M + log2 S over all ranges;
//   pass 2: D = K_tile . Q^T (tokens in TMEM lanes, N = NR): each thread sums
//           exp2(s_rt - threshold_r) over a quarter of the rows for its
//           token; the quarters are added in shared memory.
constexpr int kScoreEpiWarps = 16;
constexpr int kScoreEpiThreads = kScoreEpiWarps * 32;
constexpr int kScoreThreads = kScoreEpiThreads + 32;
constexpr int kScoreTile = 128;
constexpr int kScoreTilesPerRange = 8;
constexpr int kScoreRange = kScoreTilesPerRange * kScoreTile;
constexpr int kScoreStages = 4;
constexpr int kScoreMaxBufs = 4;                   // TMEM accumulator buffers
constexpr long long kScoreWaitCycles = 4000000000LL;   // ~2 s at 2 GHz

struct ScoreArgs {
  int T, n_obs, Hq, Hkv;
  float scale_log2;     // softmax_scale * log2(e)
  float2* stats;        // [B*Hkv, n_ranges, NR] (max, sum) per range, log2 units
  float* thr;           // [B*Hkv, NR] M + log2 S per row
  int n_ranges;
  int n_items;          // B * Hkv * n_ranges
};

// 2^x (ex2.approx.ftz: relative error ~2^-22; results below 2^-126 flush to 0)
__device__ __forceinline__ float sc_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// TMA tensor copies into this CTA's shared memory, completion as transaction bytes on `bar`.
__device__ __forceinline__ void sc_tma3(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(vc_smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(vc_smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void sc_tma2(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(vc_smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(vc_smem_addr(bar))
      : "memory");
}

template <int MT, int D>
struct ScoreCfg {
  static constexpr int NR = 16 * MT;               // rows = G * n_obs
  static constexpr int KS = D / 16;                // products along the channel axis
  static constexpr int REG = D / 64;               // 64-channel regions (TMA boxes) per tile
  // pass 1: a second M = 128 product for rows NR - 128 .. NR - 1 when NR > 128
  static constexpr bool TWO = NR > 128;
  static constexpr int S2 = NR - 128;              // its first row
  static constexpr int cols1 = TWO ? 256 : 128;
  // TMEM buffers: stride a multiple of 32 columns (the allocation unit), as
  // many as fit in 512 columns, at most kScoreMaxBufs
  static constexpr int stride1 = cols1;
  static constexpr int stride2 = (NR + 31) / 32 * 32;
  static constexpr int bufs1 = 512 / stride1 < kScoreMaxBufs ? 512 / stride1 : kScoreMaxBufs;
  static constexpr int bufs2 = 512 / stride2 < kScoreMaxBufs ? 512 / stride2 : kScoreMaxBufs;
  // pass 2: NCG column groups of CW rows of q (CW in 16 .. 64, a multiple of 8)
  static constexpr int NCG = NR >= 64 ? 4 : NR / 16;
  static constexpr int CW = NR / NCG;
  // highest q row a pass-1 product reads (for NR < 128, rows past NR feed unused lanes)
  static constexpr int max_row = TWO ? NR - 1 : 127;
  static constexpr uint32_t q_bytes = NR * D * 2;
  // the last region's rows may run past the q tile: keep them inside the q region
  static constexpr uint32_t q_reach = (REG - 1) * NR * 128 + (max_row + 1) * 128;
  static constexpr uint32_t q_region = ((q_reach > q_bytes ? q_reach : q_bytes) + 1023) / 1024 * 1024;
  static constexpr uint32_t k_bytes = kScoreTile * D * 2;                  // one K stage
  static constexpr uint32_t off_k = q_region;
  static constexpr uint32_t off_red = off_k + kScoreStages * k_bytes;     // pass 1: [2][4][NR] float2
  static constexpr uint32_t off_sum = off_red + 2 * 4 * NR * 8;           // pass 2: [2][4][128] float
  static constexpr uint32_t off_thr = off_sum + 2 * 4 * kScoreTile * 4;   // pass 2: [NR] float
  static constexpr uint32_t off_bar = off_thr + NR * 4;                   // 17 mbarriers, TMEM base, abort
  static constexpr uint32_t smem = off_bar + 17 * 8 + 8 + 1024;       // + alignment slack
  static_assert(smem <= 227 * 1024, "shared memory");

};

__host__ __device__ constexpr uint32_t sc_pow2_cols(int c) {
  return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512;
}

// Position in a CTA's tile sequence: item (slice, range) and tile within it.
struct ScoreCursor {
  int item, tile, n_tiles, bh, t0;
  __device__ __forceinline__ void set(const ScoreArgs& a, int it) {
    item = it;
    tile = 0;
    bh = it / a.n_ranges;
    const int r0 = (it % a.n_ranges) * kScoreRange;
    n_tiles = min(kScoreTilesPerRange, (a.T - r0 + kScoreTile - 1) / kScoreTile);
    t0 = r0;
  }
  __device__ __forceinline__ void next(const ScoreArgs& a) {
    if (++tile < n_tiles) {
      t0 += kScoreTile;
    } else {
      set(a, item + 1);
    }
  }
};

// The products of one tile into TMEM columns from `tmem`, issued by one
// thread.  A descriptor moves with its start address: desc + (bytes >> 4)
// (the address field cannot carry: shared addresses stay below 256 KB).
// Channel step kk: region kk / 4 (q: NR * 128 B, K tile: 128 * 128 B apart),
// +32 B per step inside the region; row r: +128 r B.
template <int PASS, int MT, int D>
__device__ __forceinline__ uint64_t score_koff(int kk, uint32_t region_bytes) {
  return static_cast<uint64_t>(((kk >> 2) * region_bytes + (kk & 3) * 32) >> 4);
}
template <int PASS, int MT, int D>
__device__ __forceinline__ void score_issue(uint32_t tmem, uint32_t q_addr, uint32_t k_addr) {
  using C = ScoreCfg<MT, D>;
  constexpr uint32_t QR = C::NR * 128, KR = kScoreTile * 128;
  const uint64_t dq = vc_tc_desc_sw128(q_addr), dk = vc_tc_desc_sw128(k_addr);
  if (PASS == 1) {
    constexpr uint32_t id128 = vc_tc_idesc_bf16(128, kScoreTile);
#pragma unroll
    for (int kk = 0; kk < C::KS; ++kk)
      vc_tc_mma(tmem, dq + score_koff<PASS, MT, D>(kk, QR), dk + score_koff<PASS, MT, D>(kk, KR), id128, kk > 0);
    if constexpr (C::TWO) {
#pragma unroll
      for (int kk = 0; kk < C::KS; ++kk)
        vc_tc_mma(tmem + 128, dq + ((C::S2 * 128) >> 4) + score_koff<PASS, MT, D>(kk, QR),
                  dk + score_koff<PASS, MT, D>(kk, KR), id128, kk > 0);
    }
  } else {
    constexpr uint32_t idesc = vc_tc_idesc_bf16(kScoreTile, C::NR);
#pragma unroll
    for (int kk = 0; kk < C::KS; ++kk)
      vc_tc_mma(tmem, dk + score_koff<PASS, MT, D>(kk, KR), dq + score_koff<PASS, MT, D>(kk, QR), idesc, kk > 0);
  }
}

// Online (max, sum exp2) of one row over 32 tokens first_t .. first_t + 31 (scores s).
__device__ __forceinline__ void score_fold32(float* s, const ScoreArgs& a, bool masked, int first_t, int last,
                                             float& m, float& l) {
  if (masked) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (first_t + j > last) s[j] = -INFINITY;
  }
  float mx = s[0];
#pragma unroll
  for (int j = 1; j < 32; ++j) mx = fmaxf(mx, s[j]);
  const float mn = fmaxf(m, mx * a.scale_log2);    // log2 units (scale > 0)
  if (mn == -INFINITY) return;                     // nothing visible yet
  float add = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) add += sc_exp2(fmaf(s[j], a.scale_log2, -mn));
  l = l * sc_exp2(m - mn) + add;
  m = mn;
}

// Columns [0, N) of the warp's TMEM lanes from taddr, in one statement.
template <int N>
__device__ __forceinline__ void score_ld(uint32_t taddr, float (&v)[N]) {
  if constexpr (N == 8) vc_tc_ld8(taddr, v);
  else if constexpr (N == 16) vc_tc_ld16(taddr, v);
  else if constexpr (N == 24) vc_tc_ld24(taddr, v);
  else if constexpr (N == 32) vc_tc_ld32(taddr, v);
  else if constexpr (N == 40) vc_tc_ld40(taddr, v);
  else if constexpr (N == 48) vc_tc_ld48(taddr, v);
  else if constexpr (N == 56) vc_tc_ld56(taddr, v);
  else vc_tc_ld64(taddr, v);
}

// Pass 2: acc += exp2(s_j * scale - threshold) over N columns from cbase for
// token t, skipping the rows that do not see t.
template <int N>
__device__ __forceinline__ void score_acc(const float (&s)[N], const float* thr_s, int cbase, bool masked, int t,
                                          const ScoreArgs& a, float& acc) {
  if (masked) {                                    // row r sees t iff t <= T - n_obs + r % n_obs
    const int lag = t - (a.T - a.n_obs);           // row r needs r % n_obs >= lag
    int o = cbase % a.n_obs;
#pragma unroll
    for (int jj = 0; jj < N; ++jj) {
      if (o >= lag) acc += sc_exp2(fmaf(s[jj], a.scale_log2, -thr_s[cbase + jj]));
      o = o + 1 == a.n_obs ? 0 : o + 1;
    }
    return;
  }
#pragma unroll
  for (int jj = 0; jj < N; jj += 4) {
    const float4 v = *reinterpret_cast<const float4*>(thr_s + cbase + jj);
    acc += sc_exp2(fmaf(s[jj], a.scale_log2, -v.x));
    acc += sc_exp2(fmaf(s[jj + 1], a.scale_log2, -v.y));
    acc += sc_exp2(fmaf(s[jj + 2], a.scale_log2, -v.z));
    acc += sc_exp2(fmaf(s[jj + 3], a.scale_log2, -v.w));
  }
}

// grid = min(SMs, items), one CTA per SM.  PASS 1 writes the range statistics, PASS 2 the scores.
template <int PASS, int MT, int D>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_pass(ScoreArgs a, const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tq,
               float* __restrict__ score) {
  using C = ScoreCfg<MT, D>;
  constexpr int NR = C::NR;
  constexpr int COLS = PASS == 1 ? C::stride1 : C::stride2;    // TMEM buffer stride
  constexpr int BUFS = PASS == 1 ? C::bufs1 : C::bufs2;
  constexpr uint32_t NCOLS = sc_pow2_cols(COLS * BUFS);
  extern __shared__ __align__(16) uint8_t smem_raw[];
  // swizzled tiles: 1024-byte aligned (1024 bytes of slack are allocated)
  uint8_t* smem = smem_raw + ((1024u - (vc_smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* q_s = smem;
  uint8_t* k_s = smem + C::off_k;
  float2* red = reinterpret_cast<float2*>(smem + C::off_red);
  float* tsum = reinterpret_cast<float*>(smem + C::off_sum);
  float* thr_s = reinterpret_cast<float*>(smem + C::off_thr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::off_bar);   // [kScoreStages]
  uint64_t* empty = full + kScoreStages;                              // [kScoreStages]
  uint64_t* tfull = empty + kScoreStages;                             // [kScoreMaxBufs]
  uint64_t* tempty = tfull + kScoreMaxBufs;                           // [kScoreMaxBufs]
  uint64_t* qbar = tempty + kScoreMaxBufs;
  uint32_t* slot = reinterpret_cast<uint32_t*>(qbar + 1);
  volatile uint32_t* abort = slot + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3, grp = warp >> 2;
  const int i0 = static_cast<int>(static_cast<long long>(blockIdx.x) * a.n_items / gridDim.x);
  const int i1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * a.n_items / gridDim.x);
  int n = 0;                                       // tiles in this CTA's sequence
  for (int it = i0; it < i1; ++it) {
    const int r0 = (it % a.n_ranges) * kScoreRange;
    n += min(kScoreTilesPerRange, (a.T - r0 + kScoreTile - 1) / kScoreTile);
  }

  if (warp == 0) vc_tc_alloc(slot, NCOLS);
  if (threadIdx.x == kScoreEpiThreads) {
    for (int s = 0; s < kScoreStages; ++s) {
      vc_mbar_init(full + s, 1);
      vc_mbar_init(empty + s, 1);
    }
    for (int b = 0; b < kScoreMaxBufs; ++b) {
      vc_mbar_init(tfull + b, 1);
      vc_mbar_init(tempty + b, kScoreEpiWarps);
    }
    vc_mbar_init(qbar, 1);
    *abort = 0u;
    vc_fence_mbar_init();
  }
  vc_tc_fence_before();
  __syncthreads();
  vc_tc_fence_after();
  const uint32_t tmem = *slot;

  if (warp == kScoreEpiWarps) {
    // ---------------- loads and products (one thread)
    if (lane == 0 && n > 0) {
      const int G = a.Hq / a.Hkv;
      const uint32_t q_addr = vc_smem_addr(q_s), k_addr = vc_smem_addr(k_s);
      auto load_q = [&](int bh) {
        const int y = ((bh / a.Hkv) * a.Hq + (bh % a.Hkv) * G) * a.n_obs;
        vc_mbar_arrive_expect_tx(qbar, C::q_bytes);
        for (int h = 0; h < C::REG; ++h) sc_tma2(q_s + h * NR * 128, &tq, 64 * h, y, qbar);
      };
      auto load_k = [&](const ScoreCursor& cu, int stage) {
        uint64_t* bar = full + stage;
        vc_mbar_arrive_expect_tx(bar, C::k_bytes);
        for (int h = 0; h < C::REG; ++h)
          sc_tma3(k_s + stage * C::k_bytes + h * kScoreTile * 128, &tk, 64 * h, cu.t0, cu.bh, bar);
      };
      ScoreCursor mc, ld;
      mc.set(a, i0);
      ld = mc;
      int q_bh = mc.bh;
      uint32_t q_phase = 0;
      load_q(q_bh);
      for (int s = 0; s < kScoreStages && s < n; ++s) {
        load_k(ld, s);
        ld.next(a);
      }
      bool ok = vc_mbar_wait_or_abort(qbar, q_phase, abort, kScoreWaitCycles);
      q_phase ^= 1u;
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % kScoreStages, b = j % BUFS;
        if (mc.bh != q_bh) {                       // every earlier product done, then this slice's q
          ok = vc_mbar_wait_or_abort(empty + (j - 1) % kScoreStages, ((j - 1) / kScoreStages) & 1, abort,
                                     kScoreWaitCycles);
          if (!ok) break;
          q_bh = mc.bh;
          load_q(q_bh);
          ok = vc_mbar_wait_or_abort(qbar, q_phase, abort, kScoreWaitCycles);
          q_phase ^= 1u;
          if (!ok) break;
        }
        ok = vc_mbar_wait_or_abort(full + s, (j / kScoreStages) & 1, abort, kScoreWaitCycles);
        // the buffer's previous tile p = j - BUFS has been read out (its
        // epilogue completes phase p / BUFS of tempty[b])
        if (ok && j >= BUFS)
          ok = vc_mbar_wait_or_abort(tempty + b, ((j - BUFS) / BUFS) & 1, abort, kScoreWaitCycles);
        if (!ok) break;
        vc_tc_fence_after();
        score_issue<PASS, MT, D>(tmem + b * COLS, q_addr, k_addr + s * C::k_bytes);
        vc_tc_commit(tfull + b);
        vc_tc_commit(empty + s);
        mc.next(a);
        // refill the stage of tile j - 1 with tile j + kScoreStages - 1
        if (j >= 1 && j + kScoreStages - 1 < n) {
          const int sp = (j - 1) % kScoreStages;
          ok = vc_mbar_wait_or_abort(empty + sp, ((j - 1) / kScoreStages) & 1, abort, kScoreWaitCycles);
          if (!ok) break;
          load_k(ld, sp);
          ld.next(a);
        }
      }
      if (!ok) *abort = 1u;
    }
  } else {
    // ---------------- epilogue warps
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    // pass-1 pieces of this warp, both over tokens 32 grp .. 32 grp + 31 of a
    // tile: A = row quarter * 32 + lane of the first product, B = row
    // S2 + quarter * 32 + lane of the second (only its rows >= 128 are new)
    const int rowA = quarter * 32 + lane;
    const bool liveA = quarter * 32 < NR;
    const int rowB = C::S2 + quarter * 32 + lane;
    const bool liveB = C::TWO && C::S2 + quarter * 32 + 31 >= 128;
    const bool newB = liveB && rowB >= 128;
    const int lastA = a.T - a.n_obs + rowA % a.n_obs, lastB = a.T - a.n_obs + rowB % a.n_obs;
    float mA = -INFINITY, lA = 0.0f, mB = -INFINITY, lB = 0.0f;
    int n_items_done = 0, thr_bh = -1;
    ScoreCursor ec;
    ec.set(a, i0);
    for (int j = 0; j < n; ++j) {
      const int b = j % BUFS;
      // after an abort every warp still takes every named barrier below
      bool live = *abort == 0u && vc_mbar_wait_or_abort(tfull + b, (j / BUFS) & 1, abort, kScoreWaitCycles);
      live = __all_sync(0xffffffffu, live);
      vc_tc_fence_after();
      const uint32_t tb = t_lane + b * COLS;
      const bool masked = ec.t0 + kScoreTile > a.T - a.n_obs;   // tile reaches the observation window
      if (PASS == 1) {
        if (live && liveA && liveB) {              // both pieces in one TMEM round trip
          float s[64];
          vc_tc_ld32x2(tb + grp * 32, tb + 128 + grp * 32, s);
          score_fold32(s, a, masked, ec.t0 + grp * 32, lastA, mA, lA);
          score_fold32(s + 32, a, masked, ec.t0 + grp * 32, lastB, mB, lB);
        } else if (live && liveA) {
          float s[32];
          vc_tc_ld32(tb + grp * 32, s);
          score_fold32(s, a, masked, ec.t0 + grp * 32, lastA, mA, lA);
        }
      } else {
        if (ec.bh != thr_bh) {                     // this slice's row thresholds into shared memory
          vc_bar_sync(1, kScoreEpiThreads);
          for (int r = threadIdx.x; r < NR; r += kScoreEpiThreads) thr_s[r] = a.thr[static_cast<size_t>(ec.bh) * NR + r];
          vc_bar_sync(1, kScoreEpiThreads);
          thr_bh = ec.bh;
        }
        float acc = 0.0f;
        if (live && grp < C::NCG) {
          const int t = ec.t0 + quarter * 32 + lane;
          const int c0 = grp * C::CW;
          constexpr int H1 = C::CW > 32 ? 32 : C::CW, H2 = C::CW - H1;   // at most two TMEM round trips
          {
            float s[H1];
            score_ld<H1>(tb + c0, s);
            score_acc<H1>(s, thr_s, c0, masked, t, a, acc);
          }
          if constexpr (H2 > 0) {
            float s[H2];
            score_ld<H2>(tb + c0 + H1, s);
            score_acc<H2>(s, thr_s, c0 + H1, masked, t, a, acc);
          }
        }
        if (grp < C::NCG) tsum[(j & 1) * 4 * kScoreTile + grp * kScoreTile + quarter * 32 + lane] = acc;
      }
      vc_tc_fence_before();                        // TMEM reads done before the buffer is refilled
      __syncwarp();
      if (lane == 0) vc_mbar_arrive(tempty + b);
      if (PASS == 1) {
        if (ec.tile + 1 == ec.n_tiles) {           // item done: merge the 4 partials of every row
          float2* rd = red + (n_items_done & 1) * 4 * NR;
          if (liveA && rowA < NR) rd[grp * NR + rowA] = make_float2(mA, lA);
          if (newB) rd[grp * NR + rowB] = make_float2(mB, lB);
          vc_bar_sync(1, kScoreEpiThreads);
          float2* out = a.stats + static_cast<size_t>(ec.item) * NR;   // item = bh * n_ranges + range
          for (int r = threadIdx.x; r < NR && *abort == 0u; r += kScoreEpiThreads) {
            float M = -INFINITY;
#pragma unroll
            for (int s = 0; s < 4; ++s) M = fmaxf(M, rd[s * NR + r].x);
            float S = 0.0f;
            if (M != -INFINITY) {
#pragma unroll
              for (int s = 0; s < 4; ++s) {
                const float2 v = rd[s * NR + r];
                if (v.x != -INFINITY) S += v.y * exp2f(v.x - M);
              }
            }
            out[r] = make_float2(M, S);
          }
          ++n_items_done;
          mA = mB = -INFINITY;
          lA = lB = 0.0f;
        }
      } else {
        vc_bar_sync(2 + quarter, 128);             // the column groups of this quarter's tokens are in tsum
        if (grp == 0 && *abort == 0u) {
          const int t = ec.t0 + quarter * 32 + lane;
          const float* ts = tsum + (j & 1) * 4 * kScoreTile + quarter * 32 + lane;
          float x = 0.0f;
#pragma unroll
          for (int g = 0; g < C::NCG; ++g) x += ts[g * kScoreTile];
          if (t < a.T) score[static_cast<size_t>(ec.bh) * a.T + t] = x;
        }
      }
      ec.next(a);
    }
  }
  vc_tc_fence_before();
  __syncthreads();
  vc_tc_fence_after();
  if (threadIdx.x == 0 && *abort != 0u) atomicOr(&g_quant_status, VC_DEV_BARRIER_TIMEOUT);
  if (warp == 0) vc_tc_dealloc(tmem, NCOLS);
}

// grid (B*Hkv): per row, the threshold M + log2 S over the ranges.
__global__ void score_merge(ScoreArgs a, int NR) {
  const int bh = blockIdx.x;
  for (int r = threadIdx.x; r < NR; r += blockDim.x) {
    const float2* st = a.stats + static_cast<size_t>(bh) * a.n_ranges * NR + r;
    float M = -INFINITY;
    for (int x = 0; x < a.n_ranges; ++x) M = fmaxf(M, st[static_cast<size_t>(x) * NR].x);
    float S = 0.0f;
    for (int x = 0; x < a.n_ranges; ++x) {
      const float2 v = st[static_cast<size_t>(x) * NR];
      if (v.x != -INFINITY) S += v.y * exp2f(v.x - M);
    }
    a.thr[static_cast<size_t>(bh) * NR + r] = M + log2f(S);
  }
}

// ------------------------------------------------------------------ select
constexpr int kSelThreads = 1024;

// Order-preserving map of fp32 to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// pooled keys: grid (ceil(T/256), B*Hkv)
__global__ void pool_kernel(const float* __restrict__ score, int T, int pool, uint32_t* __restrict__ keys) {
  const int bh = blockIdx.y;
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int r = pool / 2;
  const float* s = score + static_cast<size_t>(bh) * T;
  float m = -INFINITY;
  const int lo = max(0, t - r), hi = min(T - 1, t + r);
  for (int u = lo; u <= hi; ++u) m = fmaxf(m, s[u]);
  keys[static_cast<size_t>(bh) * T + t] = float_key(m);
}

// Block-wide exclusive scan of one int per thread (kSelThreads threads).
__device__ int block_exclusive_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < kSelThreads / 32) ? tmp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    tmp[lane] = w;                      // inclusive per warp
  }
  __syncthreads();
  const int before = (warp > 0 ? tmp[warp - 1] : 0) + x - v;
  if (total) *total = tmp[kSelThreads / 32 - 1];
  __syncthreads();
  return before;
}

// One CTA per (b, h): radix-select the n_top-th largest key among candidates
// [0, cand), then emit, in index order, keys above it plus the lowest-index
// keys equal to it, then the keep_last tail tokens.
__global__ void __launch_bounds__(kSelThreads) select_kernel(const uint32_t* __restrict__ keys_all, int T,
                                                             int keep, int keep_last,
                                                             int32_t* __restrict__ idx) {
  __shared__ int hist[256];
  __shared__ int tmp[32];
  __shared__ uint32_t prefix_s;
  __shared__ int remain_s;
  const int bh = blockIdx.x;
  const uint32_t* keys = keys_all + static_cast<size_t>(bh) * T;
  const int cand = T - keep_last;
  const int n_top = keep - keep_last;
  int32_t* out = idx + static_cast<size_t>(bh) * keep;
  uint32_t prefix = 0, mask = 0;
  int remain = n_top;                    // rank (1-based) still to find inside the prefix
  if (n_top > 0) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int t = threadIdx.x; t < cand; t += blockDim.x) {
        const uint32_t k = keys[t];
        if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int acc = 0, bin = 255;
        for (; bin >= 0; --bin) {
          if (acc + hist[bin] >= remain) break;
          acc += hist[bin];
        }
        prefix_s = prefix | (static_cast<uint32_t>(bin) << shift);
        remain_s = remain - acc;
      }
      __syncthreads();
      prefix = prefix_s;
      remain = remain_s;
      mask |= 255u << shift;
      __syncthreads();
    }
  }
  const uint32_t thr = prefix;           // the n_top-th largest key
  const int need_eq = remain;            // how many keys == thr to take (lowest index first)
  // contiguous chunk per thread, in index order
  const int per = (cand + kSelThreads - 1) / kSelThreads;
  const int lo = min(cand, threadIdx.x * per), hi = min(cand, lo + per);
  int n_eq = 0;
  if (n_top > 0)
    for (int t = lo; t < hi; ++t) n_eq += (keys[t] == thr);
  const int eq_before = block_exclusive_scan(n_eq, tmp, nullptr);
  int n_sel = 0;
  if (n_top > 0) {
    int e = eq_before;
    for (int t = lo; t < hi; ++t) {
      const uint32_t k = keys[t];
      const bool sel = k > thr || (k == thr && e < need_eq);
      e += (k == thr);
      n_sel += sel;
    }
  }
  int total = 0;
  int pos = block_exclusive_scan(n_sel, tmp, &total);
  if (n_top > 0) {
    int e = eq_before;
    for (int t = lo; t < hi; ++t) {
      const uint32_t k = keys[t];
      const bool sel = k > thr || (k == thr && e < need_eq);
      e += (k == thr);
      if (sel) out[pos++] = t;
    }
  }
  for (int j = threadIdx.x; j < keep_last; j += blockDim.x) out[n_top + j] = cand + j;
}

// ------------------------------------------------------------------ gather
__global__ void gather_kernel(const int32_t* __restrict__ idx, int T, int keep, int d,
                              const uint16_t* __restrict__ K, const uint16_t* __restrict__ V,
                              uint16_t* __restrict__ Ko, uint16_t* __restrict__ Vo) {
  const int bh = blockIdx.y;
  const int vec = d / 8;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= keep * vec) return;
  const int j = i / vec, v = i % vec;
  const int t = idx[static_cast<size_t>(bh) * keep + j];
  const size_t o = (static_cast<size_t>(bh) * keep + j) * d + v * 8;
  if (t < 0 || t >= T) {
    atomicOr(&g_quant_status, VC_DEV_BAD_INDEX);
    *reinterpret_cast<uint4*>(Ko + o) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(Vo + o) = make_uint4(0, 0, 0, 0);
    return;
  }
  const size_t s = (static_cast<size_t>(bh) * T + t) * d + v * 8;
  *reinterpret_cast<uint4*>(Ko + o) = *reinterpret_cast<const uint4*>(K + s);
  *reinterpret_cast<uint4*>(Vo + o) = *reinterpret_cast<const uint4*>(V + s);
}

vc_status_t check_shape(const vc_shape_t* s, bool need_bits) {
  VC_REQUIRE(s != nullptr, "shape is NULL");
  VC_REQUIRE(s->B >= 1 && s->Hkv >= 1, "need B >= 1 and Hkv >= 1");
  if (s->d != 64 && s->d != 128) VC_FAIL(VC_ERR_UNSUPPORTED, "head dim %d not in {64, 128}", s->d);
  if (need_bits && s->bits != 2 && s->bits != 4 && s->bits != 8)
    VC_FAIL(VC_ERR_UNSUPPORTED, "bits %d not in {2, 4, 8}", s->bits);
  return VC_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" vc_status_t vc_quant_packed_bytes(const vc_shape_t* s, int32_t T_cap, size_t* kc_bytes,
                                             size_t* ksz_bytes, size_t* vc_bytes, size_t* vsz_bytes) {
  vc_status_t st = check_shape(s, true);
  if (st != VC_OK) return st;
  VC_REQUIRE(T_cap >= 0 && T_cap % kGroup == 0, "T_cap must be a non-negative multiple of 32 (got %d)", T_cap);
  const size_t tok = static_cast<size_t>(s->B) * s->Hkv * T_cap;
  if (kc_bytes) *kc_bytes = tok * s->d * s->bits / 8;
  if (vc_bytes) *vc_bytes = tok * s->d * s->bits / 8;
  if (ksz_bytes) *ksz_bytes = tok / kGroup * s->d * 4;
  if (vsz_bytes) *vsz_bytes = tok * (s->d / kGroup) * 4;
  return VC_OK;
}

extern "C" vc_status_t vc_quant_kv_pack(const vc_shape_t* s, int32_t T, int32_t T_cap, const uint16_t* K,
                                        const uint16_t* V, uint32_t* kc, uint16_t* ksz, uint32_t* vc,
                                        uint16_t* vsz, vc_stream_t stream) {
  vc_status_t st = check_shape(s, true);
  if (st != VC_OK) return st;
  VC_REQUIRE(T >= 0 && T % kGroup == 0 && T <= T_cap && T_cap % kGroup == 0,
             "need 0 <= T <= T_cap, both multiples of 32 (T=%d, T_cap=%d)", T, T_cap);
  VC_REQUIRE(K && V && kc && ksz && vc && vsz, "NULL pointer");
  VC_REQUIRE(vc_aligned16(K) && vc_aligned16(V) && vc_aligned16(kc) && vc_aligned16(ksz) && vc_aligned16(vc) &&
                 vc_aligned16(vsz), "pointers must be 16-byte aligned");
  if (T == 0) return VC_OK;
  VC_REQUIRE(static_cast<int64_t>(s->B) * s->Hkv <= 65535, "B*Hkv <= 65535");
  dim3 grid(T / kGroup, s->B * s->Hkv);
  Packed p{kc, ksz, vc, vsz};
  auto cs = reinterpret_cast<cudaStream_t>(stream);
#define VC_PACK(BITS, D) pack_kernel<BITS, D><<<grid, kPackThreads, 0, cs>>>(K, V, T, T_cap, p)
  if (s->d == 128) {
    if (s->bits == 2) VC_PACK(2, 128);
    else if (s->bits == 4) VC_PACK(4, 128);
    else VC_PACK(8, 128);
  } else {
    if (s->bits == 2) VC_PACK(2, 64);
    else if (s->bits == 4) VC_PACK(4, 64);
    else VC_PACK(8, 64);
  }
#undef VC_PACK
  VC_LAUNCH_CHECK("pack_kernel");
  return VC_OK;
}

extern "C" vc_status_t vc_quant_kv_unpack(const vc_shape_t* s, int32_t T, int32_t T_cap, const uint32_t* kc,
                                          const uint16_t* ksz, const uint32_t* vc, const uint16_t* vsz,
                                          float* K_hat, float* V_hat, vc_stream_t stream) {
  vc_status_t st = check_shape(s, true);
  if (st != VC_OK) return st;
  VC_REQUIRE(T >= 0 && T % kGroup == 0 && T <= T_cap && T_cap % kGroup == 0, "bad T / T_cap");
  VC_REQUIRE(kc && ksz && vc && vsz && K_hat && V_hat, "NULL pointer");
  if (T == 0) return VC_OK;
  dim3 grid(T / kGroup, s->B * s->Hkv);
  Packed p{const_cast<uint32_t*>(kc), const_cast<uint16_t*>(ksz), const_cast<uint32_t*>(vc),
           const_cast<uint16_t*>(vsz)};
  auto cs = reinterpret_cast<cudaStream_t>(stream);
  if (s->bits == 2)
    unpack_kernel<2><<<grid, 256, 0, cs>>>(T, T_cap, s->d, p, K_hat, V_hat);
  else if (s->bits == 4)
    unpack_kernel<4><<<grid, 256, 0, cs>>>(T, T_cap, s->d, p, K_hat, V_hat);
  else
    unpack_kernel<8><<<grid, 256, 0, cs>>>(T, T_cap, s->d, p, K_hat, V_hat);
  VC_LAUNCH_CHECK("unpack_kernel");
  return VC_OK;
}

extern "C" vc_status_t vc_quant_kv_append(const vc_shape_t* s, const uint16_t* k_new, const uint16_t* v_new,
                                          const int32_t* n_acc, uint16_t* tail_k, uint16_t* tail_v,
                                          int32_t* tail_len, int32_t tail_cap, uint32_t* kc, uint16_t* ksz,
                                          uint32_t* vc, uint16_t* vsz, int32_t* packed_len, int32_t T_cap,
                                          vc_stream_t stream) {
  vc_status_t st = check_shape(s, true);
  if (st != VC_OK) return st;
  VC_REQUIRE(s->k >= 0, "k >= 0");
  VC_REQUIRE(tail_cap >= s->k + 1 && T_cap % kGroup == 0 && T_cap >= 0, "tail_cap >= k+1 and T_cap % 32 == 0");
  VC_REQUIRE(k_new && v_new && tail_k && tail_v && tail_len && kc && ksz && vc && vsz && packed_len, "NULL pointer");
  VC_REQUIRE(vc_aligned16(k_new) && vc_aligned16(v_new) && vc_aligned16(tail_k) && vc_aligned16(tail_v),
             "bf16 pointers must be 16-byte aligned");
  Packed p{kc, ksz, vc, vsz};
  const size_t sm = append_smem(s->d);
  auto cs = reinterpret_cast<cudaStream_t>(stream);
#define VC_APPEND(BITS, D)                                                                                    \
  append_kernel<BITS, D><<<dim3(s->Hkv, s->B), kPackThreads, sm, cs>>>(k_new, v_new, n_acc, s->k, s->Hkv, tail_k, \
                                                                       tail_v, tail_len, tail_cap, p, packed_len, T_cap)
  if (s->d == 128) {
    if (s->bits == 2) VC_APPEND(2, 128);
    else if (s->bits == 4) VC_APPEND(4, 128);
    else VC_APPEND(8, 128);
  } else {
    if (s->bits == 2) VC_APPEND(2, 64);
    else if (s->bits == 4) VC_APPEND(4, 64);
    else VC_APPEND(8, 64);
  }
#undef VC_APPEND
  VC_LAUNCH_CHECK("append_kernel");
  append_lengths_kernel<<<1, 256, 0, cs>>>(n_acc, s->B, s->k, tail_len, tail_cap, packed_len, T_cap);
  VC_LAUNCH_CHECK("append_lengths_kernel");
  return VC_OK;
}

namespace {
// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to
// the driver library); null when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

int score_ranges(int T) { return (T + kScoreRange - 1) / kScoreRange; }

vc_status_t check_score(const vc_shape_t* s, int T, int n_obs, int* NR) {
  vc_status_t st = check_shape(s, false);
  if (st != VC_OK) return st;
  VC_REQUIRE(s->Hq >= 1 && s->Hq % s->Hkv == 0, "Hq must be a multiple of Hkv");
  const int G = s->Hq / s->Hkv;
  if (G > 8) VC_FAIL(VC_ERR_UNSUPPORTED, "G = %d > 8", G);
  VC_REQUIRE(n_obs >= 1 && n_obs <= 32 && T >= n_obs, "need 1 <= n_obs <= 32 and T >= n_obs");
  *NR = G * n_obs;
  if (*NR % 16 != 0) VC_FAIL(VC_ERR_UNSUPPORTED, "G * n_obs = %d must be a multiple of 16", *NR);
  return VC_OK;
}
}  // namespace

extern "C" vc_status_t vc_token_score_workspace_size(const vc_shape_t* s, int32_t T, int32_t n_obs, size_t* bytes) {
  int NR = 0;
  vc_status_t st = check_score(s, T, n_obs, &NR);
  if (st != VC_OK) return st;
  VC_REQUIRE(bytes, "bytes is NULL");
  *bytes = static_cast<size_t>(s->B) * s->Hkv * (score_ranges(T) + 1) * NR * sizeof(float2);
  return VC_OK;
}

extern "C" vc_status_t vc_token_score(const vc_shape_t* s, int32_t T, int32_t n_obs, const uint16_t* q_obs,
                                      const uint16_t* K, float* score, void* workspace, size_t workspace_bytes,
                                      vc_stream_t stream) {
  int NR = 0;
  vc_status_t st = check_score(s, T, n_obs, &NR);
  if (st != VC_OK) return st;
  VC_REQUIRE(q_obs && K && score, "NULL pointer");
  VC_REQUIRE(vc_aligned16(q_obs) && vc_aligned16(K), "q_obs and K must be 16-byte aligned");
  size_t need = 0;
  vc_token_score_workspace_size(s, T, n_obs, &need);
  if (!workspace || workspace_bytes < need)
    VC_FAIL(VC_ERR_WORKSPACE, "score workspace needs %zu bytes (got %zu)", need, workspace_bytes);
  ScoreArgs a;
  a.T = T; a.n_obs = n_obs; a.Hq = s->Hq; a.Hkv = s->Hkv;
  a.scale_log2 = s->softmax_scale * 1.4426950408889634f;
  a.n_ranges = score_ranges(T);
  a.n_items = s->B * s->Hkv * a.n_ranges;
  a.stats = static_cast<float2*>(workspace);
  a.thr = reinterpret_cast<float*>(a.stats + static_cast<size_t>(s->B) * s->Hkv * a.n_ranges * NR);
  // TMA maps (128-byte swizzle): K as [B*Hkv][T][d] in boxes of 64 channels x
  // 128 tokens (zero past T), q as [B*Hq*n_obs][d] in boxes of 64 channels x NR rows
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) VC_FAIL(VC_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  CUtensorMap tk, tq;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(s->d), static_cast<cuuint64_t>(T),
                                static_cast<cuuint64_t>(s->B) * s->Hkv};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(s->d) * 2, static_cast<cuuint64_t>(T) * s->d * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kScoreTile), 1}, es[3] = {1, 1, 1};
    CUresult r = encode(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(K), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) VC_FAIL(VC_ERR_CUDA, "K tensor map: error %d", static_cast<int>(r));
    const cuuint64_t qd[2] = {static_cast<cuuint64_t>(s->d), static_cast<cuuint64_t>(s->B) * s->Hq * n_obs};
    const cuuint64_t qs[1] = {static_cast<cuuint64_t>(s->d) * 2};
    const cuuint32_t qb[2] = {64, static_cast<cuuint32_t>(NR)};
    r = encode(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(q_obs), qd, qs, qb, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) VC_FAIL(VC_ERR_CUDA, "q tensor map: error %d", static_cast<int>(r));
  }
  auto cs = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  VC_CUDA_CHECK(cudaGetDevice(&dev));
  VC_CUDA_CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const dim3 grid(a.n_items < sms ? a.n_items : sms);
  const int bhs = s->B * s->Hkv;
#define VC_SCORE_CASE(M, D)                                                                          \
  case M: {                                                                                          \
    const int sm = static_cast<int>(ScoreCfg<M, D>::smem);                                           \
    cudaFuncSetAttribute(score_pass<1, M, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);      \
    cudaFuncSetAttribute(score_pass<2, M, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);      \
    score_pass<1, M, D><<<grid, kScoreThreads, sm, cs>>>(a, tk, tq, score);                          \
    score_merge<<<bhs, 256, 0, cs>>>(a, NR);                                                         \
    score_pass<2, M, D><<<grid, kScoreThreads, sm, cs>>>(a, tk, tq, score);                          \
    break;                                                                                           \
  }
#define VC_SCORE_SWITCH(D)                                                                           \
  switch (NR / 16) {                                                                                 \
    VC_SCORE_CASE(1, D)                                                                              \
    VC_SCORE_CASE(2, D)                                                                              \
    VC_SCORE_CASE(4, D)                                                                              \
    VC_SCORE_CASE(6, D)                                                                              \
    VC_SCORE_CASE(8, D)                                                                              \
    VC_SCORE_CASE(10, D)                                                                             \
    VC_SCORE_CASE(12, D)                                                                             \
    VC_SCORE_CASE(14, D)                                                                             \
    VC_SCORE_CASE(16, D)                                                                             \
    default:                                                                                         \
      VC_FAIL(VC_ERR_UNSUPPORTED, "G * n_obs = %d not built (need 16 * {1,2,4,6,...,16})", NR);      \
  }
  if (s->d == 128) {
    VC_SCORE_SWITCH(128)
  } else {
    VC_SCORE_SWITCH(64)
  }
#undef VC_SCORE_SWITCH
#undef VC_SCORE_CASE
  VC_LAUNCH_CHECK("token score");
  return VC_OK;
}

extern "C" vc_status_t vc_token_select_workspace_size(int32_t B, int32_t Hkv, int32_t T, size_t* bytes) {
  VC_REQUIRE(B >= 1 && Hkv >= 1 && T >= 1 && bytes, "bad arguments");
  *bytes = static_cast<size_t>(B) * Hkv * T * sizeof(uint32_t);
  return VC_OK;
}

extern "C" vc_status_t vc_token_select(int32_t B, int32_t Hkv, int32_t T, const float* score, int32_t keep,
                                       int32_t keep_last, int32_t pool, int32_t* idx, void* workspace,
                                       size_t workspace_bytes, vc_stream_t stream) {
  VC_REQUIRE(B >= 1 && Hkv >= 1 && T >= 1, "need B, Hkv, T >= 1");
  VC_REQUIRE(keep_last >= 0 && keep_last <= keep && keep <= T, "need 0 <= keep_last <= keep <= T");
  VC_REQUIRE(pool >= 1 && pool <= 15 && (pool & 1), "pool must be odd, 1..15");
  VC_REQUIRE(score && idx, "NULL pointer");
  const size_t need = static_cast<size_t>(B) * Hkv * T * sizeof(uint32_t);
  if (!workspace || workspace_bytes < need)
    VC_FAIL(VC_ERR_WORKSPACE, "select workspace needs %zu bytes (got %zu)", need, workspace_bytes);
  auto cs = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* keys = static_cast<uint32_t*>(workspace);
  pool_kernel<<<dim3((T + 255) / 256, B * Hkv), 256, 0, cs>>>(score, T, pool, keys);
  VC_LAUNCH_CHECK("pool_kernel");
  select_kernel<<<B * Hkv, kSelThreads, 0, cs>>>(keys, T, keep, keep_last, idx);
  VC_LAUNCH_CHECK("select_kernel");
  return VC_OK;
}

extern "C" vc_status_t vc_gather_kv(const vc_shape_t* s, int32_t T, int32_t keep, const int32_t* idx,
                                    const uint16_t* K, const uint16_t* V, uint16_t* K_out, uint16_t* V_out,
                                    vc_stream_t stream) {
  vc_status_t st = check_shape(s, false);
  if (st != VC_OK) return st;
  VC_REQUIRE(T >= 1 && keep >= 0, "need T >= 1, keep >= 0");
  VC_REQUIRE(idx && K && V && K_out && V_out, "NULL pointer");
  VC_REQUIRE(vc_aligned16(K) && vc_aligned16(V) && vc_aligned16(K_out) && vc_aligned16(V_out),
             "pointers must be 16-byte aligned");
  if (keep == 0) return VC_OK;
  const int vec = s->d / 8;
  dim3 grid((keep * vec + 255) / 256, s->B * s->Hkv);
  gather_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(idx, T, keep, s->d, K, V, K_out, V_out);
  VC_LAUNCH_CHECK("gather_kernel");
  return VC_OK;
}

// Groups [g0, g1) of every (request, KV head) of a packed cache held in pinned
// host memory (layout of the device arrays with host_ng groups per (b, h)) into
// the device arrays of capacity T_cap: one 2-D copy per array.
extern "C" vc_status_t vc_quant_kv_stage_groups(const vc_shape_t* s, const uint32_t* host_kc, const uint16_t* host_ksz,
                                                const uint32_t* host_vc, const uint16_t* host_vsz, int32_t host_ng,
                                                int32_t g0, int32_t g1, int32_t T_cap, uint32_t* kc, uint16_t* ksz,
                                                uint32_t* vc, uint16_t* vsz, vc_stream_t stream) {
  vc_status_t st = check_shape(s, true);
  if (st != VC_OK) return st;
  VC_REQUIRE(host_kc && host_ksz && host_vc && host_vsz && kc && ksz && vc && vsz, "NULL pointer");
  VC_REQUIRE(T_cap >= 0 && T_cap % kGroup == 0, "T_cap must be a non-negative multiple of 32 (got %d)", T_cap);
  const int NG = T_cap / kGroup;
  VC_REQUIRE(0 <= g0 && g0 <= g1 && g1 <= host_ng && g1 <= NG, "need 0 <= g0 <= g1 <= min(host_ng, T_cap/32)");
  if (g0 == g1) return VC_OK;
  for (const void* p : {static_cast<const void*>(host_kc), static_cast<const void*>(host_ksz),
                        static_cast<const void*>(host_vc), static_cast<const void*>(host_vsz)}) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess || at.type != cudaMemoryTypeHost) {
      cudaGetLastError();
      VC_FAIL(VC_ERR_INVALID_ARG, "the host store must be pinned host memory (cudaHostAlloc / pin_memory)");
    }
  }
  const size_t rows = static_cast<size_t>(s->B) * s->Hkv;
  const size_t code_g = static_cast<size_t>(s->d) * s->bits * 4;    // bytes of one group's codes
  const size_t meta_g = static_cast<size_t>(s->d) * 4;              // bytes of one group's metadata
  auto cs = reinterpret_cast<cudaStream_t>(stream);
  auto copy2d = [&](void* dst, const void* src, size_t gb) -> cudaError_t {
    return cudaMemcpy2DAsync(static_cast<char*>(dst) + g0 * gb, NG * gb, static_cast<const char*>(src) + g0 * gb,
                             static_cast<size_t>(host_ng) * gb, static_cast<size_t>(g1 - g0) * gb, rows,
                             cudaMemcpyHostToDevice, cs);
  };
  VC_CUDA_CHECK(copy2d(kc, host_kc, code_g));
  VC_CUDA_CHECK(copy2d(ksz, host_ksz, meta_g));
  VC_CUDA_CHECK(copy2d(vc, host_vc, code_g));
  VC_CUDA_CHECK(copy2d(vsz, host_vsz, meta_g));
  return VC_OK;
}

extern "C" vc_status_t vc_quant_kv_device_status(uint32_t* status) {
  VC_REQUIRE(status, "status is NULL");
  VC_CUDA_CHECK(cudaDeviceSynchronize());
  uint32_t v = 0, zero = 0;
  VC_CUDA_CHECK(cudaMemcpyFromSymbol(&v, g_quant_status, sizeof(v)));
  VC_CUDA_CHECK(cudaMemcpyToSymbol(g_quant_status, &zero, sizeof(zero)));
  *status = v;
  return VC_OK;
}
