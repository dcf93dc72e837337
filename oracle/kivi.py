"""KIVI-style quantiser of the draft KV cache (oracle).

VeriCache drafts with a compressed KV cache and names KIVI among the
quantisation methods its compressor interface takes (VeriCache, Technical
Summary, Architecture Support).  The recipe, step by step, for one group of
32 bf16 values x (widened exactly to fp32):

1. mn = min(x), mx = max(x)                 (b = 2, 4 or 8)
2. s32 = (mx - mn) / (2^b - 1)             fp32, correctly rounded
3. s = fp16(s32), z = fp16(mn)             round to nearest even
4. code = clamp(rint((x - float(z)) / float(s)), 0, 2^b - 1)
   (each of the subtract and the divide is one rounded fp32 operation; rint
   rounds half to even); if s == 0 every code is 0
5. dequantised value x^ = fma(code, s, z) in fp32 (one rounding)

Keys form their groups along 32 consecutive tokens of one channel; values
along 32 consecutive channels of one token.

Packed layout (the library's format; written out from the rules next to
the packing functions below).  Per (request, KV head) and group of 32
tokens:

* K codes uint32 [B, Hkv, T/32, d*b] and V codes uint32 [B, Hkv, T/32, d*b]:
  32 lanes x d*b/32 words, each code a b-bit field at a position given by its
  token and channel (K and V use different maps); no field crosses bit 31.
* K meta fp16 [B, Hkv, T/32, 2, d]: scales of the group's channels, then zeros.
* V meta fp16 [B, Hkv, T/32, d/32, 2, 32]: per channel group, the 32 tokens'
  scales, then zeros, tokens in a fixed permuted order.

Numbers are numpy arrays.  bf16 inputs are uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np

GROUP = 32


def _bf16_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def quantize_groups(x: np.ndarray, bits: int):
    """Quantise groups laid out along the LAST axis (length 32).

    x: fp32 array [..., 32].  Returns (codes uint8 [..., 32], scale fp16 [...],
    zero fp16 [...]).  Steps 1-4 of the recipe above, in that order.
    """
    assert x.dtype == np.float32 and x.shape[-1] == GROUP
    qmax = (1 << bits) - 1
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    s32 = (mx - mn) / np.float32(qmax)                 # fp32 subtract, fp32 divide
    s = s32.astype(np.float16)                          # RNE
    z = mn.astype(np.float16)                           # RNE
    sf = s.astype(np.float32)[..., None]
    zf = z.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        diff = x - zf                                   # one fp32 rounding
        ratio = diff / sf                               # one fp32 rounding
        r = np.rint(ratio)                              # half to even
    r = np.where(sf == 0, np.float32(0), r)
    codes = np.clip(r, 0, qmax).astype(np.uint8)
    return codes, s, z


def dequantize(codes, scale, zero):
    """x^ = fma(code, s, z) in fp32.

    code*s is exact in fp64 (code < 16, s has 11 significant bits), and so is
    adding z (both are multiples of 2^-24 well inside 2^53), so one cast of
    the fp64 sum to fp32 is exactly one rounding: the fused multiply-add.
    """
    exact = codes.astype(np.float64) * scale.astype(np.float64) + zero.astype(np.float64)
    return exact.astype(np.float32)


def quantize_kv(K, V, bits: int):
    """Quantise a [B, Hkv, T, d] bf16 K/V pair (T a multiple of 32).

    Returns the unpacked codes and metadata in "logical" form:
    kcode uint8 [B,Hkv,T,d], kscale/kzero fp16 [B,Hkv,T/32,d],
    vcode uint8 [B,Hkv,T,d], vscale/vzero fp16 [B,Hkv,T,d/32].
    """
    Kf = _bf16_to_f32(K)
    Vf = _bf16_to_f32(V)
    B, H, T, d = Kf.shape
    assert T % GROUP == 0 and d % GROUP == 0
    # keys: groups of 32 tokens of one channel -> move the token axis last
    kg = Kf.reshape(B, H, T // GROUP, GROUP, d).transpose(0, 1, 2, 4, 3)
    kc, ks, kz = quantize_groups(np.ascontiguousarray(kg), bits)      # [B,H,G,d,32]
    kcode = kc.transpose(0, 1, 2, 4, 3).reshape(B, H, T, d)
    # values: groups of 32 channels of one token
    vg = Vf.reshape(B, H, T, d // GROUP, GROUP)
    vc, vs, vz = quantize_groups(np.ascontiguousarray(vg), bits)      # [B,H,T,d/32,32]
    vcode = vc.reshape(B, H, T, d)
    return kcode, ks, kz, vcode, vs, vz


def dequantize_kv(kcode, kscale, kzero, vcode, vscale, vzero):
    """Logical codes + metadata -> fp32 K^, V^ [B, Hkv, T, d]."""
    B, H, T, d = kcode.shape
    ks = np.repeat(kscale, GROUP, axis=2)              # [B,H,T,d]
    kz = np.repeat(kzero, GROUP, axis=2)
    Kh = dequantize(kcode, ks, kz)
    vs = np.repeat(vscale, GROUP, axis=3)              # [B,H,T,d]
    vz = np.repeat(vzero, GROUP, axis=3)
    Vh = dequantize(vcode, vs, vz)
    return Kh, Vh


# ------------------------------------------------------------ packed layout
#
# The bit placement below is this library's own format (the quantiser fixes
# only the codes and the fp16 scale/zero).  It follows the register fragments
# of the 16x8x16 half-precision tensor-core product that consumes it, so that a
# lane finds each pair of codes it feeds to one operand register 16 bits apart
# in one word.  Written out per group of 32 tokens; d channels, b bits.

def _field_pos(bits: int, u: int, r: int, e: int) -> int:
    """Lowest bit of a field.  b = 2: slot (u, r, e) starts at 16e + 4u + 2(1 - r).
    b = 4: slot (u, e) starts at 16e + 4u; b = 8: slot (u, e) at 16e + 8u (r
    unused for b = 4, 8).  The e = 1 field of a slot sits exactly 16 bits above
    its e = 0 field, in the high half-word."""
    if bits == 2:
        return 16 * e + 4 * u + 2 * (1 - r)
    return 16 * e + bits * u


def _word_index(L: int, w: int) -> int:
    """Word w of lane L sits at (w // 4) * 128 + 4 L + w % 4 within the group."""
    return (w // 4) * 128 + 4 * L + w % 4


def _slot(bits: int, i: int, r: int):
    """Fragment index i of a lane (and its r) -> (word, u) of its field.
    b = 2: word i // 4, u = i % 4.  b = 4, 8: i2 = 2i + r, and a word holds
    32 / (2b) slots: word i2 // (16 / b), u = i2 % (16 / b)."""
    if bits == 2:
        return i // 4, i % 4
    i2 = 2 * i + r
    per = 16 // bits
    return i2 // per, i2 % per


def _k_fields(d: int, bits: int):
    """(word index, field start, token, channel) of every K code of one group.

    Lane L = 4a + c holds tokens 4a + j (j < 4) and channels (d/4) c + 4k + 2r + e
    (k < d/16, r, e < 2); its fragment index is i = j*(d/16) + k."""
    KS = d // 16
    rows = []
    for L in range(32):
        a, c = divmod(L, 4)
        for j in range(4):
            for k in range(KS):
                for r in range(2):
                    for e in range(2):
                        w, u = _slot(bits, j * KS + k, r)
                        rows.append((_word_index(L, w), _field_pos(bits, u, r, e),
                                     4 * a + j, (d // 4) * c + 4 * k + 2 * r + e))
    return np.array(rows, dtype=np.int64)


def _v_fields(d: int, bits: int):
    """(word index, field start, token, channel) of every V code of one group.

    Lane L = 4a + c holds tokens 8c + 4e + 2s + r (s, r, e < 2) and channels
    8n + a (n < d/8); its fragment index is i = s*(d/8) + n."""
    NT = d // 8
    rows = []
    for L in range(32):
        a, c = divmod(L, 4)
        for s in range(2):
            for n in range(NT):
                for r in range(2):
                    for e in range(2):
                        w, u = _slot(bits, s * NT + n, r)
                        rows.append((_word_index(L, w), _field_pos(bits, u, r, e),
                                     8 * c + 4 * e + 2 * s + r, 8 * n + a))
    return np.array(rows, dtype=np.int64)


def _pack(code: np.ndarray, bits: int, fields) -> np.ndarray:
    """Logical codes uint8 [B,H,T,d] -> words uint32 [B,H,T/32,d*b]."""
    B, H, T, d = code.shape
    c = code.reshape(B, H, T // GROUP, GROUP, d)
    order = np.argsort(fields[:, 0], kind="stable")          # group fields by word
    f = fields[order]
    vals = c[..., f[:, 2], f[:, 3]]                          # [B,H,NG,F]
    placed = vals.astype(np.uint64) << f[:, 1].astype(np.uint64)
    n_words = d * bits
    per = f.shape[0] // n_words
    words = np.bitwise_or.reduce(placed.reshape(B, H, T // GROUP, n_words, per), axis=-1)
    return words.astype(np.uint32)


def _unpack(words: np.ndarray, bits: int, d: int, fields) -> np.ndarray:
    B, H, NG, n_words = words.shape
    assert n_words == d * bits
    w = words[..., fields[:, 0]].astype(np.uint64)           # [B,H,NG,F]
    vals = ((w >> fields[:, 1].astype(np.uint64)) & np.uint64((1 << bits) - 1)).astype(np.uint8)
    code = np.zeros((B, H, NG, GROUP, d), np.uint8)
    code[..., fields[:, 2], fields[:, 3]] = vals
    return code.reshape(B, H, NG * GROUP, d)


def pack_kcodes(code, bits: int):
    """K codes uint8 [B,H,T,d] -> words uint32 [B,H,T/32,d*b]."""
    return _pack(code, bits, _k_fields(code.shape[-1], bits))


def unpack_kcodes(words, bits: int, d: int):
    return _unpack(words, bits, d, _k_fields(d, bits))


def pack_vcodes(code, bits: int):
    """V codes uint8 [B,H,T,d] -> words uint32 [B,H,T/32,d*b]."""
    return _pack(code, bits, _v_fields(code.shape[-1], bits))


def unpack_vcodes(words, bits: int, d: int):
    return _unpack(words, bits, d, _v_fields(d, bits))


def pack_kmeta(kscale, kzero):
    """fp16 [B,H,T/32,d] x2 -> fp16 [B,H,T/32,2,d] (scales, then zeros)."""
    return np.ascontiguousarray(np.stack([kscale, kzero], axis=-2))


def unpack_kmeta(ksz):
    return ksz[..., 0, :], ksz[..., 1, :]


def _vmeta_token_of_entry():
    """Entry p = 8c + 4s + 2r + e of a 32-entry row holds token 8c + 4e + 2s + r."""
    p = np.arange(GROUP)
    c, s, r, e = p // 8, (p // 4) % 2, (p // 2) % 2, p % 2
    return 8 * c + 4 * e + 2 * s + r


def pack_vmeta(vscale, vzero):
    """fp16 [B,H,T,d/32] x2 -> fp16 [B,H,T/32,d/32,2,32]."""
    B, H, T, NC = vscale.shape
    m = np.stack([vscale, vzero], axis=-1).reshape(B, H, T // GROUP, GROUP, NC, 2)
    m = m.transpose(0, 1, 2, 4, 5, 3)                        # [B,H,NG,NC,2,32 tokens]
    return np.ascontiguousarray(m[..., _vmeta_token_of_entry()])


def unpack_vmeta(vsz):
    """fp16 [B,H,T/32,d/32,2,32] -> (scale, zero) fp16 [B,H,T,d/32]."""
    B, H, NG, NC, _, _ = vsz.shape
    m = np.empty_like(vsz)
    m[..., _vmeta_token_of_entry()] = vsz                    # back to token order
    m = m.transpose(0, 1, 2, 5, 3, 4).reshape(B, H, NG * GROUP, NC, 2)
    return m[..., 0], m[..., 1]


def quant_pack(K, V, bits: int):
    """bf16 K/V [B,Hkv,T,d] -> packed (kc, ksz, vc, vsz) in the library layout."""
    kcode, ks, kz, vcode, vs, vz = quantize_kv(K, V, bits)
    return (pack_kcodes(kcode, bits), pack_kmeta(ks, kz),
            pack_vcodes(vcode, bits), pack_vmeta(vs, vz))


def unpack_dequant(kc, ksz, vc, vsz, bits: int, d: int, T: int | None = None):
    """Packed cache -> fp32 K^, V^ [B,Hkv,T,d] (first T tokens)."""
    kcode = unpack_kcodes(kc, bits, d)
    vcode = unpack_vcodes(vc, bits, d)
    ks, kz = unpack_kmeta(ksz)
    vs, vz = unpack_vmeta(vsz)
    Kh, Vh = dequantize_kv(kcode, ks, kz, vcode, vs, vz)
    if T is not None:
        Kh, Vh = Kh[:, :, :T], Vh[:, :, :T]
    return Kh, Vh
