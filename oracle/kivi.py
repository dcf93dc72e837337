"""KIVI-style quantiser of the draft KV cache (oracle).

VeriCache drafts with a compressed KV cache and names KIVI among the
quantisation methods its compressor interface takes (VeriCache, Technical
Summary, Architecture Support).  The recipe, step by step, for one group of
32 bf16 values x (widened exactly to fp32):

1. mn = min(x), mx = max(x)
2. s32 = (mx - mn) / (2^b - 1)             fp32, correctly rounded
3. s = fp16(s32), z = fp16(mn)             round to nearest even
4. code = clamp(rint((x - float(z)) / float(s)), 0, 2^b - 1)
   (each of the subtract and the divide is one rounded fp32 operation; rint
   rounds half to even); if s == 0 every code is 0
5. dequantised value x^ = fma(code, s, z) in fp32 (one rounding)

Keys form their groups along 32 consecutive tokens of one channel; values
along 32 consecutive channels of one token.

Packed layout (the library's format; the oracle writes it from this text):
W = d*b/32 32-bit words per token.

* K codes uint32 [B, Hkv, T/32, W, 32]: word (g, w, t) holds token 32g+t,
  channels w*(32/b) + j for j < 32/b, code j at bits [b*j, b*j+b).
* K meta fp16 [B, Hkv, T/32, d, 2]: (scale, zero) of channel c in group g.
* V codes uint32 [B, Hkv, T/32, W, 32]: same packing as K codes.
* V meta fp16 [B, Hkv, T/32, d/32, 32, 2]: (scale, zero) of token 32g+t over
  channels 32cg .. 32cg+31.

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

def pack_codes(code: np.ndarray, bits: int) -> np.ndarray:
    """Logical codes uint8 [B,H,T,d] -> words uint32 [B,H,T/32,W,32]."""
    B, H, T, d = code.shape
    per = 32 // bits
    W = d // per
    c = code.reshape(B, H, T // GROUP, GROUP, W, per).astype(np.uint32)
    words = np.zeros((B, H, T // GROUP, GROUP, W), np.uint32)
    for j in range(per):
        words |= c[..., j] << np.uint32(bits * j)
    return np.ascontiguousarray(words.transpose(0, 1, 2, 4, 3))


def unpack_codes(words: np.ndarray, bits: int, d: int) -> np.ndarray:
    """Words uint32 [B,H,T/32,W,32] -> logical codes uint8 [B,H,T,d]."""
    B, H, NG, W, _ = words.shape
    per = 32 // bits
    assert W * per == d
    w = words.transpose(0, 1, 2, 4, 3)                 # [B,H,NG,32,W]
    mask = np.uint32((1 << bits) - 1)
    parts = [((w >> np.uint32(bits * j)) & mask) for j in range(per)]
    c = np.stack(parts, axis=-1)                       # [B,H,NG,32,W,per]
    return c.reshape(B, H, NG * GROUP, d).astype(np.uint8)


def pack_kmeta(kscale, kzero):
    """fp16 [B,H,T/32,d] x2 -> fp16 [B,H,T/32,d,2]."""
    return np.ascontiguousarray(np.stack([kscale, kzero], axis=-1))


def pack_vmeta(vscale, vzero):
    """fp16 [B,H,T,d/32] x2 -> fp16 [B,H,T/32,d/32,32,2]."""
    B, H, T, NC = vscale.shape
    m = np.stack([vscale, vzero], axis=-1).reshape(B, H, T // GROUP, GROUP, NC, 2)
    return np.ascontiguousarray(m.transpose(0, 1, 2, 4, 3, 5))


def unpack_vmeta(vsz):
    """fp16 [B,H,T/32,d/32,32,2] -> (scale, zero) fp16 [B,H,T,d/32]."""
    B, H, NG, NC, _, _ = vsz.shape
    m = vsz.transpose(0, 1, 2, 4, 3, 5).reshape(B, H, NG * GROUP, NC, 2)
    return m[..., 0], m[..., 1]


def quant_pack(K, V, bits: int):
    """bf16 K/V [B,Hkv,T,d] -> packed (kc, ksz, vc, vsz) in the library layout."""
    kcode, ks, kz, vcode, vs, vz = quantize_kv(K, V, bits)
    return (pack_codes(kcode, bits), pack_kmeta(ks, kz),
            pack_codes(vcode, bits), pack_vmeta(vs, vz))


def unpack_dequant(kc, ksz, vc, vsz, bits: int, d: int, T: int | None = None):
    """Packed cache -> fp32 K^, V^ [B,Hkv,T,d] (first T tokens)."""
    kcode = unpack_codes(kc, bits, d)
    vcode = unpack_codes(vc, bits, d)
    ks, kz = ksz[..., 0], ksz[..., 1]
    vs, vz = unpack_vmeta(vsz)
    Kh, Vh = dequantize_kv(kcode, ks, kz, vcode, vs, vz)
    if T is not None:
        Kh, Vh = Kh[:, :, :T], Vh[:, :, :T]
    return Kh, Vh
