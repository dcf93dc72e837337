"""ctypes binding of include/vc.h: same names, argument marshalling only.

Every function takes torch tensors (or raw integer addresses) and forwards
their data pointers to the C ABI; streams are ``torch.cuda.Stream`` objects
(or None for the current stream).  A non-zero status raises ``VcError`` with
the library's one-line reason.  Nothing here computes: if the shared
libraries are missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_size_t, c_uint32, c_void_p

LIBDIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib")
LIB_NAMES = ("vc_core", "vc_quant_kv", "vc_draft_attn", "vc_verify_attn", "vc_accept")


class VcError(RuntimeError):
    def __init__(self, status: int, fn: str, reason: str):
        super().__init__(f"{fn}: status {status} ({STATUS.get(status, '?')}): {reason}")
        self.status = status


STATUS = {0: "VC_OK", 1: "VC_ERR_INVALID_ARG", 2: "VC_ERR_UNSUPPORTED", 3: "VC_ERR_CUDA",
          4: "VC_ERR_TIMEOUT", 5: "VC_ERR_WORKSPACE", 6: "VC_ERR_CAPACITY"}


class vc_shape_t(ctypes.Structure):
    _fields_ = [("B", c_int32), ("Hq", c_int32), ("Hkv", c_int32), ("d", c_int32),
                ("k", c_int32), ("bits", c_int32), ("softmax_scale", c_float)]


def shape(B, Hq, Hkv, d, k=0, bits=2, softmax_scale=1.0) -> vc_shape_t:
    return vc_shape_t(int(B), int(Hq), int(Hkv), int(d), int(k), int(bits), float(softmax_scale))


def _load():
    libs = {}
    for name in LIB_NAMES:
        path = os.path.join(LIBDIR, f"lib{name}.so")
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build the CUDA libraries first "
                              "(python -m verify_compressed_kv_gb300.build)")
        # RTLD_GLOBAL for the core so the others resolve its symbols once
        mode = ctypes.RTLD_GLOBAL if name == "vc_core" else ctypes.RTLD_LOCAL
        libs[name] = ctypes.CDLL(path, mode=mode)
    return libs


_LIBS = _load()
_core = _LIBS["vc_core"]
_core.vc_status_str.restype = ctypes.c_char_p
_core.vc_status_str.argtypes = [c_int32]
_core.vc_last_error.restype = ctypes.c_char_p
_core.vc_last_error.argtypes = []

P = c_void_p
S = POINTER(vc_shape_t)
I32 = c_int32
SZ = c_size_t

_SIGS = {
    "vc_quant_kv": {
        "vc_quant_packed_bytes": [S, I32, POINTER(c_size_t), POINTER(c_size_t), POINTER(c_size_t), POINTER(c_size_t)],
        "vc_quant_kv_pack": [S, I32, I32, P, P, P, P, P, P, P],
        "vc_quant_kv_unpack": [S, I32, I32, P, P, P, P, P, P, P],
        "vc_quant_kv_append": [S, P, P, P, P, P, P, I32, P, P, P, P, P, I32, P],
        "vc_token_score_workspace_size": [S, I32, I32, POINTER(c_size_t)],
        "vc_token_score": [S, I32, I32, P, P, P, P, SZ, P],
        "vc_token_select_workspace_size": [I32, I32, I32, POINTER(c_size_t)],
        "vc_token_select": [I32, I32, I32, P, I32, I32, I32, P, P, SZ, P],
        "vc_gather_kv": [S, I32, I32, P, P, P, P, P, P],
        "vc_quant_kv_stage_groups": [S, P, P, P, P, I32, I32, I32, I32, P, P, P, P, P],
        "vc_quant_kv_device_status": [POINTER(c_uint32)],
    },
    "vc_draft_attn": {
        "vc_draft_attn_workspace_size": [S, I32, POINTER(c_size_t)],
        "vc_draft_attn": [S, P, P, P, P, P, P, P, P, I32, I32, P, P, P, I32, I32, P, P, SZ, c_uint32, P],
        "vc_draft_attn_device_status": [POINTER(c_uint32)],
        "vc_draft_attn_test_hooks": [ctypes.c_int64, I32],
        "vc_draft_attn_partition": [S, I32, I32, POINTER(c_int32), P, I32, POINTER(c_int32)],
    },
    "vc_verify_attn": {
        "vc_verify_attn_workspace_size": [S, I32, POINTER(c_size_t)],
        "vc_verify_attn_parts": [S, I32, POINTER(c_int32)],
        "vc_verify_attn_chunk": [S, P, P, I32, I32, P, I32, I32, P, SZ, P],
        "vc_verify_attn_finish": [S, P, P, P, I32, I32, P, P, SZ, P],
        "vc_verify_pipeline_create": [I32, POINTER(c_void_p)],
        "vc_verify_pipeline_destroy": [P],
        "vc_verify_prefetch": [P, S, P, I32, I32, I32, P, P],
        "vc_verify_attn_streamed": [P, S, P, P, I32, I32, I32, P, P, P, P, P, I32, P, SZ, P, P],
        "vc_verify_commit": [S, P, P, P, P, P, I32, I32, P],
        "vc_verify_attn_device_status": [POINTER(c_uint32)],
    },
    "vc_accept": {
        "vc_accept_workspace_size": [I32, I32, I32, POINTER(c_size_t)],
        "vc_accept": [I32, I32, I32, P, P, P, P, P, P, SZ, P],
        "vc_accept_noalloc": [I32, I32, I32, P, P, P, P, P, P],
    },
}

_FUNCS = {}
for _lib, _fns in _SIGS.items():
    for _fn, _argt in _fns.items():
        f = getattr(_LIBS[_lib], _fn)
        f.argtypes = _argt
        f.restype = c_int32
        _FUNCS[_fn] = f


def exported_symbols():
    """Every symbol include/vc.h declares, with the library that exports it."""
    out = {"vc_status_str": "vc_core", "vc_last_error": "vc_core"}
    for lib, fns in _SIGS.items():
        for fn in fns:
            out[fn] = lib
    return out


def loaded_paths():
    return [os.path.join(LIBDIR, f"lib{n}.so") for n in LIB_NAMES]


def _call(fn, *args):
    st = _FUNCS[fn](*args)
    if st != 0:
        raise VcError(st, fn, _core.vc_last_error().decode(errors="replace"))


def _ptr(x):
    """Tensor / int / None -> address."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def status_str(st: int) -> str:
    return _core.vc_status_str(st).decode()


# ------------------------------------------------------------ vc_quant_kv

def vc_quant_packed_bytes(s: vc_shape_t, T_cap: int):
    a, b, c, d = c_size_t(), c_size_t(), c_size_t(), c_size_t()
    _call("vc_quant_packed_bytes", ctypes.byref(s), T_cap, ctypes.byref(a), ctypes.byref(b),
          ctypes.byref(c), ctypes.byref(d))
    return a.value, b.value, c.value, d.value


def vc_quant_kv_pack(s, T, T_cap, K, V, kc, ksz, vc, vsz, stream=None):
    _call("vc_quant_kv_pack", ctypes.byref(s), T, T_cap, _ptr(K), _ptr(V), _ptr(kc), _ptr(ksz),
          _ptr(vc), _ptr(vsz), _stream(stream))


def vc_quant_kv_unpack(s, T, T_cap, kc, ksz, vc, vsz, K_hat, V_hat, stream=None):
    _call("vc_quant_kv_unpack", ctypes.byref(s), T, T_cap, _ptr(kc), _ptr(ksz), _ptr(vc), _ptr(vsz),
          _ptr(K_hat), _ptr(V_hat), _stream(stream))


def vc_quant_kv_append(s, k_new, v_new, n_acc, tail_k, tail_v, tail_len, tail_cap, kc, ksz, vc, vsz,
                       packed_len, T_cap, stream=None):
    _call("vc_quant_kv_append", ctypes.byref(s), _ptr(k_new), _ptr(v_new), _ptr(n_acc), _ptr(tail_k),
          _ptr(tail_v), _ptr(tail_len), tail_cap, _ptr(kc), _ptr(ksz), _ptr(vc), _ptr(vsz),
          _ptr(packed_len), T_cap, _stream(stream))


def vc_token_score_workspace_size(s, T, n_obs):
    n = c_size_t()
    _call("vc_token_score_workspace_size", ctypes.byref(s), T, n_obs, ctypes.byref(n))
    return n.value


def vc_token_score(s, T, n_obs, q_obs, K, score, ws, ws_bytes, stream=None):
    _call("vc_token_score", ctypes.byref(s), T, n_obs, _ptr(q_obs), _ptr(K), _ptr(score), _ptr(ws),
          ws_bytes, _stream(stream))


def vc_token_select_workspace_size(B, Hkv, T):
    n = c_size_t()
    _call("vc_token_select_workspace_size", B, Hkv, T, ctypes.byref(n))
    return n.value


def vc_token_select(B, Hkv, T, score, keep, keep_last, pool, idx, ws, ws_bytes, stream=None):
    _call("vc_token_select", B, Hkv, T, _ptr(score), keep, keep_last, pool, _ptr(idx), _ptr(ws),
          ws_bytes, _stream(stream))


def vc_gather_kv(s, T, keep, idx, K, V, K_out, V_out, stream=None):
    _call("vc_gather_kv", ctypes.byref(s), T, keep, _ptr(idx), _ptr(K), _ptr(V), _ptr(K_out),
          _ptr(V_out), _stream(stream))


def vc_quant_kv_stage_groups(s, host_kc, host_ksz, host_vc, host_vsz, host_ng, g0, g1, T_cap, kc, ksz, vc, vsz,
                             stream=None):
    _call("vc_quant_kv_stage_groups", ctypes.byref(s), _ptr(host_kc), _ptr(host_ksz), _ptr(host_vc), _ptr(host_vsz),
          host_ng, g0, g1, T_cap, _ptr(kc), _ptr(ksz), _ptr(vc), _ptr(vsz), _stream(stream))


def vc_quant_kv_device_status() -> int:
    v = c_uint32()
    _call("vc_quant_kv_device_status", ctypes.byref(v))
    return v.value


# ------------------------------------------------------------ vc_draft_attn

def vc_draft_attn_workspace_size(s, max_packed):
    n = c_size_t()
    _call("vc_draft_attn_workspace_size", ctypes.byref(s), max_packed, ctypes.byref(n))
    return n.value


VC_DRAFT_CHAINED = 1


def vc_draft_attn(s, q, k_cur, v_cur, kc, ksz, vc, vsz, packed_len, max_packed, T_cap, tail_k, tail_v,
                  tail_len, tail_cap, step, out, ws, ws_bytes, stream=None, flags=0):
    """`flags` is the C call's argument before the stream (0 or VC_DRAFT_CHAINED)."""
    _call("vc_draft_attn", ctypes.byref(s), _ptr(q), _ptr(k_cur), _ptr(v_cur), _ptr(kc), _ptr(ksz),
          _ptr(vc), _ptr(vsz), _ptr(packed_len), max_packed, T_cap, _ptr(tail_k), _ptr(tail_v),
          _ptr(tail_len), tail_cap, step, _ptr(out), _ptr(ws), ws_bytes, int(flags), _stream(stream))


def vc_draft_attn_partition(s, max_packed, slots):
    """(n_stream, lo [n_stream + 1] int list, max_parts) of the launch's stream-K partition."""
    n, mp = c_int32(), c_int32()
    cap = 513
    buf = (c_int32 * cap)()
    _call("vc_draft_attn_partition", ctypes.byref(s), max_packed, slots, ctypes.byref(n), ctypes.cast(buf, c_void_p),
          cap, ctypes.byref(mp))
    return n.value, list(buf[:n.value + 1]), mp.value


def vc_draft_attn_test_hooks(wait_cycles: int, withhold_first_stage: int) -> None:
    _call("vc_draft_attn_test_hooks", int(wait_cycles), int(withhold_first_stage))


def vc_draft_attn_device_status() -> int:
    v = c_uint32()
    _call("vc_draft_attn_device_status", ctypes.byref(v))
    return v.value


# ------------------------------------------------------------ vc_verify_attn

def vc_verify_attn_workspace_size(s, parts_per_chunk):
    n = c_size_t()
    _call("vc_verify_attn_workspace_size", ctypes.byref(s), parts_per_chunk, ctypes.byref(n))
    return n.value


def vc_verify_attn_parts(s, C):
    n = c_int32()
    _call("vc_verify_attn_parts", ctypes.byref(s), C, ctypes.byref(n))
    return n.value


def vc_verify_attn_chunk(s, q, kv_slot, C, chunk_start, prefix_len, parts, first, ws, ws_bytes, stream=None):
    _call("vc_verify_attn_chunk", ctypes.byref(s), _ptr(q), _ptr(kv_slot), C, chunk_start, _ptr(prefix_len),
          parts, int(first), _ptr(ws), ws_bytes, _stream(stream))


def vc_verify_attn_finish(s, q, k_new, v_new, parts, any_chunk, out, ws, ws_bytes, stream=None):
    _call("vc_verify_attn_finish", ctypes.byref(s), _ptr(q), _ptr(k_new), _ptr(v_new), parts,
          int(any_chunk), _ptr(out), _ptr(ws), ws_bytes, _stream(stream))


def vc_verify_pipeline_create(n_slots: int) -> int:
    h = c_void_p()
    _call("vc_verify_pipeline_create", n_slots, ctypes.byref(h))
    return h.value


def vc_verify_pipeline_destroy(h: int):
    _call("vc_verify_pipeline_destroy", h)


def vc_verify_prefetch(h, s, host_kv, C, max_prefix, T_cap, dev_slots, copy_stream):
    _call("vc_verify_prefetch", h, ctypes.byref(s), _ptr(host_kv), C, max_prefix, T_cap, _ptr(dev_slots),
          _stream(copy_stream))


def vc_verify_attn_streamed(h, s, q, host_kv, C, max_prefix, T_cap, prefix_len, dev_slots, k_new, v_new, out,
                            parts, ws, ws_bytes, compute_stream, copy_stream):
    _call("vc_verify_attn_streamed", h, ctypes.byref(s), _ptr(q), _ptr(host_kv), C, max_prefix, T_cap,
          _ptr(prefix_len), _ptr(dev_slots), _ptr(k_new), _ptr(v_new), _ptr(out), parts, _ptr(ws),
          ws_bytes, _stream(compute_stream), _stream(copy_stream))


def vc_verify_commit(s, k_new, v_new, n_acc, prefix_len, host_kv, C, T_cap, stream=None):
    _call("vc_verify_commit", ctypes.byref(s), _ptr(k_new), _ptr(v_new), _ptr(n_acc), _ptr(prefix_len),
          _ptr(host_kv), C, T_cap, _stream(stream))


def vc_verify_attn_device_status() -> int:
    v = c_uint32()
    _call("vc_verify_attn_device_status", ctypes.byref(v))
    return v.value


# ------------------------------------------------------------ vc_accept

def vc_accept_workspace_size(B, k, V):
    n = c_size_t()
    _call("vc_accept_workspace_size", B, k, V, ctypes.byref(n))
    return n.value


def vc_accept(B, k, V, logits, draft, n_acc, next_tok, argmax, ws, ws_bytes, stream=None):
    _call("vc_accept", B, k, V, _ptr(logits), _ptr(draft), _ptr(n_acc), _ptr(next_tok), _ptr(argmax),
          _ptr(ws), ws_bytes, _stream(stream))


def vc_accept_noalloc(B, k, V, logits, draft, n_acc, next_tok, argmax, stream=None):
    _call("vc_accept_noalloc", B, k, V, _ptr(logits), _ptr(draft), _ptr(n_acc), _ptr(next_tok), _ptr(argmax),
          _stream(stream))
