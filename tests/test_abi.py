"""The C ABI without a GPU: every library loads, every symbol include/vc.h
declares is exported, and host-side argument checks return their status codes
before anything touches CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vc.h")


@pytest.fixture(scope="module")
def vc():
    libdir = os.path.join(ROOT, "verify_compressed_kv_gb300", "lib")
    names = ["vc_core", "vc_quant_kv", "vc_draft_attn", "vc_verify_attn", "vc_accept"]
    if not all(os.path.exists(os.path.join(libdir, f"lib{n}.so")) for n in names):
        from verify_compressed_kv_gb300 import build
        build.build(jobs=5)
    from verify_compressed_kv_gb300 import _lib
    return _lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vc_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_calls():
    fns = declared_functions()
    for must in ["vc_quant_kv_pack", "vc_quant_kv_append", "vc_token_score", "vc_token_select", "vc_gather_kv",
                 "vc_draft_attn", "vc_verify_attn_chunk", "vc_verify_attn_finish", "vc_verify_attn_streamed",
                 "vc_verify_commit", "vc_accept", "vc_status_str", "vc_last_error"]:
        assert must in fns


def test_every_declared_symbol_is_exported(vc):
    exported = vc.exported_symbols()
    for fn in declared_functions():
        assert fn in exported, f"{fn} declared in vc.h but not bound"
        lib = ctypes.CDLL(os.path.join(vc.LIBDIR, f"lib{exported[fn]}.so"))
        assert hasattr(lib, fn), f"{fn} not exported by lib{exported[fn]}.so"


def test_binding_arity_matches_the_header(vc):
    """Every bound call passes as many arguments as vc.h declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decl = {m.group(1): m.group(2) for m in re.finditer(r"\b(vc_[a-z0-9_]+)\s*\(([^()]*)\)\s*;", text)}
    n = 0
    for lib, fns in vc._SIGS.items():
        for fn, argtypes in fns.items():
            params = decl[fn].strip()
            count = 0 if params in ("", "void") else params.count(",") + 1
            assert count == len(argtypes), f"{fn}: vc.h declares {count} parameters, the binding passes {len(argtypes)}"
            n += 1
    assert n >= 20


def test_status_strings(vc):
    assert vc.status_str(0) == "ok"
    assert "workspace" in vc.status_str(5)
    assert vc.status_str(99) == "unknown status"


def test_host_side_argument_checks(vc):
    s = vc.shape(1, 4, 1, 64, k=4, bits=4)
    with pytest.raises(vc.VcError) as e:
        vc.vc_accept(0, 4, 10, None, None, None, None, None, None, 0, stream=0)
    assert e.value.status == 1 and "B >= 1" in str(e.value)
    with pytest.raises(vc.VcError) as e:
        vc.vc_quant_packed_bytes(vc.shape(1, 4, 1, 96, bits=4), 64)
    assert e.value.status == 2
    with pytest.raises(vc.VcError) as e:
        vc.vc_quant_packed_bytes(vc.shape(1, 4, 1, 64, bits=3), 64)
    assert e.value.status == 2
    with pytest.raises(vc.VcError) as e:
        vc.vc_draft_attn_workspace_size(vc.shape(1, 12, 1, 64, bits=2), 64)   # G = 12
    assert e.value.status == 2
    with pytest.raises(vc.VcError) as e:
        vc.vc_verify_attn_workspace_size(vc.shape(1, 64, 1, 128, k=40), 1)    # 41 * 64 rows
    assert e.value.status == 2
    with pytest.raises(vc.VcError) as e:
        vc.vc_token_select(1, 1, 100, None, 10, 32, 7, None, None, 0, stream=0)   # keep_last > keep
    assert e.value.status == 1
    with pytest.raises(vc.VcError) as e:
        vc.vc_verify_attn_parts(s, 0)                                           # C = 0
    assert e.value.status == 1


def test_size_queries_match_the_layout(vc):
    s = vc.shape(8, 32, 8, 128, k=16, bits=2)
    kc, ksz, vcb, vsz = vc.vc_quant_packed_bytes(s, 32768)
    tok = 8 * 8 * 32768
    # codes d*b/8 bytes, key meta d*4/32, value meta (d/32)*4 per token per KV head
    assert (kc, vcb) == (tok * 32, tok * 32)
    assert (ksz, vsz) == (tok * 16, tok * 16)
    assert (kc + ksz + vcb + vsz) // tok == 96
    s4 = vc.shape(16, 40, 8, 128, k=32, bits=4)
    kc, ksz, vcb, vsz = vc.vc_quant_packed_bytes(s4, 16384)
    assert (kc + ksz + vcb + vsz) // (16 * 8 * 16384) == 160
    assert vc.vc_accept_workspace_size(8, 16, 32768) > 0


def test_misaligned_and_null_pointers_are_rejected_before_launch(vc):
    s = vc.shape(1, 4, 1, 64, k=2, bits=4)
    with pytest.raises(vc.VcError) as e:                      # logits not 16-byte aligned
        vc.vc_accept(1, 2, 16, 0x1004, 0x2000, 0x3000, 0x4000, None, 0x5000, 1 << 20, stream=0)
    assert e.value.status == 1 and "aligned" in str(e.value)
    with pytest.raises(vc.VcError) as e:
        vc.vc_quant_kv_pack(s, 64, 64, 0x1008, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, stream=0)
    assert e.value.status == 1 and "aligned" in str(e.value)
    with pytest.raises(vc.VcError) as e:
        vc.vc_quant_kv_pack(s, 48, 64, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, stream=0)   # T % 32
    assert e.value.status == 1
    with pytest.raises(vc.VcError) as e:
        vc.vc_gather_kv(s, 10, 4, None, 0x1000, 0x2000, 0x3000, 0x4000, stream=0)
    assert e.value.status == 1
    with pytest.raises(vc.VcError) as e:                      # k_cur without v_cur
        vc.vc_draft_attn(s, 0x1000, 0x2000, None, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 64, 64, 0x8000, 0x9000,
                         0xa000, 8, 0, 0xb000, 0xc000, 1 << 20, stream=0)
    assert e.value.status == 1
    with pytest.raises(vc.VcError) as e:                      # a flag bit the call does not know
        vc.vc_draft_attn(s, 0x1000, 0x2000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 64, 64, 0x8000, 0x9000,
                         0xa000, 8, 0, 0xb000, 0xc000, 1 << 20, stream=0, flags=2)
    assert e.value.status == 1 and "flags" in str(e.value)


def test_stage_groups_checks_ranges_before_any_copy(vc):
    s = vc.shape(2, 8, 2, 128, bits=2)
    args = (0x1000, 0x2000, 0x3000, 0x4000)
    dev = (0x5000, 0x6000, 0x7000, 0x8000)
    with pytest.raises(vc.VcError) as e:                     # g1 beyond the host store
        vc.vc_quant_kv_stage_groups(s, *args, 4, 0, 5, 1024, *dev, stream=0)
    assert e.value.status == 1
    with pytest.raises(vc.VcError) as e:                     # g1 beyond the device capacity
        vc.vc_quant_kv_stage_groups(s, *args, 64, 0, 40, 1024, *dev, stream=0)
    assert e.value.status == 1
    with pytest.raises(vc.VcError) as e:
        vc.vc_quant_kv_stage_groups(s, None, *args[1:], 4, 0, 1, 1024, *dev, stream=0)
    assert e.value.status == 1
    vc.vc_quant_kv_stage_groups(s, *args, 4, 2, 2, 1024, *dev, stream=0)   # empty range: nothing to do
