"""vc_accept on the GPU vs the oracle: bit-exact argmax, accepted length, next token."""
import json
import os

import numpy as np
import pytest
import torch

import synth
from oracle import accept as oacc

pytestmark = pytest.mark.gpu

GOLD = os.path.join(os.path.dirname(__file__), "golden", "accept_cases.json")


@pytest.fixture(scope="module")
def vc():
    from verify_compressed_kv_gb300 import _lib
    return _lib


def run_accept(vc, logits, draft):
    from gpu_util import dev, zeros_bytes
    B, R, V = logits.shape
    k = R - 1
    lg = dev(np.ascontiguousarray(logits, np.float32))
    dr = dev(np.ascontiguousarray(draft, np.int32).reshape(B, k)) if k > 0 else None
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    am = torch.empty((B, R), dtype=torch.int32, device="cuda")
    wsb = vc.vc_accept_workspace_size(B, k, V)
    ws = zeros_bytes(wsb)
    vc.vc_accept(B, k, V, lg, dr, n, nxt, am, ws, wsb)
    torch.cuda.synchronize()
    return n.cpu().numpy(), nxt.cpu().numpy(), am.cpu().numpy(), ws


@pytest.mark.parametrize("case", json.load(open(GOLD))["cases"], ids=lambda c: c["name"])
def test_golden(vc, case):
    logits = np.asarray(case["logits"], np.float32)[None]
    draft = np.asarray(case["draft"], np.int32).reshape(1, -1)
    n, nxt, am, _ = run_accept(vc, logits, draft)
    assert n[0] == case["n_acc"] and nxt[0] == case["next"] and am[0].tolist() == case["argmax"]


@pytest.mark.parametrize("B,k,V", [(1, 4, 1024), (3, 7, 1001), (8, 16, 32768), (2, 0, 77), (5, 3, 6),
                                   (2, 63, 500),     # the largest draft: 64 rows per request
                                   (3, 5, 1)])       # a one-token vocabulary
def test_random_with_ties(vc, B, k, V):
    rng = np.random.default_rng(B * 100 + V)
    logits = rng.integers(-4, 5, size=(B, k + 1, V)).astype(np.float32)   # many exact ties
    a = oacc.argmax_rows(logits)
    draft = np.where(rng.random((B, k)) < 0.8, a[:, :k], (a[:, :k] + 1) % V).astype(np.int32)
    n, nxt, am, ws = run_accept(vc, logits, draft)
    on, onx, oam = oacc.accept(logits, draft)
    assert np.array_equal(am, oam) and np.array_equal(n, on) and np.array_equal(nxt, onx)
    # the per-request arrival counters (the first 4*B bytes) are left at zero
    assert int(ws[:4 * B].count_nonzero()) == 0


@pytest.mark.parametrize("name", ["tiny", "mistral", "qwen", "llama", "stagger"])
def test_workload_logits(vc, name):
    w = synth.get(name)
    logits, drafts, L = synth.logits_and_drafts(w, rnd=0)
    n, nxt, am, _ = run_accept(vc, logits, drafts)
    on, onx, oam = oacc.accept(logits, drafts)
    assert np.array_equal(am, oam)
    assert np.array_equal(n, on) and np.array_equal(nxt, onx)
    assert np.array_equal(n, L)         # the generator's intended lengths are realised


def test_workspace_reuse_and_max_at_ends(vc):
    from gpu_util import dev, zeros_bytes
    B, k, V = 4, 5, 40000
    rng = np.random.default_rng(0)
    wsb = vc.vc_accept_workspace_size(B, k, V)
    ws = zeros_bytes(wsb)
    for rep in range(3):
        logits = rng.standard_normal((B, k + 1, V)).astype(np.float32)
        logits[0, 0, V - 1] = 100.0        # maximum at the last index
        logits[1, 2, 0] = 100.0            # maximum at the first index
        draft = rng.integers(0, V, size=(B, k)).astype(np.int32)
        draft[0, 0] = V - 1
        lg, dr = dev(logits), dev(draft)
        n = torch.empty(B, dtype=torch.int32, device="cuda")
        nxt = torch.empty(B, dtype=torch.int32, device="cuda")
        vc.vc_accept(B, k, V, lg, dr, n, nxt, None, ws, wsb)
        on, onx, _ = oacc.accept(logits, draft)
        assert np.array_equal(n.cpu().numpy(), on) and np.array_equal(nxt.cpu().numpy(), onx)
    assert int(ws[:4 * B].count_nonzero()) == 0


def test_one_workspace_for_changing_k_and_V(vc):
    """Calls with different draft lengths and vocabularies share one workspace
    (sized for the largest need): the arrival counters sit at a fixed place."""
    from gpu_util import dev, zeros_bytes
    B = 4
    shapes = [(16, 32768), (60, 32768), (3, 1001), (60, 128256), (16, 32768), (1, 77)]
    wsb = max(vc.vc_accept_workspace_size(B, k, V) for k, V in shapes)
    ws = zeros_bytes(wsb)
    rng = np.random.default_rng(5)
    for k, V in shapes:
        logits = rng.standard_normal((B, k + 1, V)).astype(np.float32)
        draft = rng.integers(0, V, size=(B, k)).astype(np.int32)
        L = rng.integers(0, k + 1, size=B)
        for b in range(B):
            for i in range(L[b]):
                logits[b, i, draft[b, i]] += 8.0
        n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        vc.vc_accept(B, k, V, dev(logits), dev(draft), n, nxt, None, ws, wsb)
        torch.cuda.synchronize()
        want_n, want_next, _ = oacc.accept(logits, draft)
        assert np.array_equal(n.cpu().numpy(), want_n), (k, V)
        assert np.array_equal(nxt.cpu().numpy(), want_next), (k, V)


def test_argument_errors(vc):
    with pytest.raises(vc.VcError) as e:
        vc.vc_accept(1, 2, 10, None, None, None, None, None, None, 0)
    assert e.value.status == 1
    with pytest.raises(vc.VcError) as e:
        lg = torch.zeros((1, 3, 10), device="cuda")
        dr = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
        o = torch.zeros(1, dtype=torch.int32, device="cuda")
        vc.vc_accept(1, 2, 10, lg, dr, o, o, None, torch.zeros(4, dtype=torch.uint8, device="cuda"), 4)
    assert e.value.status == 5
