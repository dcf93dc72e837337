"""Pins for the oracle's acceptance rule: hand-built cases and a brute-force loop."""
import json
import os

import numpy as np
import pytest

from oracle import accept as acc

GOLD = os.path.join(os.path.dirname(__file__), "golden", "accept_cases.json")


@pytest.mark.parametrize("case", json.load(open(GOLD))["cases"], ids=lambda c: c["name"])
def test_hand_built(case):
    logits = np.asarray(case["logits"], np.float32)[None]
    draft = np.asarray(case["draft"], np.int32).reshape(1, -1)
    n, nxt, a = acc.accept(logits, draft)
    assert int(n[0]) == case["n_acc"]
    assert int(nxt[0]) == case["next"]
    assert a[0].tolist() == case["argmax"]


def test_vectorised_argmax_equals_scalar_scan():
    rng = np.random.default_rng(1)
    x = rng.integers(-3, 4, size=(300, 57)).astype(np.float32)      # many ties
    vec = acc.argmax_rows(x)
    for r in range(x.shape[0]):
        assert vec[r] == acc.argmax_lowest(x[r])
        # and it is a maximum with nothing equal before it
        assert x[r, vec[r]] == x[r].max() and np.all(x[r, :vec[r]] < x[r].max())


def test_random_rows_against_definition():
    rng = np.random.default_rng(2)
    B, k, V = 20, 6, 50
    logits = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    a = logits.argmax(-1)
    draft = np.where(rng.random((B, k)) < 0.7, a[:, :k], (a[:, :k] + 1) % V).astype(np.int32)
    n, nxt, _ = acc.accept(logits, draft)
    for b in range(B):
        agree = [int(a[b, i]) == int(draft[b, i]) for i in range(k)]
        want = agree.index(False) if False in agree else k
        assert n[b] == want and nxt[b] == a[b, want]
