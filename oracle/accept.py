"""Acceptance rule (oracle).

VeriCache, Technical Summary, Core Algorithm, Acceptance (and the same
passage of the Korean translation): the drafted tokens are kept for as long
as they agree with the full-KV prediction; the first disagreement ends the
run; when every drafted token agrees, one more token from the full-KV pass
(the "bonus") is kept as well; the next round starts from the last kept token.

Reading of the page (it does not say what is emitted after a mismatch): the
full-KV prediction at the first mismatching position is always emitted.  When
every draft matches that is the page's bonus token; otherwise it is the
correction.  Both equal what greedy full-KV decoding would produce next, so
the output stays identical to full-KV decoding and each round makes at least
one token of progress.

Argmax ties go to the lowest vocabulary index (comparison with IEEE >, so
-0.0 and +0.0 tie).
"""
from __future__ import annotations

import numpy as np


def argmax_lowest(row: np.ndarray) -> int:
    """Index of the first (lowest) position holding the row's maximum."""
    best = 0
    for v in range(1, row.shape[0]):
        if row[v] > row[best]:
            best = v
    return best


def argmax_rows(logits: np.ndarray) -> np.ndarray:
    """Lowest-index argmax of every row: [..., V] -> int32 [...]."""
    m = logits.max(axis=-1, keepdims=True)
    hit = logits == m
    return hit.argmax(axis=-1).astype(np.int32)     # first True = lowest index


def accept(logits: np.ndarray, draft: np.ndarray):
    """logits fp32 [B, k+1, V], draft int32 [B, k] -> (n_acc, next_tok, argmax).

    a_i = argmax of row i; n = the first i < k with a_i != draft_i, else k;
    next = a_n.
    """
    B, R, V = logits.shape
    k = R - 1
    a = argmax_rows(logits)
    n_acc = np.empty(B, np.int32)
    nxt = np.empty(B, np.int32)
    for b in range(B):
        n = k
        for i in range(k):
            if a[b, i] != draft[b, i]:
                n = i
                break
        n_acc[b] = n
        nxt[b] = a[b, n]
    return n_acc, nxt, a
