"""Draft length (verification period) per request group.

VeriCache, Technical Summary, Key System Innovations (2), Extended Verification
Period: with a compressed-KV drafter the acceptance rate stays high over long
drafts, so each expensive full-KV verification can cover many draft tokens.
The pages give no rule for choosing the period; this module reads it as an
optimisation over measured quantities:

* acceptance: each draft token of a request is accepted (given all earlier
  ones were) with probability a, so the accepted length of a round with draft
  length k is min(N, k), P(N >= i) = a^i.  a is estimated from the observed
  accepted lengths, with rounds that accepted everything counted as censored:
  a = accepted tokens / (accepted tokens + rounds stopped by a mismatch);
* time: a round drafts k steps (t_step each, all layers) while the full KV of
  the round streams (t_copy, overlapped with drafting by prefetch or by
  staggering); verification needs the drafts, so its compute, which grows
  with the k + 1 rows (t_row per row), follows the drafting; then accept and
  commit (t_tail):  T(k) = max(k * t_step + (k + 1) * t_row, t_copy) + t_tail;
* tokens: B * (E[min(N, k)] + 1), E[min(N, k)] = sum_{i=1..k} a^i (the +1 is
  the bonus or correction token every round emits).

The controller picks the k in [k_min, k_max] that maximises tokens / T(k).
Everything here is host arithmetic; the kernels take any k <= the k their
buffers were sized for.
"""
from __future__ import annotations

import dataclasses


def expected_accepted(a: float, k: int) -> float:
    """E[min(N, k)] for P(N >= i) = a^i: sum_{i=1..k} a^i."""
    if k <= 0:
        return 0.0
    if a >= 1.0:
        return float(k)
    return a * (1.0 - a ** k) / (1.0 - a)


def round_time(k: int, t_step: float, t_copy: float, t_tail: float, t_row: float = 0.0) -> float:
    """T(k) = max(k * t_step + (k + 1) * t_row, t_copy) + t_tail."""
    return max(k * t_step + (k + 1) * t_row, t_copy) + t_tail


def best_k(a: float, t_step: float, t_copy: float, t_tail: float, k_min: int, k_max: int,
           choices=None, t_row: float = 0.0, t_verify=None) -> int:
    """The draft length in [k_min, k_max] (or among `choices`) with the most
    tokens per second (the smallest such k on ties: fewer draft launches).
    t_verify: optional mapping k -> verify compute time of a round drafting k
    tokens; where it has k, it replaces the linear (k + 1) * t_row."""
    ks = sorted(choices) if choices is not None else range(k_min, k_max + 1)
    best, best_rate = ks[0], -1.0
    for k in ks:
        if t_verify is not None and k in t_verify:
            t = max(k * t_step + t_verify[k], t_copy) + t_tail
        else:
            t = round_time(k, t_step, t_copy, t_tail, t_row)
        rate = (expected_accepted(a, k) + 1.0) / t
        if rate > best_rate * (1.0 + 1e-12):
            best, best_rate = k, rate
    return best


@dataclasses.dataclass
class DraftLengthController:
    """Chooses each round's draft length from what earlier rounds measured.

    prior_accepted / prior_stops: pseudo-counts of the acceptance estimate
    before any round is seen (default: a = 0.9, worth ~10 rounds' stops).
    Timings are exponential moving averages with weight `ema`."""
    k_max: int
    k_min: int = 1
    prior_accepted: float = 9.0
    prior_stops: float = 1.0
    ema: float = 0.5
    accepted: float = 0.0
    stops: float = 0.0
    t_step: float | None = None
    t_copy: float | None = None
    t_tail: float | None = None
    t_row: float | None = None       # verify compute per row, learned from rounds it was not hidden in
    choices: tuple | None = None     # allowed draft lengths (default: every k in [k_min, k_max])
    t_verify: dict | None = None     # optional k -> verify compute of a round (measured); overrides t_row

    def __post_init__(self):
        if not (1 <= self.k_min <= self.k_max):
            raise ValueError(f"need 1 <= k_min <= k_max (got {self.k_min}, {self.k_max})")
        if self.choices is not None and not all(self.k_min <= c <= self.k_max for c in self.choices):
            raise ValueError("choices must lie in [k_min, k_max]")

    def acceptance(self) -> float:
        """Censored estimate of the per-token acceptance probability."""
        s = self.accepted + self.prior_accepted
        f = self.stops + self.prior_stops
        return s / (s + f)

    def observe(self, n_acc, k_used: int, t_step: float | None = None, t_copy: float | None = None,
                t_tail: float | None = None, t_verify: float | None = None):
        """One finished round: accepted lengths per request (each <= k_used) and,
        if measured, the per-step draft time, the transfer span, the tail and
        the verify compute after drafting (only when the transfer had already
        ended, so that it measures compute, not waiting)."""
        for n in n_acc:
            n = int(n)
            if n < 0 or n > k_used:
                raise ValueError(f"accepted length {n} outside [0, {k_used}]")
            self.accepted += n
            if n < k_used:
                self.stops += 1          # a mismatch ended this request's run
        t_row = None if t_verify is None else t_verify / (k_used + 1)
        for name, v in (("t_step", t_step), ("t_copy", t_copy), ("t_tail", t_tail), ("t_row", t_row)):
            if v is None:
                continue
            old = getattr(self, name)
            setattr(self, name, v if old is None else (1.0 - self.ema) * old + self.ema * v)

    def next_k(self) -> int:
        """k_max until timings are known; then the rate-maximising length."""
        if self.t_step is None or self.t_copy is None:
            return self.k_max
        return best_k(self.acceptance(), self.t_step, self.t_copy, self.t_tail or 0.0, self.k_min, self.k_max,
                      self.choices, self.t_row or 0.0, self.t_verify)
