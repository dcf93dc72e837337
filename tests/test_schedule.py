"""Draft-length controller (host logic, no GPU)."""
import numpy as np
import pytest

from verify_compressed_kv_gb300.schedule import (DraftLengthController, best_k, expected_accepted,
                                                 round_time)


@pytest.mark.parametrize("a", [0.0, 0.3, 0.9, 0.99, 1.0])
@pytest.mark.parametrize("k", [0, 1, 5, 32])
def test_expected_accepted_matches_the_distribution(a, k):
    """E[min(N, k)] from P(N = n) = a^n (1 - a) summed term by term (N = k..inf lumped)."""
    if a == 1.0:
        want = float(k)
    else:
        pmf = [a ** n * (1 - a) for n in range(k)]
        want = sum(n * p for n, p in enumerate(pmf)) + k * a ** k
    assert expected_accepted(a, k) == pytest.approx(want, rel=1e-12, abs=1e-12)


def test_round_time_and_limits_of_the_choice():
    assert round_time(4, 1.0, 10.0, 2.0) == 12.0 and round_time(20, 1.0, 10.0, 2.0) == 22.0
    # drafting hides entirely under the transfer: the longest draft is free
    assert best_k(0.5, t_step=0.1, t_copy=100.0, t_tail=1.0, k_min=1, k_max=16) == 16
    # nothing to amortise (no transfer, no tail): one draft token per round is best
    assert best_k(0.9, t_step=1.0, t_copy=0.0, t_tail=0.0, k_min=1, k_max=16) == 1
    # a drafter that is never right: every k gives one token per round, so the cheapest k wins
    assert best_k(0.0, t_step=1.0, t_copy=0.0, t_tail=5.0, k_min=1, k_max=16) == 1


def test_choice_maximises_the_rate_against_brute_force():
    rng = np.random.default_rng(3)
    for _ in range(200):
        a = float(rng.uniform(0, 1))
        t_step, t_copy, t_tail = (float(x) for x in rng.uniform(0.01, 5.0, size=3))
        k = best_k(a, t_step, t_copy, t_tail, 1, 40)
        rates = [(expected_accepted(a, j) + 1) / round_time(j, t_step, t_copy, t_tail) for j in range(1, 41)]
        assert rates[k - 1] >= max(rates) * (1 - 1e-9)


def test_acceptance_estimate_is_unbiased_under_censoring():
    """Simulated rounds with a known a and draft length 8: the censored estimate
    recovers a (counting fully accepted rounds as mismatches would bias it low)."""
    rng = np.random.default_rng(7)
    a, k = 0.85, 8
    c = DraftLengthController(k_max=k, prior_accepted=0.0, prior_stops=0.0)
    for _ in range(4000):
        n = np.minimum(rng.geometric(1 - a, size=8) - 1, k)     # P(N >= i) = a^i, cut at k
        c.observe(n, k)
    assert abs(c.acceptance() - a) < 0.01


def test_controller_flow():
    c = DraftLengthController(k_max=24, k_min=2)
    assert c.next_k() == 24                         # no timings yet
    c.observe([24, 24, 3], 24, t_step=0.2, t_copy=20.0, t_tail=0.5)
    assert c.next_k() == 24                         # 24 steps (4.8) hide under 20 of transfer
    c.observe([0, 1, 0], 24, t_step=2.0, t_copy=0.1, t_tail=0.1)
    assert 2 <= c.next_k() < 24                     # expensive drafting, low acceptance
    with pytest.raises(ValueError):
        c.observe([25], 24)
    with pytest.raises(ValueError):
        DraftLengthController(k_max=4, k_min=5)


def test_choices_restrict_the_grid():
    c = DraftLengthController(k_max=64, k_min=4, choices=(4, 16, 32, 64))
    c.observe([10, 64, 64], 64, t_step=0.1, t_copy=5.0, t_tail=0.1)
    assert c.next_k() in (4, 16, 32, 64)
    # 64 steps (6.4) exceed the transfer (5.0): 32 still hides under it and loses few tokens
    assert best_k(0.5, 0.1, 5.0, 0.1, 4, 64, choices=(4, 16, 32, 64)) == 32
    with pytest.raises(ValueError):
        DraftLengthController(k_max=8, choices=(4, 16))


def test_verify_rows_cost_bounds_the_draft_length():
    """Verification follows the drafting and grows with k + 1 rows: with the
    Mistral-shaped costs measured on the GPU (0.107 ms per draft step, 5.2 ms of
    transfer, ~0.05 ms of verify per row) the best k stays well below the k at
    which drafting alone would fill the transfer (~48)."""
    assert round_time(10, 0.1, 5.0, 1.0, t_row=0.2) == max(10 * 0.1 + 11 * 0.2, 5.0) + 1.0
    k_no_rows = best_k(0.88, 0.107, 5.2, 0.5, 4, 60, choices=range(4, 61, 4))
    k_rows = best_k(0.88, 0.107, 5.2, 0.5, 4, 60, choices=range(4, 61, 4), t_row=0.05)
    assert k_no_rows >= 44 and k_rows < k_no_rows
    c = DraftLengthController(k_max=60, k_min=4, choices=tuple(range(4, 61, 4)))
    c.observe([5] * 8, 48, t_step=0.107, t_copy=5.2, t_tail=0.5, t_verify=49 * 0.05)
    assert c.t_row == pytest.approx(0.05) and c.next_k() == k_rows


def test_measured_verify_table_overrides_the_linear_row_term():
    """A verify cost that steps up at large k (the chunk kernel's launch geometry
    changes) must steer the choice away from those k, where the linear per-row
    term would not."""
    from verify_compressed_kv_gb300.schedule import best_k
    a, t_step, t_copy, t_tail, t_row = 0.96, 1.4, 82.0, 0.25, 0.69
    linear = best_k(a, t_step, t_copy, t_tail, 4, 60, choices=range(4, 61, 4), t_row=t_row)
    table = {k: (k + 1) * t_row * (1.0 if k <= 32 else 1.8) for k in range(4, 61, 4)}
    stepped = best_k(a, t_step, t_copy, t_tail, 4, 60, choices=range(4, 61, 4), t_row=t_row, t_verify=table)
    assert linear > 32 and stepped <= 32
    # a table equal to the linear term changes nothing
    same = {k: (k + 1) * t_row for k in range(4, 61, 4)}
    assert best_k(a, t_step, t_copy, t_tail, 4, 60, choices=range(4, 61, 4), t_row=t_row, t_verify=same) == linear


def test_controller_passes_its_verify_table():
    from verify_compressed_kv_gb300.schedule import DraftLengthController
    c = DraftLengthController(k_max=60, k_min=4, choices=tuple(range(4, 61, 4)))
    c.observe([30, 31, 28, 29], 32, t_step=1.4, t_copy=82.0, t_tail=0.25, t_verify=32 * 0.69)
    free = c.next_k()
    c.t_verify = {k: (k + 1) * 0.69 * (1.0 if k <= 32 else 1.8) for k in range(4, 61, 4)}
    assert c.next_k() <= 32 < free
