"""Pins for the per-request draft-length controller of the oracle (no GPU).

[FASER] mechanism 1: every request's previous acceptance feeds back into its
own gamma, longer where drafts are accepted, shorter where they are
rejected.  The pages give no formula; the controller's rule is fixed in the
library header.  What pins it here, independently of retyping it:
  * its acceptance estimate converges to the true per-draft acceptance of
    simulated requests (geometric trials, stopped at the first rejection);
  * the expected emitted tokens sum_{k<=g} alpha^k equal the closed form
    (1 - alpha^(g+1)) / (1 - alpha) and a Monte-Carlo count of a chain;
  * limits: alpha -> 0 gives gamma_min, alpha -> 1 gives gamma_max, and the
    chosen gamma never decreases as acceptance grows;
  * the chosen gamma maximises the simulated emitted-tokens-per-cost of a
    chain, checked by simulation over every candidate gamma.
"""

import numpy as np
import pytest

import oracle


def _steps(alpha, n_steps, gamma, rng, decay=0.9):
    st = np.zeros((1, 2))
    g = np.array([gamma], dtype=np.int32)
    for _ in range(n_steps):
        # a chain of g drafts, each accepted with probability alpha until the first rejection
        acc = 0
        while acc < g[0] and rng.random() < alpha:
            acc += 1
        err, _ = oracle.adapt_gamma([acc], [int(g[0])], st, decay, 2.0, 1, 8)
        assert err == 0
    return st


@pytest.mark.parametrize("alpha", [0.2, 0.5, 0.8, 0.95])
def test_estimate_converges_to_the_true_acceptance(alpha):
    rng = np.random.default_rng(int(alpha * 100))
    st = _steps(alpha, 4000, 6, rng, decay=0.999)
    est = (st[0, 0] + 1) / (st[0, 1] + 2)
    assert abs(est - alpha) < 0.03, (est, alpha)


@pytest.mark.parametrize("alpha", [0.1, 0.5, 0.9, 0.99])
def test_expected_tokens_closed_form_and_simulation(alpha):
    rng = np.random.default_rng(1)
    for g in (1, 3, 7):
        closed = (1 - alpha ** (g + 1)) / (1 - alpha)
        run = sum(alpha ** k for k in range(g + 1))
        assert run == pytest.approx(closed, rel=1e-12)
        n = 200_000
        acc = np.zeros(n, dtype=np.int64)
        alive = np.ones(n, dtype=bool)
        for _ in range(g):
            alive &= rng.random(n) < alpha
            acc += alive
        emitted = acc + 1  # accepted drafts plus the emitted token
        assert emitted.mean() == pytest.approx(closed, rel=0.01)


def _choice(S, N, overhead=2.0, gmin=1, gmax=8):
    st = np.array([[S, N]], dtype=np.float64)
    err, g = oracle.adapt_gamma([0], [-1], st, 1.0, overhead, gmin, gmax)  # verified < 0: no update
    assert err == 0 and g[0] == -1 and st[0, 0] == S
    # one update with a = 0 of 0 verified: counts unchanged except decay 1
    st = np.array([[S, N]], dtype=np.float64)
    err, g = oracle.adapt_gamma([0], [0], st, 1.0, overhead, gmin, gmax)
    assert err == 0
    return int(g[0]), (st[0, 0] + 1) / (st[0, 1] + 2)


def test_limits_and_monotonicity():
    g_low, a_low = _choice(0.0, 1e6)
    assert a_low < 1e-5 and g_low == 1
    g_high, a_high = _choice(1e7, 1e7)
    assert a_high > 0.999999 and g_high == 8
    prev = 0
    for S in np.linspace(0, 1000, 60):
        g, _ = _choice(S, 1000.0)
        assert g >= prev
        prev = g


@pytest.mark.parametrize("S,N", [(30.0, 60.0), (70.0, 90.0), (180.0, 200.0)])
def test_choice_maximises_simulated_tokens_per_cost(S, N):
    g_star, alpha = _choice(S, N)
    rng = np.random.default_rng(7)
    n = 400_000
    u = rng.random((n, 9))
    first_rej = np.where((u < alpha).all(axis=1), 9, np.argmin(u < alpha, axis=1))
    rates = []
    for g in range(1, 9):
        emitted = np.minimum(first_rej, g) + 1
        rates.append(emitted.mean() / (g + 1 + 2.0))
    best = int(np.argmax(rates)) + 1
    # the simulated best is the chosen gamma, or within noise of it
    assert rates[g_star - 1] >= max(rates) * (1 - 3e-3), (g_star, best, rates)


def test_bad_lengths_are_reported_and_skipped():
    st = np.zeros((2, 2))
    err, g = oracle.adapt_gamma([5, 1], [4, 4], st, 0.7, 2.0, 1, 8)
    assert err & oracle.ORC_BAD_LENGTH
    assert g[0] == -1 and (st[0] == 0).all() and g[1] >= 1
