"""Pins for the oracle's chunk-size rule (no GPU).

The rule is ours (the FASER page only says that the chunk size follows the
load): the expected bytes of a chunked step in which each draft of request i
is accepted with probability a_i, plus a fixed cost per chunk.  What pins it:
  * a Monte-Carlo run of chunked verification (drafts accepted at random,
    chunks attended until the first rejection, bytes counted per attended
    chunk) agrees with the expected cost at every chunk size, and would not
    agree with an off-by-one in the reach probability;
  * a = 1: every chunk is attended, one chunk of all rows is cheapest, and the
    cost is the plain sum of each request's bytes;
  * a -> 0: only the first chunk is attended, one row per chunk is cheapest;
  * ties go to the larger chunk; invalid requests are reported and left out.
"""

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


KV = 4096.0
ROW = 2 * 4 * 128256.0


def _simulate(rows, ctx, alpha, c, trials, rng):
    """Mean bytes read by a chunked step over `trials` random acceptances."""
    total = 0.0
    for r, x, a in zip(rows, ctx, alpha):
        acc = rng.random((trials, max(r - 1, 1))) < a  # draft j accepted (j = 1..r-1)
        # drafts 1..m all accepted
        run = np.cumprod(acc, axis=1)
        b = 0
        while b < r:
            e = min(b + c, r)
            if b == 0:
                reached = np.ones(trials, bool)
            else:
                reached = run[:, b - 1].astype(bool)  # drafts 1..b accepted
            total += reached.sum() * ((x + e) * KV + (e - b) * ROW)
            b += c
    return total / trials


def _state(alpha, n=50.0):
    # (S + 1) / (N + 2) = alpha
    N = np.full(len(alpha), n)
    S = np.asarray(alpha) * (N + 2.0) - 1.0
    return np.stack([S, N], axis=1)


def test_expected_cost_matches_a_monte_carlo_run():
    rng = np.random.default_rng(11)
    rows = [9, 5, 7, 2, 9, 4]
    ctx = [600, 4100, 12000, 800, 30000, 2500]
    alpha = [0.9, 0.6, 0.75, 0.3, 0.95, 0.5]
    st = _state(alpha)
    err, ch, cost, costs = oracle.select_chunk(rows, ctx, st, KV, ROW, 0)
    assert err == 0
    a_used = (st[:, 0] + 1.0) / (st[:, 1] + 2.0)
    for c in range(1, max(rows) + 1):
        sim = _simulate(rows, ctx, a_used, c, 40_000, rng)
        assert abs(float(costs[c - 1]) - sim) < 0.01 * sim, (c, float(costs[c - 1]), sim)
        if 2 <= c <= 4:
            # power: reaching chunk k with probability a^(k c - 1) instead of
            # a^(k c) shifts the expectation well past the tolerance (sizes
            # that give every long request several chunks)
            wrong = 0.0
            for r, x, a in zip(rows, ctx, a_used):
                for k, b in enumerate(range(0, r, c)):
                    e = min(b + c, r)
                    wrong += (a ** max(k * c - 1, 0)) * ((x + e) * KV + (e - b) * ROW)
            assert abs(wrong - sim) > 0.01 * sim
    mn = costs[: max(rows)].min()
    assert ch == max(c for c in range(1, max(rows) + 1) if costs[c - 1] == mn)
    assert cost == mn


def test_all_accepted_prefers_one_chunk_and_sums_every_byte():
    rows = [9, 3, 6]
    ctx = [1000, 2000, 3000]
    st = np.array([[20.0, 0.0]] * 3)  # (S + 1) / (N + 2) > 1: clamped to 1
    err, ch, cost, costs = oracle.select_chunk(rows, ctx, st, KV, ROW, 1000)
    assert err == 0
    assert ch == 9
    plain = 1000 + sum((x + r) * KV + r * ROW for r, x in zip(rows, ctx))
    assert cost == plain
    # two chunks re-read every context once more
    two = 2 * 1000
    for r, x in zip(rows, ctx):
        for b in range(0, r, 5):
            e = min(b + 5, r)
            two += (x + e) * KV + (e - b) * ROW
    assert costs[4] == two


def test_all_rejected_prefers_one_row_per_chunk():
    rows = [9, 3, 6]
    ctx = [1000, 2000, 3000]
    st = np.array([[0.0, 1e12]] * 3)  # a ~ 1e-12
    err, ch, cost, costs = oracle.select_chunk(rows, ctx, st, KV, ROW, 0)
    assert err == 0
    assert ch == 1
    # only the first row of each request is read (the rest within rounding)
    assert abs(cost - sum((x + 1) * KV + ROW for x in ctx)) < 10


def test_ties_go_to_the_larger_chunk_and_costs_past_max_rows_are_marked():
    rows = [4, 2]
    st = _state([0.5, 0.5])
    err, ch, cost, costs = oracle.select_chunk(rows, [10, 20], st, 0.0, 0.0, 0)
    assert err == 0 and ch == 4 and cost == 0
    assert (costs[4:] == np.iinfo(np.uint64).max).all()
    assert (costs[:4] == 0).all()


def test_invalid_requests_are_reported_and_left_out():
    good_rows, good_ctx = [5, 7], [100, 900]
    st_good = _state([0.7, 0.4])
    ref = oracle.select_chunk(good_rows, good_ctx, st_good, KV, ROW, 5000)
    for bad_row, bad_ctx, bad_st in [(0, 10, [1.0, 2.0]), (129, 10, [1.0, 2.0]),
                                     (4, -1, [1.0, 2.0]), (4, 10, [-1.0, 2.0]),
                                     (4, 10, [np.nan, 2.0])]:
        rows = good_rows + [bad_row]
        ctx = good_ctx + [bad_ctx]
        st = np.vstack([st_good, np.array([bad_st])])
        err, ch, cost, costs = oracle.select_chunk(rows, ctx, st, KV, ROW, 5000)
        assert err & oracle.ORC_BAD_LENGTH
        assert (ch, cost) == ref[1:3]
        assert np.array_equal(costs, ref[3])
