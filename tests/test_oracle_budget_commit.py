"""Pins for the oracle's budget selection, KV commit and Philox (no GPU).

Budget ([DSpark] "하드웨어 인식 Prefix 스케줄러", "기술 상세"): checked by brute
force over every prefix-closed allocation (L_1..L_R) for tiny R and gamma —
the greedy sorted admission must reach the same maximum of
Theta = tau * SPS(B).
Commit ([SwiftSpec] mechanism 2): conservation of blocks, no duplicates,
committed slot k == staged row path[k], the released blocks are exactly
those past the new length.
Philox4x32-10: the published Random123 known-answer vectors
(tests/golden/philox4x32_10_kat.txt), uniformity, counter and key
sensitivity.
"""

import itertools
import os

import numpy as np
import pytest
from scipy import stats

import oracle
from speculative_decoding_verification_padding_gb300 import workloads as wl


# ------------------------------------------------------------------ budget --

def _brute_force(c, gamma, sps):
    """Every prefix-closed allocation; S as fp32 left-to-right products (the
    oracle's stated precision), tau summed in fp64.  Returns the best Theta,
    the best allocation and the runner-up Theta of a different allocation."""
    R = c.shape[0]
    S = np.cumprod(c.astype(np.float32), axis=1, dtype=np.float32).astype(np.float64)
    scored = []
    for L in itertools.product(*[range(g + 1) for g in gamma]):
        B = R + sum(L)
        if B >= len(sps):
            continue
        tau = R + sum(S[i, :L[i]].sum() for i in range(R))
        scored.append((tau * float(sps[B]), L))
    scored.sort(key=lambda t: -t[0])
    runner = scored[1][0] if len(scored) > 1 else -np.inf
    return scored[0][0], scored[0][1], runner


@pytest.mark.parametrize("trial", range(60))
def test_budget_matches_brute_force(trial):
    rng = np.random.default_rng(trial)
    R = int(rng.integers(1, 4))
    gmax = int(rng.integers(1, 4))
    gamma = rng.integers(0, gmax + 1, R).astype(np.int32)
    c = rng.beta(4, 2, size=(R, gmax)).astype(np.float32)
    b_max = R + int(rng.integers(0, R * gmax + 2))
    B = np.arange(b_max + 1, dtype=np.float64)
    kind = trial % 3
    if kind == 0:
        sps = 1000.0 / (1.0 + B / rng.uniform(0.5, 8))
    elif kind == 1:
        sps = np.full(b_max + 1, 7.0)
    else:
        sps = 1000.0 / (1.0 + (B / 3.0) ** 2)
    sps = sps.astype(np.float32)
    err, vl, best_B, theta = oracle.select_budget(c, gamma, sps)
    assert err == 0
    ref_theta, ref_L, runner = _brute_force(c, gamma, sps)
    assert theta == pytest.approx(ref_theta, rel=1e-9)
    if ref_theta - runner > 1e-9 * ref_theta:  # unique optimum
        assert tuple(vl) == tuple(ref_L)
    assert best_B == R + vl.sum()
    assert (vl <= gamma).all()
    # the admitted set is prefix-closed and is the top of the survival order
    S = np.cumprod(c.astype(np.float64), axis=1)
    admitted = [S[i, k] for i in range(R) for k in range(vl[i])]
    rejected = [S[i, k] for i in range(R) for k in range(vl[i], gamma[i])]
    if admitted and rejected:
        assert min(admitted) >= max(rejected) - 1e-7


def test_budget_ties_go_to_lower_request_then_position():
    c = np.ones((3, 2), dtype=np.float32)  # every S = 1
    gamma = np.array([2, 2, 2], dtype=np.int32)
    sps = np.array([1.0] * 3 + [1.0] * 3 + [0.0] * 4, dtype=np.float32)  # B <= 5 useful
    err, vl, best_B, theta = oracle.select_budget(c, gamma, sps)
    assert err == 0
    # Theta grows with m up to B = 5 (m = 2); the two admitted keys are the
    # lowest request's positions 1 and 2
    assert best_B == 5
    assert list(vl) == [2, 0, 0]


def test_budget_constant_sps_admits_everything_that_fits():
    rng = np.random.default_rng(3)
    c = rng.beta(4, 2, size=(10, 4)).astype(np.float32)
    gamma = np.full(10, 4, dtype=np.int32)
    err, vl, best_B, _ = oracle.select_budget(c, gamma, np.ones(10 + 40 + 1, dtype=np.float32))
    assert (vl == 4).all() and best_B == 50
    err, vl, best_B, _ = oracle.select_budget(c, gamma, np.ones(10 + 7 + 1, dtype=np.float32))
    assert vl.sum() == 7 and best_B == 17


def test_budget_negative_zero_survival_is_zero():
    """A conditional survival of -0.0 is the value 0: its candidates sort with
    the other zero survivals, after every positive one.  (Keyed by its raw
    bits, ~bits(-0.0) would put them first.)"""
    c = np.array([[0.9, 0.8], [-0.0, 0.7]], dtype=np.float32)
    gamma = np.array([2, 2], dtype=np.int32)
    sps = np.array([1.0, 1.0, 1.0, 1.0, 0.0, 0.0, 0.0], dtype=np.float32)  # at most one admitted
    err, vl, best_B, theta = oracle.select_budget(c, gamma, sps)
    assert err == 0
    assert list(vl) == [1, 0] and best_B == 3
    assert theta == pytest.approx(2.9, rel=1e-6)
    ref_theta, ref_L, _ = _brute_force(c, gamma, sps)
    assert tuple(vl) == tuple(ref_L) and theta == pytest.approx(ref_theta, rel=1e-9)
    # the same selection as with +0.0 in its place, on random inputs too
    rng = np.random.default_rng(11)
    for _ in range(20):
        c = rng.beta(4, 2, size=(6, 3)).astype(np.float32)
        zero = rng.random(c.shape) < 0.3
        c_pos = np.where(zero, np.float32(0.0), c).astype(np.float32)
        c_neg = np.where(zero, np.float32(-0.0), c).astype(np.float32)
        gamma = rng.integers(0, 4, 6).astype(np.int32)
        sps = (1000.0 / (1.0 + np.arange(6 + 18 + 1) / 4.0)).astype(np.float32)
        a = oracle.select_budget(c_pos, gamma, sps)
        b = oracle.select_budget(c_neg, gamma, sps)
        assert np.array_equal(a[1], b[1]) and a[2] == b[2] and a[3] == b[3]


def test_budget_full_size_has_interior_optimum():
    w = wl.make_workload(wl.config("batch256"), vocab=64, ctx_scale=0.001)
    err, vl, best_B, theta = oracle.select_budget(w.cond_survival, w.gamma, w.sps)
    assert err == 0
    m = vl.sum()
    assert 0 < m < w.gamma.sum()
    assert best_B == 256 + m
    # Theta really is maximal over m (fp64 recomputation, all m)
    S = np.sort(np.cumprod(w.cond_survival.astype(np.float64), 1).ravel())[::-1]
    tau = 256 + np.concatenate([[0.0], np.cumsum(S)])
    th = tau * w.sps[256: 256 + len(tau)].astype(np.float64)
    assert int(np.argmax(th)) == m
    assert theta == pytest.approx(th.max(), rel=1e-9)


# ------------------------------------------------------------------ commit --

def _commit_case(name, T, **kw):
    w = wl.make_workload(wl.config(name), vocab=64, temperature=T, **kw)
    draft = w.draft_logits if T > 0 else None
    err, st = oracle.accept(w.batch(), w.target_logits, draft, T, w.seed)
    assert err == 0
    return w, st


@pytest.mark.parametrize("name,T,kw", [("batch64", 0.7, dict(n_req=20, ctx_scale=0.01, draft_sigma=0.5)),
                                       ("tree70b", 0.0, dict(ctx_scale=0.01, draft_sigma=0.1)),
                                       ("batch64", 0.0, dict(n_req=20, ctx_scale=0.01, draft_sigma=0.1))])
def test_commit_keeps_accepted_path_and_frees_the_rest(name, T, kw):
    w, st = _commit_case(name, T, **kw)
    kv = w.kv_copy()
    fl = w.free_list.copy()
    fc = np.array([w.free_count], dtype=np.int32)
    err = oracle.commit_kv(w.batch(), kv, st.accepted_len, st.accepted_nodes, fl, fc)
    assert err == 0
    bs = wl.BLOCK_SIZE
    freed_expected = []
    for i in range(w.n_req):
        rows = w.cu_rows[i + 1] - w.cu_rows[i]
        ctx = w.cache_lens[i]
        a = st.accepted_len[i]
        new_len = ctx + 1 + a
        assert kv["cache_lens"][i] == new_len
        for k in range(a + 1):
            src = ctx + st.accepted_nodes[i, k]
            dst = ctx + k
            sb, db = w.block_tables[i, src // bs], kv["block_tables"][i, dst // bs]
            assert np.array_equal(kv["k_cache"][db, :, dst % bs], w.k_cache[sb, :, src % bs])
            assert np.array_equal(kv["v_cache"][db, :, dst % bs], w.v_cache[sb, :, src % bs])
        keep = -(-new_len // bs)
        used = -(-(ctx + rows) // bs)
        assert (kv["block_tables"][i, keep:] == -1).all()
        assert np.array_equal(kv["block_tables"][i, :keep], w.block_tables[i, :keep])
        freed_expected += list(w.block_tables[i, keep:used])
        # context slots untouched
        for s in range(0, ctx, max(1, ctx // 7)):
            b = w.block_tables[i, s // bs]
            assert np.array_equal(kv["k_cache"][b, :, s % bs], w.k_cache[b, :, s % bs])
    n_new = fc[0] - w.free_count
    assert list(fl[w.free_count: fc[0]]) == freed_expected
    # conservation: every pool block is either in a table or on the free list, once
    in_tables = kv["block_tables"][kv["block_tables"] >= 0]
    on_list = fl[: fc[0]]
    allb = np.concatenate([in_tables, on_list])
    assert len(np.unique(allb)) == len(allb)          # no block held twice
    assert len(allb) == w.k_cache.shape[0]            # none lost
    assert n_new == len(freed_expected)


def test_commit_overlapping_slots_gather_before_scatter():
    # path [0, 2, 3]: slot ctx+1 <- ctx+2 and slot ctx+2 <- ctx+3 overlap.
    w = wl.make_workload(wl.config("tiny"), vocab=64, ctx_scale=0.25)
    kv = w.kv_copy()
    al = np.array([2], dtype=np.int32)
    an = np.full((1, w.max_rows), -1, dtype=np.int32)
    an[0, :3] = [0, 2, 3]
    fl = w.free_list.copy()
    fc = np.array([w.free_count], dtype=np.int32)
    assert oracle.commit_kv(w.batch(), kv, al, an, fl, fc) == 0
    bs = wl.BLOCK_SIZE
    ctx = int(w.cache_lens[0])
    for k, node in enumerate([0, 2, 3]):
        src, dst = ctx + node, ctx + k
        sb, db = w.block_tables[0, src // bs], kv["block_tables"][0, dst // bs]
        assert np.array_equal(kv["k_cache"][db, :, dst % bs], w.k_cache[sb, :, src % bs])


def test_commit_pool_overflow_is_reported():
    w, st = _commit_case("batch64", 0.0, n_req=20, ctx_scale=0.01, draft_sigma=3.0)
    kv = w.kv_copy()
    fl = np.full(w.free_count, -1, dtype=np.int32)  # capacity == current count: no room
    fc = np.array([w.free_count], dtype=np.int32)
    err = oracle.commit_kv(w.batch(), kv, st.accepted_len, st.accepted_nodes, fl, fc)
    assert err & oracle.ORC_POOL_OVERFLOW


# ------------------------------------------------------------------ Philox --

def test_philox_accept_uniforms_are_uniform():
    u = np.array([oracle.accept_uniform(12345, i, j) for i in range(2000) for j in range(50)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    counts = np.bincount((u * 64).astype(int), minlength=64)
    assert stats.chisquare(counts).pvalue > 1e-3
    # 24-bit grid
    assert np.all((u * 2 ** 24) == np.floor(u * 2 ** 24))


def test_philox_race_uniforms_open_interval_and_fp32_exact():
    for draw in (oracle.race_uniform, oracle.pick_uniform):
        u = np.array([draw(7, 3, 5, g) for g in range(20000)])
        assert u.min() > 0.0 and u.max() < 1.0
        assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
        assert stats.kstest(u, "uniform").pvalue > 1e-3
        # adjacent groups are uncorrelated
        assert abs(np.corrcoef(u[:-1], u[1:])[0, 1]) < 0.03
    # every group has its own uniform: the 128 groups of a block take the
    # four words of 32 counters, no word twice
    u = [oracle.race_uniform(7, 3, 5, g) for g in range(512)]
    assert len(set(u)) == 512
    # the pick and race streams are distinct
    a = np.array([oracle.race_uniform(7, 3, 5, g) for g in range(4000)])
    b = np.array([oracle.pick_uniform(7, 3, 5, g) for g in range(4000)])
    assert abs(np.corrcoef(a, b)[0, 1]) < 0.05


def test_philox_reproduces_the_published_known_answer_vectors():
    # Random123's known-answer vectors for philox4x32 with 10 rounds (Salmon
    # et al., SC'11), read from tests/golden
    path = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")
    n = 0
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        w = [int(x, 16) for x in line.split()]
        ctr, key, want = w[:4], w[4:6], w[6:10]
        assert [int(x) for x in oracle.philox4x32_10(ctr, key)] == want, line
        n += 1
    assert n == 3


def test_philox_counter_and_key_sensitivity():
    base = oracle.philox4x32_10([1, 2, 3, 4], [5, 6])
    seen = {tuple(base)}
    for w in range(4):
        for bit in (0, 7, 31):
            c = [1, 2, 3, 4]
            c[w] ^= 1 << bit
            out = oracle.philox4x32_10(c, [5, 6])
            # about half of the 128 output bits flip for a one-bit counter change
            flips = sum(bin(int(a) ^ int(b)).count("1") for a, b in zip(out, base))
            assert 40 < flips < 88
            seen.add(tuple(out))
    for k in range(2):
        key = [5, 6]
        key[k] ^= 1
        seen.add(tuple(oracle.philox4x32_10([1, 2, 3, 4], key)))
    assert len(seen) == 1 + 12 + 2
