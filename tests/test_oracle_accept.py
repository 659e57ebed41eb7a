"""Pins for the oracle's accept / reject / resample (no GPU).

What the pages fix: the accepted output is the longest matching prefix and
the rule preserves the target distribution ([DSpark] glossary,
"사전검증 디코딩"); a request stops at its first rejection and its later
rows are never examined ([FASER] mechanism 2).  The sampling rule itself
(accept with min(1, p/q), resample from normalize(max(0, p - q)), bonus from
p) is the standard lossless rule.  The pins:
  * greedy chains and trees against brute-force enumeration;
  * chi-square over 10^6 trials at vocab 16: the first emitted token is
    distributed as p (T = 1 and 0.7, 1 and 3 drafts), the resampled token
    after a rejection as normalize(max(0, p - q)), the bonus token as p;
  * the acceptance rate against sum_v min(p_v, q_v);
  * the two-step draw (a race among groups of four entries, then the entry
    inside the winning group) at a vocabulary whose last group is short,
    and a planted mistake in the second step that the statistics see;
  * row statistics against torch.logsumexp / softmax in fp64;
  * chunked verification equal to one-pass verification;
  * tree sampling (T > 0, siblings i.i.d. from q): chi-square of the first
    emitted token against p_root and of the next token against p_c given the
    accepted node c, a one-child tree equal to the chain rule, the closed
    form of the residual after several sibling rejections, and a planted
    mistake that the statistics see.
"""

import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from speculative_decoding_verification_padding_gb300 import workloads as wl


def _softmax_T(l, T):
    x = (np.asarray(l, dtype=np.float32) / np.float32(T)).astype(np.float64)
    x = x - x.max()
    e = np.exp(x)
    return e / e.sum()


def _chain_batch(n_req, gamma, tokens):
    rows = gamma + 1
    cu = np.arange(n_req + 1, dtype=np.int32) * rows
    parent = np.tile(np.arange(-1, gamma, dtype=np.int32), n_req)
    return {"cu_rows": cu, "parent": parent, "tokens": tokens.astype(np.int32).ravel(),
            "max_rows": rows}


def _chi2_ok(counts, probs, alpha=1e-3):
    n = counts.sum()
    exp = probs * n
    keep = exp >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    ex = np.append(exp[keep], exp[~keep].sum())
    if ex[-1] == 0:
        obs, ex = obs[:-1], ex[:-1]
    stat = ((obs - ex) ** 2 / ex).sum()
    dof = len(obs) - 1
    return stat, stats.chi2.ppf(1 - alpha, dof), dof


# ------------------------------------------------------------------ greedy --

def test_greedy_chain_is_longest_argmax_prefix():
    rng = np.random.default_rng(11)
    R, gamma, V = 400, 6, 32
    rows = gamma + 1
    target = rng.standard_normal((R * rows, V)).astype(np.float32)
    am = target.argmax(1)
    tokens = np.zeros(R * rows, dtype=np.int32)
    for i in range(R):
        for j in range(1, rows):
            good = am[i * rows + j - 1]
            tokens[i * rows + j] = good if rng.random() < 0.75 else (good + 1 + rng.integers(V - 1)) % V
    b = _chain_batch(R, gamma, tokens)
    err, st = oracle.accept(b, target, None, 0.0, 1)
    assert err == 0
    for i in range(R):
        a = 0
        while a < gamma and tokens[i * rows + a + 1] == am[i * rows + a]:
            a += 1
        assert st.accepted_len[i] == a
        assert list(st.accepted_nodes[i, : a + 1]) == list(range(a + 1))
        assert (st.accepted_nodes[i, a + 1:] == -1).all()
        assert st.next_token[i] == am[i * rows + a]
        assert st.done[i] == 1


def _random_tree(rng, n):
    parent = [-1] + [int(rng.integers(0, j)) for j in range(1, n)]
    return np.array(parent, dtype=np.int32)


def _all_paths(parent):
    n = len(parent)
    paths = []
    for r in range(n):
        p, m = [], r
        while m >= 0:
            p.append(m)
            m = parent[m]
        paths.append(p[::-1])
    return paths


def test_greedy_tree_is_longest_valid_path_by_enumeration():
    rng = np.random.default_rng(12)
    V = 6  # small vocabulary: duplicate sibling tokens, ties between paths
    R = 300
    parents, tokens, cu = [], [], [0]
    for _ in range(R):
        n = int(rng.integers(1, 20))
        parents.append(_random_tree(rng, n))
        cu.append(cu[-1] + n)
    total = cu[-1]
    target = rng.standard_normal((total, V)).astype(np.float32)
    am = target.argmax(1)
    for i in range(R):
        par = parents[i]
        t = np.zeros(len(par), dtype=np.int32)
        for j in range(1, len(par)):
            good = am[cu[i] + par[j]]
            t[j] = good if rng.random() < 0.6 else rng.integers(V)
        tokens.append(t)
    b = {"cu_rows": np.array(cu, dtype=np.int32), "parent": np.concatenate(parents),
         "tokens": np.concatenate(tokens), "max_rows": max(len(p) for p in parents)}
    err, st = oracle.accept(b, target, None, 0.0, 3)
    assert err == 0
    for i in range(R):
        par, tok = parents[i], tokens[i]
        valid = [p for p in _all_paths(par)
                 if all(tok[p[k]] == am[cu[i] + p[k - 1]] for k in range(1, len(p)))]
        best = min(valid, key=lambda p: (-len(p), p))
        a = st.accepted_len[i]
        assert a == len(best) - 1
        assert list(st.accepted_nodes[i, : a + 1]) == best
        assert st.next_token[i] == am[cu[i] + best[-1]]


# ---------------------------------------------------------------- sampling --

def _sampling_run(gamma, T, seed, N=1_000_000, V=16):
    rng = np.random.default_rng(100 + gamma * 10 + int(T * 10))
    rows = gamma + 1
    lt = (rng.standard_normal((rows, V)) * 2.0).astype(np.float32)
    ld = (lt + rng.standard_normal((rows, V))).astype(np.float32)
    p = [_softmax_T(lt[r], T) for r in range(rows)]
    q = [_softmax_T(ld[r], T) for r in range(rows)]
    tokens = np.zeros((N, rows), dtype=np.int32)
    for j in range(1, rows):
        tokens[:, j] = rng.choice(V, size=N, p=q[j - 1])
    b = _chain_batch(N, gamma, tokens)
    target = np.ascontiguousarray(np.broadcast_to(lt, (N, rows, V)).reshape(N * rows, V))
    draft = np.ascontiguousarray(np.broadcast_to(ld, (N, rows, V)).reshape(N * rows, V))
    err, st = oracle.accept(b, target, draft, T, seed)
    assert err == 0
    return p, q, tokens, st


@pytest.mark.parametrize("gamma,T", [(1, 1.0), (3, 1.0), (1, 0.7), (3, 0.7)])
def test_speculative_sampling_is_lossless_chi2(gamma, T):
    V = 16
    p, q, tokens, st = _sampling_run(gamma, T, seed=2024 + gamma)
    a = st.accepted_len
    assert (st.done == 1).all() and (st.next_token >= 0).all()
    assert st.ambiguous.mean() < 1e-3
    # first emitted token ~ p_0
    first = np.where(a >= 1, tokens[:, 1], st.next_token)
    s, crit, dof = _chi2_ok(np.bincount(first, minlength=V), p[0])
    assert s < crit, (s, crit, dof)
    # acceptance of draft 1: sum_v min(p0, q0)
    acc = np.minimum(p[0], q[0]).sum()
    n = len(a)
    z = ((a >= 1).mean() - acc) / np.sqrt(acc * (1 - acc) / n)
    assert abs(z) < 4.0, z
    # after a rejection at draft 1 the token is ~ normalize(max(0, p0 - q0))
    res = np.maximum(p[0] - q[0], 0)
    res /= res.sum()
    rej = st.next_token[a == 0]
    s, crit, _ = _chi2_ok(np.bincount(rej, minlength=V), res)
    assert s < crit
    # second emitted token given the first draft accepted ~ p_1
    m = a >= 1
    second = np.where(a[m] >= 2, tokens[m, 2] if gamma >= 2 else -1, st.next_token[m])
    s, crit, _ = _chi2_ok(np.bincount(second, minlength=V), p[1])
    assert s < crit


def test_bonus_token_after_all_accepted_is_p_of_last_row():
    V = 16
    p, q, tokens, st = _sampling_run(1, 1.0, seed=77)
    bonus = st.next_token[st.accepted_len == 1]
    s, crit, _ = _chi2_ok(np.bincount(bonus, minlength=V), p[1])
    assert s < crit


@pytest.mark.parametrize("V,T", [(18, 1.0), (13, 0.7)])
def test_grouped_race_with_a_short_last_group_chi2(V, T):
    # Vocabularies that are not a multiple of four: the last group of the
    # race is short.  First emitted token ~ p0, residual after a rejection ~
    # normalize(max(0, p0 - q0)), bonus ~ p1.
    p, q, tokens, st = _sampling_run(1, T, seed=31 + V, N=600_000, V=V)
    a = st.accepted_len
    assert st.ambiguous.mean() < 1e-3
    first = np.where(a >= 1, tokens[:, 1], st.next_token)
    s, crit, _ = _chi2_ok(np.bincount(first, minlength=V), p[0])
    assert s < crit
    res = np.maximum(p[0] - q[0], 0)
    res /= res.sum()
    s, crit, _ = _chi2_ok(np.bincount(st.next_token[a == 0], minlength=V), res)
    assert s < crit
    s, crit, _ = _chi2_ok(np.bincount(st.next_token[a == 1], minlength=V), p[1])
    assert s < crit


def test_chi2_detects_a_planted_mistake_inside_the_group():
    # A second step that always took the group's first entry (the group race
    # alone) gives the right group but the wrong entry: the statistics reject
    # it.
    V = 16
    p, q, tokens, st = _sampling_run(1, 1.0, seed=41, N=300_000)
    bonus = st.next_token[st.accepted_len == 1]
    s, crit, _ = _chi2_ok(np.bincount(bonus, minlength=V), p[1])
    assert s < crit
    wrong = bonus - bonus % 4
    s, crit, _ = _chi2_ok(np.bincount(wrong, minlength=V), p[1])
    assert s > crit


def test_chi2_detects_a_planted_mistake():
    # The same statistics reject a sampler that resamples from p instead of
    # the residual: the test above has the power to see that mistake.
    V = 16
    p, q, tokens, st = _sampling_run(1, 1.0, seed=99, N=300_000)
    rng = np.random.default_rng(5)
    wrong = np.where(st.accepted_len >= 1, tokens[:, 1],
                     rng.choice(V, size=len(st.accepted_len), p=p[0]))
    s, crit, _ = _chi2_ok(np.bincount(wrong, minlength=V), p[0])
    assert s > crit


def test_row_stats_match_torch_log_softmax():
    w = wl.make_workload(wl.config("batch64"), n_req=8, ctx_scale=0.02, vocab=2000)
    T = w.cfg.temperature
    err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits, T, w.seed)
    assert err == 0
    rs = st.row_stats
    for i in range(w.n_req):
        cu = w.cu_rows[i]
        rows = w.cu_rows[i + 1] - cu
        a = st.accepted_len[i]
        for r in range(rows):
            x = torch.from_numpy((w.target_logits[cu + r] / np.float32(T)).astype(np.float32)).double()
            np.testing.assert_allclose(rs[cu + r, 0], torch.logsumexp(x, 0).item(), rtol=0, atol=1e-12)
            if 1 <= r <= min(a + 1, rows - 1):
                lp = torch.log_softmax(
                    torch.from_numpy((w.target_logits[cu + r - 1] / np.float32(T)).astype(np.float32)).double(), 0)
                lq = torch.log_softmax(
                    torch.from_numpy((w.draft_logits[cu + r - 1] / np.float32(T)).astype(np.float32)).double(), 0)
                tok = w.tokens[cu + r]
                np.testing.assert_allclose(rs[cu + r, 2], lp[tok].exp().item(), rtol=1e-12)
                np.testing.assert_allclose(rs[cu + r, 3], lq[tok].exp().item(), rtol=1e-12)


# ---------------------------------------------------------------- windows --

@pytest.mark.parametrize("T", [0.7, 0.0])
def test_chunked_equals_one_pass(T):
    w = wl.make_workload(wl.config("batch64"), n_req=24, ctx_scale=0.01, vocab=300,
                         temperature=T, draft_sigma=0.6)
    H = w.cfg.n_q_heads
    draft = w.draft_logits if T > 0 else None
    err, st1 = oracle.accept(w.batch(), w.target_logits, draft, T, w.seed)
    assert err == 0
    _, _, full64 = oracle.tree_attend(w.batch(), w.kv(), w.q, H, w.softmax_scale)
    err, st2, _, ch64, attended = oracle.verify_chunked(
        w.batch(), w.kv(), w.q, H, w.softmax_scale, w.target_logits, draft, T, w.seed, chunk=2)
    assert err == 0
    assert np.array_equal(st1.accepted_len, st2.accepted_len)
    assert np.array_equal(st1.accepted_nodes, st2.accepted_nodes)
    assert np.array_equal(st1.next_token, st2.next_token)
    assert np.array_equal(st1.ambiguous, st2.ambiguous)
    # attended rows equal; rows after the chunk holding the first rejection never attended
    pruned = 0
    for i in range(w.n_req):
        cu, rows = w.cu_rows[i], w.cu_rows[i + 1] - w.cu_rows[i]
        last_chunk = st1.accepted_len[i] // 2
        for r in range(rows):
            if r // 2 <= last_chunk:
                assert np.array_equal(ch64[cu + r], full64[cu + r])
            else:
                assert np.isnan(ch64[cu + r]).all()
                pruned += 1
    assert attended == w.total_rows - pruned
    assert pruned > 0  # the workload does prune


def test_verify_len_truncates_the_chain():
    w = wl.make_workload(wl.config("batch256"), n_req=16, ctx_scale=0.01, vocab=300, draft_sigma=0.3)
    T = w.cfg.temperature
    vl = np.array([0, 1, 2, 3, 4] * 3 + [2], dtype=np.int32)
    err, st = oracle.accept(w.batch(verify_len=vl), w.target_logits, w.draft_logits, T, w.seed)
    assert err == 0
    assert (st.accepted_len <= vl).all()
    assert (st.next_token >= 0).all()
    # with all drafts considered, a request that accepted all of its first
    # vl drafts decides the same drafts in the same way
    err, full = oracle.accept(w.batch(), w.target_logits, w.draft_logits, T, w.seed)
    for i in range(w.n_req):
        if st.accepted_len[i] < vl[i]:
            assert full.accepted_len[i] == st.accepted_len[i]
            assert full.next_token[i] == st.next_token[i]
        else:
            assert full.accepted_len[i] >= vl[i]


# ------------------------------------------------------- tree sampling --
# Draft trees at T > 0 whose siblings are drawn i.i.d. from the parent's q
# (with replacement): children tried in index order against the residual
# left by the siblings rejected before them.  Lossless means the first
# emitted token is distributed as p_root, and, given that the walk accepted
# node c, the next emitted token is distributed as p_c.

def _tree_batch(n_req, parent1, tokens):
    rows = len(parent1)
    cu = np.arange(n_req + 1, dtype=np.int32) * rows
    parent = np.tile(np.asarray(parent1, dtype=np.int32), n_req)
    return {"cu_rows": cu, "parent": parent, "tokens": tokens.astype(np.int32).ravel(),
            "max_rows": rows}


def _tree_run(parent1, T, seed, N=600_000, V=16, bias=1.0):
    rng = np.random.default_rng(7 + len(parent1) * 13 + int(T * 10))
    rows = len(parent1)
    lt = (rng.standard_normal((rows, V)) * 2.0).astype(np.float32)
    ld = (lt + bias * rng.standard_normal((rows, V))).astype(np.float32)
    p = [_softmax_T(lt[r], T) for r in range(rows)]
    q = [_softmax_T(ld[r], T) for r in range(rows)]
    tokens = np.zeros((N, rows), dtype=np.int32)
    for c in range(1, rows):
        tokens[:, c] = rng.choice(V, size=N, p=q[parent1[c]])  # i.i.d. siblings from q_parent
    b = _tree_batch(N, parent1, tokens)
    target = np.ascontiguousarray(np.broadcast_to(lt, (N, rows, V)).reshape(N * rows, V))
    draft = np.ascontiguousarray(np.broadcast_to(ld, (N, rows, V)).reshape(N * rows, V))
    err, st = oracle.accept(b, target, draft, T, seed)
    assert err == 0
    return p, q, tokens, st


TREES = {
    "one child": [-1, 0],
    "three siblings": [-1, 0, 0, 0],
    "two levels": [-1, 0, 0, 1, 1, 2, 2],
}


@pytest.mark.parametrize("shape,T", [("one child", 1.0), ("three siblings", 1.0),
                                     ("three siblings", 0.7), ("two levels", 1.0)])
def test_tree_sampling_is_lossless_chi2(shape, T):
    V = 16
    par = TREES[shape]
    p, q, tokens, st = _tree_run(par, T, seed=31 + len(par))
    a = st.accepted_len
    nodes = st.accepted_nodes
    assert (st.next_token >= 0).all() and (st.done == 1).all()
    assert st.ambiguous.mean() < 1e-3
    # accepted path is a root-to-node path of the tree
    for r in range(0, len(a), 9973):
        for k in range(1, a[r] + 1):
            assert par[nodes[r, k]] == nodes[r, k - 1]
    # first emitted token ~ p_root
    n1 = nodes[:, 1]
    first = np.where(a >= 1, tokens[np.arange(len(a)), np.maximum(n1, 0)], st.next_token)
    s, crit, dof = _chi2_ok(np.bincount(first, minlength=V), p[0])
    assert s < crit, (s, crit, dof)
    # given the walk accepted node c at depth 1, the next token ~ p_c
    for c in [ch for ch in range(1, len(par)) if par[ch] == 0]:
        m = (a >= 1) & (n1 == c)
        if m.sum() < 20_000:
            continue
        n2 = nodes[m, 2] if nodes.shape[1] > 2 else np.zeros(m.sum(), dtype=np.int64)
        second = np.where(a[m] >= 2, tokens[np.where(m)[0], np.maximum(n2, 0)], st.next_token[m])
        s, crit, _ = _chi2_ok(np.bincount(second, minlength=V), p[c])
        assert s < crit, (c, s, crit)


def test_tree_sampling_with_one_child_equals_the_chain_rule():
    # A one-child tree is a chain of one draft: same decisions, same tokens.
    V = 16
    p, q, tokens, st_tree = _tree_run([-1, 0], 1.0, seed=5, N=20_000)
    b = _chain_batch(20_000, 1, tokens)
    rng = np.random.default_rng(7 + 2 * 13 + 10)
    lt = (rng.standard_normal((2, V)) * 2.0).astype(np.float32)
    ld = (lt + rng.standard_normal((2, V))).astype(np.float32)
    target = np.ascontiguousarray(np.broadcast_to(lt, (20_000, 2, V)).reshape(-1, V))
    draft = np.ascontiguousarray(np.broadcast_to(ld, (20_000, 2, V)).reshape(-1, V))
    err, st_chain = oracle.accept(b, target, draft, 1.0, 5)
    assert err == 0
    assert np.array_equal(st_tree.accepted_len, st_chain.accepted_len)
    assert np.array_equal(st_tree.next_token, st_chain.next_token)


def test_tree_sampling_chi2_detects_a_planted_mistake():
    # Resampling from p_root instead of the siblings' residual after all of
    # them were rejected is seen by the same statistics.
    V = 16
    p, q, tokens, st = _tree_run(TREES["three siblings"], 1.0, seed=44, N=300_000)
    rng = np.random.default_rng(9)
    a = st.accepted_len
    wrong = np.where(a >= 1, tokens[np.arange(len(a)), np.maximum(st.accepted_nodes[:, 1], 0)],
                     rng.choice(V, size=len(a), p=p[0]))
    s, crit, _ = _chi2_ok(np.bincount(wrong, minlength=V), p[0])
    assert s > crit


def test_tree_residual_after_sibling_rejections_matches_the_closed_form():
    # After j rejections the residual is max(0, p - c_j q) / S(c_j) with
    # c_{j+1} = c_j + S(c_j): checked against the step-by-step definition
    # normalize(max(0, p' - q)) in numpy on a random pair of rows.
    rng = np.random.default_rng(3)
    p = rng.dirichlet(np.ones(40))
    q = rng.dirichlet(np.ones(40))
    pres, c, S = p.copy(), 0.0, 1.0
    for _ in range(4):
        nxt = np.maximum(pres - q, 0.0)
        if nxt.sum() == 0:
            break
        pres = nxt / nxt.sum()
        c += S
        S = np.maximum(p - c * q, 0.0).sum()
        assert np.allclose(pres, np.maximum(p - c * q, 0.0) / S, rtol=1e-12, atol=1e-15)
