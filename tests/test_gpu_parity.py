"""GPU parity: every call of libspecverify, through the C ABI, against the
CPU oracle on the same seeded inputs.

Bars: token ids, accepted lengths and paths, block tables, free lists,
cache lengths and budget selections bit-exact (sampling decisions the oracle
or the device flags as ambiguous, |u - min(1, p/q)| < 1e-6 or a race too
close to call in fp32, are reported and excluded); attention within 1e-2
absolute and 1e-2 relative of the fp64 oracle (bf16 output, fp32
accumulation); probabilities within 1e-5 absolute.
"""

import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_padding_gb300 import api, build
from speculative_decoding_verification_padding_gb300 import sps as sps_mod
from speculative_decoding_verification_padding_gb300 import workloads as wl
from speculative_decoding_verification_padding_gb300.step import DeviceStep, HostPipeline

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
PROB_ATOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()


def _bf16_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _check_attention(gpu_out, ref64, rows):
    g = _bf16_to_f64(gpu_out)[rows]
    r = ref64[rows]
    assert np.isfinite(g).all()
    np.testing.assert_allclose(g, r, atol=ATOL, rtol=RTOL)


def _compare_accept(res, st, w, label=""):
    """Bit-exact comparison of the accept state, ambiguous requests excluded."""
    amb = (st.ambiguous != 0) | (res["ambiguous"] != 0)
    n_amb = int(amb.sum())
    ok = ~amb
    assert np.array_equal(res["accepted_len"][ok], st.accepted_len[ok]), label
    assert np.array_equal(res["next_token"][ok], st.next_token[ok]), label
    assert np.array_equal(res["done"][ok], st.done[ok]), label
    for i in np.nonzero(ok)[0]:
        a = st.accepted_len[i]
        assert np.array_equal(res["accepted_nodes"][i, : a + 1], st.accepted_nodes[i, : a + 1]), (label, i)
        assert (res["accepted_nodes"][i, a + 1:] == -1).all()
    assert n_amb <= max(1, len(amb) // 100), f"{label}: {n_amb} ambiguous decisions"
    return n_amb


# ---------------------------------------------------------------- attention --

ATTN_CASES = {
    "tiny": dict(),
    "chain8b": dict(),
    "tree70b": dict(),
    "batch64_small": dict(name="batch64", n_req=64, ctx_scale=0.05, vocab=256),
    "batch256_small": dict(name="batch256", n_req=96, ctx_scale=0.02, vocab=256),
    "ragged_ctx": dict(name="batch64", n_req=9, ctx_scale=0.0007, vocab=64),  # contexts of a few tokens
    # one-pass calls of at most four requests whose split groups all fit on
    # the GPU as 16-CTA clusters at once (14 such clusters on a GB300): every
    # split group is one thread-block cluster merging through shared memory --
    # mixed contexts (2 KV heads: 12 groups), a context shorter than sixteen
    # pages (empty splits), a long context (64-page splits)
    "cluster_mixed": dict(name="batch64", n_req=4, ctx_scale=0.5, vocab=64,
                          cfg=dict(n_q_heads=8, n_kv_heads=2)),
    "cluster_short": dict(name="chain8b", ctx_scale=0.01, vocab=64),
    "cluster_long": dict(name="chain8b", ctx_scale=4.0, vocab=64),
    # more groups than fit at once: the merge kernel instead
    "small_many_groups": dict(name="batch64", n_req=3, ctx_scale=0.004, vocab=64),
}


def _make(case, **extra):
    kw = dict(ATTN_CASES[case]) if case in ATTN_CASES else {}
    name = kw.pop("name", case)
    cfg = kw.pop("cfg", {})
    kw.setdefault("vocab", 1024 if name != "tiny" else None)
    if kw["vocab"] is None:
        kw.pop("vocab")
    kw.update(extra)
    return wl.make_workload(wl.config(name, **cfg), **kw)


@pytest.mark.parametrize("case", list(ATTN_CASES))
def test_tree_attend_matches_oracle(case):
    w = _make(case)
    s = DeviceStep(w, mode="onepass")
    s.out.fill_(float("nan"))
    s.attend()
    torch.cuda.synchronize()
    assert s.dev_status.item() == 0
    err, _, ref64 = oracle.tree_attend(w.batch(), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale)
    assert err == 0
    _check_attention(s.out, ref64, np.arange(w.total_rows))


def test_tree_attend_windows_touch_only_window_rows():
    w = _make("batch64_small")
    s = DeviceStep(w, mode="onepass")
    rows = np.diff(w.cu_rows)
    rng = np.random.default_rng(1)
    rb = np.array([rng.integers(0, r) for r in rows], dtype=np.int32)
    re = np.array([rng.integers(b, r + 1) for b, r in zip(rb, rows)], dtype=np.int32)
    b = api.Batch(s.batch.cu_rows, s.batch.parent, s.batch.tokens, w.max_rows,
                  row_begin=torch.from_numpy(rb).cuda(), row_end=torch.from_numpy(re).cuda())
    s.out.fill_(float("nan"))
    s.attend(b)
    torch.cuda.synchronize()
    err, _, ref64 = oracle.tree_attend(w.batch(), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale,
                                       row_begin=rb, row_end=re)
    inside = np.zeros(w.total_rows, bool)
    for i in range(w.n_req):
        inside[w.cu_rows[i] + rb[i]: w.cu_rows[i] + re[i]] = True
    _check_attention(s.out, ref64, np.nonzero(inside)[0])
    assert torch.isnan(s.out[torch.from_numpy(~inside).cuda()].float()).all()


# ------------------------------------------------------------------- accept --

ACCEPT_CASES = [
    ("tiny", 0.0, None), ("tiny", 1.0, None),
    ("chain8b", 1.0, 0.3), ("chain8b", 1.0, 1.0), ("chain8b", 1.0, 3.0),
    ("tree70b", 0.0, 1.0), ("tree70b", 0.0, 0.2),
    ("batch64", 0.7, 1.0), ("batch64", 0.0, 1.0),
    ("batch256", 1.0, 1.0),
]


@pytest.mark.parametrize("name,T,sigma", ACCEPT_CASES)
def test_accept_matches_oracle(name, T, sigma):
    kw = dict(temperature=T, ctx_scale=0.01)
    if sigma is not None:
        kw["draft_sigma"] = sigma
    w = wl.make_workload(wl.config(name), **kw)
    s = DeviceStep(w, mode="onepass")
    rs = torch.full((w.total_rows, 4), float("nan"), dtype=torch.float32, device="cuda")
    s.accept(row_stats=rs)
    res = s.results()
    assert res["dev_status"] == 0
    err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits if T > 0 else None, T, w.seed)
    assert err == 0
    _compare_accept(res, st, w, f"{name} T={T} sigma={sigma}")
    g = rs.cpu().numpy().astype(np.float64)
    o = st.row_stats
    if T > 0:
        for i in range(w.n_req):
            if st.ambiguous[i] or res["ambiguous"][i]:
                continue
            cu, a = w.cu_rows[i], st.accepted_len[i]
            rows = w.cu_rows[i + 1] - cu
            np.testing.assert_allclose(g[cu: cu + rows, 0], o[cu: cu + rows, 0], rtol=2e-6, atol=2e-5)
            dec = np.arange(cu + 1, cu + min(a + 2, rows))  # decided children
            np.testing.assert_allclose(g[dec, 2], o[dec, 2], atol=PROB_ATOL, rtol=0)
            np.testing.assert_allclose(g[dec, 3], o[dec, 3], atol=PROB_ATOL, rtol=0)
    else:
        assert np.array_equal(g[:, 1], o[:, 1])  # argmax
        assert np.array_equal(g[:, 0], o[:, 0])  # max logit


@pytest.mark.parametrize("vocab,T", [(1021, 0.7), (13, 1.0), (130, 1.0)])
def test_accept_odd_vocab_matches_oracle(vocab, T):
    # vocabularies that are not a multiple of four: scalar loads, and the
    # residual / bonus race has a short last group
    w = wl.make_workload(wl.config("batch64"), n_req=48, ctx_scale=0.01, vocab=vocab,
                         temperature=T, draft_sigma=0.5)
    s = DeviceStep(w, mode="onepass")
    s.accept()
    res = s.results()
    assert res["dev_status"] == 0
    err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits, T, w.seed)
    assert err == 0
    _compare_accept(res, st, w, f"vocab {vocab} T={T}")
    assert (st.accepted_len < np.diff(w.cu_rows) - 1).any()  # some residual draws


def test_accept_verify_len_truncation():
    w = wl.make_workload(wl.config("batch256"), n_req=64, ctx_scale=0.01, vocab=4096, draft_sigma=0.3)
    vl = np.random.default_rng(2).integers(0, 5, w.n_req).astype(np.int32)
    s = DeviceStep(w, mode="onepass")
    b = api.Batch(s.batch.cu_rows, s.batch.parent, s.batch.tokens, w.max_rows,
                  verify_len=torch.from_numpy(vl).cuda())
    s.accept(b)
    res = s.results()
    err, st = oracle.accept(w.batch(verify_len=vl), w.target_logits, w.draft_logits, 1.0, w.seed)
    assert err == 0
    _compare_accept(res, st, w, "verify_len")


# ------------------------------------------------------------------- commit --

@pytest.mark.parametrize("name,T,kw", [
    ("tree70b", 0.0, dict(ctx_scale=0.01, vocab=512, draft_sigma=0.05)),
    ("batch64", 0.7, dict(ctx_scale=0.01, vocab=512, draft_sigma=0.5)),
    ("tiny", 1.0, dict(vocab=64)),
])
def test_commit_matches_oracle(name, T, kw):
    w = wl.make_workload(wl.config(name), temperature=T, **kw)
    err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits if T > 0 else None, T, w.seed)
    assert err == 0
    if name == "tree70b":
        assert st.accepted_len.max() >= 2  # a path that moves slots
    s = DeviceStep(w, mode="onepass")
    s.accepted_len.copy_(torch.from_numpy(st.accepted_len))
    nodes = np.where(st.accepted_nodes < 0, -1, st.accepted_nodes).astype(np.int32)
    s.accepted_nodes.copy_(torch.from_numpy(nodes))
    s.commit()
    torch.cuda.synchronize()
    assert s.dev_status.item() == 0
    kv = w.kv_copy()
    fl = w.free_list.copy()
    fc = np.array([w.free_count], dtype=np.int32)
    assert oracle.commit_kv(w.batch(), kv, st.accepted_len, nodes, fl, fc) == 0
    assert np.array_equal(s.kv.block_tables.cpu().numpy(), kv["block_tables"])
    assert np.array_equal(s.kv.cache_lens.cpu().numpy(), kv["cache_lens"])
    assert s.pool.free_count.item() == fc[0]
    assert np.array_equal(s.pool.free_list.cpu().numpy()[: fc[0]], fl[: fc[0]])
    assert np.array_equal(s.kv.k_cache.view(torch.int16).cpu().numpy().view(np.uint16), kv["k_cache"])
    assert np.array_equal(s.kv.v_cache.view(torch.int16).cpu().numpy().view(np.uint16), kv["v_cache"])


@pytest.mark.parametrize("name,T,kw", [
    ("batch64", 0.7, dict(n_req=48, ctx_scale=0.02, vocab=2048, draft_sigma=0.5)),
    ("batch64", 0.0, dict(n_req=48, ctx_scale=0.02, vocab=2048, draft_sigma=0.1)),
    ("tree70b", 0.0, dict(ctx_scale=0.01, vocab=512, draft_sigma=0.05)),
    # several trees: one CTA per request shares the merge and the K/V moves
    # (up to eight requests), and the per-warp decision beyond that
    ("tree70b", 0.0, dict(n_req=5, ctx_scale=0.01, vocab=512, draft_sigma=0.05)),
    ("tree70b", 0.0, dict(n_req=11, ctx_scale=0.01, vocab=512, draft_sigma=0.05)),
    ("tree70b", 1.0, dict(n_req=3, ctx_scale=0.01, vocab=2048, draft_sigma=0.3)),
    ("batch256", 1.0, dict(n_req=200, ctx_scale=0.01, vocab=1024)),
])
def test_accept_commit_fused_matches_oracle(name, T, kw):
    # sv_accept_commit == oracle accept followed by oracle commit: decisions,
    # tables, lengths, the free list in order, and every K/V byte
    w = wl.make_workload(wl.config(name), temperature=T, **kw)
    vl = None
    if name == "batch256":
        _, vl, _, _ = oracle.select_budget(w.cond_survival, w.gamma, w.sps)
    s = DeviceStep(w, mode="onepass")
    b = s.batch if vl is None else api.Batch(s.batch.cu_rows, s.batch.parent, s.batch.tokens,
                                             w.max_rows, verify_len=torch.from_numpy(vl).cuda())
    s.accept_commit(b)
    res = s.results()
    assert res["dev_status"] == 0
    err, st = oracle.accept(w.batch(verify_len=vl), w.target_logits,
                            w.draft_logits if T > 0 else None, T, w.seed)
    assert err == 0
    _compare_accept(res, st, w, f"fused {name} T={T}")
    if (st.ambiguous != 0).any() or (res["ambiguous"] != 0).any():
        pytest.skip("an ambiguous decision: the commit inputs differ by construction")
    if name == "tree70b" and T == 0.0:
        assert st.accepted_len.max() >= 2  # a path that moves slots
    kv = w.kv_copy()
    fl = w.free_list.copy()
    fc = np.array([w.free_count], dtype=np.int32)
    nodes = np.where(st.accepted_nodes < 0, -1, st.accepted_nodes).astype(np.int32)
    assert oracle.commit_kv(w.batch(verify_len=vl), kv, st.accepted_len, nodes, fl, fc) == 0
    assert np.array_equal(s.kv.block_tables.cpu().numpy(), kv["block_tables"])
    assert np.array_equal(s.kv.cache_lens.cpu().numpy(), kv["cache_lens"])
    assert s.pool.free_count.item() == fc[0]
    assert np.array_equal(s.pool.free_list.cpu().numpy()[: fc[0]], fl[: fc[0]])
    assert np.array_equal(s.kv.k_cache.view(torch.int16).cpu().numpy().view(np.uint16), kv["k_cache"])
    assert np.array_equal(s.kv.v_cache.view(torch.int16).cpu().numpy().view(np.uint16), kv["v_cache"])


def test_commit_pool_overflow_is_flagged_not_faulted():
    w = wl.make_workload(wl.config("batch64"), n_req=16, ctx_scale=0.01, vocab=256,
                         temperature=0.0, draft_sigma=3.0)
    err, st = oracle.accept(w.batch(), w.target_logits, None, 0.0, w.seed)
    nodes = np.where(st.accepted_nodes < 0, -1, st.accepted_nodes).astype(np.int32)
    # the oracle, given the same full free list, must also overflow
    fl = w.free_list[: w.free_count].copy()
    fc = np.array([w.free_count], dtype=np.int32)
    assert oracle.commit_kv(w.batch(), w.kv_copy(), st.accepted_len, nodes, fl, fc) & oracle.ORC_POOL_OVERFLOW
    s = DeviceStep(w, mode="onepass")
    s.accepted_len.copy_(torch.from_numpy(st.accepted_len))
    s.accepted_nodes.copy_(torch.from_numpy(nodes))
    pool = api.BlockPool(s.pool.free_list[: w.free_count].clone(), s.pool.free_count)
    api.sv_commit_kv(s.kv, s.batch, s.accepted_len, s.accepted_nodes, pool, s.dev_status)
    torch.cuda.synchronize()
    assert s.dev_status.item() & api.N.SV_DEV_POOL_OVERFLOW
    assert pool.free_count.item() == w.free_count


# ------------------------------------------------------------------- budget --

def _budget_gpu(c, gamma, sps):
    R = c.shape[0]
    vl = torch.zeros(R, dtype=torch.int32, device="cuda")
    bB = torch.zeros(1, dtype=torch.int32, device="cuda")
    th = torch.zeros(1, dtype=torch.float64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.sv_select_budget(torch.from_numpy(c).cuda(), None if gamma is None else torch.from_numpy(gamma).cuda(),
                         torch.from_numpy(sps).cuda(), vl, bB, th, None, st)
    torch.cuda.synchronize()
    return vl.cpu().numpy(), int(bB.item()), float(th.item()), int(st.item())


def test_budget_full_size_matches_oracle():
    w = wl.make_workload(wl.config("batch256"), vocab=64, ctx_scale=0.001)
    vl, bB, th, st = _budget_gpu(w.cond_survival, w.gamma, w.sps)
    err, vl_o, bB_o, th_o = oracle.select_budget(w.cond_survival, w.gamma, w.sps)
    assert st == 0 and err == 0
    assert np.array_equal(vl, vl_o) and bB == bB_o and th == th_o


@pytest.mark.skipif(not os.path.exists(sps_mod.MEASURED), reason="no measured SPS table stored")
def test_budget_with_measured_sps_matches_oracle():
    # the SPS(B) table measured from this library's own kernels on GB300
    w = wl.make_workload(wl.config("batch256"), vocab=64, ctx_scale=0.001, sps="measured")
    vl, bB, th, st = _budget_gpu(w.cond_survival, w.gamma, w.sps)
    err, vl_o, bB_o, th_o = oracle.select_budget(w.cond_survival, w.gamma, w.sps)
    assert st == 0 and err == 0
    assert np.array_equal(vl, vl_o) and bB == bB_o and th == th_o
    assert 256 <= bB <= 256 + int(w.gamma.sum())


@pytest.mark.parametrize("trial", range(40))
def test_budget_random_matches_oracle(trial):
    rng = np.random.default_rng(1000 + trial)
    R = int(rng.integers(1, 400))
    gmax = int(rng.integers(1, 9))
    gamma = rng.integers(0, gmax + 1, R).astype(np.int32)
    c = rng.beta(4, 2, size=(R, gmax)).astype(np.float32)
    if trial % 4 == 0:
        c = np.round(c * 4) / 4  # many equal survivals: tie order matters
        c = c.astype(np.float32)
    b_max = R + int(rng.integers(0, R * gmax + 2))
    B = np.arange(b_max + 1, dtype=np.float64)
    sps = (1000.0 / (1.0 + B / rng.uniform(16, 2048))).astype(np.float32)
    vl, bB, th, st = _budget_gpu(c, gamma, sps)
    err, vl_o, bB_o, th_o = oracle.select_budget(c, gamma, sps)
    assert st == 0 and err == 0
    assert np.array_equal(vl, vl_o) and bB == bB_o and th == th_o


@pytest.mark.parametrize("R,gmax", [(1024, 8), (8192, 1), (2048, 4)])
def test_budget_at_the_largest_candidate_count_matches_oracle(R, gmax):
    # n_req * gamma_max = 8192 candidates, the documented limit, with many
    # equal survivals (tie order) and an SPS table long enough for every B
    rng = np.random.default_rng(R + gmax)
    c = (np.round(rng.beta(4, 2, size=(R, gmax)) * 16) / 16).astype(np.float32)
    gamma = rng.integers(0, gmax + 1, R).astype(np.int32)
    B = np.arange(R + R * gmax + 1, dtype=np.float64)
    sps = (1000.0 / (1.0 + B / 2048.0)).astype(np.float32)
    vl, bB, th, st = _budget_gpu(c, gamma, sps)
    err, vl_o, bB_o, th_o = oracle.select_budget(c, gamma, sps)
    assert st == 0 and err == 0
    assert np.array_equal(vl, vl_o) and bB == bB_o and th == th_o


# ------------------------------------------------------------ draft length --

def test_budget_negative_zero_survival_matches_oracle():
    """Survival factors of -0.0 mixed in: the kernel keys them as +0, like the
    oracle."""
    rng = np.random.default_rng(5)
    R, gmax = 200, 4
    c = rng.beta(4, 2, size=(R, gmax)).astype(np.float32)
    c[rng.random(c.shape) < 0.2] = np.float32(-0.0)
    gamma = rng.integers(0, gmax + 1, R).astype(np.int32)
    sps = (1000.0 / (1.0 + np.arange(R * (gmax + 1) + 1) / 256.0)).astype(np.float32)
    err, vl, bB, th = oracle.select_budget(c, gamma, sps)
    assert err == 0
    dev = "cuda"
    out_vl = torch.zeros(R, dtype=torch.int32, device=dev)
    out_B = torch.zeros(1, dtype=torch.int32, device=dev)
    out_th = torch.zeros(1, dtype=torch.float64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    api.sv_select_budget(torch.from_numpy(c).to(dev), torch.from_numpy(gamma).to(dev),
                         torch.from_numpy(sps).to(dev), out_vl, out_B, out_th, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(out_vl.cpu().numpy(), vl)
    assert out_B.item() == bB and out_th.item() == th


@pytest.mark.parametrize("trial", range(4))
def test_adapt_gamma_matches_oracle(trial):
    rng = np.random.default_rng(500 + trial)
    R = int(rng.integers(1, 3000))
    verified = rng.integers(-1, 9, R).astype(np.int32)
    acc = np.minimum(rng.integers(0, 9, R), np.maximum(verified, 0)).astype(np.int32)
    if trial == 3:
        acc[::7] = verified[::7] + 1  # some inconsistent lengths: reported, skipped
    state = (rng.random((R, 2)) * rng.integers(0, 50, (R, 1))).astype(np.float64)
    state[:, 0] = np.minimum(state[:, 0], state[:, 1])
    decay, overhead, gmin, gmax = [(0.7, 2.0, 1, 8), (0.9, 0.5, 0, 16), (1.0, 4.0, 2, 6),
                                   (0.5, 1.0, 1, 8)][trial]
    st_o = state.copy()
    err, g_o = oracle.adapt_gamma(acc, verified, st_o, decay, overhead, gmin, gmax)
    st_g = torch.from_numpy(state).cuda()
    g_g = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.sv_adapt_gamma(torch.from_numpy(acc).cuda(), torch.from_numpy(verified).cuda(), st_g, g_g,
                       decay, overhead, gmin, gmax, status)
    torch.cuda.synchronize()
    assert np.array_equal(g_g.cpu().numpy(), g_o)
    assert np.array_equal(st_g.cpu().numpy(), st_o)  # every bit of the fp64 state
    assert bool(status.item() & api.N.SV_DEV_BAD_LENGTH) == bool(err & oracle.ORC_BAD_LENGTH)


# -------------------------------------------------------------- chunk size --

def _chunk_inputs(R, seed, bad=()):
    rng = np.random.default_rng(seed)
    rows = rng.integers(1, 10, R).astype(np.int32)
    ctx = np.clip(np.rint(rng.lognormal(np.log(4096), 1.0, R)), 512, 32768).astype(np.int32)
    N = rng.uniform(0, 40, R)
    S = N * rng.uniform(0, 1, R)
    st = np.ascontiguousarray(np.stack([S, N], axis=1))
    for i in bad:
        rows[i] = 0 if i % 2 else 200
    return rows, ctx, st


@pytest.mark.parametrize("R,seed,bad,chunk_mb", [(64, 0, (), 170), (1, 1, (), 0), (1000, 2, (), 50),
                                                  (64, 3, (5, 17), 170), (300, 4, (), 0)])
def test_select_chunk_matches_oracle(R, seed, bad, chunk_mb):
    rows, ctx, st = _chunk_inputs(R, seed, bad)
    kv, row, cb = 4096.0, 2 * 4 * 128256.0, chunk_mb * 10 ** 6
    err, ch, cost, costs = oracle.select_chunk(rows, ctx, st, kv, row, cb)
    dev = "cuda"
    t_rows, t_ctx, t_st = (torch.from_numpy(rows).to(dev), torch.from_numpy(ctx).to(dev),
                           torch.from_numpy(st).to(dev))
    g_ch = torch.zeros(1, dtype=torch.int32, device=dev)
    g_cost = torch.zeros(1, dtype=torch.int64, device=dev)
    g_costs = torch.zeros(128, dtype=torch.int64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    api.sv_select_chunk(t_rows, t_ctx, t_st, kv, row, cb, g_ch, g_cost, g_costs, status)
    torch.cuda.synchronize()
    assert g_ch.item() == ch
    assert g_cost.cpu().numpy().view(np.uint64)[0] == np.uint64(cost)
    assert np.array_equal(g_costs.cpu().numpy().view(np.uint64), costs)
    assert bool(status.item() & api.N.SV_DEV_BAD_LENGTH) == bool(err & oracle.ORC_BAD_LENGTH)


def test_select_chunk_prefers_one_pass_at_batch64_on_this_gpu():
    # the bench workload's first-step acceptance, this GPU's per-chunk fixed
    # cost (about 25 us of plan, statistics and decision at 6.8 TB/s): the
    # chunked step re-reads context for little pruning, one pass is cheapest
    w = wl.make_workload(wl.config("batch64"))
    err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits, w.cfg.temperature, w.seed)
    rows = np.diff(w.cu_rows).astype(np.int32)
    a = st.accepted_len
    state = np.ascontiguousarray(np.stack([a, a + (a < rows - 1)], axis=1).astype(np.float64))
    dev = "cuda"
    g_ch = torch.zeros(1, dtype=torch.int32, device=dev)
    g_cost = torch.zeros(1, dtype=torch.int64, device=dev)
    g_costs = torch.zeros(128, dtype=torch.int64, device=dev)
    api.sv_select_chunk(torch.from_numpy(rows).to(dev),
                        torch.from_numpy(w.cache_lens.astype(np.int32)).to(dev),
                        torch.from_numpy(state).to(dev), 4096.0, 2 * 4 * 128256.0,
                        170 * 10 ** 6, g_ch, g_cost, g_costs)
    torch.cuda.synchronize()
    assert g_ch.item() == rows.max()
    c = g_costs.cpu().numpy().view(np.uint64)
    assert c[1] > c[rows.max() - 1]  # chunks of 2 cost more than one pass


# ------------------------------------------------------- chunked / budget step --

@pytest.mark.parametrize("T", [0.7, 0.0])
def test_chunked_step_matches_oracle(T):
    w = wl.make_workload(wl.config("batch64"), ctx_scale=0.05, vocab=2048, temperature=T,
                         draft_sigma=0.7)
    s = DeviceStep(w, mode="chunked")
    s.out.fill_(float("nan"))
    s.chunked()
    res = s.results()
    assert res["dev_status"] == 0
    err, st, _, ref64, attended = oracle.verify_chunked(
        w.batch(), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale, w.target_logits,
        w.draft_logits if T > 0 else None, T, w.seed, chunk=2)
    assert err == 0
    _compare_accept(res, st, w, f"chunked T={T}")
    att = ~np.isnan(ref64[:, 0, 0])
    assert int(att.sum()) == attended < w.total_rows  # pruning happened
    _check_attention(s.out, ref64, np.nonzero(att)[0])
    assert torch.isnan(s.out[torch.from_numpy(~att).cuda()].float()).all()


def _check_commit_against_oracle(s, w, st, vl=None, skip=()):
    """The cache state after a fused commit == oracle commit of the oracle's
    decisions (requests in `skip` are left as they were: the oracle is
    given an invalid length for them)."""
    kv = w.kv_copy()
    fl = w.free_list.copy()
    fc = np.array([w.free_count], dtype=np.int32)
    nodes = np.where(st.accepted_nodes < 0, -1, st.accepted_nodes).astype(np.int32)
    al = st.accepted_len.astype(np.int32).copy()
    al[list(skip)] = -1
    err = oracle.commit_kv(w.batch(verify_len=vl), kv, al, nodes, fl, fc)
    assert err == (oracle.ORC_BAD_WINDOW if len(skip) else 0)
    assert np.array_equal(s.kv.block_tables.cpu().numpy(), kv["block_tables"])
    assert np.array_equal(s.kv.cache_lens.cpu().numpy(), kv["cache_lens"])
    assert s.pool.free_count.item() == fc[0]
    assert np.array_equal(s.pool.free_list.cpu().numpy()[: fc[0]], fl[: fc[0]])
    assert np.array_equal(s.kv.k_cache.view(torch.int16).cpu().numpy().view(np.uint16), kv["k_cache"])
    assert np.array_equal(s.kv.v_cache.view(torch.int16).cpu().numpy().view(np.uint16), kv["v_cache"])


@pytest.mark.parametrize("name,T,chunk,kw", [
    ("batch64", 0.7, 2, dict(n_req=48, ctx_scale=0.02, vocab=2048, draft_sigma=0.5)),
    ("batch64", 0.0, 2, dict(n_req=48, ctx_scale=0.02, vocab=2048, draft_sigma=0.1)),
    ("batch64", 0.7, 3, dict(n_req=40, ctx_scale=0.05, vocab=2048, draft_sigma=0.3)),
    ("tree70b", 0.0, None, dict(ctx_scale=0.01, vocab=512, draft_sigma=0.05)),
    ("tree70b", 1.0, None, dict(n_req=3, ctx_scale=0.01, vocab=2048, draft_sigma=0.3)),
    # a chunked call of three requests: small splits merged by the merge kernel
    ("batch64", 0.7, 2, dict(n_req=3, ctx_scale=0.3, vocab=2048, draft_sigma=0.5)),
])
def test_chunked_commit_fused_matches_oracle(name, T, chunk, kw):
    # sv_verify_chunked_commit == oracle chunked verification followed by the
    # oracle commit: decisions, attention of the attended rows, tables,
    # lengths, the free list in order and every K/V byte.  Trees are taken
    # whole by the first chunk (chunk = max rows), at T > 0 by the tree walk.
    w = wl.make_workload(wl.config(name), temperature=T, **kw)
    chunk = chunk or w.max_rows
    s = DeviceStep(w, mode="chunked", chunk=chunk)
    s.out.fill_(float("nan"))
    s.run()
    res = s.results()
    assert res["dev_status"] == 0
    err, st, _, ref64, attended = oracle.verify_chunked(
        w.batch(), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale, w.target_logits,
        w.draft_logits if T > 0 else None, T, w.seed, chunk=chunk)
    assert err == 0
    _compare_accept(res, st, w, f"chunked commit {name} T={T} chunk={chunk}")
    att = ~np.isnan(ref64[:, 0, 0])
    assert int(att.sum()) == attended
    _check_attention(s.out, ref64, np.nonzero(att)[0])
    if name == "tree70b":
        assert st.accepted_len.max() >= 2  # a path that moves slots
    if (st.ambiguous != 0).any() or (res["ambiguous"] != 0).any():
        pytest.skip("an ambiguous decision: the commit inputs differ by construction")
    _check_commit_against_oracle(s, w, st)


def test_more_requests_than_the_planner_keeps_in_shared_memory():
    # 1300 requests: the planner's per-request records live in the workspace,
    # its threads take several requests each; one-pass attention and a chunked
    # step with the fused commit, both against the oracle
    w = wl.make_workload(wl.config("batch64"), n_req=1300, ctx_scale=0.002, vocab=64,
                         temperature=0.7, draft_sigma=0.7)
    s = DeviceStep(w, mode="onepass")
    s.out.fill_(float("nan"))
    s.attend()
    torch.cuda.synchronize()
    assert s.dev_status.item() == 0
    err, _, ref64 = oracle.tree_attend(w.batch(), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale)
    assert err == 0
    _check_attention(s.out, ref64, np.arange(w.total_rows))
    c = DeviceStep(w, mode="chunked")
    c.run()
    res = c.results()
    assert res["dev_status"] == 0
    err, st, _, _, _ = oracle.verify_chunked(
        w.batch(), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale, w.target_logits,
        w.draft_logits, 0.7, w.seed, chunk=2)
    assert err == 0
    _compare_accept(res, st, w, "1300 requests chunked")
    lens = c.kv.cache_lens.cpu().numpy()
    assert np.array_equal(lens, w.cache_lens + 1 + res["accepted_len"])


def test_chunked_commit_in_one_chunk_equals_the_one_pass_fused_commit():
    # a chunk that holds every row: the chunked step with its fused commit
    # leaves exactly the state of sv_accept_commit after sv_tree_attend
    kw = dict(n_req=24, ctx_scale=0.02, vocab=1024, temperature=0.7, draft_sigma=0.5)
    w = wl.make_workload(wl.config("batch64"), **kw)
    a = DeviceStep(w, mode="chunked", chunk=w.max_rows)
    a.run()
    ra = a.results()
    b = DeviceStep(w, mode="onepass")
    b.run()
    rb = b.results()
    assert ra["dev_status"] == 0 and rb["dev_status"] == 0
    for k in ("accepted_len", "accepted_nodes", "next_token", "ambiguous", "done"):
        assert np.array_equal(ra[k], rb[k]), k
    for x, y in ((a.kv.block_tables, b.kv.block_tables), (a.kv.cache_lens, b.kv.cache_lens),
                 (a.pool.free_count, b.pool.free_count)):
        assert torch.equal(x, y)
    n = b.pool.free_count.item()
    assert torch.equal(a.pool.free_list[:n], b.pool.free_list[:n])
    assert torch.equal(a.kv.k_cache, b.kv.k_cache) and torch.equal(a.kv.v_cache, b.kv.v_cache)


@pytest.mark.parametrize("vocab", [2, 3, 5])
def test_accept_tiny_vocab_matches_oracle(vocab):
    # one short race group (or one and a bit): the second step picks inside it
    w = wl.make_workload(wl.config("batch64"), n_req=40, ctx_scale=0.01, vocab=vocab,
                         temperature=1.0, draft_sigma=1.0)
    s = DeviceStep(w, mode="onepass")
    s.accept()
    res = s.results()
    assert res["dev_status"] == 0
    err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits, 1.0, w.seed)
    assert err == 0
    _compare_accept(res, st, w, f"vocab {vocab}")


def test_select_chunk_without_requests():
    dev = "cuda"
    e = torch.zeros(0, dtype=torch.int32, device=dev)
    ch = torch.full((1,), -5, dtype=torch.int32, device=dev)
    cost = torch.full((1,), 7, dtype=torch.int64, device=dev)
    costs = torch.zeros(128, dtype=torch.int64, device=dev)
    api.sv_select_chunk(e, e, torch.zeros((0, 2), dtype=torch.float64, device=dev), 4096.0, 1.0,
                        1000, ch, cost, costs)
    torch.cuda.synchronize()
    err, och, ocost, ocosts = oracle.select_chunk([], [], np.zeros((0, 2)), 4096.0, 1.0, 1000)
    assert err == 0
    assert ch.item() == och and cost.item() == ocost
    assert np.array_equal(costs.cpu().numpy().view(np.uint64), ocosts)


@pytest.mark.parametrize("T", [0.7, 0.0])
def test_chunked_commit_with_truncated_requests_matches_oracle(T):
    # verify_len cuts some chains short (budget-selected prefixes verified in
    # chunks): windows stop at verify_len + 1 rows, the commit still releases
    # every staged row past the accepted path
    w = wl.make_workload(wl.config("batch64"), n_req=40, ctx_scale=0.02, vocab=1024,
                         temperature=T, draft_sigma=0.3)
    rows = np.diff(w.cu_rows).astype(np.int32)
    vl = np.minimum(rows - 1, np.random.default_rng(9).integers(0, 9, w.n_req)).astype(np.int32)
    s = DeviceStep(w, mode="chunked")
    b = api.Batch(s.batch.cu_rows, s.batch.parent, s.batch.tokens, w.max_rows,
                  verify_len=torch.from_numpy(vl).cuda())
    api.sv_verify_chunked_commit(s.kv, b, s.q, s.Hq, s.scale, s.out, s.target, s.draft, s.V, s.T,
                                 w.seed, 2, s.accepted_len, s.accepted_nodes, s.next_token,
                                 s.ambiguous, s.done, s.pool, s.ws, s.dev_status)
    res = s.results()
    assert res["dev_status"] == 0
    err, st, _, _, _ = oracle.verify_chunked(
        w.batch(verify_len=vl), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale, w.target_logits,
        w.draft_logits if T > 0 else None, T, w.seed, chunk=2)
    assert err == 0
    _compare_accept(res, st, w, f"chunked commit verify_len T={T}")
    assert (st.accepted_len <= vl).all()
    if (st.ambiguous != 0).any() or (res["ambiguous"] != 0).any():
        pytest.skip("an ambiguous decision: the commit inputs differ by construction")
    _check_commit_against_oracle(s, w, st, vl=vl)


@pytest.mark.parametrize("mode,name,kw", [
    ("onepass", "batch64", dict(n_req=24, ctx_scale=0.02, vocab=1024, temperature=0.7)),
    ("chunked", "batch64", dict(n_req=24, ctx_scale=0.02, vocab=1024, temperature=0.7)),
    ("budget", "batch256", dict(n_req=48, ctx_scale=0.01, vocab=512)),
    ("onepass", "tree70b", dict(ctx_scale=0.01, vocab=512, temperature=1.0, draft_sigma=0.3)),
])
def test_results_do_not_depend_on_workspace_contents(mode, name, kw):
    # every workspace word a call reads is written by that call first: the
    # same step on a zeroed and on a garbage-filled workspace (one request
    # with an invalid window in the chunked case) leaves the same state
    w = wl.make_workload(wl.config(name), **kw)
    vl = None
    if mode == "chunked":
        vl = np.diff(w.cu_rows).astype(np.int32) - 1
        vl[3] = -1

    def run(fill):
        s = DeviceStep(w, mode=mode)
        s.ws.fill_(fill)
        if mode == "chunked":
            b = api.Batch(s.batch.cu_rows, s.batch.parent, s.batch.tokens, w.max_rows,
                          verify_len=torch.from_numpy(vl).cuda())
            api.sv_verify_chunked_commit(s.kv, b, s.q, s.Hq, s.scale, s.out, s.target, s.draft,
                                         s.V, s.T, w.seed, 2, s.accepted_len, s.accepted_nodes,
                                         s.next_token, s.ambiguous, s.done, s.pool, s.ws,
                                         s.dev_status)
        else:
            s.run()
        res = s.results()
        n = s.pool.free_count.item()
        return res, (s.kv.block_tables.cpu(), s.kv.cache_lens.cpu(), s.pool.free_list[:n].cpu(),
                     s.kv.k_cache.cpu(), s.out.cpu())

    r0, c0 = run(0)
    r1, c1 = run(0xA5)
    for k in ("accepted_len", "accepted_nodes", "next_token", "ambiguous", "dev_status"):
        assert np.array_equal(r0[k], r1[k]), k
    for x, y in zip(c0, c1):
        assert torch.equal(x, y)


def test_chunked_commit_invalid_window_is_left_alone():
    # one request with verify_len < 0: reported, never listed, never
    # committed; every other request is committed and the release still runs
    w = wl.make_workload(wl.config("batch64"), n_req=24, ctx_scale=0.02, vocab=1024,
                         temperature=0.7, draft_sigma=0.5)
    vl = np.diff(w.cu_rows).astype(np.int32) - 1
    bad = 5
    vl[bad] = -1
    s = DeviceStep(w, mode="chunked")
    b = api.Batch(s.batch.cu_rows, s.batch.parent, s.batch.tokens, w.max_rows,
                  verify_len=torch.from_numpy(vl).cuda())
    api.sv_verify_chunked_commit(s.kv, b, s.q, s.Hq, s.scale, s.out, s.target, s.draft, s.V, s.T,
                                 w.seed, 2, s.accepted_len, s.accepted_nodes, s.next_token,
                                 s.ambiguous, s.done, s.pool, s.ws, s.dev_status)
    res = s.results()
    assert res["dev_status"] & api.N.SV_DEV_BAD_WINDOW
    err, st, _, _, _ = oracle.verify_chunked(
        w.batch(verify_len=vl), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale, w.target_logits,
        w.draft_logits, 0.7, w.seed, chunk=2)
    assert err & oracle.ORC_BAD_WINDOW
    keep = np.arange(w.n_req) != bad
    amb = (st.ambiguous != 0) | (res["ambiguous"] != 0)
    ok = keep & ~amb
    assert np.array_equal(res["accepted_len"][ok], st.accepted_len[ok])
    assert np.array_equal(res["next_token"][ok], st.next_token[ok])
    if amb.any():
        pytest.skip("an ambiguous decision: the commit inputs differ by construction")
    _check_commit_against_oracle(s, w, st, vl=vl, skip=(bad,))


def test_budget_step_matches_oracle():
    w = wl.make_workload(wl.config("batch256"), ctx_scale=0.02, vocab=2048)
    s = DeviceStep(w, mode="budget")
    s.out.fill_(float("nan"))
    s.run(commit=False)
    res = s.results()
    assert res["dev_status"] == 0
    err, vl, bB, th = oracle.select_budget(w.cond_survival, w.gamma, w.sps)
    assert np.array_equal(s.verify_len.cpu().numpy(), vl) and s.best_B.item() == bB
    err, st = oracle.accept(w.batch(verify_len=vl), w.target_logits, w.draft_logits, 1.0, w.seed)
    assert err == 0
    _compare_accept(res, st, w, "budget step")
    err, _, ref64 = oracle.tree_attend(w.batch(verify_len=vl), w.kv(), w.q, w.cfg.n_q_heads,
                                       w.softmax_scale)
    att = ~np.isnan(ref64[:, 0, 0])
    assert att.sum() == w.n_req + vl.sum()
    _check_attention(s.out, ref64, np.nonzero(att)[0])


# ------------------------------------------------------------- losslessness --

@pytest.mark.parametrize("gamma,T", [(3, 1.0), (1, 0.7)])
def test_gpu_speculative_sampling_chi2(gamma, T):
    from scipy import stats
    N, V = 1_000_000, 16
    rows = gamma + 1
    rng = np.random.default_rng(77 + gamma)
    lt = (rng.standard_normal((rows, V)) * 2.0).astype(np.float32)
    ld = (lt + rng.standard_normal((rows, V))).astype(np.float32)

    def sm(l):
        x = (l / np.float32(T)).astype(np.float64)
        e = np.exp(x - x.max())
        return e / e.sum()
    p0, q0 = sm(lt[0]), sm(ld[0])
    tokens = np.zeros((N, rows), dtype=np.int32)
    for j in range(1, rows):
        tokens[:, j] = rng.choice(V, size=N, p=sm(ld[j - 1]))
    cu = (np.arange(N + 1) * rows).astype(np.int32)
    parent = np.tile(np.arange(-1, gamma, dtype=np.int32), N)
    dev = "cuda"
    b = api.Batch(torch.from_numpy(cu).to(dev), torch.from_numpy(parent).to(dev),
                  torch.from_numpy(tokens.ravel()).to(dev), rows)
    tgt = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(lt, (N, rows, V)).reshape(-1, V))).to(dev)
    drf = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(ld, (N, rows, V)).reshape(-1, V))).to(dev)
    al = torch.zeros(N, dtype=torch.int32, device=dev)
    an = torch.zeros((N, rows), dtype=torch.int32, device=dev)
    nt = torch.zeros(N, dtype=torch.int32, device=dev)
    amb = torch.zeros(N, dtype=torch.uint8, device=dev)
    ws = api.workspace(api.sv_accept_workspace(b, V))
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    api.sv_accept(b, tgt, drf, V, T, 4242, al, an, nt, amb, None, None, ws, st)
    a, nxt = al.cpu().numpy(), nt.cpu().numpy()
    assert st.item() == 0 and (nxt >= 0).all()
    first = np.where(a >= 1, tokens[:, 1], nxt)
    obs = np.bincount(first, minlength=V)
    chi = ((obs - p0 * N) ** 2 / (p0 * N)).sum()
    assert chi < stats.chi2.ppf(0.999, V - 1), chi
    acc = np.minimum(p0, q0).sum()
    z = ((a >= 1).mean() - acc) / np.sqrt(acc * (1 - acc) / N)
    assert abs(z) < 4
    # the first 20000 requests decide exactly as the oracle does
    n = 20000
    bo = {"cu_rows": cu[: n + 1], "parent": parent[: n * rows], "tokens": tokens[:n].ravel(),
          "max_rows": rows}
    err, so = oracle.accept(bo, np.broadcast_to(lt, (n, rows, V)).reshape(-1, V),
                            np.broadcast_to(ld, (n, rows, V)).reshape(-1, V), T, 4242)
    ok = (so.ambiguous == 0) & (amb.cpu().numpy()[:n] == 0)
    assert np.array_equal(a[:n][ok], so.accepted_len[ok])
    assert np.array_equal(nxt[:n][ok], so.next_token[ok])


# ---------------------------------------------------------- device findings --

def test_bad_block_id_and_bad_parent_are_flagged():
    w = _make("tiny", vocab=64)
    s = DeviceStep(w, mode="onepass")
    tbl = s.kv.block_tables.clone()
    s.kv.block_tables[0, 3] = w.k_cache.shape[0] + 5
    s.attend()
    torch.cuda.synchronize()
    assert s.dev_status.item() & api.N.SV_DEV_BAD_BLOCK_ID
    s.kv.block_tables.copy_(tbl)
    s.dev_status.zero_()
    par = s.batch.parent.clone()
    par[2] = 5
    b = api.Batch(s.batch.cu_rows, par, s.batch.tokens, w.max_rows)
    s.attend(b)
    s.accept(b)
    torch.cuda.synchronize()
    assert s.dev_status.item() & api.N.SV_DEV_BAD_PARENT


# Tree sampling (T > 0, siblings drawn i.i.d. from the parent's q): the walk,
# the sibling-residual passes and the final draw against the oracle, on the
# 64-node tree at small and full vocabulary, with several draft qualities.
@pytest.mark.parametrize("vocab,sigma,T", [(256, 1.0, 1.0), (4096, 0.5, 0.7), (4096, 3.0, 1.0),
                                           (128256, 1.0, 1.0)])
def test_tree_sampling_matches_oracle(vocab, sigma, T):
    n_same = 0
    for seed in range(6):
        w = wl.make_workload(wl.config("tree70b"), ctx_scale=0.01, vocab=vocab, temperature=T,
                             draft_sigma=sigma, step_seed=1000 + seed)
        s = DeviceStep(w, mode="onepass")
        s.accept()
        res = s.results()
        assert res["dev_status"] == 0
        err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits, T, w.seed)
        assert err == 0
        if st.ambiguous[0] or res["ambiguous"][0]:
            continue
        _compare_accept(res, st, w, f"tree vocab={vocab} sigma={sigma} seed={seed}")
        n_same += 1
    assert n_same >= 4


def test_tree_sampling_batch_of_trees_matches_oracle():
    # several trees in one call (one CTA each), mixed with nothing else
    w = wl.make_workload(wl.config("tree70b"), n_req=5, ctx_scale=0.01, vocab=2048,
                         temperature=1.0, draft_sigma=0.7)
    s = DeviceStep(w, mode="onepass")
    s.accept()
    res = s.results()
    assert res["dev_status"] == 0
    err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits, 1.0, w.seed)
    assert err == 0
    _compare_accept(res, st, w, "five trees")


def test_small_tree_sampling_walks_on_one_cta_and_matches_oracle():
    # trees of at most 16 rows are walked by a single CTA (deeper ones by a
    # 16-CTA cluster): both walks against the oracle on the same kind of input
    import dataclasses
    n_same = 0
    for seed in range(6):
        cfg = dataclasses.replace(wl.config("tree70b"), gamma=("tree", (3, 2, 2), 15), n_req=2)
        w = wl.make_workload(cfg, ctx_scale=0.01, vocab=2048, temperature=1.0, draft_sigma=0.7,
                             step_seed=2000 + seed)
        assert w.max_rows <= 16
        s = DeviceStep(w, mode="onepass")
        s.accept()
        res = s.results()
        assert res["dev_status"] == 0
        err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits, 1.0, w.seed)
        assert err == 0
        if st.ambiguous.any() or res["ambiguous"].any():
            continue
        _compare_accept(res, st, w, f"small trees seed={seed}")
        n_same += 1
    assert n_same >= 4


# ------------------------------------------------------- the largest windows --
# 128 rows per request (the 128-bit ancestor masks' upper word, decision
# windows longer than a warp, merges of more than 32 row/type pairs).

def _max_rows_workload(kind, T=0.0, sigma=0.05, n_req=3):
    import dataclasses
    if kind == "chain":
        cfg = dataclasses.replace(wl.config("chain8b"), gamma=("fixed", 127), n_req=n_req)
    else:
        cfg = dataclasses.replace(wl.config("tree70b"), gamma=("tree", (4, 3, 2, 2, 2, 2, 2), 127),
                                  n_req=n_req)
    return wl.make_workload(cfg, ctx_scale=0.01, vocab=512, draft_sigma=sigma, temperature=T)


@pytest.mark.parametrize("kind", ["chain", "tree"])
def test_attend_128_rows_matches_oracle(kind):
    w = _max_rows_workload(kind)
    assert w.max_rows == 128
    s = DeviceStep(w, mode="onepass")
    s.out.fill_(float("nan"))
    s.attend()
    torch.cuda.synchronize()
    assert s.dev_status.item() == 0
    err, _, ref64 = oracle.tree_attend(w.batch(), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale)
    assert err == 0
    _check_attention(s.out, ref64, np.arange(w.total_rows))


@pytest.mark.parametrize("kind,T,sigma", [("chain", 0.0, 0.05), ("chain", 1.0, 0.02),
                                          ("tree", 0.0, 0.05), ("tree", 1.0, 0.05)])
def test_accept_commit_128_rows_matches_oracle(kind, T, sigma):
    w = _max_rows_workload(kind, T, sigma)
    s = DeviceStep(w, mode="onepass")
    s.accept_commit()
    res = s.results()
    assert res["dev_status"] == 0
    err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits if T > 0 else None, T, w.seed)
    assert err == 0
    _compare_accept(res, st, w, f"128 rows {kind} T={T}")
    if kind == "chain":
        assert st.accepted_len.max() > 32  # the decision ran past one warp's lanes
    if (st.ambiguous != 0).any() or (res["ambiguous"] != 0).any():
        return
    kv = w.kv_copy()
    fl = w.free_list.copy()
    fc = np.array([w.free_count], dtype=np.int32)
    nodes = np.where(st.accepted_nodes < 0, -1, st.accepted_nodes).astype(np.int32)
    assert oracle.commit_kv(w.batch(), kv, st.accepted_len, nodes, fl, fc) == 0
    assert np.array_equal(s.kv.block_tables.cpu().numpy(), kv["block_tables"])
    assert np.array_equal(s.pool.free_list.cpu().numpy()[: fc[0]], fl[: fc[0]])
    assert np.array_equal(s.kv.k_cache.view(torch.int16).cpu().numpy().view(np.uint16), kv["k_cache"])


def test_chunked_128_rows_matches_one_pass():
    w = _max_rows_workload("chain", 0.7, 0.02, n_req=4)
    s = DeviceStep(w, mode="chunked")
    s.chunked()
    res = s.results()
    assert res["dev_status"] == 0
    err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits, 0.7, w.seed)
    assert err == 0
    _compare_accept(res, st, w, "chunked 128 rows")


def test_bounded_wait_times_out_and_the_context_survives():
    # the wait every kernel uses, on a barrier nothing completes: it gives up,
    # reports SV_DEV_TIMEOUT, and the next calls run normally
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.sv_selftest_bounded_wait(4096, st)
    torch.cuda.synchronize()
    assert st.item() == api.N.SV_DEV_TIMEOUT
    w = wl.make_workload(wl.config("tiny"))
    s = DeviceStep(w, mode="onepass")
    s.run()
    assert s.results()["dev_status"] == 0


def test_small_workspace_is_refused_before_launch():
    w = _make("tiny", vocab=64)
    s = DeviceStep(w, mode="onepass")
    need = api.sv_tree_attend_workspace(s.batch, s.kv, w.cfg.n_q_heads)
    with pytest.raises(api.N.SpecVerifyError, match="workspace too small"):
        api.sv_tree_attend(s.kv, s.batch, s.q, w.cfg.n_q_heads, w.softmax_scale, s.out,
                           s.ws[: need - 1], s.dev_status)


# ------------------------------------------------ full size, bench launch shape --

@pytest.fixture(scope="module")
def batch64_full():
    return wl.make_workload(wl.config("batch64"))


def test_batch64_full_size_chunked_step(batch64_full):
    """The bench workload at full size, run as the bench runs it (chunked,
    with the commit fused into the chunks): every accept output against the
    oracle, attention on a sample of requests, the new cache lengths."""
    w = batch64_full
    s = DeviceStep(w)
    assert s.mode == "chunked"
    s.out.fill_(float("nan"))
    s.run()
    res = s.results()
    assert res["dev_status"] == 0
    err, st = oracle.accept(w.batch(), w.target_logits, w.draft_logits, w.cfg.temperature, w.seed)
    assert err == 0
    _compare_accept(res, st, w, "batch64 full")
    # attention of every row the chunks reached, all 64 requests
    rb = np.zeros(w.n_req, np.int32)
    rows = np.diff(w.cu_rows).astype(np.int32)
    re = np.minimum(rows, 2 * (st.accepted_len // 2 + 1)).astype(np.int32)
    err, _, ref64 = oracle.tree_attend(w.batch(), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale,
                                       row_begin=rb, row_end=re)
    att = ~np.isnan(ref64[:, 0, 0])
    assert att.sum() == re.sum()
    _check_attention(s.out, ref64, np.nonzero(att)[0])
    # the commit fused into the step == the oracle's commit of the oracle's
    # decisions: every table entry, the cache lengths, the free list in order
    # and every K / V byte of the pool
    amb = (st.ambiguous != 0) | (res["ambiguous"] != 0)
    if amb.any():
        pytest.skip("an ambiguous decision: the commit inputs differ by construction")
    _check_commit_against_oracle(s, w, st)


# ------------------------------------------------ batch256 at full contexts --

@pytest.fixture(scope="module")
def batch256_full():
    return wl.make_workload(wl.config("batch256"))


def _sample_by_context(w, n_each=8, seed=0):
    """The requests with the longest contexts (several KV splits, merged by
    the group's last CTA), the shortest, and some drawn at random."""
    order = np.argsort(w.cache_lens, kind="stable")
    rng = np.random.default_rng(seed)
    mid = rng.choice(order[n_each:-n_each], size=n_each, replace=False)
    return np.unique(np.concatenate([order[-n_each:], order[:n_each], mid]))


def test_batch256_full_contexts_attention(batch256_full):
    """Attention of the batch256 shape (40 q / 8 KV heads: five query heads
    per KV head) at its real contexts, 1024..8192: the longest requests are
    split over the KV and merged; 24 requests against the oracle."""
    w = batch256_full
    s = DeviceStep(w, mode="onepass")
    s.out.fill_(float("nan"))
    s.attend()
    torch.cuda.synchronize()
    assert s.dev_status.item() == 0
    sample = _sample_by_context(w)
    assert len(sample) >= 16 and w.cache_lens[sample].max() > 7800
    rb = np.zeros(w.n_req, np.int32)
    re = np.zeros(w.n_req, np.int32)
    re[sample] = np.diff(w.cu_rows)[sample]
    err, _, ref64 = oracle.tree_attend(w.batch(), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale,
                                       row_begin=rb, row_end=re)
    assert err == 0
    att = ~np.isnan(ref64[:, 0, 0])
    assert att.sum() == re.sum()
    _check_attention(s.out, ref64, np.nonzero(att)[0])


def test_batch256_full_size_budget_step(batch256_full):
    """The budget-selected step as the bench runs it at full size: selection
    bit-exact, every accept result against the oracle at vocab 151936,
    attention of 24 requests on their selected prefixes, and the fused commit
    (tables, lengths, free list in order, every K / V byte)."""
    w = batch256_full
    s = DeviceStep(w, mode="budget")
    s.out.fill_(float("nan"))
    s.run()
    res = s.results()
    assert res["dev_status"] == 0
    err, vl, bB, th = oracle.select_budget(w.cond_survival, w.gamma, w.sps)
    assert err == 0
    assert np.array_equal(s.verify_len.cpu().numpy(), vl)
    assert s.best_B.item() == bB and s.best_theta.item() == th
    err, st = oracle.accept(w.batch(verify_len=vl), w.target_logits, w.draft_logits,
                            w.cfg.temperature, w.seed)
    assert err == 0
    _compare_accept(res, st, w, "batch256 full budget step")
    sample = _sample_by_context(w, seed=1)
    rb = np.zeros(w.n_req, np.int32)
    re = np.zeros(w.n_req, np.int32)
    re[sample] = vl[sample] + 1
    err, _, ref64 = oracle.tree_attend(w.batch(verify_len=vl), w.kv(), w.q, w.cfg.n_q_heads,
                                       w.softmax_scale, row_begin=rb, row_end=re)
    assert err == 0
    att = ~np.isnan(ref64[:, 0, 0])
    assert att.sum() == re.sum()
    _check_attention(s.out, ref64, np.nonzero(att)[0])
    amb = (st.ambiguous != 0) | (res["ambiguous"] != 0)
    if amb.any():
        pytest.skip("an ambiguous decision: the commit inputs differ by construction")
    _check_commit_against_oracle(s, w, st, vl=vl)


def test_bound_calls_equal_the_plain_calls():
    # DeviceStep launches through BoundCall objects (arguments marshalled once);
    # the plain api calls on the same inputs give the same bytes.
    w = _make("chain8b", ctx_scale=0.25, vocab=2048)
    s = DeviceStep(w, mode="onepass")
    s.restore_cache_state()
    s.attend()
    s.accept()
    torch.cuda.synchronize()
    out_b = s.out.clone()
    res_b = [t.clone() for t in (s.accepted_len, s.accepted_nodes, s.next_token, s.ambiguous)]
    s.out.zero_()
    api.sv_tree_attend(s.kv, s.batch, s.q, s.Hq, s.scale, s.out, s.ws, s.dev_status)
    api.sv_accept(s.batch, s.target, s.draft, s.V, s.T, s.w.seed, s.accepted_len,
                  s.accepted_nodes, s.next_token, s.ambiguous, s.done, None, s.ws, s.dev_status)
    torch.cuda.synchronize()
    assert s.dev_status.item() == 0
    assert torch.equal(out_b.view(torch.int16), s.out.view(torch.int16))
    for a_, b_ in zip(res_b, (s.accepted_len, s.accepted_nodes, s.next_token, s.ambiguous)):
        assert torch.equal(a_, b_)


@pytest.mark.parametrize("case,kw", [
    ("chain8b", dict(ctx_scale=0.25, vocab=2048)),                # one pass
    ("batch64", dict(n_req=12, ctx_scale=0.05, vocab=512)),       # chunked
    ("batch256", dict(n_req=24, ctx_scale=0.02, vocab=256)),      # budget selection
])
def test_host_pipeline_steps_equal_plain_steps(case, kw):
    # Double-buffered uploads: steps alternating between two input sets, each
    # step's results read only after the next step was submitted (so its upload
    # overlapped this step's kernels), equal a plain step on the same set.
    w = _make(case, **kw)
    s = DeviceStep(w)
    rng = np.random.default_rng(11)
    base = [t.cpu().clone() for t in s.inputs()]
    alt = [t.clone() for t in base]
    alt[0] = (alt[0].float() * 0.5).to(torch.bfloat16)  # q
    alt[1] = alt[1] + torch.from_numpy(rng.normal(0, 1.5, tuple(alt[1].shape)).astype(np.float32))
    sets = [[t.pin_memory() for t in base], [t.pin_memory() for t in alt]]
    refs = []
    for ins in sets:
        for d, h in zip(s.inputs(), ins):
            d.copy_(h)
        s.run()
        torch.cuda.synchronize()
        assert s.dev_status.item() == 0
        refs.append([t.cpu().clone() for t in s.outputs()])
    assert not torch.equal(refs[0][0].view(torch.int16), refs[1][0].view(torch.int16))
    for d in s.inputs():
        d.zero_()
    pipe = HostPipeline(s)
    pipe.begin()
    n, got, pending = 7, {}, []

    def take():
        j, host, ev = pending.pop(0)
        ev.synchronize()
        got[j] = [t.clone() for t in host]

    for i in range(n):
        pending.append((i,) + pipe.submit(sets[i % 2]))
        if len(pending) == 2:
            take()
    take()
    torch.cuda.synchronize()
    assert s.dev_status.item() == 0
    assert sorted(got) == list(range(n))
    for j in range(n):
        ref = refs[j % 2]
        assert torch.equal(got[j][0].view(torch.int16), ref[0].view(torch.int16)), j
        for a_, b_ in zip(got[j][1:], ref[1:]):
            assert torch.equal(a_, b_), j


def test_host_pipeline_rejects_mismatched_inputs():
    w = _make("chain8b", ctx_scale=0.05, vocab=256)
    s = DeviceStep(w)
    pipe = HostPipeline(s)
    ins = [t.cpu() for t in s.inputs()]
    with pytest.raises(ValueError):
        pipe.submit(ins[:-1])
    ins[1] = ins[1][:-1]
    with pytest.raises(ValueError):
        pipe.submit(ins)
