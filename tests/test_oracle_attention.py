"""Pins for the oracle's verification attention (no GPU).

Tree attention of a node is causal attention over the context followed by the
node's own root-to-node path ([SwiftSpec] core design, mechanism 2: every
tree node has its own KV prefix).  The pins rebuild that sequence explicitly,
by walking parent links, and run a library routine over it (torch SDPA in
fp64, GQA expanded), so a wrong mask, a wrong head mapping, a dropped scale
or a mis-indexed page fails here.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_padding_gb300 import workloads as wl


def _dense_keys(w, i, slots, g, which):
    cache = w.k_cache if which == "k" else w.v_cache
    out = []
    for s in slots:
        blk = w.block_tables[i, s // wl.BLOCK_SIZE]
        out.append(wl.bf16_to_f32(cache[blk, g, s % wl.BLOCK_SIZE]).astype(np.float64))
    return np.stack(out)


def _path(parent, cu, r):
    nodes = []
    m = r
    while m >= 0:
        nodes.append(m)
        m = parent[cu + m]
    return nodes[::-1]


def _sdpa_row(w, i, r, h):
    """Attention of packed row (request i, local row r), head h, by SDPA over
    the explicitly gathered key sequence context + path(root -> r)."""
    cfg = w.cfg
    group = cfg.n_q_heads // cfg.n_kv_heads
    g = h // group
    cu = int(w.cu_rows[i])
    ctx = int(w.cache_lens[i])
    slots = list(range(ctx)) + [ctx + m for m in _path(w.parent, cu, r)]
    K = torch.from_numpy(_dense_keys(w, i, slots, g, "k"))
    Vv = torch.from_numpy(_dense_keys(w, i, slots, g, "v"))
    qv = torch.from_numpy(wl.bf16_to_f32(w.q[cu + r, h]).astype(np.float64))
    o = torch.nn.functional.scaled_dot_product_attention(
        qv[None, None, None, :], K[None, None], Vv[None, None], scale=w.softmax_scale)
    return o[0, 0, 0].numpy()


def _small(name, **kw):
    cfg = wl.config(name)
    return wl.make_workload(cfg, **kw)


def test_no_drafts_equals_sdpa_with_gqa_expanded():
    # Rows = 1 (root only): plain decode attention over a paged cache.  The
    # whole head dimension goes through one SDPA call with K/V expanded to the
    # query heads (repeat_interleave), the library's GQA reading.
    cfg = wl.config("batch64", gamma=("fixed", 0))
    w = wl.make_workload(cfg, n_req=5, ctx_scale=0.05, vocab=64)
    err, out_bf16, out64 = oracle.tree_attend(w.batch(), w.kv(), w.q, cfg.n_q_heads, w.softmax_scale)
    assert err == 0
    group = cfg.n_q_heads // cfg.n_kv_heads
    for i in range(w.n_req):
        ctx = int(w.cache_lens[i])
        slots = list(range(ctx + 1))
        K = np.stack([_dense_keys(w, i, slots, g, "k") for g in range(cfg.n_kv_heads)])
        Vv = np.stack([_dense_keys(w, i, slots, g, "v") for g in range(cfg.n_kv_heads)])
        K = torch.from_numpy(K).repeat_interleave(group, dim=0)
        Vv = torch.from_numpy(Vv).repeat_interleave(group, dim=0)
        row = int(w.cu_rows[i])
        qv = torch.from_numpy(wl.bf16_to_f32(w.q[row]).astype(np.float64))  # [H, d]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qv[:, None, :], K, Vv, scale=1.0 / math.sqrt(cfg.head_dim))[:, 0]
        # the oracle takes the fp32 scale; the fp64 exact 1/sqrt(d) differs by < 1e-8
        np.testing.assert_allclose(out64[row], ref.numpy(), rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("name", ["tiny", "tree70b"])
def test_tree_rows_equal_path_attention(name):
    # Every row of a chain (tiny) and of the 64-node tree attends to exactly
    # context + its own path; checked row by row against SDPA.
    w = _small(name, ctx_scale=0.03 if name == "tree70b" else 0.25, vocab=64)
    H = w.cfg.n_q_heads
    err, _, out64 = oracle.tree_attend(w.batch(), w.kv(), w.q, H, w.softmax_scale)
    assert err == 0
    rng = np.random.default_rng(0)
    rows = range(w.total_rows) if name == "tiny" else rng.choice(w.total_rows, 20, replace=False)
    for r in rows:
        for h in ([0, H - 1, H // 2 + 1] if name == "tree70b" else range(H)):
            np.testing.assert_allclose(out64[r, h], _sdpa_row(w, 0, int(r), h), rtol=1e-9, atol=1e-12)


def test_paged_layout_is_invisible():
    # Moving every block to another pool slot (and rewriting the table) must
    # not change one bit of the result.
    w = _small("batch64", n_req=4, ctx_scale=0.05, vocab=64)
    H = w.cfg.n_q_heads
    _, a_bf16, a64 = oracle.tree_attend(w.batch(), w.kv(), w.q, H, w.softmax_scale)
    perm = np.random.default_rng(5).permutation(w.k_cache.shape[0])
    inv = np.argsort(perm)
    kv2 = {"k_cache": np.ascontiguousarray(w.k_cache[perm]),
           "v_cache": np.ascontiguousarray(w.v_cache[perm]),
           "block_tables": np.where(w.block_tables >= 0, inv[np.maximum(w.block_tables, 0)], -1)
           .astype(np.int32),
           "cache_lens": w.cache_lens}
    _, b_bf16, b64 = oracle.tree_attend(w.batch(), kv2, w.q, H, w.softmax_scale)
    assert np.array_equal(a64, b64, equal_nan=True)
    assert np.array_equal(a_bf16, b_bf16)


def test_window_rows_only_and_clipped_by_verify_len():
    w = _small("batch64", n_req=6, ctx_scale=0.03, vocab=64)
    H = w.cfg.n_q_heads
    rows = np.diff(w.cu_rows)
    rb = np.minimum(1, rows - 1).astype(np.int32)
    re = np.minimum(rb + 2, rows).astype(np.int32)
    _, full_bf16, full64 = oracle.tree_attend(w.batch(), w.kv(), w.q, H, w.softmax_scale)
    _, _, win64 = oracle.tree_attend(w.batch(), w.kv(), w.q, H, w.softmax_scale,
                                     row_begin=rb, row_end=re)
    for i in range(w.n_req):
        for r in range(rows[i]):
            p = w.cu_rows[i] + r
            if rb[i] <= r < re[i]:
                assert np.array_equal(win64[p], full64[p])
            else:
                assert np.isnan(win64[p]).all()
    # verify_len = 0 keeps only the root row of every request
    vl = np.zeros(w.n_req, dtype=np.int32)
    _, _, vl64 = oracle.tree_attend(w.batch(verify_len=vl), w.kv(), w.q, H, w.softmax_scale)
    for i in range(w.n_req):
        p = w.cu_rows[i]
        assert np.array_equal(vl64[p], full64[p])
        assert np.isnan(vl64[p + 1: w.cu_rows[i + 1]]).all()


def test_bf16_output_is_rounded_fp64():
    w = _small("tiny", ctx_scale=0.25, vocab=64)
    _, out_bf16, out64 = oracle.tree_attend(w.batch(), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale)
    back = wl.bf16_to_f32(out_bf16).astype(np.float64)
    np.testing.assert_allclose(back, out64, rtol=2 ** -8, atol=0)


def test_bad_inputs_are_reported():
    w = _small("tiny", ctx_scale=0.25, vocab=64)
    H = w.cfg.n_q_heads
    par = w.parent.copy()
    par[2] = 2  # a node that is its own parent
    b = w.batch()
    b["parent"] = par
    err, _, _ = oracle.tree_attend(b, w.kv(), w.q, H, w.softmax_scale)
    assert err & oracle.ORC_BAD_PARENT
    kv = w.kv_copy()
    kv["block_tables"][0, 0] = w.k_cache.shape[0] + 3
    err, _, _ = oracle.tree_attend(w.batch(), kv, w.q, H, w.softmax_scale)
    assert err & oracle.ORC_BAD_BLOCK
