"""The seeded input generator: shapes and structure of the five workloads."""

import numpy as np

from speculative_decoding_verification_padding_gb300 import workloads as wl


def test_tree_shape_depth_profile_and_closure():
    parent, rank = wl.tree_shape((4, 3, 2, 2, 1, 1), 64)
    assert len(parent) == 65 and parent[0] == -1
    assert all(0 <= parent[j] < j for j in range(1, 65))  # breadth-first, parents first
    depth = np.zeros(65, int)
    for j in range(1, 65):
        depth[j] = depth[parent[j]] + 1
    assert list(np.bincount(depth)) == [1, 4, 12, 20, 22, 5, 1]
    # branching never exceeds the per-depth limit
    for n in range(65):
        kids = [c for c in range(65) if parent[c] == n]
        if kids:
            assert len(kids) <= (4, 3, 2, 2, 1, 1)[depth[n]]
            assert sorted(rank[kids]) == list(range(len(kids)))


def test_workload_layout_small():
    w = wl.make_workload(wl.config("batch64"), n_req=10, ctx_scale=0.02, vocab=100)
    rows = np.diff(w.cu_rows)
    assert (rows >= 2).all() and (rows <= 9).all()
    assert w.k_cache.shape[1:] == (8, 16, 128)
    need = -(-(w.cache_lens + rows) // 16)
    used = np.concatenate([w.block_tables[i, :need[i]] for i in range(w.n_req)])
    assert len(np.unique(used)) == len(used)
    assert set(used).isdisjoint(set(w.free_list[: w.free_count]))
    assert len(used) + w.free_count == w.k_cache.shape[0]
    assert ((w.tokens >= 0) & (w.tokens < 100)).all()


def test_budget_inputs():
    w = wl.make_workload(wl.config("batch256"), vocab=32, ctx_scale=0.001)
    assert w.cond_survival.shape == (256, 4) and w.cond_survival.dtype == np.float32
    assert ((w.cond_survival > 0) & (w.cond_survival < 1)).all()
    assert w.sps.shape == (1281,) and (np.diff(w.sps) < 0).all()
    B = np.arange(1281.0)
    assert (np.diff(B * w.sps.astype(np.float64)) > 0).all()  # B * SPS(B) increasing


def test_seeded_inputs_are_reproducible():
    a = wl.make_workload(wl.config("tiny"), vocab=64)
    b = wl.make_workload(wl.config("tiny"), vocab=64)
    assert np.array_equal(a.k_cache, b.k_cache) and np.array_equal(a.tokens, b.tokens)
    assert np.array_equal(a.target_logits, b.target_logits)
