"""The bench's byte accounting (the numerator of every roofline fraction),
checked on the CPU against the definitions it states and against the
oracle's own count of attended rows.

  attend: per attended request, (ctx_i + window end) x KVB of K/V (context
          plus the staged slots up to the window end) plus Q in and out for
          the window rows, KVB = H_kv d 2 bytes x 2 (K and V);
  accept: per window row the target row (V x 4 bytes), at T > 0 the draft
          row of every row that proposes a tested draft, and the rows the
          residual (target + draft) or bonus (target) draw scans;
  chunked schedule: a request attends chunks 0 .. a // chunk, a its accepted
          drafts -- the same rows the oracle's chunked verification attends.
"""

import math

import numpy as np
import pytest

import bench
import oracle
from speculative_decoding_verification_padding_gb300 import workloads as wl


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def test_attend_bytes_of_the_tiny_step():
    w = wl.make_workload(wl.config("tiny"))
    win = bench.launch_windows(w, "onepass", np.zeros(1, np.int32))
    assert win == [[(0, 0, 5, 5)]]
    kvb = 2 * 64 * 2 * 2        # 2 KV heads, d 64, bf16, K and V
    qo = 8 * 64 * 2 * 2         # 8 q heads: Q in and out
    assert bench.attend_bytes(w, win[0]) == (256 + 5) * kvb + 5 * qo


@pytest.mark.parametrize("T", [0.7, 0.0])
def test_chunked_schedule_attends_the_oracle_rows(T):
    w = wl.make_workload(wl.config("batch64"), n_req=24, ctx_scale=0.01, vocab=256,
                         temperature=T, draft_sigma=0.7)
    err, st, _, _, attended = oracle.verify_chunked(
        w.batch(), w.kv(), w.q, w.cfg.n_q_heads, w.softmax_scale, w.target_logits,
        w.draft_logits if T > 0 else None, T, w.seed, chunk=2)
    assert err == 0
    sched = bench.launch_windows(w, "chunked", st.accepted_len, chunk=2)
    assert len(sched) == math.ceil(w.max_rows / 2)
    assert sum(e - b for ch in sched for _, b, e, _ in ch) == attended
    # and chunk by chunk: a request is listed until the chunk that stops it
    rows = np.diff(w.cu_rows)
    for c, ch in enumerate(sched):
        listed = {i for i, *_ in ch}
        for i in range(w.n_req):
            reaches = 2 * c < rows[i] and st.accepted_len[i] >= 2 * c
            assert (i in listed) == bool(reaches), (c, i)


def test_accept_bytes_follow_the_definition():
    w = wl.make_workload(wl.config("batch64"), n_req=3, ctx_scale=0.01, vocab=100)
    V = 100
    rows = [int(r) for r in np.diff(w.cu_rows)]
    win = [(i, 0, rows[i], rows[i]) for i in range(3)]
    acc = np.array([0, rows[1] - 1, min(1, rows[2] - 1)])
    got = bench.accept_bytes(w, win, acc, 0.7)
    want = 0
    for i in range(3):
        want += rows[i] * V * 4                      # target rows
        want += (rows[i] - 1) * V * 4                # draft rows with a tested child
        bonus = acc[i] == rows[i] - 1
        want += V * 4 if bonus else 2 * V * 4        # bonus: target; residual: both rows
    assert got == want
    # greedy: target rows only
    assert bench.accept_bytes(w, win, acc, 0.0) == sum(rows) * V * 4


def test_attend_flops_follow_the_definition():
    # chain: row j sees the context and rows 0..j (j + 1 staged slots)
    w = wl.make_workload(wl.config("tiny"))
    win = bench.launch_windows(w, "onepass", np.zeros(1, np.int32))
    per_key = 4 * 64 * 8        # QK^T and PV, d 64, 8 query heads
    assert bench.attend_flops(w, win[0]) == per_key * sum(256 + j + 1 for j in range(5))
    # tree: a node sees its ancestors and itself, counted by brute force over
    # the ancestor sets; the 65-row tree at context 8192 is about 17.5 GFLOP
    w = wl.make_workload(wl.config("tree70b"), vocab=64)
    par = w.parent
    depth_sum = 0
    for r in range(w.total_rows):
        anc = {r}
        m = r
        while par[m] >= 0:
            m = int(par[m])
            anc.add(m)
        depth_sum += len(anc)
    per_key = 4 * 128 * 64
    want = per_key * (65 * 8192 + depth_sum)
    win = bench.launch_windows(w, "onepass", np.zeros(1, np.int32))
    assert bench.attend_flops(w, win[0]) == want
    assert abs(want / 1e9 - 17.46) < 0.01


def test_e2e_reports_the_faster_complete_timing_and_names_it():
    t, mode = bench.e2e_choice(2.33e-3, 1.78e-3, False)
    assert t == 1.78e-3 and mode.startswith("double-buffered") and "flush" not in mode
    t, mode = bench.e2e_choice(0.105e-3, 0.205e-3, True)
    assert t == 0.105e-3 and mode.startswith("serial") and "flushed between steps" in mode
    t, mode = bench.e2e_choice(0.279e-3, 0.261e-3, True)
    assert t == 0.261e-3 and "L2 flushes inside the timed region" in mode
    t, mode = bench.e2e_choice(1e-3, 1e-3, False)  # a tie goes to the pipeline
    assert mode.startswith("double-buffered")
