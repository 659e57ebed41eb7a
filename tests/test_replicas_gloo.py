"""The N > 1 path on the CPU: two gloo ranks (no GPU).

The verification step has no exchange between ranks, so N GPUs run N
replicas; the ranks share only the timing protocol (barrier, slowest rank's
time, sum of units).  These tests run that protocol with world size 2 over
gloo, and the reference arm under torchrun, where only rank 0 may report.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    from speculative_decoding_verification_padding_gb300.replicas import Replicas
    reps = Replicas.from_env("gloo")
    # rank r "processed" 100 * (r + 1) rows in 0.5 * (r + 1) seconds
    units, secs = 100.0 * (rank + 1), 0.5 * (rank + 1)
    reps.barrier()
    t = reps.max_over_ranks(secs)
    u = reps.sum_over_ranks(units)
    thr = reps.throughput(units, secs)
    reps.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"t": t, "u": u, "thr": thr, "leader": reps.leader, "world": reps.world}, f)
    reps.close()


def test_two_gloo_ranks_share_slowest_time_and_total_units(tmp_path):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["world"] == 2
        assert d["leader"] == (r == 0)
        assert d["t"] == pytest.approx(1.0)          # the slower rank's time
        assert d["u"] == pytest.approx(300.0)        # both ranks' units
        assert d["thr"] == pytest.approx(300.0)      # units / slowest time


def test_single_process_needs_no_process_group(monkeypatch):
    from speculative_decoding_verification_padding_gb300.replicas import Replicas
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    reps = Replicas.from_env("gloo")
    assert reps.world == 1 and reps.leader
    reps.barrier()
    assert reps.max_over_ranks(2.5) == 2.5
    assert reps.throughput(10.0, 2.0) == 5.0
    reps.close()


def test_reference_arm_under_torchrun_prints_one_line():
    """`bench.py --impl reference` with two ranks: rank 0 times the oracle and
    prints the only JSON line; rank 1 exits 0 without work."""
    pytest.importorskip("numpy")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--workload", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle"
