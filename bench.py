"""Benchmark of one verification step per layer on GB300 (one JSON line).

Workload (default): batch of 64 requests, Llama-3-8B attention shape (32 q /
8 KV heads, d 128), per-request draft counts U{1..8}, contexts log-normal
(ln 4096, 1) clipped to [512, 32768], paged bf16 KV (16-token blocks,
shuffled tables), vocab 128256 fp32 logits, sampling at T = 0.7, chunked
verification in chunks of 2 with early pruning, then the KV commit.

One step = restore the block tables / lengths / free list the previous
step's commit changed, sv_verify_chunked (per chunk: windows, tree-prep +
split-KV attention + merge, row statistics + accept/reject + resampling),
sv_commit_kv.  The KV cache (1.7 GB) and the logits (0.36 GB) are larger
than L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 (torchrun, one rank per GPU) every rank runs its own replica of
the step (the path has no exchange step); the line reports the sum over
ranks divided by the slowest rank's time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify steps/s and verified tokens/s per layer; HBM GB/s vs GB300 8 TB/s"
UNIT = "verified tokens/s per layer"


def workload_description(cfg):
    return ("batch64: 64 requests, Llama-3-8B attention shape (32 q / 8 kv heads, d 128), "
            "drafts U{1..8} per request, context lognormal(ln 4096, 1) clipped to [512, 32768], "
            "paged bf16 KV in 16-token blocks with shuffled tables, vocab 128256 fp32 logits, "
            "T=0.7 sampling, chunked verification (chunk 2) with early pruning, KV commit")


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        self.proc = subprocess.Popen([exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                      "-i", str(self.index), "-lms", "100"],
                                     stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------- byte accounting --

def chunk_schedule(w, accepted_len, chunk):
    """Windows each chunk launch processed, from the step's accepted lengths
    (a request runs through chunk accepted_len // chunk)."""
    rows = [int(r) for r in np.diff(w.cu_rows)]
    n_chunks = math.ceil(w.max_rows / chunk)
    sched = []
    for c in range(n_chunks):
        act = []
        for i in range(w.n_req):
            b = c * chunk
            e = min(b + chunk, rows[i])
            if b < e and c <= int(accepted_len[i]) // chunk:
                act.append((i, b, e))
        sched.append(act)
    return sched


def attend_bytes(w, windows):
    cfg = w.cfg
    kvb = cfg.n_kv_heads * cfg.head_dim * 2 * 2
    qo = cfg.n_q_heads * cfg.head_dim * 2 * 2
    return sum((int(w.cache_lens[i]) + e) * kvb + (e - b) * qo for i, b, e in windows)


def accept_bytes(w, windows, accepted_len, T):
    V = int(w.target_logits.shape[1])
    rows = [int(r) for r in np.diff(w.cu_rows)]
    tot = 0
    for i, b, e in windows:
        tot += (e - b) * V * 4                               # target rows
        if T > 0:
            tot += (min(e, rows[i] - 1) - b) * V * 4          # draft rows with a child
            a = int(accepted_len[i])
            if b <= a < e:                                    # decided in this window
                tot += (V * 4 if a == rows[i] - 1 else 2 * V * 4)
    return tot


# ------------------------------------------------------------- CPU baseline --

def oracle_sample(w, n_req, start=0):
    """The first n_req requests of w (from `start`) as a standalone workload."""
    from speculative_decoding_verification_padding_gb300.workloads import Workload
    idx = list(range(start, start + n_req))
    cu = w.cu_rows
    rows = [slice(cu[i], cu[i + 1]) for i in idx]
    new_cu = np.zeros(n_req + 1, dtype=np.int32)
    new_cu[1:] = np.cumsum([cu[i + 1] - cu[i] for i in idx])
    cat = lambda a: np.concatenate([a[s] for s in rows])
    return Workload(cfg=w.cfg, cu_rows=new_cu, parent=cat(w.parent), tokens=cat(w.tokens),
                    max_rows=w.max_rows, k_cache=w.k_cache, v_cache=w.v_cache,
                    block_tables=np.ascontiguousarray(w.block_tables[idx]),
                    cache_lens=np.ascontiguousarray(w.cache_lens[idx]), free_list=w.free_list,
                    free_count=w.free_count, q=cat(w.q), target_logits=cat(w.target_logits),
                    draft_logits=cat(w.draft_logits), seed=w.seed)


def time_oracle(w, n_req, threads, start=0):
    import oracle
    s = oracle_sample(w, n_req, start)
    t0 = time.perf_counter()
    err, st, _, _, attended = oracle.verify_chunked(
        s.batch(), s.kv(), s.q, s.cfg.n_q_heads, s.softmax_scale, s.target_logits,
        s.draft_logits, s.cfg.temperature, s.seed, chunk=s.cfg.chunk or 2, n_threads=threads)
    dt = time.perf_counter() - t0
    return dt, attended, err


def cpu_baseline(w, budget_s=10.0):
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    dt1, att1, _ = time_oracle(w, 1, threads)
    n = int(max(1, min(w.n_req, budget_s / max(dt1, 1e-3))))
    dt, att, err = time_oracle(w, n, threads)
    return {"value": att / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {n} of {w.n_req} requests of the same step, chunked verification "
                      f"(attention + accept), {att} rows attended in {dt:.2f} s, fp64 C++ "
                      f"oracle with {threads} threads", "err": err}


# ------------------------------------------------------------------- main --

def run_reference(args, rank):
    """Reference arm: the CPU oracle, timed on this host's cores."""
    if rank != 0:
        return
    from speculative_decoding_verification_padding_gb300 import workloads as wl
    import oracle
    oracle.build()
    w = wl.make_workload(wl.config(args.workload))
    threads = os.cpu_count() or 1
    dt1, _, _ = time_oracle(w, 1, threads)
    per_step_budget = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    n = int(max(1, min(w.n_req, per_step_budget / max(dt1, 1e-3))))
    for k in range(args.warmup):
        time_oracle(w, n, threads, start=(k * n) % (w.n_req - n + 1))
    tot_t, tot_rows = 0.0, 0
    for k in range(args.steps):
        dt, att, _ = time_oracle(w, n, threads, start=(k * n) % (w.n_req - n + 1))
        tot_t += dt
        tot_rows += att
    value = tot_rows / tot_t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_description(w.cfg), "global_batch": w.n_req,
                       "parallelism": "host threads"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{n} of {w.n_req} requests per step (chunked verification: "
                                       f"attention + accept), fp64 C++ oracle, {threads} threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="batch64")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="only run this many steps (for a profiler), no timing line")
    ap.add_argument("--ctx-scale", type=float, default=1.0,
                    help="with --profile-steps: shrink every context (smaller profiler captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import torch.distributed as dist
    from speculative_decoding_verification_padding_gb300 import api
    from speculative_decoding_verification_padding_gb300 import workloads as wl
    from speculative_decoding_verification_padding_gb300.step import DeviceStep

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(dev))

    w = wl.make_workload(wl.config(args.workload),
                         ctx_scale=args.ctx_scale if args.profile_steps else 1.0)
    s = DeviceStep(w, device=dev)
    chunk = s.chunk
    stream = torch.cuda.current_stream()

    if args.profile_steps:
        for _ in range(args.profile_steps):
            s.run()
        torch.cuda.synchronize()
        return

    for _ in range(args.warmup):
        s.run()
    res = s.results()
    if res["dev_status"] != 0:
        raise SystemExit(f"device status {res['dev_status']} during warm-up")
    al = res["accepted_len"]
    sched = chunk_schedule(w, al, chunk)
    rows_attended = sum(e - b for ch in sched for _, b, e in ch)
    accepted_tokens = int((al + 1).sum())

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(x):
        if world == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)

    # ---- headline: K whole steps, device-resident inputs ----
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        s.run()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_step = max_over_ranks(e0.elapsed_time(e1) / 1e3 / args.steps)

    # ---- per-launch timing of the attention and accept calls, same steps ----
    n_chunks = math.ceil(w.max_rows / chunk)
    rb = torch.zeros(w.n_req, dtype=torch.int32, device=dev)
    re = torch.zeros(w.n_req, dtype=torch.int32, device=dev)
    bw = api.Batch(s.batch.cu_rows, s.batch.parent, s.batch.tokens, w.max_rows, row_begin=rb, row_end=re)
    n_rep = max(5, args.steps // 4)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(n_chunks)] for _ in range(n_rep)]
    torch.cuda.synchronize()
    for k in range(n_rep):
        s.restore_cache_state()
        for c in range(n_chunks):
            api.sv_chunk_windows(s.batch, c, chunk, s.done, rb, re)
            a0, a1, a2 = ev[k][c]
            a0.record(stream)
            s.attend(bw)
            a1.record(stream)
            s.accept(bw)
            a2.record(stream)
        s.commit()
    torch.cuda.synchronize()
    t_att = [[ev[k][c][0].elapsed_time(ev[k][c][1]) / 1e3 for c in range(n_chunks)] for k in range(n_rep)]
    t_acc = [[ev[k][c][1].elapsed_time(ev[k][c][2]) / 1e3 for c in range(n_chunks)] for k in range(n_rep)]
    att_b = [attend_bytes(w, sched[c]) for c in range(n_chunks)]
    acc_b = [accept_bytes(w, sched[c], al, s.T) for c in range(n_chunks)]
    att_time = float(np.mean([sum(t) for t in t_att]))
    acc_time = float(np.mean([sum(t) for t in t_acc]))
    att_gbs = sum(att_b) / att_time / 1e9
    acc_gbs = sum(acc_b) / acc_time / 1e9

    # ---- one-pass attention and accept on the whole batch (no chunking) ----
    full_sched = [(i, 0, int(w.cu_rows[i + 1] - w.cu_rows[i])) for i in range(w.n_req)]
    t1 = torch.cuda.Event(enable_timing=True)
    t2 = torch.cuda.Event(enable_timing=True)
    t3 = torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        s.attend(); s.accept()
    torch.cuda.synchronize()
    t1.record(stream)
    for _ in range(n_rep):
        s.attend()
    t2.record(stream)
    for _ in range(n_rep):
        s.accept()
    t3.record(stream)
    torch.cuda.synchronize()
    op_att = t1.elapsed_time(t2) / 1e3 / n_rep
    op_acc = t2.elapsed_time(t3) / 1e3 / n_rep
    op_att_b = attend_bytes(w, full_sched)
    op_acc_b = accept_bytes(w, full_sched, al, s.T)

    # ---- end to end through host buffers ----
    pin = lambda t: t.cpu().pin_memory()
    h_q, h_tgt, h_drf = pin(s.q), pin(s.target), pin(s.draft)
    h_tok, h_par, h_cu = pin(s.batch.tokens), pin(s.batch.parent), pin(s.batch.cu_rows)
    h_out = torch.empty_like(s.out, device="cpu").pin_memory()
    h_al = torch.empty_like(s.accepted_len, device="cpu").pin_memory()
    h_nodes = torch.empty_like(s.accepted_nodes, device="cpu").pin_memory()
    h_nt = torch.empty_like(s.next_token, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_tgt, h_drf, h_tok, h_par, h_cu))
    d2h = sum(t.numel() * t.element_size() for t in (h_out, h_al, h_nodes, h_nt))
    n_e2e = max(5, args.steps // 4)
    barrier()
    torch.cuda.synchronize()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(n_e2e):
        s.q.copy_(h_q, non_blocking=True)
        s.target.copy_(h_tgt, non_blocking=True)
        s.draft.copy_(h_drf, non_blocking=True)
        s.batch.tokens.copy_(h_tok, non_blocking=True)
        s.batch.parent.copy_(h_par, non_blocking=True)
        s.batch.cu_rows.copy_(h_cu, non_blocking=True)
        s.run()
        h_out.copy_(s.out, non_blocking=True)
        h_al.copy_(s.accepted_len, non_blocking=True)
        h_nodes.copy_(s.accepted_nodes, non_blocking=True)
        h_nt.copy_(s.next_token, non_blocking=True)
    e3.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_e2e = max_over_ranks(e2.elapsed_time(e3) / 1e3 / n_e2e)
    clk = clocks.stop()
    res2 = s.results()
    assert np.array_equal(res2["accepted_len"], al), "steps are not reproducible"

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    import json as _json
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        peaks = _json.load(open(peaks_path))
        hbm_peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    else:
        hbm_peak, peak_src = 6800.0, "fallback"
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "attend_traffic.json")
    if os.path.exists(tr_path):
        tr = _json.load(open(tr_path))
        if tr.get("workload") == args.workload and tr.get("kernel_rev") == KERNEL_REV:
            traffic = tr.get("bytes_per_launch")

    launches_per_step = n_chunks * 5 + 2
    value = world * rows_attended / t_step
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 attention (fp32 accumulate), fp32 softmax",
        "data": "synthetic",
        "config": {"workload": workload_description(w.cfg), "global_batch": w.n_req * world,
                   "rows_per_step": int(w.total_rows), "rows_attended_per_step": int(rows_attended),
                   "chunk": chunk, "vocab": int(w.target_logits.shape[1]),
                   "parallelism": f"replicas x{world}", "l2": "inputs larger than L2 (1.7 GB KV, 0.36 GB logits)"},
        "verify_steps_per_s": world / t_step,
        "accepted_tokens_per_s": world * accepted_tokens / t_step,
        "roofline": {"bound": "hbm", "achieved": att_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": att_gbs / hbm_peak, "traffic": traffic,
                     "kernel": "sv_tree_attend (plan + split-KV attention + merge), chunked launches",
                     "peak_source": f"{peak_src} hbm_gbs",
                     "bytes_per_launch": sum(att_b) / n_chunks,
                     "us_per_launch": 1e6 * att_time / n_chunks},
        "calls": {
            "attend_chunked": {"us_per_step": att_time * 1e6, "GB/s": att_gbs, "frac": att_gbs / hbm_peak},
            "accept_chunked": {"us_per_step": acc_time * 1e6, "GB/s": acc_gbs, "frac": acc_gbs / hbm_peak},
            "attend_onepass": {"us": op_att * 1e6, "GB/s": op_att_b / op_att / 1e9,
                               "frac": op_att_b / op_att / 1e9 / hbm_peak},
            "accept_onepass": {"us": op_acc * 1e6, "GB/s": op_acc_b / op_acc / 1e9,
                               "frac": op_acc_b / op_acc / 1e9 / hbm_peak},
        },
        "e2e": {"value": world * rows_attended / t_e2e, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# Revision tag of the attention kernel the stored ncu traffic belongs to.
KERNEL_REV = "attend-v2"

if __name__ == "__main__":
    main()
