"""Benchmark of one verification step per layer on GB300 (one JSON line).

Default workload (--workload batch64): 64 requests, Llama-3-8B attention
shape (32 q / 8 KV heads, d 128), per-request draft counts U{1..8},
contexts log-normal (ln 4096, 1) clipped to [512, 32768], paged bf16 KV
(16-token blocks, shuffled tables), vocab 128256 fp32 logits, sampling at
T = 0.7, chunked verification in chunks of 2 with early pruning, each
request's KV committed in the chunk that stops it.  Other workloads: tiny,
chain8b, tree70b (one pass; tree70b_t1 the same tree sampled at T = 1),
batch256 (budget-selected).

One step = restore the block tables / lengths / free list the previous
step's commit changed, then the workload's calls:
  chunked  sv_verify_chunked_commit (per chunk: attention plan with the
           chunk's windows and accept list, split-KV attention, row
           statistics, decisions with the KV commit of every request they
           stop; one resampling race per step)
  onepass  sv_tree_attend, sv_accept_commit (accept and KV commit fused)
  budget   sv_select_budget, sv_tree_attend and sv_accept_commit on the
           selected prefixes
Inputs larger than L2 are timed back to back; smaller ones step by step with
an L2 flush (a 512 MB write) between steps, outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload batch64|tiny|chain8b|tree70b|tree70b_t1|batch256]

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
L2_BYTES = 129 * 2 ** 20

WORKLOAD_TEXT = {
    "batch64": ("batch64: 64 requests, Llama-3-8B attention shape (32 q / 8 kv heads, d 128), "
                "drafts U{1..8} per request, context lognormal(ln 4096, 1) clipped to [512, 32768], "
                "paged bf16 KV in 16-token blocks with shuffled tables, vocab 128256 fp32 logits, "
                "T=0.7 sampling, chunked verification (chunk 2) with early pruning, KV commit"),
    "tiny": ("tiny: 1 request, 4 drafts, 8 q / 2 kv heads, d 64, context 256, vocab 1024, "
             "target N(0,2^2), draft = target + N(0,0.5^2), T=1 sampling, one pass, KV commit"),
    "chain8b": ("chain8b: 1 request, 5 drafts, Llama-3-8B attention shape (32 q / 8 kv, d 128), "
                "context 4096, vocab 128256 fp32 logits ~N(0,3^2), draft sigma 1, T=1 sampling, "
                "one pass, KV commit"),
    "tree70b": ("tree70b: 1 request, 64-node draft tree (depth 6, branching 4,3,2,2,1,1 "
                "truncated), Llama-3-70B attention shape (64 q / 8 kv, d 128), context 8192, vocab "
                "128256, greedy longest valid path, KV commit of the path"),
    "batch256": ("batch256: 256 requests, 40 q / 8 kv heads, d 128, context U{1024..8192}, 4 drafts, "
                 "vocab 151936, survival c ~ Beta(4,2), budget by argmax tau*SPS(B) with "
                 "SPS(B)=1000/(1+B/512), then attention + T=1 accept + commit on the selected prefixes"),
    "tree70b_t1": ("tree70b_t1: the tree70b step with T=1 tree sampling (siblings drawn from q, "
                   "children tried in index order against the parent's residual), KV commit of "
                   "the accepted path"),
}

# Workloads that are a configuration with one setting changed.
VARIANTS = {"tree70b_t1": ("tree70b", {"temperature": 1.0})}


def make_named_workload(wl, name, **kw):
    base, over = VARIANTS.get(name, (name, {}))
    return wl.make_workload(wl.config(base), **over, **kw)


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


NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s the target is stated against


def _peaks():
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    return json.load(open(peaks_path)) if os.path.exists(peaks_path) else None


def hbm_peak_gbs():
    """The HBM denominator: the machine's measured copy bandwidth, else the
    fallback figure."""
    p = _peaks()
    if p and "hbm_gbs" in p:
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak_tflops():
    """The dense bf16 tensor denominator for a kernel timed on its own (burst):
    the pool's measured cuBLAS figure, else the fallback figure."""
    p = _peaks()
    if p and "bf16_tflops" in p:
        return float(p["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# ---------------------------------------------------------- byte accounting --

def launch_windows(w, mode, accepted_len, verify_len=None, chunk=2):
    """The (request, begin, end, lim) windows of every attention / accept
    launch of one step, from the step's own results."""
    rows = [int(r) for r in np.diff(w.cu_rows)]
    R = w.n_req
    if mode == "chunked":
        sched = []
        for c in range(math.ceil(w.max_rows / chunk)):
            act = []
            for i in range(R):
                b, e = c * chunk, min(c * chunk + chunk, rows[i])
                if b < e and c <= int(accepted_len[i]) // chunk:
                    act.append((i, b, e, rows[i]))
            sched.append(act)
        return sched
    if mode == "budget":
        return [[(i, 0, int(verify_len[i]) + 1, int(verify_len[i]) + 1) for i in range(R)]]
    return [[(i, 0, rows[i], rows[i]) for i in range(R)]]


def attend_flops(w, windows):
    """Dense work of the attention: for every attended row and query head,
    4 d flops (QK^T and PV) per visible key (context + ancestors-or-self)."""
    cfg = w.cfg
    per_key = 4 * cfg.head_dim * cfg.n_q_heads
    tot = 0
    for i, b, e, _ in windows:
        base = int(w.cu_rows[i])
        for r in range(b, e):
            depth, m = 0, r
            while m >= 0:
                depth += 1
                m = int(w.parent[base + m]) if m > 0 else -1
            tot += per_key * (int(w.cache_lens[i]) + depth)
    return tot


def attend_bytes(w, windows):
    """KV of context + staged slots up to the window end, Q in, out."""
    cfg = w.cfg
    kvb = cfg.n_kv_heads * cfg.head_dim * 2 * 2
    qo = cfg.n_q_heads * cfg.head_dim * 2 * 2
    return sum((int(w.cache_lens[i]) + e) * kvb + (e - b) * qo for i, b, e, _ in windows)


def accept_bytes(w, windows, accepted_len, T):
    """Target rows of the window, draft rows that propose a tested draft
    (T > 0), and the one or two rows the residual / bonus draw scans."""
    V = int(w.target_logits.shape[1])
    tot = 0
    for i, b, e, lim in windows:
        tot += (e - b) * V * 4
        if T > 0:
            tot += max(0, min(e, lim - 1) - b) * V * 4
            a = int(accepted_len[i])
            if b <= a < e:
                tot += V * 4 if a == lim - 1 else 2 * V * 4
    return tot


# ------------------------------------------------------------- CPU baseline --

def oracle_sample(w, idx):
    """Requests `idx` of w as a standalone workload (same cache arrays)."""
    from speculative_decoding_verification_padding_gb300.workloads import Workload
    cu = w.cu_rows
    rows = [slice(cu[i], cu[i + 1]) for i in idx]
    new_cu = np.zeros(len(idx) + 1, dtype=np.int32)
    new_cu[1:] = np.cumsum([cu[i + 1] - cu[i] for i in idx])
    cat = lambda a: np.concatenate([a[s] for s in rows])
    return Workload(cfg=w.cfg, cu_rows=new_cu, parent=cat(w.parent), tokens=cat(w.tokens),
                    max_rows=w.max_rows, k_cache=w.k_cache, v_cache=w.v_cache,
                    block_tables=np.ascontiguousarray(w.block_tables[idx]),
                    cache_lens=np.ascontiguousarray(w.cache_lens[idx]), free_list=w.free_list,
                    free_count=w.free_count, q=cat(w.q), target_logits=cat(w.target_logits),
                    draft_logits=cat(w.draft_logits), seed=w.seed)


def time_oracle(w, mode, idx, threads):
    """One step of the oracle on requests `idx`: returns (seconds, rows attended)."""
    import oracle
    t0 = time.perf_counter()
    vl = None
    if mode == "budget":
        _, vl_all, _, _ = oracle.select_budget(w.cond_survival, w.gamma, w.sps)
        vl = np.ascontiguousarray(vl_all[idx])
    s = oracle_sample(w, idx)
    T = s.cfg.temperature
    draft = s.draft_logits if T > 0 else None
    if mode == "chunked":
        _, _, _, _, attended = oracle.verify_chunked(
            s.batch(), s.kv(), s.q, s.cfg.n_q_heads, s.softmax_scale, s.target_logits, draft, T,
            s.seed, chunk=s.cfg.chunk or 2, n_threads=threads)
    else:
        b = s.batch(verify_len=vl)
        oracle.tree_attend(b, s.kv(), s.q, s.cfg.n_q_heads, s.softmax_scale, n_threads=threads)
        oracle.accept(b, s.target_logits, draft, T, s.seed, n_threads=threads)
        attended = int(s.total_rows if vl is None else (vl + 1).sum())
    return time.perf_counter() - t0, attended


def cpu_baseline(w, mode, budget_s=10.0):
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    dt1, _ = time_oracle(w, mode, [0], threads)
    n = int(max(1, min(w.n_req, budget_s / max(dt1, 1e-3))))
    dt, att = time_oracle(w, mode, list(range(n)), threads)
    # the same oracle on one thread, on a smaller sample of the same step
    d1, _ = time_oracle(w, mode, [0], 1)
    n1 = int(max(1, min(n, 0.5 * budget_s / max(d1, 1e-3))))
    dts, atts = time_oracle(w, mode, list(range(n1)), 1)
    return {"value": att / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {n} of {w.n_req} requests of the same step ({mode}: attention + "
                      f"accept), {att} rows attended in {dt:.2f} s, fp64 C++ oracle with "
                      f"{threads} threads",
            "single_thread": {"value": atts / dts, "unit": UNIT,
                              "sample": f"first {n1} requests, {atts} rows in {dts:.2f} s"},
            "cpu_model": cpu_model()}


def cpu_model():
    """The host CPU as lscpu names it (model name and count of online CPUs)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        info = dict(l.split(":", 1) for l in out.splitlines() if ":" in l)
        name = (info.get("Model name") or info.get("Vendor ID") or "").strip()
        cpus = (info.get("CPU(s)") or "").strip()
        return f"{name}, {cpus} CPUs" if name else None
    except Exception:
        return None


# ------------------------------------------------------------------- main --

def mode_of(cfg):
    return "budget" if cfg.budget else "chunked" if cfg.chunk else "onepass"


def run_reference(args, rank):
    """Reference arm: the CPU oracle, timed on this host's cores."""
    if rank != 0:
        return
    from speculative_decoding_verification_padding_gb300 import workloads as wl
    import oracle
    oracle.build()
    w = make_named_workload(wl, args.workload)
    mode = mode_of(w.cfg)
    threads = os.cpu_count() or 1
    dt1, _ = time_oracle(w, mode, [0], threads)
    per_step_budget = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    n = int(max(1, min(w.n_req, per_step_budget / max(dt1, 1e-3))))
    span = w.n_req - n + 1
    for k in range(args.warmup):
        time_oracle(w, mode, [(k * n) % span + j for j in range(n)], threads)
    tot_t, tot_rows = 0.0, 0
    for k in range(args.steps):
        dt, att = time_oracle(w, mode, [(k * n) % span + j for j in range(n)], threads)
        tot_t += dt
        tot_rows += att
    value = tot_rows / tot_t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload], "global_batch": w.n_req,
                       "parallelism": "host threads"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{n} of {w.n_req} requests per step ({mode}: attention "
                                       f"+ accept), fp64 C++ oracle, {threads} threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="batch64", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="only run this many steps (for a profiler), no timing line")
    ap.add_argument("--ctx-scale", type=float, default=1.0,
                    help="with --profile-steps: shrink every context (smaller profiler captures)")
    ap.add_argument("--sps", default="synthetic", choices=["synthetic", "measured"],
                    help="budget workload: the synthetic SPS(B) table or the one measured "
                         "from this library's kernels (speculative_decoding_verification_padding_gb300/sps.py)")
    ap.add_argument("--profile-call", default="step", choices=["step", "attend", "accept"],
                    help="with --profile-steps: run the whole step, or only the one-pass "
                         "sv_tree_attend / sv_accept call on the whole batch")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    from speculative_decoding_verification_padding_gb300 import api
    from speculative_decoding_verification_padding_gb300.replicas import Replicas
    from speculative_decoding_verification_padding_gb300 import workloads as wl
    from speculative_decoding_verification_padding_gb300.step import DeviceStep, HostPipeline

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    reps = Replicas.from_env("nccl", device=dev)

    w = make_named_workload(wl, args.workload,
                         ctx_scale=args.ctx_scale if args.profile_steps else 1.0, sps=args.sps)
    s = DeviceStep(w, device=dev)
    mode, chunk, T = s.mode, s.chunk, s.T
    stream = torch.cuda.current_stream()

    if args.profile_steps:
        fn = {"step": s.run, "attend": s.attend, "accept": s.accept}[args.profile_call]
        for _ in range(args.profile_steps):
            fn()
        torch.cuda.synchronize()
        return

    for _ in range(args.warmup):
        s.run()
    res = s.results()
    if res["dev_status"] != 0:
        raise SystemExit(f"device status {res['dev_status']} during warm-up")
    al = res["accepted_len"]
    vl = s.verify_len.cpu().numpy() if mode == "budget" else None
    sched = launch_windows(w, mode, al, vl, chunk)
    rows_attended = sum(e - b for ch in sched for _, b, e, _ in ch)
    accepted_tokens = int((al + 1).sum())
    step_bytes = sum(attend_bytes(w, ch) + accept_bytes(w, ch, al, T) for ch in sched)
    flush_l2 = step_bytes < 2 * L2_BYTES
    flush_buf = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev) if flush_l2 else None

    barrier, max_over_ranks = reps.barrier, reps.max_over_ranks

    def timed(fn, n):
        """Mean seconds per call of fn over n calls (flushing L2 between calls
        for small inputs, outside the events)."""
        if not flush_l2:
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(n):
                fn()
            a1.record(stream)
            torch.cuda.synchronize()
            return a0.elapsed_time(a1) / 1e3 / n
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a0, a1 in evs:
            flush_buf.fill_(1)
            a0.record(stream)
            fn()
            a1.record(stream)
        torch.cuda.synchronize()
        return sum(a0.elapsed_time(a1) for a0, a1 in evs) / 1e3 / n

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)

    # ---- headline: K whole steps, device-resident inputs ----
    barrier()
    torch.cuda.synchronize()
    t_step = max_over_ranks(timed(s.run, args.steps))
    barrier()

    # ---- per-call timing inside the same steps ----
    n_rep = max(5, args.steps // 4)
    att_b = [attend_bytes(w, ch) for ch in sched]
    acc_b = [accept_bytes(w, ch, al, T) for ch in sched]
    ev = lambda: torch.cuda.Event(enable_timing=True)
    t_att = t_acc = t_sel = 0.0
    marks = []
    torch.cuda.synchronize()
    if mode == "chunked":
        rb = torch.zeros(w.n_req, dtype=torch.int32, device=dev)
        re = torch.zeros(w.n_req, dtype=torch.int32, device=dev)
        bw = api.Batch(s.batch.cu_rows, s.batch.parent, s.batch.tokens, w.max_rows,
                       row_begin=rb, row_end=re)
        for _ in range(n_rep):
            if flush_l2:
                flush_buf.fill_(1)
            s.restore_cache_state()
            for c in range(len(sched)):
                api.sv_chunk_windows(s.batch, c, chunk, s.done, rb, re)
                m = (ev(), ev(), ev())
                m[0].record(stream)
                s.attend(bw)
                m[1].record(stream)
                s.accept(bw)
                m[2].record(stream)
                marks.append(m)
            s.commit()
        torch.cuda.synchronize()
        t_att = sum(m[0].elapsed_time(m[1]) for m in marks) / 1e3 / n_rep
        t_acc = sum(m[1].elapsed_time(m[2]) for m in marks) / 1e3 / n_rep
    else:
        b = s.batch_sel if mode == "budget" else s.batch
        for _ in range(n_rep):
            if flush_l2:
                flush_buf.fill_(1)
            s.restore_cache_state()
            m = (ev(), ev(), ev(), ev())
            m[0].record(stream)
            if mode == "budget":
                s.select()
            m[1].record(stream)
            s.attend(b)
            m[2].record(stream)
            s.accept(b)
            m[3].record(stream)
            s.commit(b)
            marks.append(m)
        torch.cuda.synchronize()
        t_sel = sum(m[0].elapsed_time(m[1]) for m in marks) / 1e3 / n_rep
        t_att = sum(m[1].elapsed_time(m[2]) for m in marks) / 1e3 / n_rep
        t_acc = sum(m[2].elapsed_time(m[3]) for m in marks) / 1e3 / n_rep
    att_gbs = sum(att_b) / t_att / 1e9
    acc_gbs = sum(acc_b) / t_acc / 1e9
    calls = {"attend": {"us_per_step": t_att * 1e6, "GB/s": att_gbs},
             "accept": {"us_per_step": t_acc * 1e6, "GB/s": acc_gbs}}
    if mode == "budget":
        calls["select_budget"] = {"us_per_step": t_sel * 1e6}
    if mode == "chunked":
        # The per-call accept above runs a public sv_accept per chunk, each with
        # its own resampling race; inside the step the chunks share one race.
        # Derived: the step's time less its attention calls, over the same bytes.
        t_in = max(t_step - t_att, 1e-9)
        calls["accept_in_step"] = {"us_per_step": t_in * 1e6, "GB/s": sum(acc_b) / t_in / 1e9,
                                   "derived": "step time - attention calls"}

    # ---- one-pass attention and accept on the whole batch (chunked workload) ----
    if mode == "chunked":
        full = launch_windows(w, "onepass", al)[0]
        op_att = timed(lambda: s.attend(), n_rep)
        op_acc = timed(lambda: s.accept(), n_rep)
        calls["attend_onepass"] = {"us": op_att * 1e6, "GB/s": attend_bytes(w, full) / op_att / 1e9}
        calls["accept_onepass"] = {"us": op_acc * 1e6,
                                   "GB/s": accept_bytes(w, full, al, T) / op_acc / 1e9}
        s.run()  # back to the chunked step's state

    # ---- the chunk-size rule on this step's own acceptance (outside the timing) ----
    chunk_policy = None
    if mode == "chunked":
        rows_np = np.diff(w.cu_rows).astype(np.int32)
        a_np = np.asarray(al, dtype=np.int64)
        state = np.stack([a_np, a_np + (a_np < rows_np - 1)], axis=1).astype(np.float64)
        fixed_us = 25.0  # plan + statistics + decision latency of one chunk, launch list
        chunk_b = int(fixed_us * 1e-6 * hbm_peak_gbs()[0] * 1e9)
        kvb = 2.0 * 2 * w.cfg.n_kv_heads * w.cfg.head_dim
        rowb = 4.0 * w.target_logits.shape[1] * (2 if T > 0 else 1)
        g_ch = torch.zeros(1, dtype=torch.int32, device=dev)
        g_cost = torch.zeros(1, dtype=torch.int64, device=dev)
        g_costs = torch.zeros(128, dtype=torch.int64, device=dev)
        api.sv_select_chunk(torch.from_numpy(rows_np).to(dev),
                            torch.from_numpy(w.cache_lens.astype(np.int32)).to(dev),
                            torch.from_numpy(state).to(dev), kvb, rowb, chunk_b, g_ch, g_cost,
                            g_costs)
        torch.cuda.synchronize()
        cs = g_costs.cpu().numpy().view(np.uint64)
        sel = int(g_ch.item())
        chunk_policy = {
            "selected_chunk": sel, "per_chunk_fixed_MB": chunk_b / 1e6,
            "modelled_MB": {str(chunk): float(cs[chunk - 1]) / 1e6, str(sel): float(cs[sel - 1]) / 1e6},
            "measured_us": {f"chunk {chunk} step": t_step * 1e6,
                            "one pass (attend + accept)": calls["attend_onepass"]["us"]
                            + calls["accept_onepass"]["us"]}}

    # ---- end to end through host buffers ----
    # Inputs from pinned host memory and results back to it, every step, timed
    # two ways: in series (copy in, step, copy out; small workloads flush L2
    # between steps outside the events) and through the double-buffered
    # HostPipeline (step i + 1's upload overlaps step i's kernels; one event
    # pair around the run, so a small workload's L2 flushes sit inside it).
    # Both move every byte; the line reports the faster and names it.
    host_ins = [t.cpu().pin_memory() for t in s.inputs()]
    outs = [(torch.empty_like(t, device="cpu").pin_memory(), t) for t in s.outputs()]
    h2d = sum(h.numel() * h.element_size() for h in host_ins)
    d2h = sum(h.numel() * h.element_size() for h, _ in outs)

    def e2e_step():
        for d, h in zip(s.inputs(), host_ins):
            d.copy_(h, non_blocking=True)
        s.run()
        for h, d in outs:
            h.copy_(d, non_blocking=True)

    def e2e_pipelined(n):
        pipe = HostPipeline(s)
        for _ in range(3):
            pipe.submit(host_ins)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        pipe.begin()
        for _ in range(n):
            if flush_l2:
                flush_buf.fill_(1)
            pipe.submit(host_ins)
        a1.record(stream)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) / 1e3 / n

    barrier()
    torch.cuda.synchronize()
    n_e2e = max(5, args.steps // 4)
    t_e2e_serial = max_over_ranks(timed(e2e_step, n_e2e))
    t_e2e_pipe = max_over_ranks(e2e_pipelined(n_e2e))
    t_e2e, e2e_mode = e2e_choice(t_e2e_serial, t_e2e_pipe, flush_l2)
    barrier()

    # ---- step-time distribution: an event pair per step, L2 flushed before each ----
    flush_any = flush_buf if flush_buf is not None else torch.empty(512 * 2 ** 20, dtype=torch.uint8,
                                                                    device=dev)

    def per_step_ms(fn, n):
        evs = [(ev(), ev()) for _ in range(n)]
        for a0, a1 in evs:
            flush_any.fill_(1)
            a0.record(stream)
            fn()
            a1.record(stream)
        torch.cuda.synchronize()
        return sorted(a0.elapsed_time(a1) for a0, a1 in evs)

    n_dist = max(10, args.steps // 2)
    st_ms = per_step_ms(s.run, n_dist)
    step_dist = {"median_ms": st_ms[len(st_ms) // 2], "p90_ms": st_ms[int(0.9 * (len(st_ms) - 1))],
                 "steps": n_dist, "l2": "flushed (512 MB write outside the events) before each step"}

    # ---- one-request workloads: the same step replayed as one CUDA graph ----
    graph = None
    if w.n_req == 1:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                s.run()
            torch.cuda.synchronize()
            gr_ms = per_step_ms(g.replay, n_dist)
            res_g = s.results()
            assert np.array_equal(res_g["accepted_len"], al), "graph replay changed the results"
            graph = {"median_ms": gr_ms[len(gr_ms) // 2], "p90_ms": gr_ms[int(0.9 * (len(gr_ms) - 1))],
                     "steps": n_dist, "l2": step_dist["l2"]}
        except Exception as e:  # report, do not hide the headline
            graph = {"error": f"{type(e).__name__}: {e}"[:200]}
    clk = clocks.stop()
    res2 = s.results()
    assert np.array_equal(res2["accepted_len"], al), "steps are not reproducible"

    rows_all = reps.sum_over_ranks(rows_attended)  # every rank joins before the leader reports
    if not reps.leader:
        reps.close()
        return

    hbm_peak, peak_src = hbm_peak_gbs()
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "attend_traffic.json")
    if os.path.exists(tr_path):
        tr = json.load(open(tr_path))
        if tr.get("workload") == args.workload and tr.get("kernel_rev") == KERNEL_REV:
            traffic = tr.get("bytes_per_launch")
    for c in calls.values():
        if "GB/s" in c:
            c["frac"] = c["GB/s"] / hbm_peak
            c["frac_of_8TBs"] = c["GB/s"] / NOMINAL_HBM_GBS

    n_launch = len(sched)
    # The attention's roofline: the tensor pipe where the GQA group x draft
    # rows make a dense tile that the KV bytes cannot keep busy (the tree
    # workload, about 175 flops per byte), HBM elsewhere.
    att_flops = sum(attend_flops(w, ch) for ch in sched)
    kernel_name = "sv_tree_attend (planner, split-KV attention kernels, split merge)"
    if w.cfg.gamma and w.cfg.gamma[0] == "tree":
        tf_peak, tf_src = bf16_peak_tflops()
        achieved = att_flops / t_att / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": tf_peak, "unit": "TFLOP/s",
                    "frac": achieved / tf_peak, "traffic": traffic, "kernel": kernel_name,
                    "peak_source": f"{tf_src} bf16_tflops (burst: the kernel is timed alone)",
                    "flops_per_launch": att_flops / n_launch,
                    "hbm": {"GB/s": att_gbs, "frac": att_gbs / hbm_peak}}
    else:
        roofline = {"bound": "hbm", "achieved": att_gbs, "peak": hbm_peak, "unit": "GB/s",
                    "frac": att_gbs / hbm_peak, "frac_of_8TBs": att_gbs / NOMINAL_HBM_GBS,
                    "traffic": traffic, "kernel": kernel_name,
                    "peak_source": f"{peak_src} hbm_gbs"}
    roofline.update({"launches_per_step": n_launch, "bytes_per_launch": sum(att_b) / n_launch,
                     "us_per_launch": 1e6 * t_att / n_launch})
    race = 1 if T > 0 else 0
    # Chunked: plan (windows + accept list) + attend [+ tcgen05 attend] + stats + decide
    # (with the commit) per chunk [+ tree walk after the first when a chunk holds a
    # tree], one race after the last.  One-pass / budget: [select] + plan + attend
    # [+ tcgen05 attend] + fused accept-commit (stats + decide [+ tree walk] [+ race]).
    tree = 1 if (T > 0 and w.max_rows > 2) else 0
    tc = 1 if (w.cfg.head_dim == 128 and
               w.cfg.n_q_heads // w.cfg.n_kv_heads * w.max_rows >= 128) else 0
    # attention: plan, [tcgen05 kernel], mma.sync kernel, [one merge launch when
    # the tcgen05 kernel ran or the batch is small (<= 4 requests)]
    att = 2 + tc + (1 if (tc or w.n_req <= 4) else 0)
    if mode == "chunked":
        launches_per_step = n_launch * (att + 2) + race + (tree if chunk > 2 else 0)
    else:
        launches_per_step = att + 2 + tree + race + (1 if mode == "budget" else 0)
    value = rows_all / t_step
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 attention (fp32 accumulate), fp32 softmax",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "mode": mode,
                   "global_batch": w.n_req * world, "rows_per_step": int(w.total_rows),
                   "rows_attended_per_step": int(rows_attended),
                   "vocab": int(w.target_logits.shape[1]), "parallelism": f"replicas x{world}",
                   "l2": ("flushed between steps (512 MB write outside the timed events)"
                          if flush_l2 else "inputs larger than L2, no flush")},
        "verify_steps_per_s": world / t_step,
        "accepted_tokens_per_s": world * accepted_tokens / t_step,
        "roofline": roofline,
        "calls": calls,
        **({"chunk_policy": chunk_policy} if chunk_policy else {}),
        "e2e": {"value": rows_all / t_e2e, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3,
                "mode": e2e_mode,
                "serial_ms_per_step": t_e2e_serial * 1e3, "pipelined_ms_per_step": t_e2e_pipe * 1e3},
        "gpu_launches": launches_per_step * args.steps,
        "step_time_flushed": step_dist,
        "clocks": clk,
    }
    if graph is not None:
        line["graph_replay"] = graph
    if mode == "chunked":
        line["config"]["chunk"] = chunk
    if mode == "budget":
        line["config"]["sps"] = args.sps
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, mode)
    print(json.dumps(line), flush=True)
    reps.close()


def e2e_choice(t_serial, t_pipe, flush_l2):
    """The end-to-end time to report and its description: the faster of the
    series timing (copy in, step, copy out) and the double-buffered one, both
    of which move every input and result byte of every step."""
    if t_pipe <= t_serial:
        return t_pipe, ("double-buffered inputs (HostPipeline: upload of step i+1 overlaps step i"
                        + ("; L2 flushes inside the timed region)" if flush_l2 else ")"))
    return t_serial, ("serial (copy in, step, copy out"
                      + ("; L2 flushed between steps)" if flush_l2 else ")"))


# Revision tag of the attention kernel the stored ncu traffic belongs to.
KERNEL_REV = "attend-tma-v5"

if __name__ == "__main__":
    main()
