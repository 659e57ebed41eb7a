"""A measured SPS(B) table for the budget selection, from this library's own
verification kernels on the GPU it runs on.

[DSpark] "하드웨어 인식 Prefix 스케줄러" chooses the verified budget B by
argmax tau(B) * SPS(B), where SPS(B) is the throughput (steps per second) the
hardware delivers when B tokens are verified in one step, profiled
beforehand.  Here one "step" is the verification work of one layer: the
attention call over the B verified rows plus the accept call over them
(``sv_tree_attend`` + ``sv_accept`` on the budget workload's batch, with
verify_len spreading the B - R draft rows over the requests).  The time of
each sampled B is taken with CUDA events, L2 flushed before every call; the
table in between is linear in the step time, and made non-increasing in B.

    python -m speculative_decoding_verification_padding_gb300.sps [--out FILE]

writes the table (JSON) that ``workloads.make_workload(..., sps="measured")``
reads.  Nothing here runs on the verification path itself.
"""

from __future__ import annotations

import argparse
import json
import os

import numpy as np

DATA_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "data")
MEASURED = os.path.join(DATA_DIR, "sps_batch256_gb300.json")


def verify_lens(B: int, gamma: np.ndarray) -> np.ndarray:
    """verify_len per request for a budget of B verified rows (B - R drafts
    spread as evenly as the per-request draft counts allow, lower requests
    first)."""
    gamma = np.asarray(gamma, dtype=np.int64)
    R = len(gamma)
    m = int(np.clip(B - R, 0, int(gamma.sum())))
    L = np.zeros(R, dtype=np.int64)
    # water filling: raise every request by one draft per round
    while m > 0:
        room = np.nonzero(L < gamma)[0]
        take = room[: m]
        L[take] += 1
        m -= len(take)
    return L.astype(np.int32)


def table_from_samples(points, seconds, b_max: int) -> np.ndarray:
    """SPS(B) for B = 0..b_max from step times measured at `points`:
    linear in time between samples, constant beyond the ends, then made
    non-increasing (a larger budget never runs more steps per second)."""
    pts = np.asarray(points, dtype=np.float64)
    t = np.asarray(seconds, dtype=np.float64)
    order = np.argsort(pts)
    t_all = np.interp(np.arange(b_max + 1, dtype=np.float64), pts[order], t[order])
    sps = 1.0 / t_all
    return np.minimum.accumulate(sps).astype(np.float32)


def load_measured(b_max: int) -> np.ndarray:
    with open(MEASURED) as f:
        d = json.load(f)
    sps = np.asarray(d["sps"], dtype=np.float32)
    if len(sps) < b_max + 1:
        raise ValueError(f"{MEASURED} covers B <= {len(sps) - 1}, need {b_max}")
    return sps[: b_max + 1]


def measure(n_points: int = 9, reps: int = 20, device: str = "cuda") -> dict:
    import torch

    from . import api
    from . import workloads as wl
    from .step import DeviceStep

    w = wl.make_workload(wl.config("batch256"))
    s = DeviceStep(w, device=device)
    R = w.n_req
    gamma = w.gamma
    b_lo, b_hi = R, R + int(gamma.sum())
    points = sorted(set(int(round(x)) for x in np.linspace(b_lo, b_hi, n_points)))
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    vl_t = s.verify_len
    b = api.Batch(s.batch.cu_rows, s.batch.parent, s.batch.tokens, w.max_rows, verify_len=vl_t)
    secs = []
    for B in points:
        vl_t.copy_(torch.from_numpy(verify_lens(B, gamma)))
        for _ in range(3):
            s.attend(b)
            s.accept(b)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for a0, a1 in evs:
            flush.fill_(1)
            a0.record(stream)
            s.attend(b)
            s.accept(b)
            a1.record(stream)
        torch.cuda.synchronize()
        ms = sorted(a0.elapsed_time(a1) for a0, a1 in evs)
        secs.append(ms[len(ms) // 2] / 1e3)
    sps = table_from_samples(points, secs, w.cfg.sps_b_max)
    return {"what": "steps/s of one layer's verification (sv_tree_attend + sv_accept, T = 1) "
                    "on the batch256 workload with B verified rows, median of "
                    f"{reps} L2-flushed calls per sampled B",
            "device": torch.cuda.get_device_name(), "points": points,
            "seconds": secs, "sps": [float(x) for x in sps]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=MEASURED)
    ap.add_argument("--points", type=int, default=9)
    args = ap.parse_args()
    d = measure(args.points)
    os.makedirs(os.path.dirname(os.path.abspath(args.out)), exist_ok=True)
    with open(args.out, "w") as f:
        json.dump(d, f, indent=1)
    print(json.dumps({k: d[k] for k in ("device", "points", "seconds")}))


if __name__ == "__main__":
    main()
