"""CPU oracle for the speculative-decoding verification step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it; the product package never imports it.
The arithmetic lives in ``sv_oracle.cpp`` (plain C++, fp64); this module only
builds that file with g++ and marshals numpy arrays through ctypes.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle_sv.so")
_lib = None

# Error bits returned by the oracle calls.
ORC_BAD_BLOCK = 1
ORC_BAD_PARENT = 2
ORC_POOL_OVERFLOW = 4
ORC_BAD_WINDOW = 8
ORC_BAD_TOKEN = 32
ORC_UNSUPPORTED = 64
ORC_BAD_LENGTH = 128
ORC_BAD_ARG = 256


def build(force: bool = False) -> str:
    """Compile sv_oracle.cpp with g++ -O2 (no fast-math) into liboracle_sv.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        F = ctypes.c_float
        U64 = ctypes.c_uint64
        lib.orc_philox4x32_10.argtypes = [P, P, P]
        lib.orc_philox4x32_10.restype = None
        lib.orc_accept_uniform.argtypes = [U64, I, I]
        lib.orc_accept_uniform.restype = ctypes.c_double
        lib.orc_race_uniform.argtypes = [U64, I, I, I]
        lib.orc_race_uniform.restype = ctypes.c_double
        lib.orc_pick_uniform.argtypes = [U64, I, I, I]
        lib.orc_pick_uniform.restype = ctypes.c_double
        lib.orc_tree_attend.argtypes = [I, P, P, P, P, P, P, P, I, I, I, I, P, I, P, P, I, F, P, P, I]
        lib.orc_tree_attend.restype = I
        lib.orc_accept.argtypes = [I, P, P, P, P, P, P, P, P, I, F, U64, P, P, I, P, P, P, P, I]
        lib.orc_accept.restype = I
        lib.orc_commit_kv.argtypes = [I, P, P, P, I, I, I, I, P, I, P, P, P, I, P, P, I]
        lib.orc_commit_kv.restype = I
        lib.orc_select_budget.argtypes = [I, I, P, P, P, I, P, P, P]
        lib.orc_select_budget.restype = I
        lib.orc_verify_chunked.argtypes = [I, P, P, P, P, I, I, P, P, I, I, I, I, P, I, P, P, I, F,
                                           P, P, P, P, I, F, U64, P, P, P, P, P, P, I]
        lib.orc_verify_chunked.restype = I
        D = ctypes.c_double
        lib.orc_adapt_gamma.argtypes = [I, P, P, P, P, D, D, I, I]
        lib.orc_adapt_gamma.restype = I
        lib.orc_select_chunk.argtypes = [I, P, P, P, D, D, U64, P, P, P]
        lib.orc_select_chunk.restype = I
        _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ----------------------------------------------------------------- Philox --

def philox4x32_10(ctr, key) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib.orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def accept_uniform(seed: int, i: int, j: int) -> float:
    return _load().orc_accept_uniform(seed, i, j)


def race_uniform(seed: int, i: int, pos: int, g: int) -> float:
    """The race uniform of group g (entries 4g .. 4g+3)."""
    return _load().orc_race_uniform(seed, i, pos, g)


def pick_uniform(seed: int, i: int, pos: int, g: int) -> float:
    """The uniform that picks the entry inside the winning group g."""
    return _load().orc_pick_uniform(seed, i, pos, g)


# --------------------------------------------------------------- attention --

def tree_attend(batch, kv, q, n_q_heads, softmax_scale, out_bf16=None, out_f64=None,
                row_begin=None, row_end=None, n_threads=None):
    """Attention of every window row (see sv_oracle.cpp: orc_tree_attend).

    ``batch``: dict with cu_rows, parent (and optional verify_len);
    ``kv``: dict with k_cache, v_cache (uint16 bf16 bits, [nb][n_kv][bs][d]),
    block_tables [R][max_blocks], cache_lens [R].  Returns (err, out_bf16, out_f64).
    """
    lib = _load()
    cu = _i32(batch["cu_rows"])
    par = _i32(batch["parent"])
    vl = _i32(batch.get("verify_len"))
    R = cu.shape[0] - 1
    total_rows = int(cu[-1])
    kc, vc = kv["k_cache"], kv["v_cache"]
    nb, n_kv, bs, d = kc.shape
    bt = _i32(kv["block_tables"])
    cl = _i32(kv["cache_lens"])
    qa = np.ascontiguousarray(q, dtype=np.uint16)
    if out_bf16 is None:
        out_bf16 = np.zeros((total_rows, n_q_heads, d), dtype=np.uint16)
    if out_f64 is None:
        out_f64 = np.full((total_rows, n_q_heads, d), np.nan, dtype=np.float64)
    err = lib.orc_tree_attend(R, _ptr(cu), _ptr(par), _ptr(_i32(row_begin)), _ptr(_i32(row_end)),
                              _ptr(vl), _ptr(kc), _ptr(vc), nb, bs, n_kv, d, _ptr(bt),
                              bt.shape[1], _ptr(cl), _ptr(qa), n_q_heads, softmax_scale,
                              _ptr(out_f64), _ptr(out_bf16), n_threads or default_threads())
    return err, out_bf16, out_f64


# ------------------------------------------------------------------ accept --

@dataclass
class AcceptState:
    accepted_len: np.ndarray
    accepted_nodes: np.ndarray
    next_token: np.ndarray
    ambiguous: np.ndarray
    done: np.ndarray
    row_stats: np.ndarray

    @staticmethod
    def empty(n_req, max_rows, total_rows):
        return AcceptState(
            accepted_len=np.full(n_req, -7, dtype=np.int32),
            accepted_nodes=np.full((n_req, max_rows), -7, dtype=np.int32),
            next_token=np.full(n_req, -7, dtype=np.int32),
            ambiguous=np.zeros(n_req, dtype=np.uint8),
            done=np.zeros(n_req, dtype=np.int32),
            row_stats=np.full((total_rows, 4), np.nan, dtype=np.float64),
        )


def accept(batch, target_logits, draft_logits, temperature, seed, state=None,
           row_begin=None, row_end=None, n_threads=None):
    """Accept/reject (see sv_oracle.cpp: orc_accept).  Returns (err, state)."""
    lib = _load()
    cu = _i32(batch["cu_rows"])
    par = _i32(batch["parent"])
    tok = _i32(batch["tokens"])
    vl = _i32(batch.get("verify_len"))
    R = cu.shape[0] - 1
    max_rows = int(batch["max_rows"])
    tl = np.ascontiguousarray(target_logits, dtype=np.float32)
    V = tl.shape[-1]
    dl = None if draft_logits is None else np.ascontiguousarray(draft_logits, dtype=np.float32)
    if state is None:
        state = AcceptState.empty(R, max_rows, int(cu[-1]))
    err = lib.orc_accept(R, _ptr(cu), _ptr(par), _ptr(tok), _ptr(_i32(row_begin)),
                         _ptr(_i32(row_end)), _ptr(vl), _ptr(tl), _ptr(dl), V,
                         float(temperature), int(seed), _ptr(state.accepted_len),
                         _ptr(state.accepted_nodes), max_rows, _ptr(state.next_token),
                         _ptr(state.ambiguous), _ptr(state.done), _ptr(state.row_stats),
                         n_threads or default_threads())
    return err, state


# ------------------------------------------------------------------ commit --

def commit_kv(batch, kv, accepted_len, accepted_nodes, free_list, free_count):
    """Commit in place on the numpy arrays of ``kv`` / ``free_list``.

    ``free_count`` is a 1-element int32 array.  Returns err."""
    lib = _load()
    cu = _i32(batch["cu_rows"])
    R = cu.shape[0] - 1
    kc, vc = kv["k_cache"], kv["v_cache"]
    nb, n_kv, bs, d = kc.shape
    bt = kv["block_tables"]
    cl = kv["cache_lens"]
    assert bt.dtype == np.int32 and cl.dtype == np.int32 and free_list.dtype == np.int32
    al = _i32(accepted_len)
    an = _i32(accepted_nodes)
    return lib.orc_commit_kv(R, _ptr(cu), _ptr(kc), _ptr(vc), nb, bs, n_kv, d, _ptr(bt),
                             bt.shape[1], _ptr(cl), _ptr(al), _ptr(an), an.shape[1],
                             _ptr(free_list), _ptr(free_count), free_list.shape[0])


# ------------------------------------------------------------------ budget --

def select_budget(cond_survival, gamma, sps):
    """Budget selection (see sv_oracle.cpp: orc_select_budget).

    Returns (err, verify_len, best_B, best_theta)."""
    lib = _load()
    c = np.ascontiguousarray(cond_survival, dtype=np.float32)
    R, gmax = c.shape
    g = _i32(gamma)
    s = np.ascontiguousarray(sps, dtype=np.float32)
    vl = np.zeros(R, dtype=np.int32)
    bb = np.zeros(1, dtype=np.int32)
    bt = np.zeros(1, dtype=np.float64)
    err = lib.orc_select_budget(R, gmax, _ptr(c), _ptr(g), _ptr(s), s.shape[0] - 1, _ptr(vl),
                                _ptr(bb), _ptr(bt))
    return err, vl, int(bb[0]), float(bt[0])


def adapt_gamma(accepted_len, verified, state, decay, overhead, gamma_min, gamma_max):
    """Per-request draft length from the acceptance history (see
    orc_adapt_gamma).  `state` ([R][2] float64) is updated in place.

    Returns (err, gamma_next)."""
    lib = _load()
    a = _i32(accepted_len)
    v = _i32(verified)
    assert state.dtype == np.float64 and state.flags["C_CONTIGUOUS"]
    g = np.full(len(a), -1, dtype=np.int32)
    err = lib.orc_adapt_gamma(len(a), _ptr(a), _ptr(v), _ptr(state), _ptr(g), float(decay),
                              float(overhead), int(gamma_min), int(gamma_max))
    return err, g


def select_chunk(rows, ctx, state, kv_bytes, row_bytes, chunk_bytes):
    """Chunk size of least expected cost (see orc_select_chunk).

    Returns (err, chunk, cost, costs[128])."""
    lib = _load()
    r = _i32(rows)
    c = _i32(ctx)
    st = np.ascontiguousarray(state, dtype=np.float64)
    ch = np.zeros(1, dtype=np.int32)
    co = np.zeros(1, dtype=np.uint64)
    costs = np.zeros(128, dtype=np.uint64)
    err = lib.orc_select_chunk(len(r), _ptr(r), _ptr(c), _ptr(st), float(kv_bytes),
                               float(row_bytes), int(chunk_bytes), _ptr(ch), _ptr(co),
                               _ptr(costs))
    return err, int(ch[0]), int(co[0]), costs


# ----------------------------------------------------------------- chunked --

def verify_chunked(batch, kv, q, n_q_heads, softmax_scale, target_logits, draft_logits,
                   temperature, seed, chunk, n_threads=None):
    """Chunked verification with early pruning (see orc_verify_chunked).

    Returns (err, state, out_bf16, out_f64, rows_attended)."""
    lib = _load()
    cu = _i32(batch["cu_rows"])
    par = _i32(batch["parent"])
    tok = _i32(batch["tokens"])
    vl = _i32(batch.get("verify_len"))
    R = cu.shape[0] - 1
    total_rows = int(cu[-1])
    max_rows = int(batch["max_rows"])
    kc, vc = kv["k_cache"], kv["v_cache"]
    nb, n_kv, bs, d = kc.shape
    bt = _i32(kv["block_tables"])
    cl = _i32(kv["cache_lens"])
    qa = np.ascontiguousarray(q, dtype=np.uint16)
    tl = np.ascontiguousarray(target_logits, dtype=np.float32)
    V = tl.shape[-1]
    dl = None if draft_logits is None else np.ascontiguousarray(draft_logits, dtype=np.float32)
    state = AcceptState.empty(R, max_rows, total_rows)
    out_bf16 = np.zeros((total_rows, n_q_heads, d), dtype=np.uint16)
    out_f64 = np.full((total_rows, n_q_heads, d), np.nan, dtype=np.float64)
    attended = np.zeros(1, dtype=np.int32)
    err = lib.orc_verify_chunked(R, _ptr(cu), _ptr(par), _ptr(tok), _ptr(vl), max_rows, chunk,
                                 _ptr(kc), _ptr(vc), nb, bs, n_kv, d, _ptr(bt), bt.shape[1],
                                 _ptr(cl), _ptr(qa), n_q_heads, softmax_scale, _ptr(out_f64),
                                 _ptr(out_bf16), _ptr(tl), _ptr(dl), V, float(temperature),
                                 int(seed), _ptr(state.accepted_len), _ptr(state.accepted_nodes),
                                 _ptr(state.next_token), _ptr(state.ambiguous), _ptr(state.done),
                                 _ptr(attended), n_threads or default_threads())
    return err, state, out_bf16, out_f64, int(attended[0])
