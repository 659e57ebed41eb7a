"""Python binding of libspecverify for torch tensors.

Every function has the name of the C call it marshals and runs nothing but
that call: torch provides device memory and the current stream.  Tensors
must live on the current CUDA device; results land in the tensors passed in.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _native as N


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise N.SpecVerifyError("libspecverify takes device tensors")
    if not t.is_contiguous():
        raise N.SpecVerifyError("libspecverify takes contiguous tensors")
    return t.data_ptr()


def _expect(t: Optional[torch.Tensor], dtype, name):
    if t is not None and t.dtype != dtype:
        raise N.SpecVerifyError(f"{name} must be {dtype}, got {t.dtype}")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# The current stream's handle for a device index, without building a Stream
# object (a few microseconds less per call on the launch path).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _current_stream(device_index: int) -> int:
    if _raw_stream is not None:
        return _raw_stream(device_index)
    return torch.cuda.current_stream(device_index).cuda_stream


def _call(name: str, args: tuple, stream):
    N.check(getattr(N.lib(), name)(*args, _stream(stream)), name)


class BoundCall:
    """One library call with its arguments marshalled once: the dtypes
    checked, the structs built and the device pointers taken.  Calling it
    enqueues the call on the current stream of the bound tensors' device (or
    on `stream`).  The tensors it was bound to must stay allocated, and the
    Batch / PagedKV / BlockPool objects must keep the same tensors: the
    call reads their pointers as they were when it was bound."""

    __slots__ = ("_f", "_name", "_args", "_dev")

    def __init__(self, name: str, args: tuple, device: torch.device):
        self._f = getattr(N.lib(), name)
        self._name = name
        self._args = args  # ctypes byref objects keep their structs alive
        self._dev = device.index if device.index is not None else torch.cuda.current_device()

    def __call__(self, stream=None):
        st = _current_stream(self._dev) if stream is None else _stream(stream)
        status = self._f(*self._args, st)
        if status != N.SV_OK:
            N.check(status, self._name)


@dataclass
class Batch:
    """sv_batch: packed draft chains / trees (int32 device tensors)."""
    cu_rows: torch.Tensor
    parent: torch.Tensor
    tokens: torch.Tensor
    max_rows: int
    row_begin: Optional[torch.Tensor] = None
    row_end: Optional[torch.Tensor] = None
    verify_len: Optional[torch.Tensor] = None

    @property
    def n_req(self):
        return self.cu_rows.shape[0] - 1

    @property
    def total_rows(self):
        return self.parent.shape[0]

    def c(self) -> N.SvBatch:
        for name in ("cu_rows", "parent", "tokens", "row_begin", "row_end", "verify_len"):
            _expect(getattr(self, name), torch.int32, name)
        return N.SvBatch(self.n_req, self.total_rows, self.max_rows, _ptr(self.cu_rows),
                         _ptr(self.parent), _ptr(self.tokens), _ptr(self.row_begin),
                         _ptr(self.row_end), _ptr(self.verify_len))


@dataclass
class PagedKV:
    """sv_paged_kv: bf16 [num_blocks][n_kv][16][d] caches, int32 tables."""
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor
    cache_lens: torch.Tensor

    def c(self) -> N.SvPagedKV:
        _expect(self.k_cache, torch.bfloat16, "k_cache")
        _expect(self.v_cache, torch.bfloat16, "v_cache")
        _expect(self.block_tables, torch.int32, "block_tables")
        _expect(self.cache_lens, torch.int32, "cache_lens")
        nb, hkv, bs, d = self.k_cache.shape
        return N.SvPagedKV(_ptr(self.k_cache), _ptr(self.v_cache), nb, bs, hkv, d,
                           _ptr(self.block_tables), self.block_tables.shape[1],
                           _ptr(self.cache_lens))


@dataclass
class BlockPool:
    """sv_block_pool: free list and its count (int32 device tensors)."""
    free_list: torch.Tensor
    free_count: torch.Tensor

    def c(self) -> N.SvBlockPool:
        _expect(self.free_list, torch.int32, "free_list")
        _expect(self.free_count, torch.int32, "free_count")
        return N.SvBlockPool(_ptr(self.free_list), _ptr(self.free_count), self.free_list.shape[0])


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A 256-byte aligned device buffer of at least nbytes (torch allocations are)."""
    return torch.empty(max(1, nbytes), dtype=torch.uint8, device=device or "cuda")


# ------------------------------------------------------------------ calls --

def sv_tree_attend_workspace(batch: Batch, kv: PagedKV, n_q_heads: int) -> int:
    b, k = batch.c(), kv.c()
    return N.lib().sv_tree_attend_workspace(ctypes.byref(b), ctypes.byref(k), n_q_heads)


def _tree_attend_args(kv, batch, q, n_q_heads, softmax_scale, out, ws, dev_status):
    _expect(q, torch.bfloat16, "q")
    _expect(out, torch.bfloat16, "out")
    b, k = batch.c(), kv.c()
    return (ctypes.byref(k), ctypes.byref(b), _ptr(q), n_q_heads, softmax_scale, _ptr(out),
            _ptr(ws), ws.numel(), _ptr(dev_status))


def sv_tree_attend(kv: PagedKV, batch: Batch, q: torch.Tensor, n_q_heads: int,
                   softmax_scale: float, out: torch.Tensor, ws: torch.Tensor,
                   dev_status: Optional[torch.Tensor] = None, stream=None):
    _call("sv_tree_attend",
          _tree_attend_args(kv, batch, q, n_q_heads, softmax_scale, out, ws, dev_status), stream)


def bind_tree_attend(kv: PagedKV, batch: Batch, q: torch.Tensor, n_q_heads: int,
                     softmax_scale: float, out: torch.Tensor, ws: torch.Tensor,
                     dev_status: Optional[torch.Tensor] = None) -> BoundCall:
    """sv_tree_attend with its arguments marshalled once (see BoundCall)."""
    return BoundCall("sv_tree_attend",
                     _tree_attend_args(kv, batch, q, n_q_heads, softmax_scale, out, ws,
                                       dev_status), q.device)


def sv_accept_workspace(batch: Batch, vocab: int) -> int:
    b = batch.c()
    return N.lib().sv_accept_workspace(ctypes.byref(b), vocab)


def sv_accept(batch: Batch, target_logits: torch.Tensor, draft_logits: Optional[torch.Tensor],
              vocab: int, temperature: float, seed: int, accepted_len: torch.Tensor,
              accepted_nodes: torch.Tensor, next_token: torch.Tensor, ambiguous: torch.Tensor,
              done: Optional[torch.Tensor], row_stats: Optional[torch.Tensor], ws: torch.Tensor,
              dev_status: Optional[torch.Tensor] = None, stream=None):
    _call("sv_accept",
          _accept_args(batch, target_logits, draft_logits, vocab, temperature, seed, accepted_len,
                       accepted_nodes, next_token, ambiguous, done, row_stats, ws, dev_status),
          stream)


def _accept_args(batch, target_logits, draft_logits, vocab, temperature, seed, accepted_len,
                 accepted_nodes, next_token, ambiguous, done, row_stats, ws, dev_status):
    _expect(target_logits, torch.float32, "target_logits")
    _expect(draft_logits, torch.float32, "draft_logits")
    _expect(ambiguous, torch.uint8, "ambiguous")
    _expect(row_stats, torch.float32, "row_stats")
    b = batch.c()
    return (ctypes.byref(b), _ptr(target_logits), _ptr(draft_logits), vocab, temperature,
            seed & 0xFFFFFFFFFFFFFFFF, _ptr(accepted_len), _ptr(accepted_nodes),
            _ptr(next_token), _ptr(ambiguous), _ptr(done), _ptr(row_stats), _ptr(ws), ws.numel(),
            _ptr(dev_status))


def bind_accept(batch: Batch, target_logits: torch.Tensor,
                draft_logits: Optional[torch.Tensor], vocab: int, temperature: float, seed: int,
                accepted_len: torch.Tensor, accepted_nodes: torch.Tensor,
                next_token: torch.Tensor, ambiguous: torch.Tensor, done: Optional[torch.Tensor],
                row_stats: Optional[torch.Tensor], ws: torch.Tensor,
                dev_status: Optional[torch.Tensor] = None) -> BoundCall:
    """sv_accept with its arguments marshalled once (see BoundCall)."""
    return BoundCall("sv_accept",
                     _accept_args(batch, target_logits, draft_logits, vocab, temperature, seed,
                                  accepted_len, accepted_nodes, next_token, ambiguous, done,
                                  row_stats, ws, dev_status), target_logits.device)


def sv_accept_static(batch: Batch, target_logits: torch.Tensor,
                     draft_logits: Optional[torch.Tensor], vocab: int, temperature: float,
                     seed: int, accepted_len: torch.Tensor, accepted_nodes: torch.Tensor,
                     next_token: torch.Tensor, ambiguous: torch.Tensor,
                     done: Optional[torch.Tensor], row_stats: Optional[torch.Tensor],
                     dev_status: Optional[torch.Tensor] = None, stream=None):
    """sv_accept for callers that cannot allocate a workspace: the scratch is
    a fixed device array inside the library (see the header for its limit
    and for why concurrent calls must not overlap)."""
    _expect(target_logits, torch.float32, "target_logits")
    _expect(draft_logits, torch.float32, "draft_logits")
    _expect(ambiguous, torch.uint8, "ambiguous")
    _expect(row_stats, torch.float32, "row_stats")
    b = batch.c()
    N.check(N.lib().sv_accept_static(ctypes.byref(b), _ptr(target_logits), _ptr(draft_logits),
                                     vocab, temperature, seed & 0xFFFFFFFFFFFFFFFF,
                                     _ptr(accepted_len), _ptr(accepted_nodes), _ptr(next_token),
                                     _ptr(ambiguous), _ptr(done), _ptr(row_stats),
                                     _ptr(dev_status), _stream(stream)), "sv_accept_static")


def sv_commit_kv(kv: PagedKV, batch: Batch, accepted_len: torch.Tensor,
                 accepted_nodes: torch.Tensor, pool: BlockPool,
                 dev_status: Optional[torch.Tensor] = None, stream=None):
    b, k, p = batch.c(), kv.c(), pool.c()
    N.check(N.lib().sv_commit_kv(ctypes.byref(k), ctypes.byref(b), _ptr(accepted_len),
                                 _ptr(accepted_nodes), ctypes.byref(p), _ptr(dev_status),
                                 _stream(stream)), "sv_commit_kv")


def sv_accept_commit_workspace(batch: Batch, vocab: int) -> int:
    b = batch.c()
    return N.lib().sv_accept_commit_workspace(ctypes.byref(b), vocab)


def sv_accept_commit(batch: Batch, target_logits: torch.Tensor,
                     draft_logits: Optional[torch.Tensor], vocab: int, temperature: float,
                     seed: int, accepted_len: torch.Tensor, accepted_nodes: torch.Tensor,
                     next_token: torch.Tensor, ambiguous: torch.Tensor,
                     done: Optional[torch.Tensor], row_stats: Optional[torch.Tensor],
                     kv: PagedKV, pool: BlockPool, ws: torch.Tensor,
                     dev_status: Optional[torch.Tensor] = None, stream=None):
    _call("sv_accept_commit",
          _accept_commit_args(batch, target_logits, draft_logits, vocab, temperature, seed,
                              accepted_len, accepted_nodes, next_token, ambiguous, done,
                              row_stats, kv, pool, ws, dev_status), stream)


def _accept_commit_args(batch, target_logits, draft_logits, vocab, temperature, seed,
                        accepted_len, accepted_nodes, next_token, ambiguous, done, row_stats, kv,
                        pool, ws, dev_status):
    _expect(target_logits, torch.float32, "target_logits")
    _expect(draft_logits, torch.float32, "draft_logits")
    _expect(ambiguous, torch.uint8, "ambiguous")
    _expect(row_stats, torch.float32, "row_stats")
    b, k, p = batch.c(), kv.c(), pool.c()
    return (ctypes.byref(b), _ptr(target_logits), _ptr(draft_logits), vocab, temperature,
            seed & 0xFFFFFFFFFFFFFFFF, _ptr(accepted_len), _ptr(accepted_nodes),
            _ptr(next_token), _ptr(ambiguous), _ptr(done), _ptr(row_stats), ctypes.byref(k),
            ctypes.byref(p), _ptr(ws), ws.numel(), _ptr(dev_status))


def bind_accept_commit(batch: Batch, target_logits: torch.Tensor,
                       draft_logits: Optional[torch.Tensor], vocab: int, temperature: float,
                       seed: int, accepted_len: torch.Tensor, accepted_nodes: torch.Tensor,
                       next_token: torch.Tensor, ambiguous: torch.Tensor,
                       done: Optional[torch.Tensor], row_stats: Optional[torch.Tensor],
                       kv: PagedKV, pool: BlockPool, ws: torch.Tensor,
                       dev_status: Optional[torch.Tensor] = None) -> BoundCall:
    """sv_accept_commit with its arguments marshalled once (see BoundCall)."""
    return BoundCall("sv_accept_commit",
                     _accept_commit_args(batch, target_logits, draft_logits, vocab, temperature,
                                         seed, accepted_len, accepted_nodes, next_token,
                                         ambiguous, done, row_stats, kv, pool, ws, dev_status),
                     target_logits.device)


def sv_select_budget_workspace(n_req: int, gamma_max: int) -> int:
    return N.lib().sv_select_budget_workspace(n_req, gamma_max)


def sv_select_budget(cond_survival: torch.Tensor, gamma: Optional[torch.Tensor],
                     sps: torch.Tensor, verify_len: torch.Tensor, best_B: torch.Tensor,
                     best_theta: torch.Tensor, ws: Optional[torch.Tensor] = None,
                     dev_status: Optional[torch.Tensor] = None, stream=None):
    _expect(cond_survival, torch.float32, "cond_survival")
    _expect(sps, torch.float32, "sps")
    _expect(best_theta, torch.float64, "best_theta")
    R, gmax = cond_survival.shape
    _call("sv_select_budget",
          (R, gmax, _ptr(cond_survival), _ptr(gamma), _ptr(sps), sps.shape[0] - 1,
           _ptr(verify_len), _ptr(best_B), _ptr(best_theta), _ptr(ws),
           0 if ws is None else ws.numel(), _ptr(dev_status)), stream)


def bind_select_budget(cond_survival: torch.Tensor, gamma: Optional[torch.Tensor],
                       sps: torch.Tensor, verify_len: torch.Tensor, best_B: torch.Tensor,
                       best_theta: torch.Tensor, ws: Optional[torch.Tensor] = None,
                       dev_status: Optional[torch.Tensor] = None) -> BoundCall:
    """sv_select_budget with its arguments marshalled once (see BoundCall)."""
    _expect(cond_survival, torch.float32, "cond_survival")
    _expect(sps, torch.float32, "sps")
    _expect(best_theta, torch.float64, "best_theta")
    R, gmax = cond_survival.shape
    return BoundCall("sv_select_budget",
                     (R, gmax, _ptr(cond_survival), _ptr(gamma), _ptr(sps), sps.shape[0] - 1,
                      _ptr(verify_len), _ptr(best_B), _ptr(best_theta), _ptr(ws),
                      0 if ws is None else ws.numel(), _ptr(dev_status)), cond_survival.device)


def sv_adapt_gamma(accepted_len: torch.Tensor, verified: torch.Tensor, state: torch.Tensor,
                   gamma_next: torch.Tensor, decay: float = 0.7, overhead: float = 2.0,
                   gamma_min: int = 1, gamma_max: int = 8,
                   dev_status: Optional[torch.Tensor] = None, stream=None):
    _expect(accepted_len, torch.int32, "accepted_len")
    _expect(verified, torch.int32, "verified")
    _expect(state, torch.float64, "state")
    _expect(gamma_next, torch.int32, "gamma_next")
    N.check(N.lib().sv_adapt_gamma(accepted_len.numel(), _ptr(accepted_len), _ptr(verified),
                                   _ptr(state), _ptr(gamma_next), float(decay), float(overhead),
                                   int(gamma_min), int(gamma_max), _ptr(dev_status),
                                   _stream(stream)), "sv_adapt_gamma")


def sv_select_chunk(rows: torch.Tensor, ctx: torch.Tensor, state: torch.Tensor,
                    kv_bytes: float, row_bytes: float, chunk_bytes: int, chunk: torch.Tensor,
                    cost: torch.Tensor, costs: torch.Tensor,
                    dev_status: Optional[torch.Tensor] = None, stream=None):
    _expect(rows, torch.int32, "rows")
    _expect(ctx, torch.int32, "ctx")
    _expect(state, torch.float64, "state")
    _expect(chunk, torch.int32, "chunk")
    # cost and costs hold u64 values: any 8-byte integer tensor will do
    if cost.numel() < 1 or cost.element_size() != 8 or cost.is_floating_point():
        raise N.SpecVerifyError("cost: one 8-byte integer")
    if costs.numel() < 128 or costs.element_size() != 8 or costs.is_floating_point():
        raise N.SpecVerifyError("costs: 128 8-byte integers")
    N.check(N.lib().sv_select_chunk(rows.numel(), _ptr(rows), _ptr(ctx), _ptr(state),
                                    float(kv_bytes), float(row_bytes), int(chunk_bytes),
                                    _ptr(chunk), _ptr(cost), _ptr(costs), _ptr(dev_status),
                                    _stream(stream)), "sv_select_chunk")


def sv_selftest_bounded_wait(limit: int, dev_status: torch.Tensor, stream=None):
    _expect(dev_status, torch.int32, "dev_status")
    N.check(N.lib().sv_selftest_bounded_wait(int(limit), _ptr(dev_status), _stream(stream)),
            "sv_selftest_bounded_wait")


def sv_chunk_windows(batch: Batch, chunk_index: int, chunk_size: int,
                     done: Optional[torch.Tensor], row_begin: torch.Tensor,
                     row_end: torch.Tensor, stream=None):
    b = batch.c()
    N.check(N.lib().sv_chunk_windows(ctypes.byref(b), chunk_index, chunk_size, _ptr(done),
                                     _ptr(row_begin), _ptr(row_end), _stream(stream)),
            "sv_chunk_windows")


def sv_verify_chunked_workspace(batch: Batch, kv: PagedKV, n_q_heads: int, vocab: int) -> int:
    b, k = batch.c(), kv.c()
    return N.lib().sv_verify_chunked_workspace(ctypes.byref(b), ctypes.byref(k), n_q_heads, vocab)


def sv_verify_chunked(kv: PagedKV, batch: Batch, q: torch.Tensor, n_q_heads: int,
                      softmax_scale: float, out: torch.Tensor, target_logits: torch.Tensor,
                      draft_logits: Optional[torch.Tensor], vocab: int, temperature: float,
                      seed: int, chunk_size: int, accepted_len: torch.Tensor,
                      accepted_nodes: torch.Tensor, next_token: torch.Tensor,
                      ambiguous: torch.Tensor, done: torch.Tensor, ws: torch.Tensor,
                      dev_status: Optional[torch.Tensor] = None, stream=None):
    b, k = batch.c(), kv.c()
    _call("sv_verify_chunked",
          (ctypes.byref(k), ctypes.byref(b), _ptr(q), n_q_heads, softmax_scale, _ptr(out),
           _ptr(target_logits), _ptr(draft_logits), vocab, temperature,
           seed & 0xFFFFFFFFFFFFFFFF, chunk_size, _ptr(accepted_len), _ptr(accepted_nodes),
           _ptr(next_token), _ptr(ambiguous), _ptr(done), _ptr(ws), ws.numel(),
           _ptr(dev_status)), stream)


def sv_verify_chunked_commit(kv: PagedKV, batch: Batch, q: torch.Tensor, n_q_heads: int,
                             softmax_scale: float, out: torch.Tensor,
                             target_logits: torch.Tensor, draft_logits: Optional[torch.Tensor],
                             vocab: int, temperature: float, seed: int, chunk_size: int,
                             accepted_len: torch.Tensor, accepted_nodes: torch.Tensor,
                             next_token: torch.Tensor, ambiguous: torch.Tensor,
                             done: torch.Tensor, pool: BlockPool, ws: torch.Tensor,
                             dev_status: Optional[torch.Tensor] = None, stream=None):
    _call("sv_verify_chunked_commit",
          _chunked_commit_args(kv, batch, q, n_q_heads, softmax_scale, out, target_logits,
                               draft_logits, vocab, temperature, seed, chunk_size, accepted_len,
                               accepted_nodes, next_token, ambiguous, done, pool, ws,
                               dev_status), stream)


def _chunked_commit_args(kv, batch, q, n_q_heads, softmax_scale, out, target_logits,
                         draft_logits, vocab, temperature, seed, chunk_size, accepted_len,
                         accepted_nodes, next_token, ambiguous, done, pool, ws, dev_status):
    b, k, p = batch.c(), kv.c(), pool.c()
    return (ctypes.byref(k), ctypes.byref(b), _ptr(q), n_q_heads, softmax_scale, _ptr(out),
            _ptr(target_logits), _ptr(draft_logits), vocab, temperature,
            seed & 0xFFFFFFFFFFFFFFFF, chunk_size, _ptr(accepted_len), _ptr(accepted_nodes),
            _ptr(next_token), _ptr(ambiguous), _ptr(done), ctypes.byref(p), _ptr(ws), ws.numel(),
            _ptr(dev_status))


def bind_verify_chunked_commit(kv: PagedKV, batch: Batch, q: torch.Tensor, n_q_heads: int,
                               softmax_scale: float, out: torch.Tensor,
                               target_logits: torch.Tensor,
                               draft_logits: Optional[torch.Tensor], vocab: int,
                               temperature: float, seed: int, chunk_size: int,
                               accepted_len: torch.Tensor, accepted_nodes: torch.Tensor,
                               next_token: torch.Tensor, ambiguous: torch.Tensor,
                               done: torch.Tensor, pool: BlockPool, ws: torch.Tensor,
                               dev_status: Optional[torch.Tensor] = None) -> BoundCall:
    """sv_verify_chunked_commit with its arguments marshalled once (see BoundCall)."""
    return BoundCall("sv_verify_chunked_commit",
                     _chunked_commit_args(kv, batch, q, n_q_heads, softmax_scale, out,
                                          target_logits, draft_logits, vocab, temperature, seed,
                                          chunk_size, accepted_len, accepted_nodes, next_token,
                                          ambiguous, done, pool, ws, dev_status), q.device)
