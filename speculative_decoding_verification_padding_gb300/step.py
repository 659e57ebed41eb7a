"""One verification step on the GPU through the C ABI.

``DeviceStep`` uploads a workload (``workloads.Workload``) once, allocates the
outputs and workspaces with torch, and enqueues the library calls of a step:

  onepass   sv_tree_attend -> sv_accept_commit (accept and KV commit fused)
  chunked   sv_verify_chunked_commit (windows -> attend -> accept per chunk,
            early pruning; each request's KV committed in the chunk that
            stops it)
  budget    sv_select_budget -> sv_tree_attend -> sv_accept_commit,
            with the selected verify_len feeding the batch

``HostPipeline`` runs such steps on inputs that arrive in pinned host memory,
double-buffered so that the next step's upload overlaps this step's kernels.

Nothing here computes any part of the step; it only moves memory and calls.
"""

from __future__ import annotations

import copy

import numpy as np
import torch

from . import api
from .workloads import Workload


class DeviceStep:
    def __init__(self, w: Workload, device="cuda", mode: str | None = None, chunk: int | None = None):
        self.w = w
        self.device = device
        cfg = w.cfg
        self.mode = mode or ("budget" if cfg.budget else "chunked" if cfg.chunk else "onepass")
        self.chunk = chunk or cfg.chunk or 2
        self.T = float(cfg.temperature)
        self.Hq = cfg.n_q_heads
        self.V = w.target_logits.shape[1]
        self.scale = w.softmax_scale
        dev = device
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
        bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16)).view(torch.bfloat16).to(dev)
        f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)

        self.batch = api.Batch(i32(w.cu_rows), i32(w.parent), i32(w.tokens), w.max_rows)
        # The mutable cache state (block tables, cache lengths, free list and
        # count) lives in one buffer, each part on a 256-byte boundary, so that
        # restoring it before a step is a single copy.
        parts = [np.asarray(w.block_tables, dtype=np.int32), np.asarray(w.cache_lens, dtype=np.int32),
                 np.asarray(w.free_list, dtype=np.int32), np.array([w.free_count], dtype=np.int32)]
        offs, n = [], 0
        for a in parts:
            offs.append(n)
            n += (a.size + 63) // 64 * 64
        host = np.zeros(max(n, 64), dtype=np.int32)
        for a, o in zip(parts, offs):
            host[o:o + a.size] = a.ravel()
        self._state = i32(host)
        self._state0 = self._state.clone()  # pristine copy, restored before each step
        view = lambda k: self._state[offs[k]:offs[k] + parts[k].size].view(parts[k].shape)
        self.kv = api.PagedKV(bf16(w.k_cache), bf16(w.v_cache), view(0), view(1))
        self.pool = api.BlockPool(view(2), view(3))
        self.q = bf16(w.q)
        self.target = f32(w.target_logits)
        self.draft = f32(w.draft_logits) if self.T > 0 else None
        R, rows, maxr = w.n_req, w.total_rows, w.max_rows
        self.out = torch.zeros((rows, self.Hq, cfg.head_dim), dtype=torch.bfloat16, device=dev)
        self.accepted_len = torch.zeros(R, dtype=torch.int32, device=dev)
        self.accepted_nodes = torch.zeros((R, maxr), dtype=torch.int32, device=dev)
        self.next_token = torch.zeros(R, dtype=torch.int32, device=dev)
        self.ambiguous = torch.zeros(R, dtype=torch.uint8, device=dev)
        self.done = torch.zeros(R, dtype=torch.int32, device=dev)
        self.row_stats = None
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self._calls = {}
        if cfg.budget:
            self.cond = f32(w.cond_survival)
            self.gamma = i32(w.gamma)
            self.sps = f32(w.sps)
            self.verify_len = torch.zeros(R, dtype=torch.int32, device=dev)
            self.best_B = torch.zeros(1, dtype=torch.int32, device=dev)
            self.best_theta = torch.zeros(1, dtype=torch.float64, device=dev)
            self.batch_sel = api.Batch(self.batch.cu_rows, self.batch.parent, self.batch.tokens,
                                       maxr, verify_len=self.verify_len)
        ws = max(api.sv_tree_attend_workspace(self.batch, self.kv, self.Hq),
                 api.sv_accept_workspace(self.batch, self.V),
                 api.sv_accept_commit_workspace(self.batch, self.V),
                 api.sv_verify_chunked_workspace(self.batch, self.kv, self.Hq, self.V))
        self.ws = api.workspace(ws, dev)

    # ---------------------------------------------------------------------
    def restore_cache_state(self):
        self._state.copy_(self._state0)

    def _bound(self, name, batch, make):
        """The call `name` on `batch`, its arguments marshalled on first use
        (the step's tensors never move, so later calls only launch)."""
        key = (name, id(batch))
        hit = self._calls.get(key)
        if hit is None or hit[0] is not batch:
            hit = (batch, make())  # holding the batch keeps its id unique
            self._calls[key] = hit
        return hit[1]

    def attend(self, batch=None):
        b = batch or self.batch
        self._bound("attend", b, lambda: api.bind_tree_attend(
            self.kv, b, self.q, self.Hq, self.scale, self.out, self.ws, self.dev_status))()

    def accept(self, batch=None, row_stats=None):
        b = batch or self.batch
        if row_stats is not None:
            api.sv_accept(b, self.target, self.draft, self.V, self.T, self.w.seed,
                          self.accepted_len, self.accepted_nodes, self.next_token,
                          self.ambiguous, self.done, row_stats, self.ws, self.dev_status)
            return
        self._bound("accept", b, lambda: api.bind_accept(
            b, self.target, self.draft, self.V, self.T, self.w.seed, self.accepted_len,
            self.accepted_nodes, self.next_token, self.ambiguous, self.done, None, self.ws,
            self.dev_status))()

    def accept_commit(self, batch=None, row_stats=None):
        b = batch or self.batch
        if row_stats is not None:
            api.sv_accept_commit(b, self.target, self.draft, self.V, self.T, self.w.seed,
                                 self.accepted_len, self.accepted_nodes, self.next_token,
                                 self.ambiguous, self.done, row_stats, self.kv, self.pool,
                                 self.ws, self.dev_status)
            return
        self._bound("accept_commit", b, lambda: api.bind_accept_commit(
            b, self.target, self.draft, self.V, self.T, self.w.seed, self.accepted_len,
            self.accepted_nodes, self.next_token, self.ambiguous, self.done, None, self.kv,
            self.pool, self.ws, self.dev_status))()

    def chunked(self):
        api.sv_verify_chunked(self.kv, self.batch, self.q, self.Hq, self.scale, self.out,
                              self.target, self.draft, self.V, self.T, self.w.seed, self.chunk,
                              self.accepted_len, self.accepted_nodes, self.next_token,
                              self.ambiguous, self.done, self.ws, self.dev_status)

    def chunked_commit(self):
        self._bound("chunked_commit", self.batch, lambda: api.bind_verify_chunked_commit(
            self.kv, self.batch, self.q, self.Hq, self.scale, self.out, self.target, self.draft,
            self.V, self.T, self.w.seed, self.chunk, self.accepted_len, self.accepted_nodes,
            self.next_token, self.ambiguous, self.done, self.pool, self.ws, self.dev_status))()

    def select(self):
        self._bound("select", self.batch, lambda: api.bind_select_budget(
            self.cond, self.gamma, self.sps, self.verify_len, self.best_B, self.best_theta, None,
            self.dev_status))()

    def commit(self, batch=None):
        api.sv_commit_kv(self.kv, batch or self.batch, self.accepted_len, self.accepted_nodes,
                         self.pool, self.dev_status)

    def run(self, commit: bool = True, restore: bool = True):
        """Enqueue one whole step of this workload's mode on the current stream."""
        if restore:
            self.restore_cache_state()
        if self.mode == "onepass":
            self.attend()
            if commit:
                self.accept_commit()  # accept and commit fused
            else:
                self.accept()
        elif self.mode == "chunked":
            if commit:
                self.chunked_commit()  # accept and commit fused into the chunks
            else:
                self.chunked()
        elif self.mode == "budget":
            self.select()
            self.attend(self.batch_sel)
            if commit:
                self.accept_commit(self.batch_sel)
            else:
                self.accept(self.batch_sel)
        else:
            raise ValueError(self.mode)

    def inputs(self):
        """The device tensors a step reads that a caller feeds from the host each
        step, in a fixed order: q, target logits, tokens, parents, row offsets,
        then the draft logits (T > 0) and the survival inputs (budget mode)."""
        t = [self.q, self.target, self.batch.tokens, self.batch.parent, self.batch.cu_rows]
        if self.draft is not None:
            t.append(self.draft)
        if self.mode == "budget":
            t += [self.cond, self.gamma, self.sps]
        return t

    def outputs(self):
        """The device tensors a step's caller reads back: the attention output,
        accepted lengths, accepted nodes and next tokens."""
        return [self.out, self.accepted_len, self.accepted_nodes, self.next_token]

    def _twin(self):
        """A step sharing this one's KV cache, pool, outputs and workspace, with
        input tensors of its own (a second slot for double-buffered uploads)."""
        t = copy.copy(self)
        t._calls = {}
        b = self.batch
        t.batch = api.Batch(torch.empty_like(b.cu_rows), torch.empty_like(b.parent),
                            torch.empty_like(b.tokens), b.max_rows)
        t.q = torch.empty_like(self.q)
        t.target = torch.empty_like(self.target)
        t.draft = torch.empty_like(self.draft) if self.draft is not None else None
        if self.mode == "budget":
            t.cond = torch.empty_like(self.cond)
            t.gamma = torch.empty_like(self.gamma)
            t.sps = torch.empty_like(self.sps)
            t.batch_sel = api.Batch(t.batch.cu_rows, t.batch.parent, t.batch.tokens,
                                    b.max_rows, verify_len=self.verify_len)
        return t

    def results(self):
        torch.cuda.synchronize()
        return {
            "accepted_len": self.accepted_len.cpu().numpy(),
            "accepted_nodes": self.accepted_nodes.cpu().numpy(),
            "next_token": self.next_token.cpu().numpy(),
            "ambiguous": self.ambiguous.cpu().numpy(),
            "done": self.done.cpu().numpy(),
            "dev_status": int(self.dev_status.item()),
        }


class HostPipeline:
    """Steps of a ``DeviceStep`` fed from pinned host memory, inputs double-buffered.

    Each step's inputs (``DeviceStep.inputs()``) are copied from pinned host
    tensors into one of two device slots on a copy stream, and its results
    (``DeviceStep.outputs()``) are copied back to pinned host memory on the
    current stream right after its kernels.  The upload of step i + 1 goes into
    the other slot while step i's kernels run, and waits only until step i - 1
    (the slot's previous user) has finished reading it, so a step costs the
    larger of its host-link time and its kernels' time rather than their sum.
    Every step still moves all of its inputs and results across the link.
    """

    def __init__(self, step: DeviceStep):
        self.slots = [step, step._twin()]
        self.copy_stream = torch.cuda.Stream(device=step.device)
        self.uploaded = [torch.cuda.Event(), torch.cuda.Event()]
        self.released = [torch.cuda.Event(), torch.cuda.Event()]
        self.ready = [torch.cuda.Event(), torch.cuda.Event()]
        self.used = [False, False]
        self.host_out = [[torch.empty_like(t, device="cpu").pin_memory() for t in step.outputs()]
                         for _ in range(2)]
        self.n = 0
        self.begin()

    def begin(self):
        """Order the copy stream after everything enqueued so far on the current
        stream (call once before a run of steps, e.g. at the start of a timed
        region)."""
        self.copy_stream.wait_stream(torch.cuda.current_stream())

    def submit(self, host_inputs):
        """Enqueue one step on ``host_inputs`` (pinned host tensors matching
        ``DeviceStep.inputs()``) on the current stream.  Returns the slot's pinned host
        outputs and the event after which they hold this step's results; they
        stay valid until the step after next is submitted."""
        k = self.n & 1
        st, cs = self.slots[k], self.copy_stream
        main = torch.cuda.current_stream()
        dst = st.inputs()
        if len(host_inputs) != len(dst):
            raise ValueError(f"expected {len(dst)} host inputs, got {len(host_inputs)}")
        for d, h in zip(dst, host_inputs):
            if d.shape != h.shape or d.dtype != h.dtype or h.device.type != "cpu":
                raise ValueError(f"host input {tuple(h.shape)} {h.dtype} on {h.device} does not "
                                 f"match {tuple(d.shape)} {d.dtype}")
        self.n += 1
        if self.used[k]:
            cs.wait_event(self.released[k])
        self.used[k] = True
        with torch.cuda.stream(cs):
            for d, h in zip(dst, host_inputs):
                d.copy_(h, non_blocking=True)
            self.uploaded[k].record(cs)
        main.wait_event(self.uploaded[k])
        st.run()
        self.released[k].record(main)
        for h, d in zip(self.host_out[k], st.outputs()):
            h.copy_(d, non_blocking=True)
        self.ready[k].record(main)
        return self.host_out[k], self.ready[k]
