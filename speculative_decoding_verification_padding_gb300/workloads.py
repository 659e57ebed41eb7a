"""Seeded synthetic inputs for the verification step.

This module only draws random inputs with numpy and lays them out; it holds
none of the verification arithmetic.  The CUDA path and the CPU oracle are
both fed from it.  The pages measure on public datasets and real models,
which are not available here; these shapes and value distributions stand in
for them.

Workloads (one per entry of ``CONFIGS``):
  tiny      1 request, 4 drafts, 8 q / 2 kv heads, d 64, context 256,
            vocab 1024, target ~N(0, 2^2), draft = target + N(0, 0.5^2)
  chain8b   1 request, 5 drafts, 32 / 8 heads, d 128, context 4096,
            vocab 128256, target ~N(0, 3^2), draft = target + sigma z
  tree70b   1 request, 64-node draft tree (depth 6, branching 4,3,2,2,1,1
            truncated), 64 / 8 heads, d 128, context 8192, vocab 128256
  batch64   64 requests, drafts U{1..8}, 32 / 8 heads, d 128, context
            log-normal(ln 4096, 1) clipped to [512, 32768], vocab 128256
  batch256  256 requests, 4 drafts, 40 / 8 heads, d 128, context
            U{1024..8192}, vocab 151936, survival c ~ Beta(4, 2)
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16


@dataclass(frozen=True)
class Config:
    name: str
    seed: int
    n_req: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    vocab: int
    temperature: float
    target_sigma: float
    draft_sigma: float
    ctx: tuple = ()            # ("fixed", n) | ("lognormal", mu, sigma, lo, hi) | ("uniform", lo, hi)
    gamma: tuple = ()          # ("fixed", g) | ("uniform", lo, hi) | ("tree", branching, n_nodes)
    chunk: int = 0             # chunk size for pruned verification (0 = one pass)
    budget: bool = False       # budget-selected step (survival ~ Beta(4, 2), SPS table)
    sps_b_max: int = 1280


CONFIGS = {
    "tiny": Config("tiny", 0, 1, 8, 2, 64, 1024, 1.0, 2.0, 0.5, ("fixed", 256), ("fixed", 4)),
    "chain8b": Config("chain8b", 1, 1, 32, 8, 128, 128256, 1.0, 3.0, 1.0, ("fixed", 4096),
                      ("fixed", 5)),
    "tree70b": Config("tree70b", 2, 1, 64, 8, 128, 128256, 0.0, 3.0, 1.0, ("fixed", 8192),
                      ("tree", (4, 3, 2, 2, 1, 1), 64)),
    "batch64": Config("batch64", 3, 64, 32, 8, 128, 128256, 0.7, 3.0, 1.0,
                      ("lognormal", math.log(4096.0), 1.0, 512, 32768), ("uniform", 1, 8), chunk=2),
    "batch256": Config("batch256", 4, 256, 40, 8, 128, 151936, 1.0, 3.0, 1.0,
                       ("uniform", 1024, 8192), ("fixed", 4), budget=True),
}


def config(name: str, **overrides) -> Config:
    return dataclasses.replace(CONFIGS[name], **overrides)


# ------------------------------------------------------------------ helpers --

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng, shape, chunk=1 << 24):
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


def tree_shape(branching=(4, 3, 2, 2, 1, 1), n_nodes=64):
    """Draft tree: the full tree with the given branching per depth, truncated
    to the n_nodes non-root nodes of smallest (depth + sum of sibling ranks),
    ties broken by (depth, rank path).  Returns (parent, rank) in breadth-first
    order with the root at index 0 (parent -1)."""
    full = []  # (score, depth, rank_path)
    frontier = [()]
    for depth, b in enumerate(branching, start=1):
        nxt = []
        for path in frontier:
            for r in range(b):
                p = path + (r,)
                full.append((depth + sum(p), depth, p))
                nxt.append(p)
        frontier = nxt
    full.sort(key=lambda t: (t[0], t[1], t[2]))
    kept = sorted([t for t in full[:n_nodes]], key=lambda t: (t[1], t[2]))
    index = {(): 0}
    parent = [-1]
    rank = [0]
    for _, depth, p in kept:
        assert p[:-1] in index, "truncation must keep every ancestor"
        index[p] = len(parent)
        parent.append(index[p[:-1]])
        rank.append(p[-1])
    return np.array(parent, dtype=np.int32), np.array(rank, dtype=np.int32)


def _context_lengths(rng, cfg: Config, n_req: int) -> np.ndarray:
    kind = cfg.ctx[0]
    if kind == "fixed":
        return np.full(n_req, cfg.ctx[1], dtype=np.int64)
    if kind == "lognormal":
        _, mu, sig, lo, hi = cfg.ctx
        return np.clip(np.rint(rng.lognormal(mu, sig, n_req)), lo, hi).astype(np.int64)
    if kind == "uniform":
        _, lo, hi = cfg.ctx
        return rng.integers(lo, hi + 1, n_req).astype(np.int64)
    raise ValueError(kind)


def _draft_counts(rng, cfg: Config, n_req: int) -> np.ndarray:
    kind = cfg.gamma[0]
    if kind == "fixed":
        return np.full(n_req, cfg.gamma[1], dtype=np.int64)
    if kind == "uniform":
        return rng.integers(cfg.gamma[1], cfg.gamma[2] + 1, n_req).astype(np.int64)
    raise ValueError(kind)


# --------------------------------------------------------------- workload --

@dataclass
class Workload:
    cfg: Config
    # batch
    cu_rows: np.ndarray
    parent: np.ndarray
    tokens: np.ndarray
    max_rows: int
    # paged cache
    k_cache: np.ndarray           # uint16 bf16 bits [num_blocks][n_kv][16][d]
    v_cache: np.ndarray
    block_tables: np.ndarray      # int32 [R][max_blocks]
    cache_lens: np.ndarray        # int32 [R]
    free_list: np.ndarray         # int32 [num_blocks]
    free_count: int
    # step inputs
    q: np.ndarray                 # uint16 bf16 bits [rows][Hq][d]
    target_logits: np.ndarray     # fp32 [rows][V]
    draft_logits: np.ndarray      # fp32 [rows][V]
    seed: int
    # budget selection inputs
    cond_survival: np.ndarray | None = None   # fp32 [R][gamma_max]
    gamma: np.ndarray | None = None           # int32 [R]
    sps: np.ndarray | None = None             # fp32 [b_max + 1]
    extra: dict = field(default_factory=dict)

    @property
    def n_req(self):
        return self.cu_rows.shape[0] - 1

    @property
    def total_rows(self):
        return int(self.cu_rows[-1])

    @property
    def softmax_scale(self):
        return float(np.float32(1.0 / math.sqrt(self.cfg.head_dim)))

    def batch(self, verify_len=None):
        return {"cu_rows": self.cu_rows, "parent": self.parent, "tokens": self.tokens,
                "max_rows": self.max_rows, "verify_len": verify_len}

    def kv(self):
        return {"k_cache": self.k_cache, "v_cache": self.v_cache,
                "block_tables": self.block_tables, "cache_lens": self.cache_lens}

    def kv_copy(self):
        return {"k_cache": self.k_cache.copy(), "v_cache": self.v_cache.copy(),
                "block_tables": self.block_tables.copy(), "cache_lens": self.cache_lens.copy()}


def make_workload(cfg: Config, *, n_req: int | None = None, ctx_scale: float = 1.0,
                  vocab: int | None = None, draft_sigma: float | None = None,
                  temperature: float | None = None, step_seed: int | None = None,
                  slack: float = 0.10, sps: str = "synthetic") -> Workload:
    """Draw one verification step of workload ``cfg``.

    ``n_req``, ``ctx_scale`` and ``vocab`` shrink the workload for tests that
    the oracle must finish in seconds; ``draft_sigma`` sweeps acceptance;
    ``temperature`` overrides the sampling temperature used to draw drafts.
    ``sps`` (budget workloads): "synthetic" (1000 / (1 + B / 512)) or
    "measured" (the table ``sps.py`` measured from this library's kernels).
    """
    rng = np.random.default_rng(cfg.seed)
    R = cfg.n_req if n_req is None else n_req
    V = cfg.vocab if vocab is None else vocab
    T = cfg.temperature if temperature is None else temperature
    sig_d = cfg.draft_sigma if draft_sigma is None else draft_sigma
    H, Hkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim

    ctx = _context_lengths(rng, cfg, R)
    if ctx_scale != 1.0:
        ctx = np.maximum(1, np.rint(ctx * ctx_scale)).astype(np.int64)

    # ---- batch topology ----
    if cfg.gamma[0] == "tree":
        par1, rank1 = tree_shape(cfg.gamma[1], cfg.gamma[2])
        parents = [par1] * R
        ranks = [rank1] * R
    else:
        g = _draft_counts(rng, cfg, R)
        parents = [np.arange(-1, int(gi), dtype=np.int32) for gi in g]
        ranks = [np.zeros(int(gi) + 1, dtype=np.int32) for gi in g]
    rows = np.array([len(p) for p in parents], dtype=np.int64)
    cu_rows = np.zeros(R + 1, dtype=np.int32)
    cu_rows[1:] = np.cumsum(rows)
    total_rows = int(cu_rows[-1])
    parent = np.concatenate(parents).astype(np.int32)
    max_rows = int(rows.max())

    # ---- logits: target ~ N(0, sigma_t^2), draft = target + N(0, sigma_d^2) ----
    target = np.empty((total_rows, V), dtype=np.float32)
    draft = np.empty((total_rows, V), dtype=np.float32)
    for r in range(total_rows):
        target[r] = rng.standard_normal(V, dtype=np.float32) * np.float32(cfg.target_sigma)
    noise_rng = np.random.default_rng(cfg.seed + 1000)  # same z for every sigma of a sweep
    for r in range(total_rows):
        draft[r] = target[r] + noise_rng.standard_normal(V, dtype=np.float32) * np.float32(sig_d)

    # ---- draft tokens (the drafter's proposals) ----
    tok_rng = np.random.default_rng(cfg.seed + 2000)
    tokens = np.zeros(total_rows, dtype=np.int32)
    for i in range(R):
        base = int(cu_rows[i])
        tokens[base] = tok_rng.integers(0, V)  # root: last committed token
        if cfg.gamma[0] == "tree" and T > 0:
            # sampling: siblings drawn independently from softmax(draft at the
            # parent / T), with replacement (Gumbel-max)
            for j in range(1, rows[i]):
                row = draft[base + int(parents[i][j])]
                gum = tok_rng.gumbel(size=V)
                tokens[base + j] = int(np.argmax(row.astype(np.float64) / T + gum))
        elif cfg.gamma[0] == "tree":
            # greedy: siblings are the top-b draft tokens at the parent
            # (distinct, lower index first on ties)
            order_cache = {}
            for j in range(1, rows[i]):
                p = int(parents[i][j])
                if p not in order_cache:
                    order_cache[p] = np.argsort(-draft[base + p], kind="stable")
                tokens[base + j] = order_cache[p][ranks[i][j]]
        else:
            for j in range(1, rows[i]):
                row = draft[base + j - 1]
                if T > 0:
                    # sample from softmax(row / T) via the Gumbel-max trick
                    gum = tok_rng.gumbel(size=V)
                    tokens[base + j] = int(np.argmax(row.astype(np.float64) / T + gum))
                else:
                    tokens[base + j] = int(np.argmax(row))

    # ---- paged KV cache: blocks shuffled over a pool with `slack` spare ----
    need = (ctx + rows + BLOCK_SIZE - 1) // BLOCK_SIZE
    n_used = int(need.sum())
    num_blocks = int(math.ceil(n_used * (1.0 + slack))) + 1
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = int(need.max())
    block_tables = np.full((R, max_blocks), -1, dtype=np.int32)
    pos = 0
    for i in range(R):
        block_tables[i, : need[i]] = perm[pos: pos + need[i]]
        pos += int(need[i])
    free_list = np.full(num_blocks, -1, dtype=np.int32)
    free_count = num_blocks - pos
    free_list[:free_count] = perm[pos:]
    kv_rng = np.random.default_rng(cfg.seed + 3000)
    k_cache = _normal_bf16(kv_rng, (num_blocks, Hkv, BLOCK_SIZE, d))
    v_cache = _normal_bf16(kv_rng, (num_blocks, Hkv, BLOCK_SIZE, d))
    q = _normal_bf16(kv_rng, (total_rows, H, d))

    w = Workload(cfg=dataclasses.replace(cfg, temperature=T, draft_sigma=sig_d, vocab=V),
                 cu_rows=cu_rows, parent=parent, tokens=tokens, max_rows=max_rows,
                 k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
                 cache_lens=ctx.astype(np.int32), free_list=free_list, free_count=free_count,
                 q=q, target_logits=target, draft_logits=draft,
                 seed=(cfg.seed * 7919 + 17) if step_seed is None else step_seed)

    if cfg.budget:
        b_rng = np.random.default_rng(cfg.seed + 4000)
        gmax = int(rows.max()) - 1
        w.cond_survival = b_rng.beta(4.0, 2.0, size=(R, gmax)).astype(np.float32)
        w.gamma = (rows - 1).astype(np.int32)
        if sps == "measured":
            from .sps import load_measured
            w.sps = load_measured(cfg.sps_b_max)
        else:
            B = np.arange(cfg.sps_b_max + 1, dtype=np.float64)
            w.sps = (1000.0 / (1.0 + B / 512.0)).astype(np.float32)
    return w
