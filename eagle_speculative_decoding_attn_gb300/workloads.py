"""Seeded synthetic inputs for EAGLE-style tree verification.

This module only *draws* inputs: draft trees (parent-index arrays), paged
bf16 Q/K/V, fp32 target/draft logits and the uniforms that the sampling
acceptance consumes. It performs none of the verification arithmetic
(no attention, no softmax, no acceptance), so both the fp64 oracle and the
CUDA path can consume its output without sharing any of the method.

Workload shapes follow the five Llama-shaped cases of the tree-verification
step:  tiny parity case, Llama-2-7B-shaped (MHA 32 heads), Llama-3-70B-shaped
(GQA 64/8), a 32-request serving batch (GQA 32/8) and a long-context batch
(L = 32768).  Tree bounds follow "SGLang EAGLE-2 Speculative Decoding"
(Tech Radar), section 2 "Dynamic Tree-Attention Masking": at most 64
candidate nodes, expansion depth 4-6, up to 8 children per node.

All randomness comes from numpy PCG64 seeded with ``1000 + config index``;
numpy's PCG64 / ziggurat normals are bit-identical on x86_64 and aarch64.
bf16 values are produced by torch's round-to-nearest-even cast and are kept
as raw ``uint16`` bit patterns so numpy can carry them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

PAGE_SIZE = 16
MAX_NODES = 64


# --------------------------------------------------------------------------
# configuration
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    index: int                 # position in the list below; seed = 1000 + index
    B: int
    Hq: int
    Hkv: int
    D: int
    prefix: tuple              # ("fixed", L) | ("uniform", lo, hi) | ("loguniform", lo, hi)
    tree: str                  # "random3" | "levels" | "depth4to6" | "serving"
    n_nodes: tuple             # ("fixed", N) | ("uniform", lo, hi)
    V: int
    temperature: float         # 0 => greedy
    sigma: float
    rho: Optional[float]       # None => target and draft drawn independently
    n_layers_commit: int = 1   # layers moved by kv_commit_path in the full step
    extra_greedy: bool = False  # tiny: also run a greedy acceptance on the same tree

    @property
    def seed(self) -> int:
        return 1000 + self.index


CONFIGS: List[Config] = [
    Config("tiny", 0, B=1, Hq=4, Hkv=4, D=64, prefix=("fixed", 128), tree="random3",
           n_nodes=("fixed", 8), V=1000, temperature=1.0, sigma=2.0, rho=None,
           extra_greedy=True),
    Config("llama2_7b", 1, B=1, Hq=32, Hkv=32, D=128, prefix=("fixed", 2048), tree="levels",
           n_nodes=("fixed", 64), V=32000, temperature=0.0, sigma=2.0, rho=0.8,
           n_layers_commit=32),
    Config("llama3_70b", 2, B=8, Hq=64, Hkv=8, D=128, prefix=("uniform", 1024, 8192),
           tree="depth4to6", n_nodes=("fixed", 64), V=128256, temperature=0.7, sigma=3.0,
           rho=0.8, n_layers_commit=80),
    Config("serving", 3, B=32, Hq=32, Hkv=8, D=128, prefix=("loguniform", 256, 16384),
           tree="serving", n_nodes=("uniform", 16, 64), V=128256, temperature=0.0, sigma=3.0,
           rho=0.8, n_layers_commit=80),
    Config("long", 4, B=4, Hq=64, Hkv=8, D=128, prefix=("fixed", 32768), tree="levels",
           n_nodes=("fixed", 64), V=128256, temperature=1.0, sigma=3.0, rho=0.8,
           n_layers_commit=80),
]
CONFIG_BY_NAME = {c.name: c for c in CONFIGS}

# Level schedules (nodes per depth, root first) used for the fixed-shape trees.
# Each level holds at most 8x the previous one, so every node can keep <= 8
# children; all sum to 64 nodes.
LEVEL_SCHEDULES = {
    4: [1, 8, 24, 19, 12],
    5: [1, 8, 16, 16, 14, 9],
    6: [1, 8, 16, 16, 12, 8, 3],
}


# --------------------------------------------------------------------------
# bf16 helpers (input generation only)
# --------------------------------------------------------------------------
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even, via torch) and return uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# tree shapes (parent-index arrays, node 0 = root, parent[i] < i)
# --------------------------------------------------------------------------
def chain_tree(n: int) -> np.ndarray:
    p = np.arange(-1, n - 1, dtype=np.int32)
    return p


def star_tree(n: int) -> np.ndarray:
    p = np.zeros(n, dtype=np.int32)
    p[0] = -1
    return p


def random_recursive_tree(rng: np.random.Generator, n: int, depth: Optional[int] = None,
                          max_tries: int = 100000) -> np.ndarray:
    """parent[i] ~ U{0..i-1}; redrawn until the tree's depth equals ``depth``."""
    for _ in range(max_tries):
        p = np.empty(n, dtype=np.int32)
        p[0] = -1
        d = np.zeros(n, dtype=np.int64)
        for i in range(1, n):
            p[i] = rng.integers(0, i)
            d[i] = d[p[i]] + 1
        if depth is None or (n > 0 and int(d.max()) == depth):
            return p
    raise RuntimeError("could not draw a tree of the requested depth")


def level_tree(rng: np.random.Generator, levels: List[int], max_children: int = 8) -> np.ndarray:
    """Nodes numbered level by level; each node of level k+1 picks a random parent
    on level k that still has fewer than ``max_children`` children."""
    assert levels[0] == 1
    n = sum(levels)
    p = np.empty(n, dtype=np.int32)
    p[0] = -1
    start_prev, start = 0, 1
    for k in range(1, len(levels)):
        prev = list(range(start_prev, start_prev + levels[k - 1]))
        assert levels[k] <= max_children * len(prev)
        count = {x: 0 for x in prev}
        # every parent slot of the previous level is eligible; draw without
        # exceeding the per-node bound
        for j in range(levels[k]):
            cand = [x for x in prev if count[x] < max_children]
            x = cand[int(rng.integers(0, len(cand)))]
            count[x] += 1
            p[start + j] = x
        start_prev, start = start, start + levels[k]
    # renumber so that each node's children are contiguous and ascending in
    # the parent's order (a breadth-first numbering); parents stay < children
    order = _bfs_order(p)
    return _relabel(p, order)


def _bfs_order(p: np.ndarray) -> List[int]:
    n = len(p)
    kids = [[] for _ in range(n)]
    for i in range(1, n):
        kids[p[i]].append(i)
    order, head = [0], 0
    while head < len(order):
        order.extend(kids[order[head]])
        head += 1
    return order


def _relabel(p: np.ndarray, order: List[int]) -> np.ndarray:
    new_id = {old: new for new, old in enumerate(order)}
    q = np.empty_like(p)
    for old, new in new_id.items():
        q[new] = -1 if p[old] < 0 else new_id[int(p[old])]
    return q


def serving_levels(n: int) -> List[int]:
    """Width-8 expansion for a high-entropy row: 8 children at the root, the
    remaining nodes spread evenly over at most five further levels."""
    if n == 1:
        return [1]
    first = min(8, n - 1)
    rest = n - 1 - first
    levels = [1, first]
    n_lv = min(5, rest) if rest > 0 else 0
    for k in range(n_lv):
        levels.append(rest // n_lv + (1 if k < rest % n_lv else 0))
    return levels


def tree_depths(p: np.ndarray) -> np.ndarray:
    d = np.zeros(len(p), dtype=np.int64)
    for i in range(1, len(p)):
        d[i] = d[p[i]] + 1
    return d


def children_lists(p: np.ndarray, n: int) -> List[List[int]]:
    kids = [[] for _ in range(n)]
    for i in range(1, n):
        kids[int(p[i])].append(i)
    return kids


# --------------------------------------------------------------------------
# the workload container
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    cfg: Config
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    n_max: int
    prefix_len: np.ndarray      # int32 [B]
    n_nodes: np.ndarray         # int32 [B]
    parents: np.ndarray         # int32 [B, n_max]   (-1 past n_nodes)
    tokens: np.ndarray          # int32 [B, n_max]   (root's entry unused)
    q_bits: np.ndarray          # uint16 [B, n_max, Hq, D]   bf16 bits
    k_bits: np.ndarray          # uint16 [num_pages, Hkv, P, D]
    v_bits: np.ndarray          # uint16 [num_pages, Hkv, P, D]
    page_table: np.ndarray      # int32 [B, max_pages]  (-1 past the request's pages)
    scale: float
    V: int
    temperature: float
    target_logits: Optional[np.ndarray]  # fp32 [B, n_max, V]
    draft_logits: Optional[np.ndarray]   # fp32 [B, n_max, V] (None when greedy)
    u_accept: np.ndarray        # fp32 [B, n_max] in [0,1)
    u_sample: np.ndarray        # fp32 [B, n_max] in [0,1)

    @property
    def num_pages(self) -> int:
        return int(self.k_bits.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    # algorithmic counts of the verify attention (KV of the visible
    # positions read once, Q read once; FLOPs of masked-in pairs only)
    def attn_bytes(self) -> int:
        kv = int(np.sum(self.prefix_len.astype(np.int64) + self.n_nodes)) * self.Hkv * self.D * 2 * 2
        qb = int(np.sum(self.n_nodes)) * self.Hq * self.D * 2
        return kv + qb

    def attn_bytes_q4(self) -> int:
        """attn_bytes with K and V in the 4-bit format: D/2 code bytes and D/32
        (scale, zero) fp16 pairs per row."""
        kv = int(np.sum(self.prefix_len.astype(np.int64) + self.n_nodes)) * self.Hkv * (self.D // 2 + self.D // 8) * 2
        qb = int(np.sum(self.n_nodes)) * self.Hq * self.D * 2
        return kv + qb

    def attn_flops(self) -> int:
        tot = 0
        for b in range(self.B):
            n = int(self.n_nodes[b])
            d = tree_depths(self.parents[b, :n])
            tot += int(np.sum(int(self.prefix_len[b]) + d + 1))
        return 4 * self.D * self.Hq * tot

    def out_bytes(self) -> int:
        return int(np.sum(self.n_nodes)) * self.Hq * self.D * 2


def _draw_prefix(rng, cfg: Config, B: int) -> np.ndarray:
    kind = cfg.prefix[0]
    if kind == "fixed":
        return np.full(B, cfg.prefix[1], dtype=np.int32)
    if kind == "uniform":
        return rng.integers(cfg.prefix[1], cfg.prefix[2] + 1, size=B).astype(np.int32)
    if kind == "loguniform":
        lo, hi = math.log(cfg.prefix[1]), math.log(cfg.prefix[2])
        return np.round(np.exp(rng.uniform(lo, hi, size=B))).astype(np.int32)
    raise ValueError(kind)


def _draw_tree(rng, cfg: Config, n: int):
    """Returns (parents, is_chain)."""
    if cfg.tree == "random3":
        return random_recursive_tree(rng, n, depth=3), False
    if cfg.tree == "levels":
        return level_tree(rng, LEVEL_SCHEDULES[6]), False
    if cfg.tree == "depth4to6":
        depth = int(rng.integers(4, 7))
        return level_tree(rng, LEVEL_SCHEDULES[depth]), False
    if cfg.tree == "serving":
        if rng.random() < 0.5:                   # low-entropy row: a chain
            return chain_tree(n), True
        return level_tree(rng, serving_levels(n)), False
    raise ValueError(cfg.tree)


def _gumbel_argmax(rng, logits_row: np.ndarray, temperature: float, count: int) -> List[int]:
    """``count`` i.i.d. draws from the categorical with logits ``row / T``
    (Gumbel-max trick; the drafter's sampling, not the verifier's)."""
    out = []
    for _ in range(count):
        g = rng.gumbel(size=logits_row.shape[0]).astype(np.float64)
        out.append(int(np.argmax(logits_row.astype(np.float64) / temperature + g)))
    return out


def _gumbel_top_k(rng, logits_row: np.ndarray, temperature: float, count: int) -> List[int]:
    """``count`` distinct tokens drawn without replacement from the categorical
    with logits ``row / T``: the ``count`` largest of row / T + Gumbel noise,
    largest first (Gumbel top-k; the drafter's sampling)."""
    g = rng.gumbel(size=logits_row.shape[0]).astype(np.float64)
    z = logits_row.astype(np.float64) / temperature + g
    order = np.argsort(-z, kind="stable")[:count]
    return [int(x) for x in order]


def _top_k(logits_row: np.ndarray, k: int) -> List[int]:
    """The drafter's top-k expansion: the k largest draft logits, largest first
    (equal values by ascending token id)."""
    row = logits_row.astype(np.float64)
    k = min(k, row.shape[0])
    part = np.argpartition(-row, k - 1)[:k]
    order = sorted(part.tolist(), key=lambda t: (-row[t], t))
    return [int(x) for x in order]


def make_workload(cfg, seed: Optional[int] = None, *, with_logits: bool = True,
                  B: Optional[int] = None, siblings: str = "iid") -> Workload:
    """Draw the full synthetic input of a config.

    ``B`` overrides the batch (a prefix of the same request stream), used for
    bounded samples of a workload.  ``siblings`` selects how a sampled
    (T > 0) node's children are drafted from q: "iid" (independent draws,
    repeats possible) or "wor" (without replacement: distinct tokens, Gumbel
    top-k).
    """
    if isinstance(cfg, str):
        cfg = CONFIG_BY_NAME[cfg]
    rng = np.random.Generator(np.random.PCG64(cfg.seed if seed is None else seed))
    B = cfg.B if B is None else B
    P = PAGE_SIZE
    n_max = MAX_NODES if cfg.n_nodes[0] == "uniform" else cfg.n_nodes[1]
    prefix = _draw_prefix(rng, cfg, B)
    if cfg.n_nodes[0] == "fixed":
        n_nodes = np.full(B, cfg.n_nodes[1], dtype=np.int32)
    else:
        n_nodes = rng.integers(cfg.n_nodes[1], cfg.n_nodes[2] + 1, size=B).astype(np.int32)

    parents = np.full((B, n_max), -1, dtype=np.int32)
    chains = []
    for b in range(B):
        p, is_chain = _draw_tree(rng, cfg, int(n_nodes[b]))
        assert len(p) == n_nodes[b]
        parents[b, : len(p)] = p
        chains.append(is_chain)

    # paged KV cache: a shuffled pool of exactly the pages the batch needs
    pages_per = [(int(prefix[b]) + int(n_nodes[b]) + P - 1) // P for b in range(B)]
    num_pages = int(sum(pages_per))
    max_pages = int(max(pages_per))
    perm = rng.permutation(num_pages).astype(np.int32)
    page_table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        page_table[b, : pages_per[b]] = perm[off: off + pages_per[b]]
        off += pages_per[b]

    kv_shape = (num_pages, cfg.Hkv, P, cfg.D)
    k_bits = to_bf16_bits(rng.standard_normal(kv_shape, dtype=np.float32))
    v_bits = to_bf16_bits(rng.standard_normal(kv_shape, dtype=np.float32))
    q_bits = to_bf16_bits(rng.standard_normal((B, n_max, cfg.Hq, cfg.D), dtype=np.float32))

    V, T = cfg.V, cfg.temperature
    target = draft = None
    tokens = np.zeros((B, n_max), dtype=np.int32)
    u_accept = rng.random((B, n_max), dtype=np.float32)
    u_sample = rng.random((B, n_max), dtype=np.float32)
    if with_logits:
        target = np.zeros((B, n_max, V), dtype=np.float32)
        draft = np.zeros((B, n_max, V), dtype=np.float32)
        for b in range(B):
            n = int(n_nodes[b])
            a = rng.standard_normal((n, V), dtype=np.float32)
            if cfg.rho is None:
                bb = rng.standard_normal((n, V), dtype=np.float32)
                target[b, :n] = cfg.sigma * a
                draft[b, :n] = cfg.sigma * bb
            else:
                bb = rng.standard_normal((n, V), dtype=np.float32)
                target[b, :n] = cfg.sigma * a
                draft[b, :n] = cfg.sigma * (cfg.rho * a + math.sqrt(1.0 - cfg.rho ** 2) * bb)
            kids = children_lists(parents[b], n)
            for node in range(n):
                if not kids[node]:
                    continue
                if T > 0 and siblings == "wor":
                    toks = _gumbel_top_k(rng, draft[b, node], T, len(kids[node]))
                elif T > 0:
                    toks = _gumbel_argmax(rng, draft[b, node], T, len(kids[node]))
                else:
                    toks = _top_k(draft[b, node], len(kids[node]))
                for c, t in zip(kids[node], toks):
                    tokens[b, c] = t
        if T == 0:
            draft = None
    else:
        for b in range(B):
            tokens[b, : int(n_nodes[b])] = rng.integers(0, V, size=int(n_nodes[b]))

    return Workload(cfg=cfg, B=B, Hq=cfg.Hq, Hkv=cfg.Hkv, D=cfg.D, page_size=P, n_max=n_max,
                    prefix_len=prefix, n_nodes=n_nodes, parents=parents, tokens=tokens,
                    q_bits=q_bits, k_bits=k_bits, v_bits=v_bits, page_table=page_table,
                    scale=1.0 / math.sqrt(cfg.D), V=V, temperature=T, target_logits=target,
                    draft_logits=draft, u_accept=u_accept, u_sample=u_sample)


def make_custom(*, B, Hq, Hkv, D, prefix_len, parents_list, seed=0, V=16, temperature=0.0,
                sigma=2.0, extra_pages=0, shuffle_pages=True, n_max=None) -> Workload:
    """Small hand-shaped workloads for edge-case tests (explicit trees and prefix lengths)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    P = PAGE_SIZE
    n_nodes = np.array([len(p) for p in parents_list], dtype=np.int32)
    n_max = int(n_max or max(1, int(n_nodes.max())))
    prefix = np.asarray(prefix_len, dtype=np.int32)
    parents = np.full((B, n_max), -1, dtype=np.int32)
    for b, p in enumerate(parents_list):
        parents[b, : len(p)] = p
    pages_per = [(int(prefix[b]) + int(n_nodes[b]) + P - 1) // P for b in range(B)]
    num_pages = int(sum(pages_per)) + extra_pages
    max_pages = max(1, int(max(pages_per)))
    perm = rng.permutation(num_pages).astype(np.int32) if shuffle_pages else np.arange(num_pages, dtype=np.int32)
    page_table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        page_table[b, : pages_per[b]] = perm[off: off + pages_per[b]]
        off += pages_per[b]
    kv_shape = (max(num_pages, 1), Hkv, P, D)
    k_bits = to_bf16_bits(rng.standard_normal(kv_shape, dtype=np.float32))
    v_bits = to_bf16_bits(rng.standard_normal(kv_shape, dtype=np.float32))
    q_bits = to_bf16_bits(rng.standard_normal((B, n_max, Hq, D), dtype=np.float32))
    target = (sigma * rng.standard_normal((B, n_max, V), dtype=np.float32)).astype(np.float32)
    draft = (sigma * rng.standard_normal((B, n_max, V), dtype=np.float32)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, n_max)).astype(np.int32)
    cfg = Config("custom", -1, B=B, Hq=Hq, Hkv=Hkv, D=D, prefix=("fixed", 0), tree="custom",
                 n_nodes=("fixed", n_max), V=V, temperature=temperature, sigma=sigma, rho=None)
    return Workload(cfg=cfg, B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=P, n_max=n_max,
                    prefix_len=prefix, n_nodes=n_nodes, parents=parents, tokens=tokens,
                    q_bits=q_bits, k_bits=k_bits, v_bits=v_bits, page_table=page_table,
                    scale=1.0 / math.sqrt(D), V=V, temperature=temperature,
                    target_logits=target, draft_logits=draft if temperature > 0 else None,
                    u_accept=rng.random((B, n_max), dtype=np.float32),
                    u_sample=rng.random((B, n_max), dtype=np.float32))


# --------------------------------------------------------------------------
# dynamic tree construction inputs
# --------------------------------------------------------------------------
ROW_PEAKED, ROW_FEW, ROW_FLAT = 0, 1, 2


@dataclasses.dataclass
class ExpandWorkload:
    B: int
    n_max: int
    V: int
    draft_logits: np.ndarray    # fp32 [B, n_max, V]: the drafter's row for every node id
    kinds: np.ndarray           # int8 [B, n_max]: ROW_PEAKED / ROW_FEW / ROW_FLAT
    root_tokens: np.ndarray     # int32 [B]
    n_levels: int
    top_k: int
    max_new: int
    budget: int

    def level_bytes(self, frontier_rows: int) -> int:
        """Logit bytes one level reads for this many frontier rows in total."""
        return int(frontier_rows) * self.V * 4


def make_expand_workload(B: int, n_max: int, V: int, *, seed: int, n_levels: int = 6, top_k: int = 8,
                         max_new: int = 16, budget: Optional[int] = None, p_kinds=(0.35, 0.35, 0.30),
                         sigma_flat: float = 3.0, spike: float = 25.0) -> ExpandWorkload:
    """Synthetic drafter rows for dynamic tree construction.

    Every row is one of three kinds, drawn with probabilities ``p_kinds``:
      peaked: N(0,1) logits plus ``spike`` on one random token (a
              deterministic context: entropy near 0, a single branch);
      few:    N(0,1) logits plus spike + N(0, 0.7) on 2..6 random tokens (a
              handful of plausible continuations: perplexity between 1 and 6);
      flat:   sigma_flat * N(0,1) logits (an open context: high entropy, the
              widest branching).
    Rows exist for every node id the tree may reach; a row is read only when
    its node is on a frontier.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    kinds = rng.choice(3, size=(B, n_max), p=list(p_kinds)).astype(np.int8)
    logits = rng.standard_normal((B, n_max, V), dtype=np.float32)
    for b in range(B):
        for f in range(n_max):
            k = int(kinds[b, f])
            if k == ROW_FLAT:
                logits[b, f] *= np.float32(sigma_flat)
            elif k == ROW_PEAKED:
                logits[b, f, int(rng.integers(0, V))] += np.float32(spike)
            else:
                cnt = min(V, int(rng.integers(2, 7)))
                toks = rng.choice(V, size=cnt, replace=False)
                logits[b, f, toks] += (spike + 0.7 * rng.standard_normal(cnt)).astype(np.float32)
    root_tokens = rng.integers(0, V, size=B).astype(np.int32)
    return ExpandWorkload(B=B, n_max=n_max, V=V, draft_logits=logits, kinds=kinds, root_tokens=root_tokens,
                          n_levels=n_levels, top_k=top_k, max_new=max_new,
                          budget=n_max if budget is None else budget)


# --------------------------------------------------------------------------
# 4-bit KV caches
# --------------------------------------------------------------------------
Q4_GROUP = 32


def make_q4_cache(rng: np.random.Generator, num_pages: int, Hkv: int, D: int):
    """A random 4-bit paged cache: codes uint8 [num_pages, Hkv, 16, D/2] (two
    4-bit codes per byte, low nibble = even dim) drawn uniformly, and params
    float16 [num_pages, Hkv, 16, 2 * D / 32]: per row and group of 32 dims a
    scale ~ U(0.12, 0.30) and a zero ~ -7.5 * scale + N(0, 0.05), so decoded
    values spread like N(0, 1) around 0."""
    codes = rng.integers(0, 256, size=(num_pages, Hkv, PAGE_SIZE, D // 2), dtype=np.uint8)
    g = D // Q4_GROUP
    s = rng.uniform(0.12, 0.30, size=(num_pages, Hkv, PAGE_SIZE, g))
    z = -7.5 * s + 0.05 * rng.standard_normal(size=s.shape)
    params = np.empty((num_pages, Hkv, PAGE_SIZE, 2 * g), dtype=np.float16)
    params[..., 0::2] = s.astype(np.float16)
    params[..., 1::2] = z.astype(np.float16)
    return codes, params


def make_q3_cache(rng: np.random.Generator, num_pages: int, Hkv: int, D: int):
    """A random 3-bit paged cache: codes uint8 [num_pages, Hkv, 16, 3*D/8]
    (every bit uniform, so codes 0..7 are uniform) and params float16
    [num_pages, Hkv, 16, 2 * D / 32]: per row and group of 32 dims a scale
    ~ U(0.25, 0.60) and a zero ~ -3.5 * scale + N(0, 0.05), so decoded values
    spread like N(0, 1) around 0."""
    codes = rng.integers(0, 256, size=(num_pages, Hkv, PAGE_SIZE, 3 * D // 8), dtype=np.uint8)
    g = D // Q4_GROUP
    s = rng.uniform(0.25, 0.60, size=(num_pages, Hkv, PAGE_SIZE, g))
    z = -3.5 * s + 0.05 * rng.standard_normal(size=s.shape)
    params = np.empty((num_pages, Hkv, PAGE_SIZE, 2 * g), dtype=np.float16)
    params[..., 0::2] = s.astype(np.float16)
    params[..., 1::2] = z.astype(np.float16)
    return codes, params
