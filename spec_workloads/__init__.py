"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds none of the method's arithmetic: it only draws random
tensors with the shapes, sizes and distributions of the five verification
workloads, builds candidate-tree topologies (which the method consumes as
input), and plants target logits so that a chosen path is the greedy one.
The CUDA library and the CPU oracle both receive exactly these bits.

Floating inputs are returned as float32 arrays, or for bf16 workloads as
uint16 arrays of bf16 bit patterns (rounded to nearest even from float32).
"""

from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np


# ----------------------------------------------------------------------------
# tree topologies

def cartesian_tree(branching):
    """Cartesian-product candidate tree in breadth-first order, root included.

    Every node at depth k-1 gets branching[k-1] children, of ranks 0..b-1.
    Returns (parent int32 [T], rank int32 [T]); T = 1 + sum_k prod_{j<=k} b_j.
    """
    parent, rank = [-1], [0]
    level = [0]
    for b in branching:
        nxt = []
        for u in level:
            for r in range(int(b)):
                parent.append(u)
                rank.append(r)
                nxt.append(len(parent) - 1)
        level = nxt
    return np.array(parent, dtype=np.int32), np.array(rank, dtype=np.int32)


def chain_tree(n):
    """A chain of n nodes (root included): node i's parent is i-1."""
    return np.arange(-1, n - 1, dtype=np.int32), np.zeros(n, dtype=np.int32)


def _children(parent):
    ch = [[] for _ in range(len(parent))]
    for i in range(1, len(parent)):
        ch[int(parent[i])].append(i)
    return ch


def sparse_tree(branching=(8, 4, 2, 1), n_nodes=64, seed=64):
    """A pruned ("sparse") tree of n_nodes nodes cut from the Cartesian tree.

    Start from the root and the all-rank-0 path; then, until n_nodes are kept,
    take the frontier (children in the full tree of kept nodes, not kept yet,
    ascending full-tree index) and keep frontier[floor(u * len)], u drawn from
    numpy's Generator(Philox(seed)).  Kept nodes are relabelled in full-tree
    (breadth-first) order; rank is the node's rank in the full tree.
    """
    fp, fr = cartesian_tree(branching)
    if n_nodes > len(fp):
        raise ValueError("more nodes requested than the full tree has")
    ch = _children(fp)
    kept = {0}
    u = 0
    while ch[u]:
        u = ch[u][0]
        kept.add(u)
    rng = np.random.Generator(np.random.Philox(seed))
    while len(kept) < n_nodes:
        frontier = sorted(c for k in kept for c in ch[k] if c not in kept)
        kept.add(frontier[int(np.floor(rng.random() * len(frontier)))])
    order = sorted(kept)
    new = {old: i for i, old in enumerate(order)}
    parent = np.array([-1] + [new[int(fp[o])] for o in order[1:]], dtype=np.int32)
    rank = np.array([int(fr[o]) for o in order], dtype=np.int32)
    return parent, rank


def bfs_prefix_tree(parent, rank, n):
    """The first n nodes of a breadth-first-ordered tree (ancestor closed)."""
    return np.asarray(parent[:n], dtype=np.int32).copy(), np.asarray(rank[:n], dtype=np.int32).copy()


def random_tree(rng, T, max_depth=None, max_children=4):
    """A random tree with parent[i] < i; ranks number each node's children 0, 1, ..."""
    parent = [-1]
    depth = [0]
    nkids = [0]
    rank = [0]
    for i in range(1, T):
        while True:
            p = int(rng.integers(0, i))
            if nkids[p] < max_children and (max_depth is None or depth[p] < max_depth):
                break
        parent.append(p)
        depth.append(depth[p] + 1)
        rank.append(nkids[p])
        nkids[p] += 1
        nkids.append(0)
    return np.array(parent, dtype=np.int32), np.array(rank, dtype=np.int32)


def tree_depths(parent):
    d = np.zeros(len(parent), dtype=np.int64)
    for i in range(1, len(parent)):
        d[i] = d[parent[i]] + 1
    return d


# ----------------------------------------------------------------------------
# tensors

def f32_to_bf16_bits(x):
    """float32 -> bf16 bit patterns, round to nearest even (storage format only; finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u >> np.uint32(16)) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    return r.astype(np.uint16)


_CHUNK = 1 << 22
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        import concurrent.futures as cf
        import os
        _POOL = cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4))
    return _POOL


def normal(key, shape, std=1.0, dtype="f32"):
    """N(0, std^2) samples as float32, or as bf16 bits when dtype == 'bf16'.

    ``key`` is a tuple of integers; the array is drawn in chunks of 2^22
    elements, chunk c from numpy's default generator seeded with key + (c,),
    so the values do not depend on how many threads fill them.
    """
    shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list)) else (shape,)))
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        x = np.random.default_rng(list(key) + [c]).standard_normal(size=hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = f32_to_bf16_bits(x) if dtype == "bf16" else x

    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        list(_pool().map(fill, range(nchunks)))
    return out.reshape(shape)


def sibling_tokens(rng, parent, B, V, root_tok=None):
    """Node tokens [B, T]: uniform in [0, V), distinct among siblings."""
    T = len(parent)
    ch = _children(parent)
    tok = np.zeros((B, T), dtype=np.int32)
    for b in range(B):
        tok[b, 0] = int(rng.integers(0, V)) if root_tok is None else int(root_tok[b])
        for u in range(T):
            if ch[u]:
                picks = rng.choice(V, size=len(ch[u]), replace=False)
                tok[b, ch[u]] = picks
    return tok


def plant_greedy(rng, key, parent, node_tok, V, lengths, std=2.0):
    """Target logits [B, T, V] ~ N(0, std^2) in which greedy acceptance stops at depth lengths[b].

    For each sequence a node u_m of depth m = lengths[b] is drawn uniformly; along
    its root path every node's row gets the next path token raised to the row
    maximum + 1; at u_m itself, if the row's argmax happens to be one of u_m's
    children's tokens, another token is raised above the maximum instead.
    """
    node_tok = np.asarray(node_tok)
    B, T = node_tok.shape
    depth = tree_depths(parent)
    ch = _children(parent)
    logits = normal(key, (B, T, V), std)
    for b in range(B):
        m = int(lengths[b])
        cands = np.nonzero(depth == m)[0]
        if cands.size == 0:
            raise ValueError(f"the tree has no node of depth {m}")
        u = int(cands[int(rng.integers(0, cands.size))])
        path = []
        v = u
        while v != -1:
            path.append(v)
            v = int(parent[v])
        path = path[::-1]
        for a, nxt in zip(path[:-1], path[1:]):
            row = logits[b, a]
            row[node_tok[b, nxt]] = row.max() + np.float32(1.0)
        row = logits[b, u]
        kids = {int(node_tok[b, c]) for c in ch[u]}
        if int(np.argmax(row)) in kids:
            other = int(rng.integers(0, V))
            while other in kids:
                other = int(rng.integers(0, V))
            row[other] = row.max() + np.float32(1.0)
    return logits


# ----------------------------------------------------------------------------
# the five workloads

@dataclass
class Workload:
    name: str
    dtype: str                      # "f32" or "bf16"
    B: int
    seed: int
    # candidate tree
    tree: Tuple                     # ("cartesian", branching) | ("sparse", branching, n, seed) | ("dense_prefix", branching, n)
    # draft heads (None when the workload has no draft part)
    d: Optional[int] = None
    V: Optional[int] = None
    cond: Optional[Tuple[int, ...]] = None
    topk: Optional[Tuple[int, ...]] = None
    # tree attention (None when absent)
    Hq: Optional[int] = None
    Hkv: Optional[int] = None
    D: Optional[int] = None
    Lmax: Optional[int] = None
    prefix: Optional[Tuple[int, int]] = None   # prefix_len ~ U{lo..hi}
    # acceptance
    accept: Optional[str] = None               # "greedy" | "rejection"
    accept_lengths: Tuple[int, ...] = ()       # planted greedy lengths, drawn uniformly
    temperature: float = 1.0
    rho: float = 0.8
    logit_scale: float = 3.0
    philox_seed: int = 1234
    parts: Tuple[str, ...] = field(default_factory=tuple)


WORKLOADS = {
    1: Workload("tiny-fp32", "f32", B=1, seed=1, tree=("cartesian", (2, 3)),
                d=256, V=1000, cond=(0, 1), topk=(2, 3),
                Hq=4, Hkv=4, D=64, Lmax=128, prefix=(128, 128),
                accept="greedy", accept_lengths=(0, 1, 2),
                parts=("draft", "attention", "accept")),
    2: Workload("vicuna7b-layer", "bf16", B=1, seed=2, tree=("sparse", (8, 4, 2, 1), 64, 64),
                V=32000, Hq=32, Hkv=32, D=128, Lmax=1024, prefix=(1024, 1024),
                accept="greedy", accept_lengths=(1, 2, 3, 4),
                parts=("attention", "accept")),
    3: Workload("hydra-heads-b4", "bf16", B=4, seed=3, tree=("sparse", (8, 4, 2, 1), 64, 64),
                d=4096, V=32000, cond=(1, 1, 1, 1), topk=(8, 4, 2, 1),
                parts=("draft",)),
    4: Workload("70b-gqa-b8", "bf16", B=8, seed=4, tree=("sparse", (8, 4, 2, 1), 64, 64),
                Hq=64, Hkv=8, D=128, Lmax=4096, prefix=(2048, 4096),
                parts=("attention",)),
    5: Workload("long32k-rejection", "bf16", B=1, seed=5, tree=("cartesian", (4, 4, 4, 4)),
                V=32000, Hq=32, Hkv=32, D=128, Lmax=32768, prefix=(32768, 32768),
                accept="rejection", temperature=0.7, rho=0.8, logit_scale=3.0, philox_seed=1234,
                parts=("attention", "accept")),
}


def make_tree(spec):
    kind = spec[0]
    if kind == "cartesian":
        return cartesian_tree(spec[1])
    if kind == "sparse":
        return sparse_tree(spec[1], spec[2], spec[3])
    if kind == "dense_prefix":
        p, r = cartesian_tree(spec[1])
        return bfs_prefix_tree(p, r, spec[2])
    raise ValueError(kind)


def _rng(seed, part):
    return np.random.default_rng([int(seed), int(part)])


def draft_inputs(w, B=None, seed=None):
    """Draft-head inputs: h [B, d] ~ N(0,1); E [V, d], W1_k [d, d_in_k], b1_k [d], W2_k [V, d] ~ N(0, 0.02^2); root tokens uniform.

    d_in_k = d (cond 0), 2d (cond 1), (k + 1) d (cond 2).
    """
    B = w.B if B is None else B
    s = w.seed if seed is None else seed
    d, V = w.d, w.V
    rng = _rng(s, 1)
    out = {
        "h": normal((s, 1, 0), (B, d), 1.0, w.dtype),
        "E": normal((s, 1, 1), (V, d), 0.02, w.dtype),
        "W1": [], "b1": [], "W2": [],
        "cond": np.array(w.cond, dtype=np.int32),
        "topk": np.array(w.topk, dtype=np.int32),
        "root_tok": rng.integers(0, V, size=B).astype(np.int32),
    }
    for k, c in enumerate(w.cond):
        d_in = d * (2 if c == 1 else k + 1 if c == 2 else 1)   # cond 2: h and the path's k embeddings
        out["W1"].append(normal((s, 1, 10 + k), (d, d_in), 0.02, w.dtype))
        out["b1"].append(normal((s, 1, 30 + k), (d,), 0.02, w.dtype))
        out["W2"].append(normal((s, 1, 50 + k), (V, d), 0.02, w.dtype))
    return out


def attention_inputs(w, T, B=None, seed=None):
    """Tree-attention inputs: Q [B,Hq,T,D], caches [B,Hkv,Lmax,D], tree K/V [B,Hkv,T,D] ~ N(0,1); prefix_len ~ U{lo..hi}.

    Cache rows at or beyond prefix_len[b] hold random values too (they must be ignored).
    """
    B = w.B if B is None else B
    s = w.seed if seed is None else seed
    lo, hi = w.prefix
    return {
        "q": normal((s, 2, 0), (B, w.Hq, T, w.D), 1.0, w.dtype),
        "k_cache": normal((s, 2, 1), (B, w.Hkv, w.Lmax, w.D), 1.0, w.dtype),
        "v_cache": normal((s, 2, 2), (B, w.Hkv, w.Lmax, w.D), 1.0, w.dtype),
        "prefix_len": _rng(s, 2).integers(lo, hi + 1, size=B).astype(np.int32),
        "k_tree": normal((s, 2, 3), (B, w.Hkv, T, w.D), 1.0, w.dtype),
        "v_tree": normal((s, 2, 4), (B, w.Hkv, T, w.D), 1.0, w.dtype),
    }


def greedy_inputs(w, parent, B=None, seed=None, node_tok=None):
    """Node tokens (distinct among siblings unless given) and planted target logits [B, T, V] fp32."""
    B = w.B if B is None else B
    s = w.seed if seed is None else seed
    rng = _rng(s, 3)
    if node_tok is None:
        node_tok = sibling_tokens(rng, parent, B, w.V)
    lengths = rng.choice(np.array(w.accept_lengths), size=B)
    logits = plant_greedy(rng, (s, 3, 0), parent, node_tok, w.V, lengths)
    return {"node_tok": np.asarray(node_tok, dtype=np.int32), "logits_p": logits, "planted": lengths}


def rejection_inputs(w, parent, rank, B=None, seed=None):
    """Draft/target logits for stochastic acceptance.

    z_q ~ N(0,1), z_p = rho * z_q + sqrt(1 - rho^2) * eps; logits = logit_scale * z
    (fp32).  The children of node u carry the tokens of the top ranks of
    logits_q[u] (child of rank r: the (r+1)-th largest, ties to the lower id).
    """
    B = w.B if B is None else B
    s = w.seed if seed is None else seed
    rng = _rng(s, 4)
    T = len(parent)
    V = w.V
    zq = normal((s, 4, 0), (B, T, V))
    eps = normal((s, 4, 1), (B, T, V))
    zp = np.float32(w.rho) * zq + np.float32(np.sqrt(1.0 - w.rho ** 2)) * eps
    lq = (np.float32(w.logit_scale) * zq).astype(np.float32)
    lp = (np.float32(w.logit_scale) * zp).astype(np.float32)
    ch = _children(parent)
    tok = np.zeros((B, T), dtype=np.int32)
    tok[:, 0] = rng.integers(0, V, size=B)
    for b in range(B):
        for u in range(T):
            if ch[u]:
                order = np.argsort(-lq[b, u], kind="stable")
                for c in ch[u]:
                    tok[b, c] = order[int(rank[c])]
    return {"node_tok": tok, "logits_p": lp, "logits_q": lq}
