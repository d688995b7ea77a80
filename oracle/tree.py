"""Candidate tree and its attention mask (oracle; test infrastructure only).

Hydra Guide, section "Candidate Tree Construction": the tree's nodes are the
tokens chosen by the heads; the root is the base token x_t and a depth-k node
comes from head k.  Section "Tree Attention Matrix with Topology-Aware Causal
Masking": the tree is flattened into a 1-D sequence and M(u, v) = 0 when v is
an ancestor of u or v = u, else -inf; the prompt is always visible.

A tree is given as parent indices in that flattened order: parent[0] = -1 for
the root and 0 <= parent[i] < i for every other node (a parent precedes its
children).  rank[i] is the top-k slot node i takes among its parent head's
candidates (0 = most probable).
"""

import numpy as np


class TreeError(ValueError):
    pass


def tree_encode(parent, rank=None):
    """Validate a parent-index tree and derive what the other steps need.

    Returns a dict with
      T          number of nodes, root included
      parent     int64 [T]
      rank       int64 [T] (0 for the root; sibling order when no rank is given)
      depth      int64 [T], depth(root) = 0, depth(i) = depth(parent(i)) + 1
      anc        list of T sorted lists: anc*(i) = {i, parent(i), ..., 0}
      words      ceil(T / 64)
      anc_bits   uint64 [T, words]: bit j of row i set iff j in anc*(i)
      children   list of T lists of child indices, ascending
      max_depth  largest depth
    """
    parent = np.asarray(parent, dtype=np.int64).reshape(-1)
    T = parent.shape[0]
    if T < 1:
        raise TreeError("a tree needs at least its root")
    if parent[0] != -1:
        raise TreeError("parent[0] must be -1 (node 0 is the root)")
    for i in range(1, T):
        if not (0 <= parent[i] < i):
            raise TreeError(f"parent[{i}] = {parent[i]} is not in [0, {i})")
    if rank is None:
        # no ranks given: number each node's children 0, 1, ... in index order
        rank = np.zeros(T, dtype=np.int64)
        seen = {}
        for i in range(1, T):
            rank[i] = seen.get(int(parent[i]), 0)
            seen[int(parent[i])] = rank[i] + 1
    rank = np.asarray(rank, dtype=np.int64).reshape(-1)
    if rank.shape[0] != T:
        raise TreeError("rank must have one entry per node")
    if T > 1 and rank[1:].min() < 0:
        raise TreeError("ranks must be non-negative")

    depth = np.zeros(T, dtype=np.int64)
    children = [[] for _ in range(T)]
    for i in range(1, T):
        depth[i] = depth[parent[i]] + 1
        children[parent[i]].append(i)
    for u in range(T):
        ranks = [int(rank[c]) for c in children[u]]
        if len(set(ranks)) != len(ranks):
            raise TreeError(f"two children of node {u} claim the same rank")

    anc = []
    for i in range(T):
        chain = []
        j = i
        while j != -1:
            chain.append(j)
            j = int(parent[j])
        anc.append(sorted(chain))

    words = (T + 63) // 64
    anc_bits = np.zeros((T, words), dtype=np.uint64)
    for i in range(T):
        for j in anc[i]:
            anc_bits[i, j // 64] |= np.uint64(1) << np.uint64(j % 64)

    return {
        "T": T,
        "parent": parent,
        "rank": rank,
        "depth": depth,
        "anc": anc,
        "words": words,
        "anc_bits": anc_bits,
        "children": children,
        "max_depth": int(depth.max()),
    }


def tree_mask(tree):
    """The tree attention matrix M_tree as a T x T float64 array (0 or -inf).

    M(u, v) = 0 iff v is an ancestor of u or v = u (Hydra Guide, "Tree Attention
    Matrix with Topology-Aware Causal Masking").
    """
    T = tree["T"]
    M = np.full((T, T), -np.inf)
    for u in range(T):
        for v in tree["anc"][u]:
            M[u, v] = 0.0
    return M
