"""Pins for the oracle's tree encoding and for the workload trees (CPU only)."""

import numpy as np
import pytest

from conftest import read_golden
from oracle import tree_encode, tree_mask
from oracle.tree import TreeError
import spec_workloads as wl


def test_tree_sizes_from_pages():
    # Hydra Guide "Candidate Tree Construction": b = [3,2,2] -> 21 speculative nodes;
    # Medusa Heads "Tree Attention": top-2 x top-3 -> 6 continuations.
    rows = read_golden("hydra_guide_tree_sizes.txt")
    for branching, n in rows:
        b = [int(x) for x in branching.split(",")]
        parent, rank = wl.cartesian_tree(b)
        tree = tree_encode(parent, rank)
        depth = tree["depth"]
        if len(b) == 3:
            assert tree["T"] - 1 == int(n)
        else:
            assert int((depth == len(b)).sum()) == int(n)
        for k in range(1, len(b) + 1):
            assert int((depth == k).sum()) == int(np.prod(b[:k]))


@pytest.mark.parametrize("branching,T", [((2, 3), 9), ((3, 2, 2), 22), ((8, 4, 2, 1), 169), ((4, 4, 4, 4), 341)])
def test_cartesian_node_counts_with_root(branching, T):
    parent, rank = wl.cartesian_tree(branching)
    tree = tree_encode(parent, rank)
    assert tree["T"] == T
    assert tree["max_depth"] == len(branching)


def test_mask_table_from_hydra_guide():
    # root 0 (the prompt's last token), A=1, B=2, A.1=3, A.2=4, B.1=5
    parent = [-1, 0, 0, 1, 1, 2]
    tree = tree_encode(parent)
    M = tree_mask(tree)
    rows = read_golden("hydra_guide_mask_table.txt")
    assert len(rows) == 5
    for i, row in enumerate(rows):
        expect = [0.0 if v == "0" else -np.inf for v in row[1:]]
        # column "Prompt Hist" is the prompt, which includes the root: always visible
        got = [M[i + 1, 0]] + list(M[i + 1, 1:])
        assert got == expect, row[0]


def test_anc_bits_match_sets_and_mask():
    rng = np.random.default_rng(0)
    for T in [1, 2, 63, 64, 65, 130]:
        parent, rank = wl.random_tree(rng, T)
        tree = tree_encode(parent, rank)
        M = tree_mask(tree)
        for i in range(T):
            for j in range(T):
                bit = (int(tree["anc_bits"][i, j // 64]) >> (j % 64)) & 1
                assert bit == (1 if M[i, j] == 0 else 0)
                # ancestor relation by walking parents independently of the encoder
                k, is_anc = i, False
                while k != -1:
                    if k == j:
                        is_anc = True
                    k = int(parent[k])
                assert is_anc == bool(bit)


@pytest.mark.parametrize("parent", [[], [0], [-1, 1], [-1, 0, 3, 1], [-1, -1]])
def test_invalid_trees_rejected(parent):
    with pytest.raises(TreeError):
        tree_encode(parent)


def test_duplicate_sibling_rank_rejected():
    with pytest.raises(TreeError):
        tree_encode([-1, 0, 0], [0, 1, 1])


def test_sparse_tree_recipe():
    parent, rank = wl.sparse_tree((8, 4, 2, 1), 64, 64)
    assert len(parent) == 64
    tree = tree_encode(parent, rank)
    assert tree["max_depth"] == 4
    # the all-rank-0 path down to depth 4 is kept
    u = 0
    for _ in range(4):
        kids = [c for c in tree["children"][u] if rank[c] == 0]
        assert len(kids) == 1
        u = kids[0]
    # ranks stay within the branching of their depth
    bmax = [None, 8, 4, 2, 1]
    for i in range(1, 64):
        assert 0 <= rank[i] < bmax[tree["depth"][i]]
    # deterministic under the same seed, different under another
    p2, r2 = wl.sparse_tree((8, 4, 2, 1), 64, 64)
    assert np.array_equal(parent, p2) and np.array_equal(rank, r2)
    p3, _ = wl.sparse_tree((8, 4, 2, 1), 64, 65)
    assert not np.array_equal(parent, p3)


def test_dense_prefix_256_is_ancestor_closed():
    p, r = wl.cartesian_tree((4, 4, 4, 4))
    p256, r256 = wl.bfs_prefix_tree(p, r, 256)
    tree = tree_encode(p256, r256)
    assert tree["T"] == 256
