"""Pins for the oracle's KV commit of the accepted path (CPU only).

Independent check: the Hydra Guide's path equivalence ("Tree Attention Matrix
with Topology-Aware Causal Masking") -- after the commit, torch's
scaled_dot_product_attention (a library routine, no mask: every committed row
is visible) of the accepted node's query over the first prefix_len + m + 1
cache rows equals that node's tree attention before the commit.  Plus the
invariants of a copy: bits land unchanged, nothing else moves, invalid
sequences are left alone.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import spec_workloads as wl
from oracle import kv_commit, tree_attention, tree_encode


def _path_to(tree, u):
    path = [u]
    while path[-1] != 0:
        path.append(int(tree["parent"][path[-1]]))
    return path[::-1]


def _case(rng, B, Hq, Hkv, T, D, Lmax, prefix):
    parent, rank = wl.random_tree(rng, T, max_children=3)
    tree = tree_encode(parent, rank)
    x = dict(q=rng.standard_normal((B, Hq, T, D)).astype(np.float32),
             k_cache=rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32),
             v_cache=rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32),
             prefix_len=np.array(prefix, dtype=np.int32),
             k_tree=rng.standard_normal((B, Hkv, T, D)).astype(np.float32),
             v_tree=rng.standard_normal((B, Hkv, T, D)).astype(np.float32))
    return tree, x


def _paths(rng, tree, B):
    K1 = tree["max_depth"] + 1
    ends = [int(rng.integers(0, tree["T"])) for _ in range(B)]
    alen = np.array([tree["depth"][u] for u in ends], dtype=np.int32)
    apath = np.full((B, K1), -1, dtype=np.int32)
    for b, u in enumerate(ends):
        p = _path_to(tree, u)
        apath[b, :len(p)] = p
    return ends, alen, apath


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (6, 2)])
def test_commit_gives_path_equivalent_cache(Hq, Hkv):
    rng = np.random.default_rng(Hq * 10 + Hkv)
    B, T, D, Lmax = 3, 23, 16, 64
    tree, x = _case(rng, B, Hq, Hkv, T, D, Lmax, [0, 17, 40])
    ends, alen, apath = _paths(rng, tree, B)
    O, _ = tree_attention(**x, tree=tree, dtype="f32")
    kc, vc, L2, bad = kv_commit(x["k_tree"], x["v_tree"], x["k_cache"], x["v_cache"], x["prefix_len"], alen, apath, tree)
    assert not bad.any()
    np.testing.assert_array_equal(L2, x["prefix_len"] + alen + 1)
    g = Hq // Hkv
    for b, u in enumerate(ends):
        n = int(L2[b])
        for h in range(Hq):
            q = torch.from_numpy(x["q"][b, h, u].astype(np.float64))[None, None, None, :]
            k = torch.from_numpy(kc[b, h // g, :n].astype(np.float64))[None, None]
            v = torch.from_numpy(vc[b, h // g, :n].astype(np.float64))[None, None]
            ref = F.scaled_dot_product_attention(q, k, v)[0, 0, 0].numpy()
            np.testing.assert_allclose(O[b, h, u], ref, rtol=1e-12, atol=1e-12)


def test_copy_is_bit_exact_and_touches_nothing_else():
    rng = np.random.default_rng(5)
    B, Hkv, T, D, Lmax = 4, 3, 30, 8, 50
    parent, rank = wl.random_tree(rng, T, max_children=4)
    tree = tree_encode(parent, rank)
    bits = lambda *s: rng.integers(0, 1 << 16, size=s, dtype=np.uint16)   # arbitrary bf16 patterns
    kt, vt, kc, vc = bits(B, Hkv, T, D), bits(B, Hkv, T, D), bits(B, Hkv, Lmax, D), bits(B, Hkv, Lmax, D)
    L = np.array([0, 5, 49 - tree["max_depth"], 20], dtype=np.int32)
    ends, alen, apath = _paths(rng, tree, B)
    kc2, vc2, L2, bad = kv_commit(kt, vt, kc, vc, L, alen, apath, tree)
    assert not bad.any()
    for b in range(B):
        m, l0 = int(alen[b]), int(L[b])
        for i in range(m + 1):
            assert (kc2[b, :, l0 + i] == kt[b, :, apath[b, i]]).all()
            assert (vc2[b, :, l0 + i] == vt[b, :, apath[b, i]]).all()
        outside = np.r_[0:l0, l0 + m + 1:Lmax]
        assert (kc2[b][:, outside] == kc[b][:, outside]).all()
        assert (vc2[b][:, outside] == vc[b][:, outside]).all()


def test_root_only_and_full_depth():
    parent, rank = wl.chain_tree(6)   # depth 5
    tree = tree_encode(parent, rank)
    kt = np.arange(2 * 1 * 6 * 2, dtype=np.float32).reshape(2, 1, 6, 2)
    kc = np.zeros((2, 1, 10, 2), dtype=np.float32)
    apath = np.array([[0, -1, -1, -1, -1, -1], [0, 1, 2, 3, 4, 5]], dtype=np.int32)
    kc2, _, L2, bad = kv_commit(kt, kt, kc, kc, [3, 4], [0, 5], apath, tree)
    assert not bad.any() and list(L2) == [4, 10]
    assert (kc2[0, 0, 3] == kt[0, 0, 0]).all() and (kc2[0, 0, 4:] == 0).all()
    assert (kc2[1, 0, 4:10] == kt[1, 0, :6]).all()


def test_invalid_sequences_are_left_alone():
    parent, rank = wl.make_tree(("cartesian", (2, 2)))   # root, 2 children, 4 grandchildren
    tree = tree_encode(parent, rank)
    B = 4
    kt = np.ones((B, 2, tree["T"], 4), dtype=np.float32)
    kc = np.zeros((B, 2, 8, 4), dtype=np.float32)
    a = tree["children"][0][0]
    wrong = tree["children"][tree["children"][0][1]][0]   # a grandchild under the other child
    apath = np.array([[0, a, wrong], [1, a, -1], [0, a, -1], [0, -1, -1]], dtype=np.int32)
    alen = np.array([2, 1, 3, 0], dtype=np.int32)   # broken chain, wrong root, m > max_depth, fine
    L = np.array([0, 0, 0, 8], dtype=np.int32)      # the last one would pass Lmax
    kc2, vc2, L2, bad = kv_commit(kt, kt, kc, kc, L, alen, apath, tree)
    assert bad.tolist() == [True, True, True, True]
    assert (kc2 == kc).all() and (L2 == L).all()


# ---- the paged form: the same commit through a block table

def _paged_case(rng, B, Hkv, T, D, bs, max_blocks, prefix):
    """A pool holding every sequence's blocks in a shuffled order (plus spare blocks)."""
    parent, rank = wl.random_tree(rng, T, max_children=3)
    tree = tree_encode(parent, rank)
    num_blocks = B * max_blocks + 3
    order = rng.permutation(num_blocks)
    table = order[:B * max_blocks].reshape(B, max_blocks).astype(np.int32)
    k_pool = rng.standard_normal((num_blocks, Hkv, bs, D)).astype(np.float32)
    v_pool = rng.standard_normal((num_blocks, Hkv, bs, D)).astype(np.float32)
    k_tree = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    v_tree = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    return tree, table, k_pool, v_pool, k_tree, v_tree, np.array(prefix, dtype=np.int32)


@pytest.mark.parametrize("bs", [4, 16])
def test_paged_commit_equals_the_contiguous_commit(bs):
    """Gathering the committed pool gives the contiguous commit of the gathered cache (the
    contiguous commit is pinned above by the path equivalence through torch's SDPA)."""
    from oracle import gather_pages, kv_commit_paged
    rng = np.random.default_rng(bs)
    B, Hkv, T, D, max_blocks = 4, 2, 23, 8, 6
    prefix = [0, bs - 1, 2 * bs + 3, max_blocks * bs - 5]   # the last one crosses no block boundary
    tree, table, kp, vp, kt, vt, plen = _paged_case(rng, B, Hkv, T, D, bs, max_blocks, prefix)
    _, alen, apath = _paths(rng, tree, B)
    alen[-1] = min(int(alen[-1]), 3)        # keep the last sequence inside its capacity
    apath[-1, alen[-1] + 1:] = -1
    full = np.full(B, max_blocks * bs, dtype=np.int32)
    kc = gather_pages(kp, table, bs, full)
    vc = gather_pages(vp, table, bs, full)
    kc2, vc2, L2, bad = kv_commit(kt, vt, kc, vc, plen, alen, apath, tree)
    kp2, vp2, L3, bad3 = kv_commit_paged(kt, vt, kp, vp, table, bs, plen, alen, apath, tree)
    np.testing.assert_array_equal(bad, bad3)
    np.testing.assert_array_equal(L2, L3)
    assert not bad.any()
    np.testing.assert_array_equal(gather_pages(kp2, table, bs, full), kc2)
    np.testing.assert_array_equal(gather_pages(vp2, table, bs, full), vc2)
    # the spare blocks (in no table) are untouched
    spare = np.setdiff1d(np.arange(kp.shape[0]), table.reshape(-1))
    np.testing.assert_array_equal(kp2[spare], kp[spare])
    np.testing.assert_array_equal(vp2[spare], vp[spare])


def test_paged_commit_refusals():
    """A commit past the table's capacity, or into a block outside the pool, leaves the
    sequence unchanged and reports it; a bad entry the commit does not reach is harmless."""
    from oracle import kv_commit_paged
    rng = np.random.default_rng(7)
    B, Hkv, T, D, bs, max_blocks = 3, 1, 15, 4, 8, 3
    tree, table, kp, vp, kt, vt, _ = _paged_case(rng, B, Hkv, T, D, bs, max_blocks, [0, 0, 0])
    ends = [int(np.argmax(tree["depth"]))] * B
    m = int(tree["depth"][ends[0]])
    apath = np.full((B, tree["max_depth"] + 1), -1, dtype=np.int32)
    for b in range(B):
        p = _path_to(tree, ends[b])
        apath[b, :len(p)] = p
    alen = np.full(B, m, dtype=np.int32)
    plen = np.array([max_blocks * bs - m - 1,      # the m + 1 rows exactly fit
                     max_blocks * bs - m,          # one row too many
                     0], dtype=np.int32)
    table[2, 0] = kp.shape[0] + 5                  # sequence 2 writes into block 0: outside the pool
    table[0, 0] = -1                                # sequence 0 does not reach block 0 (m < bs)
    assert m + 1 <= bs
    kp2, vp2, L2, bad = kv_commit_paged(kt, vt, kp, vp, table, bs, plen, alen, apath, tree)
    np.testing.assert_array_equal(bad, [False, True, True])
    np.testing.assert_array_equal(L2, [plen[0] + m + 1, plen[1], plen[2]])
    touched = np.zeros(kp.shape[0], dtype=bool)
    for i in range(m + 1):
        touched[table[0, (plen[0] + i) // bs]] = True
    np.testing.assert_array_equal(kp2[~touched], kp[~touched])
