"""KV commit of the accepted path: CUDA path vs the oracle (GPU).

A copy, so the caches and prefix_len must match bit for bit.  Also chained
behind tree_accept (its outputs feed the commit directly), at the Vicuna-7B
layer shape, with invalid sequences (left unchanged, SPEC_EINVAL in the status
word), and the path equivalence through the library's own tree_attention.
"""

import numpy as np
import pytest

import oracle
import spec_workloads as wl
from gpu_util import assert_close, lib, to_dev

pytestmark = pytest.mark.gpu


def _path_to(parent, u):
    path = [u]
    while path[-1] != 0:
        path.append(int(parent[path[-1]]))
    return path[::-1]


def _paths(rng, parent, max_depth, B):
    depth = wl.tree_depths(parent)
    ends = [int(rng.integers(0, len(parent))) for _ in range(B)]
    alen = np.array([depth[u] for u in ends], dtype=np.int32)
    apath = np.full((B, max_depth + 1), -1, dtype=np.int32)
    for b, u in enumerate(ends):
        p = _path_to(parent, u)
        apath[b, :len(p)] = p
    return ends, alen, apath


def _bits(rng, dtype, *shape):
    if dtype == "bf16":
        return rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)   # any bit pattern: it is a copy
    return rng.standard_normal(shape).astype(np.float32)


def _commit(st, kt, vt, kc, vc, L, alen, apath, tree):
    kc_d, vc_d, L_d = to_dev(kc), to_dev(vc), to_dev(L)
    ws = st.tree_kv_commit(to_dev(kt), to_dev(vt), kc_d, vc_d, L_d, to_dev(alen), to_dev(apath), tree)
    status = st.spec_read_device_status(ws)
    host = lambda t: t.cpu().view(__import__("torch").int16).numpy().view(np.uint16) if t.dtype.itemsize == 2 \
        else t.cpu().numpy()
    return host(kc_d), host(vc_d), L_d.cpu().numpy(), status


CASES = [
    # dtype, B, Hkv, T (random tree), D, Lmax
    ("bf16", 3, 4, 40, 128, 300),
    ("f32", 2, 2, 17, 64, 100),
    ("bf16", 5, 1, 130, 64, 400),    # deep random tree, one KV head
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-B{c[1]}-H{c[2]}-T{c[3]}" for c in CASES])
def test_commit_matches_oracle(case):
    st = lib()
    dtype, B, Hkv, T, D, Lmax = case
    rng = np.random.default_rng(T * 7 + B)
    parent, rank = wl.random_tree(rng, T, max_children=3)
    tree_h = oracle.tree_encode(parent, rank)
    tree = st.spec_tree_build(parent, rank)
    kt, vt = _bits(rng, dtype, B, Hkv, T, D), _bits(rng, dtype, B, Hkv, T, D)
    kc, vc = _bits(rng, dtype, B, Hkv, Lmax, D), _bits(rng, dtype, B, Hkv, Lmax, D)
    L = rng.integers(0, Lmax - tree_h["max_depth"], size=B).astype(np.int32)
    _, alen, apath = _paths(rng, parent, tree_h["max_depth"], B)
    got_k, got_v, got_L, status = _commit(st, kt, vt, kc, vc, L, alen, apath, tree)
    ref_k, ref_v, ref_L, bad = oracle.kv_commit(kt, vt, kc, vc, L, alen, apath, tree_h)
    assert status == 0 and not bad.any()
    np.testing.assert_array_equal(got_L, ref_L)
    np.testing.assert_array_equal(got_k, ref_k)
    np.testing.assert_array_equal(got_v, ref_v)


def test_commit_after_tree_accept_vicuna7b_shape():
    st = lib()
    w = wl.WORKLOADS[2]
    parent, rank = wl.make_tree(w.tree)
    tree_h = oracle.tree_encode(parent, rank)
    tree = st.spec_tree_build(parent, rank)
    B, Hkv, D, Lmax, T = 2, w.Hkv, w.D, w.Lmax, len(parent)
    rng = np.random.default_rng(77)
    g = wl.greedy_inputs(w, parent, B=B)
    a, p, n, m = st.tree_accept(0, to_dev(g["logits_p"]), None, to_dev(g["node_tok"]), tree)
    alen, apath = a.cpu().numpy(), p.cpu().numpy()
    kt, vt = _bits(rng, "bf16", B, Hkv, T, D), _bits(rng, "bf16", B, Hkv, T, D)
    kc, vc = _bits(rng, "bf16", B, Hkv, Lmax, D), _bits(rng, "bf16", B, Hkv, Lmax, D)
    L = np.array([Lmax - T, 100], dtype=np.int32)
    got_k, got_v, got_L, status = _commit(st, kt, vt, kc, vc, L, alen, apath, tree)
    ref_k, ref_v, ref_L, bad = oracle.kv_commit(kt, vt, kc, vc, L, alen, apath, tree_h)
    ref_len = oracle.greedy_accept(g["logits_p"], g["node_tok"], tree_h)["accept_len"]
    assert list(alen) == list(ref_len) and status == 0 and not bad.any()
    np.testing.assert_array_equal(got_L, ref_L)
    np.testing.assert_array_equal(got_k, ref_k)
    np.testing.assert_array_equal(got_v, ref_v)


def test_invalid_sequences_are_left_unchanged():
    st = lib()
    parent, rank = wl.make_tree(("cartesian", (2, 2)))
    tree_h = oracle.tree_encode(parent, rank)
    tree = st.spec_tree_build(parent, rank)
    rng = np.random.default_rng(3)
    B, Hkv, T, D, Lmax = 5, 2, len(parent), 64, 16
    a = tree_h["children"][0][0]
    wrong = tree_h["children"][tree_h["children"][0][1]][0]
    apath = np.array([[0, a, wrong], [1, a, -1], [0, a, -1], [0, -1, -1], [0, a, -1]], dtype=np.int32)
    alen = np.array([2, 1, 3, 0, 1], dtype=np.int32)    # broken chain, wrong root, m > max depth, overflow, fine
    L = np.array([0, 0, 0, Lmax, 3], dtype=np.int32)
    kt, vt = _bits(rng, "bf16", B, Hkv, T, D), _bits(rng, "bf16", B, Hkv, T, D)
    kc, vc = _bits(rng, "bf16", B, Hkv, Lmax, D), _bits(rng, "bf16", B, Hkv, Lmax, D)
    got_k, got_v, got_L, status = _commit(st, kt, vt, kc, vc, L, alen, apath, tree)
    ref_k, ref_v, ref_L, bad = oracle.kv_commit(kt, vt, kc, vc, L, alen, apath, tree_h)
    assert bad.tolist() == [True, True, True, True, False]
    assert status == 1    # SPEC_EINVAL in the status word
    np.testing.assert_array_equal(got_L, ref_L)
    np.testing.assert_array_equal(got_k, ref_k)
    np.testing.assert_array_equal(got_v, ref_v)


def test_committed_cache_reproduces_tree_attention():
    # path equivalence through the library: the accepted node's tree attention
    # before the commit equals a one-node attention over the committed cache
    import torch
    st = lib()
    rng = np.random.default_rng(11)
    parent, rank = wl.random_tree(rng, 30, max_children=3)
    tree_h = oracle.tree_encode(parent, rank)
    tree = st.spec_tree_build(parent, rank)
    root_only = st.spec_tree_build(np.array([-1]), np.array([0]))
    B, Hq, Hkv, T, D, Lmax = 2, 8, 4, len(parent), 128, 256
    x = {k: v for k, v in wl.attention_inputs(wl.Workload("t", "bf16", B=B, seed=11, tree=None, Hq=Hq, Hkv=Hkv,
                                                                      D=D, Lmax=Lmax, prefix=(60, 200)), T).items()}
    ends, alen, apath = _paths(rng, parent, tree_h["max_depth"], B)
    dev = {k: to_dev(v) for k, v in x.items()}
    out, _ = st.tree_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["prefix_len"], dev["k_tree"],
                               dev["v_tree"], tree)
    st.tree_kv_commit(dev["k_tree"], dev["v_tree"], dev["k_cache"], dev["v_cache"], dev["prefix_len"],
                      to_dev(alen), to_dev(apath), tree)
    newL = dev["prefix_len"].cpu().numpy()
    for b, u in enumerate(ends):
        # one-node tree: its query is u's, its own key/value the last committed row
        n = int(newL[b])
        q1 = dev["q"][b:b + 1, :, u:u + 1].contiguous()
        k1 = dev["k_cache"][b:b + 1, :, n - 1:n].contiguous()
        v1 = dev["v_cache"][b:b + 1, :, n - 1:n].contiguous()
        L1 = torch.tensor([n - 1], dtype=torch.int32, device="cuda")
        o1, _ = st.tree_attention(q1, dev["k_cache"][b:b + 1].contiguous(), dev["v_cache"][b:b + 1].contiguous(),
                                  L1, k1, v1, root_only)
        assert_close(o1[0, :, 0].float().cpu().numpy(), out[b, :, u].float().cpu().numpy(), "bf16", "path equivalence")


# ---- the paged form

def _commit_paged(st, kt, vt, kp, vp, table, bs, L, alen, apath, tree):
    import torch
    kp_d, vp_d, L_d = to_dev(kp), to_dev(vp), to_dev(L)
    ws = st.tree_kv_commit_paged(to_dev(kt), to_dev(vt), kp_d, vp_d, to_dev(table), bs, L_d, to_dev(alen),
                                 to_dev(apath), tree)
    status = st.spec_read_device_status(ws)
    host = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16) if t.dtype.itemsize == 2 else t.cpu().numpy()
    return host(kp_d), host(vp_d), L_d.cpu().numpy(), status


PAGED = [
    # dtype, B, Hkv, T (random tree), D, block_size, max_blocks
    ("bf16", 4, 4, 40, 128, 64, 5),
    ("f32", 3, 2, 17, 64, 16, 6),
    ("bf16", 6, 1, 90, 64, 7, 9),    # a block size that is no power of two: commits cross blocks
]


@pytest.mark.parametrize("case", PAGED, ids=[f"{c[0]}-B{c[1]}-bs{c[5]}" for c in PAGED])
def test_paged_commit_matches_oracle(case):
    st = lib()
    dtype, B, Hkv, T, D, bs, max_blocks = case
    rng = np.random.default_rng(T * 11 + bs)
    parent, rank = wl.random_tree(rng, T, max_children=3)
    tree_h = oracle.tree_encode(parent, rank)
    tree = st.spec_tree_build(parent, rank)
    num_blocks = B * max_blocks + 2
    table = rng.permutation(num_blocks)[:B * max_blocks].reshape(B, max_blocks).astype(np.int32)
    kt, vt = _bits(rng, dtype, B, Hkv, T, D), _bits(rng, dtype, B, Hkv, T, D)
    kp, vp = _bits(rng, dtype, num_blocks, Hkv, bs, D), _bits(rng, dtype, num_blocks, Hkv, bs, D)
    _, alen, apath = _paths(rng, parent, tree_h["max_depth"], B)
    L = np.array([rng.integers(0, max_blocks * bs - int(alen[b])) for b in range(B)], dtype=np.int32)
    got_k, got_v, got_L, status = _commit_paged(st, kt, vt, kp, vp, table, bs, L, alen, apath, tree)
    ref_k, ref_v, ref_L, bad = oracle.kv_commit_paged(kt, vt, kp, vp, table, bs, L, alen, apath, tree_h)
    assert status == 0 and not bad.any()
    np.testing.assert_array_equal(got_L, ref_L)
    np.testing.assert_array_equal(got_k, ref_k)
    np.testing.assert_array_equal(got_v, ref_v)


def test_paged_commit_refusals_leave_the_pool_alone():
    """Capacity overflow and a block outside the pool: those sequences unchanged, SPEC_EINVAL in
    the status word; a valid sequence beside them commits."""
    st = lib()
    rng = np.random.default_rng(5)
    B, Hkv, T, D, bs, max_blocks = 3, 2, 20, 64, 16, 3
    parent, rank = wl.random_tree(rng, T, max_children=3)
    tree_h = oracle.tree_encode(parent, rank)
    tree = st.spec_tree_build(parent, rank)
    num_blocks = B * max_blocks
    table = rng.permutation(num_blocks).reshape(B, max_blocks).astype(np.int32)
    u = int(np.argmax(tree_h["depth"]))
    m = int(tree_h["depth"][u])
    p = _path_to(parent, u)
    apath = np.full((B, tree_h["max_depth"] + 1), -1, dtype=np.int32)
    apath[:, :len(p)] = p
    alen = np.full(B, m, dtype=np.int32)
    L = np.array([0, max_blocks * bs - m, 0], dtype=np.int32)    # sequence 1: one row past capacity
    table[2, 0] = num_blocks + 3                                  # sequence 2: a block outside the pool
    kt, vt = _bits(rng, "f32", B, Hkv, T, D), _bits(rng, "f32", B, Hkv, T, D)
    kp, vp = _bits(rng, "f32", num_blocks, Hkv, bs, D), _bits(rng, "f32", num_blocks, Hkv, bs, D)
    got_k, got_v, got_L, status = _commit_paged(st, kt, vt, kp, vp, table, bs, L, alen, apath, tree)
    ref_k, ref_v, ref_L, bad = oracle.kv_commit_paged(kt, vt, kp, vp, table, bs, L, alen, apath, tree_h)
    assert list(bad) == [False, True, True]
    assert status == 1   # SPEC_EINVAL
    np.testing.assert_array_equal(got_L, ref_L)
    np.testing.assert_array_equal(got_k, ref_k)
    np.testing.assert_array_equal(got_v, ref_v)


def test_paged_commit_then_paged_attention_is_path_equivalent():
    """After committing the accepted node's path into the pool, the library's paged tree attention
    of a one-node tree (the accepted node's query) over the grown prefix equals that node's tree
    attention before the commit (Hydra Guide, "Tree Attention Matrix with Topology-Aware Causal
    Masking": a node attends exactly to its prefix and its ancestors)."""
    import torch
    st = lib()
    rng = np.random.default_rng(12)
    B, Hq, Hkv, T, D, bs, max_blocks = 2, 4, 2, 30, 64, 64, 4
    parent, rank = wl.random_tree(rng, T, max_children=3)
    tree_h = oracle.tree_encode(parent, rank)
    tree = st.spec_tree_build(parent, rank)
    num_blocks = B * max_blocks
    table = rng.permutation(num_blocks).reshape(B, max_blocks).astype(np.int32)
    q = rng.standard_normal((B, Hq, T, D)).astype(np.float32)
    kt, vt = _bits(rng, "f32", B, Hkv, T, D), _bits(rng, "f32", B, Hkv, T, D)
    kp, vp = _bits(rng, "f32", num_blocks, Hkv, bs, D), _bits(rng, "f32", num_blocks, Hkv, bs, D)
    L = np.array([70, 133], dtype=np.int32)
    ends, alen, apath = _paths(rng, parent, tree_h["max_depth"], B)
    out0, _ = st.tree_attention_paged(to_dev(q), to_dev(kp), to_dev(vp), to_dev(table), to_dev(L), to_dev(kt), to_dev(vt),
                                      tree)
    kp_d, vp_d, L_d = to_dev(kp), to_dev(vp), to_dev(L)
    ws = st.tree_kv_commit_paged(to_dev(kt), to_dev(vt), kp_d, vp_d, to_dev(table), bs, L_d, to_dev(alen),
                                 to_dev(apath), tree)
    assert st.spec_read_device_status(ws) == 0
    # a one-node tree: the accepted node's query over the committed prefix (its own row included)
    one = st.spec_tree_build(np.array([-1], dtype=np.int32), np.array([0], dtype=np.int32))
    for b in range(B):
        qb = torch.from_numpy(np.ascontiguousarray(q[b:b + 1, :, ends[b]:ends[b] + 1])).cuda()
        kt1 = torch.from_numpy(np.ascontiguousarray(kt[b:b + 1, :, ends[b]:ends[b] + 1])).cuda()
        vt1 = torch.from_numpy(np.ascontiguousarray(vt[b:b + 1, :, ends[b]:ends[b] + 1])).cuda()
        # the committed rows hold the node itself at position L + m: drop it from the prefix and let
        # the one-node tree supply it
        Lb = (L_d[b:b + 1] - 1).contiguous()
        out1, _ = st.tree_attention_paged(qb, kp_d, vp_d, to_dev(table[b:b + 1]), Lb, kt1, vt1, one)
        assert_close(out1[0, :, 0].cpu().numpy(), out0[b, :, ends[b]].cpu().numpy(), "f32", f"seq {b}")
