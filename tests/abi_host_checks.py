"""Host-side refusals of the C-ABI entry points: every call here must fail its
argument checks before anything is queued.  The device addresses passed are
invented and never dereferenced.  tests/test_abi.py runs this file in a child
process that sees no GPU (CUDA_VISIBLE_DEVICES empty); the fixture below
refuses to run it anywhere a GPU is visible."""

import ctypes
import os

import pytest

from conftest import ROOT  # noqa: F401  (puts the repository on sys.path)


@pytest.fixture(scope="module")
def lib():
    assert os.environ.get("CUDA_VISIBLE_DEVICES") == "", "run through tests/test_abi.py (no visible GPU)"
    import __graft_entry__
    __graft_entry__.build()
    from tree_speculative_decoding_spec_gb300 import _binding
    return _binding


# ---------------------------------------------------------------- host-side validation

FAKE = 0x10000   # an aligned, never dereferenced address: these calls fail before any device access


def _build(lib, parent, rank=None, d_bytes=1 << 20, d_buf=FAKE):
    T = len(parent)
    par = (ctypes.c_int32 * max(T, 1))(*parent) if T else (ctypes.c_int32 * 1)(0)
    rk = (ctypes.c_int32 * T)(*rank) if rank is not None else None
    out = lib.spec_tree()
    return lib._lib.spec_tree_build(par, rk, T, ctypes.c_void_p(d_buf), d_bytes, ctypes.byref(out), None)


@pytest.mark.parametrize("parent,rank,code", [
    ([0, 0], None, 2),              # root must have parent -1
    ([-1, 1], None, 2),             # parent[i] < i
    ([-1, 0, 3, 1], None, 2),
    ([-1, 0, 0], [0, 1, 1], 2),     # two siblings share a rank
    ([-1, 0], [0, -1], 2),          # negative rank
    ([], None, 1),                  # empty tree
])
def test_tree_build_rejects_malformed_trees(lib, parent, rank, code):
    assert _build(lib, parent, rank) == code
    assert lib.spec_last_error() != ""


def test_tree_build_rejects_bad_buffers(lib):
    assert _build(lib, [-1, 0], d_buf=0) == 1
    assert _build(lib, [-1, 0], d_buf=FAKE + 4) == 3
    assert _build(lib, [-1, 0], d_bytes=8) == 4
    assert _build(lib, list(range(-1, 1024))) == 1     # 1025 nodes
    deep = list(range(-1, 17))                          # depth 17 chain
    assert _build(lib, deep) == 2


def _fake_tree(lib, parent):
    """A spec_tree with host fields filled as spec_tree_build would and dummy device pointers."""
    import numpy as np
    T = len(parent)
    depth = np.zeros(T, dtype=int)
    kids = np.zeros(T, dtype=int)
    for i in range(1, T):
        depth[i] = depth[parent[i]] + 1
        kids[parent[i]] += 1
    t = lib.spec_tree()
    t.T, t.words, t.max_depth = T, (T + 63) // 64, int(depth.max())
    seen = {}
    for i in range(T):
        t.n_at_depth[depth[i]] += 1
        if kids[i]:
            t.n_internal_at_depth[depth[i]] += 1
            t.n_internal += 1
    for dd in range(lib.SPEC_MAX_DEPTH + 1):
        t.max_rank_at_depth[dd] = -1
    for i in range(1, T):
        r = seen.get(parent[i], 0)
        seen[parent[i]] = r + 1
        t.max_rank_at_depth[depth[i]] = max(t.max_rank_at_depth[depth[i]], r)
    for f in ["parent", "depth", "rank", "anc", "internal", "internal_off", "row_of", "child_off", "child_idx"]:
        setattr(t, f, FAKE)
    return t


def test_workspace_sizes_and_argument_checks(lib):
    import spec_workloads as wl
    parent, _ = wl.cartesian_tree((2, 3))
    t = _fake_tree(lib, [int(x) for x in parent])
    L = lib._lib
    c = (ctypes.c_int32 * 2)(0, 1)
    k = (ctypes.c_int32 * 2)(2, 3)
    assert L.hydra_draft_workspace_size(ctypes.byref(t), 1, 256, 1000, 2, c, k, 0) > 0
    bad_k = (ctypes.c_int32 * 2)(2, 17)
    assert L.hydra_draft_workspace_size(ctypes.byref(t), 1, 256, 1000, 2, c, bad_k, 0) == 0
    small_k = (ctypes.c_int32 * 2)(2, 2)       # a depth-2 node has rank 2
    assert L.hydra_draft_workspace_size(ctypes.byref(t), 1, 256, 1000, 2, c, small_k, 0) == 0
    assert L.hydra_draft_workspace_size(ctypes.byref(t), 1, 250, 1000, 2, c, k, 0) == 0       # d % 8
    assert L.hydra_draft_workspace_size(ctypes.byref(t), 1, 256, 1000, 1, c, k, 0) == 0       # K < depth
    bad_c = (ctypes.c_int32 * 2)(0, 3)
    assert L.hydra_draft_workspace_size(ctypes.byref(t), 1, 256, 1000, 2, bad_c, k, 0) == 0
    assert L.tree_attention_workspace_size(ctypes.byref(t), 1, 4, 4, 128, 64, 0) > 0
    assert L.tree_attention_workspace_size(ctypes.byref(t), 1, 4, 3, 128, 64, 0) == 0         # Hq % Hkv
    assert L.tree_attention_workspace_size(ctypes.byref(t), 1, 4, 4, 128, 96, 0) == 0         # D
    assert L.tree_accept_workspace_size(0, ctypes.byref(t), 1, 1000) > 0
    assert L.tree_accept_workspace_size(2, ctypes.byref(t), 1, 1000) > 0       # typical acceptance
    assert L.tree_accept_workspace_size(3, ctypes.byref(t), 1, 1000) == 0
    assert L.tree_accept_workspace_size(0, ctypes.byref(t), 1, 1) == 0


def test_entry_points_reject_before_launch(lib):
    import spec_workloads as wl
    parent, _ = wl.cartesian_tree((2, 3))
    t = _fake_tree(lib, [int(x) for x in parent])
    L = lib._lib
    vp = ctypes.c_void_p
    # tree_accept: rejection without logits_q; misaligned logits; small workspace
    st = L.tree_accept(1, vp(FAKE), vp(0), vp(FAKE), ctypes.byref(t), 1, 1000, 1.0, 0, 0,
                       vp(FAKE), vp(FAKE), vp(FAKE), vp(0), vp(FAKE), 1 << 30, None)
    assert st == 1
    st = L.tree_accept(0, vp(FAKE + 4), vp(0), vp(FAKE), ctypes.byref(t), 1, 1000, 1.0, 0, 0,
                       vp(FAKE), vp(FAKE), vp(FAKE), vp(0), vp(FAKE), 1 << 30, None)
    assert st == 3
    st = L.tree_accept(0, vp(FAKE), vp(0), vp(FAKE), ctypes.byref(t), 1, 1000, 1.0, 0, 0,
                       vp(FAKE), vp(FAKE), vp(FAKE), vp(0), vp(FAKE), 16, None)
    assert st == 4
    st = L.tree_accept(1, vp(FAKE), vp(FAKE), vp(FAKE), ctypes.byref(t), 1, 1000, 0.0, 0, 0,
                       vp(FAKE), vp(FAKE), vp(FAKE), vp(0), vp(FAKE), 1 << 30, None)
    assert st == 1   # temperature 0
    # tree_attention: bad scale, NULL q
    st = L.tree_attention(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), ctypes.byref(t),
                          1, 4, 4, 128, 64, -1.0, 0, vp(FAKE), vp(0), vp(FAKE), 1 << 30, None)
    assert st == 1
    st = L.tree_attention(vp(0), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), ctypes.byref(t),
                          1, 4, 4, 128, 64, 0.125, 0, vp(FAKE), vp(0), vp(FAKE), 1 << 30, None)
    assert st == 1
    # hydra_draft: NULL weights array entry
    W = (ctypes.c_void_p * 2)(FAKE, 0)
    c = (ctypes.c_int32 * 2)(0, 1)
    k = (ctypes.c_int32 * 2)(2, 3)
    st = L.hydra_draft(vp(FAKE), vp(FAKE), 2, W, None, W, c, k, vp(FAKE), ctypes.byref(t), 1, 256, 1000, 0,
                       vp(FAKE), vp(FAKE), vp(0), vp(FAKE), 1 << 30, None)
    assert st == 1
    # mode 2 goes through tree_accept_typical; typical with a negative epsilon
    st = L.tree_accept(2, vp(FAKE), vp(0), vp(FAKE), ctypes.byref(t), 1, 1000, 1.0, 0, 0,
                       vp(FAKE), vp(FAKE), vp(FAKE), vp(0), vp(FAKE), 1 << 30, None)
    assert st == 1
    st = L.tree_accept_typical(vp(FAKE), vp(FAKE), ctypes.byref(t), 1, 1000, 1.0, -0.1, 0.3, 0, 0,
                               vp(FAKE), vp(FAKE), vp(FAKE), vp(0), vp(FAKE), 1 << 30, None)
    assert st == 1
    # a tree struct that was never built
    empty = lib.spec_tree()
    st = L.tree_accept(0, vp(FAKE), vp(0), vp(FAKE), ctypes.byref(empty), 1, 1000, 1.0, 0, 0,
                       vp(FAKE), vp(FAKE), vp(FAKE), vp(0), vp(FAKE), 1 << 30, None)
    assert st == 1


def test_fold_entries_reject_before_launch(lib):
    # every call here fails a host check, so nothing is queued (no device access)
    import spec_workloads as wl
    L = lib._lib
    vp = ctypes.c_void_p
    assert L.hydra_fold_table_bytes(4096, 32000) == 4096 * 32000 * 4
    assert L.hydra_fold_table_bytes(4092, 32000) == 0     # d % 8
    assert L.hydra_fold_table_bytes(256, 1) == 0          # V
    assert L.hydra_fold_embedding(vp(FAKE), vp(FAKE), 250, 1000, 0, vp(FAKE), None) == 1
    assert L.hydra_fold_embedding(vp(FAKE), vp(FAKE), 256, 1, 0, vp(FAKE), None) == 1
    assert L.hydra_fold_embedding(vp(0), vp(FAKE), 256, 1000, 0, vp(FAKE), None) == 1
    assert L.hydra_fold_embedding(vp(FAKE), vp(FAKE), 256, 1000, 7, vp(FAKE), None) == 1   # dtype
    assert L.hydra_fold_embedding(vp(FAKE), vp(FAKE), 256, 1000, 0, vp(FAKE + 4), None) == 3
    assert L.hydra_fold_embedding(vp(FAKE + 8), vp(FAKE), 256, 1000, 1, vp(FAKE), None) == 3
    # hydra_draft_folded: a misaligned table is refused after the other checks pass
    parent, _ = wl.cartesian_tree((2, 3))
    t = _fake_tree(lib, [int(x) for x in parent])
    W = (ctypes.c_void_p * 2)(FAKE, FAKE)
    tab = (ctypes.c_void_p * 2)(0, FAKE + 4)
    c = (ctypes.c_int32 * 2)(1, 1)
    k = (ctypes.c_int32 * 2)(2, 3)
    st = L.hydra_draft_folded(vp(FAKE), vp(FAKE), 2, W, None, W, tab, c, k, vp(FAKE), ctypes.byref(t), 1, 256, 1000, 1,
                              vp(FAKE), vp(FAKE), vp(0), vp(FAKE), 1 << 30, None)
    assert st == 3 and "folded table 1" in lib.spec_last_error()
    W0 = (ctypes.c_void_p * 2)(FAKE, 0)
    st = L.hydra_draft_folded(vp(FAKE), vp(FAKE), 2, W0, None, W, tab, c, k, vp(FAKE), ctypes.byref(t), 1, 256, 1000, 1,
                              vp(FAKE), vp(FAKE), vp(0), vp(FAKE), 1 << 30, None)
    assert st == 1


def test_kv_commit_rejects_before_launch(lib):
    # every call here fails a host check, so nothing is queued (no device access)
    import spec_workloads as wl
    parent, _ = wl.cartesian_tree((2, 3))
    t = _fake_tree(lib, [int(x) for x in parent])
    L = lib._lib
    vp = ctypes.c_void_p
    assert L.tree_kv_commit_workspace_size() == 256

    def call(k_tree=FAKE, k_cache=FAKE, D=64, dt=1, ws_bytes=256, B=1, tree=t):
        return L.tree_kv_commit(vp(k_tree), vp(FAKE), vp(k_cache), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                ctypes.byref(tree), B, 4, 128, D, dt, vp(FAKE), ws_bytes, None)
    assert call(k_tree=0) == 1                 # NULL buffer
    assert call(k_cache=FAKE + 4) == 3         # misaligned cache
    assert call(D=4) == 1                      # 8-byte rows (bf16): not 16-byte chunks
    assert call(ws_bytes=16) == 4              # workspace below its size
    assert call(dt=7) == 5                     # dtype
    assert call(B=0) == 1
    assert call(tree=lib.spec_tree()) == 1     # a tree that was never built




def test_kv_commit_paged_rejects_before_launch(lib):
    # every call here fails a host check, so nothing is queued (no device access)
    import spec_workloads as wl
    parent, _ = wl.cartesian_tree((2, 3))
    t = _fake_tree(lib, [int(x) for x in parent])
    L = lib._lib
    vp = ctypes.c_void_p

    def call(k_pool=FAKE, table=FAKE, num_blocks=8, max_blocks=4, bs=64, D=64, dt=1, ws_bytes=256):
        return L.tree_kv_commit_paged(vp(FAKE), vp(FAKE), vp(k_pool), vp(FAKE), num_blocks, vp(table), max_blocks, bs,
                                      vp(FAKE), vp(FAKE), vp(FAKE), ctypes.byref(t), 1, 4, D, dt, vp(FAKE), ws_bytes,
                                      None)
    assert call(table=0) == 1                  # no block table
    assert call(num_blocks=0) == 1
    assert call(bs=0) == 1
    assert call(max_blocks=1 << 16, bs=128) == 1   # more than 2^22 positions
    assert call(k_pool=0) == 1                 # NULL pool
    assert call(k_pool=FAKE + 4) == 3          # misaligned pool
    assert call(table=FAKE + 2) == 3           # misaligned table
    assert call(D=4) == 1                      # 8-byte rows
    assert call(ws_bytes=16) == 4
    assert call(dt=7) == 5
