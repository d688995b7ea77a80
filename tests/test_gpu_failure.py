"""Failure detection without a GPU fault (GPU).

Kernels never trap or wait without bound: a wait that runs out records
SPEC_ETIMEOUT in the workspace status word and the kernel returns, leaving the
context usable.  Host-side checks reject bad calls before anything is queued
and leave the outputs untouched.
"""

import numpy as np
import pytest
import torch

import oracle
import spec_workloads as wl
from gpu_util import assert_close, lib, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    st = lib()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    st.spec_selftest_timeout(ws, limit_ns=2_000_000)          # nothing ever completes the barrier
    assert st.spec_read_device_status(ws) == 7                 # SPEC_ETIMEOUT
    # the context is still usable: a normal call runs and matches the oracle
    rng = np.random.default_rng(1)
    parent, rank = wl.cartesian_tree((2, 2))
    tree = st.spec_tree_build(parent, rank)
    x = {k: rng.standard_normal(s, dtype=np.float32) for k, s in
         [("q", (1, 2, 7, 64)), ("k_cache", (1, 2, 40, 64)), ("v_cache", (1, 2, 40, 64)),
          ("k_tree", (1, 2, 7, 64)), ("v_tree", (1, 2, 7, 64))]}
    x["prefix_len"] = np.array([33], dtype=np.int32)
    out, _ = st.tree_attention(to_dev(x["q"]), to_dev(x["k_cache"]), to_dev(x["v_cache"]), to_dev(x["prefix_len"]),
                               to_dev(x["k_tree"]), to_dev(x["v_tree"]), tree)
    O, _ = oracle.tree_attention(**x, tree=oracle.tree_encode(parent, rank), dtype="f32")
    assert_close(out.cpu().numpy(), O, "f32", "out")


def test_status_word_is_clean_after_normal_calls():
    st = lib()
    parent, rank = wl.cartesian_tree((2, 3))
    tree = st.spec_tree_build(parent, rank)
    rng = np.random.default_rng(2)
    lp = rng.standard_normal((2, len(parent), 50), dtype=np.float32)
    tok = wl.sibling_tokens(rng, parent, 2, 50)
    ws = torch.zeros(st.tree_accept_workspace_size(1, tree, 2, 50), dtype=torch.uint8, device="cuda")
    st.tree_accept(1, to_dev(lp), to_dev(lp), to_dev(tok), tree, temperature=0.9, ws=ws)
    assert st.spec_read_device_status(ws) == 0


def test_small_workspace_is_refused_and_outputs_untouched():
    st = lib()
    parent, rank = wl.cartesian_tree((2, 3))
    tree = st.spec_tree_build(parent, rank)
    B, T, V = 2, len(parent), 64
    lp = to_dev(np.zeros((B, T, V), dtype=np.float32))
    tok = to_dev(np.zeros((B, T), dtype=np.int32))
    alen = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    apath = torch.full((B, tree.max_depth + 1), -7, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(st.SpecError) as e:
        st.tree_accept(0, lp, None, tok, tree, accept_len=alen, accept_path=apath, next_token=nxt, ws=small)
    assert e.value.status == 4   # SPEC_EWORKSPACE
    torch.cuda.synchronize()
    assert (alen == -7).all() and (apath == -7).all() and (nxt == -7).all()


def test_misaligned_pointer_is_refused():
    st = lib()
    parent, rank = wl.cartesian_tree((2,))
    tree = st.spec_tree_build(parent, rank)
    B, T, V = 1, len(parent), 32
    flat = torch.zeros(B * T * V + 1, dtype=torch.float32, device="cuda")
    lp = flat[1:].view(B, T, V)                      # 4 bytes past a 256-byte boundary
    tok = to_dev(np.zeros((B, T), dtype=np.int32))
    with pytest.raises(st.SpecError) as e:
        st.tree_accept(0, lp, None, tok, tree)
    assert e.value.status == 3   # SPEC_EALIGN


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_accept_status_is_cleared_by_each_call(mode):
    # the rows kernel clears the status word itself: a workspace whose header holds garbage,
    # then a call that flags, then a clean call on the same workspace
    st = lib()
    parent, rank = wl.chain_tree(3)
    tree = st.spec_tree_build(parent, rank)
    V = 16
    lp = np.zeros((1, 3, V), dtype=np.float32)
    bad = np.array([[0, 99, 1]], dtype=np.int32)
    good = np.array([[0, 3, 1]], dtype=np.int32)
    ws = torch.full((st.tree_accept_workspace_size(mode, tree, 1, V),), 0x7F, dtype=torch.uint8, device="cuda")

    def call(tok):
        if mode == 2:
            st.tree_accept_typical(to_dev(lp), to_dev(tok), tree, temperature=1.0, epsilon=0.3, alpha=0.09, ws=ws)
        else:
            st.tree_accept(mode, to_dev(lp), to_dev(lp) if mode == 1 else None, to_dev(tok), tree, temperature=1.0,
                           ws=ws)

    call(good)
    assert st.spec_read_device_status(ws) == 0
    if mode != 0:   # the greedy walk compares tokens without indexing by them: nothing to flag
        call(bad)
        assert st.spec_read_device_status(ws) == 1
    call(good)
    assert st.spec_read_device_status(ws) == 0


def test_draft_status_is_cleared_by_each_call():
    # the root kernel clears the status word itself and flags an out-of-vocabulary root token
    st = lib()
    w = wl.Workload("t", "bf16", B=3, seed=5, tree=("cartesian", (3, 2)), d=64, V=500, cond=(1, 1), topk=(3, 2))
    parent, rank = wl.make_tree(w.tree)
    tree = st.spec_tree_build(parent, rank)
    x = wl.draft_inputs(w)
    args = (to_dev(x["h"]), to_dev(x["E"]), [to_dev(a) for a in x["W1"]], [to_dev(a) for a in x["b1"]],
            [to_dev(a) for a in x["W2"]], list(x["cond"]), list(x["topk"]))
    ws = torch.full((st.hydra_draft_workspace_size(tree, 3, 64, 500, [1, 1], [3, 2], 1),), 0x7F, dtype=torch.uint8,
                    device="cuda")
    good = to_dev(np.array([1, 2, 3], dtype=np.int32))
    bad = to_dev(np.array([1, 500, 3], dtype=np.int32))
    for folded in (False, True):
        tabs = [st.hydra_fold_embedding(W, args[1]) for W in args[2]] if folded else None
        st.hydra_draft(*args, good, tree, ws=ws, folded=tabs)
        assert st.spec_read_device_status(ws) == 0
        tok, _, _ = st.hydra_draft(*args, bad, tree, ws=ws, folded=tabs)
        assert st.spec_read_device_status(ws) == 1
        assert tok.cpu().numpy()[1, 0] == 499        # clamped into the vocabulary
        st.hydra_draft(*args, good, tree, ws=ws, folded=tabs)
        assert st.spec_read_device_status(ws) == 0
