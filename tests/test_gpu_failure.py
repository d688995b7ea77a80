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
