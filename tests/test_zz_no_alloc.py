"""tree_attention_noalloc against tree_attention (GPU).

tree_attention_noalloc is for callers that cannot allocate device memory --
for instance a plugin inside a host engine that forbids further cudaMalloc
calls -- and uses the library's built-in scratch array instead of a caller
workspace.  Its results must equal those of tree_attention with a workspace,
on two calls in a row (the array keeps the previous call's contents), and
shapes that need more scratch than the array holds must be refused before
anything runs.  This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest

import spec_workloads as wl
from gpu_util import assert_close, lib, to_dev

pytestmark = pytest.mark.gpu


def _case(seed, dtype, B, Hq, Hkv, branching, D, Lmax, prefix):
    rng = np.random.default_rng(seed)
    parent, rank = wl.cartesian_tree(branching) if branching != "sparse" else wl.make_tree(("sparse", (8, 4, 2, 1), 64, 64))
    T = len(parent)
    enc = wl.f32_to_bf16_bits if dtype == "bf16" else (lambda a: a)
    n = lambda *s: to_dev(enc(rng.standard_normal(s, dtype=np.float32)))
    args = (n(B, Hq, T, D), n(B, Hkv, Lmax, D), n(B, Hkv, Lmax, D), to_dev(np.array(prefix, dtype=np.int32)),
            n(B, Hkv, T, D), n(B, Hkv, T, D))
    return parent, rank, args


def test_noalloc_matches_workspace_call_on_two_calls_in_a_row():
    st = lib()
    cases = [
        # the Vicuna-7B-shaped layer: bf16, 32 x 128 heads, prefix 1024, 64-node sparse tree
        (21, "bf16", 1, 32, 32, "sparse", 128, 1024, [1024]),
        # then a smaller, different one: fp32, grouped heads, ragged prefixes
        (22, "f32", 2, 8, 2, (3, 2), 64, 200, [200, 37]),
    ]
    prepared = []
    for seed, dtype, B, Hq, Hkv, br, D, Lmax, prefix in cases:
        parent, rank, args = _case(seed, dtype, B, Hq, Hkv, br, D, Lmax, prefix)
        tree = st.spec_tree_build(parent, rank)
        ref_out, ref_lse = st.tree_attention(*args, tree)
        prepared.append((dtype, tree, args, ref_out.cpu().numpy(), ref_lse.cpu().numpy()))
    results = [st.tree_attention_noalloc(*args, tree) for _, tree, args, _, _ in prepared]   # two calls in a row
    assert st.tree_attention_noalloc_status() == 0    # no failure recorded in the built-in array's status word
    for (dtype, _, _, ref_out, ref_lse), (out, lse) in zip(prepared, results):
        assert_close(out.cpu().numpy(), ref_out, dtype, "out")
        assert_close(lse.cpu().numpy(), ref_lse, dtype, "lse")


def test_noalloc_refuses_shapes_beyond_its_scratch():
    st = lib()
    from tree_speculative_decoding_spec_gb300 import _binding as b
    parent, rank = wl.cartesian_tree((4, 4, 4, 4))
    tree = st.spec_tree_build(parent, rank)
    # NULL tensors: the size check must refuse first; were it to let the call through, the
    # pointer check behind it would still stop it on the host (SPEC_EINVAL), with nothing queued
    null = ctypes.c_void_p(0)
    status = b._lib.tree_attention_noalloc(null, null, null, null, null, null, tree.ref(), 8, 64, 8, 32768, 128,
                                           0.088, 1, null, null, None)
    assert status == 4   # SPEC_EWORKSPACE
    assert "built-in" in b.spec_last_error()
