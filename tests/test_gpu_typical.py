"""Typical acceptance: CUDA path vs the oracle (GPU).

Accepted lengths, paths and extra tokens must match the oracle except where the
oracle's margin shows a decision within a relative 1e-4 of its threshold
(|p / threshold - 1|), or the draw within 1e-6 of a CDF breakpoint: fp32
probabilities and entropies over 32000 tokens carry relative errors near 1e-6.
Such cases are counted.
"""

import numpy as np
import pytest

import oracle
import spec_workloads as wl
from oracle.philox import acceptance_uniforms
from gpu_util import lib, to_dev

pytestmark = pytest.mark.gpu


def _compare(st, lp, tok, parent, rank, temp, eps, alpha, seed, offset):
    tree = st.spec_tree_build(parent, rank)
    a, p, n, m = st.tree_accept_typical(to_dev(lp), to_dev(tok), tree, temperature=temp, epsilon=eps, alpha=alpha,
                                        seed=seed, offset=offset)
    a, p, n = a.cpu().numpy(), p.cpu().numpy(), n.cpu().numpy()
    B, T, _ = lp.shape
    _, us = acceptance_uniforms(seed, offset, B, T)
    ref = oracle.typical_accept(lp, tok, oracle.tree_encode(parent, rank), temp, eps, alpha, us)
    near = 0
    for b in range(B):
        if ref["margin_decide"][b] < 1e-4:
            near += 1
            continue
        assert a[b] == ref["accept_len"][b], b
        assert np.array_equal(p[b], ref["accept_path"][b]), b
        if ref["margin_sample"][b] < 1e-6:
            near += 1
            continue
        assert n[b] == ref["next_token"][b], (b, n[b], ref["next_token"][b])
    return near, a


def test_typical_long_context_workload():
    st = lib()
    w = wl.WORKLOADS[5]
    parent, rank = wl.make_tree(w.tree)
    x = wl.rejection_inputs(w, parent, rank)
    near_total, lens = 0, []
    for offset in range(8):
        near, a = _compare(st, x["logits_p"], x["node_tok"], parent, rank, w.temperature, 0.09, 0.3, w.philox_seed,
                           offset)
        near_total += near
        lens.append(int(a[0]))
    assert near_total <= 1
    print(f"long-context typical acceptance: lengths {lens}")


@pytest.mark.parametrize("V,temp,eps,alpha", [(7, 1.0, 0.09, 0.3), (50, 0.7, 0.2, 0.5), (1000, 1.3, 0.05, 0.3),
                                               (1000, 0.5, 0.3, 10.0)])
def test_typical_random_trees(V, temp, eps, alpha):
    st = lib()
    rng = np.random.default_rng(V + int(100 * temp))
    for trial in range(3):
        T = int(rng.integers(2, 120))
        parent, rank = wl.random_tree(rng, T, max_children=3)
        B = 64
        lp = (rng.standard_normal((B, T, V), dtype=np.float32) * np.float32(2.0)).astype(np.float32)
        tok = wl.sibling_tokens(rng, parent, B, V) if V >= 4 else rng.integers(0, V, size=(B, T)).astype(np.int32)
        # raise some node tokens so that paths go deep
        for b in range(B):
            for c in range(1, T):
                if rng.random() < 0.5:
                    lp[b, parent[c], tok[b, c]] = lp[b, parent[c]].max() + np.float32(rng.random())
        near, _ = _compare(st, lp, tok, parent, rank, temp, eps, alpha, 7 + trial, trial)
        assert near <= 2


def test_typical_low_temperature_is_greedy():
    st = lib()
    rng = np.random.default_rng(3)
    parent, rank = wl.make_tree(("sparse", (8, 4, 2, 1), 64, 64))
    B, T, V = 16, len(parent), 2000
    lp = rng.standard_normal((B, T, V), dtype=np.float32)
    tok = wl.sibling_tokens(rng, parent, B, V)
    for b in range(B):
        for c in range(1, T):
            if rng.random() < 0.6:
                lp[b, parent[c], tok[b, c]] = lp[b, parent[c]].max() + np.float32(0.5)
    tree = st.spec_tree_build(parent, rank)
    a, p, n, _ = st.tree_accept_typical(to_dev(lp), to_dev(tok), tree, temperature=1e-3, seed=1, offset=0)
    g = oracle.greedy_accept(lp, tok, oracle.tree_encode(parent, rank))
    np.testing.assert_array_equal(a.cpu().numpy(), g["accept_len"])
    np.testing.assert_array_equal(p.cpu().numpy(), g["accept_path"])
    np.testing.assert_array_equal(n.cpu().numpy(), g["next_token"])


def test_typical_equal_logits():
    st = lib()
    parent, rank = wl.cartesian_tree((3, 2))
    B, T, V = 8, len(parent), 40
    lp = np.zeros((B, T, V), dtype=np.float32)
    tok = np.tile((np.arange(T) % V).astype(np.int32), (B, 1))
    tree = st.spec_tree_build(parent, rank)
    a, p, n, _ = st.tree_accept_typical(to_dev(lp), to_dev(tok), tree, temperature=0.7, seed=42, offset=3)
    _, us = acceptance_uniforms(42, 3, B, T)
    assert (a.cpu().numpy() == 2).all()
    np.testing.assert_array_equal(n.cpu().numpy(), np.floor(np.asarray(us) * V).astype(int))


def test_typical_vocabulary_past_the_walk_cache():
    """V = 50000: the extra token's draw weights are recomputed from the logits on every scan."""
    st = lib()
    rng = np.random.default_rng(50001)
    V, B = 50000, 6
    parent, rank = wl.random_tree(rng, 40, max_children=3)
    T = len(parent)
    lp = rng.standard_normal((B, T, V), dtype=np.float32) * np.float32(3.0)
    tok = wl.sibling_tokens(rng, parent, B, V)
    near_total = 0
    for offset in range(3):
        near, _ = _compare(st, lp, tok, parent, rank, 0.7, 0.09, 0.3, 11, offset)
        near_total += near
    assert near_total <= 2
