"""Pins for the oracle's typical acceptance (CPU only).

Independent of the oracle's arithmetic: scipy's entropy (a library routine)
fixes the threshold of a small hand-built case; the temperature -> 0 limit
must reproduce greedy acceptance (pinned by brute force elsewhere); equal
logits give a closed form (every edge accepted, extra token floor(u * V)); an
unreachable threshold accepts nothing; and the extra token drawn at a fixed
node follows p (chi-square).
"""

import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

import spec_workloads as wl
from oracle import greedy_accept, tree_encode, typical_accept


def _chain3():
    return tree_encode(np.array([-1, 0, 1]), np.array([0, 0, 0]))


def test_threshold_from_library_entropy():
    # root row p = softmax(z); child token 1 then grandchild token 0
    z_root = np.log(np.array([0.5, 0.3, 0.2]))
    z_child = np.log(np.array([0.2, 0.7, 0.1]))
    lp = np.stack([z_root, z_child, z_child])[None]            # [1, 3, 3]
    tok = np.array([[0, 1, 0]])
    seen = set()
    for eps, alpha in [(0.5, 1.0), (0.25, 1.0), (0.9, 0.1)]:
        out = typical_accept(lp, tok, _chain3(), 1.0, eps, alpha, [0.5])
        thr_root = min(eps, alpha * np.exp(-stats.entropy([0.5, 0.3, 0.2])))
        thr_child = min(eps, alpha * np.exp(-stats.entropy([0.2, 0.7, 0.1])))
        child_ok = 0.3 > thr_root
        grand_ok = child_ok and 0.2 > thr_child
        want = 2 if grand_ok else 1 if child_ok else 0
        assert out["accept_len"][0] == want, (eps, alpha)
        seen.add(want)
    assert seen == {0, 1, 2}   # the three cases reach every depth


def test_low_temperature_reduces_to_greedy():
    rng = np.random.default_rng(4)
    w = wl.WORKLOADS[1]
    parent, rank = wl.make_tree(w.tree)
    tree = tree_encode(parent, rank)
    B, T, V = 6, len(parent), 50
    lp = rng.standard_normal((B, T, V))
    tok = wl.sibling_tokens(rng, parent, B, V)
    # plant argmax tokens along random paths so acceptance goes deep
    for b in range(B):
        for c in range(1, T):
            if rng.random() < 0.7:
                lp[b, parent[c], tok[b, c]] = lp[b, parent[c]].max() + 1.0
    g = greedy_accept(lp, tok, tree)
    t = typical_accept(lp, tok, tree, 1e-4, 0.09, 0.3, rng.random(B))
    np.testing.assert_array_equal(t["accept_len"], g["accept_len"])
    np.testing.assert_array_equal(t["accept_path"], g["accept_path"])
    np.testing.assert_array_equal(t["next_token"], g["next_token"])


def test_equal_logits_closed_form():
    parent, rank = wl.cartesian_tree((3, 2))
    tree = tree_encode(parent, rank)
    B, T, V = 4, len(parent), 40
    lp = np.zeros((B, T, V))
    tok = np.tile(np.arange(T) % V, (B, 1))
    u = np.array([0.0, 0.26, 0.5, 0.999])
    out = typical_accept(lp, tok, tree, 0.7, 0.09, 0.3, u)   # threshold min(0.09, 0.3/40) < 1/40
    deepest = min(i for i in range(T) if tree["depth"][i] == tree["max_depth"])
    assert (out["accept_len"] == tree["max_depth"]).all()
    assert (out["accept_path"][:, -1] == deepest).all()
    np.testing.assert_array_equal(out["next_token"], np.floor(u * V).astype(int))


def test_unreachable_threshold_accepts_nothing():
    rng = np.random.default_rng(2)
    parent, rank = wl.cartesian_tree((2, 2))
    tree = tree_encode(parent, rank)
    lp = rng.standard_normal((3, len(parent), 30))
    tok = wl.sibling_tokens(rng, parent, 3, 30)
    out = typical_accept(lp, tok, tree, 1.0, 2.0, 50.0, rng.random(3))   # threshold > 1 > any p
    assert (out["accept_len"] == 0).all()
    assert (out["accept_path"][:, 0] == 0).all() and (out["accept_path"][:, 1:] == -1).all()


def test_extra_token_follows_p():
    rng = np.random.default_rng(8)
    V, n = 12, 20000
    z = rng.standard_normal(V) * 1.5
    tree = tree_encode(np.array([-1]), np.array([0]))
    lp = np.broadcast_to(z, (n, 1, V))
    out = typical_accept(lp, np.zeros((n, 1), dtype=int), tree, 1.3, 0.09, 0.3, rng.random(n))
    counts = np.bincount(out["next_token"], minlength=V)
    p = softmax(z / 1.3)
    chi2 = stats.chisquare(counts, p * n)
    assert chi2.pvalue > 1e-3
