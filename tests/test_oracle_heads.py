"""Pins for the oracle's Medusa/Hydra heads (CPU only).

Each check reduces the head to a case with a known answer computed by a
library routine (torch.nn.functional.linear / silu / topk / log_softmax):
zero-initialised heads reproduce lm_head (Medusa Heads page), Medusa heads
repeat one sibling set under every parent, a head that only sees h or only
sees the parent embedding, and a bias-only head.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from conftest import read_golden
from oracle import tree_encode, hydra_draft, silu
import spec_workloads as wl


def _chain(K):
    return tree_encode(*wl.chain_tree(K + 1))


def test_silu_matches_torch():
    x = np.linspace(-50, 50, 10001)
    np.testing.assert_allclose(silu(x), F.silu(torch.from_numpy(x)).numpy(), rtol=1e-15, atol=1e-300)
    assert silu(np.array([-1000.0]))[0] == 0.0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_init_heads_reproduce_lm_head(dtype):
    rows = {r[0]: r[1:] for r in read_golden("medusa_heads_zero_init.txt")}
    d, V, K = int(rows["hidden_size"][0]), int(rows["vocab_size"][0]), int(rows["num_heads"][0])
    assert rows["expected"] == ["True"] * K
    rng = np.random.default_rng(6)
    lm_head = rng.standard_normal((V, d)).astype(np.float32) * np.float32(0.02)
    h = rng.standard_normal((1, d)).astype(np.float32)
    if dtype == "bf16":
        lm_head, h = wl.f32_to_bf16_bits(lm_head), wl.f32_to_bf16_bits(h)
        dec = lambda a: torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).double()
    else:
        dec = lambda a: torch.from_numpy(a).double()
    zeros_w = np.zeros((d, d), dtype=np.float32 if dtype == "f32" else np.uint16)
    zeros_b = np.zeros((d,), dtype=zeros_w.dtype)
    out = hydra_draft(h, lm_head, [zeros_w] * K, [zeros_b] * K, [lm_head] * K, [0] * K, [1] * K,
                      [0], _chain(K), dtype, keep_logits=True)
    ref = F.linear(dec(h), dec(lm_head))[0].numpy()
    got = [out["logits"][(0, u)] for u in range(K)]
    for g in got:
        np.testing.assert_allclose(g, ref, rtol=1e-13, atol=1e-13)
    ref_top = int(torch.argmax(torch.from_numpy(ref)))
    assert list(out["node_tok"][0, 1:]) == [ref_top] * K


def test_medusa_siblings_repeat_under_every_parent():
    # Medusa Heads, "Tree Attention und Akzeptanz": with heads that all read the
    # same hidden state, head 2 proposes the same tokens under every head-1 branch.
    rng = np.random.default_rng(7)
    d, V = 32, 50
    parent, rank = wl.cartesian_tree((3, 4))
    tree = tree_encode(parent, rank)
    W1 = [rng.standard_normal((d, d)).astype(np.float32) * 0.3 for _ in range(2)]
    b1 = [rng.standard_normal(d).astype(np.float32) * 0.1 for _ in range(2)]
    W2 = [rng.standard_normal((V, d)).astype(np.float32) for _ in range(2)]
    E = rng.standard_normal((V, d)).astype(np.float32)
    h = rng.standard_normal((2, d)).astype(np.float32)
    out = hydra_draft(h, E, W1, b1, W2, [0, 0], [3, 4], [5, 6], tree, "f32")
    for b in range(2):
        sets = [tuple(out["node_tok"][b, tree["children"][u]]) for u in tree["children"][0]]
        assert all(s == sets[0] for s in sets)
        # with hydra conditioning they generally differ
    W1c = [W1[0], rng.standard_normal((d, 2 * d)).astype(np.float32) * 0.3]
    out2 = hydra_draft(h, E, W1c, b1, W2, [0, 1], [3, 4], [5, 6], tree, "f32")
    sets = [tuple(out2["node_tok"][0, tree["children"][u]]) for u in tree["children"][0]]
    assert len(set(sets)) > 1


def _one_depth(h, E, W1, b1, W2, cond, root_tok=0):
    """Run the oracle on a root with one child and return head 1's logits row."""
    tree = tree_encode([-1, 0])
    out = hydra_draft(h, E, [W1], [b1], [W2], [cond], [1], [root_tok], tree, "f32", keep_logits=True)
    return out["logits"][(0, 0)]


def test_conditioned_head_concat_order_and_gather():
    rng = np.random.default_rng(8)
    d, V = 16, 40
    h = rng.standard_normal((1, d)).astype(np.float32)
    E = rng.standard_normal((V, d)).astype(np.float32)
    W2 = rng.standard_normal((V, d)).astype(np.float32)
    A = rng.standard_normal((d, d)).astype(np.float32) * 0.5
    b = rng.standard_normal(d).astype(np.float32) * 0.1
    Z = np.zeros((d, d), dtype=np.float32)
    t = lambda a: torch.from_numpy(np.asarray(a)).double()
    # W1 = [A | 0]: the head sees only h
    got = _one_depth(h, E, np.concatenate([A, Z], 1), b, W2, 1, root_tok=11)
    ref = F.linear(t(h)[0] + F.silu(F.linear(t(h)[0], t(A), t(b))), t(W2))
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)
    # W1 = [0 | A]: the head sees only the parent token's embedding row E[11]
    got = _one_depth(h, E, np.concatenate([Z, A], 1), b, W2, 1, root_tok=11)
    ref = F.linear(t(h)[0] + F.silu(F.linear(t(E[11]), t(A), t(b))), t(W2))
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_bias_only_head():
    rng = np.random.default_rng(9)
    d, V = 8, 30
    h = rng.standard_normal((1, d)).astype(np.float32)
    E = rng.standard_normal((V, d)).astype(np.float32)
    W2 = rng.standard_normal((V, d)).astype(np.float32)
    b = rng.standard_normal(d).astype(np.float32)
    got = _one_depth(h, E, np.zeros((d, d), np.float32), b, W2, 0)
    t = lambda a: torch.from_numpy(np.asarray(a)).double()
    ref = F.linear(t(h)[0] + F.silu(t(b)), t(W2))
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_ranks_follow_descending_order_and_logprob_accumulates():
    # Hydra Guide "Candidate Tree Construction" (b = [3,2,2] -> 21 nodes, the
    # page's own demo shape: vocab 5000, d 512); children of rank r take the
    # (r+1)-th best token; branch probability multiplies down the tree.
    rng = np.random.default_rng(10)
    d, V = 512, 5000
    parent, rank = wl.cartesian_tree((3, 2, 2))
    tree = tree_encode(parent, rank)
    assert tree["T"] - 1 == 21
    W1 = [rng.standard_normal((d, d * c)).astype(np.float32) * 0.02 for c in (1, 2, 2)]
    b1 = [rng.standard_normal(d).astype(np.float32) * 0.02 for _ in range(3)]
    W2 = [rng.standard_normal((V, d)).astype(np.float32) * 0.02 for _ in range(3)]
    E = rng.standard_normal((V, d)).astype(np.float32)
    h = rng.standard_normal((1, d)).astype(np.float32)
    out = hydra_draft(h, E, W1, b1, W2, [0, 1, 1], [3, 2, 2], [0], tree, "f32", keep_logits=True)
    for u in range(tree["T"]):
        kids = tree["children"][u]
        if not kids:
            continue
        row = torch.from_numpy(out["logits"][(0, u)])
        vals, idx = torch.topk(row, 3)
        logp = torch.log_softmax(row, dim=0)
        for c in kids:
            assert out["node_tok"][0, c] == int(idx[rank[c]])
            assert out["node_logit"][0, c] == float(vals[rank[c]])
            np.testing.assert_allclose(out["node_logprob"][0, c],
                                       out["node_logprob"][0, u] + float(logp[idx[rank[c]]]), rtol=1e-12)
    # the probabilities of all leaves' paths sum to at most 1 and each is a product of softmax values
    probs = np.exp(out["node_logprob"][0, 1:])
    assert np.all(probs > 0) and np.all(probs <= 1)


def test_topk_ties_go_to_lower_token():
    d, V = 4, 10
    h = np.ones((1, d), dtype=np.float32)
    W2 = np.zeros((V, d), dtype=np.float32)
    W2[[2, 5, 7]] = 1.0   # three tied maxima
    tree = tree_encode([-1, 0, 0, 0], [0, 0, 1, 2])
    out = hydra_draft(h, np.zeros((V, d), np.float32), [np.zeros((d, d), np.float32)], [None], [W2],
                      [0], [3], [0], tree, "f32")
    assert list(out["node_tok"][0, 1:]) == [2, 5, 7]


def test_all_ancestor_conditioning_blocks_and_reduction():
    # Hydra Guide, "2. Generalizing to Arbitrary Tree Depths": head k reads h and the
    # embeddings of the path's tokens at depths 1..k (cond 2), depth 1 first
    rng = np.random.default_rng(21)
    d, V, K = 12, 30, 3
    tree = _chain(K)
    h = rng.standard_normal((1, d)).astype(np.float32)
    E = rng.standard_normal((V, d)).astype(np.float32)
    W2 = [rng.standard_normal((V, d)).astype(np.float32) for _ in range(K)]
    A = rng.standard_normal((d, d)).astype(np.float32) * 0.5
    b = [rng.standard_normal(d).astype(np.float32) * 0.1 for _ in range(K)]
    Z = np.zeros((d, d), dtype=np.float32)
    W1 = [rng.standard_normal((d, (k + 1) * d)).astype(np.float32) * 0.3 for k in range(K)]
    t = lambda a: torch.from_numpy(np.asarray(a)).double()
    for blocks, pick in [([Z, A, Z], 1), ([Z, Z, A], 2)]:   # head 2 sees only depth-1 / only depth-2 tokens
        W1b = list(W1)
        W1b[2] = np.concatenate(blocks, 1)
        out = hydra_draft(h, E, W1b, b, W2, [2, 2, 2], [1, 1, 1], [3], tree, "f32", keep_logits=True)
        tok = int(out["node_tok"][0, pick])
        ref = F.linear(t(h)[0] + F.silu(F.linear(t(E[tok]), t(A), t(b[2]))), t(W2[2]))
        np.testing.assert_allclose(out["logits"][(0, 2)], ref.numpy(), rtol=1e-12, atol=1e-12)
    # depth <= 1: cond 2 is cond 0 at head 0 and cond 1 at head 1
    tree2 = _chain(2)
    a = hydra_draft(h, E, W1[:2], b[:2], W2[:2], [2, 2], [1, 1], [3], tree2, "f32")
    c = hydra_draft(h, E, W1[:2], b[:2], W2[:2], [0, 1], [1, 1], [3], tree2, "f32")
    np.testing.assert_array_equal(a["node_tok"], c["node_tok"])
    np.testing.assert_allclose(a["node_logit"], c["node_logit"], rtol=0, atol=0)


def test_layernorm_fusion_head_form():
    # the head form the Hydra Guide prints as code: Linear -> SiLU -> Linear -> LayerNorm,
    # then a bias-free projection; its first head Linear -> SiLU -> LayerNorm (no W1b)
    from oracle import hydra_draft_heads
    rng = np.random.default_rng(31)
    d, V, hidden, eps = 16, 50, 24, 1e-5
    tree = tree_encode(*wl.cartesian_tree((3,)))      # root and three children: one head
    h = rng.standard_normal((1, d)).astype(np.float32)
    E = rng.standard_normal((V, d)).astype(np.float32)
    W2 = rng.standard_normal((V, d)).astype(np.float32)
    g = rng.standard_normal(d).astype(np.float32)
    be = rng.standard_normal(d).astype(np.float32)
    t = lambda a: torch.from_numpy(np.asarray(a)).double()
    root = 7
    x = torch.cat([t(h)[0], t(E[root])])               # cond 1: [h || E[root]]
    # two layers, hidden != d
    W1 = rng.standard_normal((hidden, 2 * d)).astype(np.float32) * 0.3
    b1 = rng.standard_normal(hidden).astype(np.float32) * 0.1
    W1b = rng.standard_normal((d, hidden)).astype(np.float32) * 0.3
    b1b = rng.standard_normal(d).astype(np.float32) * 0.1
    head = dict(form=1, cond=1, topk=3, W1=W1, b1=b1, W1b=W1b, b1b=b1b, gamma=g, beta=be, W2=W2)
    out = hydra_draft_heads(h, E, [head], [root], tree, "f32", ln_eps=eps, keep_logits=True)
    z = F.layer_norm(F.linear(F.silu(F.linear(x, t(W1), t(b1))), t(W1b), t(b1b)), (d,), t(g), t(be), eps)
    np.testing.assert_allclose(out["logits"][(0, 0)], F.linear(z, t(W2)).numpy(), rtol=1e-12, atol=1e-12)
    # one layer (no W1b), unconditioned: the printed first head
    W1s = rng.standard_normal((d, d)).astype(np.float32) * 0.3
    head = dict(form=1, cond=0, topk=3, W1=W1s, b1=None, W1b=None, gamma=None, beta=None, W2=W2)
    out = hydra_draft_heads(h, E, [head], [root], tree, "f32", ln_eps=eps, keep_logits=True)
    z = F.layer_norm(F.silu(F.linear(t(h)[0], t(W1s))), (d,), eps=eps)
    np.testing.assert_allclose(out["logits"][(0, 0)], F.linear(z, t(W2)).numpy(), rtol=1e-12, atol=1e-12)


def test_layernorm_head_zero_gain_gives_beta():
    # gamma = 0: every head's z is beta whatever the input, so each node's logits are W2 beta and every
    # parent's children are the same top-k of that row (closed form, independent of h, E, W1, W1b)
    from oracle import hydra_draft_heads
    rng = np.random.default_rng(32)
    d, V = 8, 40
    parent, rank = wl.cartesian_tree((3, 2))
    tree = tree_encode(parent, rank)
    h = rng.standard_normal((2, d)).astype(np.float32)
    E = rng.standard_normal((V, d)).astype(np.float32)
    heads = []
    for k, tk in enumerate((3, 2)):
        heads.append(dict(form=1, cond=k, topk=tk, W1=rng.standard_normal((12, d * (k + 1))).astype(np.float32),
                          b1=None, W1b=rng.standard_normal((d, 12)).astype(np.float32), b1b=None,
                          gamma=np.zeros(d, dtype=np.float32), beta=rng.standard_normal(d).astype(np.float32),
                          W2=rng.standard_normal((V, d)).astype(np.float32)))
    out = hydra_draft_heads(h, E, heads, [1, 2], tree, "f32")
    for b in range(2):
        for c in range(1, len(parent)):
            k = tree["depth"][c] - 1
            row = heads[k]["W2"].astype(np.float64) @ heads[k]["beta"].astype(np.float64)
            order = np.argsort(-row, kind="stable")
            assert out["node_tok"][b, c] == order[rank[c]]
            np.testing.assert_allclose(out["node_logit"][b, c], row[order[rank[c]]], rtol=1e-12)
