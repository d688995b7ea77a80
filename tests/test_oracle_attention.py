"""Pins for the oracle's tree attention (CPU only).

Independent checks: torch's scaled_dot_product_attention (a library routine)
on a chain tree (= ordinary causal attention over prompt + chain) and, per node,
on the node's own [prefix, root-to-node path] computed alone.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import tree_encode, tree_attention
import spec_workloads as wl


def _t(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float64))


def _inputs(rng, B, Hq, Hkv, T, D, Lmax, prefix):
    return dict(
        q=rng.standard_normal((B, Hq, T, D)).astype(np.float32),
        k_cache=rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32),
        v_cache=rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32),
        prefix_len=np.array(prefix, dtype=np.int32),
        k_tree=rng.standard_normal((B, Hkv, T, D)).astype(np.float32),
        v_tree=rng.standard_normal((B, Hkv, T, D)).astype(np.float32),
    )


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (6, 1)])
def test_chain_tree_equals_causal_attention(Hq, Hkv):
    # Hydra Guide: a node's attention equals autoregressive attention over
    # [prompt, its ancestors, itself]; on a chain that is plain causal attention.
    rng = np.random.default_rng(2)
    B, T, D, Lmax = 2, 7, 16, 20
    prefix = [13, 20]
    x = _inputs(rng, B, Hq, Hkv, T, D, Lmax, prefix)
    parent, rank = wl.chain_tree(T)
    tree = tree_encode(parent, rank)
    O, lse = tree_attention(**x, tree=tree, dtype="f32")
    g = Hq // Hkv
    for b in range(B):
        L = prefix[b]
        # full sequence = prefix rows then the chain; queries for the prefix rows are dummies
        k = torch.cat([_t(x["k_cache"][b, :, :L]), _t(x["k_tree"][b])], dim=1)     # [Hkv, L+T, D]
        v = torch.cat([_t(x["v_cache"][b, :, :L]), _t(x["v_tree"][b])], dim=1)
        qfull = torch.cat([torch.zeros(Hq, L, D, dtype=torch.float64), _t(x["q"][b])], dim=1)
        k = k.repeat_interleave(g, dim=0)
        v = v.repeat_interleave(g, dim=0)
        ref = F.scaled_dot_product_attention(qfull[None], k[None], v[None], is_causal=True)[0][:, L:]
        np.testing.assert_allclose(O[b], ref.numpy(), rtol=1e-10, atol=1e-12)
        s = torch.einsum("htd,hsd->hts", qfull, k) / np.sqrt(D)
        causal = torch.ones(L + T, L + T, dtype=torch.bool).tril()
        s = s.masked_fill(~causal, float("-inf"))
        np.testing.assert_allclose(lse[b], torch.logsumexp(s, dim=-1)[:, L:].numpy(), rtol=1e-12, atol=1e-12)


def test_each_node_equals_its_own_path():
    rng = np.random.default_rng(3)
    B, Hq, Hkv, T, D, Lmax = 2, 4, 2, 17, 8, 9
    prefix = [0, 9]   # an empty prefix too: the node then sees only its own path
    x = _inputs(rng, B, Hq, Hkv, T, D, Lmax, prefix)
    parent, rank = wl.random_tree(rng, T, max_children=3)
    tree = tree_encode(parent, rank)
    O, lse = tree_attention(**x, tree=tree, dtype="f32", scale=0.3)
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            for i in range(T):
                path = []
                j = i
                while j != -1:
                    path.append(j)
                    j = int(parent[j])
                path = path[::-1]
                kv = h // g
                k = torch.cat([_t(x["k_cache"][b, kv, : prefix[b]]), _t(x["k_tree"][b, kv, path])])
                v = torch.cat([_t(x["v_cache"][b, kv, : prefix[b]]), _t(x["v_tree"][b, kv, path])])
                qi = _t(x["q"][b, h, i])[None]
                ref = F.scaled_dot_product_attention(qi[None], k[None], v[None], scale=0.3)[0, 0]
                np.testing.assert_allclose(O[b, h, i], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_cache_rows_beyond_prefix_are_ignored():
    rng = np.random.default_rng(4)
    x = _inputs(rng, 1, 2, 2, 7, 8, 12, [7])
    tree = tree_encode(*wl.cartesian_tree((2, 2)))
    O1, _ = tree_attention(**x, tree=tree, dtype="f32")
    x["k_cache"][:, :, 7:] = 1e3
    x["v_cache"][:, :, 7:] = -1e3
    O2, _ = tree_attention(**x, tree=tree, dtype="f32")
    assert np.array_equal(O1, O2)


def test_bf16_inputs_decoded_exactly():
    rng = np.random.default_rng(5)
    x = _inputs(rng, 1, 2, 1, 7, 8, 6, [6])
    xb = {k: (wl.f32_to_bf16_bits(v) if v.dtype == np.float32 else v) for k, v in x.items()}
    tree = tree_encode(*wl.cartesian_tree((2, 2)))
    Ob, _ = tree_attention(**xb, tree=tree, dtype="bf16")
    # same computation on the float32 values that the bf16 bits stand for (decoded by torch)
    xf = {k: (torch.from_numpy(v.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
              if v.dtype == np.uint16 else v) for k, v in xb.items()}
    Of, _ = tree_attention(**xf, tree=tree, dtype="f32")
    assert np.array_equal(Ob, Of)
