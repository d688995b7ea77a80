"""Pins for the oracle's paged-cache tree attention (CPU only).

A paged cache is built by scattering a contiguous cache's blocks to random
pool slots.  Independent checks: the gather returns the original rows, and on
a chain tree the paged attention equals torch's scaled_dot_product_attention
(a library routine) with a causal mask over [prefix, chain] of the contiguous
rows.  Table entries past the blocks a sequence uses are garbage and must not
be read.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import spec_workloads as wl
from oracle import gather_pages, tree_attention_paged, tree_encode


def _scatter(rng, cache, prefix, bs, spare=3):
    """Pool [num_blocks, Hkv, bs, D] and table [B, n_blocks] holding cache's blocks at random slots."""
    B, Hkv, Lmax, D = cache.shape
    n_blocks = Lmax // bs
    num = B * n_blocks + spare
    pool = rng.standard_normal((num, Hkv, bs, D)).astype(cache.dtype)   # unused slots: noise
    slots = rng.permutation(num)
    table = np.full((B, n_blocks), 10 ** 6, dtype=np.int32)              # garbage past the used blocks
    k = 0
    for b in range(B):
        for j in range(-(-int(prefix[b]) // bs)):
            table[b, j] = slots[k]
            pool[slots[k]] = cache[b, :, j * bs:(j + 1) * bs]
            k += 1
    return pool, table


@pytest.mark.parametrize("bs", [64, 128])
def test_gather_returns_the_original_rows(bs):
    rng = np.random.default_rng(bs)
    B, Hkv, Lmax, D = 3, 2, 512, 8
    cache = rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32)
    prefix = np.array([0, 200, 512], dtype=np.int32)
    pool, table = _scatter(rng, cache, prefix, bs)
    got = gather_pages(pool, table, bs, prefix)
    for b in range(B):
        used = -(-int(prefix[b]) // bs) * bs
        np.testing.assert_array_equal(got[b, :, :used], cache[b, :, :used])


@pytest.mark.parametrize("bs,Hq,Hkv", [(64, 4, 2), (128, 2, 2)])
def test_paged_chain_equals_causal_attention(bs, Hq, Hkv):
    rng = np.random.default_rng(bs + Hq)
    B, T, D, Lmax = 2, 5, 16, 384
    prefix = np.array([130, 300], dtype=np.int32)
    q = rng.standard_normal((B, Hq, T, D)).astype(np.float32)
    kc = rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32)
    vc = rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32)
    kt = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    vt = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    kpool, table = _scatter(rng, kc, prefix, bs)
    vpool = np.zeros_like(kpool)
    for b in range(B):   # same slots for V
        for j in range(-(-int(prefix[b]) // bs)):
            vpool[table[b, j]] = vc[b, :, j * bs:(j + 1) * bs]
    parent, rank = wl.chain_tree(T)
    O, _ = tree_attention_paged(q, kpool, vpool, table, bs, prefix, kt, vt, tree_encode(parent, rank), "f32")
    g = Hq // Hkv
    for b in range(B):
        L = int(prefix[b])
        for h in range(Hq):
            K = np.concatenate([kc[b, h // g, :L], kt[b, h // g]]).astype(np.float64)
            V = np.concatenate([vc[b, h // g, :L], vt[b, h // g]]).astype(np.float64)
            Q = q[b, h].astype(np.float64)
            mask = np.ones((T, L + T), dtype=bool)
            mask[:, L:] = np.tril(np.ones((T, T), dtype=bool))
            ref = F.scaled_dot_product_attention(torch.from_numpy(Q)[None, None], torch.from_numpy(K)[None, None],
                                                 torch.from_numpy(V)[None, None],
                                                 attn_mask=torch.from_numpy(mask)[None, None])[0, 0].numpy()
            np.testing.assert_allclose(O[b, h], ref, rtol=1e-12, atol=1e-12)
