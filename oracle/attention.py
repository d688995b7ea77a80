"""Tree attention of one verification layer (oracle; test infrastructure only).

Hydra Guide, section "Tree Attention Matrix with Topology-Aware Causal
Masking": the T tree tokens are appended to the prompt as one flattened
sequence; every tree token sees the whole prompt (the cached prefix) and, among
the tree tokens, only itself and its ancestors: the scores get M_tree(u, v) = 0
for those and -inf for all other tree tokens.  Its attention is then the same as
autoregressive attention over [prompt, its ancestors, itself].
"Speculative Decoding", section "Beyond draft models: Medusa", and "Medusa
Heads", section "Tree Attention und Akzeptanz", describe the same mask.

The pages fix no scale and no head grouping.  Taken here: scale = 1/sqrt(D)
unless given; query head h reads key/value head h // (Hq / Hkv) (contiguous
groups); the prefix of sequence b is its first prefix_len[b] cache rows.

Brute force: the full score row, plain softmax, one matmul with the values.
"""

import numpy as np

from .bf16 import bf16_bits_to_f64
from .tree import tree_mask


def _decode(x, dtype):
    if dtype == "bf16":
        return bf16_bits_to_f64(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def tree_attention(q, k_cache, v_cache, prefix_len, k_tree, v_tree, tree, dtype,
                   scale=None, heads=None):
    """Attention of every tree node over the cached prefix and its own ancestors.

    q [B, Hq, T, D]; k_cache, v_cache [B, Hkv, Lmax, D]; prefix_len [B];
    k_tree, v_tree [B, Hkv, T, D] (keys/values of the tree tokens themselves).
    ``heads``: optional list of (b, h) pairs to compute (the rest stays NaN);
    used to sample outputs of very large cases.

    Returns (O [B, Hq, T, D] float64, lse [B, Hq, T] float64), lse being the
    natural log of the softmax denominator of the scaled scores.
    """
    q = np.asarray(q)
    B, Hq, T, D = q.shape
    Hkv = np.asarray(k_cache).shape[1]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    M = tree_mask(tree)
    prefix_len = np.asarray(prefix_len, dtype=np.int64).reshape(B)

    O = np.full((B, Hq, T, D), np.nan)
    lse = np.full((B, Hq, T), np.nan)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    by_kv = {}
    for b, h in heads:
        by_kv.setdefault((b, h // g), []).append(h)
    for (b, kvh), hs in sorted(by_kv.items()):
        L = int(prefix_len[b])
        Kp = _decode(np.asarray(k_cache)[b, kvh, :L], dtype)
        Vp = _decode(np.asarray(v_cache)[b, kvh, :L], dtype)
        Kt = _decode(np.asarray(k_tree)[b, kvh], dtype)
        Vt = _decode(np.asarray(v_tree)[b, kvh], dtype)
        for h in hs:
            Q = _decode(q[b, h], dtype)
            S = np.concatenate([scale * (Q @ Kp.T), scale * (Q @ Kt.T) + M], axis=1)
            m = S.max(axis=1, keepdims=True)
            P = np.exp(S - m)
            denom = P.sum(axis=1, keepdims=True)
            O[b, h] = (P @ np.concatenate([Vp, Vt], axis=0)) / denom
            lse[b, h] = (m + np.log(denom))[:, 0]
    return O, lse


def gather_pages(pool, block_table, block_size, prefix_len):
    """Contiguous caches [B, Hkv, n_blocks * block_size, D] from a paged pool.

    Hydra Guide, "Hydra Production Engineering Checklist", item 3 (KV-Cache
    Tree Branch Management): the cache lives in pre-allocated static blocks.
    Taken here: pool [num_blocks, Hkv, block_size, D]; block_table[b, j] is the
    pool block holding positions j*block_size .. (j+1)*block_size - 1 of
    sequence b.  Entries past the last block prefix_len[b] needs are not read
    (their rows come out as zeros).
    """
    pool = np.asarray(pool)
    block_table = np.asarray(block_table, dtype=np.int64)
    B, n_blocks = block_table.shape
    _, Hkv, bs, D = pool.shape
    if bs != block_size:
        raise ValueError("pool block size differs from block_size")
    out = np.zeros((B, Hkv, n_blocks * bs, D), dtype=pool.dtype)
    for b in range(B):
        used = -(-int(prefix_len[b]) // bs)
        for j in range(used):
            out[b, :, j * bs:(j + 1) * bs] = pool[block_table[b, j]]
    return out


def tree_attention_paged(q, k_pool, v_pool, block_table, block_size, prefix_len, k_tree, v_tree, tree, dtype,
                         scale=None, heads=None):
    """tree_attention over a paged cache: the pages gathered into contiguous rows, then the same definition."""
    k_cache = gather_pages(k_pool, block_table, block_size, prefix_len)
    v_cache = gather_pages(v_pool, block_table, block_size, prefix_len)
    return tree_attention(q, k_cache, v_cache, prefix_len, k_tree, v_tree, tree, dtype, scale=scale, heads=heads)
