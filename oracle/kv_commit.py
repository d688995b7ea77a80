"""KV commit of the accepted path (oracle; test infrastructure only).

"Speculative Decoding" (thegustafson.com), section "The acceptance criterion":
after the verification, what follows the rejection point is discarded from the
draft and target caches, and the next round starts from the last accepted
token.  Hydra Guide, section "3. Tree KV-Cache Page Sizing": the discarded
candidate nodes are rolled back at once, without deallocation.

The pages give no layout.  Taken here: the keys and values the verification
computed for the tree nodes sit in k_tree, v_tree [B, Hkv, T, D]; the cache is
k_cache, v_cache [B, Hkv, Lmax, D] with the first prefix_len[b] rows valid.
The accepted path of sequence b is accept_path[b, 0..m] (root first, m =
accept_len[b], the output of the acceptance step); its m + 1 nodes' rows are
appended to the cache at positions prefix_len[b] .. prefix_len[b] + m of every
KV head, and prefix_len[b] grows by m + 1.  The extra token the acceptance
emits is not committed: its keys and values come from the next round, as the
root of the next tree.  Nothing else changes: the rows of the rejected nodes
are never copied, so rolling them back costs nothing.

A sequence whose path is not a root-first chain of the tree (wrong root, a node
whose parent is not the previous entry, m outside 0..max_depth) or whose
commit would pass Lmax is left unchanged and reported.

Pin: the path equivalence the Hydra Guide states in section "Tree Attention
Matrix with Topology-Aware Causal Masking" -- after the commit, plain causal
attention of the accepted node's query over the first prefix_len[b] + m + 1
cache rows equals that node's tree attention before the commit.
"""

import numpy as np


def kv_commit(k_tree, v_tree, k_cache, v_cache, prefix_len, accept_len, accept_path, tree):
    """Return (k_cache', v_cache', prefix_len', bad) with the accepted paths committed.

    Inputs are not modified.  ``bad`` is a bool [B]: True where the sequence
    was left unchanged because its path or its length is invalid.  Works on
    any element type (a copy: the bits of the tree rows land unchanged).
    """
    k_cache = np.array(k_cache, copy=True)
    v_cache = np.array(v_cache, copy=True)
    k_tree = np.asarray(k_tree)
    v_tree = np.asarray(v_tree)
    prefix_len = np.array(prefix_len, dtype=np.int64, copy=True).reshape(-1)
    accept_len = np.asarray(accept_len, dtype=np.int64).reshape(-1)
    accept_path = np.asarray(accept_path, dtype=np.int64)
    B = prefix_len.shape[0]
    Lmax = k_cache.shape[2]
    parent = tree["parent"]
    bad = np.zeros(B, dtype=bool)
    for b in range(B):
        m = int(accept_len[b])
        if m < 0 or m > tree["max_depth"]:
            bad[b] = True
            continue
        path = [int(x) for x in accept_path[b, :m + 1]]
        chain = path[0] == 0 and all(0 <= path[i] < tree["T"] and parent[path[i]] == path[i - 1]
                                     for i in range(1, m + 1))
        L = int(prefix_len[b])
        if not chain or L < 0 or L + m + 1 > Lmax:
            bad[b] = True
            continue
        for i, node in enumerate(path):
            k_cache[b, :, L + i] = k_tree[b, :, node]
            v_cache[b, :, L + i] = v_tree[b, :, node]
        prefix_len[b] = L + m + 1
    return k_cache, v_cache, prefix_len, bad


def kv_commit_paged(k_tree, v_tree, k_pool, v_pool, block_table, block_size, prefix_len, accept_len, accept_path,
                    tree):
    """The same commit into a paged cache: return (k_pool', v_pool', prefix_len', bad).

    Hydra Guide, "Hydra Production Engineering Checklist", item 3 (KV-Cache
    Tree Branch Management: the cache lives in pre-allocated static blocks) with
    the layout read for the paged attention: pool [num_blocks, Hkv, block_size,
    D], block_table[b, j] the pool block of positions j*block_size ..
    (j+1)*block_size - 1 of sequence b.  Cache position L + i of sequence b is
    pool row (block_table[b, (L+i) // block_size], :, (L+i) % block_size), so
    the accepted node i's rows land there; everything else as ``kv_commit``.
    Beyond kv_commit's checks a sequence is also left unchanged (and reported)
    when its commit would pass max_blocks * block_size positions or a block it
    would write lies outside the pool.
    """
    k_pool = np.array(k_pool, copy=True)
    v_pool = np.array(v_pool, copy=True)
    k_tree = np.asarray(k_tree)
    v_tree = np.asarray(v_tree)
    block_table = np.asarray(block_table, dtype=np.int64)
    prefix_len = np.array(prefix_len, dtype=np.int64, copy=True).reshape(-1)
    accept_len = np.asarray(accept_len, dtype=np.int64).reshape(-1)
    accept_path = np.asarray(accept_path, dtype=np.int64)
    B, max_blocks = block_table.shape
    num_blocks = k_pool.shape[0]
    parent = tree["parent"]
    bad = np.zeros(B, dtype=bool)
    for b in range(B):
        m = int(accept_len[b])
        if m < 0 or m > tree["max_depth"]:
            bad[b] = True
            continue
        path = [int(x) for x in accept_path[b, :m + 1]]
        chain = path[0] == 0 and all(0 <= path[i] < tree["T"] and parent[path[i]] == path[i - 1]
                                     for i in range(1, m + 1))
        L = int(prefix_len[b])
        if not chain or L < 0 or L + m + 1 > max_blocks * block_size:
            bad[b] = True
            continue
        blocks = [int(block_table[b, (L + i) // block_size]) for i in range(m + 1)]
        if any(blk < 0 or blk >= num_blocks for blk in blocks):
            bad[b] = True
            continue
        for i, node in enumerate(path):
            k_pool[blocks[i], :, (L + i) % block_size] = k_tree[b, :, node]
            v_pool[blocks[i], :, (L + i) % block_size] = v_tree[b, :, node]
        prefix_len[b] = L + m + 1
    return k_pool, v_pool, prefix_len, bad
