"""Tree attention over a paged KV cache: CUDA path vs the oracle (GPU).

Pools are built by scattering a contiguous cache's blocks to random pool slots
(unused slots hold noise, table entries past the used blocks garbage).  The
paged call must match the oracle within the attention tolerance and, on the
same logical data, reproduce the contiguous tree_attention bit for bit (same
split plan, same tiles).
"""

import zlib

import numpy as np
import pytest

import oracle
import spec_workloads as wl
from gpu_util import assert_close, lib, to_dev

pytestmark = pytest.mark.gpu


def _scatter(rng, cache, prefix, bs, spare=5):
    B, Hkv, Lmax, D = cache.shape
    n_blocks = Lmax // bs
    num = B * n_blocks + spare
    pool = (rng.integers(0, 1 << 16, size=(num, Hkv, bs, D), dtype=np.uint16) & 0x3FFF) if cache.dtype == np.uint16 \
        else rng.standard_normal((num, Hkv, bs, D)).astype(np.float32)       # noise in unused slots (finite)
    slots = rng.permutation(num)
    table = np.full((B, n_blocks), 10 ** 7, dtype=np.int32)
    k = 0
    for b in range(B):
        for j in range(-(-int(prefix[b]) // bs)):
            table[b, j] = slots[k]
            pool[slots[k]] = cache[b, :, j * bs:(j + 1) * bs]
            k += 1
    return pool, table


def _case(dtype, B, Hq, Hkv, T, D, Lmax, prefix, bs, seed):
    rng = np.random.default_rng(seed)
    parent, rank = wl.random_tree(rng, T, max_children=4)
    enc = (lambda a: wl.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    n = lambda *s: enc(rng.standard_normal(s, dtype=np.float32))
    x = dict(q=n(B, Hq, T, D), k_cache=n(B, Hkv, Lmax, D), v_cache=n(B, Hkv, Lmax, D),
             prefix_len=np.array(prefix, dtype=np.int32), k_tree=n(B, Hkv, T, D), v_tree=n(B, Hkv, T, D))
    kpool, table = _scatter(rng, x["k_cache"], prefix, bs)
    vpool = kpool.copy()
    for b in range(B):
        for j in range(-(-int(prefix[b]) // bs)):
            vpool[table[b, j]] = x["v_cache"][b, :, j * bs:(j + 1) * bs]
    return parent, rank, x, kpool, vpool, table


CASES = [
    # dtype, B, Hq, Hkv, T, D, Lmax, prefix, block size
    ("bf16", 2, 8, 2, 70, 128, 768, [0, 700], 64),      # tensor-core path (140 rows per KV head), 64-key blocks
    ("bf16", 3, 4, 4, 64, 128, 1024, [1, 513, 1024], 128),
    ("bf16", 1, 16, 8, 100, 128, 1536, [1300], 256),
    ("bf16", 2, 4, 2, 20, 64, 320, [64, 257], 64),      # CUDA-core path (D = 64)
    ("f32", 2, 4, 4, 17, 128, 256, [100, 256], 128),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-B{c[1]}-H{c[2]}/{c[3]}-T{c[4]}-D{c[5]}-bs{c[8]}" for c in CASES])
def test_paged_matches_oracle_and_contiguous(case):
    st = lib()
    dtype, B, Hq, Hkv, T, D, Lmax, prefix, bs = case
    parent, rank, x, kpool, vpool, table = _case(dtype, B, Hq, Hkv, T, D, Lmax, prefix, bs, zlib.crc32(str(case).encode()))
    tree = st.spec_tree_build(parent, rank)
    dev = {k: to_dev(v) for k, v in x.items()}
    out_p, lse_p = st.tree_attention_paged(dev["q"], to_dev(kpool), to_dev(vpool), to_dev(table), dev["prefix_len"],
                                           dev["k_tree"], dev["v_tree"], tree)
    out_c, lse_c = st.tree_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["prefix_len"], dev["k_tree"],
                                     dev["v_tree"], tree)
    out_p, lse_p = out_p.cpu().numpy(), lse_p.cpu().numpy()
    np.testing.assert_array_equal(out_p, out_c.cpu().numpy())
    np.testing.assert_array_equal(lse_p, lse_c.cpu().numpy())
    O, L = oracle.tree_attention_paged(x["q"], kpool, vpool, table, bs, x["prefix_len"], x["k_tree"], x["v_tree"],
                                       oracle.tree_encode(parent, rank), dtype)
    assert_close(out_p, O, dtype, "out")
    assert_close(lse_p, L, dtype, "lse")


@pytest.mark.parametrize("D,Hq", [(128, 8), (64, 4)])
def test_out_of_pool_entries_are_reported(D, Hq):
    st = lib()
    B, Hkv, T, Lmax, bs = 1, 2, 40, 256, 64
    parent, rank, x, kpool, vpool, table = _case("bf16", B, Hq, Hkv, T, D, Lmax, [200], bs, 9 + D)
    table[0, 1] = kpool.shape[0] + 3     # a used block points past the pool
    table[0, 2] = -1
    tree = st.spec_tree_build(parent, rank)
    dev = {k: to_dev(v) for k, v in x.items()}
    import torch
    ws = torch.empty(st.tree_attention_paged_workspace_size(tree, B, Hq, Hkv, table.shape[1], bs, D, 1),
                     dtype=torch.uint8, device="cuda")
    out, _ = st.tree_attention_paged(dev["q"], to_dev(kpool), to_dev(vpool), to_dev(table), dev["prefix_len"],
                                     dev["k_tree"], dev["v_tree"], tree, ws=ws)
    torch.cuda.synchronize()
    assert st.spec_read_device_status(ws) == 1   # SPEC_EINVAL


def test_paged_70b_gqa_sampled():
    # the 70B-GQA layer shape (8 sequences, 64 query / 8 KV heads, prefixes 2048-4096), 128-key blocks;
    # the oracle checks a sample of (sequence, head) pairs
    st = lib()
    w = wl.WORKLOADS[4]
    parent, rank = wl.make_tree(w.tree)
    T, bs = len(parent), 128
    ax = wl.attention_inputs(w, T)
    rng = np.random.default_rng(4)
    kpool, table = _scatter(rng, ax["k_cache"], ax["prefix_len"], bs, spare=0)
    vpool = kpool.copy()
    for b in range(w.B):
        for j in range(-(-int(ax["prefix_len"][b]) // bs)):
            vpool[table[b, j]] = ax["v_cache"][b, :, j * bs:(j + 1) * bs]
    tree = st.spec_tree_build(parent, rank)
    dev = {k: to_dev(v) for k, v in ax.items()}
    out, lse = st.tree_attention_paged(dev["q"], to_dev(kpool), to_dev(vpool), to_dev(table), dev["prefix_len"],
                                       dev["k_tree"], dev["v_tree"], tree)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    heads = [(int(rng.integers(0, w.B)), int(rng.integers(0, w.Hq))) for _ in range(6)]
    O, L = oracle.tree_attention_paged(ax["q"], kpool, vpool, table, bs, ax["prefix_len"], ax["k_tree"], ax["v_tree"],
                                       oracle.tree_encode(parent, rank), "bf16", heads=heads)
    for b, h in heads:
        assert_close(out[b, h], O[b, h], "bf16", f"out[{b},{h}]")
        assert_close(lse[b, h], L[b, h], "bf16", f"lse[{b},{h}]")


def _paged_sweep(n=24, seed=4242):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = "bf16" if rng.random() < 0.75 else "f32"
        bs = int(rng.choice([64, 128, 192, 256]))
        Hkv = int(rng.choice([1, 2, 4]))
        g = int(rng.choice([1, 2, 4, 8]))
        T = int(rng.integers(1, 260))
        D = 128 if dtype == "bf16" and rng.random() < 0.8 else 64
        B = int(rng.integers(1, 5))
        Lmax = bs * int(rng.integers(1, 14))
        prefix = [int(x) for x in rng.integers(0, Lmax + 1, size=B)]
        out.append((i, dtype, B, Hkv * g, Hkv, T, D, Lmax, prefix, bs))
    return out


@pytest.mark.parametrize("case", _paged_sweep(), ids=lambda c: f"sweep{c[0]}-{c[1]}-B{c[2]}-H{c[3]}/{c[4]}-T{c[5]}-D{c[6]}-bs{c[9]}")
def test_paged_random_sweep(case):
    """Random shapes and block sizes: the paged call reproduces the contiguous call bit for bit on
    the same logical data, and matches the oracle on four sampled (sequence, head) pairs."""
    st = lib()
    i, dtype, B, Hq, Hkv, T, D, Lmax, prefix, bs = case
    parent, rank, x, kpool, vpool, table = _case(dtype, B, Hq, Hkv, T, D, Lmax, prefix, bs, 7000 + i)
    tree = st.spec_tree_build(parent, rank)
    out_p, lse_p = st.tree_attention_paged(to_dev(x["q"]), to_dev(kpool), to_dev(vpool), to_dev(table),
                                           to_dev(x["prefix_len"]), to_dev(x["k_tree"]), to_dev(x["v_tree"]), tree)
    out_c, lse_c = st.tree_attention(to_dev(x["q"]), to_dev(x["k_cache"]), to_dev(x["v_cache"]), to_dev(x["prefix_len"]),
                                     to_dev(x["k_tree"]), to_dev(x["v_tree"]), tree)
    out_p, lse_p, out_c, lse_c = (t.cpu().numpy() for t in (out_p, lse_p, out_c, lse_c))
    assert np.array_equal(out_p, out_c) and np.array_equal(lse_p, lse_c)
    rng = np.random.default_rng(i)
    pairs = [(b, h) for b in range(B) for h in range(Hq)]
    heads = [pairs[j] for j in rng.choice(len(pairs), size=min(4, len(pairs)), replace=False)]
    O, L = oracle.tree_attention(**x, tree=oracle.tree_encode(parent, rank), dtype=dtype, heads=heads)
    sel = ~np.isnan(L)
    assert_close(out_p[sel], O[sel], dtype, "out")
    assert_close(lse_p[sel], L[sel], dtype, "lse")
