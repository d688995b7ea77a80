"""Tree attention: CUDA path vs the oracle, element by element (GPU)."""

import zlib

import numpy as np
import pytest

import oracle
import spec_workloads as wl
from gpu_util import assert_close, lib, to_dev

pytestmark = pytest.mark.gpu


def _run(st, x, tree, dtype, scale=None):
    out, lse = st.tree_attention(to_dev(x["q"]), to_dev(x["k_cache"]), to_dev(x["v_cache"]),
                                 to_dev(x["prefix_len"]), to_dev(x["k_tree"]), to_dev(x["v_tree"]), tree,
                                 scale=scale)
    return out.cpu().numpy(), lse.cpu().numpy()


def _rand_inputs(rng, dtype, B, Hq, Hkv, T, D, Lmax, prefix):
    enc = (lambda a: wl.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    n = lambda *s: enc(rng.standard_normal(s, dtype=np.float32))
    return dict(q=n(B, Hq, T, D), k_cache=n(B, Hkv, Lmax, D), v_cache=n(B, Hkv, Lmax, D),
                prefix_len=np.array(prefix, dtype=np.int32), k_tree=n(B, Hkv, T, D), v_tree=n(B, Hkv, T, D))


CASES = [
    # dtype, B, Hq, Hkv, tree, D, Lmax, prefix
    ("f32", 1, 4, 4, ("cartesian", (2, 3)), 64, 128, [128]),
    ("f32", 2, 4, 2, ("random", 17), 64, 100, [0, 100]),            # empty prefix, Lmax not a tile multiple
    ("bf16", 1, 8, 1, ("random", 1), 128, 130, [130]),              # root only
    ("bf16", 3, 6, 2, ("random", 70), 128, 300, [1, 150, 300]),     # two mask words
    ("bf16", 2, 2, 2, ("random", 130), 64, 64, [64, 7]),            # three mask words
    ("bf16", 1, 32, 32, ("sparse", (8, 4, 2, 1), 64, 64), 128, 1024, [1024]),
    ("bf16", 2, 4, 2, ("random", 200), 128, 700, [333, 700]),       # two tree tiles, four mask words
    ("bf16", 1, 2, 1, ("random", 130), 128, 257, [257]),            # second tree tile: one mask word
    ("bf16", 2, 2, 2, ("sparse", (8, 4, 2, 1), 64, 64), 128, 1024, [0, 1024]),   # 8 splits merged on chip; empty prefix
    # 64 prefix splits, too many to merge on chip: the combine kernel merges 40 partials of one
    # sequence and 1 of the other, four at a time with a running maximum across the groups
    ("bf16", 2, 2, 2, ("sparse", (8, 4, 2, 1), 64, 64), 128, 8192, [5000, 77]),
    # batches whose grid slots are ranked by prefix length (64 sequences, two per lane) and one
    # past the ranking's reach (65 sequences keep the grid order)
    ("bf16", 64, 1, 1, ("sparse", (8, 4, 2, 1), 64, 64), 128, 256,
     [int(x) for x in np.random.default_rng(64).integers(0, 257, 64)]),
    ("bf16", 65, 1, 1, ("sparse", (8, 4, 2, 1), 64, 64), 128, 256,
     [int(x) for x in np.random.default_rng(65).integers(0, 257, 65)]),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-B{c[1]}-H{c[2]}/{c[3]}-{c[4][0]}-L{c[6]}" for c in CASES])
def test_attention_matches_oracle(case):
    st = lib()
    dtype, B, Hq, Hkv, tspec, D, Lmax, prefix = case
    rng = np.random.default_rng(zlib.crc32(str(case).encode()))
    if tspec[0] == "random":
        parent, rank = wl.random_tree(rng, tspec[1], max_children=4)
    else:
        parent, rank = wl.make_tree(tspec)
    tree = st.spec_tree_build(parent, rank)
    x = _rand_inputs(rng, dtype, B, Hq, Hkv, len(parent), D, Lmax, prefix)
    out, lse = _run(st, x, tree, dtype)
    O, L = oracle.tree_attention(**x, tree=oracle.tree_encode(parent, rank), dtype=dtype)
    assert_close(out, O, dtype, "out")
    assert_close(lse, L, dtype, "lse")


@pytest.mark.parametrize("cfg,sample", [(1, None), (2, None), (4, 24), (5, 6)])
def test_attention_workloads(cfg, sample):
    """Full-size workloads; for the big ones the oracle computes a sample of (sequence, head) pairs."""
    st = lib()
    w = wl.WORKLOADS[cfg]
    parent, rank = wl.make_tree(w.tree)
    tree = st.spec_tree_build(parent, rank)
    x = wl.attention_inputs(w, len(parent))
    out, lse = _run(st, x, tree, w.dtype)
    heads = None
    if sample:
        rng = np.random.default_rng(cfg)
        pairs = [(b, h) for b in range(w.B) for h in range(w.Hq)]
        heads = [pairs[i] for i in rng.choice(len(pairs), size=sample, replace=False)]
    O, L = oracle.tree_attention(**x, tree=oracle.tree_encode(parent, rank), dtype=w.dtype, heads=heads)
    sel = ~np.isnan(L)
    assert sel.any()
    assert_close(out[sel], O[sel], w.dtype, "out")
    assert_close(lse[sel], L[sel], w.dtype, "lse")


def test_attention_dense_256_variant():
    st = lib()
    w = wl.WORKLOADS[5]
    p, r = wl.cartesian_tree((4, 4, 4, 4))
    parent, rank = wl.bfs_prefix_tree(p, r, 256)
    tree = st.spec_tree_build(parent, rank)
    x = wl.attention_inputs(w, 256)
    out, lse = _run(st, x, tree, w.dtype)
    O, L = oracle.tree_attention(**x, tree=oracle.tree_encode(parent, rank), dtype=w.dtype, heads=[(0, 0), (0, 31)])
    sel = ~np.isnan(L)
    assert_close(out[sel], O[sel], w.dtype, "out")


def test_attention_is_deterministic_and_respects_scale():
    st = lib()
    rng = np.random.default_rng(5)
    parent, rank = wl.cartesian_tree((3, 2))
    tree = st.spec_tree_build(parent, rank)
    x = _rand_inputs(rng, "f32", 2, 4, 2, len(parent), 64, 90, [90, 33])
    a, _ = _run(st, x, tree, "f32", scale=0.05)
    b, _ = _run(st, x, tree, "f32", scale=0.05)
    assert np.array_equal(a, b)
    O, _ = oracle.tree_attention(**x, tree=oracle.tree_encode(parent, rank), dtype="f32", scale=0.05)
    assert_close(a, O, "f32", "out")


@pytest.mark.parametrize("dtype,Hq,Hkv,T", [("bf16", 4, 2, 100), ("f32", 4, 2, 20), ("bf16", 8, 8, 3)])
def test_attention_ignores_cache_past_prefix(dtype, Hq, Hkv, T):
    """Cache slots at or past prefix_len[b] hold NaN: no output may depend on them."""
    st = lib()
    rng = np.random.default_rng(11 + T)
    parent, rank = wl.random_tree(rng, T, max_children=3)
    tree = st.spec_tree_build(parent, rank)
    Lmax, prefix = 520, [1, 200, 519]
    x = _rand_inputs(rng, dtype, len(prefix), Hq, Hkv, T, 128, Lmax, prefix)
    nan = wl.f32_to_bf16_bits(np.float32(np.nan)) if dtype == "bf16" else np.float32(np.nan)
    for b, L in enumerate(prefix):
        x["k_cache"][b, :, L:] = nan
        x["v_cache"][b, :, L:] = nan
    out, lse = _run(st, x, tree, dtype)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    clean = dict(x)
    clean["k_cache"] = x["k_cache"].copy()
    clean["v_cache"] = x["v_cache"].copy()
    for b, L in enumerate(prefix):
        clean["k_cache"][b, :, L:] = 0
        clean["v_cache"][b, :, L:] = 0
    O, Lse = oracle.tree_attention(**clean, tree=oracle.tree_encode(parent, rank), dtype=dtype)
    assert_close(out, O, dtype, "out")
    assert_close(lse, Lse, dtype, "lse")


def _sweep_cases(n=64, seed=2024):
    """Seeded random shapes over both paths: bf16 head dim 128 with >= 64 query rows per KV head
    (tensor cores: split plans of every kind, the K/V completion forms, fused or combined
    merges) and the CUDA-core path (fp32, or few rows)."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        dtype = "bf16" if rng.random() < 0.75 else "f32"
        Hkv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.choice([1, 2, 4, 8]))
        T = int(rng.integers(1, 400))
        D = 128 if dtype == "bf16" and rng.random() < 0.8 else 64
        B = int(rng.integers(1, 7))
        Lmax = int(rng.integers(1, 5000))
        prefix = [int(x) for x in rng.integers(0, Lmax + 1, size=B)]
        cases.append((i, dtype, B, Hkv * g, Hkv, T, D, Lmax, prefix))
    return cases


@pytest.mark.parametrize("case", _sweep_cases(), ids=lambda c: f"sweep{c[0]}-{c[1]}-B{c[2]}-H{c[3]}/{c[4]}-T{c[5]}-D{c[6]}-L{c[7]}")
def test_attention_random_sweep(case):
    """Element by element against the oracle on four sampled (sequence, head) pairs per shape."""
    st = lib()
    i, dtype, B, Hq, Hkv, T, D, Lmax, prefix = case
    rng = np.random.default_rng(1000 + i)
    parent, rank = wl.random_tree(rng, T, max_children=4)
    tree = st.spec_tree_build(parent, rank)
    x = _rand_inputs(rng, dtype, B, Hq, Hkv, len(parent), D, Lmax, prefix)
    out, lse = _run(st, x, tree, dtype)
    pairs = [(b, h) for b in range(B) for h in range(Hq)]
    heads = [pairs[j] for j in rng.choice(len(pairs), size=min(4, len(pairs)), replace=False)]
    O, L = oracle.tree_attention(**x, tree=oracle.tree_encode(parent, rank), dtype=dtype, heads=heads)
    sel = ~np.isnan(L)
    assert sel.any()
    assert_close(out[sel], O[sel], dtype, "out")
    assert_close(lse[sel], L[sel], dtype, "lse")
