"""Draft heads: CUDA path vs the oracle (GPU).

Tokens must match exactly, except at near ties of the top-k: a token that
differs must score, in the oracle's own logits row, within 1e-6 (fp32 inputs)
or 1e-3 x |logit| (bf16 inputs) of the oracle's pick for that rank; such ties
are counted.  The oracle is re-run teacher-forced on the GPU's tokens so later
depths stay comparable.  Logits and log-probabilities within the tolerances.
"""

import numpy as np
import pytest

import oracle
import spec_workloads as wl
from gpu_util import assert_close, lib, to_dev

pytestmark = pytest.mark.gpu


def _run(st, x, tree):
    return st.hydra_draft(to_dev(x["h"]), to_dev(x["E"]), [to_dev(a) for a in x["W1"]],
                          None if x["b1"] is None else [to_dev(a) for a in x["b1"]],
                          [to_dev(a) for a in x["W2"]], list(x["cond"]), list(x["topk"]), to_dev(x["root_tok"]), tree)


def _compare(st, x, parent, rank, dtype):
    tree = st.spec_tree_build(parent, rank)
    tok, logit, logprob = _run(st, x, tree)
    to = oracle.tree_encode(parent, rank)
    ref_fn = lambda teacher: oracle.hydra_draft(x["h"], x["E"], x["W1"], x["b1"], x["W2"], x["cond"], x["topk"],
                                                x["root_tok"], to, dtype, teacher_tok=teacher, keep_logits=True)
    return _check(tok, logit, logprob, ref_fn, parent, dtype, x["root_tok"])


def _check(tok, logit, logprob, ref_fn, parent, dtype, root_tok):
    tok, logit, logprob = tok.cpu().numpy(), logit.cpu().numpy(), logprob.cpu().numpy()
    ref = ref_fn(tok)
    B, T = tok.shape
    near = 0        # children whose token differs from the oracle's pick (allowed only at near ties)
    tied = 0        # children whose rank the oracle itself sees within the tolerance of a neighbour rank
    for b in range(B):
        for c in range(1, T):
            row = ref["logits"].get((b, int(parent[c])))
            assert row is not None, (b, c)
            tol = 1e-6 if dtype == "f32" else 1e-3 * abs(ref["node_logit"][b, c]) + 1e-6
            r = int(np.flatnonzero(np.argsort(-row, kind="stable") == ref["node_tok"][b, c])[0])
            srt = np.sort(row)[::-1]
            if (r > 0 and srt[r - 1] - srt[r] <= tol) or (r + 1 < srt.size and srt[r] - srt[r + 1] <= tol):
                tied += 1
            if tok[b, c] == ref["node_tok"][b, c]:
                continue
            # a different token is only acceptable at a near tie: in the oracle's own row
            # it must score within the tie tolerance of the oracle's pick for that rank
            diff = abs(row[tok[b, c]] - row[ref["node_tok"][b, c]])
            assert diff <= tol, (b, c, tok[b, c], ref["node_tok"][b, c], diff, tol)
            near += 1
    # differing picks can only sit at ranks the oracle's own logits leave tied
    assert near <= tied, (near, tied)
    assert tok[:, 0].tolist() == list(root_tok)
    assert_close(logit, ref["node_logit"], dtype, "node_logit")
    assert_close(logprob, ref["node_logprob"], dtype, "node_logprob")
    return near


def test_draft_tiny_fp32_workload():
    st = lib()
    w = wl.WORKLOADS[1]
    parent, rank = wl.make_tree(w.tree)
    _compare(st, wl.draft_inputs(w), parent, rank, "f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [
    # d, V, B, branching, cond, topk
    (64, 500, 2, (3, 2, 2), (0, 1, 1), (3, 2, 2)),
    (128, 4099, 3, (4, 1), (1, 1), (5, 1)),           # vocab not a tile multiple, top-k above the ranks used
    (32, 64, 1, (8, 4), (1, 0), (8, 16)),             # Medusa head at depth 2, top-16
])
def test_draft_small_shapes(dtype, shape):
    st = lib()
    d, V, B, branching, cond, topk = shape
    w = wl.Workload("t", dtype, B=B, seed=11, tree=("cartesian", branching), d=d, V=V, cond=cond, topk=topk)
    parent, rank = wl.make_tree(w.tree)
    x = wl.draft_inputs(w)
    # larger weights than the workloads' 0.02 so the logits spread and ties are rare
    rng = np.random.default_rng(3)
    enc = (lambda a: wl.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    x["W2"] = [enc(rng.standard_normal(np.shape(a), dtype=np.float32) * np.float32(0.25)) for a in x["W2"]]
    _compare(st, x, parent, rank, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [
    # d, V, B, branching, cond, topk: all-ancestor conditioning (cond 2), alone and mixed
    (64, 500, 2, (3, 2, 2), (2, 2, 2), (3, 2, 2)),
    (64, 700, 2, (2, 2, 2, 2), (1, 2, 1, 2), (2, 2, 2, 2)),
    (32, 300, 3, (3, 3), (2, 1), (3, 3)),
    (256, 4099, 2, (4, 2, 2), (0, 2, 2), (4, 2, 2)),   # rows of 3d and 4d on the tensor-core path (bf16)
])
def test_draft_all_ancestor_conditioning(dtype, shape):
    st = lib()
    d, V, B, branching, cond, topk = shape
    if dtype == "f32" and d > 128:
        # the wide-row case targets the bf16 tensor-core path; at d = 256 with these enlarged
        # weights the fp32 log-probs reach magnitudes where the fixed 1e-5 tolerance is
        # below fp32 rounding, so the fp32 path is covered by the d <= 128 shapes
        pytest.skip("bf16 tensor-core shape")
    w = wl.Workload("t", dtype, B=B, seed=17, tree=("cartesian", branching), d=d, V=V, cond=cond, topk=topk)
    parent, rank = wl.make_tree(w.tree)
    x = wl.draft_inputs(w)
    rng = np.random.default_rng(5)
    enc = (lambda a: wl.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    x["W2"] = [enc(rng.standard_normal(np.shape(a), dtype=np.float32) * np.float32(0.25)) for a in x["W2"]]
    x["E"] = enc(rng.standard_normal(np.shape(x["E"]), dtype=np.float32))   # embeddings that move the heads
    _compare(st, x, parent, rank, dtype)


def test_draft_shared_vocabulary_projection():
    # Medusa-2 style: every head projects with the same W2 (one array for all heads)
    st = lib()
    w = wl.Workload("t", "bf16", B=2, seed=18, tree=("sparse", (8, 4, 2, 1), 64, 64), d=256, V=4000,
                    cond=(1, 1, 1, 1), topk=(8, 4, 2, 1))
    parent, rank = wl.make_tree(w.tree)
    x = wl.draft_inputs(w)
    rng = np.random.default_rng(6)
    shared = wl.f32_to_bf16_bits(rng.standard_normal((w.V, w.d), dtype=np.float32) * np.float32(0.25))
    x["W2"] = [shared] * 4
    tree = st.spec_tree_build(parent, rank)
    W2d = to_dev(shared)
    tok, logit, logprob = st.hydra_draft(to_dev(x["h"]), to_dev(x["E"]), [to_dev(a) for a in x["W1"]],
                                         [to_dev(a) for a in x["b1"]], [W2d] * 4, list(x["cond"]), list(x["topk"]),
                                         to_dev(x["root_tok"]), tree)
    ref = oracle.hydra_draft(x["h"], x["E"], x["W1"], x["b1"], x["W2"], x["cond"], x["topk"], x["root_tok"],
                             oracle.tree_encode(parent, rank), "bf16", teacher_tok=tok.cpu().numpy())
    assert_close(logit.cpu().numpy(), ref["node_logit"], "bf16", "node_logit")
    _compare(st, x, parent, rank, "bf16")


def test_draft_on_sparse_tree_with_missing_ranks():
    # pruned tree: some parents keep children of ranks {0, 2}, so top-k > children
    st = lib()
    w = wl.Workload("t", "bf16", B=2, seed=12, tree=("sparse", (8, 4, 2, 1), 64, 64), d=128, V=3000,
                    cond=(1, 1, 1, 1), topk=(8, 4, 2, 1))
    parent, rank = wl.make_tree(w.tree)
    x = wl.draft_inputs(w)
    rng = np.random.default_rng(4)
    x["W2"] = [wl.f32_to_bf16_bits(rng.standard_normal(np.shape(a), dtype=np.float32) * np.float32(0.25)) for a in x["W2"]]
    _compare(st, x, parent, rank, "bf16")


def test_draft_hydra_heads_workload():
    """The Hydra-heads workload at full size: B=4, d=4096, V=32000, 4 heads, 64-node tree."""
    st = lib()
    w = wl.WORKLOADS[3]
    parent, rank = wl.make_tree(w.tree)
    near = _compare(st, wl.draft_inputs(w), parent, rank, "bf16")
    print(f"hydra heads workload: {near} near ties")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_init_heads_reproduce_lm_head_on_gpu(dtype):
    # Medusa Heads page: zeroed feed-forward + copied lm_head -> each head predicts lm_head's top token.
    st = lib()
    d, V, K = 256, 1000, 3
    rng = np.random.default_rng(6)
    lm = rng.standard_normal((V, d), dtype=np.float32) * np.float32(0.02)
    h = rng.standard_normal((1, d), dtype=np.float32)
    enc = (lambda a: wl.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    lm, h = enc(lm), enc(h)
    zw = enc(np.zeros((d, d), dtype=np.float32))
    zb = enc(np.zeros(d, dtype=np.float32))
    parent, rank = wl.chain_tree(K + 1)
    x = dict(h=h, E=lm, W1=[zw] * K, b1=[zb] * K, W2=[lm] * K, cond=np.zeros(K, np.int32), topk=np.ones(K, np.int32),
             root_tok=np.array([0], dtype=np.int32))
    tree = st.spec_tree_build(parent, rank)
    tok, logit, _ = _run(st, x, tree)
    dec = oracle.bf16_bits_to_f64 if dtype == "bf16" else (lambda a: a.astype(np.float64))
    ref = dec(lm) @ dec(h)[0]
    assert tok.cpu().numpy()[0, 1:].tolist() == [int(np.argmax(ref))] * K
    assert_close(logit.cpu().numpy()[0, 1:], [ref.max()] * K, dtype, "logit")


def test_medusa_sibling_sets_repeat_on_gpu():
    st = lib()
    w = wl.Workload("t", "f32", B=2, seed=13, tree=("cartesian", (3, 4)), d=64, V=300, cond=(0, 0), topk=(3, 4))
    parent, rank = wl.make_tree(w.tree)
    tree = st.spec_tree_build(parent, rank)
    tok, _, _ = _run(st, wl.draft_inputs(w), tree)
    tok = tok.cpu().numpy()
    to = oracle.tree_encode(parent, rank)
    for b in range(2):
        sets = [tuple(tok[b, to["children"][u]]) for u in to["children"][0]]
        assert all(s == sets[0] for s in sets)


@pytest.mark.parametrize("dtype,d,V,hidden", [("f32", 64, 500, 96), ("bf16", 64, 700, 128), ("bf16", 256, 4099, 512)])
def test_draft_layernorm_fusion_heads(dtype, d, V, hidden):
    # the head form the Hydra Guide prints as code: head 1 Linear -> SiLU -> LayerNorm (no W1b),
    # later heads Linear -> SiLU -> Linear -> LayerNorm on [h || E[...]], bias-free projection
    st = lib()
    rng = np.random.default_rng(d + hidden)
    enc = (lambda a: wl.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    n = lambda *shape, sc=1.0: enc(rng.standard_normal(shape, dtype=np.float32) * np.float32(sc))
    parent, rank = wl.make_tree(("cartesian", (3, 2, 2)))
    B = 2
    x = {"h": n(B, d), "E": n(V, d), "root_tok": rng.integers(0, V, size=B).astype(np.int32)}
    heads = [dict(form=1, cond=0, topk=3, W1=n(d, d, sc=0.1), b1=n(d, sc=0.1), gamma=n(d), beta=n(d, sc=0.1),
                  W2=n(V, d, sc=0.25)),
             dict(form=1, cond=1, topk=2, W1=n(hidden, 2 * d, sc=0.1), b1=n(hidden, sc=0.1), W1b=n(d, hidden, sc=0.1),
                  b1b=n(d, sc=0.1), gamma=n(d), beta=None, W2=n(V, d, sc=0.25)),
             dict(form=1, cond=2, topk=2, W1=n(hidden, 3 * d, sc=0.1), b1=None, W1b=n(d, hidden, sc=0.1), b1b=None,
                  gamma=None, beta=n(d, sc=0.1), W2=n(V, d, sc=0.25))]
    tree = st.spec_tree_build(parent, rank)
    dev_heads = [{k: (to_dev(v) if isinstance(v, np.ndarray) else v) for k, v in hd.items()} for hd in heads]
    tok, logit, logprob = st.hydra_draft_heads(to_dev(x["h"]), to_dev(x["E"]), dev_heads, to_dev(x["root_tok"]), tree)
    to = oracle.tree_encode(parent, rank)
    ref_fn = lambda teacher: oracle.hydra_draft_heads(x["h"], x["E"], heads, x["root_tok"], to, dtype,
                                                      teacher_tok=teacher, keep_logits=True)
    _check(tok, logit, logprob, ref_fn, parent, dtype, x["root_tok"])


def test_draft_heads_form0_matches_hydra_draft():
    # the description entry point with form-0 heads reproduces hydra_draft bit for bit
    st = lib()
    w = wl.Workload("t", "bf16", B=2, seed=19, tree=("sparse", (8, 4, 2, 1), 64, 64), d=128, V=3000,
                    cond=(1, 2, 1, 2), topk=(8, 4, 2, 1))
    parent, rank = wl.make_tree(w.tree)
    x = wl.draft_inputs(w)
    tree = st.spec_tree_build(parent, rank)
    a = _run(st, x, tree)
    heads = [dict(form=0, cond=int(x["cond"][k]), topk=int(x["topk"][k]), W1=to_dev(x["W1"][k]), b1=to_dev(x["b1"][k]),
                  W2=to_dev(x["W2"][k])) for k in range(4)]
    b = st.hydra_draft_heads(to_dev(x["h"]), to_dev(x["E"]), heads, to_dev(x["root_tok"]), tree)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u.cpu().numpy(), v.cpu().numpy())


def test_draft_layernorm_heads_vicuna7b_shape():
    # the LayerNorm fusion head form at full size: d 4096, V 32000, inner width 1024, batch 1,
    # the 64-node sparse tree (head 1 without W1b, heads 2-4 conditioned with W1b)
    st = lib()
    rng = np.random.default_rng(47)
    d, V, hidden = 4096, 32000, 1024
    n = lambda *shape, sc=0.02: wl.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(sc))
    parent, rank = wl.make_tree(("sparse", (8, 4, 2, 1), 64, 64))
    x = {"h": n(1, d, sc=1.0), "E": n(V, d), "root_tok": rng.integers(0, V, size=1).astype(np.int32)}
    heads = [dict(form=1, cond=0, topk=8, W1=n(d, d), b1=n(d), gamma=n(d, sc=1.0), beta=n(d), W2=n(V, d))]
    for tk in (4, 2, 1):
        heads.append(dict(form=1, cond=1, topk=tk, W1=n(hidden, 2 * d), b1=n(hidden), W1b=n(d, hidden), b1b=n(d),
                          gamma=n(d, sc=1.0), beta=n(d), W2=n(V, d)))
    tree = st.spec_tree_build(parent, rank)
    dev_heads = [{k: (to_dev(v) if isinstance(v, np.ndarray) else v) for k, v in hd.items()} for hd in heads]
    tok, logit, logprob = st.hydra_draft_heads(to_dev(x["h"]), to_dev(x["E"]), dev_heads, to_dev(x["root_tok"]), tree)
    to = oracle.tree_encode(parent, rank)
    ref_fn = lambda teacher: oracle.hydra_draft_heads(x["h"], x["E"], heads, x["root_tok"], to, "bf16",
                                                      teacher_tok=teacher, keep_logits=True)
    near = _check(tok, logit, logprob, ref_fn, parent, "bf16", x["root_tok"])
    print(f"layernorm heads at full size: {near} near ties")


# ---------------------------------------------------------------- folded first layers (hydra_draft_folded)

def _bf16_to_f64(a):
    a = np.asarray(a)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d,V", [(64, 500), (256, 4099), (4096, 1000)])
def test_fold_embedding_is_the_embedding_half_product(dtype, d, V):
    # tab[v, m] = sum_j W1[m, d + j] E[v, j]: the plain product in fp64 bounds the fp32 table by
    # the accumulation error, d * 2^-24 relative to sum_j |W1[m, d + j] E[v, j]|
    st = lib()
    rng = np.random.default_rng(30 + d)
    enc = (lambda a: wl.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    W1 = enc(rng.standard_normal((d, 2 * d), dtype=np.float32) * np.float32(0.05))
    E = enc(rng.standard_normal((V, d), dtype=np.float32))
    tab = st.hydra_fold_embedding(to_dev(W1), to_dev(E)).cpu().numpy().astype(np.float64)
    W1e, Ef = _bf16_to_f64(W1)[:, d:], _bf16_to_f64(E)
    ref = Ef @ W1e.T
    bound = d * 2.0 ** -24 * (np.abs(Ef) @ np.abs(W1e).T) + 1e-30
    assert np.all(np.abs(tab - ref) <= bound), np.max(np.abs(tab - ref) / bound)


def _run_folded(st, x, tree, fold_mask):
    W1 = [to_dev(a) for a in x["W1"]]
    E = to_dev(x["E"])
    tabs = [st.hydra_fold_embedding(W1[k], E) if (fold_mask[k] and x["cond"][k] == 1) else None
            for k in range(len(W1))]
    return st.hydra_draft(to_dev(x["h"]), E, W1, None if x["b1"] is None else [to_dev(a) for a in x["b1"]],
                          [to_dev(a) for a in x["W2"]], list(x["cond"]), list(x["topk"]), to_dev(x["root_tok"]), tree,
                          folded=tabs)


def _compare_folded(st, x, parent, rank, dtype, fold_mask=None):
    tree = st.spec_tree_build(parent, rank)
    K = len(x["W1"])
    tok, logit, logprob = _run_folded(st, x, tree, fold_mask or [True] * K)
    to = oracle.tree_encode(parent, rank)
    ref_fn = lambda teacher: oracle.hydra_draft(x["h"], x["E"], x["W1"], x["b1"], x["W2"], x["cond"], x["topk"],
                                                x["root_tok"], to, dtype, teacher_tok=teacher, keep_logits=True)
    return _check(tok, logit, logprob, ref_fn, parent, dtype, x["root_tok"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [
    # d, V, B, branching, cond, topk, which heads get a table
    (64, 500, 2, (3, 2, 2), (1, 1, 1), (3, 2, 2), (1, 1, 1)),
    (128, 4099, 3, (4, 1), (1, 1), (5, 1), (1, 1)),
    (64, 700, 2, (2, 2, 2, 2), (1, 2, 1, 0), (2, 2, 2, 2), (1, 1, 1, 1)),   # tables only act on cond-1 heads
    (256, 3000, 2, (3, 2, 2), (1, 1, 1), (3, 2, 2), (0, 1, 0)),             # folded and whole layers mixed
    (256, 3000, 1, (3, 2, 2), (1, 1, 1), (3, 2, 2), (1, 0, 1)),
    (64, 500, 10, (3, 2), (1, 1), (3, 2), (1, 1)),                          # more sequences than one MMA pass
    (200, 999, 3, (2, 2), (1, 1), (2, 2), (1, 1)),                          # d not a multiple of 16 or 64
])
def test_draft_folded_matches_oracle(dtype, shape):
    st = lib()
    d, V, B, branching, cond, topk, mask = shape
    if dtype == "f32" and d > 128:
        pytest.skip("bf16 tensor-core shape")
    w = wl.Workload("t", dtype, B=B, seed=21, tree=("cartesian", branching), d=d, V=V, cond=cond, topk=topk)
    parent, rank = wl.make_tree(w.tree)
    x = wl.draft_inputs(w)
    rng = np.random.default_rng(9)
    enc = (lambda a: wl.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    x["W2"] = [enc(rng.standard_normal(np.shape(a), dtype=np.float32) * np.float32(0.25)) for a in x["W2"]]
    x["E"] = enc(rng.standard_normal(np.shape(x["E"]), dtype=np.float32))   # embeddings that move the heads
    _compare_folded(st, x, parent, rank, dtype, list(mask))


def test_draft_folded_vicuna7b_workload():
    """The Vicuna-7B draft (B=1, d=4096, V=32000, 4 cond-1 heads, 64-node tree) with every head folded."""
    st = lib()
    w = wl.Workload("vicuna7b-draft", "bf16", B=1, seed=7, tree=wl.WORKLOADS[2].tree, d=4096, V=32000,
                    cond=(1, 1, 1, 1), topk=(8, 4, 2, 1))
    parent, rank = wl.make_tree(w.tree)
    near = _compare_folded(st, wl.draft_inputs(w), parent, rank, "bf16")
    print(f"vicuna7b folded: {near} near ties")


def test_draft_folded_hydra_heads_workload():
    """The Hydra-heads workload (B=4) folded: several sequences share each a[b] pass."""
    st = lib()
    w = wl.WORKLOADS[3]
    parent, rank = wl.make_tree(w.tree)
    near = _compare_folded(st, wl.draft_inputs(w), parent, rank, "bf16")
    print(f"hydra heads folded: {near} near ties")



@pytest.mark.parametrize("dtype,d,V,folded", [("bf16", 256, 32768, False), ("bf16", 256, 32768, True),
                                               ("f32", 64, 4096, False), ("f32", 64, 4096, True)])
def test_draft_exact_ties_take_the_lower_token(dtype, d, V, folded):
    """Every vocabulary row appears four times (tokens v, v + V/4, v + V/2, v + 3V/4), so each
    logit value is tied exactly four ways, across slices that different threads and warps of the
    select hold.  The method orders equal logits by token (the lower first): the top-8 of a row is
    the four copies of the largest value in token order, then the four of the second.  On the
    tensor-core path the copies sit a multiple of two weight tiles apart, where the projection
    walks K in the same order, so the GPU's logits of a tied group are equal bit for bit too
    (copies whose K order differed would tie only up to rounding, a near tie the other tests
    allow).  Distinct values stay far apart at this scale, so no pick may differ from the
    oracle's."""
    st = lib()
    q = V // 4
    w = wl.Workload("ties", dtype, B=2, seed=31, tree=("cartesian", (8, 4)), d=d, V=V, cond=(1, 1), topk=(8, 4))
    parent, rank = wl.make_tree(w.tree)
    x = wl.draft_inputs(w)
    rng = np.random.default_rng(31)
    enc = (lambda a: wl.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    for k in range(2):
        base = rng.standard_normal((q, d), dtype=np.float32) * np.float32(0.25)
        x["W2"][k] = enc(np.tile(base, (4, 1)))
    x["E"] = enc(rng.standard_normal(np.shape(x["E"]), dtype=np.float32))
    near = (_compare_folded(st, x, parent, rank, dtype) if folded else _compare(st, x, parent, rank, dtype))
    assert near == 0, near
    # the picks themselves: each parent's children carry tied tokens in increasing order
    tree = st.spec_tree_build(parent, rank)
    tok = (_run_folded(st, x, tree, [True, True]) if folded else _run(st, x, tree))[0].cpu().numpy()
    for b in range(2):
        for u in range(len(parent)):
            kids = [c for c in range(1, len(parent)) if parent[c] == u]
            kids.sort(key=lambda c: rank[c])
            t = [int(tok[b, c]) for c in kids]
            for i in range(0, len(t), 4):
                grp = t[i:i + 4]
                assert grp == sorted(grp) and len({g % q for g in grp}) == 1, (b, u, t)


def _draft_sweep(n=20, seed=77):
    """Seeded random draft shapes: width, vocabulary, batch, branching, conditioning and top-k,
    folded or not (bf16 widths of 128 and up take the tensor-core path)."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        dtype = "bf16" if rng.random() < 0.6 else "f32"
        d = int(rng.choice([64, 128, 256] if dtype == "bf16" else [32, 64, 96]))
        V = int(rng.integers(50, 6000))
        B = int(rng.integers(1, 4))
        K = int(rng.integers(1, 4))
        branching = tuple(int(x) for x in rng.integers(1, 5, size=K))
        cond = tuple(int(x) for x in rng.choice([0, 1, 2], size=K))
        topk = tuple(int(max(b, rng.integers(1, 9))) for b in branching)
        folded = bool(rng.random() < 0.3)
        cases.append((i, dtype, d, V, B, branching, cond, topk, folded))
    return cases


@pytest.mark.parametrize("case", _draft_sweep(), ids=lambda c: f"sweep{c[0]}-{c[1]}-d{c[2]}-V{c[3]}-B{c[4]}-K{len(c[5])}{'-fold' if c[8] else ''}")
def test_draft_random_sweep(case):
    st = lib()
    i, dtype, d, V, B, branching, cond, topk, folded = case
    w = wl.Workload("sweep", dtype, B=B, seed=500 + i, tree=("cartesian", branching), d=d, V=V, cond=cond, topk=topk)
    parent, rank = wl.make_tree(w.tree)
    x = wl.draft_inputs(w)
    rng = np.random.default_rng(900 + i)
    enc = (lambda a: wl.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    x["W2"] = [enc(rng.standard_normal(np.shape(a), dtype=np.float32) * np.float32(0.25)) for a in x["W2"]]
    x["E"] = enc(rng.standard_normal(np.shape(x["E"]), dtype=np.float32))
    if folded:
        _compare_folded(st, x, parent, rank, dtype)
    else:
        _compare(st, x, parent, rank, dtype)
