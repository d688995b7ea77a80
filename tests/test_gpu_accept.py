"""Acceptance: CUDA path vs the oracle (GPU).

Greedy is exact: the argmax compares the same float32 values on both sides.
Rejection: accepted lengths, paths and tokens must match the oracle bit for
bit except where the oracle's margin shows a decision within 1e-6 of its
threshold (|u - p/q| or the sampling draw vs a CDF breakpoint), which is
counted and reported.
"""

import numpy as np
import pytest

import oracle
from oracle.philox import acceptance_uniforms, philox_uniform_pair
import spec_workloads as wl
from conftest import read_golden
from gpu_util import lib, to_dev

pytestmark = pytest.mark.gpu


def _greedy(st, lp, tok, tree):
    a, p, n, m = st.tree_accept(0, to_dev(lp), None, to_dev(tok), tree)
    return a.cpu().numpy(), p.cpu().numpy(), n.cpu().numpy(), m.cpu().numpy()


def _reject(st, lp, lq, tok, tree, temp, seed, offset):
    a, p, n, m = st.tree_accept(1, to_dev(lp), to_dev(lq), to_dev(tok), tree, temperature=temp, seed=seed, offset=offset)
    return a.cpu().numpy(), p.cpu().numpy(), n.cpu().numpy(), m.cpu().numpy()


def test_philox_stream_matches_oracle():
    st = lib()
    for seed, offset in [(1234, 0), (0, 0), (2 ** 40 + 17, 2 ** 33 + 5)]:
        ua, us = st.spec_philox_uniform(seed, offset, 3, 50)
        ua, us = ua.cpu().numpy(), us.cpu().numpy()
        for b in range(3):
            for c in range(50):
                u0, u1 = philox_uniform_pair(seed, offset, c, b)
                assert ua[b, c] == u0
                if c == 0:
                    assert us[b] == u1


@pytest.mark.parametrize("cfg,trials", [(1, 300), (2, 256)])
def test_greedy_workloads(cfg, trials):
    st = lib()
    w = wl.WORKLOADS[cfg]
    parent, rank = wl.make_tree(w.tree)
    tree = st.spec_tree_build(parent, rank)
    x = wl.greedy_inputs(w, parent, B=trials)
    a, p, n, _ = _greedy(st, x["logits_p"], x["node_tok"], tree)
    ref = oracle.greedy_accept(x["logits_p"], x["node_tok"], oracle.tree_encode(parent, rank))
    assert np.array_equal(a, ref["accept_len"])
    assert np.array_equal(p, ref["accept_path"])
    assert np.array_equal(n, ref["next_token"])
    assert np.array_equal(a, x["planted"])


def test_greedy_with_exact_ties():
    st = lib()
    rng = np.random.default_rng(21)
    for trial in range(12):
        T = int(rng.integers(1, 200))
        V = int(rng.integers(2, 7))
        parent, rank = wl.random_tree(rng, T, max_children=3)
        tree = st.spec_tree_build(parent, rank)
        B = 17
        tok = rng.integers(0, V, size=(B, T)).astype(np.int32)
        lp = rng.integers(-2, 3, size=(B, T, V)).astype(np.float32)
        a, p, n, m = _greedy(st, lp, tok, tree)
        ref = oracle.greedy_accept(lp, tok, oracle.tree_encode(parent, rank))
        assert np.array_equal(a, ref["accept_len"])
        assert np.array_equal(p, ref["accept_path"])
        assert np.array_equal(n, ref["next_token"])
        assert np.array_equal(m, ref["margin"].astype(np.float32))


def _compare_rejection(st, lp, lq, tok, parent, rank, temp, seed, offset):
    tree = st.spec_tree_build(parent, rank)
    a, p, n, m = _reject(st, lp, lq, tok, tree, temp, seed, offset)
    B, T, _ = lp.shape
    ua, us = acceptance_uniforms(seed, offset, B, T)
    ref = oracle.rejection_accept(lp, lq, tok, oracle.tree_encode(parent, rank), temp, ua, us)
    near = 0
    for b in range(B):
        if ref["margin_decide"][b] < 1e-6:
            near += 1
            continue
        assert a[b] == ref["accept_len"][b], b
        assert np.array_equal(p[b], ref["accept_path"][b]), b
        if ref["margin_sample"][b] < 1e-6:
            near += 1
            continue
        assert n[b] == ref["next_token"][b], (b, n[b], ref["next_token"][b])
    return near, a


def test_rejection_long_context_workload():
    """The long-context stochastic workload: dense 341-node tree, V = 32000, T = 0.7, seed 1234, over 32 offsets."""
    st = lib()
    w = wl.WORKLOADS[5]
    parent, rank = wl.make_tree(w.tree)
    x = wl.rejection_inputs(w, parent, rank)
    near_total = 0
    lens = []
    for offset in range(32):
        near, a = _compare_rejection(st, x["logits_p"], x["logits_q"], x["node_tok"], parent, rank, w.temperature,
                                     w.philox_seed, offset)
        near_total += near
        lens.append(int(a[0]))
    assert near_total <= 2
    print(f"long-context rejection: accepted lengths over 32 offsets {lens}, near-threshold decisions {near_total}")


@pytest.mark.parametrize("V,temp", [(7, 1.0), (50, 0.7), (1000, 1.3)])
def test_rejection_random_trees(V, temp):
    st = lib()
    rng = np.random.default_rng(V)
    for trial in range(4):
        T = int(rng.integers(2, 120))
        parent, rank = wl.random_tree(rng, T, max_children=3)
        B = 64
        lq = rng.standard_normal((B, T, V), dtype=np.float32) * np.float32(2.0)
        lp = (np.float32(0.8) * lq + np.float32(0.6) * rng.standard_normal((B, T, V), dtype=np.float32)) * np.float32(2.0)
        tok = wl.sibling_tokens(rng, parent, B, V) if V >= 4 else rng.integers(0, V, size=(B, T)).astype(np.int32)
        near, _ = _compare_rejection(st, lp.astype(np.float32), lq, tok, parent, rank, temp, 99 + trial, trial)
        assert near <= 2


def test_rejection_equal_distributions_accept_all():
    st = lib()
    rng = np.random.default_rng(7)
    parent, rank = wl.cartesian_tree((2, 2))
    tree = st.spec_tree_build(parent, rank)
    lp = rng.standard_normal((8, len(parent), 40), dtype=np.float32)
    tok = wl.sibling_tokens(rng, parent, 8, 40)
    a, p, n, _ = _reject(st, lp, lp.copy(), tok, tree, 0.7, 5, 0)
    assert a.tolist() == [2] * 8
    assert all(list(p[b]) == [0, 1, 3] for b in range(8))


def test_rejection_worked_example_on_gpu():
    # "Speculative Decoding", "A worked example": p/q per drafted token; coin at "on" rejects.
    st = lib()
    rows = read_golden("speculative_decoding_worked_example.txt")
    toks = [r for r in rows if len(r) == 4]
    V, T = 8, 6
    P = np.zeros((T, V))
    Q = np.zeros((T, V))
    for pos, r in enumerate(toks):
        p = float(r[1]) if r[1] != "-" else 0.2
        q = float(r[2]) if r[2] != "-" else 0.2
        P[pos], Q[pos] = (1 - p) / 7, (1 - q) / 7
        P[pos, pos + 1], Q[pos, pos + 1] = p, q
    P[T - 1] = Q[T - 1] = 1.0 / V
    parent, rank = wl.chain_tree(T)
    tree = st.spec_tree_build(parent, rank)
    tok = np.arange(T, dtype=np.int32)[None]
    lp = np.log(P)[None].astype(np.float32)
    lq = np.log(Q)[None].astype(np.float32)
    # find offsets whose coin at "on" (node 4) is >= p/q (a rejection) and whose other coins accept
    hits = 0
    for offset in range(200):
        us = [philox_uniform_pair(0, offset, c, 0)[0] for c in range(T)]
        if not (us[4] >= 0.34 and all(us[c] < 0.999 for c in (1, 2, 3))):
            continue
        a, p, n, _ = _reject(st, lp, lq, tok, tree, 1.0, 0, offset)
        assert a[0] == 3 and list(p[0]) == [0, 1, 2, 3, -1, -1]
        assert P[3, n[0]] > Q[3, n[0]] and n[0] != 4     # drawn from max(0, p - q), never "on"
        hits += 1
    assert hits >= 50


def test_rejection_outputs_follow_target_on_gpu():
    # Chi-square on the GPU kernel: depth-1 chains, drafts drawn from q, output token distribution = p.
    st = lib()
    rng = np.random.default_rng(31)
    V = 8
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    parent, rank = wl.chain_tree(2)
    tree = st.spec_tree_build(parent, rank)
    B = 32000
    counts = np.zeros(V, dtype=np.int64)
    lp = np.broadcast_to(np.log(np.stack([p, p])).astype(np.float32), (B, 2, V)).copy()
    lq = np.broadcast_to(np.log(np.stack([q, q])).astype(np.float32), (B, 2, V)).copy()
    for offset in range(3):
        tok = np.zeros((B, 2), dtype=np.int32)
        tok[:, 1] = rng.choice(V, size=B, p=q)
        a, _, n, _ = _reject(st, lp, lq, tok, tree, 1.0, 777, offset)
        first = np.where(a >= 1, tok[:, 1], n)
        counts += np.bincount(first, minlength=V)
    e = counts.sum() * p
    chi2 = ((counts - e) ** 2 / e).sum()
    assert chi2 < 24.3, chi2   # 7 dof, p = 0.001


def test_out_of_vocabulary_token_is_flagged():
    st = lib()
    import torch
    parent, rank = wl.chain_tree(3)
    tree = st.spec_tree_build(parent, rank)
    V = 16
    lp = np.zeros((1, 3, V), dtype=np.float32)
    tok = np.array([[0, 99, 1]], dtype=np.int32)
    ws = torch.zeros(st.tree_accept_workspace_size(1, tree, 1, V), dtype=torch.uint8, device="cuda")
    a, p, n, _ = st.tree_accept(1, to_dev(lp), to_dev(lp), to_dev(tok), tree, temperature=1.0, ws=ws)
    assert st.spec_read_device_status(ws) == 1      # SPEC_EINVAL recorded on the device
    assert int(a.cpu()[0]) == 0


def test_rejection_vocabulary_past_the_walk_cache():
    """V = 50000: above the 40,960 tokens whose draw weights the rejection walk keeps in shared
    memory, so the draw recomputes them from the logits on every scan."""
    st = lib()
    rng = np.random.default_rng(50000)
    V, B, temp = 50000, 6, 0.8
    parent, rank = wl.random_tree(rng, 40, max_children=3)
    T = len(parent)
    lq = rng.standard_normal((B, T, V), dtype=np.float32) * np.float32(2.0)
    lp = ((np.float32(0.8) * lq + np.float32(0.6) * rng.standard_normal((B, T, V), dtype=np.float32))
          * np.float32(2.0)).astype(np.float32)
    tok = wl.sibling_tokens(rng, parent, B, V)
    near_total = 0
    for offset in range(3):
        near, _ = _compare_rejection(st, lp, lq, tok, parent, rank, temp, 7, offset)
        near_total += near
    assert near_total <= 2


def _greedy_sweep(n=16, seed=31):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        T = int(rng.integers(1, 300))
        V = int(rng.choice([2, 3, 17, 1000, 32000, 50001]))
        B = int(rng.integers(1, 9))
        out.append((i, T, V, B))
    return out


@pytest.mark.parametrize("case", _greedy_sweep(), ids=lambda c: f"sweep{c[0]}-T{c[1]}-V{c[2]}-B{c[3]}")
def test_greedy_random_sweep(case):
    """Random trees, vocabularies (odd sizes and past 2^15) and batches, target logits planted to
    accept random paths, plus exact ties between the planted token and a rival: bit-exact."""
    st = lib()
    i, T, V, B = case
    rng = np.random.default_rng(100 + i)
    parent, rank = wl.random_tree(rng, T, max_children=4)
    T = len(parent)
    tree = st.spec_tree_build(parent, rank)
    tok = wl.sibling_tokens(rng, parent, B, V) if V >= 5 else rng.integers(0, V, size=(B, T)).astype(np.int32)
    lp = rng.standard_normal((B, T, V), dtype=np.float32)
    # plant: along a random path each node's row prefers its chosen child's token, some by an
    # exact tie with a lower-numbered rival (which then wins)
    for b in range(B):
        u = 0
        while True:
            kids = [c for c in range(1, T) if parent[c] == u]
            if not kids or rng.random() < 0.25:
                break
            c = kids[int(rng.integers(0, len(kids)))]
            top = float(lp[b, u].max()) + 1.0
            lp[b, u, tok[b, c]] = top
            if rng.random() < 0.3 and V > 1:
                rival = int(rng.integers(0, V))
                lp[b, u, rival] = top
            u = c
    a, p, n, _ = _greedy(st, lp, tok, tree)
    ref = oracle.greedy_accept(lp, tok, oracle.tree_encode(parent, rank))
    assert np.array_equal(a, ref["accept_len"])
    assert np.array_equal(p, ref["accept_path"])
    assert np.array_equal(n, ref["next_token"])
