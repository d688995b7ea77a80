"""Pins for the oracle's acceptance (CPU only).

Greedy: brute force over every root-to-leaf path (longest prefix matching the
target argmax) and the planted lengths of the workloads.  Rejection: the worked
example of the "Speculative Decoding" page, a chi-square test that outputs
follow p (with a planted mistake as negative control), the page's expected-
yield formula and its printed values, and the alpha = 1 special case.
"""

import numpy as np
import pytest

from conftest import read_golden
from oracle import tree_encode, greedy_accept, rejection_accept
import oracle.accept as oracle_accept
from oracle.philox import acceptance_uniforms
import spec_workloads as wl


# ---------------------------------------------------------------- greedy

def _brute_force_greedy(lp, node_tok, parent, children):
    """Longest root-to-leaf prefix whose tokens all equal the target argmax at their parent."""
    T = len(parent)
    best = (0, [0])
    leaves = [u for u in range(T) if not children[u]]
    for leaf in leaves:
        path = []
        u = leaf
        while u != -1:
            path.append(u)
            u = int(parent[u])
        path = path[::-1]
        n = 0
        for a, c in zip(path[:-1], path[1:]):
            if node_tok[c] != int(np.argmax(lp[a])):
                break
            n += 1
        cand = path[: n + 1]
        if n > best[0] or (n == best[0] and cand[-1] < best[1][-1]):
            best = (n, cand)
    return best


def test_greedy_equals_longest_matching_prefix():
    rng = np.random.default_rng(11)
    for trial in range(40):
        T = int(rng.integers(1, 30))
        V = int(rng.integers(2, 6))     # tiny vocabulary: many matches and ties
        parent, rank = wl.random_tree(rng, T, max_children=3)
        tree = tree_encode(parent, rank)
        B = 3
        node_tok = rng.integers(0, V, size=(B, T))
        lp = rng.integers(-2, 3, size=(B, T, V)).astype(np.float32)   # integer logits: exact ties
        out = greedy_accept(lp, node_tok, tree)
        for b in range(B):
            n, path = _brute_force_greedy(lp[b], node_tok[b], parent, tree["children"])
            assert out["accept_len"][b] == n
            assert list(out["accept_path"][b, : n + 1]) == path
            assert all(out["accept_path"][b, n + 1:] == -1)
            assert out["next_token"][b] == int(np.argmax(lp[b, path[-1]]))


@pytest.mark.parametrize("cfg,trials", [(1, 300), (2, 256)])
def test_planted_greedy_lengths(cfg, trials):
    w = wl.WORKLOADS[cfg]
    parent, rank = wl.make_tree(w.tree)
    tree = tree_encode(parent, rank)
    # the planting does not depend on the vocabulary size; a smaller one keeps this quick
    w = wl.Workload(**{**w.__dict__, "V": min(w.V, 2000)})
    x = wl.greedy_inputs(w, parent, B=trials, seed=100 + cfg)
    out = greedy_accept(x["logits_p"], x["node_tok"], tree)
    assert np.array_equal(out["accept_len"], x["planted"])
    counts = np.bincount(out["accept_len"], minlength=max(w.accept_lengths) + 1)[list(w.accept_lengths)]
    expected = trials / len(w.accept_lengths)
    assert ((counts - expected) ** 2 / expected).sum() < 16.3   # chi-square, <= 3 dof, p = 0.001
    if cfg == 2:
        assert abs(out["accept_len"].mean() - 2.5) < 0.25


# ---------------------------------------------------------------- rejection

def _chain_logits(V, rows):
    """Logit rows (natural log of the given probability rows)."""
    return np.log(np.asarray(rows, dtype=np.float64)).astype(np.float64)


def test_worked_example():
    rows = read_golden("speculative_decoding_worked_example.txt")
    toks = [r for r in rows if len(r) == 4]
    ratio_printed = float([r for r in rows if r[0] == "ratio_on"][0][1])
    n_acc = int([r for r in rows if r[0] == "accepted"][0][1])
    n_emit = int([r for r in rows if r[0] == "emitted"][0][1])
    # chain: root (the context) then the five drafted tokens; vocabulary of 8;
    # token ids 1..5 are the drafted words, the remaining mass goes to 0, 6, 7
    V, T = 8, 6
    parent, rank = wl.chain_tree(T)
    tree = tree_encode(parent, rank)
    P = np.full((T, V), np.nan)
    Q = np.full((T, V), np.nan)
    for pos, r in enumerate(toks):
        x = pos + 1
        p = float(r[1]) if r[1] != "-" else 0.2
        q = float(r[2]) if r[2] != "-" else 0.2
        rest_p, rest_q = (1 - p) / 7, (1 - q) / 7
        P[pos] = rest_p
        Q[pos] = rest_q
        P[pos, x], Q[pos, x] = p, q
        if r[3] == "reject":
            assert abs(p / q - ratio_printed) < 0.005
    # the spare leaf row (position after the last draft): any distribution
    P[T - 1] = Q[T - 1] = 1.0 / V
    node_tok = np.arange(T)[None]          # node i carries token i (node 0: the context)
    u_acc = np.array([[0.0, 0.99, 0.99, 0.99, 0.5, 0.01]])   # coin at "on": 0.5 >= 1/3, reject
    for u_s in np.linspace(0.0, 0.999, 25):
        out = rejection_accept(np.log(P)[None], np.log(Q)[None], node_tok, tree, 1.0, u_acc, [u_s])
        assert out["accept_len"][0] == n_acc
        assert list(out["accept_path"][0]) == [0, 1, 2, 3, -1, -1]
        assert n_acc + 1 == n_emit
        # the replacement comes from max(0, p - q) at the position of "on": never "on" itself
        x = out["next_token"][0]
        assert P[3, x] > Q[3, x] and x != 4


def _run_chain(P_rows, Q_rows, rng, trials, k):
    """Chains of k drafted tokens, each drawn from q; returns accept_len, next_token, drafted tokens."""
    V = P_rows.shape[-1]
    parent, rank = wl.chain_tree(k + 1)
    tree = tree_encode(parent, rank)
    T = k + 1
    drafts = np.stack([rng.choice(V, size=trials, p=Q_rows[i]) for i in range(k)], axis=1)
    node_tok = np.concatenate([np.zeros((trials, 1), dtype=np.int64), drafts], axis=1)
    lp = np.broadcast_to(np.log(P_rows), (trials, T, V))
    lq = np.broadcast_to(np.log(Q_rows), (trials, T, V))
    u_acc = rng.random((trials, T))
    u_smp = rng.random(trials)
    out = rejection_accept(lp, lq, node_tok, tree, 1.0, u_acc, u_smp)
    return out, node_tok


def _chi2_fit(counts, probs):
    n = counts.sum()
    e = n * probs
    return ((counts - e) ** 2 / e).sum()


def _pq(rng, V):
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    return p, q


def test_outputs_follow_target_chi_square():
    # "Speculative Decoding", "The correctness guarantee": min(p, q) accepted mass
    # plus (1 - alpha) times the normalised residual is exactly p.
    rng = np.random.default_rng(12)
    V, trials = 8, 100000
    p, q = _pq(rng, V)
    P = np.stack([p, p])
    Q = np.stack([q, q])
    out, toks = _run_chain(P, Q, rng, trials, 1)
    first = np.where(out["accept_len"] >= 1, toks[:, 1], out["next_token"])
    counts = np.bincount(first, minlength=V)
    assert _chi2_fit(counts, p) < 24.3     # chi-square, 7 dof, p = 0.001


def test_negative_control_resampling_from_p_is_detected(monkeypatch):
    # The page: resampling from p instead gives min(p, q) + (1 - alpha) p != p.
    # Plant that mistake in the oracle and check the chi-square test catches it.
    rng = np.random.default_rng(13)
    V, trials = 8, 100000
    p, q = _pq(rng, V)
    monkeypatch.setattr(oracle_accept, "_residual", lambda p_u, q_u: p_u.copy())
    out, toks = _run_chain(np.stack([p, p]), np.stack([q, q]), rng, trials, 1)
    first = np.where(out["accept_len"] >= 1, toks[:, 1], out["next_token"])
    counts = np.bincount(first, minlength=V)
    assert _chi2_fit(counts, p) > 24.3
    alpha = np.minimum(p, q).sum()
    wrong = np.minimum(p, q) + (1 - alpha) * p
    assert _chi2_fit(counts, wrong) < 24.3


def test_expected_yield_formula_and_examples():
    # "Speculative Decoding", "How much faster?": E[N] = (1 - a^(k+1)) / (1 - a),
    # limit k + 1 at a = 1; the page prints 3.4, 4.7 and 1.9 for its examples.
    for a, k, printed in read_golden("speculative_decoding_expected_yield.txt"):
        a, k, printed = float(a), int(k), float(printed)
        e = (k + 1) if a == 1.0 else (1 - a ** (k + 1)) / (1 - a)
        assert abs(e - sum(a ** i for i in range(k + 1))) < 1e-12
        assert round(e, 1) == printed or (a == 1.0 and e == printed)


@pytest.mark.parametrize("alpha_target,k", [(0.8, 4), (0.5, 4), (0.9, 5)])
def test_mean_yield_matches_formula(alpha_target, k):
    rng = np.random.default_rng(14 + k)
    V, trials = 6, 20000
    # q uniform over V; p puts mass alpha_target spread like q on the first tokens ...
    q = np.full(V, 1.0 / V)
    p = np.zeros(V)
    p[:-1] = alpha_target / (V - 1)
    p[-1] = 1 - alpha_target
    alpha = np.minimum(p, q).sum()
    P = np.tile(p, (k + 1, 1))
    Q = np.tile(q, (k + 1, 1))
    out, _ = _run_chain(P, Q, rng, trials, k)
    n = out["accept_len"] + 1
    expect = (1 - alpha ** (k + 1)) / (1 - alpha)
    assert abs(n.mean() - expect) < 4 * n.std() / np.sqrt(trials)


def test_equal_distributions_accept_everything():
    # alpha = 1: never rejects; the bonus comes from p at the deepest leaf (lowest index).
    rng = np.random.default_rng(15)
    parent, rank = wl.cartesian_tree((2, 2))
    tree = tree_encode(parent, rank)
    V = 20
    lp = rng.standard_normal((4, tree["T"], V))
    node_tok = wl.sibling_tokens(rng, parent, 4, V)
    u_acc, u_smp = acceptance_uniforms(7, 0, 4, tree["T"])
    out = rejection_accept(lp, lp.copy(), node_tok, tree, 0.7, u_acc, u_smp)
    assert list(out["accept_len"]) == [2] * 4
    assert all(list(out["accept_path"][b]) == [0, 1, 3] for b in range(4))


def test_temperature_applies_to_both():
    # scaling both logit sets by c and the temperature by c changes nothing
    rng = np.random.default_rng(16)
    parent, rank = wl.cartesian_tree((3, 2))
    tree = tree_encode(parent, rank)
    V, B = 30, 5
    lp = rng.standard_normal((B, tree["T"], V))
    lq = rng.standard_normal((B, tree["T"], V))
    tok = wl.sibling_tokens(rng, parent, B, V)
    u_acc, u_smp = acceptance_uniforms(3, 9, B, tree["T"])
    a = rejection_accept(lp, lq, tok, tree, 0.5, u_acc, u_smp)
    b = rejection_accept(lp * 4, lq * 4, tok, tree, 2.0, u_acc, u_smp)
    for key in ("accept_len", "accept_path", "next_token"):
        assert np.array_equal(a[key], b[key])


# ---------------------------------------------------------------- reporting margins, computed by hand

def test_greedy_margin_by_hand():
    # chain root -> 1 -> 2, V = 4, integer logits so every gap is exact:
    # row 0 argmax token 1 (gap 5 - 2 = 3); node 1 carries token 1: accepted.
    # row 1 argmax token 0 (gap 4 - 3.5 = 0.5); node 2 carries token 2: rejected,
    # so row 2's gap (9) is not an accepted node's and does not count.
    parent, rank = wl.chain_tree(3)
    tree = tree_encode(parent, rank)
    lp = np.array([[[0.0, 5.0, 2.0, 1.0], [4.0, 1.0, 3.5, 0.0], [9.0, 0.0, 0.0, 0.0]]])
    out = greedy_accept(lp, np.array([[7, 1, 2]]), tree)
    assert out["accept_len"][0] == 1 and out["next_token"][0] == 0
    assert out["margin"][0] == 0.5


def test_rejection_margins_by_hand():
    # root with one child carrying token 0; V = 2, temperature 1; p_0 = (.3, .7), q_0 = (.6, .4):
    # the edge's ratio is .3 / .6 = .5
    parent, rank = wl.chain_tree(2)
    tree = tree_encode(parent, rank)
    lp = np.log(np.array([[[0.3, 0.7], [0.25, 0.75]]]))
    lq = np.log(np.array([[[0.6, 0.4], [0.5, 0.5]]]))
    tok = np.array([[5, 0]])
    # u_c = .45 < .5: accepted, |u - ratio| = .05; the child is a leaf, so the draw is from
    # p_1 = (.25, .75): u' = .1 -> t = .1, CDF (.25, 1): token 0, nearest breakpoint .15 away
    out = rejection_accept(lp, lq, tok, tree, 1.0, np.array([[0.0, 0.45]]), np.array([0.1]))
    assert out["accept_len"][0] == 1 and out["next_token"][0] == 0
    assert abs(out["margin_decide"][0] - 0.05) < 1e-12
    assert abs(out["margin_sample"][0] - 0.15) < 1e-12
    assert abs(out["margin"][0] - 0.05) < 1e-12
    # u_c = .9 >= .5: rejected, |u - ratio| = .4; the draw is from the residual at the root,
    # max(p_0 - q_0, 0) = (0, .3), total .3: u' = .5 -> t = .15, CDF (0, .3): token 1,
    # nearest breakpoint .15 away, .5 of the total
    out = rejection_accept(lp, lq, tok, tree, 1.0, np.array([[0.0, 0.9]]), np.array([0.5]))
    assert out["accept_len"][0] == 0 and out["next_token"][0] == 1
    assert abs(out["margin_decide"][0] - 0.4) < 1e-12
    assert abs(out["margin_sample"][0] - 0.5) < 1e-12
    assert abs(out["margin"][0] - 0.4) < 1e-12
