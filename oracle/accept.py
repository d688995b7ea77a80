"""Acceptance over a candidate tree (oracle; test infrastructure only).

Greedy.  Hydra Guide, section "Parallel Verification and Greedy Acceptance
Algorithm": at an accepted position the target's argmax is the next token; if
it equals the token of a child on the current branch the walk advances there;
it halts when no child matches, and the target's token at the halt node is
emitted too, so a branch of length m yields m + 1 tokens.  "Medusa Heads",
section "Tree Attention und Akzeptanz": a candidate is accepted when it equals
the model's best choice and the longest accepted branch is kept.

Rejection.  "Speculative Decoding", sections "The acceptance criterion", "The
correctness guarantee", "How much faster?" and "A worked example": a draft
token x is accepted when p(x) >= q(x), else with probability p(x)/q(x); on a
rejection one token is drawn from norm(max(0, p - q)) and everything after is
discarded; when every draft is accepted a bonus token is drawn from p at the
next position.  p and q are the post-temperature distributions.

On a tree the pages give no more than the chain rule plus "keep the longest
accepted path".  Read here as: every edge (parent -> child c) is tested
independently with its own uniform u_c; a node is accepted when its parent is
and its edge passes; the deepest accepted node u* wins (lowest index on equal
depth); if u* has children (all of them were rejected) the extra token is drawn
from the residual max(p_u* - q_u*, 0), normalised (from p_u* if that residual
is all zero, the alpha = 1 case), else from p_u*.  Drawing is by inverse CDF in
ascending token order: the smallest x whose running sum exceeds u' * total.
On chains this is exactly the page's rule.
"""

import numpy as np


def _deepest(accepted, depth):
    best = 0
    for u in range(len(accepted)):
        if accepted[u] and depth[u] > depth[best]:
            best = u
    return best  # first (lowest) index among the deepest, since the scan is ascending


def _path_to(u, parent):
    path = []
    while u != -1:
        path.append(u)
        u = int(parent[u])
    return path[::-1]


def greedy_accept(logits_p, node_tok, tree):
    """Greedy longest accepted path.

    logits_p [B, T, V]: the target's logits at every tree node (row u predicts
    the token after u); node_tok [B, T].

    Returns dict: accept_len [B] (m), accept_path [B, max_depth + 1] (node ids
    root first, -1 padded), next_token [B] (target argmax at u*), margin [B]
    (smallest top-1 minus top-2 logit gap over the accepted nodes).
    """
    lp = np.asarray(logits_p, dtype=np.float64)
    B, T, V = lp.shape
    parent, depth = tree["parent"], tree["depth"]
    node_tok = np.asarray(node_tok, dtype=np.int64).reshape(B, T)
    maxd = tree["max_depth"]
    accept_len = np.zeros(B, dtype=np.int64)
    accept_path = np.full((B, maxd + 1), -1, dtype=np.int64)
    next_token = np.zeros(B, dtype=np.int64)
    margin = np.full(B, np.inf)
    for b in range(B):
        a = np.argmax(lp[b], axis=1)  # first maximum: ties go to the lowest token id
        accepted = np.zeros(T, dtype=bool)
        accepted[0] = True
        for c in range(1, T):
            accepted[c] = accepted[parent[c]] and node_tok[b, c] == a[parent[c]]
        u = _deepest(accepted, depth)
        path = _path_to(u, parent)
        accept_len[b] = depth[u]
        accept_path[b, : len(path)] = path
        next_token[b] = a[u]
        for v in np.nonzero(accepted)[0]:
            top2 = np.sort(lp[b, v])[-2:] if V >= 2 else np.array([-np.inf, lp[b, v, 0]])
            margin[b] = min(margin[b], top2[1] - top2[0])
    return {"accept_len": accept_len, "accept_path": accept_path,
            "next_token": next_token, "margin": margin}


def _residual(p_u, q_u):
    """max(p - q, 0), unnormalised ("Speculative Decoding", "The acceptance criterion")."""
    return np.maximum(p_u - q_u, 0.0)


def _log_softmax(z):
    m = z.max(axis=-1, keepdims=True)
    return z - (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))


def rejection_accept(logits_p, logits_q, node_tok, tree, temperature, u_accept, u_sample):
    """min(1, p/q) acceptance on a tree with residual resampling.

    logits_p, logits_q [B, T, V] (only rows of nodes with children are read from
    logits_q); p_u = softmax(logits_p[u] / temperature), likewise q_u.
    u_accept [B, T]: the uniform of the edge into node c (entry 0 unused);
    u_sample [B]: the uniform of the final draw.

    Returns dict as greedy_accept, plus margin_decide (smallest |u_c - ratio_c|
    over edges with an accepted parent and ratio < 1) and margin_sample
    (distance from u' * total to the nearest CDF breakpoint, over total);
    margin is the smaller of the two.
    """
    zp = np.asarray(logits_p, dtype=np.float64) / float(temperature)
    zq = np.asarray(logits_q, dtype=np.float64) / float(temperature)
    B, T, V = zp.shape
    parent, depth, children = tree["parent"], tree["depth"], tree["children"]
    node_tok = np.asarray(node_tok, dtype=np.int64).reshape(B, T)
    u_accept = np.asarray(u_accept, dtype=np.float64).reshape(B, T)
    u_sample = np.asarray(u_sample, dtype=np.float64).reshape(B)
    internal = [u for u in range(T) if children[u]]
    maxd = tree["max_depth"]
    out = {
        "accept_len": np.zeros(B, dtype=np.int64),
        "accept_path": np.full((B, maxd + 1), -1, dtype=np.int64),
        "next_token": np.zeros(B, dtype=np.int64),
        "margin": np.full(B, np.inf),
        "margin_decide": np.full(B, np.inf),
        "margin_sample": np.full(B, np.inf),
    }
    for b in range(B):
        logp = _log_softmax(zp[b])
        logq = np.full((T, V), np.nan)
        if internal:
            logq[internal] = _log_softmax(zq[b, internal])
        accepted = np.zeros(T, dtype=bool)
        accepted[0] = True
        for c in range(1, T):
            par = int(parent[c])
            x = int(node_tok[b, c])
            ratio = np.exp(logp[par, x] - logq[par, x])
            accepted[c] = accepted[par] and u_accept[b, c] < ratio
            if accepted[par] and ratio < 1.0:
                out["margin_decide"][b] = min(out["margin_decide"][b], abs(u_accept[b, c] - ratio))
        u = _deepest(accepted, depth)
        p_u = np.exp(logp[u])
        if children[u]:
            w = _residual(p_u, np.exp(logq[u]))
            if w.sum() == 0.0:
                w = p_u
        else:
            w = p_u
        cdf = np.cumsum(w)
        total = cdf[-1]
        t = u_sample[b] * total
        x = int(np.searchsorted(cdf, t, side="right"))
        path = _path_to(u, parent)
        out["accept_len"][b] = depth[u]
        out["accept_path"][b, : len(path)] = path
        out["next_token"][b] = x
        out["margin_sample"][b] = float(np.min(np.abs(cdf - t))) / total
        out["margin"][b] = min(out["margin_decide"][b], out["margin_sample"][b])
    return out


def typical_accept(logits_p, node_tok, tree, temperature, epsilon, alpha, u_sample):
    """Medusa's typical acceptance on a tree.

    "Medusa Heads" (ultralytics glossary), section "Tree Attention und
    Akzeptanz": for sampling, a candidate is kept when its probability under
    the base model exceeds a threshold tied to the entropy of that
    distribution; more tokens are accepted, at the price of an inexact
    distribution ("Speculative Decoding", section "Beyond draft models:
    Medusa").  The pages give no formula and no constants.  Taken here: with
    p_u = softmax(logits_p[u] / temperature) and H_u = -sum_x p_u(x) ln p_u(x),
    the edge into node c with token x is accepted iff
        p_par(x) > min(epsilon, alpha * exp(-H_par));
    accepted(c) = accepted(parent) and that test; u* is the deepest accepted
    node (lowest index on equal depth), and the extra token is drawn from p_u*
    by inverse CDF in ascending token order with uniform u_sample[b].

    Returns dict as greedy_accept, plus margin_decide (smallest |p / threshold - 1|
    over edges with an accepted parent: thresholds can be ~1e-4, so the distance
    is relative), margin_sample (as rejection_accept) and margin = the smaller
    of the two.
    """
    zp = np.asarray(logits_p, dtype=np.float64) / float(temperature)
    B, T, V = zp.shape
    parent, depth = tree["parent"], tree["depth"]
    node_tok = np.asarray(node_tok, dtype=np.int64).reshape(B, T)
    u_sample = np.asarray(u_sample, dtype=np.float64).reshape(B)
    maxd = tree["max_depth"]
    out = {
        "accept_len": np.zeros(B, dtype=np.int64),
        "accept_path": np.full((B, maxd + 1), -1, dtype=np.int64),
        "next_token": np.zeros(B, dtype=np.int64),
        "margin": np.full(B, np.inf),
        "margin_decide": np.full(B, np.inf),
        "margin_sample": np.full(B, np.inf),
    }
    for b in range(B):
        logp = _log_softmax(zp[b])
        p = np.exp(logp)
        H = -(p * np.where(p > 0, logp, 0.0)).sum(axis=1)
        thr = np.minimum(float(epsilon), float(alpha) * np.exp(-H))
        accepted = np.zeros(T, dtype=bool)
        accepted[0] = True
        for c in range(1, T):
            par = int(parent[c])
            pc = p[par, int(node_tok[b, c])]
            accepted[c] = accepted[par] and pc > thr[par]
            if accepted[par] and thr[par] > 0:
                out["margin_decide"][b] = min(out["margin_decide"][b], abs(pc / thr[par] - 1.0))
        u = _deepest(accepted, depth)
        cdf = np.cumsum(p[u])
        total = cdf[-1]
        t = u_sample[b] * total
        x = int(np.searchsorted(cdf, t, side="right"))
        path = _path_to(u, parent)
        out["accept_len"][b] = depth[u]
        out["accept_path"][b, : len(path)] = path
        out["next_token"][b] = x
        out["margin_sample"][b] = float(np.min(np.abs(cdf - t))) / total
        out["margin"][b] = min(out["margin_decide"][b], out["margin_sample"][b])
    return out
