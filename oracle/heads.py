"""Medusa / Hydra draft heads and the candidate tree they fill (oracle; test infrastructure only).

Head form.  "Medusa Heads", section on how the heads predict: each head is one
feed-forward layer with SiLU and a residual connection, followed by a
projection onto the vocabulary.  Hydra Guide, section "1. Embedding
Conditioning Mechanics": a downstream head also sees the base-embedding row of
the candidate token its node continues, concatenated to h_t.  Put together, for
the head of depth d and a parent node u of sequence b:

    u_in = h_b                        (cond_d = 0, Medusa / Hydra head 1)
    u_in = [h_b || E[tok(u)]]         (cond_d = 1, Hydra, parent token only)
    z    = h_b + SiLU(W1_d u_in + b1_d),   SiLU(x) = x / (1 + exp(-x))
    l    = W2_d z                      (logits over the vocabulary)

For bf16 weights z is rounded to bf16 before the projection (the projection
consumes bf16 operands).

A second head form (form 1) is the one the Hydra Guide prints as code: the
fusion MLP Linear -> SiLU -> Linear -> LayerNorm followed by a bias-free
projection (its first head: Linear -> SiLU -> LayerNorm):
    a = SiLU(W1_d u_in + b1_d)         (rounded to bf16 for bf16 weights when it feeds W1b)
    y = W1b_d a + b1b_d                 (y = a when there is no W1b)
    z = (y - mean(y)) / sqrt(var(y) + eps) * gamma_d + beta_d
with the mean and the biased variance over the d entries of y.  The head output is softmax(l); its top-k equals the
top-k of l (softmax is monotone).

Tree filling.  Hydra Guide, section "Candidate Tree Construction": head 1 takes
its top-b1 tokens; every depth-1 node runs head 2 on its own token and takes
its top-b2 continuations; and so on.  A child of rank r gets the (r+1)-th
largest logit of its parent's row (descending value, ties to the lower token
id).  The cumulative log-probability of a node is its parent's plus the
child's log-softmax value (the page's code multiplies branch probabilities).
"""

import numpy as np

from .bf16 import bf16_bits_to_f64, f64_to_bf16_bits


def _decode(x, dtype):
    if dtype == "bf16":
        return bf16_bits_to_f64(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def _logsumexp(row):
    m = row.max()
    return m + np.log(np.exp(row - m).sum())


def hydra_draft(h, E, W1, b1, W2, cond, topk, root_tok, tree, dtype,
                teacher_tok=None, keep_logits=False):
    """Every head of form 0; see hydra_draft_heads for the arguments and the result."""
    heads = [dict(form=0, cond=int(cond[k]), topk=int(topk[k]), W1=W1[k], b1=None if b1 is None else b1[k],
                  W2=W2[k]) for k in range(len(W1))]
    return hydra_draft_heads(h, E, heads, root_tok, tree, dtype, teacher_tok=teacher_tok, keep_logits=keep_logits)


def hydra_draft_heads(h, E, heads, root_tok, tree, dtype, ln_eps=1e-5, teacher_tok=None, keep_logits=False):
    """Fill the candidate tree of every sequence with draft-head tokens.

    h [B, d]; E [V, d]; heads: one dict per head k (k = 0 .. K-1, filling
    depth k+1) with cond, topk, form (0 or 1), W1 [hidden, d_in_k], b1
    [hidden] or None, W2 [V, d], and for form 1 W1b [d, hidden] or None, b1b,
    gamma, beta ([d] or None: zeros / ones / zeros); ln_eps the LayerNorm
    epsilon.  Form 0 has hidden = d.
    W2[k] [V, d]; topk[k] >= 1 + the largest rank among depth-(k+1) nodes.
    Float inputs are float32 arrays (dtype "f32") or bf16 bit patterns as
    uint16 (dtype "bf16").  root_tok [B] is the token of node 0.

    teacher_tok [B, T] (optional): tokens to condition later heads on instead of
    the oracle's own picks, so depths after a near tie stay comparable.

    Input of head k for parent node u (depth k), by cond[k]:
      0: h_b                                  (d_in = d)
      1: [h_b || E[tok(u)]]                   (d_in = 2d; Hydra Guide, "1. Embedding
                                               Conditioning Mechanics")
      2: [h_b || E[tok(a_1)] || ... || E[tok(a_k)]], a_1 .. a_k = u's path below the
         root, depth 1 first                  (d_in = (k+1) d; Hydra Guide, "2.
                                               Generalizing to Arbitrary Tree Depths":
                                               head k reads h and the embeddings of all
                                               earlier candidate tokens of its path)

    Returns dict: node_tok int64 [B, T], node_logit [B, T], node_logprob [B, T]
    (root: its token, 0, 0), topk_gap [B, T] (for each parent row, the smallest
    gap between consecutive sorted logits over the ranks its children use,
    +inf for rows without children), and, if keep_logits, logits {(b, u): row}.
    """
    K = len(heads)
    cond = [int(hd["cond"]) for hd in heads]
    topk = [int(hd["topk"]) for hd in heads]
    T = tree["T"]
    parent, rank, depth, children = tree["parent"], tree["rank"], tree["depth"], tree["children"]
    if tree["max_depth"] > K:
        raise ValueError("the tree is deeper than the number of heads")
    H = _decode(h, dtype)
    B, d = H.shape
    root_tok = np.asarray(root_tok, dtype=np.int64).reshape(B)

    node_tok = np.zeros((B, T), dtype=np.int64)
    node_logit = np.zeros((B, T))
    node_logprob = np.zeros((B, T))
    topk_gap = np.full((B, T), np.inf)
    node_tok[:, 0] = root_tok
    cond_tok = node_tok.copy()  # tokens used for conditioning (own picks or teacher's)
    logits_out = {}

    for k in range(K):
        parents = [u for u in range(T) if depth[u] == k and children[u]]
        if not parents:
            continue
        for u in parents:
            for c in children[u]:
                if rank[c] >= topk[k]:
                    raise ValueError(f"node {c} has rank {rank[c]} >= top-k {topk[k]}")
        hd = heads[k]
        W1k = _decode(hd["W1"], dtype)
        W2k = _decode(hd["W2"], dtype)
        b1k = np.zeros(W1k.shape[0]) if hd.get("b1") is None else _decode(hd["b1"], dtype)
        rows = [(b, u) for b in range(B) for u in parents]
        if cond[k] == 0:
            X = np.stack([H[b] for b, _ in rows])
        elif cond[k] == 2:
            blocks = [np.stack([H[b] for b, _ in rows])]
            paths = [[a for a in tree["anc"][u] if a != 0] for _, u in rows]   # depth order (ids grow)
            for i in range(k):
                toks = np.array([cond_tok[b, path[i]] for (b, _), path in zip(rows, paths)], dtype=np.int64)
                blocks.append(_decode(np.asarray(E)[toks], dtype))
            X = np.concatenate(blocks, axis=1)
        else:
            toks = np.array([cond_tok[b, u] for b, u in rows], dtype=np.int64)
            Erows = _decode(np.asarray(E)[toks], dtype)
            X = np.concatenate([np.stack([H[b] for b, _ in rows]), Erows], axis=1)
        A = X @ W1k.T + b1k
        if hd.get("form", 0) == 0:
            Z = np.stack([H[b] for b, _ in rows]) + silu(A)
        else:
            a = silu(A)
            if hd.get("W1b") is not None:
                if dtype == "bf16":
                    a = bf16_bits_to_f64(f64_to_bf16_bits(a))
                b1b = np.zeros(d) if hd.get("b1b") is None else _decode(hd["b1b"], dtype)
                Y = a @ _decode(hd["W1b"], dtype).T + b1b
            else:
                Y = a
            gamma = np.ones(d) if hd.get("gamma") is None else _decode(hd["gamma"], dtype)
            beta = np.zeros(d) if hd.get("beta") is None else _decode(hd["beta"], dtype)
            mu = Y.mean(axis=1, keepdims=True)
            var = ((Y - mu) ** 2).mean(axis=1, keepdims=True)
            Z = (Y - mu) / np.sqrt(var + float(ln_eps)) * gamma + beta
        if dtype == "bf16":
            Z = bf16_bits_to_f64(f64_to_bf16_bits(Z))
        L = Z @ W2k.T
        for r, (b, u) in enumerate(rows):
            row = L[r]
            order = np.argsort(-row, kind="stable")
            lse = _logsumexp(row)
            used = max(int(rank[c]) for c in children[u]) + 1
            sorted_vals = row[order[: used + 1]]
            if sorted_vals.size >= 2:
                topk_gap[b, u] = float(np.min(sorted_vals[:-1] - sorted_vals[1:]))
            for c in children[u]:
                t = int(order[rank[c]])
                node_tok[b, c] = t
                node_logit[b, c] = row[t]
                node_logprob[b, c] = node_logprob[b, u] + row[t] - lse
                cond_tok[b, c] = t if teacher_tok is None else int(teacher_tok[b, c])
            if keep_logits:
                logits_out[(b, u)] = row.copy()

    out = {"node_tok": node_tok, "node_logit": node_logit,
           "node_logprob": node_logprob, "topk_gap": topk_gap}
    if keep_logits:
        out["logits"] = logits_out
    return out
