"""A whole verification step (draft heads, tree attention, acceptance) captured
into a CUDA graph replays to the same outputs, bit for bit, as the eager calls
(GPU).

Every call takes its workspace and outputs from the caller and makes no host
synchronisation, so a step is capturable; replaying it leaves the per-call
host work (argument checks, tensor-map encoding, launch) out of the step.
"""

import numpy as np
import pytest

import spec_workloads as wl
from gpu_util import lib, to_dev

pytestmark = pytest.mark.gpu


def _step_fixture(st, w, tree_spec, folded):
    import torch
    parent, rank = wl.make_tree(tree_spec)
    T = len(parent)
    tree = st.spec_tree_build(parent, rank)
    dx = wl.draft_inputs(w)
    h, E, root = to_dev(dx["h"]), to_dev(dx["E"]), to_dev(dx["root_tok"])
    W1 = [to_dev(a) for a in dx["W1"]]
    b1 = [to_dev(a) for a in dx["b1"]]
    W2 = [to_dev(a) for a in dx["W2"]]
    cond, topk = list(w.cond), list(w.topk)
    tabs = [st.hydra_fold_embedding(W1[k], E) if cond[k] == 1 else None for k in range(len(cond))] if folded else None
    ax = wl.attention_inputs(w, T)
    q, kc, vc, plen, kt, vt = (to_dev(ax[k]) for k in ("q", "k_cache", "v_cache", "prefix_len", "k_tree", "v_tree"))
    gx = wl.greedy_inputs(w, parent)
    lp = to_dev(gx["logits_p"])
    B = w.B
    dev = h.device
    outs = {
        "node_tok": torch.empty(B, T, dtype=torch.int32, device=dev),
        "node_logit": torch.empty(B, T, dtype=torch.float32, device=dev),
        "node_logprob": torch.empty(B, T, dtype=torch.float32, device=dev),
        "out": torch.empty(B, w.Hq, T, w.D, dtype=torch.float32, device=dev),
        "lse": torch.empty(B, w.Hq, T, dtype=torch.float32, device=dev),
        "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
        "accept_path": torch.empty(B, tree.max_depth + 1, dtype=torch.int32, device=dev),
        "next_token": torch.empty(B, dtype=torch.int32, device=dev),
        "margin": torch.empty(B, dtype=torch.float32, device=dev),
    }
    dt = 1 if w.dtype == "bf16" else 0
    wsd = torch.empty(st.hydra_draft_workspace_size(tree, B, w.d, w.V, cond, topk, dt), dtype=torch.uint8, device=dev)
    wsa = torch.empty(st.tree_attention_workspace_size(tree, B, w.Hq, w.Hkv, w.Lmax, w.D, dt), dtype=torch.uint8,
                      device=dev)
    wsc = torch.empty(st.tree_accept_workspace_size(0, tree, B, w.V), dtype=torch.uint8, device=dev)

    def step():
        st.hydra_draft(h, E, W1, b1, W2, cond, topk, root, tree, node_tok=outs["node_tok"],
                       node_logit=outs["node_logit"], node_logprob=outs["node_logprob"], ws=wsd, folded=tabs)
        st.tree_attention(q, kc, vc, plen, kt, vt, tree, out=outs["out"], lse=outs["lse"], ws=wsa)
        st.tree_accept(0, lp, None, outs["node_tok"], tree, accept_len=outs["accept_len"],
                       accept_path=outs["accept_path"], next_token=outs["next_token"], margin=outs["margin"], ws=wsc)
    return step, outs


def _replay_matches_eager(w, tree_spec, folded):
    import torch
    st = lib()
    step, outs = _step_fixture(st, w, tree_spec, folded)
    step()
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in outs.items()}
    # capture on a side stream after a warm-up there (module loads, attribute setting and the
    # other first-call work stay out of the graph)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        for v in outs.values():
            v.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        for k, v in outs.items():
            a, b = v.cpu().numpy(), eager[k].cpu().numpy()
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), k


def test_tiny_fp32_step_replays_from_a_graph():
    w = wl.WORKLOADS[1]
    _replay_matches_eager(w, w.tree, folded=False)


@pytest.mark.parametrize("folded", [False, True])
def test_tensor_core_step_replays_from_a_graph(folded):
    """bf16 with 73 tree nodes: tensor-core draft heads (folded or not), tcgen05 tree attention
    with its prefix splits merged on chip, greedy acceptance."""
    w = wl.Workload("graph-step", "bf16", B=2, seed=41, tree=("cartesian", (8, 8)), d=256, V=4096, cond=(1, 1),
                    topk=(8, 8), Hq=8, Hkv=8, D=128, Lmax=1024, prefix=(700, 1024), accept="greedy",
                    accept_lengths=(0, 1, 2), parts=("draft", "attention", "accept"))
    _replay_matches_eager(w, w.tree, folded)
