#!/usr/bin/env python3
"""Benchmark of one tree-verification step on GB300.

A step is the whole hot path over one batch: the Hydra draft heads fill the
64-node candidate tree (hidden 4096, vocabulary 32000, 4 sequentially
dependent heads, top-k 8/4/2/1), the tree tokens attend over a 1024-token KV
prefix (32 heads x 128, bf16), and greedy acceptance picks the longest accepted
path (target logits planted so the mean accepted length is about 2.5).  Batch 1,
synthetic seeded inputs resident in HBM; L2 is flushed between timed steps.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on the
same workload instead (the oracle is a deliberately plain NumPy fp64 program).
Multi-GPU runs (torchrun) give every rank its own independent batch: no data
exchange, weak scaling; the reported time is the maximum over ranks.
"""

import argparse
import hashlib
import json
import os
import resource
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

METRIC = "verify steps/s & tree-node tokens/s per step; achieved HBM GB/s vs GB300 peak"
UNIT = "verify steps/s"
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Between timed steps: write a buffer larger than L2 (nothing of the last
    step stays cached), then read a second one so that the dirty lines of that
    write are written back here and not inside the next timed step."""

    def __init__(self, dev):
        import torch
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.out = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        self.torch.sum(self.r, dim=0, dtype=self.torch.int64, out=self.out)


def workload(seed):
    import spec_workloads as wl
    base = wl.WORKLOADS[2]
    return wl.Workload("vicuna7b-verify-step", "bf16", B=1, seed=seed, tree=base.tree,
                       d=4096, V=32000, cond=(1, 1, 1, 1), topk=(8, 4, 2, 1),
                       Hq=32, Hkv=32, D=128, Lmax=1024, prefix=(1024, 1024),
                       accept="greedy", accept_lengths=(1, 2, 3, 4))


def config_of(w, T):
    return {
        "workload": "vicuna7b-verify-step: Hydra draft heads (hidden 4096, vocab 32000, 4 heads, top-k 8/4/2/1) "
                    "+ tree attention (32x128 heads, prefix 1024) + greedy acceptance, 64-node sparse tree, batch 1",
        "batch": w.B, "tree_nodes": T, "prefix": w.Lmax, "hidden": w.d, "vocab": w.V,
        "attention_heads": f"{w.Hq}x{w.D}", "draft_heads": len(w.cond), "topk": list(w.topk),
        "acceptance": "greedy", "l2": "flushed between timed steps (256 MB write, then 256 MB read so no dirty line is written back inside a step)",
    }


# ---------------------------------------------------------------- distributed plumbing

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def init_dist(backend):
    import torch.distributed as dist
    rank, local, world = dist_info()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29511")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, local, world


def max_over_ranks(x, device=None):
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, every 200 ms."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.marks = {}

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def mark(self, name):
        self.marks[name] = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.samples:
            return None
        inside = [p for (t, p) in self.samples if t0 - 0.25 <= t <= t1 + 0.25]
        if len(inside) < 2:
            inside = [p for (_, p) in self.samples[-5:]]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------- roofline bookkeeping

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def algorithmic_bytes(name, ctx):
    """Algorithmic HBM bytes per launch of each kernel of the step (what the math must move)."""
    w, rows = ctx["w"], ctx["rows"]
    s = 2  # bf16
    d, V = w.d, w.V
    heads = [k for k in range(len(w.cond)) if rows[k] > 0]
    if name.startswith("draft_proj"):
        return sum(V * d * s + rows[k] * d * s for k in heads) / len(heads)
    if name == "draft_fold_h":   # W1[:, :d] once, h_b in, a (fp32) or z out, per sequence
        return d * d * s + w.B * d * (s + 4)
    if name.startswith("draft_mlp"):
        return sum(d * 2 * d * s + d * s + rows[k] * 2 * d * s + rows[k] * d * s for k in heads) / len(heads)
    if name.startswith("attn_") and name != "attn_combine":
        T = ctx["T"]
        return (sum(ctx["prefix_len"]) * w.Hkv * w.D * 2 * s + w.B * w.Hq * T * w.D * s
                + w.B * w.Hkv * T * w.D * 2 * s)
    if name == "attn_combine":
        return w.B * w.Hq * ctx["T"] * w.D * 4
    if name == "accept_rows_greedy":
        return w.B * ctx["T"] * w.V * 4
    return None


def recorded_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if its source is unchanged since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    for line in lines:
        if line.startswith("#") or not line.strip():
            continue
        parts = line.split()
        if len(parts) >= 3 and parts[0] == kernel:
            src = os.path.join(ROOT, "tree_speculative_decoding_spec_gb300", "csrc", parts[2].split(":")[0])
            want = parts[2].split(":")[1] if ":" in parts[2] else ""
            try:
                have = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
            except OSError:
                return None
            return float(parts[1]) if have == want else None
    return None


# ---------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    rank, local, world = init_dist("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import spec_workloads as wl
    import tree_speculative_decoding_spec_gb300 as st

    w = workload(seed=2 + 1000 * rank)
    parent, rank_arr = wl.make_tree(w.tree)
    T = len(parent)
    dx = wl.draft_inputs(w)
    ax = wl.attention_inputs(w, T)

    def dev_t(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    tree = st.spec_tree_build(parent, rank_arr, device=dev)
    h, E = dev_t(dx["h"]), dev_t(dx["E"])
    W1 = [dev_t(a) for a in dx["W1"]]
    b1 = [dev_t(a) for a in dx["b1"]]
    W2 = [dev_t(a) for a in dx["W2"]]
    # weight-load-time preparation (outside every timed region): the folded embedding tables,
    # their build timed with CUDA events (the second build, after a first that loads the kernels)
    tabs, fold_ms = None, None
    if not args.no_fold:
        for _ in range(2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            tabs = [st.hydra_fold_embedding(W1[k], E) if c == 1 else None for k, c in enumerate(w.cond)]
            b.record()
            torch.cuda.synchronize()
            fold_ms = a.elapsed_time(b) / max(1, sum(int(c == 1) for c in w.cond))
    root_tok = dev_t(dx["root_tok"])
    q, kc, vc = dev_t(ax["q"]), dev_t(ax["k_cache"]), dev_t(ax["v_cache"])
    plen, kt, vt = dev_t(ax["prefix_len"]), dev_t(ax["k_tree"]), dev_t(ax["v_tree"])
    cond, topk = list(w.cond), list(w.topk)
    B = w.B

    node_tok = torch.empty(B, T, dtype=torch.int32, device=dev)
    node_logit = torch.empty(B, T, dtype=torch.float32, device=dev)
    node_logprob = torch.empty(B, T, dtype=torch.float32, device=dev)
    out = torch.empty(B, w.Hq, T, w.D, dtype=torch.float32, device=dev)
    lse = torch.empty(B, w.Hq, T, dtype=torch.float32, device=dev)
    alen = torch.empty(B, dtype=torch.int32, device=dev)
    apath = torch.empty(B, tree.max_depth + 1, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    mg = torch.empty(B, dtype=torch.float32, device=dev)
    ws_d = torch.empty(st.hydra_draft_workspace_size(tree, B, w.d, w.V, cond, topk, 1), dtype=torch.uint8, device=dev)
    ws_a = torch.empty(st.tree_attention_workspace_size(tree, B, w.Hq, w.Hkv, w.Lmax, w.D, 1), dtype=torch.uint8, device=dev)
    ws_c = torch.empty(st.tree_accept_workspace_size(0, tree, B, w.V), dtype=torch.uint8, device=dev)

    def draft():
        st.hydra_draft(h, E, W1, b1, W2, cond, topk, root_tok, tree, node_tok=node_tok, node_logit=node_logit,
                       node_logprob=node_logprob, ws=ws_d, folded=tabs)

    # plant the target logits on the draft's own tokens (the target model itself is out of scope)
    draft()
    torch.cuda.synchronize()
    gx = wl.greedy_inputs(w, parent, node_tok=node_tok.cpu().numpy())
    logits_p = dev_t(gx["logits_p"])

    def attention():
        st.tree_attention(q, kc, vc, plen, kt, vt, tree, out=out, lse=lse, ws=ws_a)

    def accept():
        st.tree_accept(0, logits_p, None, node_tok, tree, accept_len=alen, accept_path=apath, next_token=nxt,
                       margin=mg, ws=ws_c)

    def step():
        draft()
        attention()
        accept()

    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    for _ in range(max(args.warmup, 0)):
        step()
        flush()
    torch.cuda.synchronize()

    # per-phase times (separate pass, not the headline)
    phase_ms = {}
    for name, fn in [("draft", draft), ("attention", attention), ("accept", accept)]:
        evs = []
        for _ in range(5):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        phase_ms[name] = statistics.median([a.elapsed_time(b) for a, b in evs])

    def timed_steps(n):
        evs = []
        for _ in range(n):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step()
            b.record(stream)
            evs.append((a, b))
            flush()
        return evs

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    # timed region: K steps exactly as a user runs them (no tracing, so the
    # dependent launches of the draft heads overlap as designed)
    launches0 = st.spec_launch_count()
    barrier(dev)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    evs = timed_steps(args.steps)
    torch.cuda.synchronize()
    barrier(dev)
    t_wall1 = time.time()
    launches = st.spec_launch_count() - launches0
    # kernel region: K more steps with every launch bracketed by CUDA events on
    # its stream (per-kernel times for the roofline; overlap is off here)
    st.spec_trace_begin(100000)
    traced = timed_steps(args.steps)
    torch.cuda.synchronize()
    kernels = st.spec_trace_end(256)
    # the same step with unfolded first layers (the whole W1 of every head streamed per step)
    unfolded = None
    if tabs is not None:
        def step_unfolded():
            st.hydra_draft(h, E, W1, b1, W2, cond, topk, root_tok, tree, node_tok=node_tok, node_logit=node_logit,
                           node_logprob=node_logprob, ws=ws_d)
            attention()
            accept()
        for _ in range(3):
            step_unfolded()
            flush()
        uev = []
        tu0 = time.time()
        for _ in range(args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step_unfolded()
            b.record(stream)
            uev.append((a, b))
            flush()
        torch.cuda.synchronize()
        tu1 = time.time()
        u_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in uev) / len(uev), dev)
        unfolded = {"value": world * 1000.0 / u_ms, "unit": UNIT, "ms_per_step": u_ms,
                    "draft_first_layer": "whole W1 streamed per step", "clocks": clocks.summary(tu0, tu1)}
    # the same step captured once into a CUDA graph and replayed (the per-call host work leaves the step)
    try:
        tg0 = time.time()
        g_list = graph_times(step, lambda: None, flush, args.steps)
        tg1 = time.time()
        g_ms = max_over_ranks(sum(g_list) / len(g_list), dev)
        graph_step = {"value": world * 1000.0 / g_ms, "unit": UNIT, "ms_per_step": g_ms,
                      "clocks": clocks.summary(tg0, tg1)}
    except Exception as e:
        graph_step = {"unavailable": str(e).splitlines()[0][:200]}
    time.sleep(0.3)
    clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    traced_ms = [a.elapsed_time(b) for a, b in traced]
    ms_per_step = max_over_ranks(sum(step_ms) / len(step_ms), dev)
    value = world * 1000.0 / ms_per_step

    # roofline of the dominant kernel
    hbm, tf_burst, tf_sust, peak_src = peaks()
    total_k = sum(v[1] for v in kernels.values())
    dom = max(kernels.items(), key=lambda kv: kv[1][1])
    dom_name, (dom_n, dom_ms) = dom
    rows = [(B * tree.struct.n_internal_at_depth[k] if cond[k] else B) if tree.struct.n_internal_at_depth[k] else 0
            for k in range(len(cond))]
    ctx = {"w": w, "rows": rows, "T": T, "prefix_len": [int(x) for x in ax["prefix_len"]]}
    abytes = algorithmic_bytes(dom_name, ctx)
    per_launch_s = dom_ms / dom_n / 1000.0
    achieved = abytes / per_launch_s / 1e9 if abytes else None
    roofline = {"kernel": dom_name, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm if achieved else None, "traffic": recorded_traffic(dom_name),
                "algorithmic_bytes_per_launch": abytes, "launch_us": per_launch_s * 1e6,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)" if peak_src == "measured"
                else "fallback 6.8 TB/s", "frac_of_nominal_8TBs": achieved / 8000.0 if achieved else None}
    kern_table = {k: {"launches": n, "ms_per_launch": ms / n, "share": ms / total_k if total_k else None,
                      "algorithmic_GBps": (algorithmic_bytes(k, ctx) / (ms / n / 1000.0) / 1e9)
                      if algorithmic_bytes(k, ctx) else None}
                  for k, (n, ms) in sorted(kernels.items(), key=lambda kv: -kv[1][1])}

    # end-to-end through the public API with host buffers (pinned), copies inside the timed region.
    # Each direction is one copy: the step's inputs sit in one pinned host buffer and the
    # device tensors the calls read are views into one device buffer (likewise the outputs).
    e2e = None
    if not args.no_e2e:
        def packed(tensors, device, pin=False):
            offs, n = [], 0
            for t in tensors:
                offs.append(n)
                n += -(-t.numel() * t.element_size() // 256) * 256
            buf = torch.empty(n, dtype=torch.uint8, device=device, pin_memory=pin)
            views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(tensors, offs)]
            return buf, views
        # two uploads per step: the draft's inputs (h_b, root tokens: 8 KB) on the compute
        # stream, then the attention's and acceptance's inputs (9.8 MB) on a copy stream,
        # overlapping the draft; the attention waits for that copy's event
        src_a = [h, root_tok]
        src_b = [q, kt, vt, plen, logits_p]
        host_a_buf, host_a = packed(src_a, "cpu", pin=True)
        host_b_buf, host_b = packed(src_b, "cpu", pin=True)
        dev_a_buf, (h_e, root_e) = packed(src_a, dev)
        dev_b_buf, (q_e, kt_e, vt_e, plen_e, lp_e) = packed(src_b, dev)
        for hv, t in zip(host_a + host_b, src_a + src_b):
            hv.copy_(t.cpu())
        copy_stream = torch.cuda.Stream(device=dev)
        b_ready = torch.cuda.Event()
        src_out = [node_tok, alen, apath, nxt]
        host_out_buf, _ = packed(src_out, "cpu", pin=True)
        dev_out_buf, (tok_e, alen_e, apath_e, nxt_e) = packed(src_out, dev)

        def step_e2e():
            st.hydra_draft(h_e, E, W1, b1, W2, cond, topk, root_e, tree, node_tok=tok_e, node_logit=node_logit,
                           node_logprob=node_logprob, ws=ws_d, folded=tabs)
            stream.wait_event(b_ready)
            st.tree_attention(q_e, kc, vc, plen_e, kt_e, vt_e, tree, out=out, lse=lse, ws=ws_a)
            st.tree_accept(0, lp_e, None, tok_e, tree, accept_len=alen_e, accept_path=apath_e, next_token=nxt_e,
                           margin=mg, ws=ws_c)

        bi = host_a_buf.numel() + host_b_buf.numel()
        bo = host_out_buf.numel()
        e_ms = []
        for i in range(args.warmup + args.steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            copy_stream.wait_stream(stream)   # after the timing event and the previous step's reads
            with torch.cuda.stream(copy_stream):
                dev_b_buf.copy_(host_b_buf, non_blocking=True)
                b_ready.record(copy_stream)
            dev_a_buf.copy_(host_a_buf, non_blocking=True)
            step_e2e()
            host_out_buf.copy_(dev_out_buf, non_blocking=True)
            b.record(stream)
            b.synchronize()
            if i >= args.warmup:
                e_ms.append(a.elapsed_time(b))
        e_mean = max_over_ranks(sum(e_ms) / len(e_ms), dev)
        e2e = {"value": world * 1000.0 / e_mean, "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "ms_per_step": e_mean, "copies_per_step": {"h2d": 2, "d2h": 1},
               "overlap": "the attention/acceptance inputs upload on a copy stream while the draft runs"}

    # every other config of the parity suite, one entry point per entry, each with its own roofline
    # and the clock record of its own timed window (rank 0 only)
    configs = None
    if rank == 0 and not args.no_configs:
        tabs = None   # the headline's fold tables (2.1 GB) are not needed any more
        torch.cuda.empty_cache()
        configs = run_configs(dev, local, args.steps)

    # CPU baseline: the oracle as it stands, one full step of the same workload, at 1 thread and at
    # every host thread (separate processes: BLAS threads are fixed when numpy loads)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_legs()

    if rank != 0:
        return
    accepted = float(alen.float().mean().item())
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; random-init head weights, N(0,1) KV)",
        "config": config_of(w, T),
        "draft_first_layer": ("whole W1 streamed per step" if args.no_fold else
                              "folded: W1[:, :d] streamed per step, W1[:, d:] E tabulated once at weight load (fp32)"),
        "tree_node_tokens_per_s": value * B * T,
        "accepted_tokens_per_s": value * B * (accepted + 1),
        "phases_ms": phase_ms,
        "kernels": kern_table,
        "roofline": roofline,
        "unfolded_step": unfolded,
        "graph_step": graph_step,
        "fold_tables_bytes": (sum(int(c == 1) for c in cond) * w.V * w.d * 4) if not args.no_fold else 0,
        "fold_table_build_ms_per_head": fold_ms,
        "configs": configs,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "ms_per_step_traced": sum(traced_ms) / len(traced_ms),
        "gpu_launches": launches,
        "gpu_launches_per_step": launches / max(args.steps, 1),
        "clocks": clocks.summary(t_wall0, t_wall1),
        "wall_s_timed": t_wall1 - t_wall0,
    }
    print(json.dumps(line), flush=True)


CONFIG_ENTRIES = [
    # (entry name, component, no_fold): every workload of the parity suite besides the headline step
    ("tiny_fp32_step", "step-tiny-fp32", False),
    ("vicuna7b_attention", "attention-vicuna7b", False),
    ("vicuna7b_greedy_accept", "accept-greedy-vicuna7b", False),
    ("hydra_heads_b4_folded", "draft-hydra-b4", False),
    ("hydra_heads_b4_unfolded", "draft-hydra-b4", True),
    ("gqa70b_b8_attention", "attention-70b-gqa", False),
    ("long32k_attention_t341", "attention-32k", False),
    ("long32k_attention_t256", "attention-32k-t256", False),
    ("long32k_rejection_accept", "accept-rejection-32k", False),
    # the entry points past the verification step itself
    ("long32k_typical_accept", "accept-typical-32k", False),
    ("gqa70b_b8_paged_attention", "attention-paged-70b-b8", False),
    ("vicuna7b_layernorm_heads", "draft-ln-heads-vicuna7b", False),
    ("vicuna7b_kv_commit", "kv-commit-vicuna7b", False),
    ("gqa70b_b8_kv_commit", "kv-commit-70b-b8", False),
    ("gqa70b_b8_kv_commit_paged", "kv-commit-paged-70b-b8", False),
]


def run_configs(dev, local, steps):
    import torch
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    flush = L2Flush(dev)
    out = {}
    try:
        for entry, name, no_fold in CONFIG_ENTRIES:
            comp = make_component(name, dev, no_fold=no_fold)
            out[entry] = {"component": name}
            out[entry].update(measure_component(comp, flush, clocks, steps))
            del comp
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
    finally:
        clocks.stop()
    return out


def cpu_baseline_legs():
    """The oracle timed on the host cores at 1 thread and at every thread, each in a child process."""
    legs = {}
    n = os.cpu_count() or 1
    for threads in (1, n):
        env = dict(os.environ)
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
            env[k] = str(threads)
        env["CUDA_VISIBLE_DEVICES"] = ""
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-step"], env=env, capture_output=True,
                           text=True, timeout=600)
        try:
            legs[threads] = json.loads(r.stdout.strip().splitlines()[-1])
        except (ValueError, IndexError):
            legs[threads] = {"error": (r.stderr or r.stdout)[-300:]}
    full = legs.get(n, {})
    one = legs.get(1, {})
    return {"value": full.get("value"), "unit": UNIT, "cores": full.get("cores"), "threads": n,
            "cores_available": n, "kind": "oracle",
            "sample": "one full verification step of the same workload (draft heads, attention, greedy acceptance), "
                      "NumPy float64 on the host cores; cores = CPU time / wall time",
            "one_thread": {"value": one.get("value"), "cores": one.get("cores"), "threads": 1},
            "all_threads": {"value": full.get("value"), "cores": full.get("cores"), "threads": n}}


def run_oracle_step_child():
    """Child of cpu_baseline_legs: one oracle step of the headline workload, one JSON line."""
    import oracle
    import spec_workloads as wl
    w = workload(seed=2)
    parent, rank_arr = wl.make_tree(w.tree)
    T = len(parent)
    dx = wl.draft_inputs(w)
    ax = wl.attention_inputs(w, T)
    to = oracle.tree_encode(parent, rank_arr)
    tok = oracle.hydra_draft(dx["h"], dx["E"], dx["W1"], dx["b1"], dx["W2"], dx["cond"], dx["topk"], dx["root_tok"],
                             to, w.dtype)["node_tok"]
    gx = wl.greedy_inputs(w, parent, node_tok=tok)
    r = time_oracle_step(w, parent, rank_arr, dx, ax, gx)
    print(json.dumps(r), flush=True)


def time_oracle_step(w, parent, rank_arr, dx, ax, gx):
    import oracle
    to = oracle.tree_encode(parent, rank_arr)
    c0 = resource.getrusage(resource.RUSAGE_SELF)
    t0 = time.perf_counter()
    ref = oracle.hydra_draft(dx["h"], dx["E"], dx["W1"], dx["b1"], dx["W2"], dx["cond"], dx["topk"],
                             dx["root_tok"], to, w.dtype)
    oracle.tree_attention(**ax, tree=to, dtype=w.dtype)
    oracle.greedy_accept(gx["logits_p"], ref["node_tok"], to)
    t1 = time.perf_counter()
    c1 = resource.getrusage(resource.RUSAGE_SELF)
    cpu_s = (c1.ru_utime - c0.ru_utime) + (c1.ru_stime - c0.ru_stime)
    return {"value": 1.0 / (t1 - t0), "unit": UNIT, "cores": round(cpu_s / (t1 - t0), 2),
            "cores_available": os.cpu_count(), "kind": "oracle",
            "sample": "one full verification step of the same workload (draft heads, attention, greedy acceptance), "
                      "NumPy float64 on the host cores; cores = CPU time / wall time"}


# ---------------------------------------------------------------- reference arm (the CPU oracle)

def run_reference(args):
    rank, local, world = dist_info()
    if rank != 0:
        return
    import oracle
    import spec_workloads as wl
    w = workload(seed=2)
    parent, rank_arr = wl.make_tree(w.tree)
    T = len(parent)
    dx = wl.draft_inputs(w)
    ax = wl.attention_inputs(w, T)
    to = oracle.tree_encode(parent, rank_arr)
    tok = oracle.hydra_draft(dx["h"], dx["E"], dx["W1"], dx["b1"], dx["W2"], dx["cond"], dx["topk"], dx["root_tok"],
                             to, w.dtype)["node_tok"]
    gx = wl.greedy_inputs(w, parent, node_tok=tok)
    for _ in range(max(args.warmup, 0)):
        time_oracle_step(w, parent, rank_arr, dx, ax, gx)
    times, cores = [], []
    for _ in range(args.steps):
        r = time_oracle_step(w, parent, rank_arr, dx, ax, gx)
        times.append(1.0 / r["value"])
        cores.append(r["cores"])
    ms = 1000.0 * sum(times) / len(times)
    value = 1000.0 / ms
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)", "config": config_of(w, T),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": round(statistics.median(cores), 2),
                         "cores_available": os.cpu_count(), "kind": "oracle",
                         "sample": "each step: one full verification step of the workload on the host cores"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


COMPONENTS = {
    # name: (workload id, part, tree override)
    "step-tiny-fp32": (1, "step", None),
    "attention-vicuna7b": (2, "attention", None),
    "attention-70b-gqa": (4, "attention", None),
    "attention-32k": (5, "attention", None),
    "attention-32k-t256": (5, "attention", ("dense_prefix", (4, 4, 4, 4), 256)),
    "draft-hydra-b4": (3, "draft", None),
    "draft-ln-heads-vicuna7b": (2, "draft_ln", ("sparse", (8, 4, 2, 1), 64, 64)),
    "accept-greedy-vicuna7b": (2, "accept", None),
    "accept-rejection-32k": (5, "accept", None),
    "accept-typical-32k": (5, "accept_typical", None),
    "attention-paged-70b-b8": (4, "attention_paged", None),
    "kv-commit-vicuna7b": (2, "commit", None),
    "kv-commit-70b-b8": (4, "commit", None),
    "kv-commit-paged-70b-b8": (4, "commit_paged", None),
}


def make_component(name, dev, no_fold=False):
    """Inputs, outputs and the library call of one entry point on one parity workload.

    Returns a dict: call (one library call), pre (untimed, before every call),
    abytes / flops (algorithmic work per call), report (extra fields after the
    measurement: near-tie counts and the like) and the workload facts."""
    import torch
    import spec_workloads as wl
    import tree_speculative_decoding_spec_gb300 as st

    wid, part, tree_spec = COMPONENTS[name]
    w = wl.WORKLOADS[wid]
    parent, rank_arr = wl.make_tree(tree_spec or w.tree)
    T = len(parent)
    tree = st.spec_tree_build(parent, rank_arr, device=dev)

    def dev_t(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    s = 2 if w.dtype == "bf16" else 4
    flops = 0.0
    if part == "step":
        # the whole verification step of the tiny fp32 workload: draft heads, attention, greedy acceptance
        dx = wl.draft_inputs(w)
        h, E, root = dev_t(dx["h"]), dev_t(dx["E"]), dev_t(dx["root_tok"])
        W1 = [dev_t(a) for a in dx["W1"]]
        b1 = [dev_t(a) for a in dx["b1"]]
        W2 = [dev_t(a) for a in dx["W2"]]
        cond, topk = list(w.cond), list(w.topk)
        nt = torch.empty(w.B, T, dtype=torch.int32, device=dev)
        nl = torch.empty(w.B, T, dtype=torch.float32, device=dev)
        nlp = torch.empty(w.B, T, dtype=torch.float32, device=dev)
        wsd = torch.empty(st.hydra_draft_workspace_size(tree, w.B, w.d, w.V, cond, topk, 0), dtype=torch.uint8, device=dev)
        ax = wl.attention_inputs(w, T)
        q, kc, vc, plen, kt, vt = (dev_t(ax[k]) for k in ("q", "k_cache", "v_cache", "prefix_len", "k_tree", "v_tree"))
        out = torch.empty(w.B, w.Hq, T, w.D, dtype=torch.float32, device=dev)
        lse = torch.empty(w.B, w.Hq, T, dtype=torch.float32, device=dev)
        wsa = torch.empty(st.tree_attention_workspace_size(tree, w.B, w.Hq, w.Hkv, w.Lmax, w.D, 0), dtype=torch.uint8,
                          device=dev)
        gx = wl.greedy_inputs(w, parent)
        lp = dev_t(gx["logits_p"])
        outs = [torch.empty(w.B, dtype=torch.int32, device=dev),
                torch.empty(w.B, tree.max_depth + 1, dtype=torch.int32, device=dev),
                torch.empty(w.B, dtype=torch.int32, device=dev), torch.empty(w.B, dtype=torch.float32, device=dev)]
        wsc = torch.empty(st.tree_accept_workspace_size(0, tree, w.B, w.V), dtype=torch.uint8, device=dev)

        def call():
            st.hydra_draft(h, E, W1, b1, W2, cond, topk, root, tree, node_tok=nt, node_logit=nl, node_logprob=nlp,
                           ws=wsd)
            st.tree_attention(q, kc, vc, plen, kt, vt, tree, out=out, lse=lse, ws=wsa)
            st.tree_accept(0, lp, None, nt, tree, accept_len=outs[0], accept_path=outs[1], next_token=outs[2],
                           margin=outs[3], ws=wsc)
        d, V, L = w.d, w.V, [int(x) for x in ax["prefix_len"]]
        abytes = 0.0
        for k in range(len(cond)):
            n_int = tree.struct.n_internal_at_depth[k]
            if n_int:
                rows = w.B * n_int if cond[k] else w.B
                d_in = d * (2 if cond[k] else 1)
                abytes += (d * d_in + d + V * d) * s + rows * (d_in + d) * s
                flops += 2.0 * rows * (d_in * d + d * V)
        abytes += (sum(L) * w.Hkv * w.D * 2 * s + w.B * w.Hq * T * w.D * s + w.B * w.Hkv * T * w.D * 2 * s
                   + w.B * w.Hq * T * (w.D + 1) * 4) + w.B * T * w.V * 4
        flops += 4.0 * w.D * w.Hq * T * sum(l + T for l in L)
    elif part == "attention":
        ax = wl.attention_inputs(w, T)
        q, kc, vc, plen, kt, vt = (dev_t(ax[k]) for k in ("q", "k_cache", "v_cache", "prefix_len", "k_tree", "v_tree"))
        out = torch.empty(w.B, w.Hq, T, w.D, dtype=torch.float32, device=dev)
        lse = torch.empty(w.B, w.Hq, T, dtype=torch.float32, device=dev)
        ws = torch.empty(st.tree_attention_workspace_size(tree, w.B, w.Hq, w.Hkv, w.Lmax, w.D, 1 if s == 2 else 0),
                         dtype=torch.uint8, device=dev)
        call = lambda: st.tree_attention(q, kc, vc, plen, kt, vt, tree, out=out, lse=lse, ws=ws)
        L = [int(x) for x in ax["prefix_len"]]
        abytes = (sum(L) * w.Hkv * w.D * 2 * s + w.B * w.Hq * T * w.D * s + w.B * w.Hkv * T * w.D * 2 * s
                  + w.B * w.Hq * T * (w.D + 1) * 4)
        flops = 4.0 * w.D * w.Hq * T * sum(l + T for l in L)
    elif part == "attention_paged":
        # the same layer over a paged pool: 128-key blocks scattered to a shuffled slot order
        ax = wl.attention_inputs(w, T)
        bs = 128
        n_blocks = w.Lmax // bs
        L = [int(x) for x in ax["prefix_len"]]
        slots = np.random.default_rng(w.seed).permutation(w.B * n_blocks)
        table = slots.reshape(w.B, n_blocks).astype(np.int32)
        kpool = np.empty((w.B * n_blocks, w.Hkv, bs, w.D), dtype=ax["k_cache"].dtype)
        vpool = np.empty_like(kpool)
        for b in range(w.B):
            for j in range(n_blocks):
                kpool[table[b, j]] = ax["k_cache"][b, :, j * bs:(j + 1) * bs]
                vpool[table[b, j]] = ax["v_cache"][b, :, j * bs:(j + 1) * bs]
        q, plen, kt, vt = (dev_t(ax[k]) for k in ("q", "prefix_len", "k_tree", "v_tree"))
        kp, vp, tb = dev_t(kpool), dev_t(vpool), dev_t(table)
        out = torch.empty(w.B, w.Hq, T, w.D, dtype=torch.float32, device=dev)
        lse = torch.empty(w.B, w.Hq, T, dtype=torch.float32, device=dev)
        ws = torch.empty(st.tree_attention_paged_workspace_size(tree, w.B, w.Hq, w.Hkv, n_blocks, bs, w.D,
                                                                1 if s == 2 else 0), dtype=torch.uint8, device=dev)
        call = lambda: st.tree_attention_paged(q, kp, vp, tb, plen, kt, vt, tree, out=out, lse=lse, ws=ws)
        abytes = (sum(L) * w.Hkv * w.D * 2 * s + w.B * w.Hq * T * w.D * s + w.B * w.Hkv * T * w.D * 2 * s
                  + w.B * w.Hq * T * (w.D + 1) * 4)
        flops = 4.0 * w.D * w.Hq * T * sum(l + T for l in L)
    elif part == "draft":
        dx = wl.draft_inputs(w)
        h, E, root = dev_t(dx["h"]), dev_t(dx["E"]), dev_t(dx["root_tok"])
        W1 = [dev_t(a) for a in dx["W1"]]
        b1 = [dev_t(a) for a in dx["b1"]]
        W2 = [dev_t(a) for a in dx["W2"]]
        cond, topk = list(w.cond), list(w.topk)
        nt = torch.empty(w.B, T, dtype=torch.int32, device=dev)
        nl = torch.empty(w.B, T, dtype=torch.float32, device=dev)
        nlp = torch.empty(w.B, T, dtype=torch.float32, device=dev)
        ws = torch.empty(st.hydra_draft_workspace_size(tree, w.B, w.d, w.V, cond, topk, 1), dtype=torch.uint8, device=dev)
        tabs = None if no_fold else [st.hydra_fold_embedding(W1[k], E) if c == 1 else None for k, c in enumerate(cond)]
        call = lambda: st.hydra_draft(h, E, W1, b1, W2, cond, topk, root, tree, node_tok=nt, node_logit=nl,
                                      node_logprob=nlp, ws=ws, folded=tabs)
        abytes, d, V = 0.0, w.d, w.V
        for k in range(len(cond)):
            n_int = tree.struct.n_internal_at_depth[k]
            if not n_int:
                continue
            rows = w.B * n_int if cond[k] else w.B
            d_in = d * (2 if cond[k] else 1)
            if tabs is not None and cond[k] == 1:
                # folded: the h_b half of W1 per sequence, a table row (fp32) per head-input row
                abytes += (d * d + d + V * d) * s + w.B * d * (s + 4) + rows * (d * 4 + 2 * d * s)
                flops += 2.0 * (w.B * d * d + rows * d * V)
            else:
                abytes += (d * d_in + d + V * d) * s + rows * (d_in + d) * s
                flops += 2.0 * rows * (d_in * d + d * V)
    elif part == "draft_ln":
        # the LayerNorm fusion head form at Vicuna-7B shape (d 4096, V 32000, inner width 1024):
        # head 1 Linear -> SiLU -> LayerNorm, heads 2-4 Linear -> SiLU -> Linear -> LayerNorm on [h || E[parent]]
        d, V, hid, B = 4096, 32000, 1024, 1
        nrm = lambda key, shape, std: dev_t(wl.normal((w.seed, 7) + key, shape, std, "bf16"))
        h, E = nrm((0,), (B, d), 1.0), nrm((1,), (V, d), 0.02)
        root = dev_t(np.zeros(B, dtype=np.int32))
        heads = [dict(form=1, cond=0, topk=8, W1=nrm((10,), (d, d), 0.02), b1=nrm((11,), (d,), 0.02),
                      gamma=nrm((12,), (d,), 1.0), beta=nrm((13,), (d,), 0.02), W2=nrm((14,), (V, d), 0.02))]
        for k, tk in zip(range(1, 4), (4, 2, 1)):
            heads.append(dict(form=1, cond=1, topk=tk, W1=nrm((20 + k,), (hid, 2 * d), 0.02),
                              b1=nrm((30 + k,), (hid,), 0.02), W1b=nrm((40 + k,), (d, hid), 0.02),
                              b1b=nrm((50 + k,), (d,), 0.02), gamma=nrm((60 + k,), (d,), 1.0),
                              beta=nrm((70 + k,), (d,), 0.02), W2=nrm((80 + k,), (V, d), 0.02)))
        nt = torch.empty(B, T, dtype=torch.int32, device=dev)
        nl = torch.empty(B, T, dtype=torch.float32, device=dev)
        nlp = torch.empty(B, T, dtype=torch.float32, device=dev)
        ws = None
        call = lambda: st.hydra_draft_heads(h, E, heads, root, tree, node_tok=nt, node_logit=nl, node_logprob=nlp)
        abytes = 0.0
        for k, hd in enumerate(heads):
            n_int = tree.struct.n_internal_at_depth[k]
            abytes += sum(hd[n].numel() * 2 for n in ("W1", "W1b", "W2") if n in hd) + B * n_int * 3 * d * 2
            flops += 2.0 * B * n_int * sum(hd[n].numel() for n in ("W1", "W1b", "W2") if n in hd)
    elif part == "accept_typical":
        # Medusa typical acceptance on the long-context workload's target logits (epsilon 0.09, alpha 0.3)
        rx = wl.rejection_inputs(w, parent, rank_arr)
        lp, tok = dev_t(rx["logits_p"]), dev_t(rx["node_tok"])
        abytes = 2.0 * w.B * T * w.V * 4    # the entropy pass reads every row; the walk reads the node rows again
        outs = [torch.empty(w.B, dtype=torch.int32, device=dev),
                torch.empty(w.B, tree.max_depth + 1, dtype=torch.int32, device=dev),
                torch.empty(w.B, dtype=torch.int32, device=dev), torch.empty(w.B, dtype=torch.float32, device=dev)]
        ws = torch.empty(st.tree_accept_workspace_size(2, tree, w.B, w.V), dtype=torch.uint8, device=dev)
        call = lambda: st.tree_accept_typical(lp, tok, tree, temperature=w.temperature, epsilon=0.09, alpha=0.3,
                                              seed=w.philox_seed, accept_len=outs[0], accept_path=outs[1],
                                              next_token=outs[2], margin=outs[3], ws=ws)
    elif part in ("commit", "commit_paged"):
        # paths from the library's own greedy acceptance on planted target logits (once, untimed)
        ax = wl.attention_inputs(w, T)
        kc, vc, kt, vt = (dev_t(ax[k]) for k in ("k_cache", "v_cache", "k_tree", "v_tree"))
        plen0 = dev_t(np.minimum(ax["prefix_len"], w.Lmax - tree.max_depth - 1).astype(np.int32))
        plen = plen0.clone()
        gw = wl.Workload("paths", "f32", B=w.B, seed=w.seed, tree=w.tree, V=4096, accept_lengths=(1, 2, 3, 4))
        gx = wl.greedy_inputs(gw, parent)
        alen, apath, _, _ = st.tree_accept(0, dev_t(gx["logits_p"]), None, dev_t(gx["node_tok"]), tree)
        ws = torch.empty(st.tree_kv_commit_workspace_size(), dtype=torch.uint8, device=dev)
        rows = int(alen.sum().item()) + w.B                   # committed rows per head, over the batch
        abytes = 2.0 * 2 * rows * w.Hkv * w.D * s             # K and V, read from the tree and written to the cache
        pre = lambda: plen.copy_(plen0)                       # every call commits onto the same prefix
        if part == "commit_paged":
            # the same commit into a paged pool: 128-row blocks in a shuffled slot order
            bs = 128
            n_blocks = -(-w.Lmax // bs)
            order = np.random.default_rng(w.seed).permutation(w.B * n_blocks).astype(np.int32)
            table = dev_t(order.reshape(w.B, n_blocks))
            kpool = torch.empty(w.B * n_blocks, w.Hkv, bs, w.D, dtype=kc.dtype, device=dev)
            vpool = torch.empty_like(kpool)
            call = lambda: st.tree_kv_commit_paged(kt, vt, kpool, vpool, table, bs, plen, alen, apath, tree, ws=ws)
        else:
            call = lambda: st.tree_kv_commit(kt, vt, kc, vc, plen, alen, apath, tree, ws=ws)
    else:
        B = w.B
        if w.accept == "greedy":
            gx = wl.greedy_inputs(w, parent)
            lp, tok = dev_t(gx["logits_p"]), dev_t(gx["node_tok"])
            lq = None
            mode, abytes = 0, B * T * w.V * 4
        else:
            rx = wl.rejection_inputs(w, parent, rank_arr)
            lp, lq, tok = dev_t(rx["logits_p"]), dev_t(rx["logits_q"]), dev_t(rx["node_tok"])
            mode = 1
            n_int = sum(tree.struct.n_internal_at_depth[k] for k in range(tree.max_depth + 1))
            abytes = B * T * w.V * 4 + B * n_int * w.V * 4
        outs = [torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, tree.max_depth + 1, dtype=torch.int32, device=dev),
                torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.float32, device=dev)]
        ws = torch.empty(st.tree_accept_workspace_size(mode, tree, B, w.V), dtype=torch.uint8, device=dev)
        call = lambda: st.tree_accept(mode, lp, lq, tok, tree, temperature=w.temperature, seed=w.philox_seed,
                                      accept_len=outs[0], accept_path=outs[1], next_token=outs[2], margin=outs[3], ws=ws)

    if part not in ("commit", "commit_paged"):
        pre = lambda: None
    comp = {"name": name, "config_id": wid, "dtype": w.dtype, "tree_nodes": T, "call": call, "pre": pre,
            "abytes": abytes, "flops": flops, "report": lambda: {}, "kernel_work": {}}
    # algorithmic work per launch of the kernels whose roofline the entry reports
    if part in ("attention", "attention_paged"):
        comp["kernel_work"]["attn_tc"] = (abytes - w.B * w.Hq * T * (w.D + 1) * 4, flops)
    elif part == "draft":
        heads = [k for k in range(len(w.cond)) if tree.struct.n_internal_at_depth[k]]
        rows = [w.B * tree.struct.n_internal_at_depth[k] if w.cond[k] else w.B for k in heads]
        comp["kernel_work"]["draft_proj_tc"] = (sum(w.V * w.d * s + r * w.d * s for r in rows) / len(rows),
                                                sum(2.0 * r * w.d * w.V for r in rows) / len(rows))
    elif part == "accept":
        comp["kernel_work"]["accept_rows_greedy" if w.accept == "greedy" else "accept_rows_lse"] = (abytes, 0.0)
    if part == "draft":
        def near_ties():
            # the drafted top-k ranks that sit within the bf16 tie tolerance (1e-3 |logit|) of the
            # next rank in the GPU's own logits (siblings of consecutive ranks)
            tok_l = nl.cpu().numpy()
            ties, pairs = 0, 0
            for u in range(T):
                kids = [c for c in range(1, T) if parent[c] == u]
                by_rank = {int(rank_arr[c]): c for c in kids}
                for r in by_rank:
                    if r + 1 in by_rank:
                        a_, b_ = tok_l[:, by_rank[r]], tok_l[:, by_rank[r + 1]]
                        pairs += a_.size
                        ties += int(np.sum(np.abs(a_ - b_) <= 1e-3 * np.abs(a_)))
            return {"near_ties": ties, "sibling_pairs_checked": pairs,
                    "near_tie_rule": "consecutive-rank siblings within 1e-3 x |logit| (bf16 tie tolerance)"}
        comp["report"] = near_ties
        comp["folded"] = tabs is not None
    if part == "accept" and w.accept == "rejection":
        def near_threshold(n_offsets=64):
            # |u - p/q| < 1e-6 decisions and CDF-breakpoint draws within 1e-6 of the total, over
            # n_offsets Philox offsets (the margin output is the smallest such distance per sequence)
            margins, lens = [], []
            for off in range(n_offsets):
                st.tree_accept(mode, lp, lq, tok, tree, temperature=w.temperature, seed=w.philox_seed, offset=off,
                               accept_len=outs[0], accept_path=outs[1], next_token=outs[2], margin=outs[3], ws=ws)
                margins.append(outs[3].cpu().numpy().copy())
                lens.append(outs[0].cpu().numpy().copy())
            m = np.concatenate(margins)
            return {"offsets": n_offsets, "near_threshold": int(np.sum(m < 1e-6)), "min_margin": float(m.min()),
                    "near_threshold_rule": "smallest |u - p/q| over decided edges, or the draw's distance to a CDF "
                                           "breakpoint over the total, below 1e-6",
                    "mean_accept_len": float(np.concatenate(lens).mean())}
        comp["report"] = near_threshold
    if part == "accept" and w.accept == "greedy":
        comp["report"] = lambda: {"exact_argmax_ties": int(np.sum(outs[3].cpu().numpy() == 0.0))}
    return comp


def graph_times(fn, pre, flush, n):
    """fn captured once into a CUDA graph (after a warm-up call on the capture stream), then
    replayed n times, each after pre() and an L2 flush, timed with CUDA events: the device time
    of the same work without the per-call host work (argument checks, tensor maps, launches)."""
    import torch
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        pre()
        fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    pre()
    with torch.cuda.graph(g):
        fn()
    evs = []
    for i in range(n + 3):
        pre()
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        if i >= 3:
            evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def measure_component(comp, flush, clocks, steps, min_wall_s=0.4):
    """CUDA-event time of one call (L2 flushed before each), a traced pass for
    per-kernel times, the clock record of the timed window, and the roofline."""
    import torch
    import tree_speculative_decoding_spec_gb300 as st
    stream = torch.cuda.current_stream()
    call, pre = comp["call"], comp["pre"]

    def timed(n):
        evs = []
        for _ in range(n):
            pre()
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    timed(3)
    ms = []
    t0 = time.time()
    while len(ms) < steps or time.time() - t0 < min_wall_s:
        ms += timed(max(steps // 2, 5))
    t1 = time.time()
    st.spec_trace_begin(100000)
    timed(max(steps // 2, 5))
    kernels = st.spec_trace_end(64)
    us = 1000.0 * statistics.median(ms)
    hbm, tf_burst, _, src = peaks()
    abytes, flops = comp["abytes"], comp["flops"]
    t_hbm, t_tc = abytes / hbm / 1e3, (flops / tf_burst / 1e6 if flops else 0.0)
    bound = "tensor" if t_tc > t_hbm else "hbm"
    kern = {k: {"launches": n, "us_per_launch": 1000.0 * t / n} for k, (n, t) in kernels.items()}
    # the kernel roofline: the entry's main kernel, its algorithmic work per launch over its mean
    # traced launch time; entries without one (the tiny launch-bound step) report the call's
    work = [(k, kw) for k, kw in comp["kernel_work"].items() if k in kern]
    if work:
        dom, (kb, kf) = max(work, key=lambda x: kern[x[0]]["us_per_launch"] * kern[x[0]]["launches"])
        dom_us = kern[dom]["us_per_launch"]
    else:
        dom, kb, kf, dom_us = "whole call", abytes, flops, us
    k_bound = "tensor" if kf / tf_burst / 1e6 > kb / hbm / 1e3 else "hbm"
    if k_bound == "tensor":
        ach = kf / dom_us / 1e6
        roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": tf_burst, "unit": "TFLOP/s",
                "frac": ach / tf_burst, "kernel_us": dom_us, "kernel_flops": kf}
    else:
        ach = kb / dom_us / 1e3
        roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "kernel_us": dom_us, "kernel_bytes": kb}
    roof["call_bound"] = bound
    roof.update({"peak_source": src, "call_hbm_frac": abytes / us / 1e3 / hbm,
                 "call_tensor_frac": (flops / us / 1e6) / tf_burst if flops else None,
                 "roofline_us": max(t_hbm, t_tc), "algorithmic_bytes": abytes, "flops": flops})
    out = {"us_per_call": us, "calls_per_s": 1e6 / us, "calls_timed": len(ms), "kernels": kern, "roofline": roof,
           "clocks": clocks.summary(t0, t1) if clocks is not None else None}
    # the same call replayed from a CUDA graph
    try:
        tg0 = time.time()
        gms = graph_times(call, pre, flush, max(steps, 20))
        tg1 = time.time()
        out["graph"] = {"us_per_call": 1000.0 * statistics.median(gms), "calls_timed": len(gms),
                        "clocks": clocks.summary(tg0, tg1) if clocks is not None else None}
    except Exception as e:   # a call that cannot be captured reports why
        out["graph"] = {"unavailable": str(e).splitlines()[0][:200]}
    out.update(comp["report"]())
    return out


def run_component(args):
    """Time one entry point on one of the parity workloads (a separate line, not the headline step)."""
    import torch
    _, local, _ = dist_info()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    comp = make_component(args.workload, dev, no_fold=args.no_fold)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    m = measure_component(comp, L2Flush(dev), clocks, args.steps)
    clocks.stop()
    line = {"workload": args.workload, "config_id": comp["config_id"], "impl": "ours", "metric": "calls/s",
            "value": m["calls_per_s"], "dtype": comp["dtype"], "steps": args.steps, "tree_nodes": comp["tree_nodes"]}
    line.update(m)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fold", action="store_true",
                    help="draft heads stream their whole first layer (no folded embedding tables)")
    ap.add_argument("--workload", choices=["step"] + sorted(COMPONENTS), default="step",
                    help="step (default): the headline verification step; otherwise one entry point on one workload")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config entries of the default line")
    ap.add_argument("--oracle-step", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_step:
        run_oracle_step_child()
        return
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "step":
        run_component(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
