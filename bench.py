#!/usr/bin/env python
"""Benchmark: Medusa verify steps per second on one GB300 (or N replicas).

One step = the whole hot path on one batch of synthetic inputs: tree-masked
attention with KV append, LM head over every tree row, acceptance, KV
compaction, the Medusa heads with top-s, and the next candidate tree -- six
libmedusa calls (11 kernels), captured once in a CUDA graph.

Default workload: Vicuna-7B shape (d=4096, V=32000, 32x128 heads), prefix
1024, 64-node greedy sparse tree (65 rows), 4 Medusa heads, batch 1, greedy
acceptance, bf16.  Weights and activations are seeded synthetic tensors;
1.48 GB of weights stream per step, more than the 126 MB L2, so nothing is
served from L2 across steps.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Medusa verify-steps/s, 7B shape, 64-node tree, bs1; % of HBM roofline"
UNIT = "verify-steps/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--plant-depth", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--loop-steps", type=int, default=48,
                    help="chained verify steps on the device around the stand-in backbone (0: skip)")
    ap.add_argument("--accept", choices=["separate", "fused"], default="separate",
                    help="acceptance reading the logits (separate) or the row statistics fused into the LM "
                         "head's epilogue (fused)")
    ap.add_argument("--no-logits", dest="logits", action="store_false",
                    help="with --accept fused and greedy acceptance: do not write the logits")
    ap.add_argument("--heads", choices=["split", "fused", "joint"], default="fused",
                    help="heads' W1 over every tree row beside the acceptance, then W2 on the accepted "
                         "row (split), W1 over every row inside the LM head's launch, then W2 (joint), or "
                         "both projections on the accepted row after the acceptance (fused)")
    ap.add_argument("--attn-branch", choices=["serial", "fork"], default="fork",
                    help="tree attention before the LM head on one stream, or on a forked graph branch")
    ap.add_argument("--attn-order", choices=["first", "after_lm", "after_accept", "after_heads"], default="after_lm",
                    help="attention enqueued before the LM head or right after it (its CTAs then fill the "
                         "SMs the LM head leaves idle)")
    ap.add_argument("--attn-splits", choices=["1", "2", "4", "8", "tc", "tc1", "tc2", "tc4", "tc8"], default=None,
                    help="CTAs that split one head's keys, or tc[N] for the tensor-core attention with N "
                         "(default: one wave of CTAs) (default: 4 for bf16)")
    return ap.parse_args()


# ------------------------------------------------------------------ bytes --

def algorithmic_bytes(w: dict, T: int, s_heads, L_list, heads_mode: str, fused_accept: bool = False,
                      logits: bool = True) -> dict:
    """Bytes each call must move at least once per step (weights once, KV
    prefix once, activations and logits once each way)."""
    e = 2 if w["dtype"] == "bf16" else 4
    B, H, Dh, d, V = w["B"], w["H"], w["Dh"], w["d"], w["V"]
    k_used = sum(1 for s in s_heads if s > 0)
    sumL = int(np.sum(L_list))
    attn = (2 * sumL * H * Dh * e          # cached K, V read
            + 3 * B * T * H * Dh * e       # q, k_new, v_new read
            + 2 * B * T * H * Dh * e       # K', V appended
            + B * T * H * Dh * e)          # out written
    lm = V * d * e + B * T * d * e + (B * T * V * 4 if logits else 0)
    accept = B * T * V * 4
    if fused_accept:  # per-group row records instead of a logits pass
        from medusa_tree_speculative_gb300 import medusa as M

        rec = M.medusa_lm_head_stat_groups(B * T, V) * B * T * 16
        lm += rec
        accept = rec
    compact = 2 * 2 * B * (w["K"] + 1) * H * Dh * e
    heads = k_used * (d * d + V * d) * e + B * k_used * V * 4 * 2
    # split heads: W1 over every tree row (u of all rows written), then W2 on the accepted row
    heads_hidden = k_used * d * d * e + B * T * d * e + B * T * k_used * d * e
    heads_w2 = k_used * V * d * e + B * k_used * d * e + B * k_used * V * 4 * 2
    cand = B * T * 4
    out = dict(tree_attn=attn, lm_head_verify=lm, accept=accept, kv_compact=compact,
               build_candidates=cand)
    if heads_mode == "split":
        out.update(heads_hidden=heads_hidden, heads_logits_topk=heads_w2)
    elif heads_mode == "joint":  # W1 streams in the LM head's launch (hidden read once for both)
        out["lm_head_verify"] += heads_hidden - B * T * d * e
        out["heads_logits_topk"] = heads_w2
    else:  # medusa_heads_topk_candidates: the candidate fill runs in the heads' last CTA
        out["heads_topk"] = heads + out.pop("build_candidates")
    out["step"] = sum(out.values())
    return out


def algorithmic_flops(w, T, s_heads, L_list):
    B, H, Dh, d, V = w["B"], w["H"], w["Dh"], w["d"], w["V"]
    k_used = sum(1 for s in s_heads if s > 0)
    return dict(tree_attn=4 * T * (int(np.sum(L_list)) + B * T) * H * Dh,
                lm_head_verify=2 * B * T * d * V,
                heads_topk=2 * B * k_used * (d * d + d * V),
                heads_hidden=2 * B * T * k_used * d * d,
                heads_logits_topk=2 * B * k_used * d * V)


def weight_bytes(w, s_heads):
    """Weights one step streams: the vocabulary matrix and the heads in use."""
    e = 2 if w["dtype"] == "bf16" else 4
    k_used = sum(1 for s in s_heads if s > 0)
    return (w["V"] * w["d"] + k_used * (w["d"] * w["d"] + w["V"] * w["d"])) * e


def floor_us(nbytes, flops, peaks):
    """max(bytes / measured copy bandwidth, flops / sustained bf16 tensor
    rate) in microseconds: the roofline floor of one call."""
    return max(nbytes / (peaks["hbm_gbs"] * 1e3), flops / (peaks["bf16_tflops_sustained"] * 1e6))


def step_floor(by, fl, peaks, ms):
    """The step's floor: all its bytes at the copy bandwidth, or all its
    flops at the sustained tensor rate, whichever is longer."""
    tb = by["step"]
    tf = sum(fl[c] for c in ("tree_attn", "lm_head_verify", "heads_topk") if c in fl)
    us = floor_us(tb, tf, peaks)
    return {"bytes": tb, "flops": tf, "floor_us": round(us, 2), "frac": round(us / (ms * 1e3), 4),
            "bound": "hbm" if tb / (peaks["hbm_gbs"] * 1e3) >= tf / (peaks["bf16_tflops_sustained"] * 1e6) else "tensor"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm_gbs=float(j["hbm_gbs"]), bf16_tflops=float(j["bf16_tflops"]),
                    bf16_tflops_sustained=float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def ncu_traffic(kernel_key: str, workload: str):
    """DRAM bytes per launch of a call on a workload, from the committed ncu
    summary (key "call@workload"), or None when there is none or the
    kernel's source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    ent = j.get(f"{kernel_key}@{workload}")
    if not ent:
        return None
    src = os.path.join(ROOT, ent["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != ent["sha"]:
        return None
    return ent["dram_bytes_per_launch_full"]


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
            os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(float(r[2]) for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- native --

def plant(w, tree, st, x, depth, torch):
    """Set the tokens along one root->node path (node at `depth`) to the
    parent-row argmax of the LM head, so acceptance takes that path; off the
    path, tokens differ from the parent's argmax.  Setup only, untimed."""
    from medusa_tree_speculative_gb300 import medusa as M

    ht = tree.host
    M.medusa_lm_head_verify(x["hidden"], st.w_lm, st.logits)
    am = torch.argmax(st.logits, dim=-1).cpu().numpy()  # [B, T]
    cands = np.nonzero(ht.depth == min(depth, ht.K))[0]
    tok = x["tokens"].cpu().numpy()
    for b in range(w["B"]):
        node = int(cands[(7 * b + 3) % len(cands)])
        path = set()
        n = node
        while n > 0:
            path.add(n)
            n = int(ht.parent[n])
        for c in range(1, ht.T):
            p = int(ht.parent[c])
            tok[b, c] = am[b, p] if c in path else (am[b, p] + 1 + c) % w["V"]
    x["tokens"].copy_(torch.from_numpy(tok))


def step_calls(st, x, s):
    """The step's library calls in stream order on one stream, as (name, call)."""
    from medusa_tree_speculative_gb300 import medusa as M

    joint = st.heads == "joint"
    c = [("tree_attn", lambda: st.attention(x, s)),
         ("lm_head_verify", (lambda: M.medusa_lm_head_verify_heads_hidden(
             x["hidden"], st.w_lm_run, st.logits.shape[-1], st.logits, st.w1_run, st.b1, st.s_heads, st.u_all,
             st.err, s, layout=st.w_layout, w1_layout=st.w1_layout)) if joint else
          (lambda: M.medusa_lm_head_verify_stats(
             x["hidden"], st.w_lm_run, st.logits if st.write_logits else None, st.stats, st.mode, st.temperature,
             st.logits.shape[-1], st.err, s, layout=st.w_layout)) if st.accept == "fused" else
          (lambda: M.medusa_lm_head_verify(x["hidden"], st.w_lm_run, st.logits, None, st.err, s,
                                           layout=st.w_layout)))]
    if st.heads == "split":
        c.append(("heads_hidden", lambda: M.medusa_heads_hidden(x["hidden"], st.w1_run, st.b1, st.s_heads, st.u_all,
                                                                st.err, s, layout=st.w1_layout)))
    c += [("accept", (lambda: M.medusa_accept_stats(
              st.stats, st.stat_groups, st.logits if st.write_logits else None, x["tokens"], st.tree, st.mode,
              st.temperature, st.eps, st.delta, st.logits.shape[-1], st.accept_len, st.accepted_nodes, st.next_root,
              st.best_node, st.best_logp, st.err, s)) if st.accept == "fused" else
           (lambda: M.medusa_accept(st.logits, x["tokens"], st.tree, st.mode, st.temperature, st.eps, st.delta,
                                    st.accept_len, st.accepted_nodes, st.next_root, st.best_node, st.best_logp,
                                    st.ws_accept, st.err, s))),
          ("kv_compact", lambda: M.medusa_kv_compact(x["k_cache"], x["v_cache"], x["seq_start"], x["prefix_len"],
                                                     st.accepted_nodes, st.accept_len, st.tree.K, st.tree.T,
                                                     st.src_slots, st.err, s))]
    if st.heads in ("split", "joint"):
        c.append(("heads_logits_topk", lambda: M.medusa_heads_logits_topk(
            st.u_all, st.T, st.best_node, st.w2, st.s_heads, st.head_logits, st.topk, st.ws_w2, st.err, s)))
        c.append(("build_candidates", lambda: M.medusa_build_candidates(st.next_root, st.topk, st.tree,
                                                                        st.next_tokens, s)))
    else:  # the heads' last CTA fills the candidates too
        c.append(("heads_topk", lambda: M.medusa_heads_topk_candidates(
            x["hidden"], st.best_node, st.w1, st.b1, st.w2, st.s_heads, st.head_logits, st.topk, st.ws_heads,
            st.next_root, st.tree, st.next_tokens, st.err, s)))
    return c


def run_native(args, w, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from medusa_tree_speculative_gb300 import medusa as M
    from medusa_tree_speculative_gb300 import step, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ht = step.build_tree(w)
    tree = M.DeviceTree(ht, dev)
    T = tree.T
    seed = 0  # every replica runs the same workload
    wts = synth.make_weights(w, seed)
    xh = synth.make_step(w, T, seed)
    dt = w["dtype"]
    wd = {k: (None if v is None else step.host_to_torch(v, dt).to(dev)) for k, v in wts.items()}
    keep_host = world == 1 and not args.no_cpu_baseline  # the CPU baseline runs on the same inputs
    if not keep_host:
        del wts
    x = {}
    for k, v in xh.items():
        x[k] = step.host_to_torch(v, dt).to(dev) if v.dtype in (np.uint16, np.float32) else torch.from_numpy(v).to(dev)
    L_list = xh["prefix_len"].copy()
    st = step.VerifyStep(w, wd, tree, max_prefix=int(L_list.max()), device=dev, heads=args.heads,
                         accept=args.accept, write_logits=args.logits, attn_order=args.attn_order,
                         attn_splits=(args.attn_splits if args.attn_splits.startswith("tc") else int(args.attn_splits))
                         if args.attn_splits else "auto")
    plant(w, tree, st, x, args.plant_depth, torch)
    prefix0 = x["prefix_len"].clone()
    s = torch.cuda.Stream(device=dev)
    # eager warm-up (JIT, attributes) then one checked step
    with torch.cuda.stream(s):
        for _ in range(2):
            x["prefix_len"].copy_(prefix0)
            st.run(x, s)
    torch.cuda.synchronize()
    if int(st.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(st.err.item())} after warm-up")
    accept_len = st.accept_len.cpu().numpy().tolist()

    # one graph holds K steps with timing events at every call boundary
    calls = [c for c, _ in step_calls(st, x, s)]
    s2 = torch.cuda.Stream(device=dev) if args.attn_branch == "fork" else None  # side branch for attention
    s3 = torch.cuda.Stream(device=dev) if args.heads == "split" else None  # branch for W1 beside the acceptance

    def capture(nsteps, with_events):
        g = torch.cuda.CUDAGraph()
        evs = []
        with torch.cuda.graph(g, stream=s):
            for _ in range(nsteps):
                if with_events or s2 is None:
                    x["prefix_len"].copy_(prefix0)
                else:
                    # every step starts from the same prefix (bench plumbing, not
                    # part of the method); only the attention's branch reads
                    # prefix_len before the compaction, so the restore runs
                    # there and the LM head does not wait for it
                    s2.wait_stream(s)
                    with torch.cuda.stream(s2):
                        x["prefix_len"].copy_(prefix0)
                if with_events:
                    e = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(calls) + 1)]
                    evs.append(e)
                    run_calls(st, x, s, e)
                else:
                    st.run(x, s, side_stream=s2, heads_stream=s3)
        return g, evs

    def run_calls(st, x, s, e):
        for i, (_, call) in enumerate(step_calls(st, x, s)):
            e[i].record(s)
            call()
        e[-1].record(s)

    g_warm, _ = capture(1, False)
    g_timed, evs = capture(args.steps, True)
    g_plain, _ = capture(args.steps, False)
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            g_warm.replay()
    torch.cuda.synchronize()

    def timed(graph):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):  # replay() launches on the current stream
            t0.record(s)
            graph.replay()
            t1.record(s)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return t0.elapsed_time(t1)

    with ClockSampler(local_rank) as clk:
        ms_plain = timed(g_plain)   # the headline number: no event nodes in the graph
        ms_events = timed(g_timed)  # same steps with per-call events
    clocks = clk.summary()
    per_call = {c: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) for i, c in enumerate(calls)}
    if int(st.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(st.err.item())} in the timed region")

    ms_total = max_over_ranks(ms_plain, dev) if world > 1 else ms_plain
    ms_step = ms_total / args.steps

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, w, st, x, xh, prefix0, s, s2, s3, torch, M)
    rej = measure_rejection(st, x, s, torch, M) if world == 1 else None
    attn_alone = (measure_attn_alone(st, x, prefix0, L_list, torch, M)
                  if world == 1 and st.attn_splits == "tc" else None)
    dloop = None
    if args.loop_steps > 0 and world == 1:
        if len(set(int(v) for v in L_list)) == 1:
            dloop = measure_loop(args, w, dev, torch, M)
        else:  # DecodeLoop starts every sequence at one prefix length
            dloop = {"skipped": "ragged prefix lengths; the decode loop runs with one prefix length for the batch"}

    return dict(host_inputs=(wts, xh) if keep_host else None, attn_alone=attn_alone,
                ms_step=ms_step, ms_events_step=ms_events / args.steps, per_call_ms=per_call, clocks=clocks,
                dloop=dloop, rej=rej,
                T=T, s_heads=st.s_heads, L_list=L_list, accept_len=accept_len, e2e=e2e,
                launches=st.launches_per_step * args.steps, tree=ht,
                attn_splits=f"tc{st.tc_splits}" if st.attn_splits == "tc" else st.attn_splits or 8)


def measure_attn_alone(st, x, prefix0, L_list, torch, M, reps=10):
    """The tree attention on its own, as its roofline is measured: the key split
    that fills the GPU (step.tc_key_splits over every SM), L2 flushed before
    each launch (a 256 MB buffer written, then read back so that L2 holds its
    clean lines: after a write alone the dirty lines' write-back lands in the
    timed launch), CUDA events around the launch alone; median of `reps`.  The
    step itself runs it beside the LM head instead."""
    from medusa_tree_speculative_gb300 import step

    B, T, H, Dh = st.out.shape
    sms = torch.cuda.get_device_properties(st.out.device).multi_processor_count
    ns = step.tc_key_splits(B, H, T, int(max(L_list)), sms)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=st.out.device)
    sink = torch.zeros(1, dtype=torch.int64, device=st.out.device)
    s = torch.cuda.Stream(device=st.out.device)

    def call():
        M.medusa_tree_attn_tc(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["seq_start"],
                              x["prefix_len"], x["seq_cap"], st.tree, st.max_prefix, st.rope_theta, st.scale,
                              st.out, st.err, s, key_splits=ns)

    ts = []
    for i in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            x["prefix_len"].copy_(prefix0)  # the steps before advanced it by the accepted tokens
            flush.fill_(1)
            sink.add_(flush.view(torch.int32).sum(dtype=torch.int64))
            e0.record(s)
            call()
            e1.record(s)
        torch.cuda.synchronize()
        if i:  # the first launch is a warm-up
            ts.append(e0.elapsed_time(e1) * 1e3)
    if int(st.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(st.err.item())} in the attention-alone launches")
    us = statistics.median(ts)
    e = st.out.element_size()
    kv = 2 * int(np.sum(L_list)) * H * Dh * e
    act = 6 * B * T * H * Dh * e  # q, k_new, v_new read; K', V' appended; out written
    return {"key_splits": ns, "us": us, "kv_bytes": kv, "bytes": kv + act, "gbs": (kv + act) / us / 1e3,
            "how": "median of %d launches, each after a 256 MB write and read-back that flush L2" % reps}


def measure_rejection(st, x, s, torch, M, reps=20):
    """medusa_accept_rejection on the step's own logits, with the heads'
    logits as the drafts and device uniforms: time per call (graph of reps
    calls) beside the greedy / typical acceptance of the same step."""
    B, T, V = st.logits.shape
    g = torch.Generator(device=st.logits.device).manual_seed(7)
    u = torch.rand((B, T, 17), generator=g, device=st.logits.device)
    al = torch.zeros(B, dtype=torch.int32, device=u.device)
    an = torch.zeros((B, st.tree.K + 1), dtype=torch.int32, device=u.device)
    nt = torch.zeros(B, dtype=torch.int32, device=u.device)
    ws = torch.empty(M.medusa_accept_rejection_workspace_size(B, V), dtype=torch.uint8, device=u.device)
    tau = st.temperature if st.mode == 1 else 1.0

    def call():
        M.medusa_accept_rejection(st.logits, st.head_logits, x["tokens"], st.tree, tau, u, al, an, nt, ws, st.err, s)

    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        for _ in range(reps):
            call()
    ts = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            gr.replay()
            e1.record(s)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / reps)
    return {"ms_per_call": statistics.median(ts), "temperature": tau, "accept_len": al.cpu().tolist(),
            "drafts": "the step's tree tokens, q = the heads' softmax, uniforms from the device generator"}


def measure_loop(args, w, dev, torch, M):
    """Chained steps (the decode loop of medusa_tree_speculative_gb300.loop):
    each step's tree comes from the previous one, on the device, around the
    stand-in backbone (an embedding lookup).  One CUDA graph of n steps,
    re-primed before every replay; the emitted tokens are checked against the
    stand-in model's greedy continuation."""
    from medusa_tree_speculative_gb300 import loop, step

    n = args.loop_steps
    tree = M.DeviceTree(step.build_tree(w), dev)
    model = loop.StandInModel(w, seed=3, device=dev)
    x0 = np.array([(97 * b + 5) % w["V"] for b in range(w["B"])])
    L0 = int(w["L"][0])
    lp = loop.DecodeLoop(w, model, tree, n, L0=L0, x0=x0, device=dev, heads=args.heads)
    s = torch.cuda.Stream(device=dev)
    s2 = torch.cuda.Stream(device=dev) if args.attn_branch == "fork" else None
    s3 = torch.cuda.Stream(device=dev) if args.heads == "split" else None

    def reset():
        with torch.cuda.stream(s):
            lp.x["prefix_len"].fill_(L0)
            lp._prime()
        torch.cuda.synchronize()

    reset()
    with torch.cuda.stream(s):
        lp.step(s, s2, s3)  # eager once (attributes, tensor maps)
    reset()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(n):
            lp.step(s, s2, s3)
    times = []
    for _ in range(3):
        reset()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if int(lp.st.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(lp.st.err.item())} in the decode loop")
    got = lp.emitted()
    ref = lp.greedy_reference(max(len(t) for t in got))
    ok = all(np.array_equal(got[b], ref[b, :len(got[b])]) for b in range(w["B"]))
    ms = statistics.median(times)
    tokens = sum(len(t) for t in got)
    return {"steps": n, "tokens": tokens, "tokens_per_step": tokens / (n * w["B"]),
            "verify_steps_per_s": n * 1e3 / ms, "tokens_per_s": tokens * 1e3 / ms,
            "ms_per_step": ms / n, "matches_greedy_decoding": bool(ok),
            "backbone": "stand-in: hidden state and q/k/v of a token = its embedding row; LM head and heads "
                        "built on a fixed next-token chain, heads' W2 with Gaussian noise (sigma 0.20-0.29)",
            "gpu_launches_per_step": lp.launches_per_step()}


def measure_e2e(args, w, st, x, xh, prefix0, s, s2, s3, torch, M):
    """Same metric through the public C-ABI calls with host buffers: per step,
    pinned host inputs -> device, the six calls, results -> pinned host."""
    # the step's inputs staged in one pinned host buffer and one device buffer
    # (one copy each way per step; the device tensors are views into it)
    names_in = ["q", "k_new", "v_new", "hidden", "tokens", "prefix_len"]
    src = {k: (prefix0 if k == "prefix_len" else x[k]) for k in names_in}
    offs, n = {}, 0
    for k in names_in:
        offs[k] = n
        n += (src[k].numel() * src[k].element_size() + 255) // 256 * 256
    host_buf = torch.empty(n, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(n, dtype=torch.uint8, device=st.logits.device)
    xe = dict(x)
    for k in names_in:
        t = src[k]
        nb = t.numel() * t.element_size()
        host_buf[offs[k]:offs[k] + nb].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
        xe[k] = dev_buf[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
    host_res = torch.empty_like(st.results, device="cpu").pin_memory()
    h2d = n
    d2h = st.results.numel() * st.results.element_size()
    steps = max(10, args.steps // 2)

    # the attention's inputs (q, k_new, v_new) on the forked branch that runs
    # the attention; the LM head's and the acceptance's (hidden, tokens,
    # prefix_len) on the main stream, so that the LM head starts after its own
    # inputs only; both by copy kernels reading the pinned buffer
    split = offs["hidden"]

    def enqueue():
        s2.wait_stream(s)
        with torch.cuda.stream(s2):
            M.medusa_copy_from_host(dev_buf[:split], host_buf[:split], s2)
        M.medusa_copy_from_host(dev_buf[split:], host_buf[split:], s)
        st.run(xe, s, side_stream=s2, heads_stream=s3)
        host_res.copy_(st.results, non_blocking=True)

    # one step = pinned host inputs -> device, the six calls, results -> pinned
    # host, captured once as a CUDA graph (as a serving loop would) and replayed
    # per step; the host waits for every step's results
    with torch.cuda.stream(s):
        enqueue()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        enqueue()

    def one():
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    dt = time.perf_counter() - t0
    return {"value": steps / dt, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps,
            "launch": "one CUDA graph per step: inputs (one pinned buffer) -> device by medusa_copy_from_host (q, "
                      "k_new, v_new on the attention's branch, the rest on the main stream), the six calls, the "
                      "step's integer results -> pinned host; the host waits for every step"}


# ------------------------------------------------------------- CPU oracle --

class OracleStep:
    """One full verify step of the CPU oracle on the bench workload's own
    inputs (the same seeded weights and activations as the GPU run), chained
    as the GPU chains it: tree attention over every head, the LM head over
    every tree row and the whole vocabulary, the acceptance on the oracle's
    own logits, compaction, both head projections at the accepted node and
    the candidate fill.  `seqs` < B keeps only the first sequences of the
    batch (a sample of whole sequences; the step's time scales by B / seqs).
    Inputs are drawn once; each call times only the oracle."""

    def __init__(self, w, seed=0, seqs=None, wts=None, xh=None):
        import oracle
        from medusa_tree_speculative_gb300 import synth

        oracle.build()
        self.w = w
        if w["tree"][0] == "cartesian":
            s = list(w["tree"][1])
            n = w["tree"][2] or sum(math.prod(s[:k]) for k in range(1, len(s) + 1))
            paths, plen = oracle.tree_cartesian(s, n)
        else:
            paths, plen = oracle.tree_greedy(synth.accuracy_table(w["K"], w["tree"][2]), w["tree"][1])
        self.ot = ot = oracle.tree_compile(paths, plen, paths.shape[1])
        self.B = w["B"]
        self.nb = nb = min(self.B, seqs or self.B)
        wts = wts if wts is not None else synth.make_weights(w, seed)
        x = xh if xh is not None else synth.make_step(w, ot.T, seed)
        s_heads = [int(ot.s[k]) if k < ot.K else 0 for k in range(w["K"])]
        self.s_heads = s_heads
        self.s_max = max(1, max(s_heads))
        self.w_lm, self.w1, self.w2 = wts["w_lm"], wts["w1"], wts["w2"]
        end = int(x["seq_start"][nb - 1] + x["seq_cap"][nb - 1])  # cache rows of the first nb sequences
        self.x = {k: np.ascontiguousarray(v[:nb]) for k, v in x.items() if k not in ("k_cache", "v_cache")}
        self.k_cache = np.ascontiguousarray(x["k_cache"][:end])
        self.v_cache = np.ascontiguousarray(x["v_cache"][:end])

    def step(self):
        """Seconds for one step of the sampled sequences, per part."""
        import oracle

        w, x, ot = self.w, self.x, self.ot
        nb, T, d, V = self.nb, ot.T, w["d"], w["V"]
        t_all = {}
        kc, vc = self.k_cache.copy(), self.v_cache.copy()
        t = time.perf_counter()
        oracle.tree_attn(x["q"], x["k_new"], x["v_new"], kc, vc, x["seq_start"], x["prefix_len"], ot)
        t_all["tree_attn"] = time.perf_counter() - t
        t = time.perf_counter()
        logits = oracle.lm_head(x["hidden"].reshape(nb * T, d), self.w_lm)
        t_all["lm_head_verify"] = time.perf_counter() - t
        mode = 1 if w["mode"] == "typical" else 0
        t = time.perf_counter()
        r = oracle.accept(logits.astype(np.float32).reshape(nb, T, V), x["tokens"], ot, mode,
                          w.get("temperature", 1.0), w.get("eps", 0.09), w.get("delta", 0.3))
        t_all["accept"] = time.perf_counter() - t
        t = time.perf_counter()
        oracle.kv_compact(kc, vc, x["seq_start"], x["prefix_len"].copy(), r["accepted_nodes"], r["accept_len"],
                          ot.K)
        t_all["kv_compact"] = time.perf_counter() - t
        t = time.perf_counter()
        _, tk, _ = oracle.heads(x["hidden"], r["best_node"], self.w1, None, self.w2, self.s_heads, self.s_max)
        t_all["heads_topk"] = time.perf_counter() - t
        t = time.perf_counter()
        oracle.build_candidates(r["next_root"], tk, ot)
        t_all["build_candidates"] = time.perf_counter() - t
        return sum(t_all.values()), t_all


def oracle_seqs(w) -> int:
    """Sequences of the batch in one timed oracle step: all of them, except
    for batches whose full step would take well over half a minute on one
    core (the 33B-shaped batch of four: one sequence)."""
    return 1 if w["B"] > 1 and w["d"] * w["V"] * w["B"] > 4 * 4096 * 32000 else w["B"]


def cpu_baseline(w, wts=None, xh=None, budget_s=30.0):
    """The oracle as it stands, single-threaded, timed on full steps of the
    bench workload (whole sequences; every head, every vocabulary row)."""
    orc = OracleStep(w, seqs=oracle_seqs(w), wts=wts, xh=xh)
    vals = []
    parts = None
    t0 = time.perf_counter()
    while not vals or (len(vals) < 3 and time.perf_counter() - t0 + vals[-1] < budget_s):
        sec, parts = orc.step()
        vals.append(sec)
    sec = statistics.median(vals) * orc.B / orc.nb  # seconds per step of the whole batch
    sample = (f"single-threaded C oracle on one host core, full verify steps (every attention head, every "
              f"vocabulary row of the LM head and of each head's W2, acceptance on the oracle's own logits); "
              f"median of {len(vals)} step(s)")
    if orc.nb < orc.B:
        sample += f"; {orc.nb} of the batch's {orc.B} sequences per step, time scaled by {orc.B}/{orc.nb}"
    return {"value": 1.0 / sec, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": sample + f"; host has {os.cpu_count()} cores",
            "seconds_per_step": sec, "steps_timed": len(vals),
            "parts_s": {k: round(v, 4) for k, v in parts.items()}}


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (the slowest rank sets a replicated
    job's time); device: where the collective's tensor lives (cuda for NCCL,
    cpu for gloo)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world: int, steps: int, ms_total: float) -> float:
    """Verify-steps per second of the whole job: every rank runs `steps`
    steps of its own replica in ms_total (the slowest rank's time)."""
    return world * steps * 1e3 / ms_total


def run_reference(args, w, rank, world, budget_s=60.0):
    """--impl reference: the CPU oracle as it stands, single-threaded, on full
    verify steps of the same workload.  A full step takes seconds, so the arm
    times as many of the requested steps as fit in about a minute (at least
    one) and reports that count: every number it prints is measured."""
    if rank != 0:
        return
    import oracle

    oracle.build()
    orc = OracleStep(w, seqs=oracle_seqs(w))
    vals = []
    parts = None
    t0 = time.perf_counter()
    while len(vals) < max(1, args.steps):
        sec, parts = orc.step()
        vals.append(sec)
        if time.perf_counter() - t0 + sec > budget_s:
            break
    wall = time.perf_counter() - t0
    sec = statistics.mean(vals) * orc.B / orc.nb
    v = 1.0 / sec
    sample = (f"full verify steps of the single-threaded C oracle on one host core (every attention head, every "
              f"vocabulary row, acceptance on the oracle's own logits); {len(vals)} of the {args.steps} requested "
              f"steps timed in {wall:.1f} s wall (a full step takes {sec:.3g} s), no warm-up step")
    if orc.nb < orc.B:
        sample += f"; {orc.nb} of the batch's {orc.B} sequences per step, time scaled by {orc.B}/{orc.nb}"
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": len(vals), "warmup": 0, "steps_requested": args.steps, "warmup_requested": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, weight_bytes=weight_bytes(w, orc.s_heads)),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample + f"; host has {os.cpu_count()} cores"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "parts_s": {k: round(x, 4) for k, x in parts.items()},
    }
    print(json.dumps(line), flush=True)


def config_dict(w, extra=None, weight_bytes=None):
    c = {"workload": w["name"], "dtype": w["dtype"], "d": w["d"], "V": w["V"], "H": w["H"], "Dh": w["Dh"],
         "B": w["B"], "prefix": str(w["L"]), "K_heads": w["K"], "tree": str(w["tree"]), "accept": w["mode"]}
    if weight_bytes is not None:
        c["l2"] = (f"inputs larger than L2 ({weight_bytes / 1e9:.2f} GB of weights stream per step)"
                   if weight_bytes > 126e6 else "inputs within L2")
    if extra:
        c.update(extra)
    return c
    if extra:
        c.update(extra)
    return c


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    from medusa_tree_speculative_gb300 import workloads

    w = workloads.get(args.workload or workloads.HEADLINE)
    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist

            dist.init_process_group("gloo")
        run_reference(args, w, rank, world)
        return
    import torch

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    r = run_native(args, w, rank, world, local_rank)
    if rank != 0:
        return
    peaks = load_peaks()
    by = algorithmic_bytes(w, r["T"], r["s_heads"], r["L_list"], args.heads, args.accept == "fused" and args.heads != "joint",
                           args.logits or w["mode"] == "typical")
    fl = algorithmic_flops(w, r["T"], r["s_heads"], r["L_list"])
    ms = r["ms_step"]
    value = whole_job_value(world, args.steps, ms * args.steps)
    step_gbs = by["step"] / (ms * 1e-3) / 1e9
    dom = max((c for c in ("heads_topk", "heads_logits_topk", "lm_head_verify", "tree_attn")
               if c in r["per_call_ms"]), key=lambda c: r["per_call_ms"][c])
    dom_ms = r["per_call_ms"][dom]
    achieved = by[dom] / (dom_ms * 1e-3) / 1e9
    traffic = ncu_traffic(dom, w["name"])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic (seeded random weights and activations)",
        "config": config_dict(w, {"parallelism": f"replicas{world}" if world > 1 else "single-gpu", "attn_branch": args.attn_branch, "attn_order": args.attn_order, "attn_splits": r["attn_splits"], "heads": args.heads, "accept_impl": args.accept,
                                  "logits_written": bool(args.logits or w["mode"] == "typical"),
                                  "T_rows": r["T"], "s": r["s_heads"], "planted_accept_len": r["accept_len"]},
                              weight_bytes=weight_bytes(w, r["s_heads"])),
        "roofline": {"bound": "hbm", "kernel": "medusa_heads_topk_candidates" if dom == "heads_topk" else f"medusa_{dom}", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "algorithmic_bytes_per_launch": by[dom], "ms_per_launch": dom_ms,
                     "peak_source": peaks["source"] + " hbm_gbs (copy)"},
        "step_roofline": {"algorithmic_bytes": by["step"], "achieved_gbs": step_gbs,
                          "frac_of_measured": step_gbs / peaks["hbm_gbs"], "frac_of_8tbs": step_gbs / 8000.0},
        "per_call": {c: {"ms": round(r["per_call_ms"][c], 5), "bytes": by[c],
                         "gbs": round(by[c] / (r["per_call_ms"][c] * 1e-3) / 1e9, 1),
                         **({"tflops": round(fl[c] / (r["per_call_ms"][c] * 1e-3) / 1e12, 1)} if c in fl else {}),
                         "floor_us": round(floor_us(by[c], fl.get(c, 0), peaks), 2),
                         "frac_of_floor": round(floor_us(by[c], fl.get(c, 0), peaks) / (r["per_call_ms"][c] * 1e3), 3)}
                     for c in r["per_call_ms"]},
        "step_floor": step_floor(by, fl, peaks, ms),
        "ms_per_step_with_call_events": r["ms_events_step"],
        "clocks": r["clocks"],
        "gpu_launches": r["launches"],
    }
    if r["e2e"] is not None:
        line["e2e"] = r["e2e"]
    if r["dloop"] is not None:
        line["decode_loop"] = r["dloop"]
    if r["rej"] is not None:
        line["rejection_accept"] = r["rej"]
    if r["attn_alone"] is not None:
        a = r["attn_alone"]
        a["frac_of_measured"] = a["gbs"] / peaks["hbm_gbs"]
        line["attn_alone"] = a
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, *r["host_inputs"])
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
