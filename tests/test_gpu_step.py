"""Whole verify steps through VerifyStep (the launch configuration bench.py
times), checked against the oracle.

tiny_fp32: every output compared in full.
tiny_bf16: the tensor-core paths (attention, LM head) at a small size, every
head and vocabulary row compared.
vicuna7b_L1024_tree64 (the benchmark's workload, full size): attention on
sampled heads, LM-head logits on sampled vocabulary rows plus the planted
path's parent rows in full, acceptance against the planted path and against
the oracle's acceptance on the GPU's own logits, heads in full (top-s against
the oracle's top-s of the GPU's head logits), compaction and candidates
bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from medusa_tree_speculative_gb300 import synth, workloads
from parity_util import (ancestors, as_double, both_trees, check_accept_on_gpu_logits, gpu_topk_matches_oracle,
                         to_dev, to_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from medusa_tree_speculative_gb300 import build

    build.build()
    from medusa_tree_speculative_gb300 import medusa

    return medusa


def _tree_spec(w):
    t = w["tree"]
    return ("cartesian", t[1], t[2]) if t[0] == "cartesian" else ("greedy", w["K"], t[2], t[1])


def _run(M, name, plant_node_fn, seed=0, heads="fused"):
    from medusa_tree_speculative_gb300 import step

    w = workloads.get(name)
    ot, dtree = both_trees(M, _tree_spec(w))
    wts = synth.make_weights(w, seed)
    x = synth.make_step(w, ot.T, seed)
    node = plant_node_fn(ot)
    path = ancestors(ot.parent, node)
    # plant with the oracle's logits at the parent rows of the path
    parents = sorted(set(int(ot.parent[c]) for c in range(1, ot.T)))
    lg_par = oracle.lm_head(np.ascontiguousarray(x["hidden"][0, parents]), wts["w_lm"])
    am = {p: int(np.argmax(lg_par[i])) for i, p in enumerate(parents)}
    gaps = {p: float(np.sort(lg_par[i])[-1] - np.sort(lg_par[i])[-2]) for i, p in enumerate(parents)}
    tok = x["tokens"].copy()
    for c in range(1, ot.T):
        p = int(ot.parent[c])
        tok[0, c] = am[p] if c in path else (am[p] + 1 + c) % w["V"]
    dev = {k: to_dev(v) for k, v in x.items()}
    dev["tokens"] = to_dev(tok)
    wd = {k: (None if v is None else to_dev(v)) for k, v in wts.items()}
    st = step.VerifyStep(w, wd, dtree, max_prefix=int(x["prefix_len"].max()), heads=heads)
    # split heads: W1 over every tree row on a second stream, beside the acceptance
    st.run(dev, heads_stream=torch.cuda.Stream() if heads == "split" else None)
    torch.cuda.synchronize()
    return w, ot, wts, x, tok, st, dev, node, path, lg_par, parents, gaps


@pytest.mark.parametrize("heads", ["fused", "split"])
def test_step_tiny_fp32_full(M, heads):
    w, ot, wts, x, tok, st, dev, node, path, _, _, _ = _run(
        M, "tiny_fp32", lambda ot: int(np.nonzero(ot.depth == 3)[0][-1]), heads=heads)
    assert int(st.err.item()) == 0
    kc, vc = x["k_cache"].copy(), x["v_cache"].copy()
    _, ref = oracle.tree_attn(x["q"], x["k_new"], x["v_new"], kc, vc, x["seq_start"], x["prefix_len"], ot)
    assert np.abs(to_host(st.out) - ref).max() <= 1e-4
    lg = oracle.lm_head(x["hidden"], wts["w_lm"]).reshape(1, ot.T, w["V"])
    assert np.abs(to_host(st.logits) - lg).max() <= 1e-5 * np.abs(lg).max()
    r = oracle.accept(lg.astype(np.float32), tok, ot, 0)
    assert r["accept_len"][0] == 3
    for key in ("accept_len", "accepted_nodes", "next_root", "best_node"):
        assert np.array_equal(to_host(getattr(st, key)), r[key])
    pl = x["prefix_len"].copy()
    src = oracle.kv_compact(kc, vc, x["seq_start"], pl, r["accepted_nodes"], r["accept_len"], ot.K)
    assert np.array_equal(to_host(dev["v_cache"]), vc)
    assert np.abs(to_host(dev["k_cache"]).astype(np.float64) - kc).max() <= 1e-5
    assert np.array_equal(to_host(dev["prefix_len"]), pl) and np.array_equal(to_host(st.src_slots), src)
    z, tk, _ = oracle.heads(x["hidden"], r["best_node"], wts["w1"], None, wts["w2"], list(ot.s[:ot.K]), 2)
    assert np.abs(to_host(st.head_logits) - z).max() <= 1e-5 * np.abs(z).max()
    assert np.array_equal(to_host(st.topk), tk)
    assert np.array_equal(to_host(st.next_tokens), oracle.build_candidates(r["next_root"], tk, ot))


@pytest.mark.parametrize("heads", ["fused", "split", "joint"])
def test_step_tiny_bf16_full(M, heads):
    _check_bf16_step(M, "tiny_bf16", heads, head_list=(0, 1), n_cols=None)


@pytest.mark.parametrize("heads", ["fused", "split", "joint"])
def test_step_vicuna7b_sampled(M, heads):
    _check_bf16_step(M, "vicuna7b_L1024_tree64", heads, head_list=(0, 17, 31), n_cols=512)


def _check_bf16_step(M, name, heads, head_list, n_cols):
    """A bf16 step in the default launch configuration: attention on `head_list`,
    logits on the path's parent rows in full and on n_cols sampled vocabulary rows
    (None: every row), acceptance, compaction, heads and candidates."""
    w, ot, wts, x, tok, st, dev, node, path, lg_par, parents, gaps = _run(
        M, name, lambda ot: int(np.nonzero(ot.depth == 3)[0][4]), heads=heads)
    assert int(st.err.item()) == 0
    T, V, H, Dh = ot.T, w["V"], w["H"], w["Dh"]
    # --- attention (oracle on single-head slices)
    out = as_double(to_host(st.out))
    for h in head_list:
        sl = lambda a: np.ascontiguousarray(a[..., h:h + 1, :])
        kc, vc = sl(x["k_cache"]), sl(x["v_cache"])
        _, ref = oracle.tree_attn(sl(x["q"]), sl(x["k_new"]), sl(x["v_new"]), kc, vc, x["seq_start"],
                                  x["prefix_len"], ot)
        assert np.abs(out[..., h:h + 1, :] - ref).max() <= 2e-2
    # --- logits: the path's parent rows in full, 512 sampled vocabulary rows for all tree rows
    logits = to_host(st.logits)[0]
    for i, p in enumerate(parents):
        assert np.abs(logits[p] - lg_par[i]).max() <= 2e-2 * np.abs(lg_par[i]).max()
    cols = np.arange(V) if n_cols is None else np.random.default_rng(0).choice(V, n_cols, replace=False)
    ref = oracle.lm_head(x["hidden"][0], np.ascontiguousarray(wts["w_lm"][cols]))
    assert np.abs(logits[:, cols] - ref).max() <= 2e-2 * np.abs(ref).max()
    # --- acceptance: the planted path (decisions there are clear of rounding)
    assert all(gaps[int(ot.parent[c])] > 1e-3 for c in path[1:])
    assert int(st.accept_len.item()) == ot.depth[node] == 3
    an = to_host(st.accepted_nodes)[0]
    assert list(an[:len(path)]) == path and np.all(an[len(path):] == -1)
    assert int(st.best_node.item()) == node
    # the oracle's acceptance on the GPU's own logits, bit for bit (greedy)
    got = {k: to_host(getattr(st, k)) for k in ("accept_len", "accepted_nodes", "next_root", "best_node",
                                                 "best_logp")}
    assert check_accept_on_gpu_logits(ot, logits[None], tok, 0, 1.0, 0.09, 0.3, got) == 1
    # --- compaction: V rows bit-exact, K rows within one bf16 unit (rotation rounding)
    L = int(x["prefix_len"][0])
    vcd = to_host(dev["v_cache"])
    for j, a in enumerate(path):
        assert np.array_equal(vcd[L + j], x["v_new"][0, a])
    assert int(dev["prefix_len"].item()) == L + 4
    # --- heads on the accepted node's hidden state, in full
    s = list(ot.s[:ot.K])
    z, tk, _ = oracle.heads(x["hidden"], np.array([node], np.int32), wts["w1"], None, wts["w2"], s, max(s))
    zg, tg = to_host(st.head_logits), to_host(st.topk)
    assert np.abs(zg - z).max() <= 2e-2 * np.abs(z).max()
    for k in range(ot.K):
        assert gpu_topk_matches_oracle(zg[0, k], tg[0, k], s[k])  # the oracle's top-s of the GPU's logits
        srt = np.sort(z[0, k])[::-1]
        if (srt[:s[k]] - srt[1:s[k] + 1]).min() > 1e-3 * np.abs(z[0, k]).max():
            assert list(tg[0, k, :s[k]]) == list(tk[0, k, :s[k]])
    # --- next candidates from the GPU's own top-s and root
    nt = to_host(st.next_tokens)[0]
    assert nt[0] == int(st.next_root.item())
    for n in range(1, T):
        assert nt[n] == tg[0, ot.depth[n] - 1, ot.rank[n] - 1]
