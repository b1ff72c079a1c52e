"""Whole verify steps at the full sizes of the other workloads, run the way
bench.py runs them (VerifyStep with the attention/compaction side branch):

  vicuna13b_L2048_tree64_typical   d=5120, 40x128 heads, L=2048, typical
  vicuna7b_L4096_tree64            d=4096, 32x128 heads, L=4096, 64-node tree
  vicuna7b_L4096_dense256          same, 256-node dense tree (T=257)
  vicuna33b_bs4_ragged             d=6656, 52x128 heads, 4 sequences with
                                   prefixes in [512, 8192], typical

Checks against the oracle on samples it computes one by one (two attention
heads of every sequence, 256 vocabulary rows of the LM head for every tree
row, the W1 pass in full and 256 vocabulary rows of every head), and
properties that hold at any size: the acceptance equals the oracle's
acceptance run on the GPU's own logits (bit for bit wherever a typical
decision is clear of float32 rounding), the compacted cache holds exactly the
accepted rows, the top-s equal the oracle's top-s of the GPU's own head
logits, and the next candidates are filled from them.
"""
import numpy as np
import pytest
import torch

import oracle
from medusa_tree_speculative_gb300 import synth, workloads
from parity_util import (ancestors, as_double, both_trees, check_accept_on_gpu_logits, gpu_topk_matches_oracle,
                         to_dev, to_host)

pytestmark = pytest.mark.gpu

CONFIGS = ["vicuna13b_L2048_tree64_typical", "vicuna7b_L4096_tree64", "vicuna7b_L4096_dense256",
           "vicuna33b_bs4_ragged"]


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


@pytest.mark.parametrize("name", CONFIGS)
def test_config_step(M, name):
    from medusa_tree_speculative_gb300 import step

    w = workloads.get(name)
    ot, dtree = both_trees(M, _tree_spec(w))
    T, B, H, Dh, d, V = ot.T, w["B"], w["H"], w["Dh"], w["d"], w["V"]
    wts = synth.make_weights(w, 0)
    x = synth.make_step(w, T, 0)
    dev = {k: to_dev(v) for k, v in x.items()}
    wd = {k: (None if v is None else to_dev(v)) for k, v in wts.items()}
    L = x["prefix_len"].astype(np.int64)
    st = step.VerifyStep(w, wd, dtree, max_prefix=int(L.max()))

    # plant one path per sequence with the GPU's own LM-head argmax (setup)
    M.medusa_lm_head_verify(dev["hidden"], st.w_lm, st.logits)
    am = torch.argmax(st.logits, dim=-1).cpu().numpy()
    tok = x["tokens"].copy()
    deep = [n for n in range(T) if ot.depth[n] == min(3, ot.K)]
    for b in range(B):
        path = set(ancestors(ot.parent, deep[(5 * b + 1) % len(deep)]))
        for c in range(1, T):
            if c in path:
                tok[b, c] = am[b, ot.parent[c]]
    dev["tokens"] = to_dev(tok)
    side = torch.cuda.Stream()
    st.run(dev, torch.cuda.current_stream(), side_stream=side)
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0

    # ---- attention: two heads of every sequence against the oracle
    out = as_double(to_host(st.out))
    for h in (0, H - 1):
        sl = lambda a: np.ascontiguousarray(a[..., h:h + 1, :])
        kc, vc = sl(x["k_cache"]), sl(x["v_cache"])
        _, ref = oracle.tree_attn(sl(x["q"]), sl(x["k_new"]), sl(x["v_new"]), kc, vc, x["seq_start"],
                                  x["prefix_len"], ot)
        assert np.abs(out[..., h:h + 1, :] - ref).max() <= 2e-2

    # ---- LM head: 256 sampled vocabulary rows for every tree row
    logits = to_host(st.logits).reshape(B * T, V)
    cols = np.random.default_rng(1).choice(V, 256, replace=False)
    ref = oracle.lm_head(np.ascontiguousarray(x["hidden"].reshape(B * T, d)),
                         np.ascontiguousarray(wts["w_lm"][cols]))
    assert np.abs(logits[:, cols] - ref).max() <= 2e-2 * np.abs(ref).max()
    logits = logits.reshape(B, T, V)

    # ---- acceptance: the oracle's acceptance on the GPU's own logits
    mode = 1 if w["mode"] == "typical" else 0
    tau, eps, delta = w.get("temperature", 1.0), w.get("eps", 0.09), w.get("delta", 0.3)
    got = {k: to_host(getattr(st, k)) for k in ("accept_len", "accepted_nodes", "next_root", "best_node",
                                                 "best_logp")}
    exact = check_accept_on_gpu_logits(ot, logits, tok, mode, tau, eps, delta, got)
    assert exact >= 0.95 * B
    if mode == 0:
        assert np.all(got["accept_len"] >= min(3, ot.K))  # the planted paths are accepted
    acc_len, acc_nodes, best = got["accept_len"], got["accepted_nodes"], got["best_node"]

    # ---- compaction: slot L+j holds tree row a_j (V exact, K rotated)
    vcd, kcd = to_host(dev["v_cache"]), to_host(dev["k_cache"])
    st_b = x["seq_start"]
    for b in range(B):
        for j in range(acc_len[b] + 1):
            a = acc_nodes[b, j]
            assert np.array_equal(vcd[st_b[b] + L[b] + j], x["v_new"][b, a])
            kref = np.stack([oracle.rope(x_h, L[b] + ot.depth[a]) for x_h in as_double(x["k_new"][b, a])])
            kerr = np.abs(as_double(kcd[st_b[b] + L[b] + j]) - kref)
            assert np.all(kerr <= 2.0 ** -7 * np.abs(kref) + 1e-6)
    assert np.array_equal(to_host(dev["prefix_len"]), (L + acc_len + 1).astype(np.int32))

    # ---- heads: W1 in full and 256 vocabulary rows of each head, on the best node
    s_heads = st.s_heads
    used = [k for k in range(w["K"]) if s_heads[k] > 0]
    hl, tk = to_host(st.head_logits), to_host(st.topk)
    one = np.ascontiguousarray(wts["w2"][:, :1])
    _, _, u = oracle.heads(x["hidden"], best.astype(np.int32), wts["w1"], None, one,
                           [1 if k in used else 0 for k in range(w["K"])], 1)
    for b in range(B):
        for k in used:
            ref = oracle.lm_head(np.ascontiguousarray(u[b, k][None]), np.ascontiguousarray(wts["w2"][k][cols]))[0]
            assert np.abs(hl[b, k, cols] - ref).max() <= 2e-2 * np.abs(ref).max()
            # the oracle's top-s on the GPU's own head logits
            assert gpu_topk_matches_oracle(hl[b, k], tk[b, k], s_heads[k])
    # ---- next candidates from the GPU's own top-s and root
    nt = to_host(st.next_tokens)
    for b in range(B):
        assert nt[b, 0] == int(to_host(st.next_root)[b])
        for n in range(1, T):
            assert nt[b, n] == tk[b, ot.depth[n] - 1, ot.rank[n] - 1]


def test_step_repeated_in_a_graph(M):
    """Thirty verify steps at L = 4096 replayed from one CUDA graph, the
    attention on its forked branch beside the LM head (the bench's launch):
    no bounded wait gives up (the device error word stays zero) and every
    step recomputes the same attention output and accepted path.  The
    attention's barriers are timing-sensitive: a hand-off whose phase could be
    overtaken shows up here as MEDUSA_DEVERR_TIMEOUT."""
    from medusa_tree_speculative_gb300 import step

    w = workloads.get("vicuna7b_L4096_tree64")
    ot, dtree = both_trees(M, _tree_spec(w))
    wts = synth.make_weights(w, 0)
    x = synth.make_step(w, ot.T, 0)
    dev = {k: to_dev(v) for k, v in x.items()}
    wd = {k: (None if v is None else to_dev(v)) for k, v in wts.items()}
    st = step.VerifyStep(w, wd, dtree, max_prefix=int(x["prefix_len"].max()))
    prefix0 = dev["prefix_len"].clone()
    s, side = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s):
        st.run(dev, s, side_stream=side)
    torch.cuda.synchronize()
    ref_out, ref_len = st.out.clone(), st.accept_len.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(30):
            dev["prefix_len"].copy_(prefix0)
            st.run(dev, s, side_stream=side)
    with torch.cuda.stream(s):
        dev["prefix_len"].copy_(prefix0)
        g.replay()
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    assert torch.equal(st.out, ref_out) and torch.equal(st.accept_len, ref_len)
