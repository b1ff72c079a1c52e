"""GPU parity: every libmedusa call against the CPU oracle on the same seeded
inputs, through the C ABI.

Bars: integer and index outputs (accepted path, lengths, next root, top-s
indices, candidate tokens, compacted cache rows) bit-exact; floating point
within the stated tolerances: attention max-abs 2e-2 and logits
2e-2 * max|logit| for bf16 (float32: 1e-4 and 1e-5 * max|logit|, from the
float32 accumulation error bound at these sizes).  Where floating point decides
an integer (an argmax or a top-s boundary), decisions are compared where the
oracle's margin exceeds the GPU's rounding error and checked for validity
against the GPU's own logits elsewhere.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from medusa_tree_speculative_gb300 import synth
from parity_util import (ancestors, as_double, both_trees, gpu_topk_matches_oracle, plant_tokens, row_gaps, to_dev,
                         to_host)

pytestmark = pytest.mark.gpu

TOL = {"f32": dict(attn=1e-4, logit=1e-5), "bf16": dict(attn=2e-2, logit=2e-2)}


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from medusa_tree_speculative_gb300 import build

    build.build()
    from medusa_tree_speculative_gb300 import medusa

    return medusa


def err_flag():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ----------------------------------------------------------- tree attention

def _attn_case(M, dt, H, Dh, L, spec, seed):
    ot, dtree = both_trees(M, spec)
    T, B = ot.T, len(L)
    q = synth.normal(seed, "q", (B, T, H, Dh), 1.0, dt)
    kn = synth.normal(seed, "k_new", (B, T, H, Dh), 1.0, dt)
    vn = synth.normal(seed, "v_new", (B, T, H, Dh), 1.0, dt)
    cap = np.array(L, np.int64) + T + 3
    st = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)
    edt = np.uint16 if dt == "bf16" else np.float32
    kc = np.zeros((int(cap.sum()), H, Dh), edt)
    vc = np.zeros_like(kc)
    for b in range(B):
        kc[st[b]:st[b] + L[b]] = synth.normal(seed, f"kp{b}", (L[b], H, Dh), 1.0, dt)
        vc[st[b]:st[b] + L[b]] = synth.normal(seed, f"vp{b}", (L[b], H, Dh), 1.0, dt)
    pl = np.array(L, np.int32)
    return ot, dtree, q, kn, vn, kc, vc, st, pl, cap


ATTN_CASES = [
    # dtype, H, Dh, prefix lengths, tree
    ("f32", 4, 64, [64], ("cartesian", (2, 2, 2), None)),
    ("f32", 2, 128, [33, 0], ("cartesian", (2, 3), None)),
    ("bf16", 4, 64, [64], ("cartesian", (2, 2, 2), None)),
    ("bf16", 4, 64, [100, 37], ("cartesian", (2, 2, 2), None)),
    ("bf16", 2, 128, [1000], ("greedy", 4, 10, 64)),
    ("bf16", 3, 128, [0], ("greedy", 4, 10, 64)),
    ("bf16", 2, 128, [130], ("cartesian", (1,), 0)),              # root only
    ("bf16", 2, 128, [300], ("cartesian", (4, 4, 4, 4), 256)),     # 257 rows
    ("bf16", 1, 64, [70], ("cartesian", (8, 8, 8), 511)),          # 512 rows (maximum)
    ("bf16", 3, 128, [4096, 777, 5], ("greedy", 5, 10, 64)),
]


_ATTN_ORACLE = {}


def _attn_oracle(case, q, kn, vn, kc, vc, st, pl, ot, scale):
    """The oracle's output and cache for one case (computed once per case)."""
    key = repr(case)
    if key not in _ATTN_ORACLE:
        kc_o, vc_o = kc.copy(), vc.copy()
        _, ref = oracle.tree_attn(q, kn, vn, kc_o, vc_o, st, pl, ot, 10000.0, scale)
        _ATTN_ORACLE[key] = (ref, kc_o, vc_o)
    return _ATTN_ORACLE[key]


@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: f"{c[0]}-H{c[1]}-Dh{c[2]}-L{c[3]}-{c[4][0]}")
def test_tree_attn(M, case):
    _check_tree_attn(M, case, None)


# bf16 key splits other than the default 8 (one CTA per unit walks every key;
# 512 tree rows make it cross several 64-node ancestor windows)
SPLIT_CASES = [ATTN_CASES[i] for i in (3, 4, 7, 8, 9)]


@pytest.mark.parametrize("key_splits", [1, 2, 4])
@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: f"{c[0]}-H{c[1]}-Dh{c[2]}-L{c[3]}-{c[4][0]}")
def test_tree_attn_key_splits(M, case, key_splits):
    _check_tree_attn(M, case, key_splits)


# the tensor-core path (bf16, Dh 128): one, several and 512 tree rows, ragged
# prefixes across sequences, an empty prefix; 1 to 8 CTAs per head's keys
# (with 8, some CTAs of a short sequence get no key tile at all)
TC_CASES = [c for c in ATTN_CASES if c[0] == "bf16" and c[2] == 128] + [
    ("bf16", 1, 128, [70], ("cartesian", (8, 8, 8), 511)),
    ("bf16", 2, 128, [127, 128, 129], ("cartesian", (2, 2, 2), None)),
]


@pytest.mark.parametrize("key_splits", [1, 2, 4, 8])
@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: f"{c[0]}-H{c[1]}-Dh{c[2]}-L{c[3]}-{c[4][0]}")
def test_tree_attn_tc(M, case, key_splits):
    _check_tree_attn(M, case, f"tc{key_splits}")


def _check_tree_attn(M, case, key_splits):
    dt, H, Dh, L, spec = case
    ot, dtree, q, kn, vn, kc, vc, st, pl, cap = _attn_case(M, dt, H, Dh, L, spec, seed=3)
    B, T = len(L), ot.T
    scale = 1.0 / math.sqrt(Dh)
    # GPU
    kc_d, vc_d = to_dev(kc), to_dev(vc)
    out_d = to_dev(np.zeros_like(q))
    ws = torch.empty(M.medusa_tree_attn_workspace_size(B, H, Dh, T, max(L)), dtype=torch.uint8, device="cuda")
    e = err_flag()
    if isinstance(key_splits, str):  # "tcN": the tensor-core path with N CTAs per head's keys
        ns = int(key_splits[2:])
        for _ in range(2):  # repeated calls append the same tree rows and give the same output
            M.medusa_tree_attn_tc(to_dev(q), to_dev(kn), to_dev(vn), kc_d, vc_d, to_dev(st), to_dev(pl),
                                  to_dev(cap), dtree, max(L), 10000.0, scale, out_d, e, key_splits=ns)
    else:
        M.medusa_tree_attn(to_dev(q), to_dev(kn), to_dev(vn), kc_d, vc_d, to_dev(st), to_dev(pl), to_dev(cap),
                           dtree, max(L), 10000.0, scale, out_d, ws, e, key_splits=key_splits)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    # oracle
    ref, kc_o, vc_o = _attn_oracle(case, q, kn, vn, kc, vc, st, pl, ot, scale)
    got = as_double(to_host(out_d))
    err = np.abs(got - ref).max()
    assert err <= TOL[dt]["attn"], f"attention max-abs error {err}"
    # cache: prefix untouched, V rows copied exactly, K rows rotated
    kg, vg = to_host(kc_d), to_host(vc_d)
    for b in range(B):
        assert np.array_equal(kg[st[b]:st[b] + L[b]], kc[st[b]:st[b] + L[b]])
        tail = slice(st[b] + L[b], st[b] + L[b] + T)
        assert np.array_equal(vg[tail], vc_o[tail])
        # rotation in float32 (GPU) vs double (oracle), then rounding to the
        # cache type: at most one unit in the last place apart
        kref = as_double(kc_o[tail])
        kerr = np.abs(as_double(kg[tail]) - kref)
        bound = (2.0 ** -7 if dt == "bf16" else 2.0 ** -21) * np.abs(kref) + 1e-6
        assert np.all(kerr <= bound)
        # slots past the tree rows stay zero
        assert not np.any(vg[st[b] + L[b] + T:st[b] + cap[b]].astype(np.float64))


def test_tree_attn_capacity_flag(M):
    ot, dtree, q, kn, vn, kc, vc, st, pl, cap = _attn_case(M, "bf16", 2, 64, [40, 20], ("cartesian", (2, 2), None), 5)
    cap = cap.copy()
    cap[1] = pl[1] + ot.T - 1  # one slot short
    B, T = 2, ot.T
    ws = torch.empty(M.medusa_tree_attn_workspace_size(B, 2, 64, T, 40), dtype=torch.uint8, device="cuda")
    out = torch.full((B, T, 2, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    e = err_flag()
    kc_d = to_dev(kc)
    M.medusa_tree_attn(to_dev(q), to_dev(kn), to_dev(vn), kc_d, to_dev(vc), to_dev(st), to_dev(pl), to_dev(cap),
                       dtree, 40, 10000.0, 0.125, out, ws, e)
    torch.cuda.synchronize()
    assert int(e.item()) & 4
    o = out.float().cpu().numpy()
    assert np.all(o[1] == 7.0)          # skipped sequence untouched
    assert not np.all(o[0] == 7.0)      # the other one computed
    assert np.array_equal(to_host(kc_d)[st[1]:st[1] + 40], kc[st[1]:st[1] + 40])


# ----------------------------------------------------------------- LM head

LM_CASES = [("f32", 15, 256, 1024), ("bf16", 15, 256, 1024), ("bf16", 65, 256, 1000),
            ("bf16", 130, 512, 3000), ("bf16", 1, 64, 17), ("bf16", 260, 128, 333),
            ("bf16", 65, 4096, 2048), ("bf16", 65, 256, 20000), ("bf16", 17, 128, 40000),
            # two tiles per item with one accumulator (129..256 rows, more tiles than SMs);
            # two row chunks sharing each weight block (257..512 rows); two such items
            ("bf16", 200, 256, 40000), ("bf16", 300, 256, 40000), ("bf16", 512, 128, 5000),
            ("bf16", 1000, 128, 700),
            # 257..264 rows: one 256-row chunk on tcgen05, the rest beside it by mma.sync
            # (one tile per item; two tiles per item with eight extra rows); 265: two chunks again
            ("bf16", 257, 4096, 2048), ("bf16", 264, 192, 40000), ("bf16", 260, 6656, 1000),
            ("bf16", 265, 128, 3000)]


@pytest.mark.parametrize("case", LM_CASES, ids=lambda c: "-".join(map(str, c)))
def test_lm_head(M, case):
    dt, rows, d, V = case
    h = synth.normal(11, "h", (rows, d), 1.0, dt)
    w = synth.normal(11, "w", (V, d), 1.0 / math.sqrt(d), dt)
    logits = torch.empty((rows, V), dtype=torch.float32, device="cuda")
    M.medusa_lm_head_verify(to_dev(h), to_dev(w), logits)
    torch.cuda.synchronize()
    ref = oracle.lm_head(h, w)
    err = np.abs(to_host(logits) - ref).max()
    scale = np.abs(ref).max()
    assert err <= TOL[dt]["logit"] * scale, f"logit error {err} vs max|logit| {scale}"


TILE_CASES = [(256, 1000), (64, 17), (4096, 2048), (128, 40000), (4096, 32000)]


@pytest.mark.parametrize("case", TILE_CASES, ids=lambda c: "-".join(map(str, c)))
def test_lm_head_tiled_layout(M, case):
    """The tile rewrite is an exact permutation (zero rows past V), and the LM
    head reading it gives the same logits bit for bit as from row-major W."""
    d, V = case
    w = synth.normal(12, "w", (V, d), 1.0 / math.sqrt(d), "bf16")
    wd = to_dev(w)
    tiled = M.medusa_lm_head_tile(wd)
    nt = (V + 127) // 128
    pad = np.zeros((nt * 128, d), np.uint16)
    pad[:V] = w
    want = pad.reshape(nt, 128, d // 64, 64).transpose(0, 2, 1, 3).ravel()
    got = to_host(tiled)
    assert got.shape == want.shape and np.array_equal(got, want)
    # element (v, j) at the documented offset, spot-checked
    rng = np.random.default_rng(0)
    for v, j in zip(rng.integers(0, V, 64), rng.integers(0, d, 64)):
        off = ((v // 128) * (d // 64) + j // 64) * 8192 + (v % 128) * 64 + j % 64
        assert got[off] == w[v, j]
    rows = 65 if V <= 32000 else 17
    h = to_dev(synth.normal(12, "h", (rows, d), 1.0, "bf16"))
    a_rows = torch.empty((rows, V), dtype=torch.float32, device="cuda")
    a_tiles = torch.full((rows, V), float("nan"), dtype=torch.float32, device="cuda")
    M.medusa_lm_head_verify(h, wd, a_rows)
    M.medusa_lm_head_verify(h, tiled, a_tiles, layout=M.W_TILES)
    torch.cuda.synchronize()
    assert torch.equal(a_rows, a_tiles)
    if d * V <= 4096 * 2048:
        ref = oracle.lm_head(to_host(h), w)
        assert np.abs(to_host(a_tiles) - ref).max() <= TOL["bf16"]["logit"] * np.abs(ref).max()


PAIR_CASES = [(129, 128, 777), (256, 192, 3000), (200, 4096, 2048), (256, 4096, 32000),
              (257, 4096, 32000), (260, 6656, 32000), (264, 128, 777)]


@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: "-".join(map(str, c)))
def test_lm_head_cta_pairs(M, case):
    """129..256 rows run on CTA pairs (one MMA of M = 256 over a vocabulary
    tile of each CTA, each CTA holding half of the hidden rows): an odd tile
    count leaves the last pair's second CTA a tile past V; 257 to 264 rows
    run as one 256-row chunk plus the extra rows by mma.sync beside it.  Both weight
    layouts give the same logits bit for bit, within tolerance of the oracle."""
    rows, d, V = case
    h = synth.normal(13, "h", (rows, d), 1.0, "bf16")
    w = synth.normal(13, "w", (V, d), 1.0 / math.sqrt(d), "bf16")
    hd, wd = to_dev(h), to_dev(w)
    if rows <= 256:
        assert M.medusa_lm_head_ctas(rows, V) % 2 == 0
    a_rows = torch.full((rows, V), float("nan"), dtype=torch.float32, device="cuda")
    a_tiles = torch.full((rows, V), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.medusa_lm_head_verify(hd, wd, a_rows, err=err)
    M.medusa_lm_head_verify(hd, M.medusa_lm_head_tile(wd), a_tiles, err=err, layout=M.W_TILES)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(a_rows, a_tiles)
    if d * V <= 4096 * 2048:
        ref = oracle.lm_head(h, w)
        assert np.abs(to_host(a_rows) - ref).max() <= TOL["bf16"]["logit"] * np.abs(ref).max()
    else:  # sampled logits against the oracle's dot products
        rng = np.random.default_rng(1)
        got = to_host(a_rows)
        scale = np.abs(got).max()
        for r, v in zip(rng.integers(0, rows, 64), rng.integers(0, V, 64)):
            want = oracle.lm_head(h[r:r + 1], w[v:v + 1])[0, 0]
            assert abs(got[r, v] - want) <= TOL["bf16"]["logit"] * scale


JOINT_CASES = [
    # rows, d, V, s, bias: plans of 2, 3 and 4 tiles per CTA (the last two at
    # 7B and 13B sizes, checked on sampled rows)
    (15, 256, 1000, (2, 2, 2), True),
    (1, 128, 17, (1,), False),
    (65, 512, 5000, (8, 6, 5, 2), False),
    (65, 1024, 32000, (8, 0, 5, 2), True),
    (65, 4096, 32000, (8, 6, 5, 2), False),
    (65, 5120, 32000, (8, 6, 5, 2, 0), False),
]


@pytest.mark.parametrize("case", JOINT_CASES, ids=lambda c: f"r{c[0]}-d{c[1]}-V{c[2]}-s{len(c[3])}")
def test_lm_head_heads_hidden_joint(M, case):
    """medusa_lm_head_verify_heads_hidden: logits and u against the oracle
    (every row for small shapes, sampled rows otherwise), and bit for bit the
    same as the two separate calls, for row-major and tiled weights."""
    rows, d, V, s, bias = case
    K = len(s)
    used = [k for k in range(K) if s[k] > 0]
    h = synth.normal(15, "h", (rows, d), 1.0, "bf16")
    w = synth.normal(15, "w", (V, d), 1.0 / math.sqrt(d), "bf16")
    w1 = synth.normal(15, "w1", (K, d, d), 1.0 / math.sqrt(d), "bf16")
    b1 = synth.normal(15, "b1", (K, d), 0.5, "bf16") if bias else None
    hd, wd, w1d = to_dev(h), to_dev(w), to_dev(w1)
    b1d = None if b1 is None else to_dev(b1)
    chk = list(range(rows)) if rows * d * (V + K * d) <= 2**28 else sorted({0, 1, rows // 2, rows - 1})
    ref = oracle.lm_head(np.ascontiguousarray(h[chk]), w)
    one = np.ascontiguousarray(w1[:, :1])  # the W2 the oracle's head call needs (unused here)
    _, _, u_ref = oracle.heads(np.ascontiguousarray(h[chk].reshape(len(chk), 1, d)), np.zeros(len(chk), np.int32),
                               w1, b1, one, [1 if k in used else 0 for k in range(K)], 1)
    # the separate calls, row-major weights
    lg_sep = torch.empty((rows, V), dtype=torch.float32, device="cuda")
    u_sep = torch.zeros((rows, K, d), dtype=torch.bfloat16, device="cuda")
    M.medusa_lm_head_verify(hd, wd, lg_sep)
    M.medusa_heads_hidden(hd, w1d, b1d, list(s), u_sep)
    wt, w1t = M.medusa_lm_head_tile(wd), M.medusa_lm_head_tile(w1d.reshape(K * d, d))
    for lay, lay1 in ((M.W_ROWS, M.W_ROWS), (M.W_TILES, M.W_TILES), (M.W_TILES, M.W_ROWS)):
        lg = torch.full((rows, V), float("nan"), dtype=torch.float32, device="cuda")
        u = torch.zeros((rows, K, d), dtype=torch.bfloat16, device="cuda")
        e = err_flag()
        M.medusa_lm_head_verify_heads_hidden(hd, wt if lay == M.W_TILES else wd, V, lg,
                                             w1t if lay1 == M.W_TILES else w1d, b1d, list(s), u, e,
                                             layout=lay, w1_layout=lay1)
        torch.cuda.synchronize()
        assert int(e.item()) == 0
        assert torch.equal(lg, lg_sep), "logits differ from medusa_lm_head_verify"
        assert torch.equal(u, u_sep), "u differs from medusa_heads_hidden"
        lgh = to_host(lg)[chk]
        assert np.abs(lgh - ref).max() <= TOL["bf16"]["logit"] * np.abs(ref).max()
        ug = as_double(to_host(u))
        for i, r in enumerate(chk):
            for k in range(K):
                if k not in used:
                    assert not np.any(ug[r, k])  # skipped head: not written
                    continue
                rk = as_double(u_ref[i, k])
                assert np.all(np.abs(ug[r, k] - rk) <= 2.0 ** -7 * np.abs(rk) + 1e-3), f"u row {r} head {k}"


# -------------------------------------------------------------- acceptance

def _accept_inputs(ot, B, V, mode, seed, plant_nodes):
    """Synthetic float32 logits; tokens planted so that the node passes."""
    rng = np.random.default_rng(seed)
    T = ot.T
    logits = (rng.standard_normal((B, T, V)) * 2.0).astype(np.float32)
    tokens = np.zeros((B, T), np.int32)
    for b in range(B):
        node = plant_nodes[b]
        path = set(ancestors(ot.parent, node))
        for c in range(1, T):
            p = ot.parent[c]
            if c in path:
                if mode == 0:
                    tokens[b, c] = int(np.argmax(logits[b, p]))
                else:
                    t = int(rng.integers(0, V))
                    logits[b, p, t] = logits[b, p].max() + 1.0  # a confident token passes
                    tokens[b, c] = t
            else:
                t = int(rng.integers(0, V))
                if mode == 0 and t == int(np.argmax(logits[b, p])):
                    t = (t + 1) % V  # off the planted path nothing passes
                tokens[b, c] = t
    return logits, tokens


def _gpu_accept(M, dtree, logits, tokens, mode, temp=0.7, eps=0.09, delta=0.3):
    B, T, V = logits.shape
    K = dtree.K
    out = dict(accept_len=torch.zeros(B, dtype=torch.int32, device="cuda"),
               accepted_nodes=torch.zeros((B, K + 1), dtype=torch.int32, device="cuda"),
               next_root=torch.zeros(B, dtype=torch.int32, device="cuda"),
               best_node=torch.zeros(B, dtype=torch.int32, device="cuda"),
               best_logp=torch.zeros(B, dtype=torch.float32, device="cuda"))
    ws = torch.zeros(M.medusa_accept_workspace_size(B, T), dtype=torch.uint8, device="cuda")
    e = err_flag()
    args = (to_dev(logits), to_dev(tokens), dtree, mode, temp, eps, delta)
    M.medusa_accept(*args, out["accept_len"], out["accepted_nodes"], out["next_root"], out["best_node"],
                    out["best_logp"], ws, e)
    # a second call on the same workspace (its counters must be zero again) gives the same results
    again = {k: torch.full_like(v, -5) for k, v in out.items()}
    M.medusa_accept(*args, again["accept_len"], again["accepted_nodes"], again["next_root"], again["best_node"],
                    again["best_logp"], ws, e)
    torch.cuda.synchronize()
    for k in out:
        assert torch.equal(out[k], again[k]), k
    return {k: to_host(v) for k, v in out.items()}, int(e.item())


ACCEPT_CASES = [
    (("cartesian", (3, 2, 2), None), 50, 0),
    (("cartesian", (3, 2, 2), None), 50, 1),
    (("greedy", 4, 10, 64), 32000, 0),
    (("greedy", 4, 10, 64), 32000, 1),
    (("cartesian", (4, 4, 4, 4), 256), 1000, 0),
    (("cartesian", (8, 8, 8), 511), 100, 1),
    (("cartesian", (1,), 0), 100, 0),
]


@pytest.mark.parametrize("case", ACCEPT_CASES, ids=lambda c: f"{c[0][0]}{c[0][1]}-V{c[1]}-mode{c[2]}")
def test_accept(M, case):
    spec, V, mode = case
    ot, dtree = both_trees(M, spec)
    T = ot.T
    rng = np.random.default_rng(7)
    # every node once as the planted endpoint, three sequences per call
    nodes = list(range(T)) if T <= 70 else list(rng.integers(0, T, 12))
    for i in range(0, len(nodes), 3):
        plant = [int(n) for n in nodes[i:i + 3]]
        B = len(plant)
        for attempt in range(20):
            logits, tokens = _accept_inputs(ot, B, V, mode, seed=100 + i + 1000 * attempt, plant_nodes=plant)
            r = oracle.accept(logits, tokens, ot, mode, temperature=0.7, eps=0.09, delta=0.3)
            # a typical decision closer to its threshold than float32 rounding
            # of p-hat could go either way; draw another input instead
            if mode == 0 or T == 1 or np.abs(r["node_margin"][:, 1:]).min() > 1e-6:
                break
        else:
            raise AssertionError("no unambiguous typical input found")
        g, e = _gpu_accept(M, dtree, logits, tokens, mode)
        assert e == 0
        for key in ("accept_len", "accepted_nodes", "next_root", "best_node"):
            assert np.array_equal(g[key], r[key]), (key, g[key], r[key])
        if mode == 0:
            for b, n in enumerate(plant):
                assert g["accept_len"][b] == ot.depth[n]
        else:
            assert np.allclose(g["best_logp"], r["best_logp"], rtol=1e-4, atol=1e-4)


def test_accept_typical_tie_break_and_low_temperature(M):
    ot, dtree = both_trees(M, ("cartesian", (2,), None))
    V = 4
    logits = np.log(np.array([[[0.1, 0.5, 0.4, 1e-9]] * 3], np.float64)).astype(np.float32)
    tokens = np.array([[0, 2, 1]], np.int32)
    g, _ = _gpu_accept(M, dtree, logits, tokens, 1, temp=1.0)
    assert g["best_node"][0] == 2 and g["accept_len"][0] == 1
    # temperature -> 0: typical reduces to greedy
    ot2, dt2 = both_trees(M, ("cartesian", (3, 2, 2), None))
    for node in range(0, ot2.T, 4):
        lg, tk = _accept_inputs(ot2, 1, 64, 0, seed=500 + node, plant_nodes=[node])
        gg, _ = _gpu_accept(M, dt2, lg, tk, 0)
        gt, _ = _gpu_accept(M, dt2, lg, tk, 1, temp=1e-3)
        for key in ("accept_len", "accepted_nodes", "next_root", "best_node"):
            assert np.array_equal(gg[key], gt[key])


def test_accept_bad_token_flag(M):
    ot, dtree = both_trees(M, ("cartesian", (2, 2), None))
    logits = np.zeros((1, ot.T, 10), np.float32)
    tokens = np.array([[0, 3, 99, 1, 1, 1, 1]], np.int32)
    g, e = _gpu_accept(M, dtree, logits, tokens, 1, temp=1.0)
    assert e & 1
    assert g["accept_len"][0] >= 0


def test_check_errors_reads_and_clears(M):
    """medusa_check_errors: the word raised by a bad token reaches pinned host
    memory and device memory in stream order; with clear the word is zero
    again for the next step."""
    ot, dtree = both_trees(M, ("cartesian", (2, 2), None))
    logits = torch.zeros((1, ot.T, 10), dtype=torch.float32, device="cuda")
    tokens = to_dev(np.array([[0, 3, 99, 1, 1, 1, 1]], np.int32))
    i32 = dict(dtype=torch.int32, device="cuda")
    outs = [torch.zeros(1, **i32), torch.zeros((1, ot.K + 1), **i32), torch.zeros(1, **i32), torch.zeros(1, **i32),
            torch.zeros(1, dtype=torch.float32, device="cuda")]
    ws = torch.zeros(M.medusa_accept_workspace_size(1, ot.T), dtype=torch.uint8, device="cuda")
    e = err_flag()
    host = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    dev_out = torch.full((1,), -1, **i32)
    s = torch.cuda.current_stream()
    M.medusa_accept(logits, tokens, dtree, 1, 1.0, 0.09, 0.3, *outs, ws, e)
    M.medusa_check_errors(e, dev_out, clear=False, stream=s)
    M.medusa_check_errors(e, host, clear=True, stream=s)
    torch.cuda.synchronize()
    assert int(host[0]) == 1 and int(dev_out.item()) == 1  # MEDUSA_DEVERR_TOKEN
    assert int(e.item()) == 0
    with pytest.raises(M.MedusaError, match="INVALID"):
        M.medusa_check_errors(e, torch.zeros(1, dtype=torch.int32))  # pageable host memory


# ------------------------------------------------------------ KV compaction

@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_kv_compact(M, dt):
    ot, dtree = both_trees(M, ("greedy", 4, 10, 64))
    H, Dh, K = 4, 64, ot.K
    L = [50, 9, 300]
    B, T = 3, ot.T
    cap = np.array(L, np.int64) + T
    st = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)
    kc = synth.normal(9, "kc", (int(cap.sum()), H, Dh), 1.0, dt)
    vc = synth.normal(9, "vc", (int(cap.sum()), H, Dh), 1.0, dt)
    rng = np.random.default_rng(9)
    nodes = [int(rng.integers(0, T)) for _ in range(B)]
    nodes[0] = max(range(T), key=lambda n: ot.depth[n])  # a deepest node
    acc_nodes = np.full((B, K + 1), -1, np.int32)
    acc_len = np.zeros(B, np.int32)
    for b, n in enumerate(nodes):
        path = ancestors(ot.parent, n)
        acc_nodes[b, :len(path)] = path
        acc_len[b] = len(path) - 1
    pl = np.array(L, np.int32)
    kd, vd, pld = to_dev(kc), to_dev(vc), to_dev(pl)
    src = torch.zeros((B, K + 1), dtype=torch.int32, device="cuda")
    e = err_flag()
    M.medusa_kv_compact(kd, vd, to_dev(st), pld, to_dev(acc_nodes), to_dev(acc_len), K, T, src, e)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    ko, vo, plo = kc.copy(), vc.copy(), pl.copy()
    so = oracle.kv_compact(ko, vo, st, plo, acc_nodes, acc_len, K)
    assert np.array_equal(to_host(kd), ko) and np.array_equal(to_host(vd), vo)
    assert np.array_equal(to_host(pld), plo) and np.array_equal(to_host(src), so)


def test_kv_compact_in_place_hazard(M):
    # accepted nodes (0, 2, 3): row 1 reads slot L+2, which row 2 overwrites
    H, Dh = 2, 64
    kc = np.arange(20 * H * Dh, dtype=np.float32).reshape(20, H, Dh)
    vc = -kc
    st, pl = np.array([0], np.int64), np.array([5], np.int32)
    an, al = np.array([[0, 2, 3, -1]], np.int32), np.array([2], np.int32)
    kd, vd, pld = to_dev(kc), to_dev(vc), to_dev(pl)
    M.medusa_kv_compact(kd, vd, to_dev(st), pld, to_dev(an), to_dev(al), 3, 7)
    ko, vo = kc.copy(), vc.copy()
    oracle.kv_compact(ko, vo, st, pl.copy(), an, al, 3)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(kd), ko) and np.array_equal(to_host(vd), vo)
    assert to_host(pld)[0] == 8


def test_kv_compact_node_outside_tree(M):
    """An accepted node at or past the tree's T rows (here 400 with a 7-row
    tree) raises MEDUSA_DEVERR_NODE and leaves that sequence untouched; a
    valid sequence in the same call is still compacted."""
    H, Dh = 2, 64
    kc = np.arange(40 * H * Dh, dtype=np.float32).reshape(40, H, Dh)
    vc = -kc
    st, pl = np.array([0, 20], np.int64), np.array([5, 5], np.int32)
    an = np.array([[0, 2, 400, -1], [0, 2, 5, -1]], np.int32)
    al = np.array([2, 2], np.int32)
    kd, vd, pld = to_dev(kc), to_dev(vc), to_dev(pl)
    e = err_flag()
    M.medusa_kv_compact(kd, vd, to_dev(st), pld, to_dev(an), to_dev(al), 3, 7, None, e)
    torch.cuda.synchronize()
    assert int(e.item()) & 2  # MEDUSA_DEVERR_NODE
    ko, vo = kc.copy(), vc.copy()
    oracle.kv_compact(ko[20:], vo[20:], st[1:] - 20, pl[1:].copy(), an[1:], al[1:], 3)
    assert np.array_equal(to_host(kd), ko) and np.array_equal(to_host(vd), vo)
    assert list(to_host(pld)) == [5, 8]


# ------------------------------------------------------------------- heads

HEAD_CASES = [
    # dtype, B, T, d, V, s per head, bias, W2 = LM head + noise
    ("f32", 1, 15, 256, 1024, (2, 2, 2), False, True),
    ("bf16", 1, 65, 256, 1000, (8, 6, 5, 2), False, False),
    ("bf16", 3, 65, 512, 3000, (8, 6, 5, 2, 0), True, False),
    ("bf16", 4, 9, 640, 5000, (16, 1), False, False),
    ("bf16", 1, 65, 4096, 32000, (8, 6, 5, 2), False, False),
    # more than four sequences: the 16-sequence kernels, a warp merging two sequences' lists
    ("bf16", 9, 9, 256, 2000, (16, 4), False, False),
    ("f32", 6, 15, 256, 1024, (3, 2), True, True),
    # bf16 with several sequences runs on the tensor cores: sixteen sequences
    # (both halves of the MMA's M), a vocabulary that is not a multiple of the
    # eight-row unit, and the 33B shape's hidden size with two sequences
    ("bf16", 16, 5, 256, 2003, (3, 2), True, False),
    ("bf16", 2, 65, 6656, 1001, (8, 6, 5, 2), False, False),
    # 325 tree rows: W1 over every row in two row chunks per weight block
    ("bf16", 5, 65, 256, 1000, (4, 3, 2), True, False),
]
# The fused call only (medusa_heads_hidden takes bf16 d in multiples of 128):
# d not a multiple of 32, the CUDA-core kernels for several sequences; d a
# multiple of 32 but not of 128 (twelve sequences: both halves of M)
FUSED_ONLY_CASES = [("bf16", 3, 9, 144, 700, (2, 2), False, False),
                    ("bf16", 4, 9, 288, 1500, (4, 2), True, False),
                    ("bf16", 12, 9, 416, 777, (3, 3, 1), False, False)]


@pytest.mark.parametrize("case", HEAD_CASES + FUSED_ONLY_CASES,
                         ids=lambda c: f"{c[0]}-B{c[1]}-d{c[3]}-V{c[4]}-s{len(c[5])}")
def test_heads_topk(M, case):
    dt, B, T, d, V, s, bias, lm_noise = case
    K = len(s)
    s_max = max(s)
    hidden = synth.normal(13, "hidden", (B, T, d), 1.0, dt)
    w1 = synth.normal(13, "w1", (K, d, d), 0.02 if lm_noise else 1 / math.sqrt(d), dt)
    if lm_noise:
        lm = synth.normal(13, "lm", (V, d), 1 / math.sqrt(d), "f32")
        w2 = np.stack([lm + synth.normal(13, f"n{k}", (V, d), 0.01, "f32") for k in range(K)])
        w2 = w2 if dt == "f32" else synth.f32_to_bf16_bits(w2)
    else:
        w2 = synth.normal(13, "w2", (K, V, d), 1 / math.sqrt(d), dt)
    b1 = synth.normal(13, "b1", (K, d), 0.5, dt) if bias else None
    last = np.array([(3 * b + 1) % T for b in range(B)], np.int32)
    hl = torch.zeros((B, K, V), dtype=torch.float32, device="cuda")
    tk = torch.zeros((B, K, s_max), dtype=torch.int32, device="cuda")
    ws = torch.zeros(M.medusa_heads_topk_workspace_size(B, K, d, V, s_max), dtype=torch.uint8, device="cuda")
    e = err_flag()
    args = (to_dev(hidden), to_dev(last), to_dev(w1), None if b1 is None else to_dev(b1), to_dev(w2), list(s))
    M.medusa_heads_topk(*args, hl, tk, ws, e)
    # a second call on the same workspace (its row counters must be ready again) gives the same bits
    hl2, tk2 = torch.full_like(hl, float("nan")), torch.full_like(tk, -7)
    M.medusa_heads_topk(*args, hl2, tk2, ws, e)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    for k in range(K):
        if s[k] > 0:
            assert torch.equal(hl[:, k], hl2[:, k])
    assert torch.equal(tk, torch.where(tk2 == -7, torch.zeros_like(tk2), tk2))
    z_ref, tk_ref, _ = oracle.heads(hidden, last, w1, b1, w2, list(s), s_max)
    zg, tg = to_host(hl), to_host(tk)
    for b in range(B):
        for k in range(K):
            if s[k] == 0:
                assert np.all(tg[b, k] == 0)  # skipped head: untouched
                continue
            scale = np.abs(z_ref[b, k]).max()
            err = np.abs(zg[b, k] - z_ref[b, k]).max()
            assert err <= TOL[dt]["logit"] * scale, f"head logit error {err} (max {scale})"
            # the oracle's top-s of the GPU's own logits equals the GPU's top-s
            assert gpu_topk_matches_oracle(zg[b, k], tg[b, k], s[k])
            assert np.all(tg[b, k, s[k]:] == -1)
            # parity with the oracle where the ranking is decided by more than
            # the GPU's rounding error
            srt = np.sort(z_ref[b, k])[::-1]
            gaps = srt[:s[k]] - srt[1:s[k] + 1]
            if gaps.min() > 1e-3 * scale:
                assert list(tg[b, k, :s[k]]) == list(tk_ref[b, k, :s[k]])


@pytest.mark.parametrize("case", HEAD_CASES, ids=lambda c: f"{c[0]}-B{c[1]}-d{c[3]}-V{c[4]}-s{len(c[5])}")
def test_heads_split(M, case):
    """medusa_heads_hidden (W1 over every tree row, both weight layouts) and
    medusa_heads_logits_topk on one row per sequence: u against the oracle
    row by row, head logits and top-s as in the fused call; the W2 call runs
    twice on one zeroed workspace (its counters must come back to zero)."""
    dt, B, T, d, V, s, bias, lm_noise = case
    K = len(s)
    s_max = max(s)
    hidden = synth.normal(14, "hidden", (B, T, d), 1.0, dt)
    w1 = synth.normal(14, "w1", (K, d, d), 1 / math.sqrt(d), dt)
    w2 = synth.normal(14, "w2", (K, V, d), 1 / math.sqrt(d), dt)
    b1 = synth.normal(14, "b1", (K, d), 0.5, dt) if bias else None
    node = np.array([(5 * b + 2) % T for b in range(B)], np.int32)
    used = [k for k in range(K) if s[k] > 0]
    hd, w1d = to_dev(hidden), to_dev(w1)
    b1d = None if b1 is None else to_dev(b1)
    layouts = [M.W_ROWS] + ([M.W_TILES] if dt == "bf16" else [])
    # rows checked against the oracle (all of them for small shapes)
    rows = list(range(B * T)) if d * d * K * B * T <= 2**28 else [0, 1, T - 1, B * T - 1]
    one = np.ascontiguousarray(w2[:, :1])
    flat = hidden.reshape(B * T, 1, d)
    _, _, u_ref = oracle.heads(np.ascontiguousarray(flat[rows]), np.zeros(len(rows), np.int32), w1, b1, one,
                               [1 if k in used else 0 for k in range(K)], 1)
    for lay in layouts:
        wsrc = M.medusa_lm_head_tile(w1d.reshape(K * d, d)) if lay == M.W_TILES else w1d
        u = torch.full((B * T, K, d), float("nan"), dtype=hd.dtype, device="cuda")
        e = err_flag()
        M.medusa_heads_hidden(hd, wsrc, b1d, list(s), u, e, layout=lay)
        torch.cuda.synchronize()
        assert int(e.item()) == 0
        ug = as_double(to_host(u))
        for i, r in enumerate(rows):
            for k in used:
                ref = as_double(u_ref[i, k])
                tol = (2.0 ** -7 * np.abs(ref) + 1e-3) if dt == "bf16" else (1e-4 * np.abs(ref) + 1e-4)
                assert np.all(np.abs(ug[r, k] - ref) <= tol), f"u row {r} head {k}"
    # W2 + top-s on the accepted rows, twice on one zeroed workspace
    hl = torch.zeros((B, K, V), dtype=torch.float32, device="cuda")
    tk = torch.zeros((B, K, s_max), dtype=torch.int32, device="cuda")
    ws = torch.zeros(M.medusa_heads_logits_topk_workspace_size(B, K, V, s_max), dtype=torch.uint8, device="cuda")
    e = err_flag()
    for rep in range(2):
        M.medusa_heads_logits_topk(u, T, to_dev(node), to_dev(w2), list(s), hl, tk, ws, e)
        torch.cuda.synchronize()
        assert int(e.item()) == 0
        zg, tg = to_host(hl), to_host(tk)
        if rep == 0:
            first = (zg.copy(), tg.copy())
        else:
            assert np.array_equal(first[0], zg) and np.array_equal(first[1], tg)
    z_ref, tk_ref, _ = oracle.heads(hidden, node, w1, b1, w2, list(s), s_max)
    for b in range(B):
        for k in range(K):
            if s[k] == 0:
                assert np.all(tg[b, k] == 0)
                continue
            scale = np.abs(z_ref[b, k]).max()
            err = np.abs(zg[b, k] - z_ref[b, k]).max()
            assert err <= TOL[dt]["logit"] * scale, f"head logit error {err} (max {scale})"
            assert gpu_topk_matches_oracle(zg[b, k], tg[b, k], s[k])
            assert np.all(tg[b, k, s[k]:] == -1)


def test_heads_init_reproduce_lm_head(M):
    """W1 = 0, W2 = the LM head: every head's top-1 is the LM head's argmax."""
    d, V, K, T = 256, 1000, 3, 7
    hidden = synth.normal(17, "h", (1, T, d), 1.0, "bf16")
    wlm = synth.normal(17, "w", (V, d), 1 / math.sqrt(d), "bf16")
    w1 = np.zeros((K, d, d), np.uint16)
    w2 = np.ascontiguousarray(np.broadcast_to(wlm, (K, V, d)))
    last = np.array([4], np.int32)
    hl = torch.zeros((1, K, V), dtype=torch.float32, device="cuda")
    tk = torch.zeros((1, K, 2), dtype=torch.int32, device="cuda")
    ws = torch.zeros(M.medusa_heads_topk_workspace_size(1, K, d, V, 2), dtype=torch.uint8, device="cuda")
    M.medusa_heads_topk(to_dev(hidden), to_dev(last), to_dev(w1), None, to_dev(w2), [2, 2, 2], hl, tk, ws)
    logits = torch.empty((T, V), dtype=torch.float32, device="cuda")
    M.medusa_lm_head_verify(to_dev(hidden), to_dev(wlm), logits)
    torch.cuda.synchronize()
    am = int(torch.argmax(logits[4]).item())
    assert all(int(tk[0, k, 0].item()) == am for k in range(K))
    lm = oracle.lm_head(hidden, wlm)
    assert int(np.argmax(lm[4])) == am


# -------------------------------------------------------------- candidates

def test_build_candidates(M):
    for spec in [("cartesian", (2, 2, 2), None), ("greedy", 4, 10, 64), ("cartesian", (8, 8, 8), 511)]:
        ot, dtree = both_trees(M, spec)
        B, K = 3, ot.K + 1
        s_max = int(max(ot.s[:ot.K]))
        rng = np.random.default_rng(19)
        topk = rng.integers(0, 32000, (B, K, s_max)).astype(np.int32)
        root = rng.integers(0, 32000, B).astype(np.int32)
        out = torch.zeros((B, ot.T), dtype=torch.int32, device="cuda")
        M.medusa_build_candidates(to_dev(root), to_dev(topk), dtree, out)
        torch.cuda.synchronize()
        ref = oracle.build_candidates(root, topk, ot)
        assert np.array_equal(to_host(out), ref)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_heads_topk_candidates(M, dt):
    """medusa_heads_topk_candidates: the same head logits and top-s as
    medusa_heads_topk, and the candidates the oracle builds from that top-s;
    three calls on one workspace (its counters, the merged-heads one
    included, must be ready again each time)."""
    for spec, B, d, V in [(("cartesian", (2, 2, 2), None), 2, 256, 1000), (("greedy", 4, 10, 64), 1, 512, 4096)]:
        ot, dtree = both_trees(M, spec)
        K = ot.K + 1  # one head past the tree's depth, unused (s = 0)
        s = [int(v) for v in ot.s[:ot.K]] + [0]
        s_max = max(s)
        T = ot.T
        hidden = synth.normal(21, "hidden", (B, T, d), 1.0, dt)
        w1 = synth.normal(21, "w1", (K, d, d), 1 / math.sqrt(d), dt)
        w2 = synth.normal(21, "w2", (K, V, d), 1 / math.sqrt(d), dt)
        node = to_dev(np.array([(2 * b + 1) % T for b in range(B)], np.int32))
        root = np.array([(7 * b + 3) % V for b in range(B)], np.int32)
        hd, w1d, w2d = to_dev(hidden), to_dev(w1), to_dev(w2)
        hl_ref = torch.zeros((B, K, V), dtype=torch.float32, device="cuda")
        tk_ref = torch.zeros((B, K, s_max), dtype=torch.int32, device="cuda")
        ws = torch.zeros(M.medusa_heads_topk_workspace_size(B, K, d, V, s_max), dtype=torch.uint8, device="cuda")
        M.medusa_heads_topk(hd, node, w1d, None, w2d, s, hl_ref, tk_ref, ws)
        for rep in range(3):
            hl = torch.zeros_like(hl_ref)
            tk = torch.zeros_like(tk_ref)
            tok = torch.full((B, T), -9, dtype=torch.int32, device="cuda")
            e = err_flag()
            M.medusa_heads_topk_candidates(hd, node, w1d, None, w2d, s, hl, tk, ws, to_dev(root), dtree, tok, e)
            torch.cuda.synchronize()
            assert int(e.item()) == 0
            assert torch.equal(hl[:, :ot.K], hl_ref[:, :ot.K]) and torch.equal(tk, tk_ref)
            assert np.array_equal(to_host(tok), oracle.build_candidates(root, to_host(tk), ot)), f"call {rep}"


@pytest.mark.parametrize("nbytes", [16, 4096 + 48, 2130688, 8 << 20])
def test_copy_from_host(M, nbytes):
    """The staging copy moves pinned host bytes to the device exactly, inside a
    CUDA graph too; unmapped host memory is refused without a launch."""
    g = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    dst = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    M.medusa_copy_from_host(dst, src)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src)
    s = torch.cuda.Stream()
    dst.zero_()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        M.medusa_copy_from_host(dst, src, s)
    src.add_(1)  # the replay reads the buffer as it is then
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src)
    # pageable memory: refused, unless the runtime maps it for the device (a
    # host whose memory the GPU reads coherently), and then copied exactly
    pageable = torch.arange(64, dtype=torch.uint8)
    if pageable.data_ptr() % 16 == 0:
        out = torch.zeros(64, dtype=torch.uint8, device="cuda")
        try:
            M.medusa_copy_from_host(out, pageable)
        except RuntimeError:
            pass
        else:
            torch.cuda.synchronize()
            assert torch.equal(out.cpu(), pageable)
