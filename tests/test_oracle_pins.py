"""Pins for the CPU oracle: facts fixed by the pages or by mathematics.

Each test ties one oracle function to something other than itself: a value the
pages print (fixtures under tests/golden/, each with its citation), a closed
form, an invariant, a library routine the definition reduces to, or brute
force on a tiny input.  Sources are cited by page title and section:
  "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
  Heads" (paper digest: Method items 1-5, the decoding-step box, Paper vs code);
  "085 | Medusa" explainer (section 二); "Speculative decoding" (Maths).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def f32_to_bf16(a):
    """bf16 bits via torch's own conversion (an independent rounding routine)."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------- bf16 rounding

def test_bf16_round_special_values(orc):
    assert orc.bf16_round(1.0) == 0x3F80
    assert orc.bf16_round(-2.5) == 0xC020
    # exactly halfway between 1 and 1+2^-7: ties to even (down)
    assert orc.bf16_round(1.0 + 2.0 ** -8) == 0x3F80
    # halfway between 1+2^-7 and 1+2^-6: ties to even (up)
    assert orc.bf16_round(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # a hair above halfway rounds up
    assert orc.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert orc.bf16_round(0.0) == 0 and orc.bf16_round(-0.0) == 0x8000


def test_bf16_round_matches_torch(orc):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(4000).astype(np.float32) * 10.0 ** rng.integers(-20, 20, 4000),
                        rng.standard_normal(1000).astype(np.float32)])
    ours = np.array([orc.bf16_round(float(v)) for v in x], np.uint16)
    assert np.array_equal(ours, f32_to_bf16(x))


# ------------------------------------------------------------ candidate tree

@pytest.mark.parametrize("case", gold("tree_counts.json")["cases"])
def test_cartesian_node_count(orc, case):
    s = case["s"]
    paths, plen = orc.tree_cartesian(s, 100000)
    assert len(plen) == case["nodes"]
    assert sum(1 for l in plen if l == len(s)) == case["leaf_paths"]
    # closed form sum_k prod_{i<=k} s_i
    assert len(plen) == sum(math.prod(s[:k]) for k in range(1, len(s) + 1))
    t = orc.tree_compile(paths, plen, len(s))
    assert t.T == case["nodes"] + 1
    assert list(t.s) == s and t.K == len(s)


def test_cartesian_truncation_breadth_first(orc):
    # 256-node dense tree: the first 256 nodes of (4,4,4,4) in breadth-first order
    paths, plen = orc.tree_cartesian([4, 4, 4, 4], 256)
    assert len(plen) == 256
    assert list(np.bincount(plen)[1:]) == [4, 16, 64, 172]
    t = orc.tree_compile(paths, plen, 4)
    assert list(t.s) == [4, 4, 4, 4]


def _walk_ancestors(parent, i):
    out = set()
    while i >= 0:
        out.add(i)
        i = parent[i]
    return out


def test_tree_compile_structure(orc):
    rng = np.random.default_rng(5)
    # a random prefix-closed set of paths, shuffled
    paths = set()
    while len(paths) < 40:
        k = int(rng.integers(1, 5))
        p = tuple(int(r) for r in rng.integers(1, 4, size=k))
        for j in range(1, k + 1):
            paths.add(p[:j])
    paths = sorted(paths)
    rng.shuffle(paths)
    K = 4
    arr = np.zeros((len(paths), K), np.int32)
    for i, p in enumerate(paths):
        arr[i, :len(p)] = p
    plen = np.array([len(p) for p in paths], np.int32)
    t = orc.tree_compile(arr, plen, K)
    assert t.T == len(paths) + 1
    # breadth-first order: (depth, lexicographic)
    keys = [tuple(t.node_paths[n, :t.depth[n]]) for n in range(t.T)]
    assert keys == sorted(keys, key=lambda p: (len(p), p))
    for n in range(1, t.T):
        assert t.parent[n] < n
        assert keys[t.parent[n]] == keys[n][:-1]
        assert t.rank[n] == keys[n][-1]
        anc = _walk_ancestors(t.parent, n)
        assert set(np.nonzero(t.anc[n])[0]) == anc


def test_tree_compile_rejects_malformed(orc):
    with pytest.raises(ValueError):  # missing prefix (1,) for (1,2)
        orc.tree_compile(np.array([[1, 2], [2, 0]]), np.array([2, 1]), 2)
    with pytest.raises(ValueError):  # duplicate
        orc.tree_compile(np.array([[1, 0], [1, 0]]), np.array([1, 1]), 2)
    with pytest.raises(ValueError):  # rank 0
        orc.tree_compile(np.array([[0, 0]]), np.array([1]), 2)


def _brute_force_top(acc, K, budget):
    """All paths up to depth K, ranked by accuracy (desc; equal within 1e-9 in
    log space), then lexicographically; a node's parent always ranks above it,
    so the top `budget` set is what greedy growth of a connected tree picks."""
    R = acc.shape[1]
    items = []
    for k in range(1, K + 1):
        for p in itertools.product(range(1, R + 1), repeat=k):
            la = sum(math.log(acc[j, p[j] - 1]) for j in range(k))
            items.append((la, p))
    # group equal accuracies, then lexicographic inside a group
    items.sort(key=lambda x: -x[0])
    groups, cur = [], [items[0]]
    for it in items[1:]:
        if abs(it[0] - cur[-1][0]) <= 1e-9:
            cur.append(it)
        else:
            groups.append(cur)
            cur = [it]
    groups.append(cur)
    out = []
    for g in groups:
        out.extend(sorted(p for _, p in g))
    return out[:budget]


def test_greedy_tree_matches_brute_force(orc):
    K, R, budget = 4, 6, 64
    acc = 0.6 * 0.7 ** np.arange(K)[:, None] * 0.5 ** np.arange(R)[None, :]
    paths, plen = orc.tree_greedy(acc, budget)
    got = [tuple(paths[i, :plen[i]]) for i in range(len(plen))]
    want = _brute_force_top(acc, K, budget)
    assert len(got) == budget
    assert set(got) == set(want)
    # connected at every step: each added node's parent was added before it
    seen = {()}
    for p in got:
        assert p[:-1] in seen
        seen.add(p)


def test_greedy_tree_64_nodes_synthetic_table(orc):
    """The 64-node tree of the synthetic accuracy table used by the 7B/13B/33B
    workloads: accuracy depends only on the depth D and on S = sum(i_j - 1),
    so classes tie exactly; depth counts and s follow from the class cut."""
    K, R = 4, 10
    acc = 0.6 * 0.7 ** np.arange(K)[:, None] * 0.5 ** np.arange(R)[None, :]
    paths, plen = orc.tree_greedy(acc, 64)
    t = orc.tree_compile(paths, plen, K)
    assert list(np.bincount(plen)[1:]) == [8, 21, 30, 5]
    assert list(t.s) == [8, 6, 5, 2]
    e = orc.tree_expected_len(paths, plen, acc)
    assert abs(e - 3.621) < 5e-4
    # the same table with a fifth head gives the same tree (no depth-5 node
    # reaches the cut)
    acc5 = 0.6 * 0.7 ** np.arange(5)[:, None] * 0.5 ** np.arange(R)[None, :]
    p5, l5 = orc.tree_greedy(acc5, 64)
    got4 = sorted(tuple(paths[i, :plen[i]]) for i in range(64))
    got5 = sorted(tuple(p5[i, :l5[i]]) for i in range(64))
    assert got4 == got5


@pytest.mark.parametrize("case", gold("spec_closed_forms.json")["cases"])
def test_expected_tokens_chain_closed_form(orc, case):
    """A chain tree with i.i.d. acceptance alpha: 1 + sum_k alpha^k equals the
    page's (1 - alpha^(gamma+1)) / (1 - alpha) and its printed value."""
    a, g = case["alpha"], case["gamma"]
    paths = np.zeros((g, g), np.int32)
    for k in range(g):
        paths[k, :k + 1] = 1
    plen = np.arange(1, g + 1, dtype=np.int32)
    acc = np.full((g, 1), a)
    e = orc.tree_expected_len(paths, plen, acc)
    assert abs(e - (1 - a ** (g + 1)) / (1 - a)) < 1e-12
    if "alpha_printed_decimals" in case:
        # alpha itself was printed rounded: the printed value must be reachable
        # from some alpha inside its rounding interval (E is monotone in alpha)
        half = 0.5 * 10 ** -case["alpha_printed_decimals"]
        lo = orc.tree_expected_len(paths, plen, np.full((g, 1), a - half))
        hi = orc.tree_expected_len(paths, plen, np.full((g, 1), a + half))
        ulp = 0.5 * 10 ** -case["printed_decimals"]
        assert lo - ulp <= case["tokens_per_pass"] <= hi + ulp
    else:
        assert round(e, case["printed_decimals"]) == case["tokens_per_pass"]
    if "speedup" in case:
        assert round(e / (g * case["c"] + 1), 2) == case["speedup"]


# ------------------------------------------------------------------- RoPE

def test_rope_closed_form_pairs(orc):
    # Dh = 4: inv_freq = (1, theta^-1/2); pairing (0,2) and (1,3)
    theta = 10000.0
    for pos in (0, 1, 7, 1000):
        y = orc.rope(np.array([1.0, 0.0, 0.0, 0.0]), pos, theta)
        a = float(np.float32(pos) * np.float32(1.0))
        assert np.allclose(y, [math.cos(a), 0, math.sin(a), 0], atol=1e-15)
        y = orc.rope(np.array([0.0, 1.0, 0.0, 0.0]), pos, theta)
        a = float(np.float32(pos) * np.float32(1.0 / math.sqrt(theta)))
        assert np.allclose(y, [0, math.cos(a), 0, math.sin(a)], atol=1e-15)
        y = orc.rope(np.array([0.0, 0.0, 1.0, 0.0]), pos, theta)
        a = float(np.float32(pos))
        assert np.allclose(y, [-math.sin(a), 0, math.cos(a), 0], atol=1e-15)


def test_rope_norm_and_relative_position(orc):
    rng = np.random.default_rng(2)
    Dh = 128
    q, k = rng.standard_normal(Dh), rng.standard_normal(Dh)
    assert abs(np.linalg.norm(orc.rope(q, 1234)) - np.linalg.norm(q)) < 1e-12
    # q_m . k_n depends only on m - n (up to the fp32 angle rounding)
    d1 = orc.rope(q, 1030) @ orc.rope(k, 1000)
    d2 = orc.rope(q, 40) @ orc.rope(k, 10)
    assert abs(d1 - d2) < 2e-3 * (np.linalg.norm(q) * np.linalg.norm(k))
    assert np.array_equal(orc.rope(q, 0), q)


# -------------------------------------------------------------- attention

def test_attn_one_matches_sdpa_float64(orc):
    rng = np.random.default_rng(3)
    for n, Dh in ((1, 8), (5, 16), (70, 64)):
        q, k, v = rng.standard_normal(Dh), rng.standard_normal((n, Dh)), rng.standard_normal((n, Dh))
        scale = 1 / math.sqrt(Dh)
        got = orc.attn_one(q, k, v, scale)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None, None, None], torch.from_numpy(k)[None, None],
            torch.from_numpy(v)[None, None], scale=scale)[0, 0, 0].numpy()
        assert np.allclose(got, ref, rtol=0, atol=1e-12)
    # one key -> its value; equal keys -> the mean of the values
    v = rng.standard_normal((1, 8))
    assert np.allclose(orc.attn_one(rng.standard_normal(8), rng.standard_normal((1, 8)), v, 0.3), v[0], atol=1e-15)
    kk = np.tile(rng.standard_normal(8), (6, 1))
    vv = rng.standard_normal((6, 8))
    assert np.allclose(orc.attn_one(rng.standard_normal(8), kk, vv, 0.3), vv.mean(0), atol=1e-14)


def _tiny_tree(orc, s=(2, 2, 2)):
    paths, plen = orc.tree_cartesian(list(s), 10000)
    return orc.tree_compile(paths, plen, len(s))


def _attn_inputs(rng, B, T, H, Dh, L, dt=np.float32):
    q = rng.standard_normal((B, T, H, Dh)).astype(np.float32)
    kn = rng.standard_normal((B, T, H, Dh)).astype(np.float32)
    vn = rng.standard_normal((B, T, H, Dh)).astype(np.float32)
    cap = np.array(L) + T
    seq_start = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)
    kc = np.zeros((int(cap.sum()), H, Dh), np.float32)
    vc = np.zeros_like(kc)
    for b in range(B):
        kc[seq_start[b]:seq_start[b] + L[b]] = rng.standard_normal((L[b], H, Dh))
        vc[seq_start[b]:seq_start[b] + L[b]] = rng.standard_normal((L[b], H, Dh))
    return q, kn, vn, kc, vc, seq_start, np.array(L, np.int32)


def test_tree_attention_equals_per_path_attention(orc):
    """Each node's result equals ordinary attention over the prefix plus the
    node's own root-to-node path at positions L..L+depth (explainer 085,
    '候选树中相同深度不表示相同上下文'; digest Method 3)."""
    rng = np.random.default_rng(4)
    t = _tiny_tree(orc)
    B, H, Dh, L = 2, 2, 16, [9, 5]
    q, kn, vn, kc, vc, st, pl = _attn_inputs(rng, B, t.T, H, Dh, L)
    kc0 = kc.copy()
    out, out_d = orc.tree_attn(q, kn, vn, kc, vc, st, pl, t, 10000.0, 1 / math.sqrt(Dh))
    for b in range(B):
        for i in range(t.T):
            path = sorted(_walk_ancestors(t.parent, i), key=lambda n: t.depth[n])
            for h in range(H):
                keys = [kc0[st[b] + j, h].astype(np.float64) for j in range(L[b])]
                vals = [vc[st[b] + j, h].astype(np.float64) for j in range(L[b])]
                for n in path:
                    keys.append(np.float32(orc.rope(kn[b, n, h], L[b] + t.depth[n])).astype(np.float64))
                    vals.append(vn[b, n, h].astype(np.float64))
                qi = orc.rope(q[b, i, h], L[b] + t.depth[i])
                ref = orc.attn_one(qi, np.array(keys), np.array(vals), 1 / math.sqrt(Dh))
                assert np.allclose(out_d[b, i, h], ref, rtol=0, atol=1e-12)
    # the prefix is untouched; tree rows were appended at L + i
    for b in range(B):
        assert np.array_equal(kc[st[b]:st[b] + L[b]], kc0[st[b]:st[b] + L[b]])
        assert np.array_equal(vc[st[b] + L[b]:st[b] + L[b] + t.T], vn[b])


def test_tree_attention_chain_is_causal_sdpa(orc):
    """A chain tree (all s_k = 1) reduces to plain causal decoding: compare with
    torch's float64 scaled_dot_product_attention under a causal mask."""
    rng = np.random.default_rng(6)
    t = _tiny_tree(orc, (1, 1, 1, 1))
    B, H, Dh, L = 1, 3, 32, [11]
    q, kn, vn, kc, vc, st, pl = _attn_inputs(rng, B, t.T, H, Dh, L)
    kc0 = kc.copy()
    _, out_d = orc.tree_attn(q, kn, vn, kc, vc, st, pl, t)
    T = t.T
    for h in range(H):
        qs = np.stack([orc.rope(q[0, i, h], L[0] + i) for i in range(T)])
        ks = np.concatenate([kc0[:L[0], h].astype(np.float64),
                             np.stack([np.float32(orc.rope(kn[0, i, h], L[0] + i)) for i in range(T)]).astype(np.float64)])
        vs = np.concatenate([vc[:L[0], h], vn[0, :, h]]).astype(np.float64)
        mask = np.ones((T, L[0] + T), bool)
        mask[:, L[0]:] = np.tril(np.ones((T, T), bool))
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qs)[None], torch.from_numpy(ks)[None], torch.from_numpy(vs)[None],
            attn_mask=torch.from_numpy(mask)[None], scale=1 / math.sqrt(Dh))[0].numpy()
        assert np.allclose(out_d[0, :, h], ref, rtol=0, atol=1e-12)


def test_tree_attention_siblings_invisible(orc):
    rng = np.random.default_rng(7)
    t = _tiny_tree(orc)
    B, H, Dh, L = 1, 2, 16, [6]
    q, kn, vn, kc, vc, st, pl = _attn_inputs(rng, B, t.T, H, Dh, L)
    _, base = orc.tree_attn(q, kn, vn, kc.copy(), vc.copy(), st, pl, t)
    n = t.T - 1  # a leaf
    for m in range(t.T):
        kn2, vn2 = kn.copy(), vn.copy()
        kn2[0, m] += 1.0
        vn2[0, m] -= 1.0
        _, o2 = orc.tree_attn(q, kn2, vn2, kc.copy(), vc.copy(), st, pl, t)
        changed = not np.array_equal(o2[0, n], base[0, n])
        assert changed == bool(t.anc[n, m])


def test_tree_attention_bf16_rounds_output(orc):
    rng = np.random.default_rng(8)
    t = _tiny_tree(orc)
    q, kn, vn, kc, vc, st, pl = _attn_inputs(rng, 1, t.T, 2, 16, [7])
    bf = lambda a: f32_to_bf16(a)
    out, out_d = orc.tree_attn(bf(q), bf(kn), bf(vn), bf(kc), bf(vc), st, pl, t)
    assert out.dtype == np.uint16
    # every stored value is the nearest bf16 of the exact result: within half
    # a unit in the last place, 2^(floor(log2|x|) - 8)
    half_ulp = np.exp2(np.floor(np.log2(np.abs(out_d))) - 8)
    assert np.all(np.abs(orc.to_double(out) - out_d) <= half_ulp)
    # and it is one of the two bf16 neighbours picked by torch's own rounding
    # of the float32-rounded value (double rounding can only move a tie)
    tb = f32_to_bf16(out_d.astype(np.float32))
    assert np.all(np.abs(out.astype(np.int32) - tb.astype(np.int32)) <= 1)


# ---------------------------------------------------------------- LM head

def test_lm_head_matches_matmul(orc):
    rng = np.random.default_rng(9)
    h = rng.standard_normal((7, 64)).astype(np.float32)
    w = rng.standard_normal((33, 64)).astype(np.float32)
    got = orc.lm_head(h, w)
    assert np.allclose(got, h.astype(np.float64) @ w.astype(np.float64).T, rtol=1e-13, atol=1e-12)
    # bf16 inputs widen exactly
    hb, wb = f32_to_bf16(h), f32_to_bf16(w)
    got = orc.lm_head(hb, wb)
    assert np.allclose(got, orc.to_double(hb) @ orc.to_double(wb).T, rtol=1e-13, atol=1e-12)
    # unit rows of W pick out hidden entries
    e = np.eye(64, dtype=np.float32)[:5]
    assert np.array_equal(orc.lm_head(h, e), h[:, :5].astype(np.float64))


# ------------------------------------------------------------- acceptance

def _planted(orc, t, V, node, rng, margin=4.0):
    """Logits with a clear argmax per row; tokens along root->node set to the
    parent row's argmax, all other tokens set to something else."""
    T = t.T
    logits = rng.standard_normal((1, T, V)).astype(np.float32)
    am = rng.integers(0, V, T)
    logits[0, np.arange(T), am] = logits[0].max(axis=1) + margin
    tok = np.zeros((1, T), np.int32)
    path = _walk_ancestors(t.parent, node)
    for c in range(1, T):
        p = t.parent[c]
        tok[0, c] = am[p] if c in path else (am[p] + 1 + c) % V
    return logits, tok, am


def test_accept_greedy_planted_every_node(orc):
    """Greedy acceptance: a node is accepted iff the parent's argmax equals its
    token, on an unbroken prefix; the longest accepted path wins (digest,
    algorithm box steps 4-5)."""
    rng = np.random.default_rng(10)
    t = _tiny_tree(orc, (3, 2, 2))
    V = 50
    for node in range(t.T):
        logits, tok, am = _planted(orc, t, V, node, rng)
        assert np.array_equal(np.argmax(logits[0], axis=1), am)
        r = orc.accept(logits, tok, t, 0)
        assert r["accept_len"][0] == t.depth[node]
        path = sorted(_walk_ancestors(t.parent, node), key=lambda n: t.depth[n])
        want = np.full(t.K + 1, -1)
        want[:len(path)] = path
        assert np.array_equal(r["accepted_nodes"][0], want)
        assert r["next_root"][0] == am[node]
        assert r["best_node"][0] == node


def test_accept_stops_at_first_rejection(orc):
    rng = np.random.default_rng(11)
    t = _tiny_tree(orc, (1, 1, 1))  # chain 0-1-2-3
    V = 20
    logits, tok, am = _planted(orc, t, V, 3, rng)
    tok[0, 2] = (am[1] + 1) % V  # break depth 2; depth 3 still "matches"
    r = orc.accept(logits, tok, t, 0)
    assert r["accept_len"][0] == 1
    assert list(r["accepted_nodes"][0]) == [0, 1, -1, -1]


def test_accept_root_always(orc):
    rng = np.random.default_rng(12)
    t = _tiny_tree(orc)
    logits, tok, am = _planted(orc, t, 40, 0, rng)
    for mode in (0, 1):
        r = orc.accept(logits, tok, t, mode, temperature=0.7, eps=0.09, delta=0.3)
        assert r["accept_len"][0] == 0
        assert r["accepted_nodes"][0][0] == 0
        assert r["next_root"][0] == am[0]


def test_typical_uniform_row_closed_form(orc):
    """Uniform row: p-hat = 1/V, H = log V, threshold min(eps, delta/V)."""
    t = _tiny_tree(orc, (1,))
    V = 8
    logits = np.zeros((1, 2, V), np.float32)
    tok = np.array([[0, 3]], np.int32)
    r = orc.accept(logits, tok, t, 1, temperature=1.0, eps=0.09, delta=0.3)
    assert r["accept_len"][0] == 1  # 0.125 > min(0.09, 0.0375)
    assert abs(r["node_margin"][0, 1] - (1 / 8 - 0.3 / 8)) < 1e-15
    r = orc.accept(logits, tok, t, 1, temperature=1.0, eps=0.2, delta=3.0)
    assert r["accept_len"][0] == 0  # 0.125 < min(0.2, 0.375)
    assert abs(r["best_logp"][0]) == 0.0


def test_typical_margin_matches_scipy(orc):
    from scipy.special import softmax
    from scipy.stats import entropy

    rng = np.random.default_rng(13)
    t = _tiny_tree(orc, (2, 2))
    V, tau, eps, delta = 100, 0.7, 0.09, 0.3
    logits = (rng.standard_normal((1, t.T, V)) * 3).astype(np.float32)
    tok = rng.integers(0, V, (1, t.T)).astype(np.int32)
    r = orc.accept(logits, tok, t, 1, temperature=tau, eps=eps, delta=delta)
    for c in range(1, t.T):
        p = softmax(logits[0, t.parent[c]].astype(np.float64) / tau)
        want = p[tok[0, c]] - min(eps, delta * math.exp(-entropy(p)))
        assert abs(r["node_margin"][0, c] - want) < 1e-12


def test_typical_low_temperature_is_greedy(orc):
    """At temperature -> 0 typical acceptance reduces to greedy (digest,
    Method 5)."""
    rng = np.random.default_rng(14)
    t = _tiny_tree(orc, (3, 2, 2))
    for node in range(0, t.T, 3):
        logits, tok, am = _planted(orc, t, 64, node, rng, margin=2.0)
        g = orc.accept(logits, tok, t, 0)
        ty = orc.accept(logits, tok, t, 1, temperature=1e-3, eps=0.09, delta=0.3)
        for key in ("accept_len", "accepted_nodes", "next_root", "best_node"):
            assert np.array_equal(g[key], ty[key])


def test_typical_tie_break_by_logprob(orc):
    """Two fully accepted paths of equal length: the one with the larger
    summed log-probability wins (digest, Paper vs code: typical acceptance)."""
    t = _tiny_tree(orc, (2,))  # root with children 1, 2
    V = 4
    logits = np.log(np.array([[[0.1, 0.5, 0.4, 1e-9]] * 3], np.float64)).astype(np.float32)
    tok = np.array([[0, 2, 1]], np.int32)  # node 1 -> p=0.4, node 2 -> p=0.5
    r = orc.accept(logits, tok, t, 1, temperature=1.0, eps=0.09, delta=0.3)
    assert r["accept_len"][0] == 1 and r["best_node"][0] == 2
    assert abs(r["best_logp"][0] - math.log(0.5)) < 1e-6


# ----------------------------------------------------------- KV compaction

def test_kv_compact_permutation_and_hazard(orc):
    H, Dh, K = 2, 4, 3
    L = [5, 3]
    T = 8
    cap = np.array(L) + T
    st = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)
    kc = np.arange(int(cap.sum()) * H * Dh, dtype=np.float32).reshape(-1, H, Dh)
    vc = -kc
    k0, v0 = kc.copy(), vc.copy()
    # seq 0: a source of row 1 (slot L+2) is the destination of row 2
    acc_nodes = np.array([[0, 2, 3, -1], [0, 4, 6, 7]], np.int32)
    acc_len = np.array([2, 3], np.int32)
    pl = np.array(L, np.int32)
    src = orc.kv_compact(kc, vc, st, pl, acc_nodes, acc_len, K)
    for b in range(2):
        for j in range(acc_len[b] + 1):
            a = acc_nodes[b, j]
            assert np.array_equal(kc[st[b] + L[b] + j], k0[st[b] + L[b] + a])
            assert np.array_equal(vc[st[b] + L[b] + j], v0[st[b] + L[b] + a])
        assert np.array_equal(kc[st[b]:st[b] + L[b]], k0[st[b]:st[b] + L[b]])
    assert list(pl) == [5 + 3, 3 + 4]
    assert list(src[0]) == [5, 7, 8, -1] and list(src[1]) == [3, 7, 9, 10]


# ------------------------------------------------------------------ heads

def test_heads_init_reproduces_lm_head(orc):
    """W1 = 0 and W2 = the LM head: each head reproduces the base model's
    next-token prediction (digest Method 1, initialisation)."""
    rng = np.random.default_rng(15)
    B, T, d, V, K = 2, 5, 32, 97, 3
    hidden = f32_to_bf16(rng.standard_normal((B, T, d)))
    wlm = f32_to_bf16(rng.standard_normal((V, d)) / math.sqrt(d))
    w1 = np.zeros((K, d, d), np.uint16)
    w2 = np.ascontiguousarray(np.broadcast_to(wlm, (K, V, d)))
    last = np.array([3, 1], np.int32)
    z, topk, u = orc.heads(hidden, last, w1, None, w2, [4, 4, 4], 4)
    lm = orc.lm_head(hidden, wlm).reshape(B, T, V)
    for b in range(B):
        assert np.array_equal(u[b, 0], hidden[b, last[b]])
        for k in range(K):
            assert np.array_equal(z[b, k], lm[b, last[b]])
            assert topk[b, k, 0] == int(np.argmax(lm[b, last[b]]))


def test_heads_match_float64_numpy(orc):
    rng = np.random.default_rng(16)
    B, T, d, V, K = 1, 3, 16, 40, 2
    hidden = rng.standard_normal((B, T, d)).astype(np.float32)
    w1 = (rng.standard_normal((K, d, d)) * 0.3).astype(np.float32)
    b1 = rng.standard_normal((K, d)).astype(np.float32)
    w2 = rng.standard_normal((K, V, d)).astype(np.float32)
    z, topk, u = orc.heads(hidden, np.array([2], np.int32), w1, b1, w2, [3, 5], 5)
    h = hidden[0, 2].astype(np.float64)
    for k in range(K):
        y = w1[k].astype(np.float64) @ h + b1[k]
        uu = (y / (1 + np.exp(-y)) + h).astype(np.float32).astype(np.float64)
        assert np.array_equal(u[0, k].astype(np.float64), uu)
        zz = w2[k].astype(np.float64) @ uu
        assert np.allclose(z[0, k], zz, rtol=1e-13, atol=1e-12)
        s = [3, 5][k]
        order = np.lexsort((np.arange(V), -zz))[:s]
        assert list(topk[0, k, :s]) == list(order)
        assert all(x == -1 for x in topk[0, k, s:])


def test_heads_hand_example(orc):
    # d = 2, V = 2: h = (1, -1), W1 = [[1, 0], [0, 0]] -> y = (1, 0)
    # u = (SiLU(1) + 1, SiLU(0) - 1) = (1.7310585786300049, -1)
    hidden = np.array([[[1.0, -1.0]]], np.float32)
    w1 = np.array([[[1.0, 0.0], [0.0, 0.0]]], np.float32)
    w2 = np.array([[[1.0, 0.0], [0.0, 1.0]]], np.float32)
    z, topk, u = orc.heads(hidden, np.array([0], np.int32), w1, None, w2, [2], 2)
    assert abs(z[0, 0, 0] - float(np.float32(1.7310585786300049))) < 1e-15
    assert z[0, 0, 1] == -1.0
    assert list(topk[0, 0]) == [0, 1]


def test_heads_skip_zero_s_and_topk_ties(orc):
    hidden = np.zeros((1, 1, 4), np.float32)
    w1 = np.zeros((2, 4, 4), np.float32)
    w2 = np.zeros((2, 6, 4), np.float32)
    z, topk, _ = orc.heads(hidden, np.array([0], np.int32), w1, None, w2, [3, 0], 3)
    assert list(topk[0, 0]) == [0, 1, 2]  # all equal: lowest indices first
    assert list(topk[0, 1]) == [-1, -1, -1]
    assert list(orc.topk_f32(np.array([1, 5, 5, 2, 5], np.float32), 3)) == [1, 2, 4]


# ------------------------------------------------------------- candidates

def test_build_candidates_fill(orc):
    """The node for path (i_1..i_k) gets the i_k-th top token of head k; the
    root gets t0 (digest, algorithm box steps 1-2)."""
    t = _tiny_tree(orc, (2, 3))
    topk = np.array([[[10, 11, -1], [20, 21, 22]]], np.int32)
    tok = orc.build_candidates(np.array([7], np.int32), topk, t)
    for n in range(t.T):
        p = tuple(t.node_paths[n, :t.depth[n]])
        want = 7 if not p else topk[0, len(p) - 1, p[-1] - 1]
        assert tok[0, n] == want


# ------------------------------------------------------ rejection sampling

def test_rejection_two_token_example(orc):
    g = gold("rejection_two_token.json")
    out, beta = orc.rejection_emit(g["p"], g["q"])
    assert abs(beta - g["beta"]) < g["tol"]
    assert np.allclose(out, g["emitted"], rtol=0, atol=g["tol"])
    # token 0 is accepted with min(1, p/q) = 0.75
    assert abs(min(1, g["p"][0] / g["q"][0]) - g["accept_prob_token0"]) < 1e-15


def test_rejection_emits_target_for_random_pairs(orc):
    rng = np.random.default_rng(17)
    for n in (2, 8, 1000):
        p = rng.random(n); p /= p.sum()
        q = rng.random(n); q /= q.sum()
        out, beta = orc.rejection_emit(p, q)
        assert np.allclose(out, p, rtol=0, atol=1e-14)
        assert abs(beta - np.minimum(p, q).sum()) < 1e-14
    out, beta = orc.rejection_emit(p, p)
    assert abs(beta - 1.0) < 1e-12 and np.allclose(out, p, atol=1e-14)


# --------------------------------------------- rejection sampling over the tree

def _cart_tree(orc, s):
    n = sum(int(np.prod(s[:k])) for k in range(1, len(s) + 1))
    paths, plen = orc.tree_cartesian(list(s), n)
    return orc.tree_compile(paths, plen, len(s))


def _first_tokens(r, tokens, n_emit):
    """The first n_emit emitted tokens of each trial: the accepted path's tokens
    (after the root), then the final draw."""
    B = len(r["accept_len"])
    out = np.full((B, n_emit), -1, np.int64)
    for b in range(B):
        seq = [tokens[b, n] for n in r["accepted_nodes"][b, 1:r["accept_len"][b] + 1]] + [r["next_token"][b]]
        out[b, :min(n_emit, len(seq))] = seq[:n_emit]
    return out


def test_rejection_tree_two_token_example_exact(orc):
    """The worked two-token example (p = (0.6, 0.4), q = (0.8, 0.2)) on a root with
    one child drafted from q: integrating the child's token over q and both
    uniforms over a midpoint grid gives the emitted distribution p."""
    g = gold("rejection_two_token.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    t = _cart_tree(orc, (1,))
    N = 300
    uu = (np.arange(N) + 0.5) / N
    U1, U2 = np.meshgrid(uu, uu, indexing="ij")
    trials = []
    for x in (0, 1):
        B = N * N
        u = np.zeros((B, 2, 2), np.float32)
        u[:, 0, 0] = U1.ravel()   # the child's test
        u[:, 0, 1] = U2.ravel()   # final draw after a rejection at the root
        u[:, 1, 0] = U2.ravel()   # final draw at the accepted (childless) child
        logits = np.broadcast_to(np.log(p).astype(np.float32), (B, 2, 2)).copy()
        draft = np.broadcast_to(np.log(q).astype(np.float32), (B, 1, 2)).copy()
        tokens = np.zeros((B, 2), np.int32)
        tokens[:, 1] = x
        r = orc.rejection_tree(logits, draft, tokens, t, 1.0, u)
        first = _first_tokens(r, tokens, 1)[:, 0]
        trials.append((q[x], np.bincount(first, minlength=2) / B))
    emitted = sum(w * h for w, h in trials)
    assert np.abs(emitted - p).max() <= 2.0 / N
    # with the child fixed to token 0 (not drafted from q) the rule emits (0.75, 0.25)
    assert np.abs(trials[0][1] - np.array([0.75, 0.25])).max() <= 2.0 / N


def test_rejection_tree_siblings_lossless(orc):
    """Three siblings drafted independently from q, tried in rank order with
    the residual update: the first emitted token is distributed as p
    (Monte Carlo, 5 sigma)."""
    rng = np.random.default_rng(23)
    V, m, B = 5, 3, 120000
    p = rng.random(V) ** 2; p /= p.sum()
    q = rng.random(V); q /= q.sum()
    t = _cart_tree(orc, (m,))
    logits = np.broadcast_to(np.log(p).astype(np.float32), (B, t.T, V)).copy()
    draft = np.broadcast_to(np.log(q).astype(np.float32), (B, 1, V)).copy()
    tokens = np.zeros((B, t.T), np.int32)
    tokens[:, 1:] = rng.choice(V, size=(B, m), p=q)
    u = rng.random((B, t.T, m + 1)).astype(np.float32)
    r = orc.rejection_tree(logits, draft, tokens, t, 1.0, u)
    first = _first_tokens(r, tokens, 1)[:, 0]
    emp = np.bincount(first, minlength=V) / B
    assert np.all(np.abs(emp - p) <= 5 * np.sqrt(p * (1 - p) / B) + 1e-12)
    # a rejected chain can end on the draw: some trials accept nothing
    assert 0 < np.mean(r["accept_len"] == 0) < 1


def test_rejection_tree_depth_two_lossless(orc):
    """Root -> two children -> two children each, every level drafted from its
    own q, the target at a node a function of its token: the first two emitted
    tokens are distributed as p_root(x1) * p_x1(x2)."""
    rng = np.random.default_rng(29)
    V, B = 3, 200000
    t = _cart_tree(orc, (2, 2))
    p_root = rng.random(V); p_root /= p_root.sum()
    table = rng.random((V, V)); table /= table.sum(1, keepdims=True)   # target after token x
    q1 = rng.random(V); q1 /= q1.sum()
    q2 = rng.random(V); q2 /= q2.sum()
    tokens = np.zeros((B, t.T), np.int32)
    for n in range(1, t.T):
        tokens[:, n] = rng.choice(V, size=B, p=q1 if t.depth[n] == 1 else q2)
    logits = np.zeros((B, t.T, V), np.float32)
    logits[:, 0] = np.log(p_root)
    for n in range(1, t.T):
        logits[:, n] = np.log(table[tokens[:, n]])
    draft = np.zeros((B, 2, V), np.float32)
    draft[:, 0], draft[:, 1] = np.log(q1), np.log(q2)
    u = rng.random((B, t.T, 3)).astype(np.float32)
    r = orc.rejection_tree(logits, draft, tokens, t, 1.0, u)
    f = _first_tokens(r, tokens, 2)
    # a trial that stopped after one token continues in the next step, whose
    # root row is the target after that token: draw it from there
    short = f[:, 1] < 0
    cdf = np.cumsum(table[f[short, 0]], axis=1)
    f[short, 1] = (rng.random(short.sum())[:, None] >= cdf).sum(1)
    joint = np.zeros((V, V))
    np.add.at(joint, (f[:, 0], f[:, 1]), 1.0)
    joint /= B
    want = p_root[:, None] * table
    assert np.all(np.abs(joint - want) <= 5 * np.sqrt(want * (1 - want) / B) + 1e-12)


def test_rejection_tree_draft_equals_target(orc):
    """q = p: every first child is accepted (u q < p for u < 1), down to a leaf."""
    rng = np.random.default_rng(31)
    V, B = 7, 500
    t = _cart_tree(orc, (2, 2, 2))
    z = rng.normal(size=V).astype(np.float32)
    logits = np.broadcast_to(z, (B, t.T, V)).copy()
    draft = np.broadcast_to(z, (B, 3, V)).copy()
    tokens = rng.integers(0, V, (B, t.T)).astype(np.int32)
    u = rng.random((B, t.T, 3)).astype(np.float32)
    r = orc.rejection_tree(logits, draft, tokens, t, 0.7, u)
    assert np.all(r["accept_len"] == 3)
    assert np.all(r["accepted_nodes"][:, 1] == 1)
