"""The closed decode loop (steps chained on the device around the stand-in
backbone of medusa_tree_speculative_gb300.loop): greedy Medusa decoding is
lossless, so the tokens it emits must be the stand-in model's plain greedy
continuation -- checked against the oracle's LM head (argmax of W_lm E[x] at
every emitted token) and against the chain the stand-in is built on -- and
the KV cache must hold, slot after slot, the rows of the emitted tokens (V
exact, K rotated at its position).  Also: medusa_append_tokens on its own.
"""
import numpy as np
import pytest
import torch

import oracle
from medusa_tree_speculative_gb300 import synth, workloads
from parity_util import as_double, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from medusa_tree_speculative_gb300 import build

    build.build()
    from medusa_tree_speculative_gb300 import medusa

    return medusa


def _loop(M, name, n_steps, B, heads, side):
    from medusa_tree_speculative_gb300 import loop, step

    w = dict(workloads.get(name), B=B)
    tree = M.DeviceTree(step.build_tree(w))
    model = loop.StandInModel(w, seed=3)
    x0 = np.array([(97 * b + 5) % w["V"] for b in range(B)])
    lp = loop.DecodeLoop(w, model, tree, n_steps, L0=w["L"][0], x0=x0, heads=heads)
    s2 = torch.cuda.Stream() if side else None
    s3 = torch.cuda.Stream() if (side and heads == "split") else None
    for _ in range(n_steps):
        lp.step(side_stream=s2, heads_stream=s3)
    torch.cuda.synchronize()
    assert int(lp.st.err.item()) == 0
    return w, model, lp


@pytest.mark.parametrize("name,B,heads,side", [("tiny_fp32", 1, "fused", False), ("tiny_fp32", 2, "split", True),
                                               ("vicuna7b_L1024_tree64", 1, "fused", True)])
def test_decode_loop_is_greedy_decoding(M, name, B, heads, side):
    n_steps = 12
    w, model, lp = _loop(M, name, n_steps, B, heads, side)
    got = lp.emitted()
    ref = lp.greedy_reference(max(len(g) for g in got))
    Eh, Wh = to_host(model.E), to_host(model.w_lm)  # float32, or bf16 bits
    E = as_double(Eh)
    for b in range(B):
        n = len(got[b])
        assert n >= n_steps  # at least the root every step
        assert np.array_equal(got[b], ref[b, :n])
        # the oracle's LM head agrees: each emitted token is the argmax after the previous one
        prev = int(lp.x0[b])
        check = got[b] if name == "tiny_fp32" else got[b][:6]
        lg = oracle.lm_head(np.ascontiguousarray(Eh[np.concatenate([[prev], check[:-1]]).astype(np.int64)]), Wh)
        assert np.array_equal(np.argmax(lg, axis=1), check)
        # cache: slot L0 + i holds token i's row (V exactly, K rotated at L0 + i)
        L0 = w["L"][0]
        cap = int(lp.x["seq_cap"][b].item())
        st0 = b * cap
        assert int(lp.x["prefix_len"][b].item()) == L0 + n
        vg = to_host(lp.x["v_cache"])[st0 + L0:st0 + L0 + n].reshape(n, -1)
        assert np.array_equal(vg, Eh[got[b]])
        kg = as_double(to_host(lp.x["k_cache"])[st0 + L0:st0 + L0 + n])
        H, Dh = w["H"], w["Dh"]
        for i in (0, n // 2, n - 1):
            kref = np.stack([oracle.rope(E[got[b][i]].reshape(H, Dh)[hh], L0 + i) for hh in range(H)])
            tol = (2.0 ** -7 if w["dtype"] == "bf16" else 2.0 ** -20) * np.abs(kref) + 1e-6
            assert np.all(np.abs(kg[i] - kref) <= tol)
    # the heads reach past the root on this stand-in
    assert sum(len(g) for g in got) > B * n_steps


def test_append_tokens(M):
    B, T, Kmax, cap = 3, 9, 3, 10
    rng = np.random.default_rng(5)
    tokens = rng.integers(0, 1000, (B, T)).astype(np.int32)
    nodes = np.array([[0, 2, 5, -1], [0, -1, -1, -1], [0, 1, 4, 8]], np.int32)
    alen = np.array([2, 0, 3], np.int32)
    out = torch.full((B, cap), -7, dtype=torch.int32, device="cuda")
    out_len = to_dev(np.array([1, 0, 7], np.int32))  # sequence 2 is one slot short
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.medusa_append_tokens(to_dev(tokens), to_dev(nodes), to_dev(alen), out, out_len, e)
    torch.cuda.synchronize()
    o, n = to_host(out), to_host(out_len)
    assert list(n) == [4, 1, 7]
    assert list(o[0, 1:4]) == [tokens[0, 0], tokens[0, 2], tokens[0, 5]] and o[0, 0] == -7
    assert o[1, 0] == tokens[1, 0]
    assert np.all(o[2] == -7)
    assert int(e.item()) & 4  # capacity
