"""Rejection-sampling acceptance over the tree on the GPU
(medusa_accept_rejection): decision-for-decision parity with the oracle on
the same uniforms, and Monte Carlo checks that the emitted tokens follow the
target distribution when the drafts are independent draws from q (the
two-token worked example, three siblings)."""
import math

import numpy as np
import pytest
import torch

import oracle
from medusa_tree_speculative_gb300 import synth
from parity_util import both_trees, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from medusa_tree_speculative_gb300 import build

    build.build()
    from medusa_tree_speculative_gb300 import medusa

    return medusa


def _run(M, dtree, logits, draft, tokens, tau, u):
    B, T, V = logits.shape
    K = dtree.K
    al = torch.zeros(B, dtype=torch.int32, device="cuda")
    an = torch.zeros((B, K + 1), dtype=torch.int32, device="cuda")
    nt = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(M.medusa_accept_rejection_workspace_size(B, V), dtype=torch.uint8, device="cuda")
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.medusa_accept_rejection(to_dev(logits), to_dev(draft), to_dev(tokens), dtree, tau, to_dev(u), al, an, nt,
                              ws, e)
    torch.cuda.synchronize()
    return to_host(al), to_host(an), to_host(nt), int(e.item())


def _first(al, an, nt, tokens, n_emit):
    B = len(al)
    out = np.full((B, n_emit), -1, np.int64)
    for b in range(B):
        seq = [tokens[b, n] for n in an[b, 1:al[b] + 1]] + [nt[b]]
        out[b, :min(n_emit, len(seq))] = seq[:n_emit]
    return out


@pytest.mark.parametrize("spec,V,tau", [(("greedy", 4, 10, 64), 32000, 0.7), (("cartesian", (2, 3, 2), None), 50, 1.0),
                                        (("cartesian", (4, 4, 4, 4), 256), 1000, 0.5)])
def test_rejection_parity(M, spec, V, tau):
    ot, dtree = both_trees(M, spec)
    B, T, K = 16, ot.T, ot.K
    rng = np.random.default_rng(41)
    logits = synth.normal(41, "tgt", (B, T, V), 2.0, "f32")
    draft = synth.normal(41, "draft", (B, K, V), 2.0, "f32")
    # drafts: a mix of the target's likely tokens and of random ones, so both outcomes occur
    tokens = np.zeros((B, T), np.int32)
    for n in range(1, T):
        p = int(ot.parent[n])
        top = np.argsort(-logits[:, p], axis=1)[:, :4]
        pick = rng.integers(0, 4, B)
        tokens[:, n] = np.where(rng.random(B) < 0.4, top[np.arange(B), pick], rng.integers(0, V, B))
    u = rng.random((B, T, 17)).astype(np.float32)
    # The oracle's margin of a sequence is the smallest distance of any of its
    # decisions from the other outcome: |u q(x) - p(x)| / max(p(x), q(x)) for
    # an acceptance test, and |u - F| for the final inverse-CDF draw, with F
    # the nearer bound of the drawn token's cumulative interval.  The GPU's
    # probabilities are float32 exponentials over sums of <= 32000 terms
    # (relative error below 1e-6; the cumulative sums are carried in double),
    # so a decision whose margin exceeds 1e-5 cannot go the other way.  A
    # sequence with a closer decision gets fresh uniforms (the oracle alone
    # decides which), at most 20 times.
    for _ in range(20):
        r = oracle.rejection_tree(logits, draft, tokens, ot, tau, u)
        close = r["margin"] <= 1e-5
        if not close.any():
            break
        u[close] = rng.random((int(close.sum()), T, 17)).astype(np.float32)
    r = oracle.rejection_tree(logits, draft, tokens, ot, tau, u)
    clear = r["margin"] > 1e-5
    assert clear.mean() >= 0.95
    al, an, nt, err = _run(M, dtree, logits, draft, tokens, tau, u)
    assert err == 0
    for b in np.nonzero(clear)[0]:
        assert al[b] == r["accept_len"][b]
        assert np.array_equal(an[b], r["accepted_nodes"][b])
        assert nt[b] == r["next_token"][b]


def test_rejection_two_token_example_monte_carlo(M):
    """p = (0.6, 0.4), q = (0.8, 0.2), the child drafted from q: the first
    emitted token is distributed as p (40 000 sequences, 5 sigma)."""
    ot, dtree = both_trees(M, ("cartesian", (1,), None))
    B, V = 40000, 2
    rng = np.random.default_rng(43)
    p, q = np.array([0.6, 0.4]), np.array([0.8, 0.2])
    logits = np.broadcast_to(np.log(p).astype(np.float32), (B, 2, V)).copy()
    draft = np.broadcast_to(np.log(q).astype(np.float32), (B, 1, V)).copy()
    tokens = np.zeros((B, 2), np.int32)
    tokens[:, 1] = rng.choice(V, size=B, p=q)
    u = rng.random((B, 2, 2)).astype(np.float32)
    al, an, nt, err = _run(M, dtree, logits, draft, tokens, 1.0, u)
    assert err == 0
    emp = np.bincount(_first(al, an, nt, tokens, 1)[:, 0], minlength=V) / B
    assert np.all(np.abs(emp - p) <= 5 * np.sqrt(p * (1 - p) / B))
    # acceptance rate of the draft: sum min(p, q) = 0.8
    assert abs(np.mean(al == 1) - 0.8) <= 5 * math.sqrt(0.16 / B)
    # the same trials through the oracle agree one by one
    r = oracle.rejection_tree(logits, draft, tokens, ot, 1.0, u)
    assert np.array_equal(al, r["accept_len"]) and np.array_equal(nt, r["next_token"])


def test_rejection_siblings_monte_carlo(M):
    ot, dtree = both_trees(M, ("cartesian", (3,), None))
    B, V, m = 60000, 5, 3
    rng = np.random.default_rng(47)
    p = rng.random(V) ** 2; p /= p.sum()
    q = rng.random(V); q /= q.sum()
    logits = np.broadcast_to(np.log(p).astype(np.float32), (B, ot.T, V)).copy()
    draft = np.broadcast_to(np.log(q).astype(np.float32), (B, 1, V)).copy()
    tokens = np.zeros((B, ot.T), np.int32)
    tokens[:, 1:] = rng.choice(V, size=(B, m), p=q)
    u = rng.random((B, ot.T, m + 1)).astype(np.float32)
    al, an, nt, err = _run(M, dtree, logits, draft, tokens, 1.0, u)
    assert err == 0
    emp = np.bincount(_first(al, an, nt, tokens, 1)[:, 0], minlength=V) / B
    assert np.all(np.abs(emp - p) <= 5 * np.sqrt(p * (1 - p) / B))


def test_rejection_bad_token_flag(M):
    ot, dtree = both_trees(M, ("cartesian", (2,), None))
    B, V = 2, 10
    logits = np.zeros((B, ot.T, V), np.float32)
    draft = np.zeros((B, 1, V), np.float32)
    tokens = np.array([[0, 99, 3], [0, 1, 2]], np.int32)  # the first-ranked child of sequence 0 is invalid
    u = np.full((B, ot.T, 3), 0.99, np.float32)
    al, an, nt, err = _run(M, dtree, logits, draft, tokens, 1.0, u)
    assert err & 1
