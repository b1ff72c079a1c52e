"""Acceptance statistics fused into the LM head's epilogue
(medusa_lm_head_verify_stats) and the acceptance that merges them
(medusa_accept_stats): the per-group records reproduce each row's argmax,
log-sum-exp and entropy (checked against float64 on the same logits), the
logits come out bit-identical to medusa_lm_head_verify, and the acceptance
matches the oracle's acceptance (the decoding-step box of the Medusa paper
digest, steps 4-5, and its Method item 5) run on the GPU's own logits, and
gives the same outputs as medusa_accept -- also with the logits not written
(greedy)."""
import math

import numpy as np
import pytest
import torch

import oracle
from medusa_tree_speculative_gb300 import synth
from parity_util import ancestors, both_trees, check_accept_on_gpu_logits, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from medusa_tree_speculative_gb300 import build

    build.build()
    from medusa_tree_speculative_gb300 import medusa

    return medusa


def _merge(rec, inv_temp):
    """records [G, rows, 4] (float32 with the index bits in column 1) -> per row
    (argmax, lse, entropy) in float64."""
    v = rec[..., 0].astype(np.float64)
    idx = rec[..., 1].copy().view(np.int32)
    S, A = rec[..., 2].astype(np.float64), rec[..., 3].astype(np.float64)
    best = np.lexsort((idx, -v), axis=0)[0]            # max value, then lowest index
    am = idx[best, np.arange(rec.shape[1])]
    m = v * inv_temp
    M_ = m.max(0)
    e = np.where(S > 0, np.exp(m - M_), 0.0)
    St = (S * e).sum(0)
    At = (e * (A + (m - M_) * S)).sum(0)
    if not (St > 0).all():  # greedy records carry no sums
        return am, None, None
    return am, M_ + np.log(St), np.log(St) - At / St


def _ref_stats(z, inv_temp):
    y = z.astype(np.float64) * inv_temp
    m = y.max(1)
    lse = m + np.log(np.exp(y - m[:, None]).sum(1))
    lp = y - lse[:, None]
    return np.argmax(z, axis=1), lse, -(np.exp(lp) * lp).sum(1)


@pytest.mark.parametrize("rows,d,V", [(15, 256, 1000), (65, 4096, 32000), (130, 512, 333), (65, 256, 40000),
                                      (200, 256, 40000), (300, 256, 5000)])
@pytest.mark.parametrize("mode", [0, 1])
def test_fused_stats_records(M, rows, d, V, mode):
    h = to_dev(synth.normal(51, "h", (rows, d), 1.0, "bf16"))
    w = to_dev(synth.normal(51, "w", (V, d), 1.0 / math.sqrt(d), "bf16"))
    tau = 0.7 if mode == 1 else 1.0
    G = M.medusa_lm_head_stat_groups(rows, V)
    stats = torch.zeros((G, rows, 4), dtype=torch.float32, device="cuda")
    lg = torch.empty((rows, V), dtype=torch.float32, device="cuda")
    ref = torch.empty((rows, V), dtype=torch.float32, device="cuda")
    M.medusa_lm_head_verify_stats(h, w, lg, stats, mode, tau, V)
    M.medusa_lm_head_verify(h, w, ref)
    torch.cuda.synchronize()
    assert torch.equal(lg, ref)
    z = to_host(ref)
    am, lse, ent = _merge(to_host(stats), 1.0 / tau)
    am_r, lse_r, ent_r = _ref_stats(z, 1.0 / tau)
    assert np.array_equal(am, am_r)
    if mode == 1:
        assert np.abs(lse - lse_r).max() <= 1e-4 * np.abs(lse_r).max()
        assert np.abs(ent - ent_r).max() <= 1e-4 * np.abs(ent_r).max() + 1e-5


@pytest.mark.parametrize("mode,write_logits", [(0, True), (0, False), (1, True)])
def test_fused_accept_matches_accept(M, mode, write_logits):
    ot, dtree = both_trees(M, ("greedy", 4, 10, 64))
    B, T, d, V = 2, ot.T, 1024, 32000
    tau, eps, delta = (0.7, 0.09, 0.3) if mode == 1 else (1.0, 0.09, 0.3)
    h = to_dev(synth.normal(53, "h", (B, T, d), 1.0, "bf16"))
    w = to_dev(synth.normal(53, "w", (V, d), 1.0 / math.sqrt(d), "bf16"))
    lg = torch.empty((B, T, V), dtype=torch.float32, device="cuda")
    M.medusa_lm_head_verify(h, w, lg)
    torch.cuda.synchronize()
    z = to_host(lg)
    # tokens: the GPU argmax along one deep path per sequence, something else elsewhere
    tok = np.zeros((B, T), np.int32)
    deep = [n for n in range(T) if ot.depth[n] == 3]
    for b in range(B):
        path = set(ancestors(ot.parent, deep[7 * b + 2]))
        for c in range(1, T):
            a = int(np.argmax(z[b, ot.parent[c]]))
            tok[b, c] = a if c in path else (a + 1 + c) % V
    tk = to_dev(tok)

    def outs():
        i32 = dict(dtype=torch.int32, device="cuda")
        return [torch.zeros(B, **i32), torch.zeros((B, ot.K + 1), **i32), torch.zeros(B, **i32),
                torch.zeros(B, **i32), torch.zeros(B, dtype=torch.float32, device="cuda")]

    o1 = outs()
    ws = torch.zeros(M.medusa_accept_workspace_size(B, T), dtype=torch.uint8, device="cuda")
    M.medusa_accept(lg, tk, dtree, mode, tau, eps, delta, *o1, ws)
    G = M.medusa_lm_head_stat_groups(B * T, V)
    stats = torch.zeros((G, B * T, 4), dtype=torch.float32, device="cuda")
    lg2 = torch.full((B, T, V), float("nan"), dtype=torch.float32, device="cuda")
    M.medusa_lm_head_verify_stats(h, w, lg2 if write_logits else None, stats, mode, tau, V)
    o2 = outs()
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.medusa_accept_stats(stats, G, lg2 if write_logits else None, tk, dtree, mode, tau, eps, delta, V, *o2, e)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    # the oracle decides on the logits the LM head wrote (bit-identical to the
    # ones the fused epilogue reduced: test_fused_stats_records)
    got = dict(zip(("accept_len", "accepted_nodes", "next_root", "best_node", "best_logp"), map(to_host, o2)))
    exact = check_accept_on_gpu_logits(ot, z, tok, mode, tau, eps, delta, got)
    assert exact == B
    for a_, b_ in zip(o1[:4], o2[:4]):
        assert torch.equal(a_, b_)
    if mode == 0:
        assert (to_host(o2[0]) == 3).all()  # the planted paths
    else:
        assert torch.allclose(o1[4], o2[4], rtol=1e-4, atol=1e-4)
    if not write_logits:
        assert torch.isnan(lg2).all()
