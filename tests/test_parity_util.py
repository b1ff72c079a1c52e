"""The parity helpers that check GPU results with the oracle (CPU only):
check_accept_on_gpu_logits accepts the oracle's own outputs, rejects a
planted mistake on a clear decision, and falls back to validity only for a
typical decision within rounding of its threshold; gpu_topk_matches_oracle
follows the lowest-index rule on equal values."""
import numpy as np
import pytest

import oracle
from parity_util import check_accept_on_gpu_logits, gpu_topk_matches_oracle, tree_paths


def _tree():
    p, l, K = tree_paths(("cartesian", (3, 2, 2), None))
    return oracle.tree_compile(p, l, K)


def _inputs(ot, B, V, seed):
    rng = np.random.default_rng(seed)
    logits = (rng.standard_normal((B, ot.T, V)) * 2).astype(np.float32)
    tokens = rng.integers(0, V, (B, ot.T)).astype(np.int32)
    for b in range(B):  # a deep accepted path per sequence
        n = int(np.nonzero(ot.depth == 3)[0][b % 4])
        while n > 0:
            p = int(ot.parent[n])
            tokens[b, n] = int(np.argmax(logits[b, p]))
            n = p
    return logits, tokens


def _oracle_outputs(ot, logits, tokens, mode):
    r = oracle.accept(logits, tokens, ot, mode, 0.7, 0.09, 0.3)
    return {k: r[k].copy() for k in ("accept_len", "accepted_nodes", "next_root", "best_node", "best_logp")}


@pytest.mark.parametrize("mode", [0, 1])
def test_accept_check_passes_the_oracle_and_catches_a_mistake(orc, mode):
    ot = _tree()
    logits, tokens = _inputs(ot, 4, 50, 3)
    got = _oracle_outputs(ot, logits, tokens, mode)
    assert check_accept_on_gpu_logits(ot, logits, tokens, mode, 0.7, 0.09, 0.3, got) == 4
    bad = {k: v.copy() for k, v in got.items()}
    bad["next_root"][1] = (bad["next_root"][1] + 1) % 50
    with pytest.raises(AssertionError):
        check_accept_on_gpu_logits(ot, logits, tokens, mode, 0.7, 0.09, 0.3, bad)
    bad = {k: v.copy() for k, v in got.items()}
    bad["accept_len"][2] -= 1
    with pytest.raises(AssertionError):
        check_accept_on_gpu_logits(ot, logits, tokens, mode, 0.7, 0.09, 0.3, bad)


def test_accept_check_validity_fallback_near_threshold(orc):
    """One typical decision sits on its threshold (delta chosen so that
    delta exp(-H) equals that token's p-hat, eps above it): both outcomes
    are accepted as valid, a clear mistake elsewhere is not."""
    ot = _tree()
    logits, tokens = _inputs(ot, 1, 50, 5)
    c = int(np.nonzero(ot.depth == 1)[0][0])
    z = logits[0, 0].astype(np.float64) / 0.7
    p_hat = np.exp(z - z.max()) / np.exp(z - z.max()).sum()
    H = -(p_hat * np.log(p_hat)).sum()
    tokens[0, c] = int(np.argsort(p_hat)[-2])       # the second most likely token at the root
    delta = float(p_hat[tokens[0, c]] * np.exp(H))  # threshold = p-hat of that token
    keys = ("accept_len", "accepted_nodes", "next_root", "best_node", "best_logp")
    outs = [oracle.accept(logits, tokens, ot, 1, 0.7, 0.99, delta * f) for f in (1 - 1e-6, 1 + 1e-6)]
    assert not np.array_equal(outs[0]["node_margin"][0] > 0, outs[1]["node_margin"][0] > 0)
    for r in outs:
        got = {k: r[k].copy() for k in keys}
        assert check_accept_on_gpu_logits(ot, logits, tokens, 1, 0.7, 0.99, delta, got) == 0  # validity only
    got = {k: outs[0][k].copy() for k in keys}
    got["next_root"][0] = (got["next_root"][0] + 1) % 50
    with pytest.raises(AssertionError):
        check_accept_on_gpu_logits(ot, logits, tokens, 1, 0.7, 0.99, delta, got)


def test_topk_check_lowest_index_on_ties(orc):
    z = np.array([0.5, 2.0, 2.0, -1.0, 2.0], np.float32)
    assert gpu_topk_matches_oracle(z, np.array([1, 2, 4]), 3)
    assert not gpu_topk_matches_oracle(z, np.array([2, 1, 4]), 3)
