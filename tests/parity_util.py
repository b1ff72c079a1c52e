"""Shared helpers for the GPU parity tests: host<->device marshalling, trees
for both sides, and token planting done with the oracle's logits."""
import math

import numpy as np
import torch

from medusa_tree_speculative_gb300 import synth


def to_dev(a: np.ndarray, dt: str = None) -> torch.Tensor:
    """numpy -> cuda tensor; uint16 arrays are bf16 bits."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_double(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return synth.bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def tree_paths(spec):
    """spec: ('cartesian', s, max_nodes) or ('greedy', K, R, budget) ->
    (paths, path_len, max_depth) built by the oracle."""
    import oracle

    if spec[0] == "cartesian":
        s, n = spec[1], spec[2]
        if n is None:
            n = sum(math.prod(s[:k]) for k in range(1, len(s) + 1))
        p, l = oracle.tree_cartesian(list(s), n)
        return p, l, len(s)
    K, R, budget = spec[1], spec[2], spec[3]
    p, l = oracle.tree_greedy(synth.accuracy_table(K, R), budget)
    return p, l, K


def both_trees(M, spec):
    import oracle

    p, l, K = tree_paths(spec)
    ot = oracle.tree_compile(p, l, K)
    dt = M.DeviceTree(M.medusa_tree_compile(p, l, K))
    assert dt.T == ot.T
    return ot, dt


def ancestors(parent, n):
    out = []
    while n >= 0:
        out.append(int(n))
        n = int(parent[n]) if n > 0 else -1
    return out[::-1]


def plant_tokens(ot, logits64: np.ndarray, node: int, V: int, rng) -> np.ndarray:
    """Tokens for one sequence: along root->node each token is the argmax of
    its parent's row (double logits from the oracle); every other node gets a
    token that is not its parent's argmax."""
    T = ot.T
    am = np.argmax(logits64, axis=1)
    tok = np.zeros(T, np.int32)
    path = set(ancestors(ot.parent, node))
    for c in range(1, T):
        p = ot.parent[c]
        if c in path:
            tok[c] = am[p]
        else:
            t = int(rng.integers(0, V))
            tok[c] = t if t != am[p] else (t + 1) % V
    tok[0] = int(rng.integers(0, V))
    return tok


def row_gaps(logits64: np.ndarray) -> np.ndarray:
    s = np.sort(logits64, axis=-1)
    return s[..., -1] - s[..., -2]


def gpu_topk_matches_oracle(z_gpu: np.ndarray, topk_gpu: np.ndarray, s: int) -> bool:
    """The oracle's top-s (value descending, lowest index first among equal
    values) run on the GPU's own float32 logits equals the GPU's top-s."""
    import oracle

    return list(oracle.topk_f32(np.ascontiguousarray(z_gpu, np.float32), s)) == list(topk_gpu[:s])


def check_accept_on_gpu_logits(ot, logits, tokens, mode, tau, eps, delta, got, rel_tol=1e-4):
    """Acceptance parity with the oracle run on the GPU's own float32 logits.

    got: host arrays accept_len [B], accepted_nodes [B,K+1], next_root [B],
    best_node [B], best_logp [B] (typical) from the GPU.

    Greedy decisions are exact comparisons of the same float32 values, so
    every sequence is compared bit for bit.  A typical decision compares
    p-hat(token) with min(eps, delta exp(-H)); the GPU forms both in float32
    (relative error of order 1e-5 at V = 32000: p-hat and exp(-H) are
    exponentials of log-space quantities with absolute errors near 1e-5), the
    oracle in double.  A decision whose oracle margin |p-hat - threshold|
    exceeds `rel_tol` times the larger of the two cannot change between them;
    neither can the tie-break between accepted nodes of equal depth when their
    summed log-probabilities differ by more than 1e-4.  (p-hat itself is the
    oracle's margin with eps = 0, where the threshold is 0.)  Sequences with a
    closer decision on a reachable node are checked for validity instead
    (every node of the GPU's path passes up to the margin, and its depth lies
    between what certainly passes and what may pass).  Returns the number of
    sequences compared bit for bit."""
    import oracle

    logits = np.ascontiguousarray(logits, np.float32)
    tokens = np.ascontiguousarray(tokens, np.int32)
    B, T, _ = logits.shape
    r = oracle.accept(logits, tokens, ot, mode, tau, eps, delta)
    if mode == 1:
        p_hat = oracle.accept(logits, tokens, ot, mode, tau, 0.0, delta)["node_margin"]
        tol = rel_tol * np.maximum(p_hat, p_hat - r["node_margin"])
    else:
        tol = np.zeros((B, T))
    exact = 0
    for b in range(B):
        mg = r["node_margin"][b]
        sure = np.zeros(T, bool)
        maybe = np.zeros(T, bool)
        sure[0] = maybe[0] = True
        for c in range(1, T):
            p = ot.parent[c]
            sure[c] = sure[p] and mg[c] > tol[b, c]
            maybe[c] = maybe[p] and mg[c] > -tol[b, c]
        clear = np.array_equal(sure, maybe)
        if clear and mode == 1:
            lp = r["node_logp"][b]
            dmax = ot.depth[np.nonzero(sure)[0]].max()
            top = np.sort(lp[(ot.depth == dmax) & sure])[::-1]
            clear = len(top) < 2 or top[0] - top[1] > 1e-4
        if clear:
            assert got["accept_len"][b] == r["accept_len"][b], b
            assert np.array_equal(got["accepted_nodes"][b], r["accepted_nodes"][b]), b
            assert got["next_root"][b] == r["next_root"][b], b
            assert got["best_node"][b] == r["best_node"][b], b
            if mode == 1:
                assert abs(float(got["best_logp"][b]) - r["best_logp"][b]) <= 1e-4 * max(1.0, abs(r["best_logp"][b]))
            exact += 1
        else:
            bn = int(got["best_node"][b])
            assert maybe[bn] and got["accept_len"][b] == ot.depth[bn]
            assert ot.depth[np.nonzero(sure)[0]].max() <= ot.depth[bn] <= ot.depth[np.nonzero(maybe)[0]].max()
            path = ancestors(ot.parent, bn)
            an = got["accepted_nodes"][b]
            assert list(an[:len(path)]) == path and np.all(an[len(path):] == -1)
            assert got["next_root"][b] == oracle.topk_f32(logits[b, bn], 1)[0]
    return exact
