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
