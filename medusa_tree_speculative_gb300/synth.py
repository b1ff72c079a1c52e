"""Seeded synthetic inputs shared by the GPU path and the CPU oracle.

This module holds none of the method's arithmetic: it only draws random
numbers and lays them out.  Every tensor is produced on the host from numpy's
PCG64 generator, keyed by (seed, tensor tag, chunk index), so the values do not
depend on the machine or on the number of threads used to draw them.

bfloat16 tensors are returned as their raw bits (``numpy.uint16``), rounded
from the float32 draw to nearest-even, so both sides read identical bits.
"""
from __future__ import annotations

import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import workloads as _wl

_CHUNK = 1 << 22
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        import os
        _POOL = ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4))
    return _POOL


def _seed_seq(seed: int, tag: str, chunk: int) -> np.random.SeedSequence:
    return np.random.SeedSequence([int(seed), zlib.crc32(tag.encode()), int(chunk)])


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    out = ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal(seed: int, tag: str, shape, std: float = 1.0, dtype: str = "f32") -> np.ndarray:
    """N(0, std^2) samples of the given shape; dtype 'f32' or 'bf16' (bits)."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, np.uint16 if dtype == "bf16" else np.float32)
    starts = list(range(0, n, _CHUNK))

    def fill(ci):
        lo = starts[ci]
        hi = min(n, lo + _CHUNK)
        g = np.random.Generator(np.random.PCG64(_seed_seq(seed, tag, ci)))
        x = g.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = f32_to_bf16_bits(x) if dtype == "bf16" else x

    if len(starts) <= 1:
        for ci in range(len(starts)):
            fill(ci)
    else:
        list(_pool().map(fill, range(len(starts))))
    return out.reshape(shape)


def integers(seed: int, tag: str, shape, lo: int, hi: int) -> np.ndarray:
    """Uniform int32 in [lo, hi)."""
    g = np.random.Generator(np.random.PCG64(_seed_seq(seed, tag, 0)))
    return g.integers(lo, hi, size=shape, dtype=np.int64).astype(np.int32)


def accuracy_table(K: int, R: int) -> np.ndarray:
    """Synthetic per-head top-i accuracy a_k^(i) = 0.6 * 0.7^(k-1) * 0.5^(i-1)."""
    k = np.arange(1, K + 1, dtype=np.float64)[:, None]
    i = np.arange(1, R + 1, dtype=np.float64)[None, :]
    return 0.6 * 0.7 ** (k - 1) * 0.5 ** (i - 1)


def prefix_lengths(w: dict, seed: int) -> np.ndarray:
    L = w["L"]
    if isinstance(L, tuple) and len(L) and L[0] == "uniform":
        return integers(seed, "prefix_len", (w["B"],), L[1], L[2] + 1)
    return np.array(L, np.int32)


def _std(spec, d):
    return 1.0 / np.sqrt(d) if spec == "inv_sqrt_d" else float(spec)


def make_weights(w: dict, seed: int = 0) -> dict:
    """W_lm [V,d], W1 [K,d,d], W2 [K,V,d] in the workload's element type."""
    d, V, K, dt = w["d"], w["V"], w["K"], w["dtype"]
    lm_std = _std(w["lm_std"], d)
    out = {}
    if w.get("w2") == "lm_plus_noise":
        # W2^(k) = W_lm + noise_k: each head starts as a copy of the LM head
        # plus a small perturbation (the heads' initialisation, perturbed).
        lm = normal(seed, "w_lm", (V, d), lm_std, "f32")
        w2 = np.empty((K, V, d), np.float32)
        for k in range(K):
            w2[k] = lm + normal(seed, f"w2_noise_{k}", (V, d), w["w2_noise_std"], "f32")
        if dt == "bf16":
            lm = f32_to_bf16_bits(lm)
            w2 = f32_to_bf16_bits(w2)
        out["w_lm"], out["w2"] = lm, w2
    else:
        out["w_lm"] = normal(seed, "w_lm", (V, d), lm_std, dt)
        w2 = np.empty((K, V, d), np.uint16 if dt == "bf16" else np.float32)
        for k in range(K):
            w2[k] = normal(seed, f"w2_{k}", (V, d), lm_std, dt)
        out["w2"] = w2
    w1 = np.empty((K, d, d), np.uint16 if dt == "bf16" else np.float32)
    for k in range(K):
        w1[k] = normal(seed, f"w1_{k}", (d, d), _std(w["w1_std"], d), dt)
    out["w1"] = w1
    out["b1"] = None
    return out


def make_step(w: dict, T: int, seed: int = 0) -> dict:
    """Per-step activations: q/k_new/v_new [B,T,H,Dh], hidden [B,T,d], a KV
    cache with a random rotated prefix per sequence, and natural tokens."""
    B, H, Dh, d, V, dt = w["B"], w["H"], w["Dh"], w["d"], w["V"], w["dtype"]
    L = prefix_lengths(w, seed)
    cap = L.astype(np.int64) + T
    seq_start = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)
    tokens_total = int(cap.sum())
    edt = np.uint16 if dt == "bf16" else np.float32
    k_cache = np.zeros((tokens_total, H, Dh), edt)
    v_cache = np.zeros((tokens_total, H, Dh), edt)
    for b in range(B):
        st, l = int(seq_start[b]), int(L[b])
        k_cache[st:st + l] = normal(seed, f"k_prefix_{b}", (l, H, Dh), 1.0, dt)
        v_cache[st:st + l] = normal(seed, f"v_prefix_{b}", (l, H, Dh), 1.0, dt)
    return dict(
        q=normal(seed, "q", (B, T, H, Dh), 1.0, dt),
        k_new=normal(seed, "k_new", (B, T, H, Dh), 1.0, dt),
        v_new=normal(seed, "v_new", (B, T, H, Dh), 1.0, dt),
        hidden=normal(seed, "hidden", (B, T, d), 1.0, dt),
        k_cache=k_cache, v_cache=v_cache,
        seq_start=seq_start, prefix_len=L.astype(np.int32), seq_cap=cap,
        tokens=integers(seed, "tokens", (B, T), 0, V),
    )


def workload(name: str) -> dict:
    return _wl.get(name)
