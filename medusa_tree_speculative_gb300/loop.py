"""A closed decode loop on the device: Medusa verify steps chained so that
each step's candidate tokens come from the previous step (decoding-step box of
the Medusa paper digest, steps 1-6, repeated), around a stand-in backbone.

The stand-in has no counterpart in the paper.  It replaces the transformer
forward over the tree by an embedding lookup, so the hidden state of a tree
token t is row t of a table E (rows of norm about 1), and the attention takes
its q, k and v from the same rows.  Its weights make the model continue a
fixed chain: the LM head row of token v is E[prev(v)], so the greedy next
token of t is next(t) = (a t + c) mod V; Medusa head k (0-based) predicts the
token k + 2 places ahead, next^(k+2)(t), from rows E[prev^(k+2)(v)] plus
Gaussian noise of standard deviation sigma_k in every weight (its score
noise), so its top-s holds the right token only part of the time; W1 = 0
(the heads' initialisation in Method 1), so the head input is h itself.

Greedy Medusa decoding is lossless, so the tokens the loop emits must be the
stand-in model's plain greedy continuation next(x0), next(next(x0)), ...,
which is what the tests check against the oracle.  Tokens per step then
measure how far the heads' top-s trees reach.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import medusa as M
from . import step as S

CHAIN_A, CHAIN_C = 7919, 12345  # next(t) = (A t + C) mod V; A is prime to every V used here


def chain_next(t: np.ndarray, V: int, n: int = 1) -> np.ndarray:
    t = np.asarray(t, np.int64)
    for _ in range(n):
        t = (CHAIN_A * t + CHAIN_C) % V
    return t


def chain_prev(v: np.ndarray, V: int, n: int = 1) -> np.ndarray:
    inv = pow(CHAIN_A, -1, V)
    v = np.asarray(v, np.int64)
    for _ in range(n):
        v = (inv * (v - CHAIN_C)) % V
    return v


class StandInModel:
    """Embedding table and weights of the stand-in (on the device)."""

    def __init__(self, w: dict, seed: int = 0, sigma=(0.20, 0.23, 0.26, 0.29, 0.32), device="cuda"):
        V, d, K = w["V"], w["d"], w["K"]
        assert math.gcd(CHAIN_A, V) == 1
        dt = S.TORCH_DT[w["dtype"]]
        g = torch.Generator(device=device).manual_seed(seed)
        E = torch.randn(V, d, generator=g, device=device) / math.sqrt(d)
        idx = np.arange(V)
        self.E = E.to(dt).contiguous()
        self.w_lm = E[torch.from_numpy(chain_prev(idx, V)).to(device)].to(dt).contiguous()
        self.w1 = torch.zeros(K, d, d, dtype=dt, device=device)
        w2 = torch.empty(K, V, d, dtype=dt, device=device)
        for k in range(K):
            rows = torch.from_numpy(chain_prev(idx, V, k + 2)).to(device)
            noise = torch.randn(V, d, generator=g, device=device) * sigma[min(k, len(sigma) - 1)]
            w2[k] = (E[rows] + noise).to(dt)
        self.w2 = w2
        self.V, self.d = V, d

    def weights(self):
        return {"w_lm": self.w_lm, "w1": self.w1, "w2": self.w2, "b1": None}


class DecodeLoop:
    """n_steps verify steps on the device, each fed by the previous one."""

    def __init__(self, w: dict, model: StandInModel, tree: M.DeviceTree, n_steps: int, L0: int, x0,
                 device="cuda", heads: str = "fused", seed: int = 0):
        B, H, Dh, d, K = w["B"], w["H"], w["Dh"], w["d"], w["K"]
        assert H * Dh == d, "the stand-in takes q, k and v from the hidden rows"
        T = tree.T
        dt = S.TORCH_DT[w["dtype"]]
        self.w, self.model, self.tree, self.n_steps = w, model, tree, n_steps
        self.B, self.T, self.K = B, T, K
        cap = L0 + n_steps * (tree.K + 1) + T + 1
        g = torch.Generator(device=device).manual_seed(seed + 1)
        kc = torch.zeros(B * cap, H, Dh, dtype=dt, device=device)
        vc = torch.zeros_like(kc)
        for b in range(B):  # a random (already rotated) prefix
            kc[b * cap:b * cap + L0] = torch.randn(L0, H, Dh, generator=g, device=device).to(dt)
            vc[b * cap:b * cap + L0] = torch.randn(L0, H, Dh, generator=g, device=device).to(dt)
        self.hidden = torch.zeros(B, T, d, dtype=dt, device=device)
        qkv = self.hidden.view(B, T, H, Dh)
        self.st = S.VerifyStep(w, model.weights(), tree, max_prefix=cap - T, device=device, heads=heads)
        self.x = {"q": qkv, "k_new": qkv, "v_new": qkv, "hidden": self.hidden, "tokens": self.st.next_tokens,
                  "k_cache": kc, "v_cache": vc,
                  "seq_start": torch.arange(B, dtype=torch.int64, device=device) * cap,
                  "prefix_len": torch.full((B,), L0, dtype=torch.int32, device=device),
                  "seq_cap": torch.full((B,), cap, dtype=torch.int64, device=device)}
        self.out = torch.zeros(B, n_steps * (tree.K + 1) + 1, dtype=torch.int32, device=device)
        self.out_len = torch.zeros(B, dtype=torch.int32, device=device)
        self.x0 = np.asarray(x0, np.int64).reshape(B)
        self._prime()

    def _prime(self):
        """The state before the first step: the root is next(x0) and the tree
        is filled from the heads at x0's hidden state (box steps 1-2)."""
        st, m = self.st, self.model
        B, d = self.B, m.d
        x0 = torch.from_numpy(self.x0.astype(np.int32)).to(self.hidden.device)
        h0 = torch.zeros(B, 1, d, dtype=self.hidden.dtype, device=self.hidden.device)
        M.medusa_standin_embed(x0, m.E, h0, st.err)
        root = torch.from_numpy(chain_next(self.x0, m.V).astype(np.int32)).to(self.hidden.device)
        zero = torch.zeros(B, dtype=torch.int32, device=self.hidden.device)
        M.medusa_heads_topk(h0, zero, m.w1, None, m.w2, st.s_heads, st.head_logits, st.topk, st.ws_heads, st.err)
        M.medusa_build_candidates(root, st.topk, self.tree, st.next_tokens)
        self.out_len.zero_()

    def launches_per_step(self) -> int:
        return 1 + self.st.launches_per_step + 1  # embed, the step, the append

    def step(self, stream=None, side_stream=None, heads_stream=None):
        st = self.st
        main = stream if stream is not None else torch.cuda.current_stream()
        M.medusa_standin_embed(st.next_tokens, self.model.E, self.hidden, st.err, main)
        st.run(self.x, main, side_stream=side_stream, heads_stream=heads_stream, append=(self.out, self.out_len))

    def emitted(self):
        """Per sequence, the tokens emitted so far (host)."""
        n = self.out_len.cpu().numpy()
        o = self.out.cpu().numpy()
        return [o[b, :n[b]] for b in range(self.B)]

    def greedy_reference(self, n_tokens: int):
        """The stand-in model's plain greedy continuation of x0 (host)."""
        out, t = [], self.x0.copy()
        for _ in range(n_tokens):
            t = chain_next(t, self.model.V)
            out.append(t.copy())
        return np.stack(out, axis=1) if out else np.zeros((self.B, 0), np.int64)
