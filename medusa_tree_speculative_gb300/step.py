"""One Medusa verify step on one GPU: device buffers and the order of the six
library calls.  Plumbing only: every step of the method runs in libmedusa.

Call order (decoding-step box of the Medusa paper digest, steps 3-6 then 1-2
for the next step):
  main chain: medusa_lm_head_verify -> medusa_accept -> heads (->
  medusa_build_candidates); medusa_tree_attn and then medusa_kv_compact either
  on the same stream or on a forked branch that joins at the end.
  heads = medusa_heads_topk_candidates on the accepted node ("fused": the
  heads' last CTA also fills the next candidates), or ("split")
  medusa_heads_hidden over every tree row -- forked after the LM head so that
  it runs beside the acceptance -- then medusa_heads_logits_topk on the
  accepted node's row, or ("joint", bf16) medusa_lm_head_verify_heads_hidden
  in place of the LM head call (logits and every row's u in one pass) and
  then medusa_heads_logits_topk.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import medusa as M

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def host_to_torch(a: np.ndarray, dt: str) -> torch.Tensor:
    """numpy (float32, or bf16 bits as uint16) -> CPU torch tensor of dtype dt."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    t = torch.from_numpy(a)
    return t if dt == "f32" else t.to(torch.bfloat16)


def tc_key_splits(B: int, H: int, T: int, max_prefix: int, sms: int) -> int:
    """Key split for medusa_tree_attn_tc: the largest of 8, 4, 2 that keeps
    the grid (splits x heads x sequences x 128-row blocks, one CTA per SM)
    within `sms` SMs and gives every CTA at least one 128-key tile; else 1.
    On its own the attention may take every SM; in the step it runs beside
    the LM head and gets the SMs the LM head leaves free."""
    ctas = B * H * -(-T // 128)
    tiles = -(-(max_prefix + T) // 128)
    return next(c for c in (8, 4, 2, 1) if c == 1 or (c * ctas <= sms and c <= tiles))


def build_tree(w: dict) -> M.HostTree:
    """The workload's candidate tree via the library's host helpers."""
    kind = w["tree"][0]
    if kind == "cartesian":
        s, max_nodes = w["tree"][1], w["tree"][2]
        n = max_nodes if max_nodes is not None else sum(math.prod(s[:k]) for k in range(1, len(s) + 1))
        paths, plen = M.medusa_tree_cartesian(list(s), n)
        return M.medusa_tree_compile(paths, plen, len(s))
    budget, R = w["tree"][1], w["tree"][2]
    from .synth import accuracy_table

    paths, plen = M.medusa_tree_greedy(accuracy_table(w["K"], R), budget)
    return M.medusa_tree_compile(paths, plen, w["K"])


class VerifyStep:
    """Owns the outputs and scratch of one verify step for fixed shapes."""

    def __init__(self, w: dict, weights: dict, tree: M.DeviceTree, max_prefix: int, device="cuda",
                 heads: str = "fused", accept: str = "separate", write_logits: bool = True,
                 attn_order: str = "after_lm", attn_splits="auto"):
        self.w, self.tree, self.max_prefix = w, tree, max_prefix
        # attention on the forked branch: enqueued before the LM head ("first"),
        # right after it ("after_lm": its CTAs then take the SMs the LM head
        # leaves idle instead of holding the LM head back), or after the
        # acceptance ("after_accept": beside the heads, whose rows are handed
        # out at run time; "after_heads": forked there but enqueued after the
        # heads' kernels), with the library's default key split (None), 1, 2,
        # 4, 8 CTAs per head, or "tc" (medusa_tree_attn_tc: bf16, Dh 128;
        # "tc1" .. "tc8" name its key split, "tc" takes the largest that keeps
        # the grid within the SMs the LM head leaves free, see tc_key_splits);
        # "auto": "tc" for bf16 with Dh 128, else 4 for bf16.  (At the
        # 7B/13B/33B shapes the heads alone outnumber the free SMs, so this is
        # one CTA per head, the fastest step measured at L = 1024 and 4096.)
        if attn_order not in ("first", "after_lm", "after_accept", "after_heads"):
            raise ValueError(f"attn_order {attn_order!r}")
        if attn_splits == "auto":
            attn_splits = ("tc" if w["Dh"] == 128 else 4) if w["dtype"] == "bf16" else None
        B, H, Dh, d, V, K = w["B"], w["H"], w["Dh"], w["d"], w["V"], w["K"]
        T = tree.T
        self.tc_splits = None
        if isinstance(attn_splits, str) and attn_splits.startswith("tc"):
            if attn_splits[2:]:
                self.tc_splits = int(attn_splits[2:])
            else:
                sms = torch.cuda.get_device_properties(device).multi_processor_count if torch.cuda.is_available() else 152
                free = sms
                if attn_order in ("first", "after_lm"):  # it runs beside the LM head
                    free = max(0, sms - M.medusa_lm_head_ctas(B * T, V))
                self.tc_splits = tc_key_splits(B, H, T, max_prefix, free)
            if self.tc_splits not in (1, 2, 4, 8):
                raise ValueError(f"attn_splits {attn_splits!r}")
            attn_splits = "tc"
        self.attn_order, self.attn_splits = attn_order, attn_splits
        self.B, self.T = B, T
        dt = TORCH_DT[w["dtype"]]
        self.w_lm, self.w1, self.b1, self.w2 = weights["w_lm"], weights["w1"], weights.get("b1"), weights["w2"]
        # bf16: the vocabulary matrix is kept resident in the 128 x 64 tile
        # layout the tensor-core LM head streams fastest (written once here)
        self.w_layout = M.W_TILES if w["dtype"] == "bf16" else M.W_ROWS
        self.w_lm_run = M.medusa_lm_head_tile(self.w_lm) if self.w_layout == M.W_TILES else self.w_lm
        # heads that feed a tree level run; the others are skipped (s_k = 0)
        self.s_heads = [tree.s[k] if k < tree.K else 0 for k in range(K)]
        self.s_max = max(1, max(self.s_heads))
        self.mode = 1 if w["mode"] == "typical" else 0
        self.temperature = float(w.get("temperature", 1.0))
        self.eps, self.delta = float(w.get("eps", 0.09)), float(w.get("delta", 0.3))
        self.rope_theta = float(w.get("rope_theta", 10000.0))
        self.scale = 1.0 / math.sqrt(Dh)
        i32 = dict(dtype=torch.int32, device=device)
        self.out = torch.empty((B, T, H, Dh), dtype=dt, device=device)
        self.logits = torch.empty((B, T, V), dtype=torch.float32, device=device)
        # the step's integer results side by side in one buffer, so that a
        # caller reads them back with a single copy (self.results)
        Kp = tree.K + 1
        self.results = torch.zeros(B * (3 + Kp + T), **i32)
        r = self.results
        self.accept_len = r[0:B]
        self.next_root = r[B:2 * B]
        self.best_node = r[2 * B:3 * B]
        self.accepted_nodes = r[3 * B:3 * B + B * Kp].view(B, Kp)
        self.best_logp = torch.zeros(B, dtype=torch.float32, device=device)
        self.src_slots = torch.zeros((B, tree.K + 1), **i32)
        self.head_logits = torch.zeros((B, K, V), dtype=torch.float32, device=device)
        self.topk = torch.zeros((B, K, self.s_max), **i32)
        self.next_tokens = r[3 * B + B * Kp:].view(B, T)
        self.err = torch.zeros(1, **i32)

        def ws(n):
            return torch.empty(max(int(n), 256), dtype=torch.uint8, device=device)

        # accept="fused" (bf16): the LM head's epilogue writes per-group row
        # statistics that medusa_accept_stats merges; greedy steps may then skip
        # writing the logits (write_logits=False)
        self.accept = accept if w["dtype"] == "bf16" else "separate"
        self.write_logits = write_logits or self.mode == 1 or self.accept != "fused"
        if self.accept == "fused":
            self.stat_groups = M.medusa_lm_head_stat_groups(B * T, V)
            self.stats = torch.zeros((self.stat_groups, B * T, 4), dtype=torch.float32, device=device)
        self.ws_attn = ws(M.medusa_tree_attn_workspace_size(B, H, Dh, T, max_prefix))
        # the acceptance keeps per-sequence counters in its workspace: zero-filled once
        self.ws_accept = torch.zeros(max(256, M.medusa_accept_workspace_size(B, T)), dtype=torch.uint8,
                                     device=device)
        # the heads' workspace holds their row counters: zero-filled once, each call leaves them ready
        self.ws_heads = torch.zeros(max(256, M.medusa_heads_topk_workspace_size(B, K, d, V, self.s_max)),
                                    dtype=torch.uint8, device=device)
        # split heads: W1 over every tree row (tile layout for bf16), u for all rows,
        # and the W2 pass's arrival counters (zero once; each call leaves them zero)
        if heads not in ("fused", "split", "joint"):
            raise ValueError(f"heads {heads!r}")
        if heads == "joint" and (w["dtype"] != "bf16" or B * T > 256):
            raise ValueError("heads='joint' needs bf16 and at most 256 tree rows")
        if heads == "joint":
            self.accept = "separate"  # the joint launch has no statistics epilogue
            self.write_logits = True
        self.heads = heads
        if heads in ("split", "joint"):
            self.w1_layout = M.W_TILES if w["dtype"] == "bf16" else M.W_ROWS
            self.w1_run = (M.medusa_lm_head_tile(self.w1.reshape(K * d, d)) if self.w1_layout == M.W_TILES
                           else self.w1)
            self.u_all = torch.zeros((B * T, K, d), dtype=dt, device=device)
            self.ws_w2 = torch.zeros(max(256, M.medusa_heads_logits_topk_workspace_size(B, K, V, self.s_max)),
                                     dtype=torch.uint8, device=device)

    def run(self, x: dict, stream=None, side_stream=None, heads_stream=None, append=None):
        """x: device tensors q, k_new, v_new, hidden, tokens, k_cache, v_cache,
        seq_start, prefix_len, seq_cap.  Updates the cache and prefix_len.

        One stream: tree attention, LM head, acceptance, heads, candidates,
        KV compaction.  With `side_stream`: the chain LM head -> acceptance ->
        heads -> candidates stays on `stream` while the tree attention and
        then the KV compaction (which needs the acceptance result) run on a
        forked branch that joins `stream` at the end.  `append` = (out,
        out_len): the step's root and accepted tokens are appended there right
        after the acceptance (so x["tokens"] may be the buffer that
        medusa_build_candidates refills at the end of the step)."""
        import torch

        main = stream if stream is not None else torch.cuda.current_stream()
        side = side_stream if side_stream is not None else main
        if side is not main and self.attn_order not in ("after_accept", "after_heads"):
            side.wait_stream(main)

        def attention():
            self.attention(x, side)

        if self.attn_order == "first":
            attention()
        if self.heads == "joint":
            M.medusa_lm_head_verify_heads_hidden(x["hidden"], self.w_lm_run, self.logits.shape[-1], self.logits,
                                                 self.w1_run, self.b1, self.s_heads, self.u_all, self.err, main,
                                                 layout=self.w_layout, w1_layout=self.w1_layout)
        elif self.accept == "fused":
            M.medusa_lm_head_verify_stats(x["hidden"], self.w_lm_run, self.logits if self.write_logits else None,
                                          self.stats, self.mode, self.temperature, self.logits.shape[-1], self.err,
                                          main, layout=self.w_layout)
        else:
            M.medusa_lm_head_verify(x["hidden"], self.w_lm_run, self.logits, None, self.err, main,
                                    layout=self.w_layout)
        if self.attn_order == "after_lm":
            attention()
        hs = heads_stream if heads_stream is not None else main
        if self.heads == "split":
            if hs is not main:
                hs.wait_stream(main)  # after the LM head: beside the acceptance
            M.medusa_heads_hidden(x["hidden"], self.w1_run, self.b1, self.s_heads, self.u_all, self.err, hs,
                                  layout=self.w1_layout)
        if self.accept == "fused":
            M.medusa_accept_stats(self.stats, self.stat_groups, self.logits if self.write_logits else None,
                                  x["tokens"], self.tree, self.mode, self.temperature, self.eps, self.delta,
                                  self.logits.shape[-1], self.accept_len, self.accepted_nodes, self.next_root,
                                  self.best_node, self.best_logp, self.err, main)
        else:
            M.medusa_accept(self.logits, x["tokens"], self.tree, self.mode, self.temperature, self.eps,
                            self.delta, self.accept_len, self.accepted_nodes, self.next_root, self.best_node,
                            self.best_logp, self.ws_accept, self.err, main)
        if append is not None:  # box step 6: the root and the accepted tokens to the output
            M.medusa_append_tokens(x["tokens"], self.accepted_nodes, self.accept_len, append[0], append[1],
                                   self.err, main)
        if side is not main:
            side.wait_stream(main)  # compaction needs the accepted path

        def compaction():
            M.medusa_kv_compact(x["k_cache"], x["v_cache"], x["seq_start"], x["prefix_len"],
                                self.accepted_nodes, self.accept_len, self.tree.K, self.tree.T, self.src_slots,
                                self.err, side)

        if self.attn_order == "after_accept":
            attention()
        if self.attn_order != "after_heads":
            compaction()
        if self.heads in ("split", "joint"):
            if hs is not main and self.heads == "split":
                main.wait_stream(hs)
            M.medusa_heads_logits_topk(self.u_all, self.T, self.best_node, self.w2, self.s_heads, self.head_logits,
                                       self.topk, self.ws_w2, self.err, main)
            M.medusa_build_candidates(self.next_root, self.topk, self.tree, self.next_tokens, main)
        else:  # the heads' last CTA also fills the next step's candidates
            M.medusa_heads_topk_candidates(x["hidden"], self.best_node, self.w1, self.b1, self.w2, self.s_heads,
                                           self.head_logits, self.topk, self.ws_heads, self.next_root, self.tree,
                                           self.next_tokens, self.err, main)
        if self.attn_order == "after_heads":  # forked after the acceptance, enqueued after the heads' launches
            attention()
            compaction()
        if side is not main:
            main.wait_stream(side)

    def attention(self, x: dict, stream):
        """The step's tree attention (box step 1) on `stream`."""
        if self.attn_splits == "tc":
            M.medusa_tree_attn_tc(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["seq_start"],
                                  x["prefix_len"], x["seq_cap"], self.tree, self.max_prefix, self.rope_theta,
                                  self.scale, self.out, self.err, stream, key_splits=self.tc_splits)
        else:
            M.medusa_tree_attn(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["seq_start"],
                               x["prefix_len"], x["seq_cap"], self.tree, self.max_prefix, self.rope_theta,
                               self.scale, self.out, self.ws_attn, self.err, stream, key_splits=self.attn_splits)

    @property
    def launches_per_step(self) -> int:
        """Kernels one run() launches: attention 1 (2 for f32), LM head 1,
        acceptance 1, compaction 1, heads 2 with the candidate fill ("fused"),
        or heads 2 ("split"; 1 "joint": W1 runs in the LM head's launch) and
        candidates 1."""
        heads = {"fused": 2, "split": 3, "joint": 2}[self.heads]
        return (1 if self.w["dtype"] == "bf16" else 2) + 1 + 1 + 1 + heads
