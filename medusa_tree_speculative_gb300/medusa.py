"""ctypes binding of libmedusa (include/medusa.h): argument marshalling only.

Every function here has the name of the C entry point it calls and takes torch
tensors (device tensors on the current CUDA device, host tensors or numpy
arrays where the header says "host").  No arithmetic of the method happens in
Python; if the library is missing this module raises on import.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmedusa.so")

MEDUSA_F32, MEDUSA_BF16 = 0, 1
MAX_T, MAX_K, MAX_S, MAX_B = 512, 8, 16, 16
STATUS = {0: "OK", -1: "INVALID", -2: "UNSUPPORTED", -3: "CAPACITY", -4: "WORKSPACE", -5: "CUDA"}
DEVERR = {1: "TOKEN", 2: "NODE", 4: "CAPACITY", 8: "LENGTH", 16: "TIMEOUT"}

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is not built; run `python -m medusa_tree_speculative_gb300.build` "
        "(the CUDA library is required; there is no fallback)")

_lib = C.CDLL(LIB_PATH)


class medusa_tree_t(C.Structure):
    _fields_ = [
        ("parent", C.c_void_p), ("depth", C.c_void_p), ("rank", C.c_void_p),
        ("anc_mask", C.c_void_p), ("T", C.c_int32), ("W", C.c_int32), ("K", C.c_int32),
        ("s", C.c_int32 * MAX_K),
    ]


P, I, F, SZ = C.c_void_p, C.c_int, C.c_float, C.c_size_t
TREE = C.POINTER(medusa_tree_t)

_SIGS = {
    "medusa_last_error": (C.c_char_p, []),
    "medusa_version": (C.c_char_p, []),
    "medusa_tree_compile": (I, [P, P, I, I, P, P, P, P, P, P, P, P]),
    "medusa_tree_cartesian": (I, [P, I, I, P, P]),
    "medusa_tree_greedy": (I, [P, I, I, I, P, P]),
    "medusa_tree_attn_workspace_size": (SZ, [I, I, I, I, I]),
    "medusa_tree_attn": (I, [P, P, P, P, P, P, P, P, TREE, I, I, I, I, F, F, I, P, P, SZ, P, P]),
    "medusa_tree_attn_splits": (I, [P, P, P, P, P, P, P, P, TREE, I, I, I, I, F, F, I, P, P, SZ, I, P, P]),
    "medusa_tree_attn_tc": (I, [P, P, P, P, P, C.c_int64, P, P, P, TREE, I, I, I, I, F, F, I, P, I, P, P]),
    "medusa_copy_from_host": (I, [P, P, SZ, P]),
    "medusa_check_errors": (I, [P, P, I, P]),
    "medusa_lm_head_workspace_size": (SZ, [I, I, I]),
    "medusa_lm_head_tiled_bytes": (SZ, [I, I]),
    "medusa_lm_head_tile": (I, [P, P, I, I, P]),
    "medusa_lm_head_verify": (I, [P, P, P, I, I, I, I, I, P, SZ, P, P]),
    "medusa_accept_workspace_size": (SZ, [I, I]),
    "medusa_accept": (I, [P, P, TREE, I, I, I, F, F, F, P, P, P, P, P, P, SZ, P, P]),
    "medusa_accept_noalloc": (I, [P, P, TREE, I, I, I, F, F, F, P, P, P, P, P, P, P]),
    "medusa_kv_compact": (I, [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P]),
    "medusa_heads_topk_workspace_size": (SZ, [I, I, I, I, I]),
    "medusa_heads_topk": (I, [P, P, I, P, P, P, P, I, I, I, I, I, P, P, I, P, SZ, P, P]),
    "medusa_heads_topk_candidates": (I, [P, P, I, P, P, P, P, I, I, I, I, I, P, P, I, P, SZ, P, TREE, P, P, P]),
    "medusa_build_candidates": (I, [P, P, I, I, TREE, I, P, P]),
    "medusa_heads_hidden": (I, [P, I, P, I, P, P, I, I, I, P, P, P]),
    "medusa_lm_head_verify_heads_hidden": (I, [P, I, I, P, I, I, P, P, I, P, P, I, P, I, P, P]),
    "medusa_append_tokens": (I, [P, P, P, I, I, I, P, P, I, P, P]),
    "medusa_lm_head_stat_groups": (I, [I, I]),
    "medusa_lm_head_ctas": (I, [I, I]),
    "medusa_lm_head_verify_stats": (I, [P, P, P, I, I, I, I, I, I, F, P, SZ, P, P]),
    "medusa_accept_stats": (I, [P, I, P, P, TREE, I, I, I, F, F, F, P, P, P, P, P, P, P]),
    "medusa_accept_rejection_workspace_size": (SZ, [I, I]),
    "medusa_accept_rejection": (I, [P, P, I, P, TREE, I, I, F, P, I, P, P, P, P, SZ, P, P]),
    "medusa_standin_embed": (I, [P, I, P, I, I, I, P, P, P]),
    "medusa_heads_logits_topk_workspace_size": (SZ, [I, I, I, I]),
    "medusa_heads_logits_topk": (I, [P, I, P, P, P, I, I, I, I, I, P, P, I, P, SZ, P, P]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTS = tuple(_SIGS)


class MedusaError(RuntimeError):
    pass


def _check(rc: int, name: str):
    if rc < 0:
        msg = _lib.medusa_last_error().decode(errors="replace")
        raise MedusaError(f"{name} -> {STATUS.get(rc, rc)}: {msg}")
    return rc


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        assert t.flags["C_CONTIGUOUS"]
        return t.ctypes.data
    assert t.is_contiguous(), "libmedusa takes dense row-major tensors"
    return t.data_ptr()


def _dtype(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return MEDUSA_BF16
    if t.dtype == torch.float32:
        return MEDUSA_F32
    raise TypeError(f"libmedusa element type must be bfloat16 or float32, got {t.dtype}")


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def medusa_version() -> str:
    return _lib.medusa_version().decode()


# ------------------------------------------------------------ host trees ---

class HostTree:
    """A compiled tree in host memory (numpy int32 / uint32 arrays)."""

    def __init__(self, parent, depth, rank, anc_mask, s, node_paths, T, K):
        self.parent, self.depth, self.rank = parent, depth, rank
        self.anc_mask, self.s, self.node_paths = anc_mask, s, node_paths
        self.T, self.K, self.W = T, K, (T + 31) // 32


def medusa_tree_compile(paths, path_len, max_depth: int) -> HostTree:
    paths = np.ascontiguousarray(paths, np.int32).reshape(-1, max_depth)
    path_len = np.ascontiguousarray(path_len, np.int32)
    n = len(path_len)
    T = n + 1
    W = (T + 31) // 32
    parent = np.zeros(T, np.int32)
    depth = np.zeros(T, np.int32)
    rank = np.zeros(T, np.int32)
    anc = np.zeros(T * W, np.uint32)
    s = np.zeros(max_depth, np.int32)
    node_paths = np.zeros((T, max_depth), np.int32)
    To, Ko = C.c_int(0), C.c_int(0)
    _check(_lib.medusa_tree_compile(_ptr(paths), _ptr(path_len), n, max_depth, _ptr(parent),
                                    _ptr(depth), _ptr(rank), _ptr(anc), _ptr(s), _ptr(node_paths),
                                    C.addressof(To), C.addressof(Ko)), "medusa_tree_compile")
    return HostTree(parent, depth, rank, anc.reshape(T, W), s, node_paths, To.value, Ko.value)


def medusa_tree_cartesian(s, max_nodes: int):
    s = np.ascontiguousarray(s, np.int32)
    K = len(s)
    paths = np.zeros((max(max_nodes, 1), K), np.int32)
    plen = np.zeros(max(max_nodes, 1), np.int32)
    n = _check(_lib.medusa_tree_cartesian(_ptr(s), K, max_nodes, _ptr(paths), _ptr(plen)),
               "medusa_tree_cartesian")
    return paths[:n].copy(), plen[:n].copy()


def medusa_tree_greedy(acc, budget: int):
    acc = np.ascontiguousarray(acc, np.float64)
    K, R = acc.shape
    paths = np.zeros((max(budget, 1), K), np.int32)
    plen = np.zeros(max(budget, 1), np.int32)
    n = _check(_lib.medusa_tree_greedy(_ptr(acc), K, R, budget, _ptr(paths), _ptr(plen)),
               "medusa_tree_greedy")
    return paths[:n].copy(), plen[:n].copy()


class DeviceTree:
    """A HostTree copied to the GPU, with the medusa_tree_t that points at it."""

    def __init__(self, ht: HostTree, device="cuda"):
        import torch

        self.host = ht
        self.parent = torch.from_numpy(ht.parent).to(device)
        self.depth = torch.from_numpy(ht.depth).to(device)
        self.rank = torch.from_numpy(ht.rank).to(device)
        self.anc_mask = torch.from_numpy(ht.anc_mask.view(np.int32).copy()).to(device)
        self.T, self.K, self.W = ht.T, ht.K, ht.W
        self.struct = medusa_tree_t()
        self.struct.parent = self.parent.data_ptr()
        self.struct.depth = self.depth.data_ptr()
        self.struct.rank = self.rank.data_ptr()
        self.struct.anc_mask = self.anc_mask.data_ptr()
        self.struct.T, self.struct.W, self.struct.K = ht.T, ht.W, ht.K
        for k in range(min(len(ht.s), MAX_K)):
            self.struct.s[k] = int(ht.s[k])

    @property
    def ref(self):
        return C.byref(self.struct)

    @property
    def s(self):
        return [int(self.struct.s[k]) for k in range(self.K)]


# ------------------------------------------------------------ step calls ---

def medusa_tree_attn_workspace_size(B, H, Dh, T, max_prefix) -> int:
    return int(_lib.medusa_tree_attn_workspace_size(B, H, Dh, T, max_prefix))


def medusa_tree_attn_tc(q, k_new, v_new, k_cache, v_cache, seq_start, prefix_len, seq_cap,
                        tree: DeviceTree, max_prefix: int, rope_theta: float, scale: float, out, err=None,
                        stream=None, key_splits=1):
    """Tensor-core tree attention (bf16, Dh 128); k_cache / v_cache [rows][H][Dh]; a cluster of
    key_splits CTAs (1, 2, 4 or 8) shares each (sequence, head, row block)'s key tiles."""
    B, T, H, Dh = q.shape
    _check(_lib.medusa_tree_attn_tc(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                    int(k_cache.shape[0]), _ptr(seq_start), _ptr(prefix_len), _ptr(seq_cap),
                                    tree.ref, B, H, Dh, max_prefix, rope_theta, scale, _dtype(q), _ptr(out),
                                    int(key_splits), _ptr(err), _stream(stream)), "medusa_tree_attn_tc")


def medusa_copy_from_host(dst, src_host, stream=None):
    """dst (device tensor) <- src_host (pinned CPU tensor of the same byte size) by a copy kernel."""
    nb = src_host.numel() * src_host.element_size()
    if dst.numel() * dst.element_size() != nb:
        raise ValueError("medusa_copy_from_host: byte sizes differ")
    _check(_lib.medusa_copy_from_host(_ptr(dst), C.c_void_p(src_host.data_ptr()), nb, _stream(stream)),
           "medusa_copy_from_host")


def medusa_check_errors(err, out, clear: bool = False, stream=None):
    """out (device tensor or pinned CPU tensor, int32, one element) <- the
    device error word err; with clear, err is then reset to 0.  Enqueued on
    the stream, no synchronisation."""
    _check(_lib.medusa_check_errors(_ptr(err), C.c_void_p(out.data_ptr()), 1 if clear else 0, _stream(stream)),
           "medusa_check_errors")


def medusa_tree_attn(q, k_new, v_new, k_cache, v_cache, seq_start, prefix_len, seq_cap,
                     tree: DeviceTree, max_prefix: int, rope_theta: float, scale: float, out,
                     workspace, err=None, stream=None, key_splits=None):
    """key_splits None: medusa_tree_attn; 1, 2, 4 or 8: medusa_tree_attn_splits."""
    B, T, H, Dh = q.shape
    args = (_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(seq_start),
            _ptr(prefix_len), _ptr(seq_cap), tree.ref, B, H, Dh, max_prefix, rope_theta, scale, _dtype(q),
            _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size())
    if key_splits is None:
        _check(_lib.medusa_tree_attn(*args, _ptr(err), _stream(stream)), "medusa_tree_attn")
    else:
        _check(_lib.medusa_tree_attn_splits(*args, int(key_splits), _ptr(err), _stream(stream)),
               "medusa_tree_attn_splits")


def medusa_lm_head_workspace_size(rows, d, V) -> int:
    return int(_lib.medusa_lm_head_workspace_size(rows, d, V))


W_ROWS, W_TILES = 0, 1  # medusa_w_layout


def medusa_lm_head_tiled_bytes(d, V) -> int:
    return int(_lib.medusa_lm_head_tiled_bytes(d, V))


def medusa_lm_head_tile(w_lm, out=None, stream=None):
    """The MEDUSA_W_TILES copy of a bf16 [V][d] matrix (a flat bf16 tensor)."""
    import torch

    V, d = w_lm.shape
    n = medusa_lm_head_tiled_bytes(d, V) // 2
    if out is None:
        out = torch.empty(n, dtype=torch.bfloat16, device=w_lm.device)
    _check(_lib.medusa_lm_head_tile(_ptr(w_lm), _ptr(out), d, V, _stream(stream)), "medusa_lm_head_tile")
    return out


def medusa_lm_head_verify(hidden, w_lm, logits, workspace=None, err=None, stream=None, layout=W_ROWS):
    """logits [rows][V] = hidden [rows][d] @ w_lm^T; V is read from logits."""
    d = hidden.shape[-1]
    rows = hidden.numel() // d
    V = logits.shape[-1]
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.medusa_lm_head_verify(_ptr(hidden), _ptr(w_lm), _ptr(logits), rows, d, V, _dtype(hidden),
                                      layout, _ptr(workspace), nbytes, _ptr(err), _stream(stream)),
           "medusa_lm_head_verify")


def medusa_accept_workspace_size(B, T) -> int:
    return int(_lib.medusa_accept_workspace_size(B, T))


def medusa_accept(logits, tokens, tree: DeviceTree, mode: int, temperature: float, eps: float,
                  delta: float, accept_len, accepted_nodes, next_root, best_node, best_logp, workspace,
                  err=None, stream=None):
    B, T, V = logits.shape
    _check(_lib.medusa_accept(_ptr(logits), _ptr(tokens), tree.ref, B, V, mode, temperature, eps, delta,
                              _ptr(accept_len), _ptr(accepted_nodes), _ptr(next_root), _ptr(best_node),
                              _ptr(best_logp), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _ptr(err), _stream(stream)),
           "medusa_accept")


def medusa_accept_noalloc(logits, tokens, tree: DeviceTree, mode: int, temperature: float, eps: float,
                          delta: float, accept_len, accepted_nodes, next_root, best_node, best_logp, err=None,
                          stream=None):
    """medusa_accept without a workspace: for callers that cannot allocate
    device memory (the library's static scratch is used instead)."""
    B, T, V = logits.shape
    _check(_lib.medusa_accept_noalloc(_ptr(logits), _ptr(tokens), tree.ref, B, V, mode, temperature, eps, delta,
                                      _ptr(accept_len), _ptr(accepted_nodes), _ptr(next_root), _ptr(best_node),
                                      _ptr(best_logp), _ptr(err), _stream(stream)), "medusa_accept_noalloc")


def medusa_kv_compact(k_cache, v_cache, seq_start, prefix_len, accepted_nodes, accept_len, Kmax: int, T: int,
                      src_slots=None, err=None, stream=None):
    _, H, Dh = k_cache.shape
    B = prefix_len.numel()
    _check(_lib.medusa_kv_compact(_ptr(k_cache), _ptr(v_cache), _ptr(seq_start), _ptr(prefix_len),
                                  _ptr(accepted_nodes), _ptr(accept_len), B, H, Dh, Kmax, T, _dtype(k_cache),
                                  _ptr(src_slots), _ptr(err), _stream(stream)), "medusa_kv_compact")


def medusa_heads_topk_workspace_size(B, K, d, V, s_max) -> int:
    return int(_lib.medusa_heads_topk_workspace_size(B, K, d, V, s_max))


def medusa_heads_topk(hidden, last_node, w1, b1, w2, s, head_logits, topk, workspace, err=None,
                      stream=None):
    B, T, d = hidden.shape
    K, V = w2.shape[0], w2.shape[1]
    s_arr = np.ascontiguousarray(s, np.int32)
    assert len(s_arr) == K
    s_max = topk.shape[-1]
    _check(_lib.medusa_heads_topk(_ptr(hidden), _ptr(last_node), T, _ptr(w1), _ptr(b1), _ptr(w2),
                                  _ptr(s_arr), K, B, d, V, _dtype(hidden), _ptr(head_logits), _ptr(topk),
                                  s_max, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _ptr(err), _stream(stream)), "medusa_heads_topk")


def medusa_heads_topk_candidates(hidden, last_node, w1, b1, w2, s, head_logits, topk, workspace, next_root,
                                 tree: "DeviceTree", tokens, err=None, stream=None):
    """medusa_heads_topk, then the next step's candidate tokens from next_root and topk, in one call."""
    B, T, d = hidden.shape
    K, V = w2.shape[0], w2.shape[1]
    s_arr = np.ascontiguousarray(s, np.int32)
    assert len(s_arr) == K
    s_max = topk.shape[-1]
    _check(_lib.medusa_heads_topk_candidates(_ptr(hidden), _ptr(last_node), T, _ptr(w1), _ptr(b1), _ptr(w2),
                                             _ptr(s_arr), K, B, d, V, _dtype(hidden), _ptr(head_logits), _ptr(topk),
                                             s_max, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                             _ptr(next_root), tree.ref, _ptr(tokens), _ptr(err), _stream(stream)),
           "medusa_heads_topk_candidates")


def medusa_heads_hidden(hidden, w1, b1, s, u, err=None, stream=None, layout=W_ROWS):
    """u [rows][K][d] = dtype(SiLU(W1_k h_r + b1_k) + h_r) for every row of hidden (any leading shape)."""
    d = hidden.shape[-1]
    rows = hidden.numel() // d
    s_arr = np.ascontiguousarray(s, np.int32)
    _check(_lib.medusa_heads_hidden(_ptr(hidden), rows, _ptr(w1), layout, _ptr(b1), _ptr(s_arr), len(s_arr), d,
                                    _dtype(hidden), _ptr(u), _ptr(err), _stream(stream)), "medusa_heads_hidden")


def medusa_lm_head_verify_heads_hidden(hidden, w_lm, V, logits, w1, b1, s, u, err=None, stream=None,
                                       layout=W_ROWS, w1_layout=W_ROWS):
    """logits [rows][V] and u [rows][K][d] in one launch (bf16).  w_lm: [V][d], or its tile copy (flat)
    with layout=W_TILES; w1: [K][d][d], or the tile copy of w1 seen as [K*d][d] with w1_layout=W_TILES."""
    d = hidden.shape[-1]
    rows = hidden.numel() // d
    s_arr = np.ascontiguousarray(s, np.int32)
    _check(_lib.medusa_lm_head_verify_heads_hidden(_ptr(hidden), rows, d, _ptr(w_lm), layout, int(V), _ptr(logits),
                                                   _ptr(w1), w1_layout, _ptr(b1), _ptr(s_arr), len(s_arr), _ptr(u),
                                                   _dtype(hidden), _ptr(err), _stream(stream)),
           "medusa_lm_head_verify_heads_hidden")


def medusa_heads_logits_topk_workspace_size(B, K, V, s_max) -> int:
    return int(_lib.medusa_heads_logits_topk_workspace_size(B, K, V, s_max))


def medusa_heads_logits_topk(u, T, node, w2, s, head_logits, topk, workspace, err=None, stream=None):
    """W2 + top-s on row b*T + node[b] of u [B*T][K][d]; the workspace must be zero on the first call."""
    K, V, d = w2.shape
    B = node.shape[0]
    s_arr = np.ascontiguousarray(s, np.int32)
    assert len(s_arr) == K
    _check(_lib.medusa_heads_logits_topk(_ptr(u), T, _ptr(node), _ptr(w2), _ptr(s_arr), K, B, d, V, _dtype(u),
                                         _ptr(head_logits), _ptr(topk), topk.shape[-1], _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _ptr(err),
                                         _stream(stream)), "medusa_heads_logits_topk")


def medusa_build_candidates(next_root, topk, tree: DeviceTree, tokens, stream=None):
    B, K, s_max = topk.shape
    _check(_lib.medusa_build_candidates(_ptr(next_root), _ptr(topk), s_max, K, tree.ref, B, _ptr(tokens),
                                        _stream(stream)), "medusa_build_candidates")


def medusa_append_tokens(tokens, accepted_nodes, accept_len, out, out_len, err=None, stream=None):
    """out[b][out_len[b]:] += tokens[b][accepted path]; out_len[b] += accept_len[b] + 1."""
    B, T = tokens.shape
    _check(_lib.medusa_append_tokens(_ptr(tokens), _ptr(accepted_nodes), _ptr(accept_len), B, T,
                                     accepted_nodes.shape[1] - 1, _ptr(out), _ptr(out_len), out.shape[1],
                                     _ptr(err), _stream(stream)), "medusa_append_tokens")


def medusa_standin_embed(tokens, emb, hidden, err=None, stream=None):
    """hidden[r] = emb[tokens[r]] over the flattened tokens (stand-in backbone)."""
    V, d = emb.shape
    _check(_lib.medusa_standin_embed(_ptr(tokens), tokens.numel(), _ptr(emb), V, d, _dtype(emb), _ptr(hidden),
                                     _ptr(err), _stream(stream)), "medusa_standin_embed")


def medusa_accept_rejection_workspace_size(B, V) -> int:
    return int(_lib.medusa_accept_rejection_workspace_size(B, V))


def medusa_accept_rejection(logits, draft_logits, tokens, tree: DeviceTree, temperature, uniforms, accept_len,
                            accepted_nodes, next_token, workspace, err=None, stream=None):
    """Rejection-sampling acceptance over the tree (uniforms [B][T][u_stride] are inputs)."""
    B, T, V = logits.shape
    _check(_lib.medusa_accept_rejection(_ptr(logits), _ptr(draft_logits), draft_logits.shape[1], _ptr(tokens),
                                        tree.ref, B, V, float(temperature), _ptr(uniforms), uniforms.shape[2],
                                        _ptr(accept_len), _ptr(accepted_nodes), _ptr(next_token), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _ptr(err),
                                        _stream(stream)), "medusa_accept_rejection")


def medusa_lm_head_stat_groups(rows, V) -> int:
    return int(_lib.medusa_lm_head_stat_groups(rows, V))


def medusa_lm_head_ctas(rows: int, V: int) -> int:
    """CTAs the bf16 LM head launches for rows x V on the current device."""
    return int(_lib.medusa_lm_head_ctas(rows, V))


def medusa_lm_head_verify_stats(hidden, w_lm, logits, stats, mode, temperature, V, err=None, stream=None,
                                layout=W_ROWS):
    """LM head + fused acceptance statistics; logits may be None in greedy mode (mode 0)."""
    d = hidden.shape[-1]
    rows = hidden.numel() // d
    _check(_lib.medusa_lm_head_verify_stats(_ptr(hidden), _ptr(w_lm), _ptr(logits), rows, d, V, _dtype(hidden),
                                            layout, mode, float(temperature), _ptr(stats),
                                            stats.numel() * stats.element_size(), _ptr(err), _stream(stream)),
           "medusa_lm_head_verify_stats")


def medusa_accept_stats(stats, groups, logits, tokens, tree: DeviceTree, mode, temperature, eps, delta, V,
                        accept_len, accepted_nodes, next_root, best_node, best_logp, err=None, stream=None):
    B = tokens.shape[0]
    _check(_lib.medusa_accept_stats(_ptr(stats), groups, _ptr(logits), _ptr(tokens), tree.ref, B, V, mode,
                                    float(temperature), float(eps), float(delta), _ptr(accept_len),
                                    _ptr(accepted_nodes), _ptr(next_root), _ptr(best_node), _ptr(best_logp),
                                    _ptr(err), _stream(stream)), "medusa_accept_stats")
