"""CPU oracle for one Medusa tree-speculative verify step (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  The product (the CUDA
library and its binding) never touches it, and it never touches the product.

The arithmetic lives in ``oracle.c`` (plain single-threaded C99, double
accumulation); this module only builds it with gcc and marshals numpy arrays.
bfloat16 tensors are passed as their raw bits (``numpy.uint16``).

Parity pins for every function are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (no fast-math) if it is missing or stale."""
    stale = (
        force
        or not os.path.exists(_LIB)
        or os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    )
    if stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = C.CDLL(_LIB)
        _declare(_lib)
    return _lib


P = C.c_void_p
I32 = C.c_int32
I = C.c_int
D = C.c_double


def _declare(L):
    L.orc_bf16_round.restype = C.c_uint16
    L.orc_bf16_round.argtypes = [D]
    L.orc_tree_compile.restype = I
    L.orc_tree_compile.argtypes = [P, P, I, I, P, P, P, P, P, P, P]
    L.orc_tree_cartesian.restype = I
    L.orc_tree_cartesian.argtypes = [P, I, I, P, P]
    L.orc_tree_greedy.restype = I
    L.orc_tree_greedy.argtypes = [P, I, I, I, P, P]
    L.orc_tree_expected_len.restype = D
    L.orc_tree_expected_len.argtypes = [P, P, I, I, P, I]
    L.orc_rope.restype = None
    L.orc_rope.argtypes = [P, I, C.c_int64, D]
    L.orc_attn_one.restype = None
    L.orc_attn_one.argtypes = [I, I, P, P, P, D, P]
    L.orc_tree_attn.restype = I
    L.orc_tree_attn.argtypes = [I, P, P, P, P, P, P, P, P, P, I, I, I, I, D, D, P, P]
    L.orc_lm_head.restype = I
    L.orc_lm_head.argtypes = [I, P, P, I, I, I, P]
    L.orc_accept.restype = I
    L.orc_accept.argtypes = [P, P, P, P, I, I, I, I, I, D, D, D, P, P, P, P, P, P, P, P]
    L.orc_kv_compact.restype = I
    L.orc_kv_compact.argtypes = [I, P, P, P, P, P, P, I, I, I, I, P]
    L.orc_heads.restype = I
    L.orc_heads.argtypes = [I, P, P, I, P, P, P, P, I, I, I, I, P, P, I, P]
    L.orc_topk_f32.restype = I
    L.orc_topk_f32.argtypes = [P, I, I, P]
    L.orc_build_candidates.restype = I
    L.orc_build_candidates.argtypes = [P, P, I, I, P, P, I, I, P]
    L.orc_rejection_emit.restype = D
    L.orc_rejection_emit.argtypes = [P, P, I, P]
    L.orc_rejection_tree.restype = I
    L.orc_rejection_tree.argtypes = [P, P, P, P, P, P, I, I, I, I, D, P, I, P, P, P, P]


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def _dt(a) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"oracle element type must be float32 or bf16 bits (uint16), got {a.dtype}")


def _chk(rc, what):
    if rc < 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")
    return rc


# ---------------------------------------------------------------- elements ---

def bf16_round(x: float) -> int:
    return int(lib().orc_bf16_round(float(x)))


def to_double(a: np.ndarray) -> np.ndarray:
    """Widen float32 or bf16 bits to float64 exactly."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# -------------------------------------------------------------------- tree ---

class Tree:
    """A compiled candidate tree (oracle's own representation)."""

    def __init__(self, node_paths, parent, depth, rank, anc, s, K):
        self.node_paths = node_paths
        self.parent = parent
        self.depth = depth
        self.rank = rank
        self.anc = anc
        self.s = s
        self.K = K
        self.T = len(parent)


def tree_compile(paths: np.ndarray, path_len: np.ndarray, max_depth: int) -> Tree:
    paths = np.ascontiguousarray(paths, dtype=np.int32).reshape(-1, max_depth)
    path_len = np.ascontiguousarray(path_len, dtype=np.int32)
    n = len(path_len)
    T = n + 1
    node_paths = np.zeros((T, max_depth), np.int32)
    parent = np.zeros(T, np.int32)
    depth = np.zeros(T, np.int32)
    rank = np.zeros(T, np.int32)
    anc = np.zeros((T, T), np.uint8)
    s = np.zeros(max_depth, np.int32)
    K = np.zeros(1, np.int32)
    _chk(lib().orc_tree_compile(_p(paths), _p(path_len), n, max_depth, _p(node_paths),
                                _p(parent), _p(depth), _p(rank), _p(anc), _p(s), _p(K)),
         "tree_compile")
    return Tree(node_paths, parent, depth, rank, anc, s, int(K[0]))


def tree_cartesian(s, max_nodes: int):
    s = np.ascontiguousarray(s, dtype=np.int32)
    K = len(s)
    paths = np.zeros((max(max_nodes, 1), K), np.int32)
    plen = np.zeros(max(max_nodes, 1), np.int32)
    n = _chk(lib().orc_tree_cartesian(_p(s), K, max_nodes, _p(paths), _p(plen)), "tree_cartesian")
    return paths[:n].copy(), plen[:n].copy()


def tree_greedy(acc: np.ndarray, budget: int):
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    K, R = acc.shape
    paths = np.zeros((max(budget, 1), K), np.int32)
    plen = np.zeros(max(budget, 1), np.int32)
    n = _chk(lib().orc_tree_greedy(_p(acc), K, R, budget, _p(paths), _p(plen)), "tree_greedy")
    return paths[:n].copy(), plen[:n].copy()


def tree_expected_len(paths, path_len, acc) -> float:
    paths = np.ascontiguousarray(paths, dtype=np.int32)
    path_len = np.ascontiguousarray(path_len, dtype=np.int32)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    return float(lib().orc_tree_expected_len(_p(paths), _p(path_len), len(path_len),
                                             paths.shape[1], _p(acc), acc.shape[1]))


# --------------------------------------------------------------- attention ---

def rope(x: np.ndarray, pos: int, theta: float = 10000.0) -> np.ndarray:
    y = np.ascontiguousarray(x, dtype=np.float64).copy()
    lib().orc_rope(_p(y), len(y), int(pos), float(theta))
    return y


def attn_one(q, k, v, scale):
    q = np.ascontiguousarray(q, np.float64)
    k = np.ascontiguousarray(k, np.float64)
    v = np.ascontiguousarray(v, np.float64)
    out = np.zeros(len(q), np.float64)
    lib().orc_attn_one(k.shape[0], len(q), _p(q), _p(k), _p(v), float(scale), _p(out))
    return out


def tree_attn(q, k_new, v_new, k_cache, v_cache, seq_start, prefix_len, tree: Tree,
              rope_theta=10000.0, scale=None):
    """Returns (out [B,T,H,Dh] in the input type, out_d float64).  k_cache and
    v_cache are updated in place (the tree rows are appended)."""
    B, T, H, Dh = q.shape
    assert T == tree.T
    dt = _dt(q)
    if scale is None:
        scale = 1.0 / np.sqrt(Dh)
    out = np.zeros_like(q)
    out_d = np.zeros(q.shape, np.float64)
    seq_start = np.ascontiguousarray(seq_start, np.int64)
    prefix_len = np.ascontiguousarray(prefix_len, np.int32)
    _chk(lib().orc_tree_attn(dt, _p(q), _p(k_new), _p(v_new), _p(k_cache), _p(v_cache),
                             _p(seq_start), _p(prefix_len), _p(tree.depth), _p(tree.anc),
                             T, B, H, Dh, float(rope_theta), float(scale), _p(out), _p(out_d)),
         "tree_attn")
    return out, out_d


# ----------------------------------------------------------------- LM head ---

def lm_head(hidden: np.ndarray, w: np.ndarray) -> np.ndarray:
    hidden = np.ascontiguousarray(hidden)
    w = np.ascontiguousarray(w)
    d = hidden.shape[-1]
    rows = hidden.size // d
    V = w.shape[0]
    assert hidden.dtype == w.dtype
    logits = np.zeros((rows, V), np.float64)
    _chk(lib().orc_lm_head(_dt(hidden), _p(hidden), _p(w), rows, d, V, _p(logits)), "lm_head")
    return logits


# -------------------------------------------------------------- acceptance ---

def accept(logits: np.ndarray, tokens: np.ndarray, tree: Tree, mode: int,
           temperature=1.0, eps=0.09, delta=0.3):
    logits = np.ascontiguousarray(logits, np.float32)
    tokens = np.ascontiguousarray(tokens, np.int32)
    B, T, V = logits.shape
    K = tree.K
    r = dict(
        accept_len=np.zeros(B, np.int32),
        accepted_nodes=np.zeros((B, K + 1), np.int32),
        next_root=np.zeros(B, np.int32),
        best_node=np.zeros(B, np.int32),
        best_logp=np.zeros(B, np.float64),
        row_gap=np.zeros((B, T), np.float64),
        node_margin=np.zeros((B, T), np.float64),
        node_logp=np.zeros((B, T), np.float64),
    )
    _chk(lib().orc_accept(_p(logits), _p(tokens), _p(tree.parent), _p(tree.depth), T, K, B, V,
                          mode, float(temperature), float(eps), float(delta),
                          _p(r["accept_len"]), _p(r["accepted_nodes"]), _p(r["next_root"]),
                          _p(r["best_node"]), _p(r["best_logp"]), _p(r["row_gap"]),
                          _p(r["node_margin"]), _p(r["node_logp"])), "accept")
    return r


# ------------------------------------------------------------ KV compaction ---

def kv_compact(k_cache, v_cache, seq_start, prefix_len, accepted_nodes, accept_len, K):
    """In place on k_cache, v_cache and prefix_len; returns src_slots."""
    tokens, H, Dh = k_cache.shape
    B = len(prefix_len)
    src = np.zeros((B, K + 1), np.int32)
    _chk(lib().orc_kv_compact(_dt(k_cache), _p(k_cache), _p(v_cache),
                              _p(np.ascontiguousarray(seq_start, np.int64)), _p(prefix_len),
                              _p(np.ascontiguousarray(accepted_nodes, np.int32)),
                              _p(np.ascontiguousarray(accept_len, np.int32)),
                              B, H, Dh, K, _p(src)), "kv_compact")
    return src


# ------------------------------------------------------------------- heads ---

def heads(hidden, last_node, w1, b1, w2, s, s_max):
    """hidden [B,T,d]; returns (head_logits [B,K,V] float64, topk [B,K,s_max], u [B,K,d])."""
    B, T, d = hidden.shape
    K, V = w2.shape[0], w2.shape[1]
    s = np.ascontiguousarray(s, np.int32)
    logits = np.zeros((B, K, V), np.float64)
    topk = np.zeros((B, K, s_max), np.int32)
    u = np.zeros((B, K, d), hidden.dtype)
    _chk(lib().orc_heads(_dt(hidden), _p(hidden), _p(np.ascontiguousarray(last_node, np.int32)), T,
                         _p(w1), _p(b1), _p(w2), _p(s), K, B, d, V, _p(logits), _p(topk), s_max,
                         _p(u)), "heads")
    return logits, topk, u


def topk_f32(z: np.ndarray, s: int) -> np.ndarray:
    z = np.ascontiguousarray(z, np.float32)
    out = np.zeros(s, np.int32)
    _chk(lib().orc_topk_f32(_p(z), len(z), s, _p(out)), "topk_f32")
    return out


# -------------------------------------------------------------- candidates ---

def build_candidates(next_root, topk, tree: Tree):
    topk = np.ascontiguousarray(topk, np.int32)
    B, K, s_max = topk.shape
    tokens = np.zeros((B, tree.T), np.int32)
    _chk(lib().orc_build_candidates(_p(np.ascontiguousarray(next_root, np.int32)), _p(topk),
                                    s_max, K, _p(tree.depth), _p(tree.rank), tree.T, B,
                                    _p(tokens)), "build_candidates")
    return tokens


# ------------------------------------------------------- rejection sampling ---

def rejection_emit(p, q):
    p = np.ascontiguousarray(p, np.float64)
    q = np.ascontiguousarray(q, np.float64)
    out = np.zeros_like(p)
    beta = lib().orc_rejection_emit(_p(p), _p(q), len(p), _p(out))
    return out, beta


def rejection_tree(logits, draft, tokens, tree: Tree, temperature, u):
    """logits [B,T,V] f32, draft [B,K,V] f32, tokens [B,T], u [B,T,S1] f32 ->
    dict(accept_len [B], accepted_nodes [B,K+1], next_token [B], margin [B])."""
    logits = np.ascontiguousarray(logits, np.float32)
    draft = np.ascontiguousarray(draft, np.float32)
    tokens = np.ascontiguousarray(tokens, np.int32)
    u = np.ascontiguousarray(u, np.float32)
    B, T, V = logits.shape
    K = tree.K
    assert draft.shape == (B, K, V) and u.shape[:2] == (B, T)
    out = dict(accept_len=np.zeros(B, np.int32), accepted_nodes=np.zeros((B, K + 1), np.int32),
               next_token=np.zeros(B, np.int32), margin=np.zeros(B, np.float64))
    _chk(lib().orc_rejection_tree(_p(logits), _p(draft), _p(tokens), _p(tree.parent), _p(tree.depth),
                                  _p(tree.rank), T, K, B, V, float(temperature), _p(u), u.shape[2],
                                  _p(out["accept_len"]), _p(out["accepted_nodes"]), _p(out["next_token"]),
                                  _p(out["margin"])), "rejection_tree")
    return out
