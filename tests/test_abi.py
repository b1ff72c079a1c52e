"""Host-side tests of libmedusa (no GPU needed): the library loads and exports
every entry point include/medusa.h declares; the host tree helpers agree with
the oracle bit for bit; argument validation rejects bad calls before any CUDA
work is enqueued."""
import ctypes as C
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def M():
    from medusa_tree_speculative_gb300 import build

    build.build()
    from medusa_tree_speculative_gb300 import medusa

    return medusa


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "medusa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(medusa_[a-z0-9_]+)\s*\(", src)))


def test_header_symbols_exported(M):
    declared = _declared_symbols()
    assert len(declared) >= 15
    lib = C.CDLL(M.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/medusa.h but not exported"
    assert set(declared) == set(M.EXPORTS), "binding and header disagree"


def test_version_and_error_string(M):
    assert "sm_103a" in M.medusa_version()
    assert isinstance(M._lib.medusa_last_error(), bytes)


@pytest.mark.parametrize("s,max_nodes", [((2, 2, 2), 14), ((2, 3), 8), ((4, 4, 4, 4), 256),
                                         ((3, 1, 2), 9), ((5,), 5)])
def test_cartesian_and_compile_match_oracle(M, orc, s, max_nodes):
    p1, l1 = M.medusa_tree_cartesian(list(s), max_nodes)
    p0, l0 = orc.tree_cartesian(list(s), max_nodes)
    assert np.array_equal(p1, p0) and np.array_equal(l1, l0)
    t1 = M.medusa_tree_compile(p1, l1, len(s))
    t0 = orc.tree_compile(p0, l0, len(s))
    assert t1.T == t0.T and t1.K == t0.K
    for f in ("parent", "depth", "rank", "node_paths"):
        assert np.array_equal(getattr(t1, f), getattr(t0, f)), f
    assert np.array_equal(t1.s[:t1.K], t0.s[:t0.K])
    # bitmask vs dense matrix
    dense = np.zeros((t1.T, t1.T), np.uint8)
    for i in range(t1.T):
        for j in range(t1.T):
            dense[i, j] = (int(t1.anc_mask[i, j // 32]) >> (j % 32)) & 1
    assert np.array_equal(dense, t0.anc)


@pytest.mark.parametrize("K,R,budget", [(4, 10, 64), (5, 10, 64), (3, 4, 20), (4, 10, 1)])
def test_greedy_matches_oracle(M, orc, K, R, budget):
    from medusa_tree_speculative_gb300.synth import accuracy_table

    acc = accuracy_table(K, R)
    p1, l1 = M.medusa_tree_greedy(acc, budget)
    p0, l0 = orc.tree_greedy(acc, budget)
    assert np.array_equal(p1, p0) and np.array_equal(l1, l0)


def test_compile_random_shuffled_sets(M, orc):
    rng = np.random.default_rng(21)
    for _ in range(20):
        paths = set()
        while len(paths) < int(rng.integers(1, 60)):
            k = int(rng.integers(1, 6))
            p = tuple(int(r) for r in rng.integers(1, 5, size=k))
            for j in range(1, k + 1):
                paths.add(p[:j])
        paths = list(paths)
        rng.shuffle(paths)
        arr = np.zeros((len(paths), 5), np.int32)
        for i, p in enumerate(paths):
            arr[i, :len(p)] = p
        plen = np.array([len(p) for p in paths], np.int32)
        t1 = M.medusa_tree_compile(arr, plen, 5)
        t0 = orc.tree_compile(arr, plen, 5)
        assert np.array_equal(t1.parent, t0.parent) and np.array_equal(t1.node_paths, t0.node_paths)


def test_compile_rejects_bad_sets(M):
    with pytest.raises(M.MedusaError, match="INVALID"):
        M.medusa_tree_compile(np.array([[1, 2], [2, 0]]), np.array([2, 1]), 2)
    with pytest.raises(M.MedusaError, match="INVALID"):
        M.medusa_tree_compile(np.array([[1, 0], [1, 0]]), np.array([1, 1]), 2)
    with pytest.raises(M.MedusaError, match="UNSUPPORTED"):  # rank above MEDUSA_MAX_S
        M.medusa_tree_compile(np.array([[17]]), np.array([1]), 1)
    with pytest.raises(M.MedusaError, match="UNSUPPORTED"):  # more than MEDUSA_MAX_T rows
        paths, plen = M.medusa_tree_cartesian([16, 16, 16], 600)
        M.medusa_tree_compile(paths, plen, 3)


# ---- argument validation: every case below fails before any CUDA call ----

FAKE = 0x10000  # never dereferenced: validation rejects the call first


def _fake_tree(M, T=15, K=3, s=(2, 2, 2)):
    t = M.medusa_tree_t()
    t.parent = t.depth = t.rank = t.anc_mask = FAKE
    t.T, t.W, t.K = T, (T + 31) // 32, K
    for k, v in enumerate(s):
        t.s[k] = v
    return t


def _no_gpu():
    import torch

    return not torch.cuda.is_available()


pytestmark_cpu = pytest.mark.skipif("not _no_gpu()")


@pytest.mark.skipif(not _no_gpu(), reason="host-only validation checks run without a GPU")
def test_validation_statuses(M):
    L = M._lib
    t = _fake_tree(M)
    ref = C.byref(t)
    # accept: bad mode, non-positive temperature, NULL output, tiny workspace
    assert L.medusa_accept(FAKE, FAKE, ref, 1, 100, 2, 1.0, 0.09, 0.3, FAKE, FAKE, FAKE, FAKE, None,
                           FAKE, 1 << 20, None, None) == -1
    assert L.medusa_accept(FAKE, FAKE, ref, 1, 100, 1, 0.0, 0.09, 0.3, FAKE, FAKE, FAKE, FAKE, None,
                           FAKE, 1 << 20, None, None) == -1
    assert L.medusa_accept(FAKE, FAKE, ref, 1, 100, 0, 1.0, 0.09, 0.3, None, FAKE, FAKE, FAKE, None,
                           FAKE, 1 << 20, None, None) == -1
    assert L.medusa_accept(FAKE, FAKE, ref, 1, 100, 0, 1.0, 0.09, 0.3, FAKE, FAKE, FAKE, FAKE, None,
                           FAKE, 4, None, None) == -4
    # tree checks: T above the maximum, wrong W, NULL tree
    big = _fake_tree(M, T=600, K=3)
    assert L.medusa_accept(FAKE, FAKE, C.byref(big), 1, 100, 0, 1.0, 0.09, 0.3, FAKE, FAKE, FAKE, FAKE,
                           None, FAKE, 1 << 20, None, None) == -2
    badw = _fake_tree(M)
    badw.W = 3
    assert L.medusa_build_candidates(FAKE, FAKE, 2, 3, C.byref(badw), 1, FAKE, None) == -1
    assert L.medusa_build_candidates(FAKE, FAKE, 2, 3, None, 1, FAKE, None) == -1
    # build_candidates: s_max below the tree's widest level, K below depth
    assert L.medusa_build_candidates(FAKE, FAKE, 1, 3, ref, 1, FAKE, None) == -1
    assert L.medusa_build_candidates(FAKE, FAKE, 2, 2, ref, 1, FAKE, None) == -1
    # attention: Dh outside {64,128}, bad dtype, small workspace
    assert L.medusa_tree_attn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ref, 1, 4, 96, 64, 1e4, 0.1,
                              1, FAKE, FAKE, 1 << 30, None, None) == -2
    assert L.medusa_tree_attn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ref, 1, 4, 64, 64, 1e4, 0.1,
                              7, FAKE, FAKE, 1 << 30, None, None) == -2
    assert L.medusa_tree_attn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ref, 1, 4, 64, 64, 1e4, 0.1,
                              0, FAKE, FAKE, 16, None, None) == -4   # f32 stages q' in scratch
    assert L.medusa_tree_attn(FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ref, 1, 4, 64, 64, 1e4, 0.1,
                              1, FAKE, None, 0, None, None) == -1    # bf16 needs 16-byte alignment
    assert L.medusa_tree_attn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ref, 17, 4, 64, 64, 1e4, 0.1,
                              1, FAKE, FAKE, 1 << 30, None, None) == -1
    # joint LM head + heads' W1: bf16 only, rows <= 256, d a multiple of 128
    s3 = (C.c_int32 * 3)(2, 2, 2)
    assert L.medusa_lm_head_verify_heads_hidden(FAKE, 15, 256, FAKE, 1, 1000, FAKE, FAKE, 1, None, s3, 3, FAKE,
                                                0, None, None) == -2
    assert L.medusa_lm_head_verify_heads_hidden(FAKE, 300, 256, FAKE, 1, 1000, FAKE, FAKE, 1, None, s3, 3, FAKE,
                                                1, None, None) == -2
    assert L.medusa_lm_head_verify_heads_hidden(FAKE, 15, 192, FAKE, 1, 1000, FAKE, FAKE, 1, None, s3, 3, FAKE,
                                                1, None, None) == -2
    assert L.medusa_lm_head_verify_heads_hidden(FAKE, 15, 256, FAKE, 1, 1000, None, FAKE, 1, None, s3, 3, FAKE,
                                                1, None, None) == -1
    assert L.medusa_lm_head_verify_heads_hidden(FAKE, 15, 256, FAKE, 3, 1000, FAKE, FAKE, 1, None, s3, 3, FAKE,
                                                1, None, None) == -1
    # key splits outside {1, 2, 4, 8}; fewer than 8 need bf16
    for ks in (0, 3, 16, -1):
        assert L.medusa_tree_attn_splits(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ref, 1, 4, 64, 64, 1e4,
                                         0.1, 1, FAKE, FAKE, 1 << 30, ks, None, None) == -2
    assert L.medusa_tree_attn_splits(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ref, 1, 4, 64, 64, 1e4,
                                     0.1, 0, FAKE, FAKE, 1 << 30, 1, None, None) == -2
    # tensor-core attention: key splits outside {1, 2, 4, 8}, Dh other than 128, f32
    def tc(dh, dt, ks):
        return L.medusa_tree_attn_tc(FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, FAKE, FAKE, FAKE, ref, 1, 4, dh, 64,
                                     1e4, 0.1, dt, FAKE, ks, None, None)
    for ks in (0, 3, 16, -1):
        assert tc(128, 1, ks) == -2
    assert tc(64, 1, 1) == -2
    assert tc(128, 0, 1) == -2
    # host-to-device staging copy: nothing to do, NULL, misaligned, memory that is not mapped pinned memory
    assert L.medusa_copy_from_host(FAKE, FAKE, 0, None) == 0
    assert L.medusa_copy_from_host(None, FAKE, 64, None) == -1
    assert L.medusa_copy_from_host(FAKE, FAKE + 8, 64, None) == -1
    assert L.medusa_copy_from_host(FAKE, FAKE, 40, None) == -1
    buf = np.zeros(64, np.uint8)
    assert L.medusa_copy_from_host(FAKE, buf.ctypes.data + (-buf.ctypes.data % 16), 32, None) == -1
    # LM head: d not a multiple of 64 for bf16; misaligned pointers
    assert L.medusa_lm_head_verify(FAKE, FAKE, FAKE, 15, 100, 1000, 1, 0, None, 0, None, None) == -2
    assert L.medusa_lm_head_verify(FAKE + 2, FAKE, FAKE, 15, 256, 1000, 1, 0, None, 0, None, None) == -1
    # LM head layouts: unknown layout, tiles are bf16 only
    assert L.medusa_lm_head_verify(FAKE, FAKE, FAKE, 15, 256, 1000, 1, 2, None, 0, None, None) == -1
    assert L.medusa_lm_head_verify(FAKE, FAKE, FAKE, 15, 256, 1000, 0, 1, None, 0, None, None) == -2
    # tiling: d not a multiple of 64, misaligned, overlapping source and destination
    assert L.medusa_lm_head_tile(FAKE, FAKE + (1 << 24), 100, 1000, None) == -2
    assert L.medusa_lm_head_tile(FAKE + 8, FAKE + (1 << 24), 256, 1000, None) == -1
    assert L.medusa_lm_head_tile(FAKE, FAKE + 4096, 256, 1000, None) == -1
    assert b"overlaps" in L.medusa_last_error()
    # error-word read-out: NULL or misaligned pointers (rejected before any CUDA call)
    assert L.medusa_check_errors(None, FAKE, 1, None) == -1
    assert L.medusa_check_errors(FAKE + 2, FAKE, 1, None) == -1
    # KV compaction: Kmax above the maximum, misaligned cache, tree rows outside 1..MEDUSA_MAX_T
    assert L.medusa_kv_compact(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 64, 9, 65, 1, None, None, None) == -2
    assert L.medusa_kv_compact(FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 64, 3, 65, 1, None, None, None) == -1
    assert L.medusa_kv_compact(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 64, 3, 0, 1, None, None, None) == -1
    assert L.medusa_kv_compact(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 64, 3, 513, 1, None, None, None) == -1
    # heads: s_k above s_max, too-small workspace, K above the maximum
    s = (C.c_int32 * 3)(2, 9, 2)
    assert L.medusa_heads_topk(FAKE, FAKE, 15, FAKE, None, FAKE, s, 3, 1, 256, 1000, 1, FAKE, FAKE, 8,
                               FAKE, 1 << 30, None, None) == -1
    s = (C.c_int32 * 3)(2, 2, 2)
    assert L.medusa_heads_topk(FAKE, FAKE, 15, FAKE, None, FAKE, s, 3, 1, 256, 1000, 1, FAKE, FAKE, 8,
                               FAKE, 8, None, None) == -4
    assert L.medusa_heads_topk(FAKE, FAKE, 15, FAKE, None, FAKE, s, 9, 1, 256, 1000, 1, FAKE, FAKE, 8,
                               FAKE, 1 << 30, None, None) == -2
    assert b"medusa_heads_topk" in L.medusa_last_error()
    # heads + candidate fill: no tree, no tokens, fewer heads than tree levels, tree s above s_max
    assert L.medusa_heads_topk_candidates(FAKE, FAKE, 15, FAKE, None, FAKE, s, 3, 1, 256, 1000, 1, FAKE, FAKE, 8,
                                          FAKE, 1 << 30, FAKE, None, FAKE, None, None) == -1
    assert L.medusa_heads_topk_candidates(FAKE, FAKE, 15, FAKE, None, FAKE, s, 3, 1, 256, 1000, 1, FAKE, FAKE, 8,
                                          FAKE, 1 << 30, FAKE, ref, None, None, None) == -1
    assert L.medusa_heads_topk_candidates(FAKE, FAKE, 15, FAKE, None, FAKE, s, 2, 1, 256, 1000, 1, FAKE, FAKE, 8,
                                          FAKE, 1 << 30, FAKE, ref, FAKE, None, None) == -1
    assert L.medusa_heads_topk_candidates(FAKE, FAKE, 15, FAKE, None, FAKE, s, 3, 1, 256, 1000, 1, FAKE, FAKE, 1,
                                          FAKE, 1 << 30, FAKE, ref, FAKE, None, None) == -1
    # heads over every row: bf16 needs d a multiple of 128; K above the maximum; bad layout
    s = (C.c_int32 * 3)(2, 2, 2)
    assert L.medusa_heads_hidden(FAKE, 65, FAKE, 0, None, s, 3, 320, 1, FAKE, None, None) == -2
    assert L.medusa_heads_hidden(FAKE, 65, FAKE, 0, None, s, 9, 256, 1, FAKE, None, None) == -2
    assert L.medusa_heads_hidden(FAKE, 65, FAKE, 5, None, s, 3, 256, 1, FAKE, None, None) == -1
    assert L.medusa_heads_hidden(FAKE, 65, FAKE, 1, None, s, 3, 256, 0, FAKE, None, None) == -2  # f32: rows only
    zero = (C.c_int32 * 3)(0, 0, 0)
    assert L.medusa_heads_hidden(FAKE, 65, FAKE, 0, None, zero, 3, 256, 1, FAKE, None, None) == 0  # nothing to do
    # W2 on the accepted row: small workspace, s_k above s_max
    assert L.medusa_heads_logits_topk(FAKE, 65, FAKE, FAKE, s, 3, 1, 256, 1000, 1, FAKE, FAKE, 8, FAKE, 8,
                                      None, None) == -4
    s9 = (C.c_int32 * 3)(2, 9, 2)
    assert L.medusa_heads_logits_topk(FAKE, 65, FAKE, FAKE, s9, 3, 1, 256, 1000, 1, FAKE, FAKE, 8, FAKE, 1 << 30,
                                      None, None) == -1


def test_workspace_queries(M):
    assert M.medusa_accept_workspace_size(1, 65) >= 65 * 16
    assert M.medusa_heads_topk_workspace_size(1, 4, 4096, 32000, 8) >= 4 * 4096 * 2
    n = M.medusa_tree_attn_workspace_size(1, 32, 128, 65, 1024)
    assert n >= 65 * 32 * 128 * 4
    assert M.medusa_lm_head_workspace_size(65, 4096, 32000) == 0
    assert M.medusa_heads_logits_topk_workspace_size(1, 4, 32000, 8) >= 4 * 4
    assert M.medusa_lm_head_tiled_bytes(4096, 32000) == 32000 * 4096 * 2
    assert M.medusa_lm_head_tiled_bytes(256, 1000) == 1024 * 256 * 2  # last block padded to 128 rows
    assert M.medusa_lm_head_tiled_bytes(100, 1000) == 0


def test_tc_key_splits(M):
    """The tensor-core attention's default key split (host logic): one wave of
    one-CTA-per-SM clusters, at least one key tile per CTA."""
    from medusa_tree_speculative_gb300.step import tc_key_splits

    assert tc_key_splits(1, 32, 65, 1024, 152) == 4    # 7B, one sequence: 128 CTAs
    assert tc_key_splits(1, 40, 65, 2048, 152) == 2    # 13B: 40 heads
    assert tc_key_splits(4, 52, 65, 8192, 152) == 1    # 33B, four sequences: 208 CTAs already
    assert tc_key_splits(1, 2, 15, 300, 152) == 2      # 3 key tiles: 4 would leave a CTA none
    assert tc_key_splits(1, 1, 15, 0, 152) == 1        # one key tile only
    assert tc_key_splits(1, 32, 257, 4096, 152) == 1   # three row blocks: 96 CTAs
    assert tc_key_splits(1, 16, 65, 1024, 152) == 8
    # in the step: the 27 SMs the 7B LM head (125 CTAs) leaves free
    assert tc_key_splits(1, 32, 65, 4096, 27) == 1
    assert tc_key_splits(1, 4, 65, 4096, 27) == 4      # 16 CTAs; 8 splits would need 32 SMs


def test_lm_head_plans(M):
    """CTAs the bf16 LM head launches per row plan (host logic, one CTA per
    SM): two weight tiles per work item up to 128 rows; CTA pairs (an even
    count) from 129 to 256 rows; one 256-row chunk plus the extra rows by
    mma.sync from 257 to 264; chunks sharing each weight block beyond."""
    assert M.medusa_lm_head_ctas(0, 32000) == 0
    assert M.medusa_lm_head_ctas(65, 0) == 0
    assert M.medusa_lm_head_ctas(65, 32000) == 125            # 250 tiles, two per item
    for rows in (129, 200, 256):
        assert M.medusa_lm_head_ctas(rows, 32000) == 126      # 63 pairs, four tiles each
        assert M.medusa_lm_head_ctas(rows, 1000) % 2 == 0     # 8 tiles: four pairs
    for rows in (257, 260, 264, 265, 512):
        assert M.medusa_lm_head_ctas(rows, 32000) == 125
