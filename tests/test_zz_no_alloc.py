"""medusa_accept_noalloc against medusa_accept.

Some callers of this library cannot allocate device memory: a plugin or a C
host program that is handed only input and output pointers, or a decode loop
that must not call cudaMalloc because it can synchronise the device.  For
them, medusa_accept_noalloc takes no workspace and uses a fixed scratch array
inside the library.  This test calls it through the C ABI twice in a row, on
different inputs (typical acceptance, then greedy), and checks each result
against medusa_accept on the same inputs (integer outputs bit-exact, the
summed log-probability within 1e-6) and against the oracle's acceptance on
the same logits (integer outputs bit-exact).

This file is collected last so that a run stopping at the first failure has
already run every other test.  It also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from parity_util import both_trees, check_accept_on_gpu_logits, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from medusa_tree_speculative_gb300 import build

    build.build()
    from medusa_tree_speculative_gb300 import medusa

    return medusa


def _tree(M):
    """The 64-node greedy tree, as the oracle's tree and as the library's."""
    return both_trees(M, ("greedy", 4, 10, 64))


def _inputs(tree, B, V, mode, seed):
    """Logits with a planted accepted path per sequence, on the device."""
    rng = np.random.default_rng(seed)
    ht = tree.host
    T = ht.T
    logits = (rng.standard_normal((B, T, V)) * 2.0).astype(np.float32)
    tokens = rng.integers(0, V, (B, T)).astype(np.int32)
    for b in range(B):
        n = int(rng.integers(1, T))
        while n > 0:
            p = int(ht.parent[n])
            if mode == 0:
                tokens[b, n] = int(np.argmax(logits[b, p]))
            else:
                logits[b, p, tokens[b, n]] = logits[b, p].max() + 1.0
            n = p
    return torch.from_numpy(logits).cuda(), torch.from_numpy(tokens).cuda()


def _outputs(B, K):
    z = lambda *s: torch.zeros(s, dtype=torch.int32, device="cuda")
    return dict(accept_len=z(B), accepted_nodes=z(B, K + 1), next_root=z(B), best_node=z(B),
                best_logp=torch.zeros(B, dtype=torch.float32, device="cuda"))


def test_accept_noalloc_matches_accept_on_two_calls(M):
    ot, tree = _tree(M)
    B, V = 3, 32000
    for mode, seed in ((1, 11), (0, 12)):
        logits, tokens = _inputs(tree, B, V, mode, seed)
        ref, got = _outputs(B, tree.K), _outputs(B, tree.K)
        ws = torch.zeros(M.medusa_accept_workspace_size(B, tree.T), dtype=torch.uint8, device="cuda")
        err_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        err_got = torch.zeros(1, dtype=torch.int32, device="cuda")
        M.medusa_accept(logits, tokens, tree, mode, 0.7, 0.09, 0.3, ref["accept_len"], ref["accepted_nodes"],
                        ref["next_root"], ref["best_node"], ref["best_logp"], ws, err_ref)
        M.medusa_accept_noalloc(logits, tokens, tree, mode, 0.7, 0.09, 0.3, got["accept_len"],
                                got["accepted_nodes"], got["next_root"], got["best_node"], got["best_logp"],
                                err_got)
        torch.cuda.synchronize()
        assert int(err_ref.item()) == 0 and int(err_got.item()) == 0
        for key in ("accept_len", "accepted_nodes", "next_root", "best_node"):
            assert torch.equal(ref[key], got[key]), key
        assert torch.allclose(ref["best_logp"], got["best_logp"], rtol=0, atol=1e-6)
        assert int(got["accept_len"].max().item()) >= 1  # the planted paths were taken
        host = {k: to_host(v) for k, v in got.items()}
        assert check_accept_on_gpu_logits(ot, to_host(logits), to_host(tokens), mode, 0.7, 0.09, 0.3, host) == B


def test_accept_noalloc_rejects_oversize(M):
    # 17 sequences of a 512-row tree need 8704 row records; the scratch holds
    # MEDUSA_ACCEPT_NOALLOC_MAX_ROWS = 8192.  Rejected before any launch.
    paths, plen = M.medusa_tree_cartesian([8, 8, 8], 511)
    tree = M.DeviceTree(M.medusa_tree_compile(paths, plen, 3))
    assert tree.T == 512
    logits = torch.zeros((17, tree.T, 8), dtype=torch.float32, device="cuda")
    tokens = torch.zeros((17, tree.T), dtype=torch.int32, device="cuda")
    o = _outputs(17, tree.K)
    with pytest.raises(M.MedusaError, match="CAPACITY"):
        M.medusa_accept_noalloc(logits, tokens, tree, 0, 1.0, 0.09, 0.3, o["accept_len"], o["accepted_nodes"],
                                o["next_root"], o["best_node"], o["best_logp"])
