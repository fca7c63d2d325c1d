"""GPU parity of tree_build_dynamic against the oracle: the kept set, its
flattened parent array, tokens, pool indices, ancestry masks, depths,
positions and status, all bit-exact (the path values are the same fp32
recurrence on both sides, so the ranking is identical)."""
import numpy as np
import pytest
import torch

from oracle import dynamic as D
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tree_attention_speculative_gb300 import _build
    _build.build()


def run_gpu(parent, logp, token, prefix_len, n):
    import tree_attention_speculative_gb300 as ts
    B, M = parent.shape
    dev = "cuda"

    def i32(x):
        return torch.from_numpy(np.ascontiguousarray(x, np.int32)).to(dev)

    W_ = (n + 63) // 64
    out = dict(parent=torch.full((B, n), -9, dtype=torch.int32, device=dev),
               tokens=torch.full((B, n), -9, dtype=torch.int32, device=dev),
               sel=torch.full((B, n), -9, dtype=torch.int32, device=dev),
               anc=torch.zeros((B, n, W_), dtype=torch.int64, device=dev),
               depth=torch.full((B, n), -9, dtype=torch.int32, device=dev),
               pos=torch.full((B, n), -9, dtype=torch.int32, device=dev),
               status=torch.full((B,), 77, dtype=torch.int32, device=dev))
    ts.tree_build_dynamic(i32(parent), torch.from_numpy(np.ascontiguousarray(logp, np.float32)).to(dev), i32(token),
                          i32(prefix_len), out["parent"], out["tokens"], out["sel"], out["anc"], out["depth"],
                          out["pos"], out["status"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def check(parent, logp, token, prefix_len, n):
    got = run_gpu(parent, logp, token, prefix_len, n)
    p, tok, sel, anc, dep, pos, st = D.build_dynamic(parent, logp, token, prefix_len, n)
    np.testing.assert_array_equal(got["status"], st)
    ok = st == 0
    np.testing.assert_array_equal(got["parent"][ok], p[ok])
    np.testing.assert_array_equal(got["tokens"][ok], tok[ok])
    np.testing.assert_array_equal(got["sel"][ok], sel[ok])
    np.testing.assert_array_equal(got["anc"][ok].view(np.uint64), anc[ok])
    np.testing.assert_array_equal(got["depth"][ok], dep[ok])
    np.testing.assert_array_equal(got["pos"][ok], pos[ok])
    return got


@pytest.mark.parametrize("B,depth,topk,n", [(4, 5, 4, 30), (64, 8, 8, 64), (3, 10, 10, 256), (5, 3, 6, 1),
                                            (2, 4, 3, 40)])
def test_dynamic_matches_oracle(B, depth, topk, n):
    pool = W.candidate_pool(depth * 100 + topk, B, depth, topk, 128256)
    M = pool.parent.shape[1]
    n = min(n, M)
    plen = W.rng(n, "dyn-plen").integers(0, 5000, B)
    check(pool.parent, pool.logp, pool.token, plen, n)


def test_whole_pool_ties_infinities_and_chains():
    g = W.rng(1, "dyn-edge")
    B, M = 6, 120
    parent = np.stack([W.tree_random_recursive(g, M) for _ in range(B)])
    # quantised log-probabilities: many exact ties, decided by pool index
    logp = -g.integers(0, 4, (B, M)).astype(np.float32) * np.float32(0.25)
    logp[:, 0] = 0
    logp[1, 5:40] = -np.inf
    parent[2] = W.tree_chain(M)
    parent[3] = W.tree_star(M)
    token = g.integers(0, 1000, (B, M))
    for n in (1, 2, 64, 120):
        check(parent, logp, token, np.arange(B) * 10, n)
    # the largest pool, and a chain of it (1023 levels)
    pool = W.candidate_pool(7, 2, 10, 10, 5000)
    pp = np.concatenate([pool.parent, np.full((2, 1024 - pool.parent.shape[1]), 0, np.int32)], 1)
    lp = np.concatenate([pool.logp, np.full((2, 1024 - pool.parent.shape[1]), -30, np.float32)], 1)
    tk = np.concatenate([pool.token, np.zeros((2, 1024 - pool.parent.shape[1]), np.int32)], 1)
    pp[1] = W.tree_chain(1024)
    check(pp, lp, tk, [3, 4], 256)


def test_invalid_pools_report_and_leave_a_star():
    g = W.rng(2, "dyn-bad")
    pool = W.candidate_pool(2, 4, 4, 4, 1000)
    parent, logp = pool.parent.copy(), pool.logp.copy()
    parent[0, 7] = 9            # not topological
    logp[1, 3] = 0.5            # positive log-probability
    logp[2, 4] = np.nan
    got = check(parent, logp, pool.token, [1, 2, 3, 4], 16)
    assert got["status"].tolist() == [-3, -3, -3, 0]
    for b in range(3):
        assert got["parent"][b].tolist() == [-1] + [0] * 15
        assert got["depth"][b].tolist() == [0] + [1] * 15
        assert (got["anc"][b, :, 0].view(np.uint64) == (np.uint64(1) | (np.uint64(1) << np.arange(16, dtype=np.uint64)))).all()
