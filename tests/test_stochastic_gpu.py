"""GPU parity of tree_verify_stochastic against the oracle.

Inputs are seeded; the coins of a sequence are redrawn (by the oracle alone)
until every acceptance comparison of its walk is at least 1e-3 away from its
threshold in relative terms, so that fp32 and fp64 must take the same accept /
reject decisions: paths, lengths and status are compared exactly.  The bonus
token is compared exactly when coins[0] lies more than 1e-4 (in probability
mass) from an inversion boundary; otherwise the token drawn must be one with
mass whose cumulative interval lies within 2e-5 of coins[0], which is what
fp32 sums over the vocabulary can guarantee.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import stochastic as S
import workloads as W

pytestmark = pytest.mark.gpu

ACC_MARGIN = 1e-3
SMP_MARGIN = 1e-4
SMP_TOL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tree_attention_speculative_gb300 import _build
    _build.build()


def robust_coins(si, parent, max_depth, seed):
    """Redraw the coins of sequences whose walk decides an acceptance within
    ACC_MARGIN of its threshold (oracle only)."""
    g = W.rng(seed, "coins-redraw")
    coins = si.coins.copy()
    for _ in range(50):
        _, _, _, _, m = S.verify_stochastic(si.draft, si.logits, si.q, parent, coins, si.temperature, max_depth)
        bad = np.nonzero(m[:, 0] < ACC_MARGIN)[0]
        if len(bad) == 0:
            return coins
        coins[bad] = g.random((len(bad), coins.shape[1]), dtype=np.float32)
    raise AssertionError("could not draw coins away from the acceptance thresholds")


def run_gpu(draft, logits, q, parent, coins, T, max_depth):
    import tree_attention_speculative_gb300 as ts
    B, N = parent.shape
    dev = "cuda"
    d = torch.from_numpy(np.ascontiguousarray(draft, np.int32)).to(dev)
    lg = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).to(dev)
    qq = torch.from_numpy(np.ascontiguousarray(q, np.float32)).to(dev)
    p = torch.from_numpy(np.ascontiguousarray(parent, np.int32)).to(dev)
    c = torch.from_numpy(np.ascontiguousarray(coins, np.float32)).to(dev)
    acc = torch.full((B, max_depth + 1), -7, dtype=torch.int32, device=dev)
    L = torch.full((B,), -7, dtype=torch.int32, device=dev)
    bonus = torch.full((B,), -7, dtype=torch.int32, device=dev)
    st = torch.zeros(B, dtype=torch.int32, device=dev)
    ts.tree_verify_stochastic(d, lg, qq, p, c, T, acc, L, bonus, st)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), L.cpu().numpy(), bonus.cpu().numpy(), st.cpu().numpy()


def check(draft, logits, q, parent, coins, T, max_depth):
    acc, L, bonus, st = run_gpu(draft, logits, q, parent, coins, T, max_depth)
    exact = 0
    for b in range(parent.shape[0]):
        path, l, bo, s, am, sm, r = S.walk_stochastic(parent[b], draft[b], logits[b], q[b], coins[b], T, max_depth,
                                                       final=True)
        assert st[b] == s, (b, st[b], s)
        assert acc[b].tolist() == path.tolist(), (b, acc[b], path)
        assert L[b] == l, (b, L[b], l)
        if s == oracle.ERR_BAD_TREE:
            assert bonus[b] == 0
            continue
        assert am >= ACC_MARGIN, "inputs must keep acceptance decisions away from thresholds"
        if bonus[b] == bo:
            exact += 1
            continue
        assert sm < SMP_MARGIN, (b, bonus[b], bo, sm)
        v = int(bonus[b])
        cum = np.cumsum(r)
        lo = cum[v - 1] if v > 0 else 0.0
        c0 = float(coins[b][0])
        assert r[v] > 0 and lo - SMP_TOL <= c0 <= cum[v] + SMP_TOL, (b, v, bo, lo, cum[v], c0)
    return exact


CASES = [
    # (tag, B, N, depth, V, T)
    ("small-vocab", 6, 40, 6, 1000, 1.0),
    ("odd-vocab", 4, 33, 5, 1001, 0.7),        # rows not 16-byte aligned: plain loads
    ("two-cta", 5, 64, 8, 4100, 1.3),
    ("llama3-vocab", 4, 64, 8, 128256, 1.0),
    ("wide", 2, 256, 12, 5000, 0.9),
]


@pytest.mark.parametrize("tag,B,N,depth,V,T", CASES)
def test_stochastic_matches_oracle(tag, B, N, depth, V, T):
    g = W.rng(len(tag) * 7 + N, "stoch-gpu-" + tag)
    parent = np.stack([W.tree_random_levels(g, N, depth) for _ in range(B)])
    si = W.stochastic_inputs(11 + N, parent, V, temperature=T)
    coins = robust_coins(si, parent, depth, 5)
    exact = check(si.draft, si.logits, si.q, parent, coins, T, depth)
    if V <= 5000:
        assert exact >= B // 2


def test_edge_cases():
    V = 3000
    g = W.rng(4, "stoch-edge")
    N = 12
    parent = np.stack([W.tree_random_levels(g, N, 4) for _ in range(6)])
    parent[0] = W.tree_star(N)
    parent[1] = W.tree_chain(N)
    parent[2, 5] = 7               # not topological: a bad tree
    si = W.stochastic_inputs(4, parent, V)
    si.draft[3, 4] = V             # a draft token outside the vocabulary
    parent[5] = W.tree_chain(N)
    coins = robust_coins(si, parent, 4, 9)
    coins[5, 1:] = 0.0             # chain accepted all the way: longer than max_depth 4
    acc, L, bonus, st = run_gpu(si.draft, si.logits, si.q, parent, coins, 1.0, 4)
    assert st[2] == oracle.ERR_BAD_TREE and st[3] == oracle.ERR_BAD_TREE
    assert (acc[2] == -1).all() and (acc[3] == -1).all() and bonus[2] == 0 and bonus[3] == 0
    assert st[5] == -2 and L[5] == N - 1 and (acc[5] == -1).all()
    check(si.draft, si.logits, si.q, parent, coins, 1.0, 4)
    # a single node: the bonus is drawn from the root's own target distribution
    one = np.full((3, 1), -1, np.int32)
    si1 = W.stochastic_inputs(5, one, V)
    check(si1.draft, si1.logits, si1.q, one, si1.coins, 0.8, 0)


def test_greedy_limit_matches_greedy_verify():
    """A one-hot target makes the stochastic walk the greedy walk; compare with
    the greedy oracle on the planted greedy workload."""
    g = W.rng(8, "greedy-limit-tree")
    parents = np.stack([W.tree_random_levels(g, 64, 8) for _ in range(8)])
    plant = W.rng(8, "greedy-limit-plant").integers(0, 9, size=8)
    case = W.build_case("greedy-limit", 8, parents, [16] * 8, Hq=1, Hkv=1, D=64, bs=16, permute=False,
                        vocab=128256, plant_len=plant)
    lg = case.logits.copy()
    am = oracle.verify.greedy_argmax(lg)
    B, N, V = lg.shape
    lg[np.arange(B)[:, None], np.arange(N)[None, :], am] += 800.0
    q = np.full((B, N, V), 1.0 / V, np.float32)
    coins = W.rng(1, "greedy-limit").random((B, N), dtype=np.float32)
    acc, L, bonus, st = run_gpu(case.draft, lg, q, case.parent, coins, 1.0, 8)
    gacc, gL, gbonus, _, gst = oracle.verify.verify_greedy(case.draft, case.logits, case.parent, 8)
    np.testing.assert_array_equal(acc, gacc)
    np.testing.assert_array_equal(L, gL)
    np.testing.assert_array_equal(bonus, gbonus)
    np.testing.assert_array_equal(st, gst)
    np.testing.assert_array_equal(L, case.planted_len)


def test_full_size_batch64_all_sequences_and_determinism():
    """The bench's stochastic workload: batch 64, 64-node depth-8 trees over the
    128256-token vocabulary; every sequence checked, and a second run is
    bit-identical."""
    g = W.rng(20260004, "tree")
    parent = np.stack([W.tree_random_levels(g, 64, 8) for _ in range(64)])
    si = W.stochastic_inputs(20260004, parent, 128256, temperature=1.0)
    coins = robust_coins(si, parent, 8, 3)
    check(si.draft, si.logits, si.q, parent, coins, 1.0, 8)
    r1 = run_gpu(si.draft, si.logits, si.q, parent, coins, 1.0, 8)
    r2 = run_gpu(si.draft, si.logits, si.q, parent, coins, 1.0, 8)
    for x, y in zip(r1, r2):
        np.testing.assert_array_equal(x, y)
