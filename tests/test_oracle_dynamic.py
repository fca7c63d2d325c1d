"""Pins for the oracle's dynamic tree construction (reranking a candidate pool).

Against: a pool worked by hand, brute force over every tree of N nodes that
can be cut from small pools (the kept tree maximises the expected number of
accepted tokens, sum of exp(value)), special cases (whole pool, root only,
chain, star, ties), and the ancestry of the flattened tree by the independent
tree oracle.
"""
import itertools

import numpy as np
import pytest

from oracle import dynamic as D
from oracle import tree as T
import workloads as W


def _lp(*p):
    return [0.0] + [float(np.float32(np.log(x))) for x in p]


# root; A .6, B .25, C .15 under the root; D .7, E .3 under A; F .9 under B.
# Path probabilities: A .6, D .42, B .25, F .225, E .18, C .15.
HAND_PARENT = [-1, 0, 0, 0, 1, 1, 2]
HAND_LOGP = _lp(0.6, 0.25, 0.15, 0.7, 0.3, 0.9)
HAND_TOKEN = [9, 11, 12, 13, 14, 15, 16]


@pytest.mark.parametrize("n,keep,parent", [
    (1, [0], [-1]),
    (2, [0, 1], [-1, 0]),
    (4, [0, 1, 2, 4], [-1, 0, 0, 1]),           # root, A, B, D
    (5, [0, 1, 2, 4, 6], [-1, 0, 0, 1, 2]),     # + F: the demo tree's shape
    (6, [0, 1, 2, 4, 5, 6], [-1, 0, 0, 1, 1, 2]),
    (7, [0, 1, 2, 3, 4, 5, 6], HAND_PARENT),
])
def test_hand_pool(n, keep, parent):
    p, tok, sel, anc, dep, pos, st = D.build_dynamic([HAND_PARENT], [HAND_LOGP], [HAND_TOKEN], [100], n)
    assert st[0] == 0
    assert sel[0].tolist() == keep
    assert p[0].tolist() == parent
    assert tok[0].tolist() == [HAND_TOKEN[c] for c in keep]
    assert pos[0].tolist() == (100 + T.depths(parent)).tolist()


def _closed_subsets(parent, n):
    m = len(parent)
    for rest in itertools.combinations(range(1, m), n - 1):
        s = {0, *rest}
        if all(parent[c] in s for c in rest):
            yield sorted(s)


def test_kept_tree_maximises_expected_accepted_tokens():
    g = np.random.default_rng(4)
    for trial in range(300):
        m = int(g.integers(1, 10))
        par = W.tree_random_recursive(g, m)
        lp = np.log(g.uniform(0.05, 1.0, m)).astype(np.float32)
        lp[0] = 0.0
        n = int(g.integers(1, m + 1))
        v = D.path_values(par, lp).astype(np.float64)
        best = max(sum(np.exp(v[c]) for c in s) for s in _closed_subsets(par, n))
        keep = D.rerank(par, lp, n).tolist()
        assert 0 in keep and len(set(keep)) == n
        assert all(par[c] in keep for c in keep if c != 0), (par, keep)
        got = sum(np.exp(v[c]) for c in keep)
        assert got >= best - 1e-12, (trial, got, best)
        winners = [s for s in _closed_subsets(par, n) if sum(np.exp(v[c]) for c in s) >= best - 1e-12]
        if len(winners) == 1:
            assert keep == winners[0]


def test_special_cases():
    g = np.random.default_rng(5)
    m = 12
    par = W.tree_random_recursive(g, m)
    lp = np.log(g.uniform(0.1, 1.0, m)).astype(np.float32)
    lp[0] = 0
    # the whole pool: identity
    p, tok, sel, *_ , st = D.build_dynamic([par], [lp], [np.arange(m)], [0], m)
    assert sel[0].tolist() == list(range(m)) and p[0].tolist() == par.tolist()
    # a chain keeps its first n nodes
    chain = W.tree_chain(m)
    for n in (1, 3, m):
        assert D.rerank(chain, lp, n).tolist() == list(range(n))
    # a star keeps the n-1 most probable children (ties: smaller index)
    star = W.tree_star(m)
    lps = np.array([0, -1, -0.5, -0.5, -3, -0.1, -2, -0.5, -1, -1, -4, -0.2], np.float32)
    assert D.rerank(star, lps, 5).tolist() == [0, 2, 3, 5, 11]
    assert D.rerank(star, lps, 6).tolist() == [0, 2, 3, 5, 7, 11]


def test_flattened_tree_and_masks():
    pool = W.candidate_pool(3, 4, 5, 4, 1000)
    n = 30
    p, tok, sel, anc, dep, pos, st = D.build_dynamic(pool.parent, pool.logp, pool.token, [7, 8, 9, 10], n)
    assert (st == 0).all()
    a2, d2, p2, s2 = T.build_ancestry(p, np.array([7, 8, 9, 10]))
    np.testing.assert_array_equal(anc, a2)
    np.testing.assert_array_equal(dep, d2)
    np.testing.assert_array_equal(pos, p2)
    for b in range(4):
        assert T.is_valid_tree(p[b])
        assert (np.diff(sel[b]) > 0).all()
        for k in range(1, n):
            assert sel[b][p[b][k]] == pool.parent[b][sel[b][k]]
        np.testing.assert_array_equal(tok[b], pool.token[b][sel[b]])


def test_invalid_pools():
    ok = ([HAND_PARENT], [HAND_LOGP], [HAND_TOKEN], [0])
    assert D.build_dynamic(*ok, 7)[-1][0] == 0
    assert D.build_dynamic(*ok, 8)[-1][0] == -3                        # pool smaller than the tree
    bad_lp = list(HAND_LOGP)
    bad_lp[3] = 0.1
    assert D.build_dynamic([HAND_PARENT], [bad_lp], [HAND_TOKEN], [0], 4)[-1][0] == -3
    bad_lp[3] = float("nan")
    assert D.build_dynamic([HAND_PARENT], [bad_lp], [HAND_TOKEN], [0], 4)[-1][0] == -3
    bad_par = list(HAND_PARENT)
    bad_par[4] = 5
    assert D.build_dynamic([bad_par], [HAND_LOGP], [HAND_TOKEN], [0], 4)[-1][0] == -3
    # a zero-probability candidate (logp = -inf) is allowed and ranks last
    lp = list(HAND_LOGP)
    lp[1] = float("-inf")
    p, tok, sel, *_, st = D.build_dynamic([HAND_PARENT], [lp], [HAND_TOKEN], [0], 7)
    assert st[0] == 0 and sel[0].tolist() == list(range(7))
    assert D.rerank(HAND_PARENT, np.array(lp, np.float32), 4).tolist() == [0, 2, 3, 6]


def test_generator_contract():
    pool = W.candidate_pool(9, 3, 6, 5, 500)
    M = 1 + 5 + 5 * 25
    assert pool.parent.shape == (3, M)
    for b in range(3):
        assert T.is_valid_tree(pool.parent[b])
        assert (pool.logp[b][1:] <= 0).all() and pool.logp[b][0] == 0
        for u in range(M):
            kids = np.nonzero(pool.parent[b] == u)[0]
            assert len(kids) in (0, 5)
            assert len(set(pool.token[b][kids].tolist())) == len(kids)
