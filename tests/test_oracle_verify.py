"""Pins for the oracle's greedy verification.

Against: the hand-worked acceptance cases on the demo tree (golden file), the
listing's own flattened scan on chain trees (shifted by one position, since a
node's logits predict its child), a top-down search written independently of
the oracle's bottom-up chain test on every small tree, planted argmax indices,
and planted ties.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import verify as V
import workloads as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example_5node.json")))


@pytest.mark.parametrize("k", range(len(GOLD["acceptance_cases_by_hand"])))
def test_worked_example_acceptance(k):
    case = GOLD["acceptance_cases_by_hand"][k]
    path, L, bonus, st = V.accept_walk(GOLD["parent"], GOLD["token_ids"], case["argmax"], GOLD["max_depth"])
    assert st == 0
    assert path.tolist() == case["path"]
    assert L == case["accept_len"]
    assert bonus == case["bonus"]


def test_chain_matches_listing_scan_shifted():
    g = np.random.default_rng(3)
    for _ in range(300):
        n = int(g.integers(1, 12))
        draft = g.integers(0, 3, n)
        am = g.integers(0, 3, n)
        # the listing scans index by index and stops at the first mismatch; on a
        # chain the prediction for node i sits at node i-1
        scan = 0
        for i in range(1, n):
            if draft[i] == am[i - 1]:
                scan += 1
            else:
                break
        path, L, bonus, st = V.accept_walk(W.tree_chain(n), draft, am, n)
        assert st == 0 and L == scan
        assert path[: L + 1].tolist() == list(range(L + 1))
        assert bonus == am[L]


def _top_down(parent, draft, am):
    """Breadth-first from the root, entering a child only if its draft equals the
    parent's prediction; the last node reached at the greatest depth, smallest index."""
    n = len(parent)
    kids = [[c for c in range(n) if parent[c] == p] for p in range(n)]
    frontier, depth, best = [0], 0, (0, 0)
    while frontier:
        for x in sorted(frontier):
            if depth > best[0] or (depth == best[0] and x < best[1]):
                best = (depth, x)
        nxt = []
        for x in frontier:
            nxt += [c for c in kids[x] if draft[c] == am[x]]
        frontier, depth = nxt, depth + 1
    return best


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_brute_force_small_trees_all_tokens(n):
    for rest in itertools.product(*[range(i) for i in range(1, n)]):
        parent = (-1,) + rest
        for draft in itertools.product(range(2), repeat=n):
            for am in itertools.product(range(2), repeat=n):
                path, L, bonus, st = V.accept_walk(parent, draft, am, n)
                d, x = _top_down(parent, draft, am)
                assert (L, path[L]) == (d, x)
                assert bonus == am[x]


def test_brute_force_random_larger_trees():
    g = np.random.default_rng(11)
    for _ in range(2000):
        n = int(g.integers(5, 9))
        parent = W.tree_random_recursive(g, n)
        draft = g.integers(0, 3, n)
        am = g.integers(0, 3, n)
        path, L, bonus, st = V.accept_walk(parent, draft, am, n)
        d, x = _top_down(parent.tolist(), draft, am)
        assert (L, path[L]) == (d, x)
        # path is the parent chain of x, root first
        chain = []
        y = x
        while y != -1:
            chain.append(y)
            y = parent[y]
        assert path[: L + 1].tolist() == chain[::-1]


def test_argmax_planted_and_ties():
    g = np.random.default_rng(5)
    x = g.standard_normal((6, 1000)).astype(np.float32)
    x[0, 17] = 9.0
    x[1, 999] = 9.0
    x[2, 5] = 9.0
    x[2, 700] = 9.0        # tie: first wins
    x[3, :] = 0.0
    x[3, 0] = -0.0         # -0 == +0: tie, index 0
    x[4, 3] = np.float32(1e30)
    x[4, 4] = np.float32(1e30)
    x[5, :] = -np.float32(3.0)
    x[5, 42] = -np.float32(2.9999998)
    am = V.greedy_argmax(x)
    assert am.tolist() == [17, 999, 5, 0, 3, 42]


def test_planted_workload_lengths_and_argmax():
    c = W.c1()
    acc, L, bonus, am, st = V.verify_greedy(c.draft, c.logits, c.parent, 4)
    assert st.tolist() == [0]
    assert acc[0].tolist() == [0, 1, 3, -1, -1] and L.tolist() == [2]
    assert (am == c.planted_argmax).all()
    g = W.rng(3, "x")
    parents = np.stack([W.tree_random_levels(g, 40, 5) for _ in range(6)])
    case = W.build_case("t", 3, parents, [4] * 6, Hq=1, Hkv=1, D=8, bs=4, permute=False,
                        vocab=500, plant_len=[0, 1, 2, 3, 4, 5])
    acc, L, bonus, am, st = V.verify_greedy(case.draft, case.logits, case.parent, 5)
    assert L.tolist() == [0, 1, 2, 3, 4, 5]
    assert (am == case.planted_argmax).all()
    assert acc[np.arange(6), L].tolist() == case.planted_target.tolist()


def test_path_too_long_for_buffer():
    path, L, bonus, st = V.accept_walk(W.tree_chain(4), [0, 1, 2, 3], [1, 2, 3, 4], 2)
    assert st == V.ERR_SHAPE and L == 3 and bonus == 4 and path.tolist() == [-1, -1, -1]


def test_invalid_tree_status():
    _, _, _, st = V.accept_walk([-1, 2, 0], [0, 0, 0], [0, 0, 0], 3)
    assert st == V.ERR_BAD_TREE
