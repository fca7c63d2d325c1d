"""Pins for the oracle's forests: decomposition into separate trees (each run
through the pinned tree oracle, results mapped back), the single-root and
all-roots special cases, a worked two-tree example and invalid forests."""
import numpy as np
import pytest

from oracle import forest as F
from oracle import tree as T
from oracle import verify as V
import workloads as W


def _components(parent):
    roots = F.roots_of(parent)
    comps = {}
    for i, r in enumerate(roots):
        comps.setdefault(int(r), []).append(i)
    return [comps[r] for r in sorted(comps)]


def test_masks_by_decomposition():
    g = np.random.default_rng(1)
    for trial in range(100):
        n = int(g.integers(1, 40))
        par = W.forest_random(g, n, int(g.integers(1, min(n, 6) + 1)), 5)
        assert F.is_valid_forest(par)
        anc, dep, pos, st = F.build_ancestry_forest(par[None], [100])
        assert st[0] == 0
        m = np.zeros((n, n), bool)
        d = np.zeros(n, np.int64)
        for comp in _components(par):
            loc = {c: k for k, c in enumerate(comp)}
            lp = np.array([-1 if par[c] < 0 else loc[int(par[c])] for c in comp])
            mm = T.ancestry_matrix(lp)
            d[comp] = T.depths(lp)
            for a_, ca in enumerate(comp):
                for b_, cb in enumerate(comp):
                    m[ca, cb] = mm[a_, b_]
        np.testing.assert_array_equal(anc[0], T.pack_rows(m))
        np.testing.assert_array_equal(dep[0], d)
        np.testing.assert_array_equal(pos[0], 100 + d)


def test_acceptance_by_decomposition():
    g = np.random.default_rng(2)
    for trial in range(300):
        n = int(g.integers(1, 30))
        par = W.forest_random(g, n, int(g.integers(1, min(n, 5) + 1)), 5)
        draft = g.integers(0, 3, n)
        am = g.integers(0, 3, n)
        md = int(g.integers(0, 7))
        path, L, bonus, st = F.accept_walk_forest(par, draft, am, 10)
        best = None
        for comp in _components(par):
            loc = {c: k for k, c in enumerate(comp)}
            lp = [-1 if par[c] < 0 else loc[int(par[c])] for c in comp]
            p2, l2, b2, s2 = V.accept_walk(lp, draft[comp], am[comp], 10)
            nstar = comp[int(p2[l2])]
            cand = (l2, -nstar, [comp[int(x)] for x in p2[: l2 + 1]], b2)
            if best is None or cand[:2] > best[:2]:
                best = cand
        assert st == 0 and L == best[0] and path[: L + 1].tolist() == best[2] and bonus == best[3], trial
        path2, L2, bonus2, st2 = F.accept_walk_forest(par, draft, am, md)
        assert (L2, bonus2) == (L, bonus)
        assert (st2, path2.tolist()) == ((0, path[: md + 1].tolist()) if L <= md else (-2, [-1] * (md + 1)))


def test_single_root_is_the_tree_rule_and_all_roots():
    g = np.random.default_rng(3)
    for trial in range(100):
        n = int(g.integers(1, 20))
        par = W.tree_random_recursive(g, n)
        draft = g.integers(0, 3, n)
        am = g.integers(0, 3, n)
        a = F.accept_walk_forest(par, draft, am, n)
        b = V.accept_walk(par, draft, am, n)
        assert a[0].tolist() == b[0].tolist() and a[1:] == b[1:]
    roots = np.full(7, -1)
    anc, dep, pos, st = F.build_ancestry_forest(roots[None], [5])
    assert anc[0, :, 0].tolist() == [1 << i for i in range(7)] and dep.sum() == 0 and (pos == 5).all()
    path, L, bonus, st = F.accept_walk_forest(roots, np.arange(7), np.arange(7) + 3, 3)
    assert path.tolist() == [0, -1, -1, -1] and L == 0 and bonus == 3 and st == 0


def test_worked_two_demo_trees():
    # two copies of the demo tree side by side: nodes 0-4 and 5-9
    par = [-1, 0, 0, 1, 2, -1, 5, 5, 6, 7]
    draft = [0, 10, 11, 12, 13, 0, 20, 21, 22, 23]
    am = [10, 99, 99, 99, 99, 20, 22, 99, 99, 99]   # tree 1 accepts 0->1; tree 2 accepts 5->6->8
    assert F.accept_walk_forest(par, draft, am, 4)[:2][1] == 2
    path, L, bonus, st = F.accept_walk_forest(par, draft, am, 4)
    assert path.tolist() == [5, 6, 8, -1, -1] and bonus == 99 and st == 0
    am2 = [10, 12, 99, 99, 99, 20, 22, 99, 77, 99]   # both accept two: the smaller index (3) wins
    path, L, bonus, st = F.accept_walk_forest(par, draft, am2, 4)
    assert path.tolist() == [0, 1, 3, -1, -1] and L == 2 and bonus == 99


def test_invalid_forests():
    for bad in ([0, -1], [-1, 1], [-1, 0, 3, 0], [-1, -2]):
        assert not F.is_valid_forest(bad)
        assert F.build_ancestry_forest(np.array([bad]), [0])[3][0] == -3
        assert F.accept_walk_forest(bad, [0] * len(bad), [0] * len(bad), 3)[3] == -3
    assert F.is_valid_forest([-1, -1, 0, 1, -1])


def test_generator_interleaves_trees():
    g = np.random.default_rng(4)
    par = W.forest_random(g, 50, 4, 5)
    assert F.is_valid_forest(par) and (par == -1).sum() == 4
    roots = F.roots_of(par)
    assert not all(roots[i] <= roots[i + 1] for i in range(49))   # not simply concatenated
