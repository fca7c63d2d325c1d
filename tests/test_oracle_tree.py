"""Pins for the oracle's tree part: validity, ancestry mask, depth, positions.

Each check compares against something other than the oracle's own walk: the
values the demo tree prints, hand-derived masks, a transitive closure computed
by boolean matrix powers, closed forms for chains and stars, and structural
invariants of an ancestor relation.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import tree as T
import workloads as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example_5node.json")))


def test_worked_example_mask_words_and_sparsity():
    parent = np.array(GOLD["parent"])
    m = T.ancestry_matrix(parent)
    for i, vis in enumerate(GOLD["visible_by_hand"]):
        assert sorted(np.nonzero(m[i])[0].tolist()) == vis
    words = T.pack_rows(m)
    assert words[:, 0].tolist() == GOLD["mask_words_by_hand"]
    assert abs(T.mask_sparsity(m) - GOLD["sparsity_by_hand"]) < 1e-12


def test_worked_example_depth_pos_match_printed_records():
    parent = np.array([GOLD["parent"]])
    anc, dep, pos, st = T.build_ancestry(parent, np.array([GOLD["prefix_len"]]))
    assert st.tolist() == [0]
    assert dep[0].tolist() == GOLD["depth_printed"]
    assert pos[0].tolist() == GOLD["pos_by_hand"]
    assert anc[0, :, 0].tolist() == GOLD["mask_words_by_hand"]
    # the printed child lists are the inverse of the parent pointers
    for i, kids in enumerate(GOLD["children_printed"]):
        assert [j for j in range(5) if GOLD["parent"][j] == i] == kids


def _closure(parent):
    """Ancestor-or-self relation as reflexive-transitive closure of the parent edge,
    by repeated boolean squaring (no walking)."""
    n = len(parent)
    a = np.eye(n, dtype=bool)
    for i, p in enumerate(parent):
        if p >= 0:
            a[i, p] = True
    while True:
        a2 = (a.astype(np.int64) @ a.astype(np.int64)) > 0
        if (a2 == a).all():
            return a
        a = a2


def _all_trees(n):
    for choice in itertools.product(*[range(i) for i in range(1, n)]):
        yield np.array((-1,) + choice, np.int64)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7])
def test_mask_equals_transitive_closure_all_trees(n):
    for parent in _all_trees(n):
        m = T.ancestry_matrix(parent)
        assert (m == _closure(parent)).all()
        dep = T.depths(parent)
        # popcount of a row = depth + 1 (itself plus one ancestor per level)
        assert (m.sum(1) == dep + 1).all()
        for i in range(1, n):
            p = parent[i]
            # row i = row of the parent plus i itself
            expect = m[p].copy()
            expect[i] = True
            assert (m[i] == expect).all()
        # siblings share exactly their parent's row
        for i in range(1, n):
            for j in range(i + 1, n):
                if parent[i] == parent[j]:
                    assert ((m[i] & m[j]) == m[parent[i]]).all()


@pytest.mark.parametrize("n", [1, 63, 64, 65, 128, 129, 192, 256])
def test_chain_words_closed_form(n):
    parent = W.tree_chain(n)
    anc, dep, pos, st = T.build_ancestry(parent[None], np.array([7]))
    assert st[0] == 0
    assert dep[0].tolist() == list(range(n))
    assert pos[0].tolist() == [7 + i for i in range(n)]
    for i in range(n):
        for w in range(anc.shape[2]):
            lo, hi = 64 * w, min(i, 64 * w + 63)
            cnt = max(0, hi - lo + 1)
            expect = (1 << cnt) - 1 if cnt < 64 else (1 << 64) - 1
            assert int(anc[0, i, w]) == expect


@pytest.mark.parametrize("n", [2, 65, 200])
def test_star_words_closed_form(n):
    anc, dep, pos, st = T.build_ancestry(W.tree_star(n)[None], np.array([0]))
    for i in range(1, n):
        bits = {0, i}
        for w in range(anc.shape[2]):
            expect = sum(1 << (j - 64 * w) for j in bits if 64 * w <= j < 64 * w + 64)
            assert int(anc[0, i, w]) == expect
    assert dep[0, 1:].tolist() == [1] * (n - 1)


@pytest.mark.parametrize("parent,valid", [
    ([-1], True),
    ([-1, 0, 0, 1, 2], True),
    ([0, 0], False),            # root must be -1
    ([-1, -1], False),          # second root
    ([-1, 1], False),           # self loop
    ([-1, 2, 0], False),        # parent after child
    ([-1, 0, 5], False),        # out of range
    ([-1, 0, -2], False),       # negative non-root
    ([], False),
])
def test_validity_cases(parent, valid):
    assert T.is_valid_tree(parent) == valid


def test_invalid_tree_status():
    parent = np.array([[-1, 0, 0], [-1, 2, 0]])
    _, _, _, st = T.build_ancestry(parent, np.array([3, 3]))
    assert st.tolist() == [0, -3]


def test_generated_trees_have_requested_shape():
    g = W.rng(1, "t")
    for n, d in [(64, 6), (64, 8), (192, 10), (5, 4)]:
        p = W.tree_random_levels(g, n, d)
        assert T.is_valid_tree(p)
        assert T.depths(p).max() == min(d, n - 1)
    p = W.tree_from_widths([4, 3, 2, 1, 1])
    assert len(p) == 26 and T.is_valid_tree(p)
    assert np.bincount(T.depths(p)).tolist() == [1, 4, 12, 6, 2, 1]
