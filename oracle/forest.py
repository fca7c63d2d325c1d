"""Oracle: forests of draft trees in one flattened sequence (test infrastructure only).

[P3] The Future of Reasoning (speculative forest exploration): the verifier
evaluates whole forests of candidate continuations in parallel.  [P1] Key
Mechanisms > Modified Causal Attention Mask and [P2] How It Works: a node
sees the verified prefix, itself and its ancestors, nothing of another
branch; the acceptance rule follows one valid path (P2) up to the first
rejection (P1 Multi-Token Acceptance & Rollback).

Readings where the pages are silent:
  * A forest is flattened in topological order: node 0 is a root
    (parent -1), and every other node is either another root (parent -1) or
    has a parent with a smaller index.
  * Every root is a given token, attended at position P_b like the single
    root of a tree; a node's mask, depth and position follow its chain up to
    its own root (so nodes of different trees never see each other).
  * Greedy acceptance generalises the tree rule: every root is accepted;
    node c is accepted iff every node x on its chain below its root has
    draft[x] == argmax(logits[parent[x]]).  n* is the deepest accepted node of
    the whole forest, ties to the smallest index; the accepted path runs from
    n*'s root to n*; accept_len = depth(n*); bonus = argmax(logits[n*]).
  * Invalid forests give status -3; a path longer than max_depth status -2,
    as for trees.

The attention of a forest needs nothing new: the tree attention oracle
follows parent pointers until -1 and so already stops at each node's root.
"""
from __future__ import annotations

import numpy as np

from .tree import ancestry_matrix, depths, pack_rows
from .verify import greedy_argmax

ERR_SHAPE = -2
ERR_BAD_TREE = -3


def is_valid_forest(parent) -> bool:
    parent = [int(p) for p in parent]
    if len(parent) < 1 or parent[0] != -1:
        return False
    return all(p == -1 or 0 <= p < i for i, p in enumerate(parent) if i > 0)


def roots_of(parent) -> np.ndarray:
    parent = [int(p) for p in parent]
    out = np.zeros(len(parent), np.int64)
    for i in range(len(parent)):
        r = i
        while parent[r] != -1:
            r = parent[r]
        out[i] = r
    return out


def build_ancestry_forest(parent, prefix_len):
    """parent [B, N] -> anc [B, N, W] uint64, depth [B, N], pos [B, N], status [B]."""
    parent = np.asarray(parent)
    B, N = parent.shape
    W = (N + 63) // 64
    anc = np.zeros((B, N, W), np.uint64)
    dep = np.zeros((B, N), np.int32)
    pos = np.zeros((B, N), np.int32)
    status = np.zeros(B, np.int32)
    for b in range(B):
        if not is_valid_forest(parent[b]):
            status[b] = ERR_BAD_TREE
            continue
        anc[b] = pack_rows(ancestry_matrix(parent[b]))
        dep[b] = depths(parent[b])
        pos[b] = int(prefix_len[b]) + dep[b]
    return anc, dep, pos, status


def accept_walk_forest(parent, draft, am, max_depth: int):
    """Acceptance by definition for one forest: (path[max_depth+1], L, bonus, status)."""
    parent = [int(p) for p in parent]
    n = len(parent)
    path = np.full(max_depth + 1, -1, np.int32)
    if not is_valid_forest(parent):
        return path, 0, 0, ERR_BAD_TREE
    best, best_d = 0, 0
    for c in range(n):
        ok, x, d = True, c, 0
        while parent[x] != -1:
            if int(draft[x]) != int(am[parent[x]]):
                ok = False
            x = parent[x]
            d += 1
        if ok and d > best_d:
            best, best_d = c, d
    bonus = int(am[best])
    if best_d > max_depth:
        return path, best_d, bonus, ERR_SHAPE
    x = best
    for k in range(best_d, -1, -1):
        path[k] = x
        x = parent[x]
    return path, best_d, bonus, 0


def verify_greedy_forest(draft, logits, parent, max_depth: int):
    """Batched like oracle.verify.verify_greedy, for forests."""
    draft = np.asarray(draft)
    parent = np.asarray(parent)
    B, N = draft.shape
    am = greedy_argmax(np.asarray(logits, np.float32))
    acc = np.full((B, max_depth + 1), -1, np.int32)
    L = np.zeros(B, np.int32)
    bonus = np.zeros(B, np.int32)
    status = np.zeros(B, np.int32)
    for b in range(B):
        acc[b], L[b], bonus[b], status[b] = accept_walk_forest(parent[b], draft[b], am[b], max_depth)
    return acc, L, bonus, am, status
