"""Oracle: greedy verification of a scored draft tree (test infrastructure only).

[P3] code listing, verify_candidate_tree: the target's greedy prediction at each
node is the argmax of that node's logits over the vocabulary.  [P1] Key
Mechanisms > Multi-Token Acceptance & Rollback, and Integration with
Speculative Decoding: the longest valid prefix of the tree, from the root up to
the first rejection, is accepted.  [P2] How It Works: the acceptance rule
follows one valid path through the scored tree.

The listing's own loop compares draft and prediction at the same flattened
index and stops at the first mismatch; that is not tree-aware (it would accept
a sibling) and is not followed.  The rule written out here:

  * A node's logits predict its children.  The root (node 0) is the last
    verified token: it is never checked and is always accepted.
  * Node c >= 1 is accepted iff for every node x on its chain c -> ... -> the
    root's child, draft[x] == argmax(logits[parent[x]]).
  * n* is the accepted node of greatest depth; ties go to the smaller index
    (several valid paths exist only when siblings share a draft token).
  * The accepted path is root -> n*, root first, padded with -1 to
    max_depth + 1 entries; accept_len = depth(n*) counts accepted drafts
    (the root excluded); bonus = argmax(logits[n*]) is the target's next token.

Readings: argmax ties go to the first index (as torch.argmax documents);
logits are finite.  If depth(n*) > max_depth the path does not fit: status -2,
the path row stays all -1, accept_len and bonus are still reported.  An invalid
tree gives status -3 and unspecified outputs (zeros here).
"""
from __future__ import annotations

import numpy as np

from .tree import is_valid_tree

ERR_SHAPE = -2
ERR_BAD_TREE = -3


def greedy_argmax(logits: np.ndarray) -> np.ndarray:
    """Index of the first maximum along the last axis, compared in the logits' own fp32."""
    return np.argmax(logits, axis=-1).astype(np.int32)


def accept_walk(parent, draft, am, max_depth: int):
    """Acceptance by definition for one tree: returns (path[max_depth+1], L, bonus, status)."""
    parent = [int(p) for p in parent]
    n = len(parent)
    path = np.full(max_depth + 1, -1, np.int32)
    if not is_valid_tree(parent):
        return path, 0, 0, ERR_BAD_TREE
    accepted = [False] * n
    depth = [0] * n
    accepted[0] = True
    for c in range(1, n):
        ok, x, d = True, c, 0
        while x != 0:
            p = parent[x]
            if int(draft[x]) != int(am[p]):
                ok = False
            x = p
            d += 1
        accepted[c] = ok
        depth[c] = d
    best = 0
    for c in range(1, n):
        if accepted[c] and depth[c] > depth[best]:
            best = c
    L = depth[best]
    bonus = int(am[best])
    if L > max_depth:
        return path, L, bonus, ERR_SHAPE
    x = best
    while x != -1:
        path[depth[x]] = x
        x = parent[x]
    return path, L, bonus, 0


def verify_greedy(draft, logits, parent, max_depth: int):
    """Batched: draft [B,N], logits [B,N,V] fp32, parent [B,N] ->
    accepted [B,max_depth+1], accept_len [B], bonus [B], argmax [B,N], status [B]."""
    draft = np.asarray(draft)
    parent = np.asarray(parent)
    B, N = draft.shape
    am = greedy_argmax(np.asarray(logits, np.float32))
    acc = np.full((B, max_depth + 1), -1, np.int32)
    L = np.zeros(B, np.int32)
    bonus = np.zeros(B, np.int32)
    status = np.zeros(B, np.int32)
    for b in range(B):
        path, l, bo, st = accept_walk(parent[b], draft[b], am[b], max_depth)
        acc[b] = path
        L[b] = l
        bonus[b] = bo
        status[b] = st
    return acc, L, bonus, am, status
