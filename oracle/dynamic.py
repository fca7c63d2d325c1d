"""Oracle: dynamic draft-tree construction by reranking (test infrastructure only).

[P2] Common Confusions: the tree shape may be fixed, learned or selected
dynamically; Where It Appears (EAGLE-2, context-aware dynamic draft trees): the
tree changes per context and the ancestry mask is built after reranking.
[P1] Key Mechanisms > Tree-Structured Candidate Generation: the draft proposes
several continuations at each branching point, giving a prefix tree.  [P2]
Tradeoffs: tree construction and flattening are part of the cost.

The pages give no procedure.  The reading taken here:

  * Input: a candidate pool already expanded by the draft, in topological
    order (pool_parent[0] = -1 is the root, the last verified token; every
    other candidate's parent has a smaller index), with the draft's
    log-probability of each candidate given its parent (<= 0) and its token.
  * A candidate's value is the draft's log-probability of its whole path:
    value(root) = 0, value(c) = value(parent(c)) + logp(c), accumulated from
    the root down in fp32 (the precision the GPU works in, so that both sides
    rank identically).
  * Reranking keeps the root and the N - 1 candidates of highest value, ties
    to the smaller pool index.  Because logp <= 0 a parent's value is at least
    its child's and its index smaller, so the kept set contains every kept
    node's parent: it is a tree.
  * Flattening keeps the pool order of the kept candidates (topological);
    node k of the tree is the k-th kept candidate.  Then the ancestry mask,
    depths and positions of that tree follow as for any tree.
  * A pool that is not topological, has a positive or NaN log-probability, or
    is smaller than N is invalid: status -3, outputs unspecified (zeros here).

Under the model in which a drafted token is accepted with the probability the
draft gave it, exp(value(c)) is the chance that c is accepted, and the kept
set maximises the expected number of accepted tokens over all trees of N
nodes cut from the pool; the tests check that by brute force.
"""
from __future__ import annotations

import numpy as np

from .tree import ancestry_matrix, depths, pack_rows

ERR_BAD_TREE = -3


def pool_valid(pool_parent, pool_logp, n: int) -> bool:
    par = [int(p) for p in pool_parent]
    m = len(par)
    if m < n or n < 1 or par[0] != -1:
        return False
    for c in range(1, m):
        if not (0 <= par[c] < c):
            return False
        lp = float(pool_logp[c])
        if not (lp <= 0.0):  # positive or NaN
            return False
    return True


def path_values(pool_parent, pool_logp) -> np.ndarray:
    """value(c) = value(parent) + logp(c), root 0, in fp32 from the root down."""
    m = len(pool_parent)
    v = np.zeros(m, np.float32)
    for c in range(1, m):
        v[c] = np.float32(v[int(pool_parent[c])] + np.float32(pool_logp[c]))
    return v


def rerank(pool_parent, pool_logp, n: int) -> np.ndarray:
    """Pool indices of the kept candidates, in pool order (the root first)."""
    v = path_values(pool_parent, pool_logp)
    order = sorted(range(len(v)), key=lambda c: (-float(v[c]), c))
    return np.array(sorted(order[:n]), np.int64)


def build_dynamic(pool_parent, pool_logp, pool_token, prefix_len, n: int):
    """Batched: pool_parent/logp/token [B, M] -> parent [B, n], tokens [B, n],
    sel [B, n] (pool index of each tree node), anc [B, n, W], depth [B, n],
    pos [B, n], status [B]."""
    pool_parent = np.asarray(pool_parent)
    B = pool_parent.shape[0]
    W = (n + 63) // 64
    parent = np.zeros((B, n), np.int32)
    tokens = np.zeros((B, n), np.int32)
    sel = np.zeros((B, n), np.int32)
    anc = np.zeros((B, n, W), np.uint64)
    dep = np.zeros((B, n), np.int32)
    pos = np.zeros((B, n), np.int32)
    status = np.zeros(B, np.int32)
    for b in range(B):
        if not pool_valid(pool_parent[b], pool_logp[b], n):
            status[b] = ERR_BAD_TREE
            continue
        keep = rerank(pool_parent[b], pool_logp[b], n)
        new = {int(c): k for k, c in enumerate(keep)}
        par = [-1 if k == 0 else new[int(pool_parent[b][c])] for k, c in enumerate(keep)]
        parent[b] = par
        tokens[b] = np.asarray(pool_token[b])[keep]
        sel[b] = keep
        anc[b] = pack_rows(ancestry_matrix(par))
        dep[b] = depths(par)
        pos[b] = int(prefix_len[b]) + dep[b]
    return parent, tokens, sel, anc, dep, pos, status
