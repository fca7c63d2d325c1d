"""Oracle: stochastic (temperature) verification of a scored draft tree (test infrastructure only).

[P3] Production Inference Runtimes section: every accepted token is checked
against the target model's own probability distribution by rejection sampling,
so the emitted text has exactly the distribution of plain autoregressive
decoding.  [P3] code listing, verify_candidate_tree (its comment): the target's
prediction is greedy or temperature-sampled.  [P1] Key Mechanisms >
Multi-Token Acceptance & Rollback: the walk keeps the accepted branch up to the
first rejection and discards the rest.

The pages give no rule for several drafts under one node.  The reading taken
here is recursive rejection sampling over the siblings, the drafts of a node
having been drawn from the draft distribution without replacement (which is
what distinct sibling tokens imply):

  * p_u = softmax(target_logits[u] / T) is the target distribution after
    node u; q_u = draft_probs[u] is the distribution u's children were drawn
    from, used as given.
  * Walk from the root.  At node u start with r = p_u and q' = q_u; try u's
    children c in increasing index order, with x = draft[c]:
      - accept c iff coins[c] * q'(x) < r(x)   (probability min(1, r(x)/q'(x)));
        then c joins the path and the walk moves to c;
      - otherwise r <- max(r - q', 0) renormalised (kept unchanged if that
        leaves no mass, which only rounding can cause), and x leaves the draft
        distribution: q'(x) <- 0, q' renormalised to the remaining mass (all
        zero if none remains).
  * The walk ends at a node with no children, or when every child of u was
    rejected.  The bonus token is then drawn from r by inversion with
    coins[0]: the smallest v with r(0) + ... + r(v) > coins[0] (the last v
    with r(v) > 0 if rounding leaves none).
  * accepted = the path root .. n*, padded with -1 to max_depth + 1 entries;
    accept_len = depth(n*).  If depth(n*) > max_depth the row stays all -1,
    accept_len and bonus are still reported and the status is -2.  An invalid
    tree, or a draft token outside [0, V) on a node other than the root, gives
    status -3, an all -1 row and zeros.

Each step is the single-draft speculative sampling step applied to the current
residual, so the first token the walk emits (an accepted draft or the bonus)
is distributed as p_root whatever q is; tests check that by sampling.

For the tests the walk also returns two decision margins: how close any
acceptance comparison came to going the other way (relative to the larger side
compared), and how far coins[0] fell from the nearest boundary of the inversion
(in units of probability mass).  A fp32 implementation takes the same decisions
wherever a margin is well above its rounding.  Over a large vocabulary the
inversion margin is of the order of one token's probability, so a fp32 sum may
legitimately pick a neighbouring token; the tests then check that the token
picked lies within rounding of the inversion boundaries of ``final``, the
distribution the bonus was drawn from.
"""
from __future__ import annotations

import numpy as np

from .tree import is_valid_tree

ERR_SHAPE = -2
ERR_BAD_TREE = -3


def target_probs(logits_row, temperature: float) -> np.ndarray:
    """softmax(l / T) in fp64 from the fp32 logits."""
    z = np.asarray(logits_row, np.float64) / float(temperature)
    e = np.exp(z - z.max())
    return e / e.sum()


def sample_inverse(r: np.ndarray, coin: float):
    """Smallest v with cumsum(r)[v] > coin; returns (v, margin)."""
    c = np.cumsum(r)
    hit = np.nonzero(c > coin)[0]
    if len(hit) == 0:
        pos = np.nonzero(r > 0)[0]
        return int(pos[-1]), 0.0
    v = int(hit[0])
    lo = c[v - 1] if v > 0 else 0.0
    return v, float(min(coin - lo, c[v] - coin) / c[-1])


def walk_stochastic(parent, draft, logits, q, coins, temperature: float, max_depth: int, final: bool = False):
    """One tree.  logits [N, V] fp32, q [N, V] draft probabilities, coins [N] in [0, 1).
    Returns (path[max_depth + 1], accept_len, bonus, status, accept_margin, sample_margin),
    plus the bonus token's distribution when ``final``."""
    parent = [int(p) for p in parent]
    n = len(parent)
    path = np.full(max_depth + 1, -1, np.int32)
    V = np.asarray(logits).shape[-1]
    if not is_valid_tree(parent) or any(not (0 <= int(draft[c]) < V) for c in range(1, n)):
        out = (path, 0, 0, ERR_BAD_TREE, np.inf, np.inf)
        return out + (None,) if final else out
    kids = [[c for c in range(n) if parent[c] == u] for u in range(n)]
    acc_margin = np.inf
    walk = [0]
    u = 0
    while True:
        r = target_probs(logits[u], temperature)
        qc = np.array(q[u], np.float64, copy=True)
        nxt = -1
        for c in kids[u]:
            x = int(draft[c])
            a = float(coins[c]) * qc[x]
            b = r[x]
            acc_margin = min(acc_margin, abs(a - b) / max(a, b) if max(a, b) > 0 else 0.0)
            if a < b:
                nxt = c
                break
            res = np.maximum(r - qc, 0.0)
            s = res.sum()
            if s > 0:
                r = res / s
            left = 1.0 - qc[x]
            qc[x] = 0.0
            qc = qc / left if left > 0 else np.zeros_like(qc)
        if nxt < 0:
            bonus, smp_margin = sample_inverse(r, float(coins[0]))
            break
        walk.append(nxt)
        u = nxt
    L = len(walk) - 1
    status = 0
    if L > max_depth:
        status = ERR_SHAPE
    else:
        path[: L + 1] = walk
    out = (path, L, bonus, status, acc_margin, smp_margin)
    return out + (r,) if final else out


def verify_stochastic(draft, logits, q, parent, coins, temperature: float, max_depth: int):
    """Batched: draft [B,N], logits [B,N,V] fp32, q [B,N,V], parent [B,N], coins [B,N] ->
    accepted [B,max_depth+1], accept_len [B], bonus [B], status [B],
    margins [B, 2] (acceptance, inversion)."""
    draft = np.asarray(draft)
    parent = np.asarray(parent)
    B, N = draft.shape
    acc = np.full((B, max_depth + 1), -1, np.int32)
    L = np.zeros(B, np.int32)
    bonus = np.zeros(B, np.int32)
    status = np.zeros(B, np.int32)
    margin = np.zeros((B, 2), np.float64)
    for b in range(B):
        acc[b], L[b], bonus[b], status[b], margin[b, 0], margin[b, 1] = walk_stochastic(
            parent[b], draft[b], logits[b], q[b], coins[b], temperature, max_depth)
    return acc, L, bonus, status, margin
