"""Oracle: tree validity, ancestry mask, depth and positions (test infrastructure only).

[P1] Key Mechanisms > Modified Causal Attention Mask: a node sees every token on
its ancestral path back to the root and itself, and nothing from sibling
branches.  [P2] How It Works: a node may attend to the verified prefix, itself
and its ancestors, never to a sibling or a node of another branch.  [P3] code
listing, build_tree_attention_mask: a dense N x N boolean matrix, filled by
setting the diagonal and then walking parent pointers until the root's -1.

Readings where the pages are silent:
  * Flattened order is topological with a single root at index 0
    (parent[0] == -1, 0 <= parent[i] < i); the demo tree of [P3] is in this
    breadth-first order.  Anything else is an invalid tree.
  * Packing: mask row i is stored as W = ceil(N/64) little-endian uint64 words;
    node j is bit (j mod 64) of word (j div 64); bits for j >= N are zero.
  * [P2] Tradeoffs names "position bookkeeping" without a formula; the position
    of node i is prefix_len + depth(i), the root being the last verified token.
"""
from __future__ import annotations

import numpy as np

ERR_BAD_TREE = -3


def is_valid_tree(parent) -> bool:
    """Single root at index 0, every other node's parent strictly earlier."""
    parent = [int(p) for p in parent]
    n = len(parent)
    if n < 1 or parent[0] != -1:
        return False
    for i in range(1, n):
        if not (0 <= parent[i] < i):
            return False
    return True


def ancestry_matrix(parent) -> np.ndarray:
    """Explicit N x N bool mask by the page's walk: M[i,i]; then M[i,c] for every
    c reached by repeatedly following parent pointers until -1."""
    parent = [int(p) for p in parent]
    n = len(parent)
    m = np.zeros((n, n), dtype=bool)
    for i in range(n):
        m[i, i] = True
        c = parent[i]
        while c != -1:
            m[i, c] = True
            c = parent[c]
    return m


def depths(parent) -> np.ndarray:
    """Number of parent steps from each node to the root (the same walk, counted)."""
    parent = [int(p) for p in parent]
    out = np.zeros(len(parent), np.int64)
    for i in range(len(parent)):
        d, c = 0, parent[i]
        while c != -1:
            d += 1
            c = parent[c]
        out[i] = d
    return out


def pack_rows(m: np.ndarray) -> np.ndarray:
    """Pack each bool row into ceil(N/64) uint64 words, node j -> bit j%64 of word j//64."""
    n = m.shape[1]
    w = (n + 63) // 64
    words = np.zeros((m.shape[0], w), np.uint64)
    for i in range(m.shape[0]):
        for j in range(n):
            if m[i, j]:
                words[i, j // 64] |= np.uint64(1) << np.uint64(j % 64)
    return words


def build_ancestry(parent: np.ndarray, prefix_len: np.ndarray):
    """Per sequence: packed ancestry words, depth, position and a status code.

    parent [B, N] int, prefix_len [B] int -> anc [B, N, W] uint64, depth [B, N] int32,
    pos [B, N] int32, status [B] int32 (0, or -3 for an invalid tree; the other
    outputs of an invalid sequence are unspecified and reported here as zeros).
    """
    parent = np.asarray(parent)
    B, N = parent.shape
    W = (N + 63) // 64
    anc = np.zeros((B, N, W), np.uint64)
    dep = np.zeros((B, N), np.int32)
    pos = np.zeros((B, N), np.int32)
    status = np.zeros(B, np.int32)
    for b in range(B):
        if not is_valid_tree(parent[b]):
            status[b] = ERR_BAD_TREE
            continue
        anc[b] = pack_rows(ancestry_matrix(parent[b]))
        dep[b] = depths(parent[b])
        pos[b] = int(prefix_len[b]) + dep[b]
    return anc, dep, pos, status


def mask_sparsity(m: np.ndarray) -> float:
    """Fraction of masked-out entries, as printed by the [P3] demo."""
    return float((~m).mean())
