"""Oracle: commit the accepted path's keys/values to the paged cache (test infrastructure only).

[P1] Key Mechanisms > Speculative KV Cache Reuse: the keys/values computed for
the tree nodes are reused rather than recomputed; Multi-Token Acceptance &
Rollback: the tokens of the accepted path are kept and the rejected branches
are discarded; Integration with Speculative Decoding: the accepted prefix is
appended to the output and generation continues from the new state.

Readings where the pages are silent:
  * The root is the last verified token and is attended as tree node 0 at
    position P_b, so it is not yet in the cache: the committed tokens are the
    path root, x1, ..., n* at positions P_b, P_b + 1, ..., P_b + L, and the new
    prefix length is P_b + L + 1.  Nothing else is written: discarding the
    rejected branches needs no work because their keys/values never entered
    the cache.
  * The position t goes to row (t mod bs) of block block_table[b, t div bs];
    the caller provides blocks for every position it may commit to.
  * A sequence whose verify status is not 0 commits nothing and keeps its
    prefix length.
"""
from __future__ import annotations

import numpy as np


def commit_accepted(k_tree, v_tree, accepted, accept_len, status, prefix_len, k_cache, v_cache, block_table):
    """Copy the accepted path's rows into (copies of) the caches.

    k_tree/v_tree [B, N, Hkv, D], accepted [B, max_depth+1] (node ids, root
    first), accept_len [B], status [B], prefix_len [B], k_cache/v_cache
    [blocks, Hkv, bs, D], block_table [B, max_blocks].
    Returns (k_cache', v_cache', new_prefix_len [B]).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    bs = kc.shape[2]
    B = len(prefix_len)
    new_len = np.array(prefix_len, np.int32, copy=True)
    for b in range(B):
        if int(status[b]) != 0:
            continue
        P = int(prefix_len[b])
        L = int(accept_len[b])
        for d in range(L + 1):
            node = int(accepted[b][d])
            t = P + d
            blk = int(block_table[b][t // bs])
            kc[blk, :, t % bs] = k_tree[b, node]
            vc[blk, :, t % bs] = v_tree[b, node]
        new_len[b] = P + L + 1
    return kc, vc, new_len
