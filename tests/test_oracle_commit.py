"""Pins for the oracle's commit of the accepted path.

The pages imply one exact check: after the accepted path is appended to the
cache, the deepest accepted node's output is ordinary single-query decode
attention over the new prefix (its tree-attention row saw exactly the prefix
and its root path, which is what was committed).  Also closed forms on chains
and the untouched rest of the pool.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as W


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(seed, B, N, plant, bs=16, P=(37, 5, 64), depth=6, vocab=300):
    g = W.rng(seed, "commit")
    parents = np.stack([W.tree_random_levels(g, N, depth) for _ in range(B)])
    return W.build_case("commit", seed, parents, list(P)[:B], Hq=4, Hkv=2, D=32, bs=bs, permute=True,
                        vocab=vocab, plant_len=plant, spare_tokens=depth + 1)


def _commit(c, max_depth):
    acc, L, bonus, am, st = oracle.verify.verify_greedy(c.draft, c.logits, c.parent, max_depth)
    kc, vc, new_len = oracle.commit.commit_accepted(c.k_tree, c.v_tree, acc, L, st, c.prefix_len, c.k_cache,
                                                    c.v_cache, c.block_table)
    return acc, L, st, kc, vc, new_len


@pytest.mark.parametrize("seed,plant", [(1, [3, 0, 6]), (2, [1, 5, 2]), (3, [6, 6, 0])])
def test_deepest_node_equals_decode_over_committed_cache(seed, plant):
    c = _case(seed, 3, 24, plant)
    acc, L, st, kc, vc, new_len = _commit(c, 6)
    assert L.tolist() == plant and (new_len == c.prefix_len + L + 1).all()
    out, _ = oracle.attention.tree_attention_case(c)
    G = c.Hq // c.Hkv
    for b in range(c.B):
        nstar = int(acc[b, L[b]])
        t = np.arange(int(new_len[b]))
        for h in range(c.Hq):
            g = h // G
            keys = _f64(kc[c.block_table[b, t // c.bs], g, t % c.bs])
            vals = _f64(vc[c.block_table[b, t // c.bs], g, t % c.bs])
            q = torch.from_numpy(_f64(c.q[b, nstar, h]))[None, None, None]
            ref = F.scaled_dot_product_attention(q, torch.from_numpy(keys)[None, None],
                                                 torch.from_numpy(vals)[None, None], scale=c.scale)
            np.testing.assert_allclose(out[b, nstar, h], ref[0, 0, 0].numpy(), rtol=1e-12, atol=1e-12)


def test_chain_commits_nodes_in_order_and_nothing_else():
    N, P, L = 8, 13, 5
    c = W.build_case("chain", 4, W.tree_chain(N), [P], Hq=2, Hkv=2, D=16, bs=8, permute=True, vocab=50,
                     plant_len=[L], spare_tokens=N)
    acc, Ls, st, kc, vc, new_len = _commit(c, N - 1)
    assert Ls.tolist() == [L] and new_len.tolist() == [P + L + 1]
    for d in range(L + 1):
        t = P + d
        blk = c.block_table[0, t // 8]
        assert (kc[blk, :, t % 8] == c.k_tree[0, d]).all() and (vc[blk, :, t % 8] == c.v_tree[0, d]).all()
    # every other pool row is untouched
    touched = np.zeros(kc.shape[:3], bool)
    for d in range(L + 1):
        t = P + d
        touched[c.block_table[0, t // 8], :, t % 8] = True
    assert (kc[~touched] == c.k_cache[~touched]).all() and (vc[~touched] == c.v_cache[~touched]).all()


def test_failed_sequence_commits_nothing():
    c = _case(5, 2, 10, [2, 3], P=(20, 9))
    acc, L, bonus, am, st = oracle.verify.verify_greedy(c.draft, c.logits, c.parent, 6)
    st = np.array([0, -3], np.int32)
    kc, vc, new_len = oracle.commit.commit_accepted(c.k_tree, c.v_tree, acc, L, st, c.prefix_len, c.k_cache,
                                                    c.v_cache, c.block_table)
    assert new_len.tolist() == [20 + 2 + 1, 9]
    blk_rows = {(int(c.block_table[1, t // 16]), t % 16) for t in range(9, 9 + 7)}
    for blk, row in blk_rows:
        assert (kc[blk, :, row] == c.k_cache[blk, :, row]).all()
