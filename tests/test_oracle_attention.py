"""Pins for the oracle's tree attention.

The pages fix two facts that can be checked without the oracle's own loop:
each node's result must equal ordinary causal attention run over the prefix
followed by its own root-to-node path ([P2] How It Works: a node's state
matches its own root-to-node history; [P1] Modified Causal Attention Mask: the
autoregressive property holds within each candidate sequence), and a chain
tree is plain causal attention.  Those are computed here with torch's
scaled_dot_product_attention in fp64 on the CPU, on keys gathered from the
paged pool by vectorised indexing (not the oracle's gather).  Further pins:
single-token decode for N = 1, constant values, lse by scipy's logsumexp, and
relabelling invariance.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

from oracle import attention as A
from oracle import tree as T
import workloads as W


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _prefix_vectorised(cache, table, b, g, plen, bs):
    t = np.arange(plen)
    return _f64(cache[table[b, t // bs], g, t % bs])


def _path(parent, i):
    out = []
    while i != -1:
        out.append(i)
        i = parent[i]
    return out[::-1]


def _case(seed, B, N, Hq, Hkv, D, plens, bs, tree="random", permute=True):
    g = W.rng(seed, "tree")
    if tree == "random":
        parent = np.stack([W.tree_random_recursive(g, N) for _ in range(B)])
    elif tree == "chain":
        parent = W.tree_chain(N)
    elif tree == "star":
        parent = W.tree_star(N)
    else:
        parent = tree
    return W.build_case("t", seed, parent, plens, Hq=Hq, Hkv=Hkv, D=D, bs=bs, permute=permute)


def _sdpa_last_rows(qrows, keys, vals, scale):
    """Causal SDPA over a sequence whose last len(qrows) positions carry the queries."""
    S = keys.shape[0]
    L = qrows.shape[0]
    D = keys.shape[1]
    q = torch.zeros(1, 1, S, D, dtype=torch.float64)
    q[0, 0, S - L:] = torch.from_numpy(qrows)
    k = torch.from_numpy(keys)[None, None]
    v = torch.from_numpy(vals)[None, None]
    o = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=scale)
    return o[0, 0, S - L:].numpy()


@pytest.mark.parametrize("seed,B,N,Hq,Hkv,D,plens,bs", [
    (1, 2, 9, 4, 2, 16, [0, 21], 8),
    (2, 1, 17, 6, 3, 32, [40], 16),
    (3, 3, 5, 2, 2, 64, [16, 1, 33], 16),
])
def test_each_node_equals_causal_attention_on_its_path(seed, B, N, Hq, Hkv, D, plens, bs):
    c = _case(seed, B, N, Hq, Hkv, D, plens, bs)
    out, lse = A.tree_attention_case(c)
    G = Hq // Hkv
    for b in range(B):
        for i in range(N):
            path = _path(c.parent[b], i)
            for h in range(Hq):
                g = h // G
                kp = _prefix_vectorised(c.k_cache, c.block_table, b, g, plens[b], bs)
                vp = _prefix_vectorised(c.v_cache, c.block_table, b, g, plens[b], bs)
                keys = np.concatenate([kp, _f64(c.k_tree[b, path, g])])
                vals = np.concatenate([vp, _f64(c.v_tree[b, path, g])])
                ref = _sdpa_last_rows(_f64(c.q[b, i, h])[None], keys, vals, c.scale)[0]
                np.testing.assert_allclose(out[b, i, h], ref, rtol=1e-12, atol=1e-12)
                s = c.scale * keys @ _f64(c.q[b, i, h])
                assert abs(lse[b, i, h] - logsumexp(s)) < 1e-10


def test_chain_tree_is_full_causal_attention():
    N, P, D = 12, 19, 32
    c = _case(5, 1, N, 2, 1, D, [P], 8, tree="chain")
    out, _ = A.tree_attention_case(c)
    kp = _prefix_vectorised(c.k_cache, c.block_table, 0, 0, P, 8)
    vp = _prefix_vectorised(c.v_cache, c.block_table, 0, 0, P, 8)
    keys = np.concatenate([kp, _f64(c.k_tree[0, :, 0])])
    vals = np.concatenate([vp, _f64(c.v_tree[0, :, 0])])
    for h in range(2):
        ref = _sdpa_last_rows(_f64(c.q[0, :, h]), keys, vals, c.scale)
        np.testing.assert_allclose(out[0, :, h], ref, rtol=1e-12, atol=1e-12)


def test_single_node_is_single_token_decode():
    c = _case(6, 2, 1, 8, 2, 64, [100, 3], 16)
    out, _ = A.tree_attention_case(c)
    for b in range(2):
        for h in range(8):
            g = h // 4
            keys = np.concatenate([_prefix_vectorised(c.k_cache, c.block_table, b, g, c.prefix_len[b], 16),
                                   _f64(c.k_tree[b, :1, g])])
            vals = np.concatenate([_prefix_vectorised(c.v_cache, c.block_table, b, g, c.prefix_len[b], 16),
                                   _f64(c.v_tree[b, :1, g])])
            q = torch.from_numpy(_f64(c.q[b, 0, h]))[None, None, None]
            ref = F.scaled_dot_product_attention(q, torch.from_numpy(keys)[None, None],
                                                 torch.from_numpy(vals)[None, None], scale=c.scale)
            np.testing.assert_allclose(out[b, 0, h], ref[0, 0, 0].numpy(), rtol=1e-12, atol=1e-12)


def test_star_tree_sees_prefix_root_and_self():
    c = _case(7, 1, 6, 2, 2, 16, [10], 16, tree="star")
    out, _ = A.tree_attention_case(c)
    for i in range(6):
        vis = [0] if i == 0 else [0, i]
        for h in range(2):
            keys = np.concatenate([_prefix_vectorised(c.k_cache, c.block_table, 0, h, 10, 16), _f64(c.k_tree[0, vis, h])])
            vals = np.concatenate([_prefix_vectorised(c.v_cache, c.block_table, 0, h, 10, 16), _f64(c.v_tree[0, vis, h])])
            s = c.scale * keys @ _f64(c.q[0, i, h])
            p = np.exp(s - s.max())
            np.testing.assert_allclose(out[0, i, h], p @ vals / p.sum(), rtol=1e-12, atol=1e-12)


def test_constant_values_give_that_constant():
    c = _case(8, 2, 7, 4, 1, 16, [5, 0], 4)
    val = W.bf16_bits(np.float32(0.375) * np.ones(16, np.float32))
    c.v_cache[:] = val
    c.v_tree[:] = val
    out, _ = A.tree_attention_case(c)
    np.testing.assert_allclose(out, 0.375, rtol=0, atol=1e-15)


def test_zero_prefix_root_sees_only_itself():
    c = _case(9, 1, 4, 2, 2, 8, [0], 16)
    out, lse = A.tree_attention_case(c)
    np.testing.assert_array_equal(out[0, 0, 1], _f64(c.v_tree[0, 0, 1]))
    s = c.scale * _f64(c.q[0, 0, 1]) @ _f64(c.k_tree[0, 0, 1])
    assert abs(lse[0, 0, 1] - s) < 1e-12


def test_relabelling_permutes_rows():
    # two topological numberings of the same tree: swap the subtrees of the root's children
    p1 = np.array([-1, 0, 0, 1, 2, 3])
    p2 = np.array([-1, 0, 0, 1, 2, 4])    # new 1 = old 2, new 3 = old 4 (under new 1), new 5 under new 4 = old 3
    perm = [0, 2, 1, 4, 3, 5]            # new index k holds old node perm[k]
    c1 = W.build_case("t", 11, p1, [9], Hq=2, Hkv=1, D=16, bs=4, permute=True)
    c2 = W.build_case("t", 11, p2, [9], Hq=2, Hkv=1, D=16, bs=4, permute=True)
    for name in ("q", "k_tree", "v_tree"):
        getattr(c2, name)[0] = getattr(c1, name)[0][perm]
    assert (T.ancestry_matrix(p2)[np.ix_(range(6), range(6))] ==
            T.ancestry_matrix(p1)[np.ix_(perm, perm)]).all()
    o1, _ = A.tree_attention_case(c1)
    o2, _ = A.tree_attention_case(c2)
    np.testing.assert_allclose(o2[0], o1[0][perm], rtol=1e-13, atol=1e-13)


def test_gqa_grouping_is_consecutive():
    # with Hq=4, Hkv=2: heads 0,1 read kv head 0; heads 2,3 read kv head 1
    c = _case(12, 1, 3, 4, 2, 16, [6], 8)
    c.k_cache[:, 1] = 0
    c.k_tree[:, :, 1] = 0          # kv head 1 keys all zero -> uniform weights over visible keys
    out, _ = A.tree_attention_case(c)
    vp = _prefix_vectorised(c.v_cache, c.block_table, 0, 1, 6, 8)
    for i in range(3):
        vis = _path(c.parent[0], i)
        vals = np.concatenate([vp, _f64(c.v_tree[0, vis, 1])])
        for h in (2, 3):
            np.testing.assert_allclose(out[0, i, h], vals.mean(0), rtol=1e-12, atol=1e-12)
