"""Oracle: tree-masked attention over the verified prefix and the tree (test infrastructure only).

What one attention layer of the verification pass computes ([P1] Key
Mechanisms > Batched Parallel Verification and Modified Causal Attention Mask;
[P2] How It Works): for sequence b, query head h and tree node i, the keys are
the whole verified prefix of b followed by the tree nodes j that the ancestry
mask lets node i see (its ancestors and itself).  Softmax attention in fp64:

    s_t = scale * <q[b,i,h], k_t>,  m = max_t s_t,  p_t = exp(s_t - m)
    out[b,i,h] = sum_t p_t v_t / sum_t p_t,   lse[b,i,h] = m + ln sum_t p_t

Readings where the pages are silent:
  * Grouped-query attention: query head h reads KV head h // (Hq/Hkv)
    (consecutive grouping).
  * scale defaults to 1/sqrt(head_dim).
  * Prefix token t of sequence b lives in the paged pool at
    cache[block_table[b, t // bs], kv_head, t % bs, :] (pool [blocks, Hkv, bs, D]).
  * Tree keys/values are inputs k_tree/v_tree [B, N, Hkv, D] ([P1] Speculative
    KV Cache Reuse leaves their provenance to the runtime).
  * Masked-out tree keys contribute nothing; every row sees at least itself.
  * No rotary embedding is applied: the inputs are taken as already positioned.

Inputs are bf16 bit patterns (uint16), widened exactly to fp64 here.
"""
from __future__ import annotations

import numpy as np

from .tree import ancestry_matrix


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def prefix_kv(cache_bits: np.ndarray, block_table: np.ndarray, b: int, g: int, plen: int, bs: int) -> np.ndarray:
    """Gather the prefix rows of sequence b, KV head g, token by token: [plen, D] fp64."""
    D = cache_bits.shape[-1]
    out = np.empty((plen, D), np.float64)
    for t in range(plen):
        blk = int(block_table[b, t // bs])
        out[t] = bf16_to_f64(cache_bits[blk, g, t % bs])
    return out


def attend_rows(q_rows: np.ndarray, keys: np.ndarray, vals: np.ndarray, visible: np.ndarray, scale: float):
    """Softmax attention of each query row over the key rows it may see.

    q_rows [R, D], keys/vals [T, D], visible [R, T] bool -> out [R, D], lse [R].
    """
    s = scale * (q_rows @ keys.T)
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)                       # exp(-inf) = 0 for masked keys
    l = p.sum(axis=1, keepdims=True)
    out = (p @ vals) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def tree_attention(q, k_cache, v_cache, block_table, prefix_len, k_tree, v_tree, parent,
                   scale=None, units=None):
    """fp64 tree attention for every (b, node, head), or only for the given units.

    q [B,N,Hq,D], k/v_cache [blocks,Hkv,bs,D], k/v_tree [B,N,Hkv,D]: bf16 bits.
    block_table [B, max_blocks] int, prefix_len [B] int, parent [B,N] int.
    ``units``: optional iterable of (b, kv_head); rows outside them are NaN.
    Returns out [B,N,Hq,D] fp64 and lse [B,N,Hq] fp64 (natural log).
    """
    B, N, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    bs = k_cache.shape[2]
    G = Hq // Hkv
    if scale is None or scale == 0.0:
        scale = 1.0 / np.sqrt(D)
    out = np.full((B, N, Hq, D), np.nan)
    lse = np.full((B, N, Hq), np.nan)
    if units is None:
        units = [(b, g) for b in range(B) for g in range(Hkv)]
    masks = {}
    for b, g in units:
        if b not in masks:
            masks[b] = ancestry_matrix(parent[b])
        m = masks[b]
        plen = int(prefix_len[b])
        kp = prefix_kv(k_cache, block_table, b, g, plen, bs)
        vp = prefix_kv(v_cache, block_table, b, g, plen, bs)
        kt = bf16_to_f64(k_tree[b, :, g])
        vt = bf16_to_f64(v_tree[b, :, g])
        keys = np.concatenate([kp, kt], axis=0)
        vals = np.concatenate([vp, vt], axis=0)
        for hh in range(G):
            h = g * G + hh
            qr = bf16_to_f64(q[b, :, h])                     # [N, D]
            visible = np.concatenate([np.ones((N, plen), bool), m], axis=1)
            o, l = attend_rows(qr, keys, vals, visible, scale)
            out[b, :, h] = o
            lse[b, :, h] = l
    return out, lse


def tree_attention_case(case, units=None):
    """Convenience wrapper over a ``workloads.Case``."""
    return tree_attention(case.q, case.k_cache, case.v_cache, case.block_table, case.prefix_len,
                          case.k_tree, case.v_tree, case.parent, case.scale, units=units)
