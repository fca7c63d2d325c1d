"""Numerics of the split combine as the kernels store it (CPU).

The attention kernel leaves, per split of the prefix, a normalised partial
output in bf16 and its log-sum-exp in fp32; the combine merges them as
    out = sum_s 2^(L_s - M) O_s / sum_s 2^(L_s - M).
This models exactly those roundings in numpy (partials rounded to bf16 with
round-to-nearest-even, lse rounded to fp32, the merged output rounded to bf16)
and checks the result against the fp64 softmax over all keys, on the value
distributions of the workloads (N(0,1), and 1% of key rows scaled by 8), with
as many splits as the planner uses.  The error must stay well inside the
parity bound 1e-2 + 1e-2 |ref| (under half of it), leaving the rest for the
kernel's other roundings (bf16 P, fp32 accumulation)."""
import numpy as np
import pytest

import workloads as W

ATOL, RTOL = 1e-2, 1e-2


def bf16(x):
    return (W.bf16_bits(np.asarray(x, np.float32)).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def reference(q, k, v, scale):
    s = scale * q @ k.T
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    return (p @ v) / p.sum(axis=1, keepdims=True)


def split_combine(q, k, v, scale, splits):
    parts, lses = [], []
    for ks, vs in zip(np.array_split(k, splits), np.array_split(v, splits)):
        s = scale * np.log2(np.e) * q @ ks.T              # base-2 scores, as the kernel
        m = s.max(axis=1, keepdims=True)
        p = np.exp2(s - m)
        l = p.sum(axis=1, keepdims=True)
        parts.append(bf16((p @ vs) / l))                   # bf16 partial
        lses.append(np.float32(m + np.log2(l)).astype(np.float64))  # fp32 lse
    L = np.stack(lses)                                     # [S, R, 1]
    M = L.max(axis=0)
    w = np.exp2(L - M)
    out = (w * np.stack(parts)).sum(axis=0) / w.sum(axis=0)
    return bf16(out)


@pytest.mark.parametrize("rows,keys,splits,hot", [(64, 4096, 9, 0.0), (104, 16384, 4, 0.0), (96, 16384, 7, 0.01),
                                                 (64, 2048, 17, 0.01)])
def test_bf16_partials_stay_inside_half_the_bound(rows, keys, splits, hot):
    g = np.random.default_rng(rows + keys + splits)
    D = 128
    q = bf16(g.standard_normal((rows, D)))
    k = g.standard_normal((keys, D))
    if hot:
        k[g.random(keys) < hot] *= 8.0
    k = bf16(k)
    v = bf16(g.standard_normal((keys, D)))
    scale = 1.0 / np.sqrt(D)
    ref = reference(q, k, v, scale)
    got = split_combine(q, k, v, scale, splits)
    ratio = np.abs(got - ref) / (ATOL + RTOL * np.abs(ref))
    assert ratio.max() < 0.5, ratio.max()


def test_one_split_is_the_plain_softmax():
    g = np.random.default_rng(3)
    q, k, v = (bf16(g.standard_normal(s)) for s in ((8, 64), (300, 64), (300, 64)))
    got = split_combine(q, k, v, 0.125, 1)
    np.testing.assert_allclose(got, bf16(reference(q, k, v, 0.125)), rtol=0, atol=0)
