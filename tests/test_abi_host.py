"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching a GPU.  None of
these calls launches a kernel, so they run without a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ts():
    from tree_attention_speculative_gb300 import _build
    _build.build()
    import tree_attention_speculative_gb300 as ts
    ts.lib()
    return ts


def _header_symbols():
    src = open(os.path.join(ROOT, "include", "treespec.h")).read()
    return sorted(set(re.findall(r"TS_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)))


def test_header_declares_the_expected_calls():
    syms = _header_symbols()
    for name in ("tree_build_ancestry", "tree_attn_fwd", "tree_verify_greedy"):
        assert name in syms


def test_library_exports_every_header_symbol(ts):
    L = ts.lib()
    syms = _header_symbols()
    assert syms, "no declarations found"
    for name in syms:
        assert hasattr(L, name), name
    assert sorted(ts.EXPORTS) == syms


def test_status_strings(ts):
    for code in range(-8, 1):
        assert ts.ts_status_str(code)
    assert "invalid tree" in ts.ts_status_str(-3)


class _FakeTensor:
    """Stands in for a device tensor on a GPU-less host: shape + a fake aligned address."""
    def __init__(self, shape, addr=0x10000):
        self.shape = shape
        self._addr = addr

    def data_ptr(self):
        return self._addr

    def cpu(self):
        return self


def _params(ts, B=2, N=26, Hq=32, Hkv=8, D=128, bs=16, P=(1000, 3000), **kw):
    nblk = max(1, sum(-(-p // bs) for p in P))
    maxb = max(1, max(-(-p // bs) for p in P))
    f = _FakeTensor
    args = dict(q=f((B, N, Hq, D)), k_cache=f((nblk, Hkv, bs, D)), v_cache=f((nblk, Hkv, bs, D)),
                block_table=f((B, maxb)), prefix_len=f((B,)), prefix_len_host=np.array(P, np.int32),
                k_tree=f((B, N, Hkv, D)), v_tree=f((B, N, Hkv, D)), anc_mask=f((B, N, 1)), pos=f((B, N)),
                out=f((B, N, Hq, D)), lse=None, status=f((B,)))
    args.update(kw)
    return ts.attn_params(**args)


def test_attn_workspace_query_and_plan(ts):
    p = _params(ts)
    n = ts.tree_attn_workspace_size(p)
    assert n > 0 and n % 256 == 0
    # bf16 partial outputs of at least two splits of every output row
    assert n >= 2 * 26 * 32 * 128 * 2


def test_attn_plan_query(ts):
    p = _params(ts)
    plan = ts.tree_attn_plan(p)
    assert plan["chunk_tiles"] >= 1 and plan["max_splits"] >= 1 and plan["tree_split"] in (0, 1)
    assert ts.lib().tree_attn_plan(ctypes.byref(p), None, None, None) == 0
    bad = _params(ts, D=96)
    assert ts.lib().tree_attn_plan(ctypes.byref(bad), None, None, None) == -4


@pytest.mark.parametrize("B,N,Hq,Hkv,D,bs,P", [
    (1, 64, 32, 8, 128, 4096, (4096,)),                  # c2-shaped: one wave, tree on its own split
    (16, 26, 32, 8, 128, 16, tuple(range(1024, 16385, 1024))),
    (64, 64, 64, 8, 128, 16, (8192,) * 64),              # many waves: one split per unit
    (4, 192, 32, 8, 128, 64, (131072,) * 4),
    (3, 5, 2, 2, 64, 16, (0, 0, 0)),                     # no prefix at all
    (2, 256, 1, 1, 64, 16, (0, 5000)),
])
def test_attn_plan_covers_the_prefix_and_sizes_the_workspace(ts, B, N, Hq, Hkv, D, bs, P):
    p = _params(ts, B=B, N=N, Hq=Hq, Hkv=Hkv, D=D, bs=bs, P=P)
    plan = ts.tree_attn_plan(p)
    chunk, splits, tsplit = plan["chunk_tiles"], plan["max_splits"], plan["tree_split"]
    tiles = max(-(-x // 128) for x in P)
    # the prefix splits of the longest sequence hold all its tiles, and no split is empty
    assert chunk * (splits - tsplit) >= tiles
    if tiles:
        assert chunk * (splits - tsplit - 1) < tiles
    else:
        assert splits == 1
    rows = B * N * Hq
    ws = ts.tree_attn_workspace_size(p)
    # 256 bytes for the persistent kernel's item counter, then the partials
    if splits == 1:
        assert ws == 256
    else:
        r256 = lambda x: -(-x // 256) * 256
        assert ws == 256 + r256(splits * rows * D * 2) + r256(splits * rows * 4)


def test_attn_plan_gives_the_tree_its_own_split_on_one_wave(ts):
    plan = ts.tree_attn_plan(_params(ts, B=1, N=64, Hq=32, Hkv=8, D=128, bs=4096, P=(4096,)))
    assert plan == {"chunk_tiles": 4, "max_splits": 9, "tree_split": 1}
    plan = ts.tree_attn_plan(_params(ts, B=64, N=64, Hq=64, Hkv=8, D=128, bs=16, P=(8192,) * 64))
    assert plan["max_splits"] == 1 and plan["tree_split"] == 0


def test_attn_plan_keeps_one_split_when_a_combine_would_cost_more(ts):
    """A split plan pays the combine kernel's launch whatever its size: the
    5-node demo tree on a 16-token prefix runs as one split with the tree
    block on it (a split of its own would save one tile and add a kernel)."""
    plan = ts.tree_attn_plan(_params(ts, B=1, N=5, Hq=2, Hkv=2, D=64, bs=16, P=(16,)))
    assert plan == {"chunk_tiles": 1, "max_splits": 1, "tree_split": 0}


def _plan_of(ts, name, B, N, Hq, Hkv, D, plens, bs, tree):
    return ts.tree_attn_plan(_params(ts, B=B, N=N, Hq=Hq, Hkv=Hkv, D=D, bs=bs, P=tuple(plens)))


def test_small_parity_cases_cover_every_split_layout(ts):
    """The element-wise GPU parity cases must exercise each kernel layout."""
    from tests.gpu_util import SMALL
    layouts = set()
    for spec in SMALL:
        plan = _plan_of(ts, *spec)
        if plan["max_splits"] == 1:
            layouts.add("direct")
        else:
            layouts.add("tree split" if plan["tree_split"] else "tree on last prefix split")
    assert layouts == {"direct", "tree split", "tree on last prefix split"}


@pytest.mark.parametrize("change,code", [
    (dict(q=None), -1),
    (dict(D=96), -4),
    (dict(Hq=24, Hkv=8), -4),      # G = 3
    (dict(Hq=30, Hkv=8), -2),      # not a multiple
    (dict(N=257), -4),
    (dict(bs=40), -4),             # block sizes must be multiples of 16
    (dict(bs=8), -4),
    (dict(rope_theta=10000.0), -4),
    (dict(misalign=True), -2),
    (dict(neg_prefix=True), -2),
    (dict(huge_prefix=True), -4),
])
def test_attn_rejects_before_launch(ts, change, code):
    change = dict(change)
    if change.pop("misalign", False):
        p = _params(ts)
        p.q = 0x10002
    elif change.pop("neg_prefix", False):
        p = _params(ts, P=(5, -1))
    elif change.pop("huge_prefix", False):
        p = _params(ts, P=(5, (1 << 30) + 16))
    elif "q" in change:
        p = _params(ts)
        p.q = None
    else:
        p = _params(ts)
        for k, v in change.items():
            setattr(p, k if k != "bs" else "block_size", v)
    assert ts.tree_attn_workspace_size(p) == 0
    ws = _FakeTensor((1,), 0x20000)
    ws.numel = lambda: 1 << 30
    ws.element_size = lambda: 1
    st = ts.lib().tree_attn_fwd(ctypes.byref(p), ctypes.c_void_p(0x20000), 1 << 30, None)
    assert st == code


def test_attn_rejects_small_workspace(ts):
    p = _params(ts)
    need = ts.tree_attn_workspace_size(p)
    assert ts.lib().tree_attn_fwd(ctypes.byref(p), ctypes.c_void_p(0x20000), need - 256, None) == -8
    assert ts.lib().tree_attn_fwd(ctypes.byref(p), None, need, None) == -8
    assert ts.lib().tree_attn_fwd(ctypes.byref(p), ctypes.c_void_p(0x20010), need, None) == -8


def test_verify_and_ancestry_reject_before_launch(ts):
    L = ts.lib()
    a = ctypes.c_void_p(0x10000)
    assert L.tree_build_ancestry(None, a, 1, 5, a, a, a, a, None) == -1
    assert L.tree_build_ancestry(a, a, 1, 257, a, a, a, a, None) == -4
    assert L.tree_build_ancestry(a, a, 0, 5, a, a, a, a, None) == -4
    assert ts.tree_verify_workspace_size(1, 5, 1000) > 0
    assert ts.tree_verify_workspace_size(1, 300, 1000) == 0
    need = ts.tree_verify_workspace_size(4, 64, 128256)
    args = [a, a, a, 4, 64, 128256, 8, a, a, a, a, a, a, need, None]
    bad = list(args); bad[1] = None
    assert L.tree_verify_greedy(*bad) == -1
    bad = list(args); bad[6] = -1
    assert L.tree_verify_greedy(*bad) == -4
    bad = list(args); bad[13] = need - 1
    assert L.tree_verify_greedy(*bad) == -8


def test_commit_stochastic_and_dynamic_reject_before_launch(ts):
    L = ts.lib()
    a = ctypes.c_void_p(0x10000)
    # tree_commit_accepted: k_tree, v_tree, accepted, accept_len, prefix_len, k_cache, v_cache, table,
    #                       B, N, Hkv, D, bs, num_blocks, max_blocks, max_depth, new_len, status, stream
    args = [a, a, a, a, a, a, a, a, 2, 8, 2, 128, 16, 10, 4, 4, a, a, None]
    bad = list(args); bad[0] = None
    assert L.tree_commit_accepted(*bad) == -1
    bad = list(args); bad[11] = 96
    assert L.tree_commit_accepted(*bad) == -4
    bad = list(args); bad[8] = 0
    assert L.tree_commit_accepted(*bad) == -2
    # tree_verify_stochastic: draft, logits, q, parent, coins, B, N, V, max_depth, T, acc, L, bonus, status, stream
    args = [a, a, a, a, a, 4, 64, 128256, 8, ctypes.c_float(1.0), a, a, a, a, None]
    bad = list(args); bad[2] = None
    assert L.tree_verify_stochastic(*bad) == -1
    for i, v in ((9, ctypes.c_float(0.0)), (9, ctypes.c_float(-1.0)), (9, ctypes.c_float(float("inf"))),
                 (6, 257), (7, 409601), (8, -1), (5, 70000)):
        bad = list(args); bad[i] = v
        assert L.tree_verify_stochastic(*bad) == -4, (i, v)
    # tree_build_dynamic: pool_parent, logp, token, prefix_len, B, M, N, parent, tokens, sel, anc, depth, pos,
    #                     status, stream
    args = [a, a, a, a, 4, 457, 64, a, a, a, a, a, a, a, None]
    bad = list(args); bad[1] = None
    assert L.tree_build_dynamic(*bad) == -1
    bad = list(args); bad[5] = 63
    assert L.tree_build_dynamic(*bad) == -2
    bad = list(args); bad[5] = 1025
    assert L.tree_build_dynamic(*bad) == -4
    bad = list(args); bad[6] = 257; bad[5] = 1000
    assert L.tree_build_dynamic(*bad) == -4


def test_forest_calls_reject_before_launch(ts):
    L = ts.lib()
    a = ctypes.c_void_p(0x10000)
    assert L.tree_build_ancestry_forest(None, a, 1, 5, a, a, a, a, None) == -1
    assert L.tree_build_ancestry_forest(a, a, 1, 257, a, a, a, a, None) == -4
    need = ts.tree_verify_workspace_size(4, 64, 128256)
    args = [a, a, a, 4, 64, 128256, 8, a, a, a, a, a, a, need, None]
    bad = list(args); bad[2] = None
    assert L.tree_verify_greedy_forest(*bad) == -1
    bad = list(args); bad[13] = need - 1
    assert L.tree_verify_greedy_forest(*bad) == -8


def _expected_pairs(P, chunk, splits, tsplit, tree_tiles):
    """(length in tiles, first prefix tile) of every (sequence, split) pair when
    each prefix of T tiles is cut into ceil(T / chunk) splits of near-equal
    length, split s starting at floor(T s / splits), and the tree block rides on
    the sequence's last split (or a split of its own)."""
    out = {}
    for b, p in enumerate(P):
        tiles = -(-p // 128)
        ps = -(-tiles // chunk)
        ns = ps + 1 if tsplit else max(ps, 1)
        for s in range(splits):
            start = tiles * s // ps if s < ps else 0
            n = (tiles * (s + 1) // ps - start) if s < ps else 0
            if s == ns - 1:
                n += tree_tiles
            out[(b, s)] = (n, start)
    return out


@pytest.mark.parametrize("B,N,Hq,Hkv,P", [
    (16, 26, 32, 8, (1207, 1427, 1497, 1964, 2939, 4413, 5913, 6798, 7843, 7953, 8097, 8622, 10608, 11850, 13284,
                     15195)),
    (8, 33, 8, 2, (0, 17, 1000, 4096, 130, 2500, 3999, 1)),
    (1, 64, 32, 8, (4096,)),
    (4, 192, 32, 8, (131072,) * 4),
    (6, 30, 8, 2, (700, 3000, 130, 1900, 0, 2500)),
    (256, 3, 2, 1, tuple(16 * (i % 7) for i in range(256))),
])
def test_attn_plan_order_is_every_pair_longest_first(ts, B, N, Hq, Hkv, P):
    p = _params(ts, B=B, N=N, Hq=Hq, Hkv=Hkv, D=128 if N > 3 else 64, bs=16, P=P)
    plan = ts.tree_attn_plan(p)
    order = ts.tree_attn_plan_order(p)
    pairs = B * plan["max_splits"]
    assert len(order) == (pairs if pairs <= 256 else 0)
    exp = _expected_pairs(P, plan["chunk_tiles"], plan["max_splits"], plan["tree_split"], -(-N // 128))
    got = [(e >> 24, (e >> 15) & 0x1FF, e & 0x7FFF) for e in order]
    assert sorted((b, s) for b, s, _ in got) == sorted(exp)          # every pair exactly once
    lens = [exp[(b, s)][0] for b, s, _ in got]
    assert lens == sorted(lens, reverse=True)                        # longest first
    for i in range(1, len(got)):                                     # ties keep sequence, then split order
        if lens[i] == lens[i - 1]:
            assert got[i][:2] > got[i - 1][:2]
    for b, s, start in got:                                          # the first tile of each split
        assert start == min(exp[(b, s)][1], 0x7FFF)
    for b in range(B):                                               # splits cover the prefix, none over the chunk
        tiles = -(-P[b] // 128)
        ps = -(-tiles // plan["chunk_tiles"])
        sizes = [tiles * (s + 1) // ps - tiles * s // ps for s in range(ps)]
        assert sum(sizes) == tiles and all(0 < x <= plan["chunk_tiles"] for x in sizes)


def test_attn_plan_order_counts_without_a_table_past_256_pairs(ts):
    P = tuple(16 * (i % 5) + 2000 * (i == 7) for i in range(300))
    p = _params(ts, B=300, N=3, Hq=2, Hkv=1, D=64, bs=16, P=P)
    assert ts.tree_attn_plan(p)["max_splits"] >= 2
    assert ts.tree_attn_plan_order(p) == []
    n = ctypes.c_int32(-1)
    assert ts.lib().tree_attn_plan_order(ctypes.byref(p), None, 0, ctypes.byref(n)) == 0 and n.value == 0
    small = _params(ts, B=2, N=26, Hq=32, Hkv=8, D=128, bs=16, P=(1000, 3000))
    assert ts.lib().tree_attn_plan_order(ctypes.byref(small), None, 0, ctypes.byref(n)) == -2   # cap 0 < count
    assert ts.lib().tree_attn_plan_order(ctypes.byref(small), None, -1, ctypes.byref(n)) == -2
    assert ts.lib().tree_attn_plan_order(ctypes.byref(small), None, 0, None) == -1
