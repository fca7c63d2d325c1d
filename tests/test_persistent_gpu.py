"""The persistent attention kernel: work items shared out through a counter.

tree_attn_fwd runs one attention CTA per SM; each takes work items (a 128-row
tile of one (sequence, KV head) and one split of its prefix) from a counter
in the workspace until none is left, and the last request of all puts the
counter back to zero.  The ordinary tests give most CTAs a single item, so
these cap the CTAs (tree_attn_fwd_ctas_test) to send many items through each
CTA: items of unequal length, empty splits past a short prefix, the tree
block on a split of its own, the last item stored by TMA and the others by
plain stores.  Each result is compared element by element with the oracle;
calls are repeated on one workspace (the counter must come back to zero, or
the next call would skip items); and a stalled item must report the timeout
for the items its CTA had taken and not finished, leave every other output
right, and leave the counter at zero for the next call.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import SMALL, LSE_ATOL, assert_close_attention, out_f64, to_dev

pytestmark = pytest.mark.gpu

TS_ERR_TIMEOUT = -6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tree_attention_speculative_gb300 import _build
    _build.build()
    import tree_attention_speculative_gb300 as ts
    ts.lib()
    torch.cuda.init()


def _small_case(name, B, N, Hq, Hkv, D, plens, bs, tree):
    g = W.rng(len(name), name)
    if tree == "random":
        parent = np.stack([W.tree_random_recursive(g, N) for _ in range(B)])
    elif tree == "levels":
        parent = np.stack([W.tree_random_levels(g, N, 8) for _ in range(B)])
    elif tree == "chain":
        parent = W.tree_chain(N)
    elif tree == "worked":
        parent = W.tree_worked_example()
    else:
        parent = W.tree_from_widths([4, 3, 2, 1, 1])
    permute = bs < max(max(plens), 1)
    return W.build_case(name, 7, parent, plens, Hq=Hq, Hkv=Hkv, D=D, bs=bs, permute=permute)


def _step(case):
    """The step, the call's parameters, and the device inputs they point into
    (which the caller must keep alive while it uses the parameters)."""
    from tree_attention_speculative_gb300.step import TreeVerifyStep
    t = to_dev(case)
    step = TreeVerifyStep(case.B, case.N, case.Hq, case.Hkv, case.D, case.prefix_len)
    step.ancestry(t["parent"], t["prefix_len"])
    p = step._params(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"], t["k_tree"],
                     t["v_tree"])
    return step, p, t


def _check(step, case, ref, ref_lse, what, skip=()):
    got = out_f64(step)
    lse = step.lse.cpu().numpy()
    for b in range(case.B):
        if b in skip:
            continue
        assert_close_attention(got[b], ref[b], f"{what}, sequence {b}")
        np.testing.assert_allclose(lse[b], ref_lse[b], rtol=0, atol=LSE_ATOL)


@pytest.mark.parametrize("ctas", [1, 2, 3, 7])
@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_few_ctas_take_every_item(spec, ctas):
    import tree_attention_speculative_gb300 as ts
    case = _small_case(*spec)
    step, p, _t = _step(case)
    ws = torch.zeros(ts.tree_attn_workspace_size(p), dtype=torch.uint8, device="cuda")
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    for rep in range(2):   # the same workspace twice: its counter is back at zero after each call
        step.out.zero_()
        ts.tree_attn_fwd_ctas_test(p, ws, ctas)
        torch.cuda.synchronize()
        assert step.status.cpu().tolist() == [0] * case.B
        _check(step, case, ref, ref_lse, f"{spec[0]} on {ctas} CTAs, call {rep}")
        assert ws[:256].cpu().numpy().tobytes() == bytes(256), "item counter not back at zero"


def test_variable_prefixes_with_empty_splits():
    """Prefixes from empty to several splits long, on fewer CTAs than items:
    most CTAs meet empty splits (past a short prefix) between real items."""
    import tree_attention_speculative_gb300 as ts
    plens = [0, 17, 1000, 4096, 130, 2500, 3999, 1]
    g = W.rng(5, "var")
    parent = np.stack([W.tree_random_levels(g, 33, 6) for _ in plens])
    case = W.build_case("var", 5, parent, plens, Hq=8, Hkv=2, D=128, bs=16, permute=True)
    step, p, _t = _step(case)
    plan = ts.tree_attn_plan(p)
    assert plan["max_splits"] >= 2, plan
    ws = torch.zeros(ts.tree_attn_workspace_size(p), dtype=torch.uint8, device="cuda")
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    for ctas in (1, 4, 5, 1000):
        step.out.zero_()
        ts.tree_attn_fwd_ctas_test(p, ws, ctas)
        torch.cuda.synchronize()
        assert step.status.cpu().tolist() == [0] * case.B
        _check(step, case, ref, ref_lse, f"{ctas} CTAs")
    # and the ordinary call after them
    step.out.zero_()
    ts.tree_attn_fwd(p, ws)
    torch.cuda.synchronize()
    _check(step, case, ref, ref_lse, "ordinary call")


@pytest.mark.parametrize("stall_seq", [0, 2])
def test_timeout_on_one_cta_reports_its_unfinished_items(stall_seq):
    """All items on one CTA, one sequence stalled: the items taken before the
    stalled one are finished and right; the stalled one and every item the
    CTA takes after it report the timeout; the counter is back at zero, so an
    ordinary call on the same workspace right after is right everywhere."""
    import tree_attention_speculative_gb300 as ts
    g = W.rng(9, "stall1")
    plens = [600, 900, 300, 700]
    parent = np.stack([W.tree_random_levels(g, 20, 5) for _ in plens])
    case = W.build_case("stall1", 9, parent, plens, Hq=4, Hkv=2, D=128, bs=16, permute=True)
    step, p, _t = _step(case)
    ws = torch.zeros(ts.tree_attn_workspace_size(p), dtype=torch.uint8, device="cuda")
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    step.status.zero_()
    ts.tree_attn_fwd_ctas_test(p, ws, 1, stall_seq, 0, 2000)
    torch.cuda.synchronize()
    st = step.status.cpu().tolist()
    assert st[stall_seq] == TS_ERR_TIMEOUT, st
    assert all(s in (0, TS_ERR_TIMEOUT) for s in st), st
    assert ws[:256].cpu().numpy().tobytes() == bytes(256)
    # the sequences reported fine are right
    _check(step, case, ref, ref_lse, "beside the stall", skip={b for b in range(case.B) if st[b] != 0})
    # the context and the workspace are usable at once
    step.status.zero_()
    step.out.zero_()
    ts.tree_attn_fwd(p, ws)
    torch.cuda.synchronize()
    assert step.status.cpu().tolist() == [0] * case.B
    _check(step, case, ref, ref_lse, "ordinary call after the timeout")


def test_ctas_test_rejects_bad_arguments():
    import ctypes
    import tree_attention_speculative_gb300 as ts
    case = _small_case(*SMALL[0])
    step, p, _t = _step(case)
    ws = torch.zeros(ts.tree_attn_workspace_size(p), dtype=torch.uint8, device="cuda")
    L = ts.lib()
    nb = ws.numel()
    w = ctypes.c_void_p(ws.data_ptr())
    assert L.tree_attn_fwd_ctas_test(ctypes.byref(p), w, nb, 0, -1, 0, 2000, None) == -4
    assert L.tree_attn_fwd_ctas_test(ctypes.byref(p), w, nb, 1, -2, 0, 2000, None) == -2
    assert L.tree_attn_fwd_ctas_test(ctypes.byref(p), w, nb, 1, case.B, 0, 2000, None) == -2
    assert L.tree_attn_fwd_ctas_test(ctypes.byref(p), w, nb, 1, 0, -1, 2000, None) == -2
    assert L.tree_attn_fwd_ctas_test(ctypes.byref(p), w, nb, 1, -1, 0, 50, None) == -4


# --------------------------------------------------------------------------- tail items
#
# With one split per unit, N items on C CTAs leave N mod C for the last round;
# when that is at most C/2 those items are cut into two halves (the first half
# of the prefix tiles; the rest and the tree block), and the half that ends
# second merges the two.  These cases have one split per unit and are run on
# CTA counts that leave such a last round.

def _tail_case(name, B, N, Hq, Hkv, D, plens, bs=16):
    g = W.rng(len(name) + 3, name)
    parent = np.stack([W.tree_random_levels(g, N, 6) for _ in range(B)])
    return W.build_case(name, 11, parent, plens, Hq=Hq, Hkv=Hkv, D=D, bs=bs, permute=True)


def _ticket_bytes_zero(ws):
    # the counter (first 256 bytes) and the tail tickets (the last region)
    return ws[:256].cpu().numpy().tobytes() == bytes(256) and not ws[-256:].cpu().numpy().any()


TAIL_CASES = [
    # name, B, N, Hq, Hkv, D, prefix lengths, CTA counts (items n; a tail where n mod C <= C/2)
    ("tail_d128", 20, 26, 32, 8, 128, [1500 - 37 * i for i in range(20)], [50, 70, 150]),
    # prefixes of 0-2 tiles: first halves with no tile at all
    ("tail_short", 40, 20, 16, 4, 128, [(53 * i) % 260 for i in range(40)], [50, 70, 150]),
    ("tail_d64", 24, 26, 32, 8, 64, [1400 - 41 * i for i in range(24)], [90, 150, 180]),
]


@pytest.mark.parametrize("spec", TAIL_CASES, ids=[c[0] for c in TAIL_CASES])
def test_tail_items_cut_in_halves(spec):
    import tree_attention_speculative_gb300 as ts
    name, B, N, Hq, Hkv, D, plens, ctas_list = spec
    case = _tail_case(name, B, N, Hq, Hkv, D, plens)
    step, p, _t = _step(case)
    plan = ts.tree_attn_plan(p)
    assert plan["max_splits"] == 1, plan   # one split per unit: the tail rule applies
    items = -(-N * (Hq // Hkv) // 128) * B * Hkv
    ws = torch.zeros(ts.tree_attn_workspace_size(p), dtype=torch.uint8, device="cuda")
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    tails = 0
    for ctas in ctas_list:
        rem = items % ctas
        tails += 0 < 2 * rem <= ctas
        for rep in range(2):
            step.out.zero_()
            step.lse.zero_()
            ts.tree_attn_fwd_ctas_test(p, ws, ctas)
            torch.cuda.synchronize()
            assert step.status.cpu().tolist() == [0] * case.B
            _check(step, case, ref, ref_lse, f"{name} on {ctas} CTAs ({items} items), call {rep}")
            assert _ticket_bytes_zero(ws), "counter or tail tickets not back at zero"
    assert tails > 0, "no CTA count left a tail to cut"


def test_stall_on_tail_halves_keeps_tickets_at_zero():
    """A stalled sequence whose last-round items are cut in halves: its
    timeout is reported, every sequence reported fine is right, and the
    counter and the tail tickets end at zero, so the next ordinary call is
    right everywhere."""
    import tree_attention_speculative_gb300 as ts
    B, N, Hq, Hkv, D = 20, 26, 32, 8, 128
    case = _tail_case("tail_stall", B, N, Hq, Hkv, D, [1500 - 37 * i for i in range(B)])
    step, p, _t = _step(case)
    assert ts.tree_attn_plan(p)["max_splits"] == 1
    items = -(-N * (Hq // Hkv) // 128) * B * Hkv     # 160, one per (sequence, KV head)
    ctas = 50                                          # 160 mod 50 = 10: the last 10 items in halves
    assert 0 < 2 * (items % ctas) <= ctas
    ws = torch.zeros(ts.tree_attn_workspace_size(p), dtype=torch.uint8, device="cuda")
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    for stall_seq in (B - 1, B - 2, 0):   # the last two sequences' items are the tail items
        step.status.zero_()
        ts.tree_attn_fwd_ctas_test(p, ws, ctas, stall_seq, 0, 2000)
        torch.cuda.synchronize()
        st = step.status.cpu().tolist()
        assert st[stall_seq] == TS_ERR_TIMEOUT, st
        assert all(s in (0, TS_ERR_TIMEOUT) for s in st), st
        assert _ticket_bytes_zero(ws), "counter or tail tickets not back at zero after a timeout"
        _check(step, case, ref, ref_lse, f"beside stalled sequence {stall_seq}",
               skip={b for b in range(case.B) if st[b] != 0})
        step.status.zero_()
        step.out.zero_()
        ts.tree_attn_fwd_ctas_test(p, ws, ctas)
        torch.cuda.synchronize()
        assert step.status.cpu().tolist() == [0] * case.B
        _check(step, case, ref, ref_lse, f"call after stalling sequence {stall_seq}")
