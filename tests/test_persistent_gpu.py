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
