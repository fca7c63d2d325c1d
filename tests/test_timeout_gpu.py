"""The attention kernel's failure path: a bounded wait that runs out.

Every wait inside the attention kernel is bounded.  tree_attn_fwd_stall_test
runs the ordinary call with one sequence's key stream stopped before a given
tile (those loads are never issued, so nothing is left in flight) and a short
wait limit.  The wait for that tile must run out, the CTA must wind down and
report TS_ERR_TIMEOUT for that sequence only, the other sequences must still
get the oracle's result, and the device must stay usable: an ordinary call
right after, in the same process, passes parity.  No fault, trap or endless
loop is involved: the kernel returns by itself.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import LSE_ATOL, assert_close_attention, out_f64, run_case, to_dev

pytestmark = pytest.mark.gpu

TS_ERR_TIMEOUT = -6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tree_attention_speculative_gb300 import _build
    _build.build()
    import tree_attention_speculative_gb300 as ts
    ts.lib()
    torch.cuda.init()


def _case():
    g = W.rng(11, "stall")
    parent = np.stack([W.tree_random_levels(g, 37, 6) for _ in range(3)])
    return W.build_case("stall", 11, parent, [700, 1100, 129], Hq=8, Hkv=2, D=128, bs=16, permute=True)


@pytest.mark.parametrize("stall_seq,stall_tile", [(1, 0), (1, 1), (0, 0), (2, 1)])
def test_attention_wait_runs_out_and_reports_timeout(stall_seq, stall_tile):
    import tree_attention_speculative_gb300 as ts
    from tree_attention_speculative_gb300.step import TreeVerifyStep
    case = _case()
    t = to_dev(case)
    step = TreeVerifyStep(case.B, case.N, case.Hq, case.Hkv, case.D, case.prefix_len)
    step.ancestry(t["parent"], t["prefix_len"])
    p = step._params(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"], t["k_tree"],
                     t["v_tree"])
    # the longest split of the sequence holds more than stall_tile tiles (its
    # ceil(tiles / chunk) splits differ by one tile at most), so its CTAs do
    # reach the withheld tile
    plan = ts.tree_attn_plan(p)
    tiles = -(-int(case.prefix_len[stall_seq]) // 128)
    ps = -(-tiles // plan["chunk_tiles"])
    assert -(-tiles // ps) > stall_tile, plan
    ws = torch.zeros(ts.tree_attn_workspace_size(p), dtype=torch.uint8, device="cuda")
    ts.tree_attn_fwd_stall_test(p, ws, stall_seq, stall_tile, 2000)
    torch.cuda.synchronize()     # the call returns by itself: no hang, no fault
    st = step.status.cpu().tolist()
    assert st == [TS_ERR_TIMEOUT if b == stall_seq else 0 for b in range(case.B)], st
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    got = out_f64(step)
    lse = step.lse.cpu().numpy()
    for b in range(case.B):
        if b == stall_seq:
            continue
        assert_close_attention(got[b], ref[b], f"sequence {b} beside the stalled one")
        np.testing.assert_allclose(lse[b], ref_lse[b], rtol=0, atol=LSE_ATOL)
    # the context is still usable: the ordinary call on the same inputs passes parity
    s2, _ = run_case(case)
    assert s2.status.cpu().tolist() == [0] * case.B
    assert_close_attention(out_f64(s2), ref, "ordinary call after the timeout")
    np.testing.assert_allclose(s2.lse.cpu().numpy(), ref_lse, rtol=0, atol=LSE_ATOL)


def test_stall_test_rejects_bad_arguments():
    import tree_attention_speculative_gb300 as ts
    from tree_attention_speculative_gb300.step import TreeVerifyStep
    case = _case()
    t = to_dev(case)
    step = TreeVerifyStep(case.B, case.N, case.Hq, case.Hkv, case.D, case.prefix_len)
    p = step._params(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"], t["k_tree"],
                     t["v_tree"])
    ws = torch.zeros(ts.tree_attn_workspace_size(p), dtype=torch.uint8, device="cuda")
    L = ts.lib()
    import ctypes
    nb = ws.numel()
    assert L.tree_attn_fwd_stall_test(ctypes.byref(p), ctypes.c_void_p(ws.data_ptr()), nb, 3, 0, 2000, None) == -2
    assert L.tree_attn_fwd_stall_test(ctypes.byref(p), ctypes.c_void_p(ws.data_ptr()), nb, 0, -1, 2000, None) == -2
    assert L.tree_attn_fwd_stall_test(ctypes.byref(p), ctypes.c_void_p(ws.data_ptr()), nb, 0, 0, 50, None) == -4
