"""The order of the attention kernel's work items, and its equal splits.

The host cuts each sequence's prefix into splits of near-equal length and
orders every (sequence, split) pair longest first by the prefix lengths it
was given (with the first prefix tile of each split as a hint); the kernel
takes the items in that order and works on each with the prefix length it
finds on the device.  These cases compare every output element with the
oracle where host and device disagree, and where no order table is used:

- host lengths permuted among the sequences: for most items the hint names
  the wrong first tile (the block-table entries loaded with it must be
  loaded again), and sequences have more or fewer splits than the table
  expects (splits the table ranks last, as empty, have work);
- a batch with more (sequence, split) pairs than one table holds: items go
  in unit-major order; and one with exactly as many as it holds.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import LSE_ATOL, assert_close_attention, out_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tree_attention_speculative_gb300 import _build
    _build.build()
    import tree_attention_speculative_gb300 as ts
    ts.lib()
    torch.cuda.init()


def _run(case, host_len, ctas=None):
    import tree_attention_speculative_gb300 as ts
    from tree_attention_speculative_gb300.step import TreeVerifyStep
    t = to_dev(case)
    step = TreeVerifyStep(case.B, case.N, case.Hq, case.Hkv, case.D, host_len)
    step.ancestry(t["parent"], t["prefix_len"])
    p = step._params(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"], t["k_tree"],
                     t["v_tree"])
    ws = torch.zeros(ts.tree_attn_workspace_size(p), dtype=torch.uint8, device="cuda")
    if ctas is None:
        ts.tree_attn_fwd(p, ws)
    else:
        ts.tree_attn_fwd_ctas_test(p, ws, ctas)
    torch.cuda.synchronize()
    assert ws[:256].cpu().numpy().tobytes() == bytes(256), "item counter not back at zero"
    return step, dict(ts.tree_attn_plan(p), pairs=len(ts.tree_attn_plan_order(p)))


def _check(step, case, what):
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    assert step.status.cpu().tolist() == [0] * case.B
    got = out_f64(step)
    lse = step.lse.cpu().numpy()
    for b in range(case.B):
        assert_close_attention(got[b], ref[b], f"{what}, sequence {b}")
        np.testing.assert_allclose(lse[b], ref_lse[b], rtol=0, atol=LSE_ATOL)


@pytest.mark.parametrize("ctas", [None, 1, 3])
def test_host_lengths_permuted_among_sequences(ctas):
    plens = [700, 3000, 130, 1900, 0, 2500]
    g = W.rng(11, "order")
    parent = np.stack([W.tree_random_levels(g, 30, 5) for _ in plens])
    case = W.build_case("order", 11, parent, plens, Hq=8, Hkv=2, D=128, bs=16, permute=True)
    host = plens[::-1]     # same multiset: same plan, wrong length for every sequence
    step, plan = _run(case, host, ctas)
    assert plan["max_splits"] >= 2, plan
    _check(step, case, f"host lengths reversed, {ctas} CTAs")


def test_more_pairs_than_one_table_holds():
    g = W.rng(12, "pairs")
    plens = [int(x) for x in g.integers(0, 600, 300)]
    plens[7] = 2000      # one long prefix: several splits for every sequence's slot
    parent = np.stack([W.tree_random_levels(g, 3, 2) for _ in plens])
    case = W.build_case("pairs", 12, parent, plens, Hq=2, Hkv=1, D=64, bs=16, permute=True)
    step, plan = _run(case, plens)
    assert case.B * plan["max_splits"] > 256 and plan["pairs"] == 0, plan
    _check(step, case, "unit-major order")


def test_exactly_one_full_table_of_pairs():
    """256 (sequence, split) pairs, the most one order table holds: sequence
    255 is the largest the entries' 8-bit field carries."""
    g = W.rng(14, "t256")
    plens = [int(x) for x in g.integers(0, 250, 256)]
    parent = np.stack([W.tree_random_levels(g, 3, 2) for _ in plens])
    case = W.build_case("t256", 14, parent, plens, Hq=2, Hkv=1, D=64, bs=16, permute=True)
    step, plan = _run(case, plens)
    assert plan["pairs"] == 256 and case.B * plan["max_splits"] == 256, plan
    _check(step, case, "a full order table")
