"""GPU parity of tree_commit_accepted against the oracle (bit-exact: a pure copy).

A full verification step runs on the GPU (ancestry, attention, verify), then
the accepted paths are appended to the paged cache; the whole pool and the new
prefix lengths must equal the oracle's.  Covers accepted lengths 0..max,
contiguous and permuted pools, a sequence whose verify failed, a destination
block missing from the table, and updating the prefix lengths in place.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import run_case, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tree_attention_speculative_gb300 import _build
    _build.build()


def _run(case, max_depth, in_place=False, status_override=None, table_override=None):
    import tree_attention_speculative_gb300 as ts
    step, t = run_case(case, max_depth=max_depth)
    if status_override is not None:
        step.status.copy_(torch.from_numpy(np.asarray(status_override, np.int32)))
    table = t["block_table"]
    if table_override is not None:
        table = torch.from_numpy(table_override.astype(np.int32)).cuda()
    new_len = t["prefix_len"] if in_place else torch.empty_like(t["prefix_len"])
    ts.tree_commit_accepted(t["k_tree"], t["v_tree"], step.accepted, step.accept_len, t["prefix_len"], t["k_cache"],
                            t["v_cache"], table, new_len, step.status)
    torch.cuda.synchronize()
    got = dict(k=t["k_cache"].view(torch.int16).cpu().numpy().view(np.uint16),
               v=t["v_cache"].view(torch.int16).cpu().numpy().view(np.uint16),
               new_len=new_len.cpu().numpy(), status=step.status.cpu().numpy(),
               accepted=step.accepted.cpu().numpy(), accept_len=step.accept_len.cpu().numpy())
    return got


def _ref(case, got, table=None):
    table = case.block_table if table is None else table
    return oracle.commit.commit_accepted(case.k_tree, case.v_tree, got["accepted"], got["accept_len"], got["status"],
                                         case.prefix_len, case.k_cache, case.v_cache, table)


@pytest.mark.parametrize("bs,permute", [(16, True), (64, True), (128, False)])
def test_commit_matches_oracle(bs, permute):
    g = W.rng(bs, "commit-gpu")
    B, N, depth = 6, 40, 7
    parents = np.stack([W.tree_random_levels(g, N, depth) for _ in range(B)])
    plens = [0, 1, 127, 128, 300, 513]
    case = W.build_case("commit", bs, parents, plens, Hq=8, Hkv=2, D=128, bs=bs, permute=permute, vocab=500,
                        plant_len=[0, 7, 3, 1, 5, 2], spare_tokens=depth + 1)
    got = _run(case, depth)
    # the GPU's acceptance equals the oracle's before anything is committed
    acc, L, bonus, am, st = oracle.verify.verify_greedy(case.draft, case.logits, case.parent, depth)
    np.testing.assert_array_equal(got["accepted"], acc)
    kc, vc, new_len = _ref(case, got)
    np.testing.assert_array_equal(got["new_len"], new_len)
    np.testing.assert_array_equal(got["k"], kc)
    np.testing.assert_array_equal(got["v"], vc)
    assert (got["new_len"] == np.array(plens) + np.array([0, 7, 3, 1, 5, 2]) + 1).all()


def test_commit_skips_failed_and_rejects_missing_block_in_place():
    g = W.rng(9, "commit-gpu2")
    B, N, depth = 3, 20, 5
    parents = np.stack([W.tree_random_levels(g, N, depth) for _ in range(B)])
    case = W.build_case("commit", 9, parents, [50, 31, 16], Hq=2, Hkv=1, D=64, bs=16, permute=True, vocab=300,
                        plant_len=[4, 5, 3], spare_tokens=depth + 1)
    table = case.block_table.copy()
    # sequence 2 commits positions 16..19: its second block entry goes missing
    table[2, 1] = -1
    got = _run(case, depth, in_place=True, status_override=[0, -3, 0], table_override=table)
    assert got["status"].tolist() == [0, -3, -5]
    assert got["new_len"].tolist() == [50 + 4 + 1, 31, 16]
    kc, vc, _ = _ref(case, dict(got, status=np.array([0, -3, -5])), table)
    np.testing.assert_array_equal(got["k"], kc)
    np.testing.assert_array_equal(got["v"], vc)
