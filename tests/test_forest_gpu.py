"""GPU parity of a forest verification step (several roots per sequence):
tree_build_ancestry_forest, tree_attn_fwd on the forest's masks,
tree_verify_greedy_forest and tree_commit_accepted, against the forest oracle
(masks, acceptance: bit-exact) and the fp64 attention oracle (tolerance)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import forest as F
import workloads as W
from tests.gpu_util import assert_close_attention, out_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tree_attention_speculative_gb300 import _build
    _build.build()


def _forest_case(seed, B, N, roots, depth, plens, Hq, Hkv, D, bs, vocab, planted):
    g = W.rng(seed, "forest-gpu")
    parents = np.stack([W.forest_random(g, N, roots, depth) for _ in range(B)])
    # plant in a tree other than node 0's when there is one
    tgt = []
    for b in range(B):
        lv = W._levels_of(parents[b])
        cands = np.nonzero(lv == planted[b])[0]
        r = F.roots_of(parents[b])
        other = [c for c in cands if r[c] != 0]
        tgt.append(int((other or list(cands))[-1]))
    return W.build_case("forest", seed, parents, plens, Hq=Hq, Hkv=Hkv, D=D, bs=bs, permute=True, vocab=vocab,
                        plant_len=planted, plant_target=tgt, spare_tokens=N)


def run_forest(case, max_depth):
    import tree_attention_speculative_gb300 as ts
    from tree_attention_speculative_gb300.step import TreeVerifyStep
    t = to_dev(case)
    step = TreeVerifyStep(case.B, case.N, case.Hq, case.Hkv, case.D, case.prefix_len, vocab=case.vocab,
                          max_depth=max_depth, forest=True)
    step.run(t["parent"], t["prefix_len"], t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["k_tree"],
             t["v_tree"], t["draft"], t["logits"])
    new_len = torch.empty_like(t["prefix_len"])
    ts.tree_commit_accepted(t["k_tree"], t["v_tree"], step.accepted, step.accept_len, t["prefix_len"], t["k_cache"],
                            t["v_cache"], t["block_table"], new_len, step.status)
    torch.cuda.synchronize()
    return step, t, new_len


@pytest.mark.parametrize("seed,B,N,roots,depth,D,bs", [(1, 3, 40, 3, 5, 128, 16), (2, 2, 130, 5, 7, 64, 64),
                                                       (3, 4, 9, 9, 0, 128, 16)])
def test_forest_step_matches_oracle(seed, B, N, roots, depth, D, bs):
    plens = [0, 77, 300, 1000][:B]
    planted = [min(depth, 3)] * B if depth else [0] * B
    case = _forest_case(seed, B, N, roots, depth, plens, 8, 2, D, bs, 700, planted)
    md = depth + 1
    step, t, new_len = run_forest(case, md)
    anc, dep, pos, st = F.build_ancestry_forest(case.parent, case.prefix_len)
    np.testing.assert_array_equal(step.anc.cpu().numpy().view(np.uint64), anc)
    np.testing.assert_array_equal(step.depth.cpu().numpy(), dep)
    np.testing.assert_array_equal(step.pos.cpu().numpy(), pos)
    ref, lse = oracle.attention.tree_attention_case(case)
    assert_close_attention(out_f64(step), ref, "forest attention")
    acc, L, bonus, am, vst = F.verify_greedy_forest(case.draft, case.logits, case.parent, md)
    np.testing.assert_array_equal(step.accepted.cpu().numpy(), acc)
    np.testing.assert_array_equal(step.accept_len.cpu().numpy(), L)
    np.testing.assert_array_equal(step.bonus.cpu().numpy(), bonus)
    np.testing.assert_array_equal(step.argmax.cpu().numpy(), am)
    np.testing.assert_array_equal(step.status.cpu().numpy(), vst)
    np.testing.assert_array_equal(L, planted)
    kc, vc, nl = oracle.commit.commit_accepted(case.k_tree, case.v_tree, acc, L, vst, case.prefix_len, case.k_cache,
                                               case.v_cache, case.block_table)
    np.testing.assert_array_equal(new_len.cpu().numpy(), nl)
    np.testing.assert_array_equal(t["k_cache"].view(torch.int16).cpu().numpy().view(np.uint16), kc)


def test_single_root_calls_reject_forests_and_forest_calls_accept_trees():
    import tree_attention_speculative_gb300 as ts
    g = W.rng(5, "forest-reject")
    par = np.stack([W.forest_random(g, 20, 3, 4), W.tree_random_levels(g, 20, 4)]).astype(np.int32)
    p = torch.from_numpy(par).cuda()
    pl = torch.zeros(2, dtype=torch.int32, device="cuda")
    anc = torch.zeros(2, 20, 1, dtype=torch.int64, device="cuda")
    d, pos = torch.zeros(2, 20, dtype=torch.int32, device="cuda"), torch.zeros(2, 20, dtype=torch.int32, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    ts.tree_build_ancestry(p, pl, anc, d, pos, st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [-3, 0]
    ts.tree_build_ancestry_forest(p, pl, anc, d, pos, st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, 0]
    a2, d2, p2, s2 = F.build_ancestry_forest(par, [0, 0])
    np.testing.assert_array_equal(anc.cpu().numpy().view(np.uint64), a2)
