"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Integer outputs (ancestry words, depths, positions, argmax, accepted paths,
lengths, bonus tokens, status codes) must match bit for bit.  Attention
outputs are bf16 and must satisfy |out - ref| <= 1e-2 + 1e-2 |ref| against the
fp64 oracle; the natural-log lse must be within 1e-3.
Small cases are compared element by element; the five named workloads at full
size are compared on every output row the oracle can afford (all rows for the
small ones, seeded samples of (sequence, kv head) units for the large ones).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import SMALL, LSE_ATOL, assert_close_attention, out_f64, run_case, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tree_attention_speculative_gb300 import _build
    _build.build()
    import tree_attention_speculative_gb300 as ts
    ts.lib()
    torch.cuda.init()


# --------------------------------------------------------------------------- ancestry

def _anc_gpu(parent, prefix_len):
    from tree_attention_speculative_gb300 import tree_build_ancestry
    B, N = parent.shape
    W_ = (N + 63) // 64
    dev = "cuda"
    anc = torch.full((B, N, W_), -7, dtype=torch.int64, device=dev)
    depth = torch.full((B, N), -7, dtype=torch.int32, device=dev)
    pos = torch.full((B, N), -7, dtype=torch.int32, device=dev)
    status = torch.full((B,), -7, dtype=torch.int32, device=dev)
    tree_build_ancestry(torch.from_numpy(parent.astype(np.int32)).to(dev),
                        torch.from_numpy(prefix_len.astype(np.int32)).to(dev), anc, depth, pos, status)
    torch.cuda.synchronize()
    return (anc.cpu().numpy().view(np.uint64), depth.cpu().numpy(), pos.cpu().numpy(), status.cpu().numpy())


@pytest.mark.parametrize("n", [1, 2, 5, 31, 32, 33, 63, 64, 65, 127, 128, 129, 192, 200, 255, 256])
def test_ancestry_random_trees_bit_exact(n):
    g = W.rng(n, "anc")
    parents = np.stack([W.tree_random_recursive(g, n), W.tree_chain(n), W.tree_star(n),
                        W.tree_random_levels(g, n, 10)])
    plen = np.array([0, 1, 131072, 4096], np.int32)
    got = _anc_gpu(parents, plen)
    ref = oracle.tree.build_ancestry(parents, plen)
    for x, y in zip(got, ref):
        np.testing.assert_array_equal(x, y)


def test_ancestry_worked_example_and_invalid_trees():
    parents = np.array([[-1, 0, 0, 1, 2], [-1, 0, 0, 4, 2], [0, 0, 0, 1, 2], [-1, 0, -1, 1, 2],
                        [-1, 0, 0, 1, 7]], np.int32)
    plen = np.array([16, 16, 16, 16, 16], np.int32)
    got = _anc_gpu(parents, plen)
    ref = oracle.tree.build_ancestry(parents, plen)
    for x, y in zip(got, ref):
        np.testing.assert_array_equal(x, y)
    assert got[0][0, :, 0].tolist() == [1, 3, 5, 11, 21]
    assert got[3].tolist() == [0, -3, -3, -3, -3]


# --------------------------------------------------------------------------- attention

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


@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_attention_small_elementwise(spec):
    case = _small_case(*spec)
    step, _ = run_case(case)
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    assert step.status.cpu().tolist() == [0] * case.B
    assert_close_attention(out_f64(step), ref, spec[0])
    np.testing.assert_allclose(step.lse.cpu().numpy(), ref_lse, rtol=0, atol=LSE_ATOL)


@pytest.mark.parametrize("plens", [[896, 300], [1000, 129], [1920, 640], [2000, 0]],
                         ids=["8-splits", "9-splits", "16-splits", "17-splits"])
def test_attention_combine_group_boundaries(plens):
    """Split counts on both sides of the combine's load groups (8 and 16 splits
    a round trip), with a second, shorter sequence whose rows use fewer splits
    than the grid holds."""
    case = _small_case("groups", 2, 33, 4, 1, 128, plens, 64, "levels")
    step, _ = run_case(case)
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    assert step.status.cpu().tolist() == [0, 0]
    assert_close_attention(out_f64(step), ref, f"splits {plens}")
    np.testing.assert_allclose(step.lse.cpu().numpy(), ref_lse, rtol=0, atol=LSE_ATOL)


def test_attention_combine_of_few_splits_d64():
    """Plans of 2..4 splits are merged by the combine's 16-channel form (two
    16-byte pieces a lane, splits in groups of 4); with D = 64 a row is 4 lanes."""
    import tree_attention_speculative_gb300 as ts
    g = W.rng(21, "c16")
    plens = [3000, 2900, 400, 2000] * 4
    parent = np.stack([W.tree_random_levels(g, 20, 5) for _ in plens])
    case = W.build_case("c16", 21, parent, plens, Hq=8, Hkv=8, D=64, bs=16, permute=True)
    step, t = run_case(case)
    p = step._params(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"], t["k_tree"], t["v_tree"])
    assert 2 <= ts.tree_attn_plan(p)["max_splits"] <= 4
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    assert step.status.cpu().tolist() == [0] * case.B
    assert_close_attention(out_f64(step), ref, "few splits, D = 64")
    np.testing.assert_allclose(step.lse.cpu().numpy(), ref_lse, rtol=0, atol=LSE_ATOL)


def test_attention_hot_keys_softmax_range():
    case = W.build_case("hot", 3, W.tree_random_levels(W.rng(1, "h"), 48, 6), [700, 1500], Hq=8, Hkv=2,
                        D=128, bs=64, permute=True, hot_key_frac=0.05, hot_key_scale=8.0)
    step, _ = run_case(case)
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    assert_close_attention(out_f64(step), ref, "hot keys")
    np.testing.assert_allclose(step.lse.cpu().numpy(), ref_lse, rtol=0, atol=LSE_ATOL)


def test_attention_bad_block_id_reported():
    case = _small_case("g4_ragged", 2, 37, 8, 2, 128, [0, 300], 16, "random")
    case.block_table[1, 3] = case.num_blocks + 5
    step, _ = run_case(case)
    assert step.status.cpu().tolist() == [0, -5]


def test_attention_deterministic():
    case = _small_case("g2_multi_tile", 3, 70, 4, 2, 128, [129, 1, 640], 32, "levels")
    s1, _ = run_case(case)
    o1 = s1.out.clone()
    s2, _ = run_case(case)
    assert torch.equal(o1, s2.out)


# --------------------------------------------------------------------------- verify

def _verify_check(case, max_depth):
    step, _ = run_case(case, max_depth=max_depth)
    acc, L, bonus, am, st = oracle.verify.verify_greedy(case.draft, case.logits, case.parent, max_depth)
    np.testing.assert_array_equal(step.argmax.cpu().numpy(), am)
    np.testing.assert_array_equal(step.status.cpu().numpy(), st)
    np.testing.assert_array_equal(step.accept_len.cpu().numpy(), L)
    np.testing.assert_array_equal(step.bonus.cpu().numpy(), bonus)
    np.testing.assert_array_equal(step.accepted.cpu().numpy(), acc)
    _assert_tickets_zero(step, case.B, case.N)
    return step, acc, L


def _assert_tickets_zero(step, B, N):
    """The verify workspace (a packed argmax key per node, then an arrival counter
    per sequence) is all zero again after the call, ready for the next one."""
    ws = step.ws_verify.cpu().numpy()
    assert not ws.any()


@pytest.mark.parametrize("vocab", [13, 1000, 8192, 8193, 20000, 128256])
def test_verify_planted(vocab):
    g = W.rng(vocab, "v")
    B, N = 5, 33
    if vocab < 100:   # a chain: one child per node, so a small vocabulary can still plant
        parents = np.stack([W.tree_chain(N)] * B)
    else:
        parents = np.stack([W.tree_random_levels(g, N, 6) for _ in range(B)])
    plant = [0, 1, 3, 6, 2]
    case = W.build_case("v", vocab, parents, [4] * B, Hq=1, Hkv=1, D=64, bs=16, permute=False,
                        vocab=vocab, plant_len=plant)
    step, acc, L = _verify_check(case, 6)
    assert L.tolist() == plant


def test_verify_ties_and_chunk_boundaries():
    B, N, V = 2, 6, 3 * 8192 + 4
    parent = W.tree_chain(N)
    case = W.build_case("t", 1, parent, [4, 4], Hq=1, Hkv=1, D=64, bs=16, permute=False, vocab=V, plant_len=[2, 0])
    lg = case.logits
    lg[0, 3, :] = 0.0
    lg[0, 3, 8191] = 5.0
    lg[0, 3, 8192] = 5.0          # tie across a chunk boundary: first wins
    lg[1, 0, V - 1] = 50.0
    lg[1, 0, 2 * 8192] = 50.0     # tie between chunk 2's first and the row's last
    lg[1, 2, :] = -1.0
    lg[1, 2, 0] = -0.5
    _verify_check(case, 5)


@pytest.mark.parametrize("first", ["neg", "pos"])
def test_verify_signed_zero_tie_across_chunks(first):
    """A row whose maximum is zero, held by -0.0 and +0.0 in different 8192-logit
    chunks (one CTA each): the two compare equal, so the first index wins,
    whichever sign comes first and wherever the chunk boundaries fall."""
    B, N, V = 2, 4, 3 * 8192 + 8
    case = W.build_case("z", 5, W.tree_chain(N), [4, 4], Hq=1, Hkv=1, D=64, bs=16, permute=False, vocab=V,
                        plant_len=[0, 0])
    lg = case.logits
    a, b = (np.float32(-0.0), np.float32(0.0)) if first == "neg" else (np.float32(0.0), np.float32(-0.0))
    for s in range(B):
        for r in range(N):
            lg[s, r, :] = -1.0
    lg[0, 0, 100] = a               # chunk 0
    lg[0, 0, 2 * 8192 + 5] = b      # chunk 2
    lg[0, 1, 8191] = a              # the last of chunk 0 ...
    lg[0, 1, 8192] = b              # ... and the first of chunk 1
    lg[1, 2, 8192 + 3] = a          # chunk 1
    lg[1, 2, V - 1] = b             # the row's scalar tail, chunk 3
    lg[1, 3, 0] = a                 # index 0 against the next CTA's zero
    lg[1, 3, 8192] = b
    step, acc, L = _verify_check(case, 3)
    am = step.argmax.cpu().numpy()
    assert am[0, 0] == 100 and am[0, 1] == 8191 and am[1, 2] == 8192 + 3 and am[1, 3] == 0


@pytest.mark.parametrize("vocab", [3, 8])
def test_verify_duplicate_sibling_drafts(vocab):
    """Several valid paths: drafts and argmax drawn from a tiny vocabulary, so
    siblings often share a draft token and more than one root path matches.  The
    deepest accepted node wins, the smaller index on ties; paths, lengths, bonus
    and argmax must equal the oracle's bit for bit over hundreds of trees."""
    g = W.rng(vocab, "dup")
    B, N = 400, 12
    parents = np.stack([W.tree_random_recursive(g, N) if b % 2 else W.tree_random_levels(g, N, 4)
                        for b in range(B)])
    case = W.build_case("dup", vocab, parents, [4] * B, Hq=1, Hkv=1, D=64, bs=16, permute=False)
    case.vocab = vocab
    case.draft = g.integers(0, 3, size=(B, N)).astype(np.int32)
    lg = g.standard_normal((B, N, vocab)).astype(np.float32)
    want = g.integers(0, 3, size=(B, N))           # the planted argmax, also from {0, 1, 2}
    np.put_along_axis(lg, want[..., None], lg.max(axis=-1, keepdims=True) + np.float32(1.0), axis=-1)
    case.logits = lg
    step, acc, L = _verify_check(case, N - 1)
    # the inputs really hold several valid paths in many sequences: more
    # accepted nodes than one path of length L can hold
    am = oracle.verify.greedy_argmax(case.logits)
    several = 0
    for b in range(B):
        ok = np.zeros(N, bool)
        for c in range(1, N):
            ok[c] = (ok[case.parent[b, c]] or case.parent[b, c] == 0) and case.draft[b, c] == am[b, case.parent[b, c]]
        several += int(ok.sum()) > int(L[b])
    assert several > B // 10 and L.max() >= 3


def test_verify_negative_infinity_rows():
    """Masked logits: a row of nothing but -inf takes index 0 (the first maximum),
    and -inf entries never beat a finite one, across chunk boundaries."""
    B, N, V = 2, 5, 2 * 8192 + 20
    case = W.build_case("ninf", 3, W.tree_chain(N), [4, 4], Hq=1, Hkv=1, D=64, bs=16, permute=False, vocab=V,
                        plant_len=[1, 0])
    lg = case.logits
    lg[0, 1, :] = -np.inf
    lg[0, 2, :] = -np.inf
    lg[0, 2, 8192 + 7] = -3e38    # the only finite value, in the second chunk
    lg[1, 3, : 8192] = -np.inf
    lg[1, 4, 1:] = -np.inf        # finite only at index 0
    _verify_check(case, 4)


def test_verify_path_too_long_and_bad_tree():
    g = W.rng(3, "x")
    parents = np.stack([W.tree_chain(12), W.tree_random_levels(g, 12, 5), W.tree_chain(12)])
    case = W.build_case("t", 2, parents, [4] * 3, Hq=1, Hkv=1, D=64, bs=16, permute=False, vocab=300,
                        plant_len=[11, 5, 2])
    case.parent[2, 5] = 9          # invalid: parent after child
    step, acc, L = _verify_check(case, 4)
    assert step.status.cpu().tolist() == [-2, -2, -3]


def test_verify_repeated_calls_reuse_workspace():
    case = W.c1()
    s1, _ = run_case(case, max_depth=4)
    t = to_dev(case)
    for _ in range(3):
        s1.verify(t["draft"], t["logits"], t["parent"])
    torch.cuda.synchronize()
    assert s1.accepted.cpu().tolist() == [[0, 1, 3, -1, -1]]
    _assert_tickets_zero(s1, case.B, case.N)


# --------------------------------------------------------------------------- the named workloads

def test_c1_full():
    case = W.c1()
    step, _ = run_case(case, max_depth=4)
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    assert_close_attention(out_f64(step), ref, "c1")
    np.testing.assert_allclose(step.lse.cpu().numpy(), ref_lse, rtol=0, atol=LSE_ATOL)
    anc, dep, pos, st = oracle.tree.build_ancestry(case.parent, case.prefix_len)
    np.testing.assert_array_equal(step.anc.cpu().numpy().view(np.uint64), anc)
    np.testing.assert_array_equal(step.pos.cpu().numpy(), pos)
    assert step.accepted.cpu().tolist() == [[0, 1, 3, -1, -1]]
    assert step.accept_len.cpu().tolist() == [2]


def test_c2_full():
    case = W.c2()
    step, _ = run_case(case, max_depth=6)
    ref, ref_lse = oracle.attention.tree_attention_case(case)
    assert_close_attention(out_f64(step), ref, "c2")
    np.testing.assert_allclose(step.lse.cpu().numpy(), ref_lse, rtol=0, atol=LSE_ATOL)
    acc, L, bonus, am, st = oracle.verify.verify_greedy(case.draft, case.logits, case.parent, 6)
    np.testing.assert_array_equal(step.accepted.cpu().numpy(), acc)
    np.testing.assert_array_equal(step.argmax.cpu().numpy(), am)
    assert L.tolist() == case.planted_len.tolist()


def _sampled_units(case, k, seed):
    """k distinct (sequence, kv head) units drawn with a fixed seed, plus the first and the last."""
    g = np.random.default_rng(seed)
    pick = g.choice(case.B * case.Hkv, size=min(k, case.B * case.Hkv), replace=False)
    units = {(int(u) // case.Hkv, int(u) % case.Hkv) for u in pick}
    units |= {(0, 0), (case.B - 1, case.Hkv - 1)}
    return sorted(units)


@pytest.mark.parametrize("name,k", [("c3", None), ("c4", 64), ("c5", None)])
def test_named_workload_sampled(name, k):
    """c3 and c5 check every (sequence, kv head) unit; c4 a seeded sample of
    64 of its 512 units plus the first and the last."""
    case = W.make(name)
    vocab = case.vocab
    step, _ = run_case(case, max_depth=12 if vocab else None)
    units = (sorted((b, h) for b in range(case.B) for h in range(case.Hkv)) if k is None
             else _sampled_units(case, k, 99))
    ref, ref_lse = oracle.attention.tree_attention_case(case, units=units)
    got = out_f64(step)
    glse = step.lse.cpu().numpy()
    G = case.G
    for b, g in units:
        hs = slice(g * G, (g + 1) * G)
        assert_close_attention(got[b, :, hs], ref[b, :, hs], f"{name} unit {(b, g)}")
        np.testing.assert_allclose(glse[b, :, hs], ref_lse[b, :, hs], rtol=0, atol=LSE_ATOL)
    assert np.isfinite(got).all()
    assert step.status.cpu().tolist() == [0] * case.B
    anc, dep, pos, st = oracle.tree.build_ancestry(case.parent, case.prefix_len)
    np.testing.assert_array_equal(step.anc.cpu().numpy().view(np.uint64), anc)
    np.testing.assert_array_equal(step.pos.cpu().numpy(), pos)
    if vocab:
        acc, L, bonus, am, st = oracle.verify.verify_greedy(case.draft, case.logits, case.parent, 12)
        np.testing.assert_array_equal(step.argmax.cpu().numpy(), am)
        np.testing.assert_array_equal(step.accepted.cpu().numpy(), acc)
        np.testing.assert_array_equal(step.bonus.cpu().numpy(), bonus)
        assert L.tolist() == case.planted_len.tolist()
