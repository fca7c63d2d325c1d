"""Helpers for the GPU parity tests: move a ``workloads.Case`` to the device and
run one verification step through the library's C ABI."""
import numpy as np
import torch

# Attention cases compared element by element with the oracle:
# name, B, N, Hq, Hkv, D, prefix lengths, block size, tree kind.  Between them
# they take every layout the split planner can choose (tests/test_abi_host.py
# checks that): one split per unit (the kernel writes the output itself), the
# tree block on the last prefix split, and the tree block on a split of its own.
SMALL = [
    ("g4_ragged", 2, 37, 8, 2, 128, [0, 300], 16, "random"),
    ("g1_d64", 1, 5, 2, 2, 64, [16], 16, "worked"),
    ("g2_multi_tile", 3, 70, 4, 2, 128, [129, 1, 640], 32, "levels"),
    ("g8_rows_over_tile", 2, 40, 16, 2, 128, [257, 96], 64, "random"),
    ("g16", 1, 9, 16, 1, 64, [383], 128, "chain"),
    ("w3_192_nodes", 1, 192, 2, 1, 128, [200], 16, "levels"),
    ("w4_256_nodes", 1, 256, 1, 1, 64, [0], 16, "random"),
    ("contiguous_2k", 2, 26, 8, 2, 128, [2048, 2048], 2048, "widths"),
    ("tree_on_last_split", 5, 130, 8, 8, 128, [6000, 5963, 5926, 5889, 5852], 16, "levels"),
    ("one_split_per_unit", 16, 26, 32, 8, 128, [1500 - 37 * i for i in range(16)], 16, "widths"),
    # block sizes that neither divide a 128-token tile nor are multiples of it
    ("bs48", 2, 37, 8, 2, 128, [300, 1000], 48, "random"),
    ("bs144", 1, 40, 16, 2, 128, [700], 144, "levels"),
    ("bs80_d64", 2, 20, 4, 2, 64, [333, 150], 80, "random"),
    # a contiguous cache whose prefixes are not multiples of 16: one 304-row block per sequence
    ("contiguous_300", 2, 26, 8, 2, 128, [300, 290], 304, "widths"),
]

ATOL = 1e-2   # |out - ref| <= ATOL + RTOL * |ref| for bf16 attention outputs
RTOL = 1e-2
LSE_ATOL = 1e-3


def to_dev(case, dev="cuda"):
    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

    def i32(x):
        return torch.from_numpy(np.ascontiguousarray(x, np.int32)).to(dev)

    t = dict(parent=i32(case.parent), prefix_len=i32(case.prefix_len), q=bf(case.q), k_cache=bf(case.k_cache),
             v_cache=bf(case.v_cache), block_table=i32(case.block_table), k_tree=bf(case.k_tree),
             v_tree=bf(case.v_tree))
    if case.logits is not None:
        t["draft"] = i32(case.draft)
        t["logits"] = torch.from_numpy(case.logits).to(dev)
    return t


def run_case(case, max_depth=None, scale=0.0):
    from tree_attention_speculative_gb300.step import TreeVerifyStep
    t = to_dev(case)
    step = TreeVerifyStep(case.B, case.N, case.Hq, case.Hkv, case.D, case.prefix_len, vocab=case.vocab,
                          max_depth=max_depth, scale=scale)
    step.run(t["parent"], t["prefix_len"], t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["k_tree"],
             t["v_tree"], t.get("draft"), t.get("logits"))
    torch.cuda.synchronize()
    return step, t


def out_f64(step):
    return step.out.float().cpu().numpy().astype(np.float64)


def assert_close_attention(got, ref, what=""):
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {idx.tolist()} "
                             f"got {got[tuple(idx[0])]} ref {ref[tuple(idx[0])]} max err {err.max()}")
