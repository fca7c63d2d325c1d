"""tree_verify_greedy_noalloc: the verify entry point for callers that may not
allocate device memory (for example a plugin inside another serving engine
that is handed only its input and output buffers, or a latency-critical loop
where a cudaMalloc could stall the device).  It must give exactly what the
workspace-taking tree_verify_greedy gives, call after call, although every
call reuses the same library-owned scratch array.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _lib():
    from tree_attention_speculative_gb300 import _build
    _build.build()
    import tree_attention_speculative_gb300 as ts
    ts.lib()
    return ts


def _case(seed, B, N, V, plant):
    g = W.rng(seed, "noalloc")
    parents = np.stack([W.tree_random_levels(g, N, 8) for _ in range(B)])
    return W.build_case("noalloc", seed, parents, [4] * B, Hq=1, Hkv=1, D=64, bs=16, permute=False,
                        vocab=V, plant_len=plant)


def _outputs(B, N, max_depth, dev):
    i32 = dict(dtype=torch.int32, device=dev)
    return dict(accepted=torch.full((B, max_depth + 1), -7, **i32), accept_len=torch.full((B,), -7, **i32),
                bonus=torch.full((B,), -7, **i32), argmax=torch.full((B, N), -7, **i32),
                status=torch.zeros((B,), **i32))


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    ts = _lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cases = [_case(1, 6, 64, 128256, [0, 3, 8, 1, 5, 2]), _case(2, 9, 37, 20000, [4, 0, 2, 6, 1, 3, 8, 7, 5]),
             _case(1, 6, 64, 128256, [0, 3, 8, 1, 5, 2])]
    max_depth = 8
    for case in cases:
        draft = torch.from_numpy(case.draft).to(dev)
        logits = torch.from_numpy(case.logits).to(dev)
        parent = torch.from_numpy(case.parent).to(dev)
        # the existing entry point, with a caller-owned zeroed workspace
        ref = _outputs(case.B, case.N, max_depth, dev)
        ws = torch.zeros(ts.tree_verify_workspace_size(case.B, case.N, case.vocab), dtype=torch.uint8, device=dev)
        ts.tree_verify_greedy(draft, logits, parent, max_depth, ref["accepted"], ref["accept_len"], ref["bonus"],
                              ref["argmax"], ref["status"], ws)
        # the no-allocation entry point, twice in a row on the same inputs
        for _ in range(2):
            got = _outputs(case.B, case.N, max_depth, dev)
            ts.tree_verify_greedy_noalloc(draft, logits, parent, max_depth, got["accepted"], got["accept_len"],
                                          got["bonus"], got["argmax"], got["status"])
            torch.cuda.synchronize()
            for k in ref:
                assert torch.equal(got[k], ref[k]), k
        assert ref["accept_len"].cpu().tolist() == case.planted_len.tolist()
        # and the CPU oracle, which shares no code with either entry point
        acc, L, bonus, am, st = oracle.verify.verify_greedy(case.draft, case.logits, case.parent, max_depth)
        np.testing.assert_array_equal(got["accepted"].cpu().numpy(), acc)
        np.testing.assert_array_equal(got["accept_len"].cpu().numpy(), L)
        np.testing.assert_array_equal(got["bonus"].cpu().numpy(), bonus)
        np.testing.assert_array_equal(got["argmax"].cpu().numpy(), am)
        np.testing.assert_array_equal(got["status"].cpu().numpy(), st)


def test_noalloc_rejects_problems_beyond_its_scratch():
    ts = _lib()
    a = ctypes.c_void_p(0x10000)
    B, N, V = 2100, 256, 128256      # needs about 4.1 MiB of scratch (8 bytes a node)
    assert ts.tree_verify_workspace_size(B, N, V) > ts.NOALLOC_SCRATCH_BYTES
    st = ts.lib().tree_verify_greedy_noalloc(a, a, a, B, N, V, 8, a, a, a, a, a, None)
    assert st == -8     # TS_ERR_WORKSPACE, returned before anything is launched
    assert ts.tree_verify_workspace_size(4, 64, 128256) < ts.NOALLOC_SCRATCH_BYTES
