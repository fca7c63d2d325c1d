"""Python binding of libtreespec (GB300 tree-attention speculative verification).

Argument marshalling only: every function below forwards torch tensors'
device pointers, sizes and the current CUDA stream to the C entry point of
the same name in ``include/treespec.h`` and raises ``TreeSpecError`` on a
non-zero status.  All work runs in the library's CUDA kernels; there is no
other implementation behind these names, and the package refuses to work if
the library has not been built (``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

from ._build import LIB as LIB_PATH

__all__ = [
    "TreeSpecError", "lib", "ts_status_str", "tree_build_ancestry", "AttnParams", "attn_params",
    "tree_attn_workspace_size", "tree_attn_plan", "tree_attn_plan_order", "tree_attn_fwd",
    "tree_verify_workspace_size", "tree_verify_greedy",
    "tree_verify_greedy_noalloc", "tree_commit_accepted", "tree_verify_stochastic", "tree_build_dynamic",
    "tree_build_ancestry_forest", "tree_verify_greedy_forest", "NOALLOC_SCRATCH_BYTES",
    "STATUS",
]

STATUS = {
    0: "TS_OK", -1: "TS_ERR_NULL", -2: "TS_ERR_SHAPE", -3: "TS_ERR_BAD_TREE", -4: "TS_ERR_UNSUPPORTED",
    -5: "TS_ERR_BAD_BLOCK", -6: "TS_ERR_TIMEOUT", -7: "TS_ERR_CUDA", -8: "TS_ERR_WORKSPACE",
}


class TreeSpecError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({ts_status_str(status)})")


class AttnParams(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("prefix_len", ctypes.c_void_p),
        ("prefix_len_host", ctypes.c_void_p), ("k_tree", ctypes.c_void_p), ("v_tree", ctypes.c_void_p),
        ("anc_mask", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("lse", ctypes.c_void_p), ("status", ctypes.c_void_p),
        ("B", ctypes.c_int), ("N", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("D", ctypes.c_int), ("block_size", ctypes.c_int), ("num_blocks", ctypes.c_int),
        ("max_blocks", ctypes.c_int), ("scale", ctypes.c_float), ("rope_theta", ctypes.c_float),
    ]


_LIB: Optional[ctypes.CDLL] = None

# every symbol include/treespec.h declares
EXPORTS = ("ts_status_str", "tree_build_ancestry", "tree_attn_workspace_size", "tree_attn_plan", "tree_attn_plan_order",
           "tree_attn_fwd",
           "tree_verify_workspace_size", "tree_verify_greedy", "tree_verify_greedy_noalloc",
           "tree_commit_accepted", "tree_verify_stochastic", "tree_build_dynamic", "tree_build_ancestry_forest",
           "tree_verify_greedy_forest", "tree_attn_fwd_stall_test", "tree_attn_fwd_ctas_test")

# TS_VERIFY_NOALLOC_SCRATCH_BYTES of treespec.h
NOALLOC_SCRATCH_BYTES = 4 << 20


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtreespec is not built ({LIB_PATH} missing); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.ts_status_str.argtypes = [i32]
        L.ts_status_str.restype = ctypes.c_char_p
        L.tree_build_ancestry.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, vp]
        L.tree_build_ancestry.restype = i32
        L.tree_attn_workspace_size.argtypes = [ctypes.POINTER(AttnParams)]
        L.tree_attn_workspace_size.restype = sz
        L.tree_attn_plan.argtypes = [ctypes.POINTER(AttnParams), vp, vp, vp]
        L.tree_attn_plan.restype = i32
        L.tree_attn_plan_order.argtypes = [ctypes.POINTER(AttnParams), vp, i32, vp]
        L.tree_attn_plan_order.restype = i32
        L.tree_attn_fwd.argtypes = [ctypes.POINTER(AttnParams), vp, sz, vp]
        L.tree_attn_fwd.restype = i32
        L.tree_attn_fwd_stall_test.argtypes = [ctypes.POINTER(AttnParams), vp, sz, i32, i32, ctypes.c_uint32, vp]
        L.tree_attn_fwd_stall_test.restype = i32
        L.tree_attn_fwd_ctas_test.argtypes = [ctypes.POINTER(AttnParams), vp, sz, i32, i32, i32, ctypes.c_uint32, vp]
        L.tree_attn_fwd_ctas_test.restype = i32
        L.tree_verify_workspace_size.argtypes = [i32, i32, i32]
        L.tree_verify_workspace_size.restype = sz
        L.tree_verify_greedy.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.tree_verify_greedy.restype = i32
        L.tree_verify_greedy_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.tree_verify_greedy_noalloc.restype = i32
        L.tree_commit_accepted.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                           vp, vp, vp]
        L.tree_commit_accepted.restype = i32
        L.tree_verify_stochastic.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_float, vp, vp, vp, vp,
                                             vp]
        L.tree_verify_stochastic.restype = i32
        L.tree_build_dynamic.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.tree_build_dynamic.restype = i32
        L.tree_build_ancestry_forest.argtypes = L.tree_build_ancestry.argtypes
        L.tree_build_ancestry_forest.restype = i32
        L.tree_verify_greedy_forest.argtypes = L.tree_verify_greedy.argtypes
        L.tree_verify_greedy_forest.restype = i32
        _LIB = L
    return _LIB


def ts_status_str(status: int) -> str:
    return lib().ts_status_str(int(status)).decode()


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(st: int, where: str):
    if st != 0:
        raise TreeSpecError(st, where)


def tree_build_ancestry(parent_idx: torch.Tensor, prefix_len: torch.Tensor, anc_mask: torch.Tensor,
                        depth: torch.Tensor, pos: torch.Tensor, status: torch.Tensor, stream=None) -> None:
    """parent_idx [B,N] i32, prefix_len [B] i32 -> anc_mask [B,N,W] u64 (int64 tensor), depth, pos [B,N] i32, status [B] i32."""
    B, N = parent_idx.shape
    _check(lib().tree_build_ancestry(_p(parent_idx), _p(prefix_len), B, N, _p(anc_mask), _p(depth), _p(pos),
                                     _p(status), _s(stream)), "tree_build_ancestry")


def tree_build_ancestry_forest(parent_idx: torch.Tensor, prefix_len: torch.Tensor, anc_mask: torch.Tensor,
                               depth: torch.Tensor, pos: torch.Tensor, status: torch.Tensor, stream=None) -> None:
    """tree_build_ancestry for forests (several parent -1 entries; node 0 is a root)."""
    B, N = parent_idx.shape
    _check(lib().tree_build_ancestry_forest(_p(parent_idx), _p(prefix_len), B, N, _p(anc_mask), _p(depth), _p(pos),
                                            _p(status), _s(stream)), "tree_build_ancestry_forest")


def attn_params(q, k_cache, v_cache, block_table, prefix_len, prefix_len_host, k_tree, v_tree, anc_mask, pos,
                out, lse=None, status=None, scale: float = 0.0, rope_theta: float = 0.0) -> AttnParams:
    """Fill the C parameter block from tensors (shapes as in treespec.h).

    ``prefix_len_host`` is a host int32 tensor/array; the returned object keeps
    it alive.
    """
    B, N, Hq, D = q.shape
    nblk, Hkv, bs, _ = k_cache.shape
    host = np.ascontiguousarray(np.asarray(prefix_len_host.cpu() if torch.is_tensor(prefix_len_host)
                                           else prefix_len_host, dtype=np.int32))
    p = AttnParams(q=q.data_ptr(), k_cache=k_cache.data_ptr(), v_cache=v_cache.data_ptr(),
                   block_table=block_table.data_ptr(), prefix_len=prefix_len.data_ptr(),
                   prefix_len_host=host.ctypes.data, k_tree=k_tree.data_ptr(), v_tree=v_tree.data_ptr(),
                   anc_mask=anc_mask.data_ptr(), pos=pos.data_ptr() if pos is not None else None,
                   out=out.data_ptr(), lse=lse.data_ptr() if lse is not None else None,
                   status=status.data_ptr() if status is not None else None,
                   B=B, N=N, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, num_blocks=nblk,
                   max_blocks=block_table.shape[1], scale=scale, rope_theta=rope_theta)
    p._keep = (host,)
    return p


def tree_attn_workspace_size(params: AttnParams) -> int:
    return int(lib().tree_attn_workspace_size(ctypes.byref(params)))


def tree_attn_plan(params: AttnParams) -> dict:
    """The split plan tree_attn_fwd uses for these arguments (host only)."""
    c, s, t = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(lib().tree_attn_plan(ctypes.byref(params), ctypes.byref(c), ctypes.byref(s), ctypes.byref(t)),
           "tree_attn_plan")
    return {"chunk_tiles": c.value, "max_splits": s.value, "tree_split": t.value}


def tree_attn_plan_order(params: AttnParams) -> list:
    """The packed (sequence, split, first tile) entries in the order the
    attention kernel takes its items (host only); [] when it orders none."""
    n = ctypes.c_int32()
    buf = (ctypes.c_uint32 * 256)()  # the most pairs the kernel orders
    _check(lib().tree_attn_plan_order(ctypes.byref(params), buf, 256, ctypes.byref(n)), "tree_attn_plan_order")
    return [int(buf[i]) for i in range(n.value)]


def tree_attn_fwd(params: AttnParams, workspace: torch.Tensor, stream=None) -> None:
    _check(lib().tree_attn_fwd(ctypes.byref(params), _p(workspace), workspace.numel() * workspace.element_size(),
                               _s(stream)), "tree_attn_fwd")


def tree_attn_fwd_stall_test(params: AttnParams, workspace: torch.Tensor, stall_seq: int, stall_tile: int,
                             wait_limit_us: int, stream=None) -> None:
    """Testing only: tree_attn_fwd with sequence ``stall_seq``'s key stream
    stopped before tile ``stall_tile``, so its bounded wait runs out."""
    _check(lib().tree_attn_fwd_stall_test(ctypes.byref(params), _p(workspace),
                                          workspace.numel() * workspace.element_size(), stall_seq, stall_tile,
                                          wait_limit_us, _s(stream)), "tree_attn_fwd_stall_test")


def tree_attn_fwd_ctas_test(params: AttnParams, workspace: torch.Tensor, max_ctas: int, stall_seq: int = -1,
                            stall_tile: int = 0, wait_limit_us: int = 1000000, stream=None) -> None:
    """Testing only: tree_attn_fwd on at most ``max_ctas`` CTAs (and, with
    ``stall_seq >= 0``, that sequence's key stream stopped as in
    tree_attn_fwd_stall_test)."""
    _check(lib().tree_attn_fwd_ctas_test(ctypes.byref(params), _p(workspace),
                                         workspace.numel() * workspace.element_size(), max_ctas, stall_seq,
                                         stall_tile, wait_limit_us, _s(stream)), "tree_attn_fwd_ctas_test")


def tree_verify_workspace_size(B: int, N: int, V: int) -> int:
    return int(lib().tree_verify_workspace_size(B, N, V))


def tree_verify_greedy(draft_tokens, target_logits, parent_idx, max_depth: int, accepted, accept_len, bonus,
                       argmax_out, status, workspace, stream=None) -> None:
    B, N, V = target_logits.shape
    _check(lib().tree_verify_greedy(_p(draft_tokens), _p(target_logits), _p(parent_idx), B, N, V, max_depth,
                                    _p(accepted), _p(accept_len), _p(bonus), _p(argmax_out), _p(status),
                                    _p(workspace), workspace.numel() * workspace.element_size(), _s(stream)),
           "tree_verify_greedy")


def tree_verify_greedy_forest(draft_tokens, target_logits, parent_idx, max_depth: int, accepted, accept_len, bonus,
                              argmax_out, status, workspace, stream=None) -> None:
    """tree_verify_greedy for forests; same workspace size."""
    B, N, V = target_logits.shape
    _check(lib().tree_verify_greedy_forest(_p(draft_tokens), _p(target_logits), _p(parent_idx), B, N, V, max_depth,
                                           _p(accepted), _p(accept_len), _p(bonus), _p(argmax_out), _p(status),
                                           _p(workspace), workspace.numel() * workspace.element_size(), _s(stream)),
           "tree_verify_greedy_forest")


def tree_commit_accepted(k_tree, v_tree, accepted, accept_len, prefix_len, k_cache, v_cache, block_table,
                         new_prefix_len, status=None, stream=None) -> None:
    """Append the accepted path (root .. n*) of every sequence to the paged cache."""
    B, N, Hkv, D = k_tree.shape
    nblk, _, bs, _ = k_cache.shape
    _check(lib().tree_commit_accepted(_p(k_tree), _p(v_tree), _p(accepted), _p(accept_len), _p(prefix_len),
                                      _p(k_cache), _p(v_cache), _p(block_table), B, N, Hkv, D, bs, nblk,
                                      block_table.shape[1], accepted.shape[1] - 1, _p(new_prefix_len), _p(status),
                                      _s(stream)), "tree_commit_accepted")


def tree_verify_stochastic(draft_tokens, target_logits, draft_probs, parent_idx, coins, temperature: float,
                           accepted, accept_len, bonus, status, stream=None) -> None:
    """Rejection-sampling verification at the given temperature; max_depth is
    accepted.shape[1] - 1.  coins [B, N] are the uniforms the walk consumes."""
    B, N, V = target_logits.shape
    _check(lib().tree_verify_stochastic(_p(draft_tokens), _p(target_logits), _p(draft_probs), _p(parent_idx),
                                        _p(coins), B, N, V, accepted.shape[1] - 1, float(temperature),
                                        _p(accepted), _p(accept_len), _p(bonus), _p(status), _s(stream)),
           "tree_verify_stochastic")


def tree_build_dynamic(pool_parent, pool_logp, pool_token, prefix_len, parent_idx, draft_tokens, sel_index,
                       anc_mask, depth, pos, status, stream=None) -> None:
    """Rerank a candidate pool [B, M] into the N-node tree of parent_idx [B, N]
    and build its masks, depths and positions."""
    B, M = pool_parent.shape
    N = parent_idx.shape[1]
    _check(lib().tree_build_dynamic(_p(pool_parent), _p(pool_logp), _p(pool_token), _p(prefix_len), B, M, N,
                                    _p(parent_idx), _p(draft_tokens), _p(sel_index), _p(anc_mask), _p(depth),
                                    _p(pos), _p(status), _s(stream)), "tree_build_dynamic")


def tree_verify_greedy_noalloc(draft_tokens, target_logits, parent_idx, max_depth: int, accepted, accept_len, bonus,
                               argmax_out, status, stream=None) -> None:
    """tree_verify_greedy without a workspace, for callers that may not allocate
    device memory (e.g. a plugin handed only its input/output buffers).  Runs on
    a fixed 4 MiB scratch array inside the library; larger problems raise
    TS_ERR_WORKSPACE.  Calls on one device share that array, so keep them
    ordered on one stream; make the first call on a device outside any stream
    capture (it looks up the array's device address)."""
    B, N, V = target_logits.shape
    _check(lib().tree_verify_greedy_noalloc(_p(draft_tokens), _p(target_logits), _p(parent_idx), B, N, V, max_depth,
                                            _p(accepted), _p(accept_len), _p(bonus), _p(argmax_out), _p(status),
                                            _s(stream)), "tree_verify_greedy_noalloc")
