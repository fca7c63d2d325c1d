"""One verification step on the GPU: device buffers plus the three library calls.

``TreeVerifyStep`` owns the output and workspace buffers (allocated with torch,
which is only the allocator here) for fixed sizes and enqueues
tree_build_ancestry -> tree_attn_fwd -> tree_verify_greedy on one stream (their
_forest variants with ``forest=True``).  Every computation happens in the
library's kernels.  ``PackedInputs`` stages a step's inputs from host memory
in one copy.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import (attn_params, tree_attn_fwd, tree_attn_workspace_size, tree_build_ancestry,
               tree_build_ancestry_forest, tree_verify_greedy, tree_verify_greedy_forest,
               tree_verify_workspace_size)


class PackedInputs:
    """A step's inputs packed into one pinned host buffer and one device buffer
    (every tensor at a 256-byte aligned offset), so that the whole host-to-device
    upload of a step is a single copy, which can run on a stream of its own
    while the previous step computes.

    ``arrays`` maps names to CPU tensors (any dtype); ``device(name)`` is the
    device view to hand to the library's calls, ``upload(stream)`` enqueues the
    copy.  Torch is only the allocator and the copy call here.
    """

    ALIGN = 256

    def __init__(self, arrays: dict, device):
        self.layout = {}
        off = 0
        for name, t in arrays.items():
            t = t.contiguous()
            self.layout[name] = (off, tuple(t.shape), t.dtype)
            off += -(-(t.numel() * t.element_size()) // self.ALIGN) * self.ALIGN
        self.nbytes = off
        self.host = torch.empty(off, dtype=torch.uint8)
        if torch.device(device).type == "cuda":
            self.host = self.host.pin_memory()
        self.dev = torch.empty(off, dtype=torch.uint8, device=device)
        for name, t in arrays.items():
            self.host_view(name).copy_(t)

    def _view(self, buf: torch.Tensor, name: str) -> torch.Tensor:
        off, shape, dtype = self.layout[name]
        n = int(np.prod(shape, dtype=np.int64)) * torch.empty((), dtype=dtype).element_size()
        return buf[off:off + n].view(dtype).view(shape)

    def host_view(self, name: str) -> torch.Tensor:
        return self._view(self.host, name)

    def device(self, name: str) -> torch.Tensor:
        return self._view(self.dev, name)

    def upload(self, stream=None) -> None:
        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream(self.dev.device)):
            self.dev.copy_(self.host, non_blocking=True)


class TreeVerifyStep:
    def __init__(self, B: int, N: int, Hq: int, Hkv: int, D: int, prefix_len_host, vocab: int = 0,
                 max_depth: Optional[int] = None, device="cuda", scale: float = 0.0, forest: bool = False):
        self.B, self.N, self.Hq, self.Hkv, self.D = B, N, Hq, Hkv, D
        self.forest = forest
        self.vocab = vocab
        self.max_depth = N - 1 if max_depth is None else max_depth
        self.scale = scale
        self.device = torch.device(device)
        self.prefix_len_host = np.ascontiguousarray(np.asarray(prefix_len_host, np.int32))
        W = (N + 63) // 64
        dev = self.device
        i32 = dict(dtype=torch.int32, device=dev)
        self.anc = torch.zeros(B, N, W, dtype=torch.int64, device=dev)
        self.depth = torch.zeros(B, N, **i32)
        self.pos = torch.zeros(B, N, **i32)
        self.status = torch.zeros(B, **i32)
        self.out = torch.empty(B, N, Hq, D, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(B, N, Hq, dtype=torch.float32, device=dev)
        self.ws_attn = None
        if vocab > 0:
            nb = tree_verify_workspace_size(B, N, vocab)
            # zero-filled once; the verify kernel leaves its counters at zero
            self.ws_verify = torch.zeros(nb, dtype=torch.uint8, device=dev)
            self.accepted = torch.empty(B, self.max_depth + 1, **i32)
            self.accept_len = torch.empty(B, **i32)
            self.bonus = torch.empty(B, **i32)
            self.argmax = torch.empty(B, N, **i32)

    def _params(self, q, k_cache, v_cache, block_table, prefix_len, k_tree, v_tree):
        return attn_params(q, k_cache, v_cache, block_table, prefix_len, self.prefix_len_host, k_tree, v_tree,
                           self.anc, self.pos, self.out, self.lse, self.status, scale=self.scale)

    def attn_workspace_bytes(self, q, k_cache, v_cache, block_table, prefix_len, k_tree, v_tree) -> int:
        return tree_attn_workspace_size(self._params(q, k_cache, v_cache, block_table, prefix_len, k_tree, v_tree))

    def ancestry(self, parent, prefix_len, stream=None):
        build = tree_build_ancestry_forest if self.forest else tree_build_ancestry
        build(parent, prefix_len, self.anc, self.depth, self.pos, self.status, stream)

    def attention(self, q, k_cache, v_cache, block_table, prefix_len, k_tree, v_tree, stream=None):
        p = self._params(q, k_cache, v_cache, block_table, prefix_len, k_tree, v_tree)
        need = tree_attn_workspace_size(p)
        if need == 0:
            raise ValueError("tree_attn_fwd would reject these arguments")
        if self.ws_attn is None or self.ws_attn.numel() < need:
            # zero-filled once; every call leaves its head (the item counter) zero again
            self.ws_attn = torch.zeros(need, dtype=torch.uint8, device=self.device)
        tree_attn_fwd(p, self.ws_attn, stream)

    def verify(self, draft, logits, parent, stream=None):
        verify = tree_verify_greedy_forest if self.forest else tree_verify_greedy
        verify(draft, logits, parent, self.max_depth, self.accepted, self.accept_len, self.bonus, self.argmax,
               self.status, self.ws_verify, stream)

    def run(self, parent, prefix_len, q, k_cache, v_cache, block_table, k_tree, v_tree, draft=None, logits=None,
            stream=None):
        self.ancestry(parent, prefix_len, stream)
        self.attention(q, k_cache, v_cache, block_table, prefix_len, k_tree, v_tree, stream)
        if logits is not None:
            self.verify(draft, logits, parent, stream)
