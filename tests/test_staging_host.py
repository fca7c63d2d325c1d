"""Host-side checks of PackedInputs (one pinned buffer per step's inputs):
every tensor sits at a 256-byte aligned offset and its view reproduces the
input bit for bit.  Runs on the CPU (device "cpu", no pinning)."""
import numpy as np
import torch

from tree_attention_speculative_gb300.step import PackedInputs


def test_packed_views_are_aligned_and_exact():
    g = np.random.default_rng(0)
    arrays = {
        "parent": torch.from_numpy(g.integers(-1, 5, (3, 7)).astype(np.int32)),
        "q": torch.from_numpy(g.standard_normal((2, 5, 4, 64)).astype(np.float32)).to(torch.bfloat16),
        "prefix_len": torch.tensor([17], dtype=torch.int32),
        "logits": torch.from_numpy(g.standard_normal((2, 5, 1001)).astype(np.float32)),
    }
    p = PackedInputs(arrays, "cpu")
    assert p.nbytes % 256 == 0
    for name, t in arrays.items():
        off, shape, dtype = p.layout[name]
        assert off % 256 == 0 and shape == tuple(t.shape) and dtype == t.dtype
        for view in (p.host_view(name), p.device(name)):
            assert view.dtype == t.dtype and tuple(view.shape) == tuple(t.shape)
        assert torch.equal(p.host_view(name).view(torch.uint8), t.contiguous().view(torch.uint8))
    # the views do not overlap
    spans = sorted((off, off + arrays[n].numel() * arrays[n].element_size()) for n, (off, _, _) in p.layout.items())
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    # the device buffer receives everything in one copy
    p.dev.copy_(p.host)
    for name, t in arrays.items():
        assert torch.equal(p.device(name).view(torch.uint8), t.contiguous().view(torch.uint8))
