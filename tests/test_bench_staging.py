"""Host logic of bench.py's end-to-end staging, on CPU: one flat buffer carved
into contiguous, typed, 256-byte-aligned views that cover disjoint bytes, so
that a step's inputs (and its outputs) move as one copy."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_staged_views_are_aligned_disjoint_and_typed():
    import bench
    specs = [((1, 3314, 28, 128), torch.bfloat16), ((1, 3314, 4, 128), torch.bfloat16),
             ((1, 3314, 4, 128), torch.bfloat16), ((1, 28, 3314), torch.float32), ((3,), torch.int32)]
    buf, views = bench._staged(specs, torch.device("cpu"))
    assert buf.dtype == torch.uint8 and buf.dim() == 1
    base = buf.data_ptr()
    spans = []
    for (shape, dtype), v in zip(specs, views):
        assert tuple(v.shape) == shape and v.dtype == dtype and v.is_contiguous()
        off = v.data_ptr() - base
        assert off % 256 == 0
        spans.append((off, off + v.numel() * v.element_size()))
    spans.sort()
    assert spans[0][0] == 0 and spans[-1][1] <= buf.numel()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:])), "views overlap"
    # writing through the views lands in the flat buffer, and a copy of the
    # buffer carries every view's contents
    for i, v in enumerate(views):
        v.fill_(i + 1)
    copy = buf.clone()
    for i, ((shape, dtype), v) in enumerate(zip(specs, views)):
        off = v.data_ptr() - base
        n = v.numel() * v.element_size()
        assert torch.equal(copy[off:off + n].view(dtype).view(shape), v)
        assert torch.all(v == i + 1)
