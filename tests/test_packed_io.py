"""The round's host-facing tensors share one allocation per direction
(runtime._packed): every view starts on a 256-byte boundary, no two views
overlap, the buffer starts zeroed, and one copy of the flat buffer carries
every tensor (what the end-to-end loop relies on)."""
import torch

from eagle_feature_level_gb300.runtime import _packed


SPECS = [((3,), torch.int32), ((3, 64), torch.float32), ((3,), torch.int32), ((3,), torch.float32),
         ((3, 27, 1000), torch.float32), ((3, 27, 64), torch.float32), ((3, 27, 4, 32), torch.bfloat16),
         ((3, 27, 2, 32), torch.bfloat16), ((3, 27, 2, 32), torch.bfloat16), ((1,), torch.float64)]


def _span(flat, t):
    start = t.data_ptr() - flat.data_ptr()
    return start, start + t.numel() * t.element_size()


def test_views_aligned_disjoint_and_zeroed():
    flat, views = _packed(SPECS, "cpu")
    assert flat.dtype == torch.uint8 and int(flat.abs().sum()) == 0
    spans = []
    for (shape, dtype), v in zip(SPECS, views):
        assert tuple(v.shape) == shape and v.dtype == dtype and v.is_contiguous()
        lo, hi = _span(flat, v)
        assert lo % 256 == 0 and 0 <= lo < hi <= flat.numel()
        spans.append((lo, hi))
    spans.sort()
    for (_, a_hi), (b_lo, _) in zip(spans, spans[1:]):
        assert a_hi <= b_lo


def test_one_flat_copy_moves_every_tensor():
    src_flat, src = _packed(SPECS, "cpu")
    g = torch.Generator().manual_seed(7)
    for v in src:
        if v.dtype.is_floating_point:
            v.copy_(torch.randn(v.shape, generator=g).to(v.dtype))
        else:
            v.copy_(torch.randint(-1000, 1000, v.shape, generator=g).to(v.dtype))
    dst_flat, dst = _packed(SPECS, "cpu")
    dst_flat.copy_(src_flat)
    for a, b in zip(src, dst):
        assert torch.equal(a, b)
