"""Host-side: the packed-buffer layout of conv_bn_silu_gb300.host_io (one
copy each way per step) places every tensor at an aligned offset, without
overlap, and its views read and write the buffer in place."""
import torch

from conv_bn_silu_gb300.host_io import pack_layout, packed_views


def test_pack_layout_aligned_and_disjoint():
    like = [torch.empty(3, 5, dtype=torch.float32), torch.empty(7, dtype=torch.bfloat16),
            torch.empty(0, dtype=torch.float32), torch.empty(64, dtype=torch.int8), torch.empty(2, 2)]
    offsets, total = pack_layout(like, align=256)
    ends = [o + t.numel() * t.element_size() for o, t in zip(offsets, like)]
    assert all(o % 256 == 0 for o in offsets)
    assert all(e <= n for e, n in zip(ends, offsets[1:] + [total]))   # each tensor ends before the next starts
    assert total % 256 == 0 and total == offsets[-1] + 256
    assert offsets == [0, 256, 512, 512, 768]                        # an empty tensor takes no room


def test_packed_views_alias_the_buffer():
    like = [torch.empty(2, 3, dtype=torch.float32), torch.empty(4, dtype=torch.int16)]
    offsets, total = pack_layout(like, align=16)
    buf = torch.zeros(total, dtype=torch.uint8)
    a, b = packed_views(buf, like, offsets)
    assert a.shape == (2, 3) and a.dtype == torch.float32 and b.shape == (4,) and b.dtype == torch.int16
    a.fill_(1.5)
    b.copy_(torch.tensor([1, -2, 3, -4], dtype=torch.int16))
    assert torch.equal(buf[:24].view(torch.float32), torch.full((6,), 1.5))
    assert torch.equal(buf[offsets[1]:offsets[1] + 8].view(torch.int16), torch.tensor([1, -2, 3, -4], dtype=torch.int16))
    assert torch.count_nonzero(buf[24:offsets[1]]) == 0                # the gap stays untouched
