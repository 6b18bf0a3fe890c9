"""The write-guard helper catches writes outside a view (on CPU tensors):
one element past either end of a guarded buffer must be reported, writes
inside it must not."""
import pytest
import torch

from tests._guard import PAD, Guards


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.uint8, torch.int32])
def test_guard_reports_a_write_past_either_end(dtype):
    for side in (-1, 1):
        g = Guards("cpu")
        v = g.new((3, 5), dtype)
        v.fill_(1)                              # every element of the view: allowed
        g.check("inside")
        raw = g.bufs[0][0]
        n = g.bufs[0][1]
        esz = torch.empty((), dtype=dtype).element_size()
        at = PAD - esz if side < 0 else PAD + n  # the element just outside the view
        raw[at:at + esz] = 0
        with pytest.raises(AssertionError):
            g.check("outside")


def test_guard_view_is_aligned_and_contiguous():
    g = Guards("cpu")
    v = g.new((7, 9), torch.float32)
    assert v.is_contiguous() and v.shape == (7, 9)
    assert (v.data_ptr() - g.bufs[0][0].data_ptr()) == PAD and PAD % 256 == 0
