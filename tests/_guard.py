"""Guarded output buffers for the write-guard tests: a view into a larger
allocation whose bytes before and after it carry a sentinel pattern, and a
check that those bytes are untouched."""
import torch

PAD = 4096        # guard bytes on each side (keeps the view 256-byte aligned)
SENTINEL = 0xA5


class Guards:
    """Allocates guarded output views and checks their guard bands."""

    def __init__(self, device="cuda"):
        self.device = device
        self.bufs = []

    def new(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((PAD + nbytes + PAD,), SENTINEL, dtype=torch.uint8, device=self.device)
        view = raw[PAD:PAD + nbytes].view(dtype).view(*shape) if n else torch.empty(shape, dtype=dtype,
                                                                                     device=self.device)
        self.bufs.append((raw, nbytes))
        return view

    def like(self, t):
        return self.new(tuple(t.shape), t.dtype)

    def check(self, what):
        if self.device != "cpu":
            torch.cuda.synchronize()
        for i, (raw, nbytes) in enumerate(self.bufs):
            head, tail = raw[:PAD], raw[PAD + nbytes:]
            bad = int((head != SENTINEL).sum().item() + (tail != SENTINEL).sum().item())
            assert bad == 0, f"{what}: {bad} guard bytes of output buffer {i} changed"
