"""Guard margins around the device buffers a test hands to the library.

compute-sanitizer is not available on the GPU pool, so writes past the end
(or before the start) of an output are caught this way instead: each buffer is
the middle of a larger allocation whose 64 KiB margins on both sides hold a
fixed byte pattern, and ``check()`` asserts after the call that no byte of the
margins changed."""
import torch

MARGIN = 64 << 10
PATTERN = 0xA5


class Guarded:
    def __init__(self, shape, dtype, device="cuda", align=256, fill=None):
        numel = 1
        for s in shape:
            numel *= s
        esize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = numel * esize
        self.raw = torch.full((2 * MARGIN + self.nbytes + align,), PATTERN, dtype=torch.uint8,
                              device=device)
        # the view starts MARGIN (+ padding to ``align``) bytes into the buffer
        self.off = MARGIN + (-(self.raw.data_ptr() + MARGIN)) % align
        self.t = self.raw[self.off:self.off + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self, what):
        head = self.raw[:self.off]
        tail = self.raw[self.off + self.nbytes:]
        assert bool((head == PATTERN).all()), f"{what}: bytes before the buffer were written"
        assert bool((tail == PATTERN).all()), f"{what}: bytes after the buffer were written"


def guarded(shape, dtype=torch.float32, **kw):
    return Guarded(shape, dtype, **kw)
