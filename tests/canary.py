"""Guard regions around output buffers, the test-side half of the sanitizer substitute.

Each guarded output is the middle of a larger device allocation whose head and tail (4 KiB
each) hold a byte pattern.  A kernel that writes past either end of its output changes the
pattern; check() finds it.  (Writes that stay inside the output but miss their place are
caught by the parity checks, and unwritten elements by outputs prefilled with NaN.)
"""
from __future__ import annotations

import math

import torch

GUARD_BYTES = 4096
PATTERN = 0xA5


class Guarded:
    def __init__(self, shape, dtype, device="cuda", fill=None):
        self.shape = tuple(shape)
        itemsize = torch.empty(0, dtype=dtype).element_size()
        self.nbytes = math.prod(self.shape) * itemsize
        body = max(256, -(-self.nbytes // 256) * 256)
        self.raw = torch.full((GUARD_BYTES + body + GUARD_BYTES,), PATTERN, dtype=torch.uint8,
                              device=device)
        self.tensor = self.raw[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(self.shape)
        if fill is not None:
            self.tensor.fill_(fill)

    def check(self, what=""):
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.nbytes:]
        bad_h = int((head != PATTERN).sum())
        bad_t = int((tail != PATTERN).sum())
        assert bad_h == 0 and bad_t == 0, \
            f"{what}: {bad_h} guard bytes before and {bad_t} after the output were overwritten"


def guarded_like(shape, dtype, device="cuda", fill=float("nan")):
    """A guarded output prefilled with `fill` (NaN shows unwritten floating-point elements)."""
    if not dtype.is_floating_point and isinstance(fill, float) and math.isnan(fill):
        fill = -7
    return Guarded(shape, dtype, device, fill)
