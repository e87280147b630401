"""Guard bands around output buffers, standing in for a memory checker.

A kernel that writes past either end of an output (a masked tail store that
is off by one, a strided dw store with a wrong bound, a reduction that runs a
row too far) would go unseen when the bytes it hits belong to nothing the test
reads. Each guarded buffer sits inside a larger allocation: GUARD_BYTES before
and after it are filled with a fixed byte pattern, and `check()` asserts that
those bytes are unchanged after the call. The interior starts filled with
0xFF bytes (a NaN in fp32, fp16 and bf16), so an element the kernel never
writes also fails the parity comparison's finiteness check.
"""

from __future__ import annotations

import torch

GUARD_BYTES = 4096
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape` and `dtype` with guard bands on both sides.

    `offset_elems` shifts the interior by that many elements past the guard
    (for misaligned views); the tensor is `self.t`."""

    def __init__(self, shape, dtype, device="cuda", offset_elems: int = 0, fill: int = 0xFF):
        n = 1
        for d in shape:
            n *= int(d)
        self.es = torch.empty((), dtype=dtype).element_size()
        self.lead = GUARD_BYTES + offset_elems * self.es
        self.nbytes = n * self.es
        total = self.lead + self.nbytes + GUARD_BYTES
        total = (total + self.es - 1) // self.es * self.es
        self.raw = torch.full((total,), PATTERN, dtype=torch.uint8, device=device)
        self.raw[self.lead:self.lead + self.nbytes] = fill
        self.t = self.raw[self.lead:self.lead + self.nbytes].view(dtype).view(tuple(shape))
        self.name = ""

    def check(self, name: str = "") -> None:
        head = self.raw[:self.lead]
        tail = self.raw[self.lead + self.nbytes:]
        bad_head = int((head != PATTERN).sum())
        bad_tail = int((tail != PATTERN).sum())
        assert bad_head == 0 and bad_tail == 0, (
            f"{name or self.name}: {bad_head} guard bytes changed before the buffer, {bad_tail} after it")


def guarded(shape, dtype, device="cuda", **kw) -> Guarded:
    return Guarded(shape, dtype, device, **kw)


def workspace(nbytes: int, device="cuda") -> Guarded:
    """A guarded uint8 workspace of exactly the size a workspace query returned
    (its interior filled with the guard pattern too: the kernels must not rely
    on its contents)."""
    return Guarded((max(int(nbytes), 0),), torch.uint8, device, fill=PATTERN)


def check_all(guards: dict) -> None:
    for k, g in guards.items():
        g.check(k)
