"""Buffers with guard regions, for out-of-bounds write checks without a
sanitizer: each tensor is a view into a larger byte allocation whose 4 KiB
head and tail hold a fixed pattern; after the kernels ran, both must be
unchanged.  The payload starts 4096 bytes into the allocation, so it keeps
the allocation's alignment (TMA and vector stores need 16 bytes, the
workspaces 256)."""
from __future__ import annotations

import math

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    def __init__(self):
        self._allocs = []

    def empty(self, shape, dtype, device):
        """A tensor of `shape` and `dtype` between two guard regions."""
        import torch
        nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        body = (nbytes + GUARD - 1) // GUARD * GUARD
        raw = torch.full((GUARD + body + GUARD,), PATTERN, dtype=torch.uint8, device=device)
        self._allocs.append((raw, nbytes))
        return raw[GUARD:GUARD + nbytes].view(dtype).view(shape)

    def empty_like(self, t):
        return self.empty(tuple(t.shape), t.dtype, t.device)

    def bytes(self, n, device):
        """A workspace of n bytes (uint8) between guard regions."""
        import torch
        return self.empty((max(int(n), 1),), torch.uint8, device)

    def damaged(self):
        """Indices of allocations whose head or tail guard changed (including the slack between the
        payload and the tail guard, which no kernel may touch either)."""
        bad = []
        for i, (raw, nbytes) in enumerate(self._allocs):
            head = raw[:GUARD]
            tail = raw[GUARD + nbytes:]
            if not bool((head == PATTERN).all()) or not bool((tail == PATTERN).all()):
                bad.append(i)
        return bad
