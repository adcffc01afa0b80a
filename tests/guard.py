"""Canary guard bands around device buffers (a stand-in for a memory checker).

Every output buffer of a layer under test is replaced by a view (256-byte
aligned) into a larger allocation whose margins (at least MARGIN bytes before
and after) are filled with a sentinel byte.  After the step, the margins
must still hold the sentinel: a kernel that stores past either end of an
output (a TMA store at a wrong coordinate, a ragged tile not clipped, a
token-chunk map off by one) changes them.  The inputs are snapshotted too and must come back unchanged.
"""
from __future__ import annotations

import torch

MARGIN = 64 * 1024   # bytes on each side; a multiple of 256 keeps the view aligned
SENTINEL = 0xA5


class GuardBands:
    def __init__(self):
        self._bufs = []     # (name, raw uint8 allocation, view start, view bytes)
        self._inputs = []   # (name, tensor, snapshot)

    def like(self, x: torch.Tensor, name: str) -> torch.Tensor:
        """A tensor with x's shape, dtype and device (contents: the sentinel
        bytes), inside a guarded allocation."""
        n = x.numel() * x.element_size()
        raw = torch.full((MARGIN + n + MARGIN + 256,), SENTINEL, dtype=torch.uint8,
                         device=x.device)
        start = MARGIN + (-(raw.data_ptr() + MARGIN)) % 256  # the view starts 256-byte aligned
        view = raw[start:start + n].view(x.dtype).view(x.shape)
        self._bufs.append((name, raw, start, n))
        return view

    def guard(self, obj, names) -> None:
        """Replace obj.<name> (a tensor or a list of tensors) by guarded ones."""
        for name in names:
            cur = getattr(obj, name)
            if isinstance(cur, list):
                setattr(obj, name, [self.like(x, f"{name}[{i}]") for i, x in enumerate(cur)])
            else:
                setattr(obj, name, self.like(cur, name))

    def watch_inputs(self, obj, names) -> None:
        for name in names:
            cur = getattr(obj, name)
            for i, x in enumerate(cur if isinstance(cur, list) else [cur]):
                self._inputs.append((f"{name}[{i}]", x, x.clone()))

    def check(self) -> None:
        """Raise AssertionError naming every buffer whose margins changed (and
        every watched input that changed)."""
        bad = []
        for name, raw, start, n in self._bufs:
            head, tail = raw[:start], raw[start + n:]
            for where, band in (("before", head), ("after", tail)):
                hit = torch.nonzero(band != SENTINEL)
                if hit.numel():
                    off = int(hit[0]) if where == "after" else start - int(hit[-1])
                    bad.append(f"{name}: {hit.numel()} byte(s) {where} the buffer changed "
                               f"(nearest {off} byte(s) from its {'end' if where == 'after' else 'start'})")
        for name, x, snap in self._inputs:
            if not torch.equal(x, snap):
                bad.append(f"input {name} was modified")
        assert not bad, "guard bands: " + "; ".join(bad)
