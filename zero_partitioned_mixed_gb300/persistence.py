"""ZeRO-3 parameter persistence: small tensors keep a resident 16-bit copy.

"ZeRO Stage 1/2/3" guide, ZeRO-3 config, param_persistence_threshold:
parameter tensors with fewer elements than the threshold stay replicated
instead of being gathered layer by layer.  The flat buffer puts the
partitioned tensors first and the persistent ones after them, each group
in model order, so the persistent tensors are one region [p0, psi).  Only
the 16-bit copies change place: gradients and fp32 master/m/v stay
partitioned, and the region is reduce-scattered and updated like the rest.
Zero3Schedule (schedule.py) keeps the region's N copies resident, skips it
in the forward and backward gathers, and refreshes it with one gather
after each step's update.

Host logic only: this module computes offsets and bucket lists.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Sequence, Tuple


@dataclass(frozen=True)
class PersistentLayout:
    order: Tuple[int, ...]                 # model index of each tensor, in flat-buffer order
    ranges: Dict[str, Tuple[int, int]]     # tensor name -> [a, b) in the flat buffer
    p0: int                                # start of the persistent region
    psi: int                               # real parameter count
    threshold: int

    @property
    def n_persistent(self) -> int:
        return sum(1 for a, b in self.ranges.values() if a >= self.p0 and b > a)

    @property
    def psi_persistent(self) -> int:
        return self.psi - self.p0

    def persistent_from(self, psi_pad: int) -> int:
        """Start of the resident region in a buffer padded to psi_pad: p0, or
        psi_pad when no tensor is persistent (the padding is then partitioned
        with the last tensor)."""
        return self.p0 if self.p0 < self.psi else psi_pad


def persistent_layout(shapes: Sequence[Tuple[str, Sequence[int]]], threshold: int) -> PersistentLayout:
    """Flat layout of a named tensor list under a persistence threshold.

    A tensor is persistent when its element count is strictly below the
    threshold (threshold 0: none is).
    """
    sizes = []
    for _, shp in shapes:
        k = 1
        for d in shp:
            k *= int(d)
        sizes.append(k)
    small = [k < threshold for k in sizes]
    order = [i for i in range(len(sizes)) if not small[i]] + [i for i in range(len(sizes)) if small[i]]
    ranges = {}
    pos, p0 = 0, None
    for i in order:
        if small[i] and p0 is None:
            p0 = pos
        ranges[shapes[i][0]] = (pos, pos + sizes[i])
        pos += sizes[i]
    return PersistentLayout(tuple(order), ranges, pos if p0 is None else p0, pos, threshold)


def tensor_buckets(layout: PersistentLayout, psi_pad: int) -> List[Tuple[int, int]]:
    """One bucket per partitioned tensor, then the persistent region as one
    bucket; the padding [psi, psi_pad) joins the last bucket.  The buckets
    tile [0, psi_pad) and have a boundary at p0."""
    out = sorted(r for r in layout.ranges.values() if r[1] <= layout.p0 and r[1] > r[0])
    if layout.p0 < layout.psi:
        out.append((layout.p0, layout.psi))
    if not out:
        return [(0, psi_pad)] if psi_pad else []
    a, _ = out[-1]
    out[-1] = (a, psi_pad)
    return out
