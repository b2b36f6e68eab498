"""Oracle evaluation at full size, streamed over every element.

The step is elementwise apart from the global norm and the overflow flag.
A full-size step is therefore checked chunk by chunk: the main thread copies
one chunk of the device buffers to host memory (the N gradient rows, the
fp32 state before and after the step, the 16-bit copies), and a pool of
threads runs the oracle on it (numpy drops the GIL in its array loops).
Every element is compared bit for bit.  Each chunk also returns its sums
of squares per owner shard (left to right, fp64); the global norm adds them
shard by shard in chunk order, then over the shards in rank order -- the
oracle's definition, re-associated at chunk boundaries, which moves it by
far less than the 1e-5 relative tolerance.

A skipped (overflowed) step must leave the state untouched: chunks then
carry digests (BLAKE2b) of the state and 16-bit copies, which are compared
with the digests taken from the same buffers after the last applied step.
"""

from __future__ import annotations

import hashlib
import math
import os
from collections import deque
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

import oracle as O

CHUNK = 1 << 23


def _ordered(bits: np.ndarray, sign: int) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & (sign - 1)
    return np.where(b & sign, -mag, mag)


def _ulp(a: np.ndarray, b: np.ndarray, sign: int) -> np.ndarray:
    return np.abs(_ordered(a, sign) - _ordered(b, sign))


@dataclass
class Tally:
    """What a streamed comparison found, merged over its chunks."""
    compared: int = 0
    mismatches: int = 0
    max_ulp32: int = 0
    max_ulp16: int = 0
    bad: bool = False
    sums: Dict[int, Dict[int, float]] = field(default_factory=dict)   # shard -> {chunk start: sum}
    digests: Dict[Tuple[str, int], bytes] = field(default_factory=dict)

    def merge(self, d: dict) -> None:
        self.compared += d["compared"]
        self.mismatches += d["mismatches"]
        self.max_ulp32 = max(self.max_ulp32, d["max_ulp32"])
        self.max_ulp16 = max(self.max_ulp16, d["max_ulp16"])
        self.bad |= d["bad"]
        for r, v in d["sums"].items():
            self.sums.setdefault(r, {})[d["start"]] = v
        self.digests.update(d["digests"])

    def norm(self, n_ranks: int) -> float:
        total = 0.0
        for r in range(n_ranks):
            s = 0.0
            parts = self.sums.get(r, {})
            for k in sorted(parts):
                s = s + parts[k]
            total = total + s
        return math.sqrt(total)


def _digest(x: np.ndarray) -> bytes:
    return hashlib.blake2b(np.ascontiguousarray(x).view(np.uint8), digest_size=16).digest()


def _check_chunk(start: int, psi: int, shard: int, n: int, dtype: str, gbits: Optional[np.ndarray],
                 old: Optional[Sequence[np.ndarray]], new: Optional[Sequence[np.ndarray]],
                 q: Optional[np.ndarray], loss_scale: float, sc: Optional[O.StepScalars],
                 clip: Optional[np.float32], digest: bool) -> dict:
    """The oracle on elements [start, start + L) of one step.

    gbits (N, L) uint16: the ranks' gradients.  old/new: (master, m, v)
    before and after the step.  q (R, L) uint16: the 16-bit copies after
    the step.  With sc given, new and q are compared with the oracle's
    update of old; with digest, new and q are hashed instead of (or as
    well as) compared.
    """
    out = {"start": start, "compared": 0, "mismatches": 0, "max_ulp32": 0, "max_ulp16": 0,
           "bad": False, "sums": {}, "digests": {}}
    L = None
    ghat = None
    if gbits is not None:
        L = gbits.shape[1]
        real = max(0, min(L, psi - start))
        g = [O.widen16(gbits[r, :real], dtype) for r in range(n)]
        ghat = O.unscale(O.rank_sum(g), n, loss_scale)
        out["bad"] = O.has_overflow(ghat)
        pos = 0
        while pos < real:
            r = (start + pos) // shard
            end = min(real, (r + 1) * shard - start)
            out["sums"][r] = O.sq_sum_sequential(ghat[pos:end])
            pos = end
    if sc is not None:
        real = ghat.size
        gg = ghat if clip is None else ghat * clip
        p2, m2, v2 = O.adam_update(old[0][:real], old[1][:real], old[2][:real], gg, sc)
        L = new[0].size
        for got, val in zip(new, (p2, m2, v2)):
            want = np.zeros(L, np.float32)
            want[:real] = val
            d = _ulp(got.view(np.uint32), want.view(np.uint32), 1 << 31)
            out["max_ulp32"] = max(out["max_ulp32"], int(d.max()) if d.size else 0)
            out["mismatches"] += int(np.count_nonzero(d))
            out["compared"] += d.size
        wp = np.zeros(L, np.float32)
        wp[:real] = p2
        wq = O.rne16(wp, dtype)
        for row in q:
            d = _ulp(row, wq, 1 << 15)
            out["max_ulp16"] = max(out["max_ulp16"], int(d.max()) if d.size else 0)
            out["mismatches"] += int(np.count_nonzero(d))
            out["compared"] += d.size
    if digest:
        for name, x in zip(("master", "m", "v"), new):
            out["digests"][(name, start)] = _digest(x)
        for r, row in enumerate(q):
            out["digests"][(f"q{r}", start)] = _digest(row)
    return out


def _host16(t, lo: int, hi: int) -> np.ndarray:
    """Columns [lo, hi) of a (R, cols) or (cols,) 16-bit device tensor as (R, hi - lo) uint16."""
    import torch
    rows = t.unsqueeze(0) if t.dim() == 1 else t
    host = torch.empty((rows.shape[0], hi - lo), dtype=torch.int16)
    for r in range(rows.shape[0]):
        host[r].copy_(rows[r, lo:hi].view(torch.int16))
    return host.numpy().view(np.uint16)


def _host32(t, lo: int, hi: int) -> np.ndarray:
    return t[lo:hi].cpu().numpy()


class FullCheck:
    """Streams device buffers to host chunk by chunk and runs the oracle on them in threads."""

    def __init__(self, workers: Optional[int] = None, chunk: int = CHUNK):
        self.workers = workers or max(1, min(16, (os.cpu_count() or 2)))
        self.pool = ThreadPoolExecutor(self.workers)
        self.chunk = chunk

    def close(self):
        self.pool.shutdown(wait=True)

    def compare(self, a: int, b: int, *, psi: int, part: O.Partition, dtype: str,
                grads=None, g_base: int = 0, old=None, new=None, q=None, q_base: int = 0,
                loss_scale: float = 1.0, sc: Optional[O.StepScalars] = None,
                clip: Optional[np.float32] = None, digest: bool = False,
                tally: Optional[Tally] = None) -> Tally:
        """Elements [a, b) of one step.

        grads: (N, cols) device tensor of 16-bit rows, flat element i at
        column i - g_base (or None).  old/new: (master, m, v) device fp32
        vectors indexed by flat element.  q: 16-bit device tensor, (R, cols)
        replicas or the (cols,) stage-3 shard, flat element i at column
        i - q_base.  sc: the step's Adam scalars when the step applied.
        """
        tally = tally or Tally()
        pending = deque()
        n = part.n_ranks
        for s in range(a, b, self.chunk):
            e = min(b, s + self.chunk)
            gb = _host16(grads, s - g_base, e - g_base) if grads is not None else None
            o3 = [_host32(x, s, e) for x in old] if old is not None else None
            n3 = [_host32(x, s, e) for x in new] if new is not None else None
            qh = _host16(q, s - q_base, e - q_base) if q is not None else None
            pending.append(self.pool.submit(_check_chunk, s, psi, part.shard, n, dtype, gb, o3, n3, qh,
                                            loss_scale, sc, clip, digest))
            while len(pending) >= 2 * self.workers:
                tally.merge(pending.popleft().result())
        while pending:
            tally.merge(pending.popleft().result())
        return tally
