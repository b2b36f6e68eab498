"""Oracle evaluation at full size, streamed over every element.

The step is elementwise apart from the global norm and the overflow flag.
A full-size step is therefore checked chunk by chunk: the main thread copies
one chunk of the device buffers to pinned host memory (the N gradient rows,
the fp32 state before and after the step, the 16-bit copies), and a pool of
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


class FullCheck:
    """Streams device buffers to host chunk by chunk and runs the oracle on them in threads.

    The chunks land in a ring of pinned host slots (async copies on a side
    stream, one event per chunk that its worker waits on); a slot is reused
    once the worker that read it has finished.
    """

    def __init__(self, workers: Optional[int] = None, slot_bytes: int = 1 << 29, max_chunk: int = CHUNK):
        self.workers = workers or max(1, min(16, (os.cpu_count() or 2)))
        self.pool = ThreadPoolExecutor(self.workers)
        self.slot_bytes = slot_bytes
        self.max_chunk = max_chunk
        self.slots = [None] * (2 * self.workers)
        self.stream = None

    def close(self):
        self.pool.shutdown(wait=True)
        self.slots = []

    def _slot(self, i: int):
        import torch
        if self.slots[i] is None:
            self.slots[i] = torch.empty(self.slot_bytes, dtype=torch.uint8, pin_memory=True)
        return self.slots[i]

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
        import torch
        tally = tally or Tally()
        n = part.n_ranks
        qrows = None if q is None else (q.unsqueeze(0) if q.dim() == 1 else q)
        ng = grads.shape[0] if grads is not None else 0
        nq = qrows.shape[0] if qrows is not None else 0
        per_elem = 2 * ng + 4 * 3 * ((old is not None) + (new is not None)) + 2 * nq
        chunk = self.max_chunk
        while chunk > 1024 and chunk * per_elem + 16 * 256 > self.slot_bytes:
            chunk //= 2
        if self.stream is None:
            self.stream = torch.cuda.Stream()
        self.stream.wait_stream(torch.cuda.current_stream())
        pending = deque()
        k = 0
        for s in range(a, b, chunk):
            e = min(b, s + chunk)
            L = e - s
            if len(pending) == len(self.slots):
                tally.merge(pending.popleft().result())
            buf = self._slot(k % len(self.slots))
            k += 1
            off = 0

            def take(nbytes):
                nonlocal off
                v = buf[off:off + nbytes]
                off += (nbytes + 255) // 256 * 256
                return v

            with torch.cuda.stream(self.stream):
                gb = o3 = n3 = qh = None
                if grads is not None:
                    t = take(2 * ng * L).view(torch.int16).view(ng, L)
                    for r in range(ng):
                        t[r].copy_(grads[r, s - g_base:e - g_base].view(torch.int16), non_blocking=True)
                    gb = t.numpy().view(np.uint16)
                if old is not None:
                    o3 = []
                    for x in old:
                        t = take(4 * L).view(torch.float32)
                        t.copy_(x[s:e], non_blocking=True)
                        o3.append(t.numpy())
                if new is not None:
                    n3 = []
                    for x in new:
                        t = take(4 * L).view(torch.float32)
                        t.copy_(x[s:e], non_blocking=True)
                        n3.append(t.numpy())
                if qrows is not None:
                    t = take(2 * nq * L).view(torch.int16).view(nq, L)
                    for r in range(nq):
                        t[r].copy_(qrows[r, s - q_base:e - q_base].view(torch.int16), non_blocking=True)
                    qh = t.numpy().view(np.uint16)
                ev = torch.cuda.Event()
                ev.record(self.stream)

            def job(ev=ev, s=s, gb=gb, o3=o3, n3=n3, qh=qh):
                ev.synchronize()
                return _check_chunk(s, psi, part.shard, n, dtype, gb, o3, n3, qh, loss_scale, sc, clip, digest)

            pending.append(self.pool.submit(job))
        while pending:
            tally.merge(pending.popleft().result())
        return tally
