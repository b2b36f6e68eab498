"""Oracle evaluation at full size: sampled elements and a streamed global norm.

The step is elementwise apart from the norm and the overflow flag, so at
full size the oracle computes the expected state of a sample of elements
one by one.  The norm and flag over all elements come from a pool of
oracle threads that each reduce a chunk of the gradients copied from the
device to host memory.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import List, Sequence, Tuple

import numpy as np

import oracle as O

CHUNK = 1 << 24


def _chunk_partials(bits: np.ndarray, start: int, psi: int, dtype: str, loss_scale: float,
                    shard: int) -> Tuple[dict, bool]:
    """Per-owner-shard fp64 sums of squares of g_hat over [start, start + bits.shape[1])."""
    n, length = bits.shape
    real = max(0, min(length, psi - start))
    g = [O.widen16(bits[r, :real], dtype) for r in range(n)]
    ghat = O.unscale(O.rank_sum(g), n, loss_scale)
    bad = O.has_overflow(ghat)
    out = {}
    pos = 0
    while pos < real:
        r = (start + pos) // shard
        end = min(real, (r + 1) * shard - start)
        x = ghat[pos:end].astype(np.float64)
        out[r] = out.get(r, 0.0) + float(np.sum(x * x))
        pos = end
    return out, bad


class NormPool:
    """Threads running the oracle on chunks (numpy drops the GIL in its array loops)."""

    def __init__(self, workers: int = None):
        self.workers = workers or max(1, min(16, (os.cpu_count() or 2)))
        self.pool = ThreadPoolExecutor(self.workers)

    def close(self):
        self.pool.shutdown(wait=True)

    def norm_and_flag(self, rows: Sequence, psi: int, part: O.Partition, dtype: str,
                      loss_scale: float) -> Tuple[float, bool]:
        """Oracle norm and overflow flag of the N device rows (each >= psi long)."""
        import torch
        n = len(rows)
        futures = []
        sums = {}
        bad = False

        def drain(f):
            nonlocal bad
            d, b = f.result()
            bad |= b
            for r, v in d.items():
                sums.setdefault(r, []).append(v)

        for start in range(0, psi, CHUNK):
            length = min(CHUNK, psi - start)
            host = torch.empty((n, length), dtype=torch.int16)
            for r in range(n):
                host[r].copy_(rows[r][start:start + length].view(torch.int16))
            bits = host.numpy().view(np.uint16)
            futures.append(self.pool.submit(_chunk_partials, bits, start, psi, dtype, loss_scale, part.shard))
            if len(futures) >= 2 * self.workers:
                drain(futures.pop(0))
        for f in futures:
            drain(f)
        total = 0.0
        for r in range(part.n_ranks):
            total = total + math.fsum(sums.get(r, []))
        return math.sqrt(total), bad


def sample_indices(psi_pad: int, part: O.Partition, k: int, seed: int, extra=()) -> np.ndarray:
    """k random indices plus both ends, every shard boundary, and `extra`."""
    rng = np.random.default_rng(seed)
    idx = set(int(i) for i in rng.integers(0, psi_pad, k))
    for lo in [0] + list(part.offsets) + [psi_pad]:
        for d in range(-8, 8):
            if 0 <= lo + d < psi_pad:
                idx.add(lo + d)
    for e in extra:
        idx.add(int(e))
    return np.array(sorted(idx), dtype=np.int64)


def gather_bits16(t, idx_t) -> np.ndarray:
    import torch
    return t.index_select(-1, idx_t).contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def gather_f32(t, idx_t) -> np.ndarray:
    return t.index_select(0, idx_t).cpu().numpy()


def oracle_sampled_step(p, m, v, gbits, n, dtype, loss_scale, h: O.Hyper, t_next: int,
                        clip, valid_mask) -> Tuple[np.ndarray, np.ndarray, np.ndarray, bool]:
    """The oracle's step on a sample: returns new (p, m, v) and the sampled overflow flag."""
    keep = valid_mask.astype(bool)
    g = [np.where(keep, O.widen16(gbits[r], dtype), np.float32(0)) for r in range(n)]
    ghat = O.unscale(O.rank_sum(g), n, loss_scale)
    bad = O.has_overflow(ghat[keep])
    if bad:
        return p, m, v, True
    if clip is not None:
        ghat = ghat * clip
    sc = O.step_scalars(h, t_next)
    p2, m2, v2 = O.adam_update(p, m, v, ghat, sc)
    p2 = np.where(keep, p2, np.float32(0)); m2 = np.where(keep, m2, np.float32(0)); v2 = np.where(keep, v2, np.float32(0))
    return p2.astype(np.float32), m2.astype(np.float32), v2.astype(np.float32), False
