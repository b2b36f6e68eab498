"""ZeRO-3 step schedule: gathers prefetched on a side stream, CUDA-graph capture.

ZeRO summary Sec. 5 (P_os+g+p): the parameter all-gather is spread across
forward propagation, each layer's parameters fetched just before use and
discarded after; backward fetches them again in reverse order and
reduce-scatters each layer's gradients as they appear; a layer may be
prefetched while the previous one computes.  The "ZeRO Stage 1/2/3" guide
names the corresponding knob (prefetch_bucket_size).

Here the gather of bucket b+1 (forward) or b-1 (backward) is issued on a
side stream one bucket ahead, into the other of two output buffer sets,
while the main stream runs the caller's work on bucket b (its forward or
backward compute, then the reduce-scatter).  Events order every reuse of a
buffer set.  All launches go through the C ABI; nothing here computes.

With a persistence boundary p0 (param_persistence_threshold; layout in
persistence.py) the region [p0, psi_pad) keeps N resident 16-bit copies:
its buckets are not gathered in forward or backward, their gradients are
reduce-scattered after the backward pass (a persistent tensor's gradient
is complete only then), and one gather after the update refreshes the
copies.

With fuse=True (the default) the backward pass issues no separate gathers
after its first: each bucket's reduce-scatter carries the gather of the next
bucket in the same launch (zero_reduce_scatter_gather_bucket), whose CTAs
start the gather as they finish their share of the reduce-scatter.  The two
output sets alternate; one stream orders everything.  The forward pass is
as above.  Measured at psi = 2^29 with 5e7-element buckets: 3.66 against
3.89 ms per step at N = 2, 6.41 against 6.57 ms at N = 8.

A step whose buffers and hyper-parameters stay fixed can be captured once
into a CUDA graph and replayed: the library's calls never synchronise or
allocate after the first (warm-up) step, and its step count, loss scale
and state slot live on the device, so each replay is the next step.
"""

from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch

from . import _binding as B
from .buffers import RankBuffers


class Zero3Schedule:
    """One ZeRO-3 step over fixed buckets with one-ahead gather prefetch.

    buf: a stage-3 RankBuffers; buckets: [(a, b)] tiling [0, psi_pad).
    grad_rows(i) -> list of N device tensors holding rank r's gradient of
    bucket i (the caller's backward writes them), or their pointer_array; forward(i, rows) and
    backward(i, rows) are the caller's per-bucket work on the gathered
    16-bit parameters (default: none).
    """

    def __init__(self, buf: RankBuffers, buckets: Sequence[Tuple[int, int]], prefetch: bool = True,
                 persistent_from: Optional[int] = None, fuse: bool = True):
        if buf.stage != 3:
            raise ValueError("Zero3Schedule needs a stage-3 RankBuffers")
        self.buf = buf
        self.buckets = list(buckets)
        self.prefetch = prefetch
        self.fuse = fuse
        P = buf.psi_pad
        self.p0 = P if persistent_from is None else int(persistent_from)
        if not 0 <= self.p0 <= P:
            raise ValueError("persistent_from must lie in [0, psi_pad]")
        for a, b in self.buckets:
            if a < self.p0 < b:
                raise ValueError("a bucket straddles the persistence boundary")
        # the handle's accounting counts the resident region's memory and traffic
        B.zero_set_persistent(buf.h, self.p0)
        self.gathered = [i for i, (a, b) in enumerate(self.buckets) if b <= self.p0 and a < self.p0]
        gset = set(self.gathered)
        self.kept = [i for i in range(len(self.buckets)) if i not in gset]
        self.resident: Optional[torch.Tensor] = None
        self._fresh = False
        if self.p0 < P:
            lp = max(8, (P - self.p0 + 7) // 8 * 8)
            self.resident = torch.empty((buf.n, lp), dtype=buf.params.dtype, device=buf.params.device)
            self._resident_ptrs = B.pointer_array([self.resident[r] for r in range(buf.n)])
        sizes = [self.buckets[i][1] - self.buckets[i][0] for i in self.gathered]
        lmax = max(sizes) if sizes else 0
        lpad = max(8, (lmax + 7) // 8 * 8)
        td = buf.params.dtype
        nsets = 2 if (prefetch or fuse) else 1
        self.outs = [torch.empty((buf.n, lpad), dtype=td, device=buf.params.device) for _ in range(nsets)]
        # the library calls take the rows' pointer arrays, built once
        self._out_ptrs = [B.pointer_array([o[r] for r in range(buf.n)]) for o in self.outs]
        self.side = torch.cuda.Stream(device=buf.params.device) if prefetch else None
        self.graph: Optional[torch.cuda.CUDAGraph] = None

    def _rows(self, k: int) -> List[torch.Tensor]:
        o = self.outs[k % len(self.outs)]
        return [o[r] for r in range(self.buf.n)]

    def _pass(self, order: Sequence[int], work: Optional[Callable], rs: Optional[Callable]) -> None:
        main = torch.cuda.current_stream()
        buf = self.buf
        order = list(order)
        if not self.prefetch:
            for i in order:
                a, b = self.buckets[i]
                buf.gather(a, b, self._out_ptrs[0], main)
                if work is not None:
                    work(i, self._rows(0))
                if rs is not None:
                    rs(i)
            return
        n = len(order)
        ready = [torch.cuda.Event() for _ in range(n)]       # gather k done (side stream)
        free = [torch.cuda.Event() for _ in range(2)]        # output set released (main stream)
        for e in free:
            e.record(main)

        def issue(k):
            a, b = self.buckets[order[k]]
            self.side.wait_event(free[k % 2])
            with torch.cuda.stream(self.side):
                buf.gather(a, b, self._out_ptrs[k % len(self.outs)], self.side)
                ready[k].record(self.side)

        if n:
            issue(0)
        for k in range(n):
            if k + 1 < n:
                issue(k + 1)                                   # prefetch the next bucket
            main.wait_event(ready[k])
            if work is not None:
                work(order[k], self._rows(k))
            if rs is not None:
                rs(order[k])
            free[k % 2].record(main)
        # every gather was joined into the main stream through ready[k]

    def _backward_fused(self, order: Sequence[int], work: Optional[Callable], hyp, grad_rows) -> None:
        """Backward over `order`: bucket k's reduce-scatter and bucket k+1's
        gather in one call, into output sets that alternate."""
        main = torch.cuda.current_stream()
        buf = self.buf
        order = list(order)
        if not order:
            return
        a, b = self.buckets[order[0]]
        buf.gather(a, b, self._out_ptrs[0], main)
        for k, i in enumerate(order):
            if work is not None:
                work(i, self._rows(k))
            a, b = self.buckets[i]
            if k + 1 < len(order):
                ga, gb = self.buckets[order[k + 1]]
                buf.reduce_scatter_gather(a, b, grad_rows(i), hyp, ga, gb, self._out_ptrs[(k + 1) % 2], main)
            else:
                buf.reduce_scatter(a, b, grad_rows(i), hyp, main)

    def resident_rows(self) -> List[torch.Tensor]:
        """The N resident copies of [p0, psi_pad) (rank r's is row r)."""
        if self.resident is None:
            return []
        return [self.resident[r] for r in range(self.buf.n)]

    def refresh(self) -> None:
        """Gather [p0, psi_pad) from the owners' shards into the resident copies."""
        if self.resident is not None:
            self.buf.gather(self.p0, self.buf.psi_pad, self._resident_ptrs, torch.cuda.current_stream())
            self._fresh = True

    def step(self, hyp, grad_rows: Callable[[int], List[torch.Tensor]],
             forward: Optional[Callable] = None, backward: Optional[Callable] = None) -> None:
        """Forward gathers, backward gathers + reduce-scatters, the persistent
        buckets' reduce-scatters, zero_step, then the resident refresh."""
        buf = self.buf
        if self.resident is not None and not self._fresh:
            self.refresh()
        self._pass(self.gathered, forward, None)

        def rs(i):
            a, b = self.buckets[i]
            buf.reduce_scatter(a, b, grad_rows(i), hyp)

        if self.fuse:
            self._backward_fused(self.gathered[::-1], backward, hyp, grad_rows)
        else:
            self._pass(self.gathered[::-1], backward, rs)
        for i in self.kept:
            rs(i)
        buf.step(hyp)
        self.refresh()

    def capture(self, hyp, grad_rows, forward=None, backward=None) -> torch.cuda.CUDAGraph:
        """Capture one step into a CUDA graph (call after one eager warm-up step)."""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.step(hyp, grad_rows, forward, backward)
        torch.cuda.current_stream().wait_stream(s)
        self.graph = g
        return g
