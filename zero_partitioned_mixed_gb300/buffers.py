"""Device buffers for the N simulated ranks, allocated with PyTorch.

Layout in HBM (all 16-byte aligned):
  * grads  [N, stride] 16-bit: rank r's gradient is row r (stages 0-2);
  * params [N, stride] 16-bit replicas (stages 0-2) or [stride] 16-bit
    concatenation of the owner shards (stage 3);
  * master, m, v: fp32, ``slots * psi_pad`` floats with the N owner shards
    back to back in each slot (stages 1-3), or ``N * psi_pad`` (stage 0,
    one full replica per rank).
stride is psi_pad rounded up to 8 elements so every row starts on 16 bytes.
"""

from __future__ import annotations

from typing import List, Optional

import torch

from . import _binding as B
from .synth import torch_dtype

_ZDT = {"fp16": B.ZERO_FP16, "bf16": B.ZERO_BF16}


def _round8(x: int) -> int:
    return (x + 7) // 8 * 8


class RankBuffers:
    """A handle plus the caller-owned buffers of one partitioned flat model.

    grads and params are written in place (the handle keeps their row
    pointers); rebinding the attributes to other tensors is not supported.
    """

    def __init__(self, psi: int, n_ranks: int, stage: int, dtype: str = "bf16", align: int = 8,
                 double_buffer: Optional[bool] = True, device="cuda", alloc_grads: bool = True):
        if stage == 0:
            double_buffer = False
        if double_buffer is None:
            double_buffer = self.second_slot_fits(psi, n_ranks, stage, align, alloc_grads, device)
        self.psi, self.n, self.stage, self.dtype = psi, n_ranks, stage, dtype
        self.double_buffer = double_buffer
        self.h = B.zero_init_partition(psi, n_ranks, stage, _ZDT[dtype], align,
                                       B.ZERO_F_DOUBLE_BUFFER if double_buffer else 0)
        self.psi_pad, self.shard, self.offsets, self.real = B.zero_partition_info(self.h)
        td = torch_dtype(dtype)
        self.stride = max(8, _round8(self.psi_pad))
        self.grads = (torch.zeros((n_ranks, self.stride), dtype=td, device=device)
                      if (alloc_grads and stage != 3) else None)
        if stage == 3:
            self.params = torch.zeros((self.stride,), dtype=td, device=device)
        else:
            self.params = torch.zeros((n_ranks, self.stride), dtype=td, device=device)
        slots = 2 if double_buffer else 1
        rows = n_ranks if stage == 0 else slots
        size = max(4, rows * self.psi_pad)
        self.master = torch.zeros(size, dtype=torch.float32, device=device)
        self.m = torch.zeros(size, dtype=torch.float32, device=device)
        self.v = torch.zeros(size, dtype=torch.float32, device=device)
        # the rows never move: their pointer arrays are built once (at N = 32
        # building them costs more host time than the step's GPU time)
        self._grad_ptrs = B._ptr_array(self.grad_rows()) if self.grads is not None else None
        self._param_ptrs = B._ptr_array(self.param_rows())

    @staticmethod
    def second_slot_fits(psi: int, n_ranks: int, stage: int, align: int = 8, alloc_grads: bool = True,
                         device="cuda", margin: float = 0.05) -> bool:
        """Whether the speculative mode's second master/m/v slot fits in the
        device's free memory next to everything else these buffers hold
        (with a 5 % margin); when it does not, single-buffered state makes
        the library's AUTO mode take the two-pass step instead."""
        unit = n_ranks * align
        pp = (psi + unit - 1) // unit * unit
        stride = max(8, _round8(pp))
        sixteen = 2 * stride * ((n_ranks if alloc_grads and stage != 3 else 0) + (1 if stage == 3 else n_ranks))
        state_one = 3 * 4 * pp
        free, _ = torch.cuda.mem_get_info(torch.device(device))
        return sixteen + 2 * state_one <= free * (1.0 - margin)

    # -- views
    def grad_rows(self) -> List[torch.Tensor]:
        return [self.grads[r] for r in range(self.n)]

    def param_rows(self) -> List[torch.Tensor]:
        if self.stage == 3:
            return [self.params]
        return [self.params[r] for r in range(self.n)]

    def state(self, slot: int = 0):
        """(master, m, v) views of one slot (stages 1-3) or all N replicas (stage 0)."""
        P = self.psi_pad
        if self.stage == 0:
            return (self.master[: self.n * P].view(self.n, P), self.m[: self.n * P].view(self.n, P),
                    self.v[: self.n * P].view(self.n, P))
        return (self.master[slot * P:(slot + 1) * P], self.m[slot * P:(slot + 1) * P],
                self.v[slot * P:(slot + 1) * P])

    # -- calls
    def set_scaler(self, loss_scale: float, steps_applied: int = 0, slot: int = 0, stream=None):
        B.zero_set_scaler(self.h, loss_scale, steps_applied, slot, stream)

    def step(self, hyp, grads: Optional[List] = None, stream=None):
        if self.stage == 3:
            B.zero_step(self.h, None, self._param_ptrs, self.master, self.m, self.v, hyp, stream)
        else:
            B.zero_step(self.h, grads if grads is not None else self._grad_ptrs, self._param_ptrs,
                        self.master, self.m, self.v, hyp, stream)

    def gather(self, a: int, b: int, out: List, stream=None):
        B.zero_gather_bucket(self.h, a, b, self.params, out, stream)

    def reduce_scatter(self, a: int, b: int, grads: List, hyp, stream=None):
        """Reduce-scatter of one bucket: stage 3, or stage 2 reduced during backward."""
        if self.stage == 2:
            B.zero_reduce_scatter_bucket_replicas(self.h, a, b, grads, self.master, self.m, self.v,
                                                  self._param_ptrs, hyp, stream)
        else:
            B.zero_reduce_scatter_bucket(self.h, a, b, grads, self.master, self.m, self.v, self.params, hyp,
                                         stream)

    def reduce_scatter_gather(self, a: int, b: int, grads: List, hyp, ga: int, gb: int, out: List, stream=None):
        """Stage 3: reduce-scatter of bucket [a, b) and gather of [ga, gb) into out, in one call."""
        B.zero_reduce_scatter_gather_bucket(self.h, a, b, grads, self.master, self.m, self.v, self.params, hyp,
                                            ga, gb, out, stream)

    def finish_bucketed_step(self, hyp, stream=None):
        """zero_step after the step's buckets were reduce-scattered (stages 2 and 3)."""
        B.zero_step(self.h, None, self._param_ptrs, self.master, self.m, self.v, hyp, stream)

    def status(self, stream=None) -> dict:
        return B.zero_get_status(self.h, stream)

    def bytes_moved(self) -> dict:
        return B.zero_bytes_moved(self.h)

    def close(self):
        if self.h:
            B.zero_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
