"""Helpers that run the CUDA path and the oracle on the same seeded inputs
and compare them element by element (used by the gpu-marked tests)."""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

import oracle as O
from zero_partitioned_mixed_gb300 import _binding as B
from zero_partitioned_mixed_gb300 import synth as S
from zero_partitioned_mixed_gb300.buffers import RankBuffers

# tolerances stated for this path: fp32 master/m/v within 2 ulp, 16-bit
# parameters within 1 ulp, global norm within 1e-5 relative; integers exact.
ULP32 = 2
ULP16 = 1
NORM_RTOL = 1e-5


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits32(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int32).cpu().numpy().view(np.uint32)


def _ordered(bits: np.ndarray, sign: int) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & (sign - 1)
    return np.where(b & sign, -mag, mag)


def ulp32(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(_ordered(a_bits, 1 << 31) - _ordered(b_bits, 1 << 31))


def ulp16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(_ordered(a_bits, 1 << 15) - _ordered(b_bits, 1 << 15))


@dataclass
class Stats:
    max_ulp32: int = 0
    max_ulp16: int = 0
    mismatches: int = 0     # elements not bit-identical
    compared: int = 0
    norm_rel: float = 0.0
    steps: int = 0

    def add32(self, a, b):
        d = ulp32(a, b)
        if d.size:
            self.max_ulp32 = max(self.max_ulp32, int(d.max()))
        self.mismatches += int(np.count_nonzero(d))
        self.compared += d.size

    def add16(self, a, b):
        d = ulp16(a, b)
        if d.size:
            self.max_ulp16 = max(self.max_ulp16, int(d.max()))
        self.mismatches += int(np.count_nonzero(d))
        self.compared += d.size

    def check(self):
        assert self.max_ulp32 <= ULP32, f"fp32 state off by {self.max_ulp32} ulp"
        assert self.max_ulp16 <= ULP16, f"16-bit params off by {self.max_ulp16} ulp"
        assert self.norm_rel <= NORM_RTOL, f"norm rel err {self.norm_rel}"


def hyper_pair(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, max_norm=0.0, mode=0):
    return (B.hyper(lr, beta1, beta2, eps, weight_decay, max_norm, mode),
            O.Hyper(lr, beta1, beta2, eps, weight_decay, max_norm))


def _draw(shape, sigma, seed, dtype=torch.float32, absolute=False):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device="cuda", dtype=torch.float32) * sigma
    if absolute:
        x = x.abs()
    return x.to(dtype)


def run_case(psi: int, n: int, stage: int, dtype: str = "bf16", steps: int = 2, align: int = 8,
             mode: int = 0, double_buffer: bool = True, loss_scale: float = 1.0, hyper_kw=None,
             buckets: Optional[Sequence[Tuple[int, int]]] = None, inject=None, sigma: float = 1e-2,
             seed: int = 0, warm: bool = True, hyper_steps=None, fused: bool = False) -> Stats:
    """Run `steps` steps on the GPU and in the oracle; compare after each step.

    inject: list of (step, rank, index, value) written into the gradients.
    hyper_steps: per step, hyper-parameter overrides on top of hyper_kw (a
    schedule: learning rate, weight decay, ... changing between steps).
    fused: stage 3, backward through zero_reduce_scatter_gather_bucket (each
    bucket's reduce-scatter carries the next bucket's gather).
    """
    hyper_kw = dict(hyper_kw or {})
    hb, ho = hyper_pair(mode=mode, **hyper_kw)
    buf = RankBuffers(psi, n, stage, dtype, align=align, double_buffer=double_buffer)
    part = O.partition(psi, n, align)
    assert (buf.psi_pad, buf.shard) == (part.psi_pad, part.shard)
    assert list(buf.offsets) == list(part.offsets) and list(buf.real) == list(part.real)
    P = part.psi_pad
    td = S.torch_dtype(dtype)
    st = Stats()
    # initial state: master N(0, 0.02^2); warm m/v or zeros; replicas = RNE(master)
    master0 = _draw((psi,), 0.02, seed * 7 + 1)
    m0 = _draw((psi,), 1e-4, seed * 7 + 2) if warm else torch.zeros(psi, device="cuda")
    v0 = _draw((psi,), 1e-6, seed * 7 + 3, absolute=True) if warm else torch.zeros(psi, device="cuda")
    ost = O.init_state(stage, dtype, part, master0.cpu().numpy(), m0.cpu().numpy(), v0.cpu().numpy(),
                       loss_scale=loss_scale)
    # load the oracle's initial placement into the device buffers
    if stage == 0:
        mv, mm, vv = buf.state()
        mv.copy_(torch.from_numpy(ost.master)); mm.copy_(torch.from_numpy(ost.m)); vv.copy_(torch.from_numpy(ost.v))
        buf.params[:, :P].copy_(torch.from_numpy(ost.params.view(np.int16)).view(td))
    else:
        mv, mm, vv = buf.state(0)
        mv.copy_(torch.from_numpy(ost.master)); mm.copy_(torch.from_numpy(ost.m)); vv.copy_(torch.from_numpy(ost.v))
        if stage == 3:
            buf.params[:P].copy_(torch.from_numpy(ost.params.view(np.int16)).view(td))
        else:
            buf.params[:, :P].copy_(torch.from_numpy(ost.params.view(np.int16)).view(td))
    buf.set_scaler(loss_scale, 0, 0)
    if stage == 3 and buckets is None:
        buckets = [(0, P)]
    for k in range(steps):
        if hyper_steps is not None:
            hb, ho = hyper_pair(mode=mode, **{**hyper_kw, **hyper_steps[k]})
        scale_now = ost.loss_scale
        # gradients for this step (already multiplied by the current scale)
        grads = torch.zeros((n, buf.stride), dtype=td, device="cuda")
        if psi:
            g = _draw((n, psi), sigma * scale_now, seed * 1000 + 17 * k + 5)
            grads[:, :psi] = g.to(td)
        for (ks, r, i, val) in (inject or []):
            if ks == k:
                grads[r, i] = val
        gbits = bits16(grads)
        res_gather_fwd, res_gather_bwd = [], []
        if stage == 3:
            for (a, b) in buckets:
                L = b - a
                outs = [torch.zeros((max(8, (L + 7) // 8 * 8),), dtype=td, device="cuda") for _ in range(n)]
                buf.gather(a, b, outs)
                res_gather_fwd.append([bits16(o[:L]) for o in outs])
            order = list(range(len(buckets) - 1, -1, -1))

            def new_outs(i):
                L = buckets[i][1] - buckets[i][0]
                return [torch.zeros((max(8, (L + 7) // 8 * 8),), dtype=td, device="cuda") for _ in range(n)]

            bwd = {}
            if fused and order:
                bwd[order[0]] = new_outs(order[0])
                buf.gather(buckets[order[0]][0], buckets[order[0]][1], bwd[order[0]])
            for k, idx in enumerate(order):
                a, b = buckets[idx]
                L = b - a
                if not fused:
                    bwd[idx] = new_outs(idx)
                    buf.gather(a, b, bwd[idx])
                gb = [torch.zeros((max(8, (L + 7) // 8 * 8),), dtype=td, device="cuda") for _ in range(n)]
                for r in range(n):
                    gb[r][:L].copy_(grads[r, a:b])
                if fused and k + 1 < len(order):
                    nxt = order[k + 1]
                    bwd[nxt] = new_outs(nxt)
                    buf.reduce_scatter_gather(a, b, gb, hb, buckets[nxt][0], buckets[nxt][1], bwd[nxt])
                else:
                    buf.reduce_scatter(a, b, gb, hb)
            for idx in range(len(buckets)):
                L = buckets[idx][1] - buckets[idx][0]
                res_gather_bwd.append([bits16(o[:L]) for o in bwd[idx]])
            buf.step(hb)
            ost, ores = O.step_stage3(ost, [gbits[:, a:b] for (a, b) in buckets], buckets, ho)
            for bi in range(len(buckets)):
                for r in range(n):
                    assert np.array_equal(res_gather_fwd[bi][r], ores.gathered_fwd[bi][r])
                    assert np.array_equal(res_gather_bwd[bi][r], ores.gathered_bwd[bi][r])
        elif stage == 2 and buckets is not None:
            # ZeRO-2 reduced during backward: buckets in reverse order, each
            # copied into one constant-size buffer per rank that is reused
            lmax = max(b - a for a, b in buckets)
            cb = torch.zeros((n, max(8, (lmax + 7) // 8 * 8)), dtype=td, device="cuda")
            for (a, b) in reversed(buckets):
                cb[:, :b - a].copy_(grads[:, a:b])
                buf.reduce_scatter(a, b, [cb[r] for r in range(n)], hb)
            buf.finish_bucketed_step(hb)
            ost, ores = O.step(ost, gbits, ho)
        else:
            buf.step(hb, buf_grads_rows(grads, n))
            ost, ores = O.step(ost, gbits, ho)
        torch.cuda.synchronize()
        s = buf.status()
        assert bool(s["overflow"]) == ores.overflow, (k, s, ores)
        assert bool(s["applied"]) == ores.applied
        assert s["steps_applied"] == ost.t
        assert s["loss_scale"] == np.float32(ost.loss_scale)
        if ores.applied:
            rel = abs(s["grad_norm"] - ores.norm) / max(ores.norm, 1e-300)
            st.norm_rel = max(st.norm_rel, rel)
            want_clip = float(ores.clip) if ores.clip is not None else 1.0
            assert s["clip_coef"] == want_clip, (s["clip_coef"], want_clip)
        slot = s["state_slot"]
        gm, gmm, gv = buf.state(slot)
        st.add32(bits32(gm), ost.master.view(np.uint32))
        st.add32(bits32(gmm), ost.m.view(np.uint32))
        st.add32(bits32(gv), ost.v.view(np.uint32))
        if stage == 3:
            st.add16(bits16(buf.params[:P]), ost.params)
        else:
            st.add16(bits16(buf.params[:, :P]), ost.params)
        st.steps += 1
    buf.close()
    return st


def buf_grads_rows(grads: torch.Tensor, n: int):
    return [grads[r] for r in range(n)]
