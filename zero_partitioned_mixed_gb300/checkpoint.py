"""Checkpoint and resume of the partitioned model state.

Saved: the live slot of the fp32 master/m/v (the N owner shards back to
back, or the N replicas at stage 0), the 16-bit parameters, and the
device-side scaler state (loss scale, applied-step count t).  Resuming
copies them into slot 0 of fresh buffers and sets the scaler, so the next
step computes exactly what it would have without the interruption.

What is reproduced is the arithmetic state: master, m, v, the 16-bit
parameters, the loss scale and t, and with them every later step, bit for
bit.  The count of skipped (overflowed) steps is a statistic outside that
state; setting the scaler restarts it at 0, so after a resume it counts the
skips since the resume only.
"""

from __future__ import annotations

import torch

from .buffers import RankBuffers


def save(buf: RankBuffers, path: str) -> None:
    st = buf.status()
    master, m, v = buf.state(st["state_slot"])
    torch.save({
        "meta": {"psi": buf.psi, "n_ranks": buf.n, "stage": buf.stage, "dtype": buf.dtype,
                 "psi_pad": buf.psi_pad},
        "master": master.detach().cpu().clone(), "m": m.detach().cpu().clone(), "v": v.detach().cpu().clone(),
        "params": buf.params.detach().cpu().clone(),
        "loss_scale": float(st["loss_scale"]), "steps_applied": int(st["steps_applied"]),
    }, path)


def load(path: str, buf: RankBuffers) -> None:
    ck = torch.load(path, map_location="cpu")
    meta = ck["meta"]
    if (meta["psi"], meta["n_ranks"], meta["stage"], meta["dtype"], meta["psi_pad"]) != (
            buf.psi, buf.n, buf.stage, buf.dtype, buf.psi_pad):
        raise ValueError(f"checkpoint is for {meta}, buffers are psi={buf.psi} N={buf.n} stage={buf.stage}")
    master, m, v = buf.state(0)
    master.copy_(ck["master"])
    m.copy_(ck["m"])
    v.copy_(ck["v"])
    buf.params.copy_(ck["params"])
    buf.set_scaler(ck["loss_scale"], ck["steps_applied"], 0)
