"""Seeded synthetic inputs for the ZeRO step (shared by tests, bench and the oracle side).

This module draws random numbers and lays out buffers; it holds none of the
method's arithmetic.  Values come from ``torch`` generators seeded per
(workload, purpose, step, rank), drawn in fixed chunks (the same seed
and device type give the same bits), then rounded to 16 bits by torch's
round-to-nearest-even cast.  The oracle side receives copies of the very
tensors the GPU side consumes.

Workload shapes:
  * toy GPT flat buffer of the "zero-stages-simulation" README (psi = 637,824,
    N = 32);
  * a GPT-2-small parameter list (12 layers, d 768, ffn 3072, vocab 50257,
    ctx 1024, tied head) -- psi = 124,439,808;
  * a flat 1.5B buffer (the GPT-2 1.5B size of the ZeRO paper's Sec. 3.1
    example);
  * a Llama-7B parameter list (32 layers, hidden 4096, ffn 11008, vocab
    32000, untied head) -- psi = 6,738,415,616, one bucket per layer.
"""

from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import torch

CHUNK = 1 << 24   # elements drawn per generator call


def seed_of(*parts) -> int:
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def torch_dtype(dtype: str) -> torch.dtype:
    return {"fp16": torch.float16, "bf16": torch.bfloat16}[dtype]


# ---------------------------------------------------------------- parameter lists
def gpt2_small_shapes() -> List[Tuple[str, Tuple[int, ...]]]:
    d, ffn, vocab, ctx, layers = 768, 3072, 50257, 1024, 12
    out = [("wte", (vocab, d)), ("wpe", (ctx, d))]
    for i in range(layers):
        out += [(f"h{i}.ln_1.w", (d,)), (f"h{i}.ln_1.b", (d,)),
                (f"h{i}.attn.c_attn.w", (3 * d, d)), (f"h{i}.attn.c_attn.b", (3 * d,)),
                (f"h{i}.attn.c_proj.w", (d, d)), (f"h{i}.attn.c_proj.b", (d,)),
                (f"h{i}.ln_2.w", (d,)), (f"h{i}.ln_2.b", (d,)),
                (f"h{i}.mlp.c_fc.w", (ffn, d)), (f"h{i}.mlp.c_fc.b", (ffn,)),
                (f"h{i}.mlp.c_proj.w", (d, ffn)), (f"h{i}.mlp.c_proj.b", (d,))]
    out += [("ln_f.w", (d,)), ("ln_f.b", (d,))]
    return out


def llama7b_shapes() -> List[Tuple[str, Tuple[int, ...]]]:
    d, ffn, vocab, layers = 4096, 11008, 32000, 32
    out = [("embed", (vocab, d))]
    for i in range(layers):
        out += [(f"l{i}.q", (d, d)), (f"l{i}.k", (d, d)), (f"l{i}.v", (d, d)), (f"l{i}.o", (d, d)),
                (f"l{i}.gate", (ffn, d)), (f"l{i}.up", (ffn, d)), (f"l{i}.down", (d, ffn)),
                (f"l{i}.norm_attn", (d,)), (f"l{i}.norm_mlp", (d,))]
    out += [("norm", (d,)), ("lm_head", (vocab, d))]
    return out


def numel(shape: Sequence[int]) -> int:
    return int(math.prod(shape))


def layer_buckets(shapes, psi_pad: int) -> List[Tuple[int, int]]:
    """One bucket per layer of a Llama-style list: [embed], each layer, [norm + head + padding]."""
    bounds = [0]
    pos = 0
    group = None
    for name, shp in shapes:
        g = name.split(".")[0] if name.startswith("l") and name[1].isdigit() else name
        if group is not None and g != group and not (group in ("norm", "lm_head") and g in ("norm", "lm_head")):
            bounds.append(pos)
        group = g
        pos += numel(shp)
    out = list(zip(bounds, bounds[1:] + [psi_pad]))
    return out


def flat_buckets(psi_pad: int, n_ranks: int, size: int) -> List[Tuple[int, int]]:
    """Constant-size buckets rounded down to a multiple of N*8; the last may be partial."""
    size = max(n_ranks * 8, size // (n_ranks * 8) * (n_ranks * 8))
    return [(a, min(a + size, psi_pad)) for a in range(0, psi_pad, size)]


# ---------------------------------------------------------------- workloads
@dataclass(frozen=True)
class Workload:
    name: str
    psi: int
    n_ranks: int
    stage: int
    dtype: str
    steps: int
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    max_norm: float = 0.0
    loss_scale: float = 1.0
    grad_sigma: float = 1e-2
    fan_in_scaled: bool = False
    warm_state: bool = False
    inject_step: int = 0         # 1-based step with one +inf (0 = none)
    inject_rank: int = 0
    shapes: str = ""             # "gpt2" | "llama" | ""


TOY = Workload("toy_gpt_flat_psi637824_n32", 637824, 32, 1, "fp16", 3, grad_sigma=1e-2)
GPT2 = Workload("gpt2_small_psi124439808_n8_stage2", 124439808, 8, 2, "bf16", 5, weight_decay=0.1,
                max_norm=1.0, grad_sigma=1e-3, fan_in_scaled=True, warm_state=True, shapes="gpt2")
FLAT15B = Workload("flat_psi1.5e9_n8_stage1_fp16_ls65536", 1_500_000_000, 8, 1, "fp16", 4,
                   loss_scale=65536.0, grad_sigma=1e-3, warm_state=True, inject_step=3, inject_rank=5)
LLAMA7B = Workload("llama7b_zero3_n8_bf16", 6_738_415_616, 8, 3, "bf16", 1, grad_sigma=1e-3, shapes="llama")


def sweep_points() -> List[Tuple[int, int]]:
    """(psi, N) of the bandwidth sweep, with N*2*psi gradient bytes <= 120 GB."""
    out = []
    for psi in (1 << 20, 1 << 24, 1 << 27, 1 << 29, 1 << 30):
        for n in (2, 4, 8, 16, 32, 64):
            if n * 2 * psi <= 120 * 10 ** 9:
                out.append((psi, n))
    return out


# ---------------------------------------------------------------- drawing
def _gen(device, *seed_parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed_of(*seed_parts))
    return g


def fill_normal(out: torch.Tensor, sigma, gen: torch.Generator, scale_vec: Optional[torch.Tensor] = None,
                absolute: bool = False, multiplier: float = 1.0) -> torch.Tensor:
    """out[i] = cast(N(0,1) * sigma (* scale_vec[i]) (* multiplier)), drawn in CHUNK pieces."""
    flat = out.view(-1)
    n = flat.numel()
    for a in range(0, n, CHUNK):
        b = min(n, a + CHUNK)
        x = torch.randn(b - a, generator=gen, device=out.device, dtype=torch.float32)
        x.mul_(sigma)
        if scale_vec is not None:
            x.mul_(scale_vec[a:b])
        if multiplier != 1.0:
            x.mul_(multiplier)
        if absolute:
            x.abs_()
        flat[a:b].copy_(x)
    return out


def fan_in_scale(shapes, device) -> torch.Tensor:
    """Per-element 1/sqrt(fan_in) with fan_in = shape[-1] (Linear [out, in], Embedding [V, d], 1-D: length)."""
    parts = [torch.full((numel(s),), 1.0 / math.sqrt(s[-1]), dtype=torch.float32, device=device)
             for _, s in shapes]
    return torch.cat(parts)


def shapes_of(w: Workload):
    return {"gpt2": gpt2_small_shapes, "llama": llama7b_shapes}[w.shapes]() if w.shapes else None


def draw_master(w: Workload, out: torch.Tensor, psi: int) -> None:
    """fp32 master N(0, 0.02^2) over [0, psi); padding zero."""
    out.zero_()
    fill_normal(out[:psi], 0.02, _gen(out.device, w.name, "master"))


def draw_moments(w: Workload, m: torch.Tensor, v: torch.Tensor, psi: int) -> None:
    """m N(0, 1e-4^2), v |N(0, 1e-6^2)| when the workload starts warm, else zeros."""
    m.zero_()
    v.zero_()
    if w.warm_state:
        fill_normal(m[:psi], 1e-4, _gen(m.device, w.name, "m"))
        fill_normal(v[:psi], 1e-6, _gen(v.device, w.name, "v"), absolute=True)


def draw_grads(w: Workload, out: torch.Tensor, psi: int, step: int, rank: int, loss_scale: float,
               scale_vec: Optional[torch.Tensor] = None, offset: int = 0) -> None:
    """Rank `rank`'s 16-bit gradient of `step` for global elements [offset, offset+len(out)).

    N(0, sigma^2) (times 1/sqrt(fan_in) per tensor when the workload says so)
    times the current loss scale; elements at or past psi are zero.  The
    stream is keyed by (workload, step, rank, offset) so buckets draw
    independently.
    """
    out.zero_()
    real = max(0, min(out.numel(), psi - offset))
    if real == 0:
        return
    sv = scale_vec[offset:offset + real] if scale_vec is not None else None
    fill_normal(out[:real], w.grad_sigma, _gen(out.device, w.name, "grad", step, rank, offset), sv,
                multiplier=loss_scale)


def inject_index(w: Workload, psi: int) -> int:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed_of(w.name, "inject"))
    return int(torch.randint(0, psi, (1,), generator=g).item())


def inject_inf(w: Workload, grads_rank: torch.Tensor, psi: int) -> int:
    """Write +inf at the workload's seeded index; return that index."""
    idx = inject_index(w, psi)
    grads_rank.view(-1)[idx] = float("inf")
    return idx
