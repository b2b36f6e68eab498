"""Oracle: the ZeRO partitioned mixed-precision step, written out plainly.

TEST INFRASTRUCTURE ONLY (see the package docstring).  numpy, one core,
no blocking or fusion: every array statement below is one step of the
method in the order the pages give it.

Sources (web pages on ZeRO; cited by title and section):

* "zero-stages-simulation" README (32 virtual GPUs): the mixed-precision
  layout table (2+2+4+4+4 bytes per parameter), the flat contiguous
  partition ("GPU r owns chunk r"), the per-stage schedule table
  (all-reduce / reduce-scatter / all-gather per stage), and the
  equivalence claim that all stages give identical trained weights.
* "ZeRO Stage 1/2/3" guide: per-stage memory formulas and the worked
  7B / 13B tables.
* "ZeRO: Memory Optimizations Toward Training Trillion Parameter Models"
  summary: Sec. 3.1 model-state memory (2Psi + 2Psi + K Psi, K = 12),
  Sec. 5 stages P_os / P_os+g / P_os+g+p with their memory equations,
  Sec. 7 communication volume (2 Psi, 2 Psi, 3 Psi), the flattened buffer
  used for the gradient-norm computation (residual states).
* "CMU 11-868 L18: How ZeRO Cuts Data-Parallel Memory": the ZeRO-1 call
  sequence (reduce-scatter that sums and averages into an FP32 shard,
  update of the FP32 shard, copy to FP16, all-gather), ZeRO-2 reduce to
  owner, ZeRO-3 broadcast from owner before forward and again before
  backward.

Readings taken where the pages are silent:

* Adam: Kingma & Ba with the eps added to the bias-corrected sqrt(v);
  written with t = number of applied steps + 1 and these fp32 operations,
  each rounded once, in this order::

      p   = p * dfac                       dfac = f32(1 - lr*wd)   (AdamW)
      m   = b1*m + a1*g                    a1 = f32(1 - b1)
      v   = b2*v + a2*(g*g)                a2 = f32(1 - b2)
      den = sqrt(v) / bc2s + eps           bc2s = f32(sqrt(1 - b2**t))
      p   = p - step_size * (m / den)      step_size = f32(lr / (1 - b1**t))

  The scalar coefficients are formed in double from the fp32 hyper
  parameters and rounded once to fp32.
* Reduction: s = +0.0; s = s + f32(g_r) for r = 0..N-1 (fixed order);
  g_hat = s / f32(N * loss_scale).
* Overflow: any non-finite g_hat over the real elements -> the step is
  skipped, all model state is left bit-identical, the loss scale halves
  (floor 1.0) and t does not advance.
* Norm: sum of g_hat**2 in fp64, left to right within each owner shard,
  then the shards' sums in rank order; clip factor c = max_norm /
  (norm + 1e-6) in double, applied as g_hat * f32(c) only when
  max_norm > 0 and c < 1.
* Cast: IEEE round-to-nearest-even to fp16 (overflow to inf) or bf16.
* Padding elements [psi, psi_pad) are never updated; they stay zero.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

FP16 = "fp16"
BF16 = "bf16"

__all__ = [
    "FP16", "BF16", "Partition", "partition", "model_state_bytes",
    "comm_elems_paper", "comm_elems_ring", "comm_elems_ring_allreduce_zero1",
    "widen16", "rne16", "Hyper", "StepScalars", "step_scalars",
    "rank_sum", "unscale", "has_overflow", "sq_sum_sequential", "grad_norm", "clip_factor",
    "adam_update", "State", "StepResult", "init_state", "step",
    "step_stage0", "step_stage1", "step_stage2", "step_stage3",
    "all_reduce_mean", "reduce_scatter_mean", "all_gather",
    "Q_BLOCK", "quantize_blocks", "dequantize_blocks", "pack_int4", "unpack_int4",
    "quantized_gather", "step_stage3_quantized",
    "persistent_layout", "comm_elems_persistent", "comm_elems_ring_persistent",
    "model_state_bytes_persistent",
    "step_stage3_persistent",
]


# ---------------------------------------------------------------------------
# a1: the flat partition
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Partition:
    psi: int
    n_ranks: int
    align: int
    psi_pad: int
    shard: int
    offsets: Tuple[int, ...]
    real: Tuple[int, ...]


def partition(psi: int, n_ranks: int, align: int = 8) -> Partition:
    """Split the flat buffer into N equal contiguous chunks; rank r owns chunk r.

    "zero-stages-simulation" README, section on flat partitioning: every
    parameter tensor is flattened and split into N near-equal contiguous
    chunks, GPU r owning chunk r.  ZeRO summary Sec. 5 (P_os): the states
    are divided into N_d equal partitions.  Equal partitions need padding:
    psi_pad is the smallest multiple of N*align that is >= psi.
    """
    if psi < 0 or n_ranks < 1 or align < 1:
        raise ValueError("psi >= 0, n_ranks >= 1, align >= 1 required")
    unit = n_ranks * align
    psi_pad = ((psi + unit - 1) // unit) * unit
    shard = psi_pad // n_ranks
    offsets = tuple(r * shard for r in range(n_ranks))
    real = tuple(max(0, min(psi - off, shard)) for off in offsets)
    return Partition(psi, n_ranks, align, psi_pad, shard, offsets, real)


# ---------------------------------------------------------------------------
# D4 / D5: model-state bytes and communication volume (exact integers)
# ---------------------------------------------------------------------------
def model_state_bytes(psi: int, n_ranks: int, stage: int, k: int = 12) -> int:
    """Per-rank model-state bytes of one stage.

    ZeRO summary Sec. 3.1: M = 2Psi + 2Psi + K Psi with K = 12.  Sec. 5:
    P_os = 4Psi + K Psi/N, P_os+g = 2Psi + (2+K)Psi/N, P_os+g+p = (4+K)Psi/N.
    Exact integers when psi is a multiple of n_ranks (pass psi_pad).
    """
    if stage == 0:
        return (4 + k) * psi
    if stage == 1:
        return 4 * psi + (k * psi) // n_ranks
    if stage == 2:
        return 2 * psi + ((2 + k) * psi) // n_ranks
    if stage == 3:
        return ((4 + k) * psi) // n_ranks
    raise ValueError("stage must be 0..3")


def comm_elems_paper(psi: int, stage: int) -> int:
    """Elements a rank communicates per step, the paper's count.

    ZeRO summary Sec. 7: baseline DP all-reduce = reduce-scatter (Psi) +
    all-gather (Psi) = 2Psi; P_os and P_os+g also 2Psi; P_os+g+p adds the
    forward and backward parameter broadcasts: 3Psi.
    """
    if stage in (0, 1, 2):
        return 2 * psi
    if stage == 3:
        return 3 * psi
    raise ValueError("stage must be 0..3")


def comm_elems_ring(psi: int, n_ranks: int, stage: int) -> int:
    """Ring-model elements sent per rank per step: each collective moves (N-1)/N of its size.

    "zero-stages-simulation" README, stage table (1.94 Psi at N = 32 is
    2*(N-1)/N).  Exact when psi is a multiple of n_ranks.
    """
    per = psi // n_ranks * (n_ranks - 1)
    if stage in (0, 1, 2):
        return 2 * per
    if stage == 3:
        return 3 * per
    raise ValueError("stage must be 0..3")


def comm_elems_ring_allreduce_zero1(psi: int, n_ranks: int) -> int:
    """The README's own ZeRO-1 variant: all-reduce grads, then all-gather params.

    "zero-stages-simulation" README, footnote to the stage table: 3*(N-1)/N*Psi.
    """
    return 3 * (psi // n_ranks * (n_ranks - 1))


# ---------------------------------------------------------------------------
# 16-bit formats (IEEE binary16 and bfloat16), bit patterns as uint16
# ---------------------------------------------------------------------------
def widen16(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of 16-bit floats (given as uint16 bit patterns) to fp32."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == FP16:
        return bits.view(np.float16).astype(np.float32)
    if dtype == BF16:
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    raise ValueError(dtype)


def rne16(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 -> 16-bit bit patterns, IEEE round to nearest, ties to even.

    fp16: numpy's float16 conversion (RNE, overflow to inf, subnormals).
    bf16: keep the high half after adding 0x7FFF plus the kept half's lowest
    bit (ties to even); a NaN keeps its sign and gets the quiet bit.
    """
    x = np.asarray(x, dtype=np.float32)
    if dtype == FP16:
        with np.errstate(over="ignore"):
            return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        u = x.view(np.uint32).astype(np.uint64)
        lsb = (u >> np.uint64(16)) & np.uint64(1)
        rounded = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
        nan = np.isnan(x)
        quiet = ((u >> np.uint64(16)).astype(np.uint16)) | np.uint16(0x0040)
        return np.where(nan, quiet, rounded).astype(np.uint16)
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# a7: Adam / AdamW scalars and the elementwise update
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Hyper:
    """Optimizer hyper-parameters, held as fp32 like the C interface does."""
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    max_norm: float = 0.0   # 0 = no clipping


@dataclass(frozen=True)
class StepScalars:
    b1: np.float32
    b2: np.float32
    a1: np.float32
    a2: np.float32
    eps: np.float32
    dfac: np.float32
    step_size: np.float32
    bc2s: np.float32


def _f32(x) -> float:
    return float(np.float32(x))


def step_scalars(h: Hyper, t: int) -> StepScalars:
    """Per-step Adam coefficients for step t (1-based).

    ZeRO summary Sec. 3.1 names mixed-precision Adam with fp32 master,
    momentum and variance; the coefficients are Kingma & Ba's bias
    corrections 1 - beta^t, formed in double and rounded once to fp32.
    """
    if t < 1:
        raise ValueError("t is 1-based")
    lr, b1, b2 = _f32(h.lr), _f32(h.beta1), _f32(h.beta2)
    eps, wd = _f32(h.eps), _f32(h.weight_decay)
    bc1 = 1.0 - math.pow(b1, t)
    bc2 = 1.0 - math.pow(b2, t)
    return StepScalars(
        b1=np.float32(b1), b2=np.float32(b2),
        a1=np.float32(1.0 - b1), a2=np.float32(1.0 - b2),
        eps=np.float32(eps), dfac=np.float32(1.0 - lr * wd),
        step_size=np.float32(lr / bc1), bc2s=np.float32(math.sqrt(bc2)),
    )


def adam_update(p: np.ndarray, m: np.ndarray, v: np.ndarray, g: np.ndarray,
                sc: StepScalars) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """One AdamW update of fp32 master p, momentum m, variance v with gradient g.

    "zero-stages-simulation" README, layout table: the update happens on the
    fp32 master weights, with fp32 m and v.  Each statement is one fp32
    operation (numpy rounds every ufunc result to fp32; nothing is fused).
    """
    p = np.asarray(p, np.float32)
    m = np.asarray(m, np.float32)
    v = np.asarray(v, np.float32)
    g = np.asarray(g, np.float32)
    p = p * sc.dfac
    m = sc.b1 * m + sc.a1 * g
    v = sc.b2 * v + sc.a2 * (g * g)
    den = np.sqrt(v) / sc.bc2s + sc.eps
    p = p - sc.step_size * (m / den)
    return p.astype(np.float32), m.astype(np.float32), v.astype(np.float32)


# ---------------------------------------------------------------------------
# a2..a6: reduction, unscale, overflow, norm, clip
# ---------------------------------------------------------------------------
def rank_sum(grads_f32: Sequence[np.ndarray]) -> np.ndarray:
    """s_i = sum over ranks r = 0..N-1, in that order, in fp32.

    CMU 11-868 notes, ZeRO-1 step 3: the reduce-scatter sums the ranks'
    gradients into an FP32 result.  Starts from +0.0.
    """
    s = np.zeros(np.asarray(grads_f32[0]).shape, np.float32)
    for g in grads_f32:
        s = s + np.asarray(g, np.float32)
    return s


def unscale(s: np.ndarray, n_ranks: int, loss_scale: float) -> np.ndarray:
    """Average over ranks and remove the loss scale: s / f32(N * scale)."""
    den = np.float32(n_ranks) * np.float32(loss_scale)
    return (np.asarray(s, np.float32) / den).astype(np.float32)


def has_overflow(ghat_real: np.ndarray) -> bool:
    """True if any real element of the averaged gradient is inf or nan."""
    return not bool(np.all(np.isfinite(ghat_real)))


def sq_sum_sequential(x: np.ndarray) -> float:
    """sum of x_i**2 in fp64, added left to right from +0 (one rounding per addition).

    np.cumsum adds strictly in order; its last entry is the sequential sum.
    """
    x = np.asarray(x, np.float64)
    if x.size == 0:
        return 0.0
    return float(np.cumsum(x * x)[-1])


def grad_norm(ghat: np.ndarray, part: Partition) -> float:
    """Global L2 norm over the flattened gradient (real elements only).

    ZeRO summary, residual states: the gradient-norm computation runs over
    the flattened gradient buffer.  Each owner sums its shard's squares in
    fp64 sequentially, then the ranks' sums are added in rank order.
    """
    total = 0.0
    for off, real in zip(part.offsets, part.real):
        total = total + sq_sum_sequential(ghat[off:off + real])
    return math.sqrt(total)


def clip_factor(norm: float, max_norm: float) -> Optional[np.float32]:
    """fp32 multiplier for clipping, or None when no clipping applies."""
    if _f32(max_norm) <= 0.0:
        return None
    c = _f32(max_norm) / (norm + 1e-6)
    if c < 1.0:
        return np.float32(c)
    return None


def all_reduce_mean(grads_f32: Sequence[np.ndarray], n: int, scale: float) -> List[np.ndarray]:
    """All-reduce: every rank receives the full averaged gradient."""
    ghat = unscale(rank_sum(grads_f32), n, scale)
    return [ghat.copy() for _ in range(n)]


def reduce_scatter_mean(grads_f32: Sequence[np.ndarray], part: Partition,
                        scale: float) -> List[np.ndarray]:
    """Reduce-scatter: rank r receives only its own shard of the averaged gradient.

    ZeRO summary Sec. 5 (P_os+g): the reduced gradients are scattered so
    each process holds the partition it updates.
    """
    out = []
    for off in part.offsets:
        sl = [np.asarray(g[off:off + part.shard]) for g in grads_f32]
        out.append(unscale(rank_sum(sl), part.n_ranks, scale))
    return out


def all_gather(shards: Sequence[np.ndarray]) -> np.ndarray:
    """All-gather: concatenation of every rank's shard, received by every rank."""
    return np.concatenate([np.asarray(s) for s in shards])


# ---------------------------------------------------------------------------
# the step, per stage
# ---------------------------------------------------------------------------
@dataclass
class State:
    """Model states of all simulated ranks.

    stages 1/2/3: master, m, v are the N owner shards concatenated in rank
    order (length psi_pad).  stage 0: shape (N, psi_pad), one replica each.
    params: (N, psi_pad) uint16 replicas (stages 0/1/2) or the (psi_pad,)
    uint16 concatenation of the N owner shards (stage 3).
    """
    stage: int
    dtype: str
    part: Partition
    master: np.ndarray
    m: np.ndarray
    v: np.ndarray
    params: np.ndarray
    loss_scale: float = 1.0
    t: int = 0           # applied steps so far

    def copy(self) -> "State":
        return State(self.stage, self.dtype, self.part, self.master.copy(),
                     self.m.copy(), self.v.copy(), self.params.copy(),
                     self.loss_scale, self.t)


@dataclass
class StepResult:
    overflow: bool
    applied: bool
    norm: float
    clip: Optional[np.float32]
    gathered_fwd: List[List[np.ndarray]] = field(default_factory=list)
    gathered_bwd: List[List[np.ndarray]] = field(default_factory=list)


def init_state(stage: int, dtype: str, part: Partition, master: np.ndarray,
               m: Optional[np.ndarray] = None, v: Optional[np.ndarray] = None,
               loss_scale: float = 1.0) -> State:
    """Build the per-stage placement of one fp32 master vector (length psi).

    Padding [psi, psi_pad) is zero.  The 16-bit parameters are the RNE cast
    of the master weights (CMU notes, ZeRO-1 step 5).
    """
    psi, pp, n = part.psi, part.psi_pad, part.n_ranks

    def padded(x):
        out = np.zeros(pp, np.float32)
        if x is not None:
            out[:psi] = np.asarray(x, np.float32)[:psi]
        return out

    pm, mm, vv = padded(master), padded(m), padded(v)
    q = rne16(pm, dtype)
    if stage == 0:
        return State(0, dtype, part, np.tile(pm, (n, 1)), np.tile(mm, (n, 1)),
                     np.tile(vv, (n, 1)), np.tile(q, (n, 1)), loss_scale, 0)
    if stage in (1, 2):
        return State(stage, dtype, part, pm, mm, vv, np.tile(q, (n, 1)), loss_scale, 0)
    if stage == 3:
        return State(3, dtype, part, pm, mm, vv, q.copy(), loss_scale, 0)
    raise ValueError("stage must be 0..3")


def _skip(state: State) -> State:
    """Overflow: nothing changes but the loss scale, which halves (floor 1)."""
    out = state.copy()
    out.loss_scale = max(state.loss_scale / 2.0, 1.0)
    return out


def _grads_f32(grads_bits: np.ndarray, dtype: str, psi: int, psi_pad: int) -> List[np.ndarray]:
    """Widen each rank's gradient; padding elements read as zero."""
    out = []
    for g in grads_bits:
        x = widen16(np.asarray(g)[:psi_pad], dtype)
        x = x.copy()
        x[psi:] = 0.0
        out.append(x)
    return out


def step_stage0(state: State, grads_bits: np.ndarray, h: Hyper) -> Tuple[State, StepResult]:
    """ZeRO-0 (plain DP): all-reduce mean, full Adam on every rank, no re-sync.

    "zero-stages-simulation" README, stage table row ZeRO-0; ZeRO summary
    Sec. 7 baseline DP.
    """
    part, n, psi = state.part, state.part.n_ranks, state.part.psi
    g = _grads_f32(grads_bits, state.dtype, psi, part.psi_pad)
    ghat_r = all_reduce_mean(g, n, state.loss_scale)
    if has_overflow(ghat_r[0][:psi]):
        return _skip(state), StepResult(True, False, float("nan"), None)
    norm = grad_norm(ghat_r[0], part)
    c = clip_factor(norm, h.max_norm)
    sc = step_scalars(h, state.t + 1)
    out = state.copy()
    for r in range(n):
        gr = ghat_r[r][:psi]
        if c is not None:
            gr = gr * c
        p, m, v = adam_update(state.master[r][:psi], state.m[r][:psi], state.v[r][:psi], gr, sc)
        out.master[r][:psi], out.m[r][:psi], out.v[r][:psi] = p, m, v
        out.params[r][:psi] = rne16(p, state.dtype)
    out.t = state.t + 1
    return out, StepResult(False, True, norm, c)


def _update_shards(state: State, ghat_shards: Sequence[np.ndarray], h: Hyper,
                   norm: float) -> Tuple[State, Optional[np.float32]]:
    """Each owner updates its own shard of master/m/v (ZeRO summary Sec. 5, P_os)."""
    part = state.part
    c = clip_factor(norm, h.max_norm)
    sc = step_scalars(h, state.t + 1)
    out = state.copy()
    for r, (off, real) in enumerate(zip(part.offsets, part.real)):
        if real == 0:
            continue
        gr = np.asarray(ghat_shards[r][:real], np.float32)
        if c is not None:
            gr = gr * c
        sl = slice(off, off + real)
        p, m, v = adam_update(state.master[sl], state.m[sl], state.v[sl], gr, sc)
        out.master[sl], out.m[sl], out.v[sl] = p, m, v
    out.t = state.t + 1
    return out, c


def _norm_from_shards(ghat_shards: Sequence[np.ndarray], part: Partition) -> float:
    """The norm of grad_norm, from the owners' shards of the averaged gradient."""
    total = 0.0
    for r, real in enumerate(part.real):
        total = total + sq_sum_sequential(ghat_shards[r][:real])
    return math.sqrt(total)


def step_stage1(state: State, grads_bits: np.ndarray, h: Hyper) -> Tuple[State, StepResult]:
    """ZeRO-1 (P_os): full averaged gradient on every rank, owner updates its shard, all-gather.

    ZeRO summary Sec. 5 (P_os): gradients still fully reduced; each process
    updates its partition; an all-gather collects the updated parameters.
    """
    part, n, psi = state.part, state.part.n_ranks, state.part.psi
    g = _grads_f32(grads_bits, state.dtype, psi, part.psi_pad)
    ghat_r = all_reduce_mean(g, n, state.loss_scale)
    if has_overflow(ghat_r[0][:psi]):
        return _skip(state), StepResult(True, False, float("nan"), None)
    shards = [ghat_r[r][off:off + part.shard] for r, off in enumerate(part.offsets)]
    norm = _norm_from_shards(shards, part)
    out, c = _update_shards(state, shards, h, norm)
    q = all_gather([rne16(out.master[off:off + part.shard], state.dtype) for off in part.offsets])
    for r in range(n):
        out.params[r][:psi] = q[:psi]
    return out, StepResult(False, True, norm, c)


def step_stage2(state: State, grads_bits: np.ndarray, h: Hyper) -> Tuple[State, StepResult]:
    """ZeRO-2 (P_os+g): reduce-scatter to owners, owner update, all-gather.

    ZeRO summary Sec. 5 (P_os+g) and Sec. 7: reduce-scatter (Psi) then
    all-gather of the updated parameters (Psi).
    """
    part, n, psi = state.part, state.part.n_ranks, state.part.psi
    g = _grads_f32(grads_bits, state.dtype, psi, part.psi_pad)
    shards = reduce_scatter_mean(g, part, state.loss_scale)
    real_vals = np.concatenate([shards[r][:part.real[r]] for r in range(n)])
    if has_overflow(real_vals):
        return _skip(state), StepResult(True, False, float("nan"), None)
    norm = _norm_from_shards(shards, part)
    out, c = _update_shards(state, shards, h, norm)
    q = all_gather([rne16(out.master[off:off + part.shard], state.dtype) for off in part.offsets])
    for r in range(n):
        out.params[r][:psi] = q[:psi]
    return out, StepResult(False, True, norm, c)


def step_stage3(state: State, bucket_grads: Sequence[np.ndarray],
                buckets: Sequence[Tuple[int, int]], h: Hyper) -> Tuple[State, StepResult]:
    """ZeRO-3 (P_os+g+p): per-bucket gather before forward and before backward,
    per-bucket reduce-scatter to owners, owner update of the 16-bit shard.

    ZeRO summary Sec. 5 (P_os+g+p): parameters broadcast by their owner
    before each layer's forward, again in reverse order in backward, and the
    gradients reduce-scattered as they appear.  CMU notes, ZeRO-3: broadcast
    from owner, compute, discard; backward reduces each segment to its owner.

    bucket_grads[b] has shape (N, b_end - b_start): rank r's 16-bit
    gradient for bucket b.  Buckets must tile [0, psi_pad).
    """
    part, n, psi = state.part, state.part.n_ranks, state.part.psi
    pp = part.psi_pad
    ranges = sorted(buckets)
    if ranges and (ranges[0][0] != 0 or ranges[-1][1] != pp or
                   any(ranges[i][1] != ranges[i + 1][0] for i in range(len(ranges) - 1))):
        raise ValueError("buckets must tile [0, psi_pad)")
    res = StepResult(False, True, 0.0, None)
    # forward: gather every bucket from the owners' shards, in order
    for (a, b) in buckets:
        res.gathered_fwd.append([state.params[a:b].copy() for _ in range(n)])
    # backward: reverse order; gather again, then reduce-scatter the bucket
    ghat = np.zeros(pp, np.float32)
    for idx in range(len(buckets) - 1, -1, -1):
        a, b = buckets[idx]
        res.gathered_bwd.insert(0, [state.params[a:b].copy() for _ in range(n)])
        gb = np.asarray(bucket_grads[idx])
        g = []
        for r in range(n):
            x = widen16(gb[r][:b - a], state.dtype).copy()
            lo = max(0, min(psi, b) - a)
            x[lo:] = 0.0
            g.append(x)
        ghat[a:b] = unscale(rank_sum(g), n, state.loss_scale)
    if has_overflow(ghat[:psi]):
        return _skip(state), StepResult(True, False, float("nan"), None,
                                        res.gathered_fwd, res.gathered_bwd)
    shards = [ghat[off:off + part.shard] for off in part.offsets]
    norm = _norm_from_shards(shards, part)
    out, c = _update_shards(state, shards, h, norm)
    out.params[:psi] = rne16(out.master[:psi], state.dtype)
    res.norm, res.clip = norm, c
    return out, res


# ---------------------------------------------------------------------------
# ZeRO-3 with param_persistence_threshold
# ---------------------------------------------------------------------------
def persistent_layout(sizes: Sequence[int], threshold: int) -> Tuple[List[int], int, int]:
    """Tensor order of the flat buffer when small tensors stay replicated.

    "ZeRO Stage 1/2/3" guide, ZeRO-3 config: parameters with fewer elements
    than param_persistence_threshold stay replicated (the comparison is
    strict: a tensor of exactly the threshold is partitioned).  Reading:
    the partitioned tensors come first and the persistent ones after them,
    each group in model order, so the persistent tensors form one region
    [p0, psi) of the flat buffer.

    Returns (order, p0, psi): order[k] is the model index of the k-th tensor
    in the flat buffer.
    """
    order = []
    for i, n in enumerate(sizes):
        if not n < threshold:
            order.append(i)
    p0 = 0
    for i in order:
        p0 += int(sizes[i])
    for i, n in enumerate(sizes):
        if n < threshold:
            order.append(i)
    return order, p0, int(sum(int(n) for n in sizes))


def comm_elems_persistent(psi: int, psi_pers: int) -> int:
    """Elements a rank communicates per ZeRO-3 step with a persistent region.

    ZeRO summary Sec. 7 counts P_os+g+p as a forward gather (Psi), a
    backward gather (Psi) and a gradient reduce-scatter (Psi).  Persistent
    parameters are not gathered in forward or backward; their replicas are
    refreshed by one all-gather of psi_pers after the update, which is how
    the stage 1/2 parameters are refreshed.
    """
    return 2 * (psi - psi_pers) + psi + psi_pers


def comm_elems_ring_persistent(psi: int, psi_pers: int, n_ranks: int) -> int:
    """Ring-model elements sent per rank per ZeRO-3 step with a persistent region.

    Each collective moves (N-1)/N of its elements ("zero-stages-simulation"
    README, stage table): the forward and backward gathers of the
    partitioned psi - psi_pers, the reduce-scatter of psi and the refresh
    gather of psi_pers, i.e. (N-1)/N of comm_elems_persistent, rounded down.
    """
    return (n_ranks - 1) * comm_elems_persistent(psi, psi_pers) // n_ranks


def model_state_bytes_persistent(psi: int, psi_pers: int, n_ranks: int, k: int = 12) -> int:
    """Per-rank model-state bytes of ZeRO-3 with a persistent region.

    ZeRO summary Sec. 5: P_os+g+p holds (4 + K) Psi / N.  Each rank also
    holds the full 16-bit copy of the persistent parameters (2 psi_pers);
    their owner shards stay, as the source of the refresh.  Exact when psi
    is a multiple of n_ranks (pass psi_pad).
    """
    return ((4 + k) * psi) // n_ranks + 2 * psi_pers


def step_stage3_persistent(state: State, bucket_grads: Sequence[np.ndarray],
                           buckets: Sequence[Tuple[int, int]], h: Hyper,
                           p0: int) -> Tuple[State, StepResult, List[np.ndarray]]:
    """ZeRO-3 step whose region [p0, psi_pad) stays replicated.

    Same update as step_stage3 (persistence moves no value, only where the
    16-bit copies live): buckets ending at or before p0 are gathered in
    forward and in backward; buckets starting at or after p0 are only
    reduce-scattered.  After the update every rank's persistent copy is the
    all-gather of the new shards over [p0, psi_pad); after a skipped step it
    is the unchanged old one.

    Returns (state, result, replicas) with replicas a list of N uint16
    arrays of length psi_pad - p0.  result.gathered_fwd / gathered_bwd hold
    the gathered buckets only.
    """
    for (a, b) in buckets:
        if a < p0 < b:
            raise ValueError("a bucket straddles the persistent boundary")
    out, res = step_stage3(state, bucket_grads, buckets, h)
    keep = [i for i, (a, b) in enumerate(buckets) if b <= p0 and a < p0]
    res.gathered_fwd = [res.gathered_fwd[i] for i in keep]
    res.gathered_bwd = [res.gathered_bwd[i] for i in keep]
    pp = state.part.psi_pad
    replicas = [out.params[p0:pp].copy() for _ in range(state.part.n_ranks)]
    return out, res, replicas


def step(state: State, grads_bits: np.ndarray, h: Hyper,
         buckets: Optional[Sequence[Tuple[int, int]]] = None) -> Tuple[State, StepResult]:
    """Dispatch one step by stage.  grads_bits: (N, >= psi_pad) uint16.

    For stage 3 the full gradients are cut into the given buckets (default:
    one bucket covering [0, psi_pad)).
    """
    if state.stage == 0:
        return step_stage0(state, grads_bits, h)
    if state.stage == 1:
        return step_stage1(state, grads_bits, h)
    if state.stage == 2:
        return step_stage2(state, grads_bits, h)
    if state.stage == 3:
        pp = state.part.psi_pad
        if buckets is None:
            buckets = [(0, pp)]
        bg = [np.asarray(grads_bits)[:, a:b] for (a, b) in buckets]
        return step_stage3(state, bg, buckets, h)
    raise ValueError("stage must be 0..3")


# ---------------------------------------------------------------------------
# ZeRO++ quantized collectives (block-wise zero-point quantization)
# ---------------------------------------------------------------------------
Q_BLOCK = 256


def quantize_blocks(x: np.ndarray, bits: int, block: int = Q_BLOCK):
    """Block-wise zero-point (asymmetric) quantization of fp32 values.

    "CMU 11-868 L18" notes, other memory optimizations (ZeRO++): parameters
    are block-quantized from FP16 to INT8 with zero-point quantization for
    the forward gather, and the backward reduce-scatter is quantized to INT8
    or INT4.  The notes give no formula; the reading taken is the plain
    zero-point definition: blocks of `block` consecutive elements from the
    start of the buffer (the last one may be short); per block lo = min,
    hi = max and scale = (hi - lo) / (2^bits - 1); code q = rint((x - lo) / scale)
    clamped to [0, 2^bits - 1], or 0 when scale is 0.  Every operation is
    one fp32 operation rounded once (subtract, divide, then round half to
    even).  min/max propagate NaN (a NaN element makes its whole block NaN
    after dequantization, so overflow detection still sees it); a code that
    comes out NaN is stored as 0.  Returns
    (codes uint8, one per element; scale fp32; lo fp32).
    """
    if bits not in (4, 8):
        raise ValueError("bits must be 4 or 8")
    x = np.asarray(x, np.float32)
    n = x.size
    nb = (n + block - 1) // block
    qmax = np.float32((1 << bits) - 1)
    codes = np.zeros(n, np.uint8)
    scale = np.zeros(nb, np.float32)
    lo = np.zeros(nb, np.float32)
    for k in range(nb):
        blk = x[k * block:(k + 1) * block]
        # min/max with NaN propagation; a zero bound is taken as +0
        l = np.float32(blk.min()) + np.float32(0.0)
        hgh = np.float32(blk.max()) + np.float32(0.0)
        rng = np.float32(hgh - l)
        s = rng / qmax
        scale[k], lo[k] = s, l
        if s != 0:
            with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
                q = np.rint((blk - l) / s)
            q = np.where(np.isnan(q), 0, q)          # a NaN's code is 0 (its block is NaN anyway)
            codes[k * block:(k + 1) * block] = np.clip(q, 0, qmax).astype(np.uint8)
    return codes, scale, lo


def dequantize_blocks(codes: np.ndarray, scale: np.ndarray, lo: np.ndarray, block: int = Q_BLOCK) -> np.ndarray:
    """x' = lo + q * scale per block, in fp32 (a multiply, then an add)."""
    codes = np.asarray(codes)
    k = np.arange(codes.size) // block
    with np.errstate(invalid="ignore", over="ignore"):
        return (lo[k] + codes.astype(np.float32) * scale[k]).astype(np.float32)


def pack_int4(codes: np.ndarray) -> np.ndarray:
    """Two 4-bit codes per byte: element 2i in the low nibble, 2i+1 in the high one."""
    c = np.asarray(codes, np.uint8)
    if c.size % 2:
        c = np.concatenate([c, np.zeros(1, np.uint8)])
    return (c[0::2] & 0x0F) | ((c[1::2] & 0x0F) << 4)


def unpack_int4(packed: np.ndarray, n: int) -> np.ndarray:
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.size * 2, np.uint8)
    out[0::2] = p & 0x0F
    out[1::2] = p >> 4
    return out[:n]


def quantized_gather(shard16: np.ndarray, a: int, b: int, dtype: str, n_ranks: int):
    """ZeRO++ weight gather of bucket [a, b): the owners' 16-bit values are
    block-quantized to INT8 once and every rank receives codes and scales;
    a rank's view of the parameters is their dequantization, cast to 16 bits."""
    x = widen16(np.asarray(shard16)[a:b], dtype)
    codes, scale, lo = quantize_blocks(x, 8)
    view16 = rne16(dequantize_blocks(codes, scale, lo), dtype)
    return [(codes.copy(), scale.copy(), lo.copy()) for _ in range(n_ranks)], view16


def step_stage3_quantized(state: "State", bucket_grads: Sequence[np.ndarray],
                          buckets: Sequence[Tuple[int, int]], h: "Hyper", bits: int) -> Tuple["State", "StepResult"]:
    """ZeRO-3 step whose gradient reduce-scatter is quantized (ZeRO++ qgZ).

    Each rank block-quantizes its bucket gradient (blocks from the bucket's
    start) to `bits`; the owner sums the N dequantized gradients in rank order
    and the step proceeds exactly as step_stage3 (unscale, flag, norm, clip,
    AdamW, cast).  Gathers are not modelled here (see quantized_gather).
    """
    part, n, psi = state.part, state.part.n_ranks, state.part.psi
    pp = part.psi_pad
    ghat = np.zeros(pp, np.float32)
    for idx in range(len(buckets) - 1, -1, -1):
        a, b = buckets[idx]
        gb = np.asarray(bucket_grads[idx])
        g = []
        lo_i = max(0, min(psi, b) - a)
        for r in range(n):
            x = widen16(gb[r][:b - a], state.dtype)
            codes, scale, lo = quantize_blocks(x, bits)
            xq = dequantize_blocks(codes, scale, lo)
            xq[lo_i:] = 0.0          # padding reads as zero after the exchange
            g.append(xq)
        ghat[a:b] = unscale(rank_sum(g), n, state.loss_scale)
    res = StepResult(False, True, 0.0, None)
    if has_overflow(ghat[:psi]):
        return _skip(state), StepResult(True, False, float("nan"), None)
    shards = [ghat[off:off + part.shard] for off in part.offsets]
    norm = _norm_from_shards(shards, part)
    out, c = _update_shards(state, shards, h, norm)
    out.params[:psi] = rne16(out.master[:psi], state.dtype)
    res.norm, res.clip = norm, c
    return out, res
