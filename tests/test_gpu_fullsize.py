"""Parity at the full sizes of the workloads, in the launch configuration the
bench times, over every element: the 1.5B stage-1 step (with its overflow
step), the GPT-2-small stage-2 step with clipping, the toy buffer at all
four stages, one Llama-7B ZeRO-3 step, and corners of the bandwidth sweep
(psi = 2^30 at N = 2, 2^29 at N = 4, 2^27 at N = 64).

Each applied step is checked in full: its new fp32 state and every 16-bit
copy against the oracle's update of the state the step started from (read
back from the device's other state slot, itself checked by the step
before), its global norm and overflow flag against the oracle's over all
elements (tests/_fullsize.py streams the buffers chunk by chunk).  A
skipped step must leave the state and copies unchanged: their digests are
compared with those taken after the last applied step.
"""

import numpy as np
import pytest
import torch

import oracle as O
from _fullsize import FullCheck
from _parity import NORM_RTOL, ULP16, ULP32, run_case
from zero_partitioned_mixed_gb300 import _binding as B
from zero_partitioned_mixed_gb300 import synth as S
from zero_partitioned_mixed_gb300.buffers import RankBuffers

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def fc():
    p = FullCheck()
    yield p
    p.close()


def _hyper(w, mode=B.ZERO_MODE_AUTO):
    return (B.hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm, mode),
            O.Hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm))


def _assert_exact(tal, count):
    assert tal.compared == count, (tal.compared, count)
    assert tal.max_ulp32 <= ULP32 and tal.max_ulp16 <= ULP16
    assert tal.mismatches == 0, f"{tal.mismatches} of {tal.compared} elements differ"


def _assert_norm(got, want):
    assert abs(got - want) <= NORM_RTOL * want, (got, want)


@pytest.mark.parametrize("mode", [B.ZERO_MODE_AUTO, B.ZERO_MODE_SPECULATIVE_STAGED])
def test_flat_1p5b_stage1_four_steps_with_overflow(fc, mode):
    # the bench's workload in both of its launch configurations
    w = S.FLAT15B
    hb, ho = _hyper(w, mode)
    n, dt = w.n_ranks, w.dtype
    buf = RankBuffers(w.psi, n, w.stage, dt, double_buffer=True, alloc_grads=False)
    P = buf.psi_pad
    part = O.partition(w.psi, n, 8)
    mv, mm, vv = buf.state(0)
    S.draw_master(w, mv, w.psi)
    S.draw_moments(w, mm, vv, w.psi)
    buf.params[:, :P].copy_(mv.to(S.torch_dtype(dt)).unsqueeze(0).expand(n, P))
    grads = torch.empty((n, buf.stride), dtype=S.torch_dtype(dt), device="cuda")
    buf.set_scaler(w.loss_scale, 0, 0)
    scale, t, slot, saved = w.loss_scale, 0, 0, None
    for k in range(w.steps):
        for r in range(n):
            S.draw_grads(w, grads[r], w.psi, k + 1, r, scale)
        if k + 1 == w.inject_step:
            S.inject_inf(w, grads[w.inject_rank], w.psi)
        buf.step(hb, [grads[r] for r in range(n)])
        st = buf.status()
        assert bool(st["overflow"]) == (k + 1 == w.inject_step)
        if not st["overflow"]:
            tal = fc.compare(0, P, psi=w.psi, part=part, dtype=dt, grads=grads, old=buf.state(slot),
                             new=buf.state(st["state_slot"]), q=buf.params, loss_scale=scale,
                             sc=O.step_scalars(ho, t + 1), digest=True)
            assert not tal.bad
            _assert_exact(tal, (3 + n) * P)
            _assert_norm(st["grad_norm"], tal.norm(n))
            saved = tal.digests
            t += 1
        else:
            # the oracle's flag over every element; state and replicas untouched
            tal = fc.compare(0, P, psi=w.psi, part=part, dtype=dt, grads=grads, loss_scale=scale)
            assert tal.bad
            assert st["state_slot"] == slot
            kept = fc.compare(0, P, psi=w.psi, part=part, dtype=dt, new=buf.state(slot), q=buf.params,
                              digest=True)
            assert kept.digests == saved
            scale = max(scale / 2, 1.0)
        slot = st["state_slot"]
        assert st["steps_applied"] == t and st["loss_scale"] == np.float32(scale)
    buf.close()
    del grads, buf
    torch.cuda.empty_cache()


@pytest.mark.parametrize("double_buffer", [False, True])
def test_gpt2_small_stage2_clip_five_steps(fc, double_buffer):
    # two-pass (clip decided before the update, state updated in place) and
    # speculative (redo only if the norm exceeds max_norm, which it does not here)
    w = S.GPT2
    hb, ho = _hyper(w)
    n, dt = w.n_ranks, w.dtype
    buf = RankBuffers(w.psi, n, 2, dt, double_buffer=double_buffer, alloc_grads=False)
    P = buf.psi_pad
    part = O.partition(w.psi, n, 8)
    mv, mm, vv = buf.state(0)
    S.draw_master(w, mv, w.psi)
    S.draw_moments(w, mm, vv, w.psi)
    buf.params[:, :P].copy_(mv.to(S.torch_dtype(dt)).unsqueeze(0).expand(n, P))
    sv = S.fan_in_scale(S.gpt2_small_shapes(), "cuda")
    grads = torch.empty((n, buf.stride), dtype=S.torch_dtype(dt), device="cuda")
    buf.set_scaler(1.0, 0, 0)
    slot = 0
    for k in range(w.steps):
        for r in range(n):
            S.draw_grads(w, grads[r], w.psi, k + 1, r, 1.0, sv)
        pre = fc.compare(0, P, psi=w.psi, part=part, dtype=dt, grads=grads)
        norm = pre.norm(n)
        clip = O.clip_factor(norm, w.max_norm)
        old = buf.state(slot) if double_buffer else [x.clone() for x in buf.state(0)]
        buf.step(hb, [grads[r] for r in range(n)])
        st = buf.status()
        assert not pre.bad and not st["overflow"]
        _assert_norm(st["grad_norm"], norm)
        assert st["clip_coef"] == (float(clip) if clip is not None else 1.0)
        tal = fc.compare(0, P, psi=w.psi, part=part, dtype=dt, grads=grads, old=old,
                         new=buf.state(st["state_slot"]), q=buf.params, sc=O.step_scalars(ho, k + 1), clip=clip)
        _assert_exact(tal, (3 + n) * P)
        slot = st["state_slot"]
        del old
    buf.close()
    del grads, sv, buf
    torch.cuda.empty_cache()


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_toy_buffer_all_stages_full(stage):
    # psi = 637,824 over 32 ranks, fp16, 3 steps: compared element by element in full
    buckets = None
    if stage == 3:
        buckets = S.flat_buckets(637_952, 32, 50_000)
    st = run_case(637_824, 32, stage, "fp16", steps=3, sigma=1e-2, warm=False,
                  double_buffer=(stage != 0), buckets=buckets)
    st.check()
    assert st.mismatches == 0


def _zero3_step(fc, w, buf, part, buckets, hb, ho, step, fused=True):
    """One ZeRO-3 step over the given buckets (gathers before forward and
    backward, each bucket's gradients drawn on the device and
    reduce-scattered; with `fused` each backward reduce-scatter carries the
    next bucket's gather, as the bench times it), checked in full."""
    n, dt = w.n_ranks, w.dtype
    td = S.torch_dtype(dt)
    lmax = max(b - a for a, b in buckets)
    lpad = (lmax + 7) // 8 * 8
    outs = torch.empty((2, n, lpad), dtype=td, device="cuda")
    gbuf = torch.empty((n, lpad), dtype=td, device="cuda")
    shard0 = buf.params.clone()

    def check_gather(a, b, o):
        # the gather is a copy of the owners' values: every rank's row equals the shard
        for r in range(n):
            assert torch.equal(o[r, :b - a], shard0[a:b])

    def draw(a):
        for r in range(n):
            S.draw_grads(w, gbuf[r], w.psi, step, r, 1.0, offset=a)

    st0 = buf.status()
    slot = st0["state_slot"]
    for (a, b) in buckets:                       # forward
        buf.gather(a, b, [outs[0, r] for r in range(n)])
        check_gather(a, b, outs[0])
    back = list(reversed(buckets))               # backward
    if fused:
        buf.gather(back[0][0], back[0][1], [outs[0, r] for r in range(n)])
        check_gather(back[0][0], back[0][1], outs[0])
        for k, (a, b) in enumerate(back):
            draw(a)
            if k + 1 < len(back):
                ga, gb = back[k + 1]
                o = outs[(k + 1) % 2]
                buf.reduce_scatter_gather(a, b, [gbuf[r] for r in range(n)], hb, ga, gb, [o[r] for r in range(n)])
                check_gather(ga, gb, o)
            else:
                buf.reduce_scatter(a, b, [gbuf[r] for r in range(n)], hb)
    else:
        for (a, b) in back:
            buf.gather(a, b, [outs[0, r] for r in range(n)])
            check_gather(a, b, outs[0])
            draw(a)
            buf.reduce_scatter(a, b, [gbuf[r] for r in range(n)], hb)
    buf.step(hb)
    st = buf.status()
    assert not st["overflow"] and st["applied"] and st["steps_applied"] == st0["steps_applied"] + 1
    # the same gradients again (same generator, offset and buffer length), bucket by bucket
    tal = None
    for (a, b) in buckets:
        draw(a)
        tal = fc.compare(a, b, psi=w.psi, part=part, dtype=dt, grads=gbuf, g_base=a, old=buf.state(slot),
                         new=buf.state(st["state_slot"]), q=buf.params, loss_scale=1.0,
                         sc=O.step_scalars(ho, st0["steps_applied"] + 1), tally=tal)
    assert not tal.bad
    _assert_exact(tal, 4 * part.psi_pad)
    _assert_norm(st["grad_norm"], tal.norm(n))
    del outs, gbuf, shard0


def test_llama7b_zero3_one_step(fc):
    w = S.LLAMA7B
    hb, ho = _hyper(w)
    n, dt = w.n_ranks, w.dtype
    buf = RankBuffers(w.psi, n, 3, dt, double_buffer=True)
    P = buf.psi_pad
    part = O.partition(w.psi, n, 8)
    buckets = S.layer_buckets(S.llama7b_shapes(), P)
    assert len(buckets) == 34 and buckets[1][1] - buckets[1][0] == 202_383_360
    mv, mm, vv = buf.state(0)
    S.draw_master(w, mv, w.psi)
    S.draw_moments(w, mm, vv, w.psi)
    buf.params[:P].copy_(mv.to(S.torch_dtype(dt)))
    buf.set_scaler(1.0, 0, 0)
    _zero3_step(fc, w, buf, part, buckets, hb, ho, 1)
    buf.close()
    del buf
    torch.cuda.empty_cache()


# corners of the bandwidth sweep: the longest chunks of the one-pass step
# (psi = 2^30, N = 2), the reduce-scatter's chunk cap for N <= 4, and the
# widest rank loops (N = 64); bf16 N(0, 1e-3^2), Adam defaults, 2 steps
SWEEP_CORNERS = [(1 << 30, 2, 1), (1 << 30, 2, 3), (1 << 29, 4, 3), (1 << 27, 64, 1), (1 << 27, 64, 3)]


@pytest.mark.parametrize("psi,n,stage", SWEEP_CORNERS)
def test_sweep_corner(fc, psi, n, stage):
    w = S.Workload(f"sweep_psi{psi}_n{n}", psi, n, stage, "bf16", 2, grad_sigma=1e-3)
    hb, ho = _hyper(w)
    dt = w.dtype
    td = S.torch_dtype(dt)
    buf = RankBuffers(psi, n, stage, dt, double_buffer=True, alloc_grads=False)
    P = buf.psi_pad
    part = O.partition(psi, n, 8)
    mv, mm, vv = buf.state(0)
    S.draw_master(w, mv, psi)
    S.draw_moments(w, mm, vv, psi)
    buf.set_scaler(1.0, 0, 0)
    if stage == 3:
        buf.params[:P].copy_(mv.to(td))
        buckets = S.flat_buckets(P, n, 50_000_000)
        for k in range(w.steps):
            _zero3_step(fc, w, buf, part, buckets, hb, ho, k + 1)
    else:
        buf.params[:, :P].copy_(mv.to(td).unsqueeze(0).expand(n, P))
        grads = torch.empty((n, buf.stride), dtype=td, device="cuda")
        slot = 0
        for k in range(w.steps):
            for r in range(n):
                S.draw_grads(w, grads[r], psi, k + 1, r, 1.0)
            buf.step(hb, [grads[r] for r in range(n)])
            st = buf.status()
            assert not st["overflow"] and st["steps_applied"] == k + 1
            tal = fc.compare(0, P, psi=psi, part=part, dtype=dt, grads=grads, old=buf.state(slot),
                             new=buf.state(st["state_slot"]), q=buf.params, sc=O.step_scalars(ho, k + 1))
            assert not tal.bad
            _assert_exact(tal, (3 + n) * P)
            _assert_norm(st["grad_norm"], tal.norm(n))
            slot = st["state_slot"]
        del grads
    buf.close()
    del buf
    torch.cuda.empty_cache()
