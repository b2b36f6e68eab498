"""Parity at the full sizes of the workloads, in the launch configuration the
bench times: the 1.5B stage-1 step (with its overflow step), the GPT-2-small
stage-2 step with clipping, the toy buffer at all four stages, and one
Llama-7B ZeRO-3 step.  Elements are compared on samples (both ends, every
shard boundary, the injected index and random positions) against the
oracle computing them one by one; the global norm and overflow flag of the
first steps are compared against the oracle over all elements.
"""

import numpy as np
import pytest
import torch

import oracle as O
from _fullsize import NormPool, gather_bits16, gather_f32, oracle_sampled_step, sample_indices
from _parity import NORM_RTOL, ULP16, ULP32, bits16, bits32, run_case, ulp16, ulp32
from zero_partitioned_mixed_gb300 import _binding as B
from zero_partitioned_mixed_gb300 import synth as S
from zero_partitioned_mixed_gb300.buffers import RankBuffers

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def pool():
    p = NormPool()
    yield p
    p.close()


def _hyper(w, mode=B.ZERO_MODE_AUTO):
    return (B.hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm, mode),
            O.Hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm))


def _check_samples(buf, slot, idx_t, p, m, v, dtype, n, stage):
    gm, gmm, gv = buf.state(slot)
    for dev, ref in ((gm, p), (gmm, m), (gv, v)):
        got = gather_f32(dev, idx_t)
        assert int(ulp32(got.view(np.uint32), ref.view(np.uint32)).max()) <= ULP32
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    want_q = O.rne16(p, dtype)
    if stage == 3:
        q = gather_bits16(buf.params, idx_t)
        assert int(ulp16(q, want_q).max()) <= ULP16 and np.array_equal(q, want_q)
    else:
        q = gather_bits16(buf.params, idx_t)    # (N, K)
        for r in range(n):
            assert int(ulp16(q[r], want_q).max()) <= ULP16 and np.array_equal(q[r], want_q)


@pytest.mark.parametrize("mode", [B.ZERO_MODE_AUTO, B.ZERO_MODE_SPECULATIVE_STAGED])
def test_flat_1p5b_stage1_four_steps_with_overflow(pool, mode):
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
    inj = S.inject_index(w, w.psi)
    idx = sample_indices(P, part, 1 << 16, 5, extra=[inj, inj - 1, inj + 1])
    idx_t = torch.from_numpy(idx).cuda()
    valid = (idx < w.psi).astype(np.float32)
    p, m, v = gather_f32(mv, idx_t), gather_f32(mm, idx_t), gather_f32(vv, idx_t)
    buf.set_scaler(w.loss_scale, 0, 0)
    scale, t = w.loss_scale, 0
    for k in range(w.steps):
        for r in range(n):
            S.draw_grads(w, grads[r], w.psi, k + 1, r, scale)
        if k + 1 == w.inject_step:
            S.inject_inf(w, grads[w.inject_rank], w.psi)
        gs = gather_bits16(grads, idx_t)
        if k == 0:
            norm, bad_full = pool.norm_and_flag([grads[r] for r in range(n)], w.psi, part, dt, scale)
        buf.step(hb, [grads[r] for r in range(n)])
        st = buf.status()
        p2, m2, v2, bad = oracle_sampled_step(p, m, v, gs, n, dt, scale, ho, t + 1, None, valid)
        assert bool(st["overflow"]) == bad == (k + 1 == w.inject_step)
        if k == 0:
            assert not bad_full
            assert abs(st["grad_norm"] - norm) <= NORM_RTOL * norm
        if bad:
            scale = max(scale / 2, 1.0)
        else:
            t += 1
            p, m, v = p2, m2, v2
        assert st["steps_applied"] == t and st["loss_scale"] == np.float32(scale)
        _check_samples(buf, st["state_slot"], idx_t, p, m, v, dt, n, 1)
    buf.close()
    del grads, buf
    torch.cuda.empty_cache()


@pytest.mark.parametrize("double_buffer", [False, True])
def test_gpt2_small_stage2_clip_five_steps(pool, double_buffer):
    # two-pass (clip decided before the update) and speculative (redo only
    # if the norm exceeds max_norm, which it does not here)
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
    idx = sample_indices(P, part, 1 << 16, 6)
    idx_t = torch.from_numpy(idx).cuda()
    valid = (idx < w.psi).astype(np.float32)
    p, m, v = gather_f32(mv, idx_t), gather_f32(mm, idx_t), gather_f32(vv, idx_t)
    buf.set_scaler(1.0, 0, 0)
    for k in range(w.steps):
        for r in range(n):
            S.draw_grads(w, grads[r], w.psi, k + 1, r, 1.0, sv)
        norm, bad_full = pool.norm_and_flag([grads[r] for r in range(n)], w.psi, part, dt, 1.0)
        clip = O.clip_factor(norm, w.max_norm)
        gs = gather_bits16(grads, idx_t)
        buf.step(hb, [grads[r] for r in range(n)])
        st = buf.status()
        assert not bad_full and not st["overflow"]
        assert abs(st["grad_norm"] - norm) <= NORM_RTOL * norm
        assert st["clip_coef"] == (float(clip) if clip is not None else 1.0)
        p, m, v, bad = oracle_sampled_step(p, m, v, gs, n, dt, 1.0, ho, k + 1, clip, valid)
        assert not bad
        _check_samples(buf, st["state_slot"], idx_t, p, m, v, dt, n, 2)
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


def test_llama7b_zero3_one_step():
    w = S.LLAMA7B
    hb, ho = _hyper(w)
    n, dt = w.n_ranks, w.dtype
    td = S.torch_dtype(dt)
    buf = RankBuffers(w.psi, n, 3, dt, double_buffer=True)
    P = buf.psi_pad
    part = O.partition(w.psi, n, 8)
    buckets = S.layer_buckets(S.llama7b_shapes(), P)
    assert len(buckets) == 34 and buckets[1][1] - buckets[1][0] == 202_383_360
    mv, mm, vv = buf.state(0)
    S.draw_master(w, mv, w.psi)
    S.draw_moments(w, mm, vv, w.psi)
    buf.params[:P].copy_(mv.to(td))
    idx = sample_indices(P, part, 1 << 16, 7, extra=[a for a, _ in buckets] + [b - 1 for _, b in buckets])
    idx_t = torch.from_numpy(idx).cuda()
    shard0 = gather_bits16(buf.params, idx_t)
    p, m, v = gather_f32(mv, idx_t), gather_f32(mm, idx_t), gather_f32(vv, idx_t)
    lmax = max(b - a for a, b in buckets)
    lpad = (lmax + 7) // 8 * 8
    outs = torch.empty((n, lpad), dtype=td, device="cuda")
    gbuf = torch.empty((n, lpad), dtype=td, device="cuda")
    gs = np.zeros((n, idx.size), np.uint16)
    buf.set_scaler(1.0, 0, 0)

    def check_gather(a, b):
        sel = (idx >= a) & (idx < b)
        loc = torch.from_numpy(idx[sel] - a).cuda()
        got = gather_bits16(outs, loc)
        for r in range(n):
            assert np.array_equal(got[r], shard0[sel])

    for (a, b) in buckets:                       # forward
        buf.gather(a, b, [outs[r] for r in range(n)])
        check_gather(a, b)
    for bi in range(len(buckets) - 1, -1, -1):   # backward
        a, b = buckets[bi]
        buf.gather(a, b, [outs[r] for r in range(n)])
        check_gather(a, b)
        for r in range(n):
            S.draw_grads(w, gbuf[r], w.psi, 1, r, 1.0, offset=a)
        sel = np.nonzero((idx >= a) & (idx < b))[0]
        loc = torch.from_numpy(idx[sel] - a).cuda()
        gs[:, sel] = gather_bits16(gbuf, loc)
        buf.reduce_scatter(a, b, [gbuf[r] for r in range(n)], hb)
    buf.step(hb)
    st = buf.status()
    valid = (idx < w.psi).astype(np.float32)
    p2, m2, v2, bad = oracle_sampled_step(p, m, v, gs, n, dt, 1.0, ho, 1, None, valid)
    assert not bad and not st["overflow"] and st["applied"] and st["steps_applied"] == 1
    assert st["grad_norm"] > 0
    _check_samples(buf, st["state_slot"], idx_t, p2, m2, v2, dt, n, 3)
    buf.close()
    del outs, gbuf, buf
    torch.cuda.empty_cache()
