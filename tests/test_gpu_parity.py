"""CUDA path vs the oracle, element by element, through the C ABI.

Sizes span several 8-element groups per thread, several blocks and a
ragged tail; every stage, mode and dtype; overflow, clipping, padding,
non-power-of-two scales, N up to 64, empty inputs and unaligned buckets.
"""

import numpy as np
import pytest
import torch

from _parity import ULP16, ULP32, bits16, bits32, run_case, ulp16, ulp32

pytestmark = pytest.mark.gpu

INF, NINF, NAN = float("inf"), float("-inf"), float("nan")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("stage", [1, 2])
@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_stage12_modes(stage, mode, dtype):
    st = run_case(300_007, 8, stage, dtype, steps=3, mode=mode, double_buffer=(mode in (0, 3)),
                  hyper_kw=dict(weight_decay=0.1))
    st.check()
    assert st.mismatches == 0, st


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_stage0_toy_shape(dtype):
    # the README's toy buffer: psi = 637,824 over 32 simulated ranks
    st = run_case(637_824, 32, 0, dtype, steps=2, double_buffer=False)
    st.check()
    assert st.mismatches == 0, st


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("double_buffer", [True, False])
def test_stage3_layer_buckets(dtype, double_buffer):
    psi, n = 200_003, 4
    pp = (psi + 31) // 32 * 32
    buckets = [(0, 40_000), (40_000, 40_008), (40_008, 123_456), (123_456, 123_457), (123_457, pp)]
    st = run_case(psi, n, 3, dtype, steps=3, buckets=buckets, double_buffer=double_buffer)
    st.check()
    assert st.mismatches == 0, st


@pytest.mark.parametrize("stage", [1, 2, 3])
def test_overflow_skip_and_scale_halving(stage):
    n, psi = 8, 100_000
    inject = [(1, 5, 4_321, INF), (2, 0, 99_999, NAN), (3, 7, 0, NINF)]
    st = run_case(psi, n, stage, "fp16", steps=5, loss_scale=65536.0, sigma=1e-3, inject=inject,
                  buckets=[(0, 50_000), (50_000, 100_032)] if stage == 3 else None)
    st.check()
    assert st.mismatches == 0, st


def test_overflow_in_padding_is_ignored():
    # psi = 1001, N = 4, align 8 -> psi_pad 1024; an inf at index 1010 is padding
    st = run_case(1001, 4, 2, "fp16", steps=2, inject=[(0, 2, 1010, INF)])
    st.check()
    assert st.mismatches == 0


def test_two_pass_stage0_overflow():
    st = run_case(5000, 3, 0, "bf16", steps=3, double_buffer=False, inject=[(1, 1, 17, INF)])
    st.check()
    assert st.mismatches == 0


@pytest.mark.parametrize("stage,mode", [(1, 1), (2, 2), (0, 0), (3, 0)])
def test_clipping_active(stage, mode):
    # max_norm well below the norm: every gradient scaled by max_norm / (norm + 1e-6)
    st = run_case(250_000, 4, stage, "bf16", steps=3, mode=mode, double_buffer=(stage == 3),
                  hyper_kw=dict(max_norm=0.05, weight_decay=0.01))
    st.check()


def test_clip_inactive_when_norm_small():
    st = run_case(250_000, 4, 2, "bf16", steps=2, mode=1, double_buffer=False,
                  hyper_kw=dict(max_norm=1e6))
    st.check()
    assert st.mismatches == 0


@pytest.mark.parametrize("n", [1, 3, 5, 13, 64])
def test_rank_counts_and_nonpow2_scale(n):
    # N * scale not a power of two -> the kernels divide; ragged psi
    st = run_case(20_011, n, 2, "fp16", steps=2, loss_scale=1000.0, sigma=1e-3, mode=3)
    st.check()
    assert st.mismatches == 0


@pytest.mark.parametrize("align", [1, 2])
def test_elementwise_path_when_not_multiple_of_8(align):
    # psi_pad % 8 != 0 takes the element-wise kernels
    st = run_case(1001, 3, 1, "bf16", steps=2, align=align, mode=1, double_buffer=False)
    st.check()
    assert st.mismatches == 0


def test_tiny_hand_case_through_the_abi():
    # psi = 5, N = 2, align = 2: the hand-worked case, lr 2^-6, b = (0.5, 0.75), eps 0
    import oracle as O
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    buf = RankBuffers(5, 2, 1, "fp16", align=2, double_buffer=False)
    assert (buf.psi_pad, buf.shard, buf.offsets, buf.real) == (8, 4, [0, 4], [4, 1])
    p0 = torch.tensor([0.5, 0.25, 0.0, -0.5, 1.0, 0, 0, 0], device="cuda")
    mv, _, _ = buf.state(0)
    mv.copy_(p0)
    buf.params[:, :8].copy_(p0.to(torch.float16))
    buf.grads[0, :8].copy_(torch.tensor([1, 2, -1, 0.5, 4, 0, 0, 0], device="cuda"))
    buf.grads[1, :8].copy_(torch.tensor([3, 2, -3, -2.5, 0, 0, 0, 0], device="cuda"))
    buf.step(B.hyper(lr=2.0 ** -6, beta1=0.5, beta2=0.75, eps=0.0, mode=1))
    s = buf.status()
    assert s["grad_norm"] == 17 ** 0.5 and s["applied"] == 1
    want = [0.484375, 0.234375, 0.015625, -0.484375, 0.984375, 0, 0, 0]
    assert mv.cpu().tolist() == want
    assert buf.params[0, :8].float().cpu().tolist() == want
    assert buf.params[1, :8].float().cpu().tolist() == want
    buf.close()


def test_empty_psi():
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    for stage in (0, 1, 2, 3):
        buf = RankBuffers(0, 4, stage, "bf16")
        assert buf.psi_pad == 0
        buf.step(B.hyper())
        s = buf.status()
        assert s["applied"] == 1 and s["overflow"] == 0 and s["grad_norm"] == 0.0
        buf.close()


def test_errors_are_returned_not_raised_on_device():
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    buf = RankBuffers(1024, 2, 2, "bf16")
    bad = buf.grads.view(-1)[1:]            # 2-byte offset: misaligned
    with pytest.raises(B.ZeroError) as e:
        B.zero_step(buf.h, [bad, buf.grads[1]], buf.param_rows(), buf.master, buf.m, buf.v, B.hyper())
    assert e.value.code == 1 and "aligned" in str(e.value)
    with pytest.raises(B.ZeroError):
        B.zero_gather_bucket(buf.h, 0, 8, buf.params, buf.param_rows())   # not stage 3
    buf.close()
    b3 = RankBuffers(1024, 2, 3, "bf16")
    with pytest.raises(B.ZeroError) as e:
        b3.step(B.hyper())                  # no bucket reduced yet
    assert e.value.code == 5
    g = [torch.zeros(512, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(B.ZeroError) as e:
        b3.reduce_scatter(0, 512, g, B.hyper(max_norm=1.0, mode=3))   # bucketed: no speculative clip
    assert e.value.code == 1
    b3.reduce_scatter(0, 512, g, B.hyper())
    with pytest.raises(B.ZeroError) as e:
        b3.reduce_scatter(256, 768, g, B.hyper())   # overlaps
    assert e.value.code == 5
    b3.close()


def test_state_slot_and_resume():
    # resume from (scale, t, slot) gives the same result as running on
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    torch.manual_seed(0)
    a = RankBuffers(4096, 4, 1, "bf16")
    a.master[:4096].normal_(0, 0.02)
    a.params[:, :4096].copy_(a.master[:4096].to(torch.bfloat16))
    a.grads.normal_(0, 1e-2)
    h = B.hyper()
    a.step(h)
    a.step(h)
    s = a.status()
    assert s["state_slot"] == 0 and s["steps_applied"] == 2
    b = RankBuffers(4096, 4, 1, "bf16")
    b.master.copy_(a.master); b.m.copy_(a.m); b.v.copy_(a.v); b.params.copy_(a.params)
    b.grads.copy_(a.grads)
    b.set_scaler(s["loss_scale"], s["steps_applied"], s["state_slot"])
    a.step(h)
    b.step(h)
    sa, sb = a.status(), b.status()
    assert sa["state_slot"] == sb["state_slot"] == 1
    assert torch.equal(a.master, b.master) and torch.equal(a.params, b.params)
    a.close(); b.close()


@pytest.mark.parametrize("stage", [1, 3])
def test_state_only_16_byte_aligned_takes_the_128_bit_path(stage):
    # master/m/v 16- but not 32-byte aligned: the kernels fall back to 128-bit
    # fp32 accesses; results must equal the 256-bit path bit for bit
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    psi, n = 100_000, 4
    a = RankBuffers(psi, n, stage, "bf16")
    b = RankBuffers(psi, n, stage, "bf16")
    P = a.psi_pad
    torch.manual_seed(3)
    a.master[:psi].normal_(0, 0.02)
    a.m[:psi].normal_(0, 1e-4)
    a.v[:psi].normal_(0, 1e-6).abs_()
    if stage == 3:
        a.params[:P].copy_(a.master[:P].to(torch.bfloat16))
    else:
        a.params[:, :P].copy_(a.master[:P].to(torch.bfloat16))
    b.params.copy_(a.params)
    off = {}
    for name in ("master", "m", "v"):
        big = torch.zeros(2 * P + 8, dtype=torch.float32, device="cuda")
        view = big[4:4 + 2 * P]
        assert view.data_ptr() % 32 == 16
        view.copy_(getattr(a, name))
        off[name] = view
    b.master, b.m, b.v = off["master"], off["m"], off["v"]
    g = torch.randn((n, a.stride), device="cuda").mul_(1e-2).to(torch.bfloat16)
    g[:, psi:] = 0
    h = B.hyper(weight_decay=0.1)
    for buf in (a, b):
        if stage == 3:
            rows = [g[r] for r in range(n)]
            buf.reduce_scatter(0, P, rows, h)
            buf.step(h)
        else:
            buf.step(h, [g[r] for r in range(n)])
    torch.cuda.synchronize()
    assert torch.equal(a.master.view(torch.int32), b.master.view(torch.int32))
    assert torch.equal(a.m.view(torch.int32), b.m.view(torch.int32))
    assert torch.equal(a.v.view(torch.int32), b.v.view(torch.int32))
    assert torch.equal(a.params.view(torch.int16), b.params.view(torch.int16))
    a.close(); b.close()


@pytest.mark.parametrize("stage", [1, 3])
def test_gradients_in_pinned_host_memory(stage):
    # the kernels may read the ranks' gradients straight from pinned host memory
    # (unified addresses); results must equal those from device-resident gradients
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    psi, n = 300_000, 8
    a = RankBuffers(psi, n, stage, "fp16")
    b = RankBuffers(psi, n, stage, "fp16")
    P = a.psi_pad
    torch.manual_seed(4)
    a.master[:psi].normal_(0, 0.02)
    b.master.copy_(a.master)
    q = a.master[:P].to(torch.float16)
    for buf in (a, b):
        if stage == 3:
            buf.params[:P].copy_(q)
        else:
            buf.params[:, :P].copy_(q.unsqueeze(0).expand(n, P))
    g_dev = (torch.randn((n, a.stride), device="cuda") * 1e-2 * 1024).to(torch.float16)
    g_dev[:, psi:] = 0
    g_host = torch.empty((n, a.stride), dtype=torch.float16, pin_memory=True)
    g_host.copy_(g_dev)
    h = B.hyper(weight_decay=0.01)
    for buf, g in ((a, g_dev), (b, g_host)):
        buf.set_scaler(1024.0, 0, 0)
        for _ in range(2):
            if stage == 3:
                buf.reduce_scatter(0, P, [g[r] for r in range(n)], h)
                buf.step(h)
            else:
                buf.step(h, [g[r] for r in range(n)])
    torch.cuda.synchronize()
    assert a.status()["grad_norm"] == b.status()["grad_norm"]
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(a.params.view(torch.int16), b.params.view(torch.int16))
    a.close(); b.close()


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("double_buffer", [True, False])
def test_stage2_reduced_during_backward_constant_buffer(dtype, double_buffer):
    # ZeRO-2 with the reduce-scatter interleaved with backward, one constant-size
    # gradient buffer per rank reused for every bucket; same result as one step
    psi, n = 200_003, 4
    pp = (psi + 31) // 32 * 32
    buckets = [(0, 65_536), (65_536, 65_544), (65_544, 131_072), (131_072, 131_073), (131_073, pp)]
    inject = [(1, 2, 70_000, INF)]
    st = run_case(psi, n, 2, dtype, steps=3, buckets=buckets, double_buffer=double_buffer,
                  loss_scale=256.0, inject=inject, hyper_kw=dict(weight_decay=0.1))
    st.check()
    assert st.mismatches == 0, st


def test_stage2_bucketed_with_clipping_and_errors():
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    st = run_case(100_000, 4, 2, "bf16", steps=2, buckets=[(0, 50_000), (50_000, 100_000)],
                  double_buffer=False, hyper_kw=dict(max_norm=0.05))
    st.check()
    b2 = RankBuffers(1024, 2, 2, "bf16")
    g = [torch.zeros(512, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    b2.reduce_scatter(0, 512, g, B.hyper())
    with pytest.raises(B.ZeroError) as e:
        b2.finish_bucketed_step(B.hyper())      # half the buffer not reduced yet
    assert e.value.code == 5
    with pytest.raises(B.ZeroError) as e:
        b2.reduce_scatter(512, 1024, g, B.hyper(mode=B.ZERO_MODE_TWO_PASS_REREAD))
    assert e.value.code == 1                    # hyper differs within the step
    b2.close()
    b1 = RankBuffers(1024, 2, 1, "bf16")
    with pytest.raises(B.ZeroError):
        B.zero_reduce_scatter_bucket_replicas(b1.h, 0, 512, g, b1.master, b1.m, b1.v, b1.param_rows(), B.hyper())
    b1.close()



@pytest.mark.parametrize("stage", [1, 2])
@pytest.mark.parametrize("max_norm", [0.05, 1e6])
def test_speculative_step_with_clipping(stage, max_norm):
    # one pass assuming no clip; a step whose norm needs clipping is redone
    # from the old slot (max_norm 0.05: every step clips; 1e6: none does)
    inject = [(2, 1, 1234, INF)]
    st = run_case(250_000, 8, stage, "bf16", steps=4, mode=3, double_buffer=True, inject=inject,
                  hyper_kw=dict(max_norm=max_norm, weight_decay=0.1))
    st.check()
    if max_norm > 1:
        assert st.mismatches == 0


@pytest.mark.parametrize("stage", [0, 2, 3])
def test_checkpoint_resume_is_bit_identical(stage, tmp_path):
    # run 4 steps; checkpoint after step 2 (with an overflow at step 2), resume in
    # fresh buffers and run steps 3-4: identical to the uninterrupted run
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300 import checkpoint
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    psi, n = 50_000, 4
    torch.manual_seed(5)
    gs = []
    for k in range(4):
        g = (torch.randn((n, psi), device="cuda") * 1e-2 * 256).to(torch.float16)
        if k == 1:
            g[1, 77] = float("inf")
        gs.append(g)
    h = B.hyper(weight_decay=0.05)

    def make():
        b = RankBuffers(psi, n, stage, "fp16")
        P = b.psi_pad
        mv, _, _ = b.state(0)
        if stage == 0:
            mv.copy_(torch.linspace(-0.1, 0.1, P, device="cuda").expand(n, P))
            b.params[:, :P].copy_(mv.to(torch.float16))
        else:
            mv.copy_(torch.linspace(-0.1, 0.1, P, device="cuda"))
            if stage == 3:
                b.params[:P].copy_(mv.to(torch.float16))
            else:
                b.params[:, :P].copy_(mv.to(torch.float16).unsqueeze(0).expand(n, P))
        b.set_scaler(256.0, 0, 0)
        return b

    def run(b, k):
        rows = torch.zeros((n, b.stride), dtype=torch.float16, device="cuda")
        rows[:, :psi] = gs[k]
        if stage == 3:
            b.reduce_scatter(0, b.psi_pad, [rows[r] for r in range(n)], h)
            b.step(h)
        else:
            b.step(h, [rows[r] for r in range(n)])

    a = make()
    for k in range(4):
        run(a, k)
        if k == 1:
            checkpoint.save(a, str(tmp_path / "ck.pt"))
    b = make()
    checkpoint.load(str(tmp_path / "ck.pt"), b)
    for k in (2, 3):
        run(b, k)
    sa, sb = a.status(), b.status()
    assert (sa["steps_applied"], sa["loss_scale"]) == (sb["steps_applied"], sb["loss_scale"]) == (3, 128.0)
    # the skip count is not part of the resumed state: it restarts with the scaler
    assert (sa["steps_skipped"], sb["steps_skipped"]) == (1, 0)
    for x, y in zip(a.state(sa["state_slot"]), b.state(sb["state_slot"])):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(a.params.view(torch.int16), b.params.view(torch.int16))
    a.close(); b.close()


@pytest.mark.parametrize("stage", [1, 2])
@pytest.mark.parametrize("where", [5, 2_600_000, 7_999_990])
def test_overflow_stops_the_pass_early(stage, where):
    # 8M elements over 4 ranks is about 8.6 waves of the persistent grid: an
    # inf near the start, the middle or the end stops the one-pass step there.
    # The rollback then restores only what the pass may have written, and
    # every element of state and replicas must still match the oracle.
    st = run_case(8_000_011, 4, stage, "fp16", steps=3, mode=3, double_buffer=True, loss_scale=1024.0,
                  sigma=1e-3, inject=[(1, 2, where, INF)])
    st.check()
    assert st.mismatches == 0, st


@pytest.mark.parametrize("psi,bucket", [(6_000_001, 1_000_000), (140_000_003, 36_000_000)])
@pytest.mark.parametrize("stage,mode", [(1, 3), (2, 1), (3, 0), (1, 4)])
def test_norm_is_bitwise_deterministic(stage, mode, psi, bucket):
    _repeat_bitwise(stage, mode, psi, bucket, 8)


@pytest.mark.parametrize("n", [2, 4])
def test_norm_is_bitwise_deterministic_long_rs_chunks(n):
    # with N <= 4 the reduce-scatter takes chunks of up to 16 x 256 vectors;
    # one 140M bucket gives 4273 of them (more than 4096: grouped sums)
    _repeat_bitwise(3, 0, 140_000_003, 140_000_064, n)


def _repeat_bitwise(stage, mode, psi, bucket, n):
    # CTAs take chunks of work in whatever order they reach the counter, but
    # norm partials are formed per chunk, then per group of chunks (launches
    # of more than 4096 chunks: the 140M case), in a fixed order: repeated
    # runs give the same bits.
    import struct
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    g = torch.Generator(device="cuda")
    g.manual_seed(23)
    width = (psi + 8 * n - 1) // (8 * n) * (8 * n)
    grads = (torch.randn((n, width), generator=g, device="cuda") * 1e-2).to(torch.bfloat16)
    master0 = torch.randn(psi, generator=g, device="cuda") * 0.02
    runs = []
    for _ in range(3):
        buf = RankBuffers(psi, n, stage, "bf16", double_buffer=(mode in (0, 3, 4)))
        P = buf.psi_pad
        mv, _, _ = buf.state(0)
        mv[:psi].copy_(master0)
        if stage == 3:
            buf.params[:P].copy_(mv.to(torch.bfloat16))
        else:
            buf.params[:, :P].copy_(mv.to(torch.bfloat16).unsqueeze(0).expand(n, P))
        hyp = B.hyper(max_norm=1e6, mode=mode)
        for _ in range(2):
            if stage == 3:
                for a0 in range(0, P, bucket):
                    b0 = min(P, a0 + bucket)
                    buf.reduce_scatter(a0, b0, [grads[r, a0:b0] for r in range(n)], hyp)
                buf.step(hyp)
            else:
                buf.step(hyp, [grads[r, :P] for r in range(n)])
        s = buf.status()
        m, _, _ = buf.state(s["state_slot"])
        runs.append((struct.pack("<d", s["grad_norm"]), m.cpu().numpy().tobytes()))
        buf.close()
    assert runs[0] == runs[1] == runs[2]


def test_overflow_stop_on_the_grouped_path():
    # 140M elements over 2 ranks: 17.5M vectors, 4273 chunks of 16 x 256 --
    # above the 4096 chunks summed directly, so norm partials go through
    # group tickets.  An inf at 30 % stops the pass with groups left
    # incomplete; the finaliser must reset their tickets (the next steps'
    # norms and every element of state and replicas must still match the
    # oracle).
    st = run_case(140_000_003, 2, 1, "bf16", steps=3, mode=3, double_buffer=True, sigma=1e-3,
                  inject=[(1, 1, 42_000_000, INF)])
    st.check()
    assert st.mismatches == 0, st


@pytest.mark.parametrize("psi,n,buckets", [
    # N = 4: the reduce-scatter's chunks grow to 5 x 256 vectors on the 24M
    # buckets (2344 chunks, summed directly) and the gather runs full
    # 4-vector batches; an 8-element bucket between them, and the last
    # bucket ends in the padding
    (48_000_005, 4, [(0, 24_000_000), (24_000_000, 24_000_008), (24_000_008, 48_000_032)]),
    # N = 2, one 140M bucket: 16 x 256-vector chunks, 4273 of them -- above
    # the 4096 summed directly, so the norm goes through group tickets
    (140_000_003, 2, None),
])
def test_stage3_long_chunks_few_ranks(psi, n, buckets):
    st = run_case(psi, n, 3, "bf16", steps=2, buckets=buckets, double_buffer=True, sigma=1e-3)
    st.check()
    assert st.mismatches == 0, st


@pytest.mark.parametrize("stage,mode", [(1, 3), (2, 1), (3, 0), (1, 4)])
def test_hyper_parameters_changing_between_steps(stage, mode):
    # A learning-rate schedule, and a weight decay that changes once: the
    # one-pass kernels read step scalars that the previous step's finaliser
    # computed for the hyper-parameters it was given, and must compute their
    # own whenever this step's differ.  Step 3 repeats step 2's values (the
    # cached scalars are valid again).
    sched = [dict(lr=1e-3), dict(lr=5e-4), dict(lr=5e-4), dict(lr=2.5e-4, weight_decay=0.05),
             dict(lr=1e-4, weight_decay=0.05)]
    st = run_case(250_003, 4, stage, "bf16", steps=len(sched), mode=mode, double_buffer=True,
                  hyper_steps=sched)
    st.check()
    assert st.mismatches == 0, st


@pytest.mark.parametrize("chunks", [456, 457, 915])
@pytest.mark.parametrize("stage", [1, 3])
def test_chunk_counts_around_the_grid(stage, chunks):
    # The step and reduce-scatter kernels run 3 CTAs of 256 threads per SM
    # (456 on a GB300) and hand out chunks of 256 vectors at these sizes: a
    # CTA's first chunk is its own index, later ones come from the counter.
    # Exactly one chunk per CTA, one chunk more, and two rounds plus three.
    n = 8
    psi = chunks * 256 * 8 - 5   # the last chunk ragged
    inject = [(1, 3, psi - 2, INF)]
    st = run_case(psi, n, stage, "bf16", steps=3, mode=3 if stage == 1 else 0, double_buffer=True,
                  inject=inject, buckets=[(0, (psi + 63) // 64 * 64)] if stage == 3 else None)
    st.check()
    assert st.mismatches == 0, st


@pytest.mark.parametrize("stage", [1, 3])
def test_missing_rank_is_refused(stage):
    # a rank whose gradient (or, stage 3, bucket) row is missing: ZERO_EINVAL
    # before any launch, and the handle stays usable
    from zero_partitioned_mixed_gb300 import _binding as B
    n = 4
    h = B.zero_init_partition(4096, n, stage, B.ZERO_BF16, 8, B.ZERO_F_DOUBLE_BUFFER)
    try:
        P = B.zero_partition_info(h)[0]
        rows = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        rows[2] = None
        master, m, v = (torch.zeros(2 * P, device="cuda") for _ in range(3))
        if stage == 3:
            shard = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
            with pytest.raises(B.ZeroError, match="ZERO_EINVAL"):
                B.zero_reduce_scatter_bucket(h, 0, P, rows, master, m, v, shard, B.hyper())
        else:
            params = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
            with pytest.raises(B.ZeroError, match="ZERO_EINVAL"):
                B.zero_step(h, rows, params, master, m, v, B.hyper())
            rows[2] = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
            B.zero_step(h, rows, params, master, m, v, B.hyper())
            torch.cuda.synchronize()
            assert B.zero_get_status(h)["steps_applied"] == 1
    finally:
        B.zero_destroy(h)


def test_double_buffer_chosen_from_free_memory():
    # double_buffer=None: the second state slot is taken when it fits in
    # free device memory, and not when it cannot (AUTO then runs two-pass)
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    free, _ = torch.cuda.mem_get_info()
    assert RankBuffers.second_slot_fits(1 << 20, 8, 3)
    too_big = int(free // 12) + (1 << 20)      # one state slot alone exceeds free memory
    assert not RankBuffers.second_slot_fits(too_big, 8, 3, alloc_grads=False)
    buf = RankBuffers(1 << 20, 8, 3, "bf16", double_buffer=None)
    assert buf.double_buffer
    buf.close()


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("stage", [1, 3])
def test_cast_at_the_limits_of_the_16_bit_formats(dtype, stage):
    # Zero gradients and zero moments leave the master unchanged (AdamW
    # without decay adds -step * 0 / (0 + eps)), so the replicas or the shard
    # after a step are the cast of the master: values at fp16's overflow
    # threshold (65520 rounds to inf, 65519.996 to 65504), past bf16's
    # largest finite value, in the subnormal ranges, and at ties to even.
    import oracle as O
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    vals = np.array([65504.0, 65519.996, 65520.0, -65520.0, 1e10, -1e38, 3.3895314e38, 3.4e38,
                     2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14 * 1.5, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                     1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1e-40, -1e-45, 0.0, -0.0], np.float32)
    psi, n = 4096, 4
    master = np.resize(vals, psi).astype(np.float32)
    buf = RankBuffers(psi, n, stage, dtype)
    P = buf.psi_pad
    part = O.partition(psi, n, 8)
    ost = O.init_state(stage, dtype, part, master)
    buf.master[:P].copy_(torch.from_numpy(ost.master))
    td = torch.float16 if dtype == "fp16" else torch.bfloat16
    if stage == 3:
        buf.params[:P].copy_(torch.from_numpy(ost.params.view(np.int16)).view(td))
        buf.reduce_scatter(0, P, [torch.zeros(P, dtype=td, device="cuda") for _ in range(n)], B.hyper())
        buf.step(B.hyper())
    else:
        buf.params[:, :P].copy_(torch.from_numpy(ost.params.view(np.int16)).view(td))
        buf.grads.zero_()
        buf.step(B.hyper())
    zeros = np.zeros((n, P), np.uint16)
    ost, res = O.step(ost, zeros, O.Hyper(), [(0, P)] if stage == 3 else None)
    s = buf.status()
    assert s["applied"] and res.applied
    got = buf.params[:P] if stage == 3 else buf.params[:, :P]
    got = got.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ost.params)
    want = O.rne16(master, dtype)
    first = got[:psi] if stage == 3 else got[0, :psi]
    assert np.array_equal(first, want)
    buf.close()


@pytest.mark.parametrize("stage", [1, 3])
@pytest.mark.parametrize("mag", [2.0 ** 70, 2.0 ** -75, "mixed"])
def test_norm_of_gradients_whose_squares_leave_fp32(stage, mag):
    # bf16 gradients reach magnitudes whose fp32 squares overflow (|g| >= 2^64)
    # or fall below the normal range (|g| < 2^-63); the norm is defined in
    # fp64, where every such square is exact.  With clipping on, the norm
    # decides the clip factor and so the update.
    import oracle as O
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    psi, n = 5003, 3
    rng = np.random.default_rng(17 + stage)
    part = O.partition(psi, n, 8)
    P = part.psi_pad
    master = (rng.normal(0, 0.02, psi)).astype(np.float32)
    sign = np.where(rng.random((n, psi)) < 0.5, -1.0, 1.0)
    g = sign * (1.0 + rng.random((n, psi)))
    if mag == "mixed":
        # squares near fp32's top (a group's sum overflows), below its
        # normal range, and ordinary, side by side
        g = g * rng.choice([2.0 ** 62, 2.0 ** -75, 1.0], size=(n, psi))
    else:
        g = g * mag
    gbits = np.zeros((n, P), np.uint16)
    gbits[:, :psi] = O.rne16(g.astype(np.float32), "bf16")
    buf = RankBuffers(psi, n, stage, "bf16")
    ost = O.init_state(stage, "bf16", part, master)
    buf.master[:P].copy_(torch.from_numpy(ost.master))
    dev = torch.from_numpy(gbits.view(np.int16)).cuda().view(torch.bfloat16)
    hb, ho = B.hyper(max_norm=1.0), O.Hyper(max_norm=1.0)
    if stage == 3:
        buf.params[:P].copy_(torch.from_numpy(ost.params.view(np.int16)).view(torch.bfloat16))
        buf.reduce_scatter(0, P, [dev[r] for r in range(n)], hb)
        buf.step(hb)
    else:
        buf.params[:, :P].copy_(torch.from_numpy(ost.params.view(np.int16)).view(torch.bfloat16))
        buf.grads[:, :P].copy_(dev)
        buf.step(hb)
    with np.errstate(over="ignore"):            # fp32 squares of the update may overflow
        ost, res = O.step(ost, gbits, ho, [(0, P)] if stage == 3 else None)
    s = buf.status()
    assert res.applied and s["applied"] and not s["overflow"]
    assert np.isfinite(res.norm) and res.norm > 0
    assert abs(s["grad_norm"] - res.norm) <= 1e-5 * res.norm, (s["grad_norm"], res.norm)
    want_clip = float(res.clip) if res.clip is not None else 1.0
    assert s["clip_coef"] == want_clip
    gm, gmm, gv = buf.state(s["state_slot"])
    for got, want in ((gm, ost.master), (gmm, ost.m), (gv, ost.v)):
        assert int(ulp32(bits32(got), want.view(np.uint32)).max()) <= ULP32
    got16 = bits16(buf.params[:P]) if stage == 3 else bits16(buf.params[:, :P])
    assert int(ulp16(got16, ost.params).max()) <= ULP16
    buf.close()
