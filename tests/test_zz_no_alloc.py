"""zero_step_noalloc: the step for callers that cannot allocate device memory.

Such callers (code whose framework's caching allocator owns the device
memory, code under a fixed memory budget) cannot create a handle, because
zero_init_partition allocates a workspace.  zero_step_noalloc keeps all of
its scratch in a static device array instead.  These tests call it through
the C ABI and check that two calls in a row give what the handle-based
zero_step gives on the same inputs, and what the oracle computes, within the
tolerances of the other parity tests; that a call leaves the device's free
memory unchanged; and that a result pointer the GPU cannot write is refused
before anything runs.  The file is named so that pytest collects it last.
"""

import pytest

from zero_partitioned_mixed_gb300 import _binding as B


def test_noalloc_rejects_sizes_beyond_its_static_scratch():
    B.load_library()
    h = B.hyper()
    cap = 1 << 22
    with pytest.raises(B.ZeroError) as e:
        B.zero_step_noalloc(cap + 1, 2, 1, B.ZERO_BF16, 8, None, None, None, None, None, h, 1.0, 0, None, 0)
    assert e.value.code == 1 and "static scratch" in str(e.value)
    # psi itself fits but its padding to a multiple of N*align does not
    with pytest.raises(B.ZeroError) as e:
        B.zero_step_noalloc(cap - 1, 3, 2, B.ZERO_FP16, 8, None, None, None, None, None, h, 1.0, 0, None, 0)
    assert e.value.code == 1 and "psi_pad" in str(e.value)
    with pytest.raises(B.ZeroError) as e:
        B.zero_step_noalloc(100, 2, 3, B.ZERO_FP16, 8, None, None, None, None, None, h, 1.0, 0, None, 0)
    assert e.value.code == 1


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,max_norm,inject", [("bf16", 0.0, False), ("fp16", 0.05, False),
                                                    ("fp16", 0.0, True)])
def test_noalloc_matches_zero_step_on_two_calls(dtype, max_norm, inject):
    import numpy as np
    import torch

    from _parity import NORM_RTOL, ULP16, ULP32, bits16, bits32, ulp16, ulp32
    from zero_partitioned_mixed_gb300 import synth as S
    from zero_partitioned_mixed_gb300.buffers import RankBuffers

    import oracle as O

    psi, n, stage, align = 1_000_003, 8, 2, 8
    zdt = B.ZERO_BF16 if dtype == "bf16" else B.ZERO_FP16
    td = S.torch_dtype(dtype)
    loss_scale = 1024.0
    # the handle-based path, two-pass with its workspace
    ref = RankBuffers(psi, n, stage, dtype, align=align, double_buffer=False)
    P = ref.psi_pad
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    ref.master[:psi].copy_(torch.randn(psi, generator=g, device="cuda") * 0.02)
    ref.m[:psi].copy_(torch.randn(psi, generator=g, device="cuda") * 1e-4)
    ref.v[:psi].copy_((torch.randn(psi, generator=g, device="cuda") * 1e-6).abs())
    ref.params[:, :P].copy_(ref.master[:P].to(td).unsqueeze(0).expand(n, P))
    # the caller-owned buffers of the no-alloc path: same starting values
    master, m, v = ref.master.clone(), ref.m.clone(), ref.v.clone()
    params = ref.params.clone()
    result = torch.zeros(64, dtype=torch.uint8, device="cuda")
    hyp = B.hyper(lr=1e-3, weight_decay=0.1, max_norm=max_norm, mode=B.ZERO_MODE_TWO_PASS_WS)
    ref.set_scaler(loss_scale, 0, 0)
    scale, t = loss_scale, 0
    # the oracle, from the same starting state
    part = O.partition(psi, n, align)
    ost = O.init_state(stage, dtype, part, ref.master[:psi].cpu().numpy(), ref.m[:psi].cpu().numpy(),
                       ref.v[:psi].cpu().numpy(), loss_scale=loss_scale)
    oh = O.Hyper(lr=1e-3, weight_decay=0.1, max_norm=max_norm)
    for k in range(2):
        grads = torch.zeros((n, ref.stride), dtype=td, device="cuda")
        grads[:, :psi] = (torch.randn((n, psi), generator=g, device="cuda") * 1e-2 * scale).to(td)
        if inject and k == 0:
            grads[3, 12345] = float("inf")
        rows = [grads[r] for r in range(n)]
        ref.step(hyp, rows)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        B.zero_step_noalloc(psi, n, stage, zdt, align, rows, [params[r] for r in range(n)],
                            master, m, v, hyp, scale, t, result)
        torch.cuda.synchronize()
        if k == 1:      # after the first call has loaded the kernels: nothing allocated
            assert torch.cuda.mem_get_info()[0] == free0
        ost, ores = O.step(ost, bits16(grads[:, :P]), oh)
        want = ref.status()
        got = B.result_from_device(result)
        for key in ("overflow", "applied", "steps_applied", "loss_scale", "clip_coef"):
            assert got[key] == want[key], (k, key, got, want)
        assert got["steps_skipped"] == got["overflow"]   # counts this call only
        if want["applied"]:
            assert abs(got["grad_norm"] - want["grad_norm"]) <= NORM_RTOL * want["grad_norm"]
        for a, b in ((master, ref.master), (m, ref.m), (v, ref.v)):
            assert int(ulp32(bits32(a[:P]), bits32(b[:P])).max()) <= ULP32
        assert int(ulp16(bits16(params[:, :P]), bits16(ref.params[:, :P])).max()) <= ULP16
        # and against the oracle directly
        assert bool(got["overflow"]) == ores.overflow and got["steps_applied"] == ost.t
        assert got["loss_scale"] == np.float32(ost.loss_scale)
        if ores.applied:
            assert abs(got["grad_norm"] - ores.norm) <= NORM_RTOL * ores.norm
            assert got["clip_coef"] == (float(ores.clip) if ores.clip is not None else 1.0)
        for a, b in ((master, ost.master), (m, ost.m), (v, ost.v)):
            assert int(ulp32(bits32(a[:P]), b.view(np.uint32)).max()) <= ULP32
        assert int(ulp16(bits16(params[:, :P]), ost.params).max()) <= ULP16
        scale, t = got["loss_scale"], got["steps_applied"]
    assert t == (1 if inject else 2)
    ref.close()


@pytest.mark.gpu
def test_noalloc_refuses_a_result_the_gpu_cannot_write():
    # pageable host memory for the result: refused before any launch (the
    # gradients are missing too, so had the result passed, that check would
    # refuse the call instead, with another message, and still launch nothing)
    import ctypes
    import torch

    host = (ctypes.c_uint64 * 8)()
    torch.cuda.init()
    with pytest.raises(B.ZeroError) as e:
        B.zero_step_noalloc(1000, 2, 1, B.ZERO_BF16, 8, None, None, None, None, None, B.hyper(), 1.0, 0,
                            ctypes.addressof(host), 0)
    assert e.value.code == 1 and "result must be device, managed or pinned host memory" in str(e.value)
