"""zero_reduce_scatter_gather_bucket against the oracle: ZeRO-3 steps whose
backward pass gathers each next bucket in the same call as the current
bucket's reduce-scatter.  Every gathered row, the state, the shard, the norm
and the flags are compared with the oracle element by element.  Covers the
one-launch path (8-aligned buckets), the two-call path (unaligned buckets),
both modes, overflow, launches whose reduce-scatter part has fewer chunks
than the grid or more than the directly summed ones, and the refusals."""

import pytest
import torch

from _parity import run_case
from zero_partitioned_mixed_gb300 import _binding as B
from zero_partitioned_mixed_gb300.buffers import RankBuffers

pytestmark = pytest.mark.gpu

INF = float("inf")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("double_buffer", [True, False])
@pytest.mark.parametrize("n", [1, 2, 3, 8])
def test_fused_backward_matches_oracle(dtype, double_buffer, n):
    psi = 200_003
    pp = (psi + 8 * n - 1) // (8 * n) * (8 * n)
    # 8-aligned buckets (one launch each) and unaligned ones (two calls)
    buckets = [(0, 40_000), (40_000, 40_008), (40_008, 123_456), (123_456, 123_457), (123_457, pp)]
    st = run_case(psi, n, 3, dtype, steps=3, buckets=buckets, double_buffer=double_buffer, fused=True)
    st.check()
    assert st.mismatches == 0, st


def test_fused_backward_with_overflow_and_scale():
    psi, n = 300_007, 4
    pp = (psi + 31) // 32 * 32
    buckets = [(0, 100_000), (100_000, 200_000), (200_000, pp)]
    st = run_case(psi, n, 3, "fp16", steps=4, buckets=buckets, double_buffer=True, loss_scale=1024.0,
                  sigma=1e-3, inject=[(1, 2, 150_001, INF)], fused=True)
    st.check()
    assert st.mismatches == 0, st


@pytest.mark.parametrize("psi,buckets", [
    # backward starts with the 64-element last bucket, whose reduce-scatter
    # carries the gather of a 999,936-element bucket: most CTAs start on gather chunks
    (1_000_000, [(0, 999_936), (999_936, 1_000_000)]),
    # a 140M-element reduce-scatter (4272 chunks of 16 x 256 vectors at N = 2:
    # the grouped norm partials) carrying an 8000-element gather
    (140_000_000, [(0, 8_000), (8_000, 140_000_000)]),
])
def test_fused_chunk_geometry(psi, buckets):
    st = run_case(psi, 2, 3, "bf16", steps=2, buckets=buckets, double_buffer=True, sigma=1e-3, fused=True)
    st.check()
    assert st.mismatches == 0, st


def test_fused_refusals():
    psi, n = 10_000, 4
    buf = RankBuffers(psi, n, 3, "bf16")
    P = buf.psi_pad
    hyp = B.hyper()
    grads = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    outs = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(n)]

    def refused(*args, msg):
        with pytest.raises(B.ZeroError) as e:
            buf.reduce_scatter_gather(*args)
        assert e.value.code == 1 and msg in str(e.value), str(e.value)

    refused(0, 4_000, grads, hyp, 3_992, 8_000, outs, msg="overlaps the reduce-scattered one")
    refused(0, 4_000, grads, hyp, 4_000, P + 8, outs, msg="0 <= ga <= gb <= psi_pad")
    # an output row that is one of the gradient rows
    refused(0, 4_000, grads, hyp, 4_000, 8_000, [grads[1]] + outs[1:], msg="overlaps a gradient row")
    # an output row inside the shard, or inside the fp32 state
    refused(0, 4_000, grads, hyp, 4_000, 8_000, [buf.params[4_000:]] + outs[1:], msg="overlaps the 16-bit shard")
    refused(0, 4_000, grads, hyp, 4_000, 8_000, outs[:3] + [buf.m.view(torch.bfloat16)[16:]],
            msg="overlaps master, m or v")
    # nothing was reduced: a whole step still goes through
    for (a, b), (ga, gb) in (((0, 4_000), (4_000, 8_000)), ((4_000, 8_000), (8_000, P)), ((8_000, P), (0, 0))):
        buf.reduce_scatter_gather(a, b, grads, hyp, ga, gb, outs)
    buf.finish_bucketed_step(hyp)
    assert buf.status()["applied"] == 1
    buf.close()
    b2 = RankBuffers(psi, n, 2, "bf16")
    with pytest.raises(B.ZeroError):
        B.zero_reduce_scatter_gather_bucket(b2.h, 0, 8, grads, b2.master, b2.m, b2.v, b2.params[0], hyp, 8, 16,
                                            outs)
    b2.close()


@pytest.mark.parametrize("stage,fused", [(3, False), (3, True), (2, False)])
def test_bucketed_steps_when_psi_pad_is_not_a_multiple_of_8(stage, fused):
    # N = 5 and align 2 give psi_pad = 31,910: the second state slot starts
    # off an 8-float boundary, so the 8-aligned buckets must still take the
    # element-wise path (an 8-wide access there would be misaligned)
    psi, n = 31_910, 5
    buckets = [(0, 13_520), (13_520, 16_280), (16_280, 17_952), (17_952, 24_864), (24_864, 31_910)]
    st = run_case(psi, n, stage, "bf16", steps=3, align=2, double_buffer=True, loss_scale=65536.0,
                  buckets=buckets, fused=fused)
    st.check()
    assert st.mismatches == 0, st
