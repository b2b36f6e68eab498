"""The staged speculative step (inputs through shared memory by bulk copies)
against the oracle, element by element.

Sizes cover: no full tile (tail only), whole tiles and a tail, more tiles
per CTA than pipeline stages (the stage ring wraps), N from 1 to 19 (the
largest N whose two stages fit), overflow, clipping (the speculative redo),
and the argument checks that refuse the mode.
"""

import numpy as np
import pytest
import torch

from _parity import run_case
from zero_partitioned_mixed_gb300 import _binding as B

pytestmark = pytest.mark.gpu

STAGED = B.ZERO_MODE_SPECULATIVE_STAGED
INF, NAN = float("inf"), float("nan")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("stage", [1, 2])
def test_staged_matches_oracle(stage, dtype):
    st = run_case(300_007, 8, stage, dtype, steps=3, mode=STAGED, hyper_kw=dict(weight_decay=0.1))
    st.check()
    assert st.mismatches == 0, st


@pytest.mark.parametrize("psi,n", [(1000, 4), (2048 * 8, 8), (2048 * 8 + 8, 1), (77_777, 3),
                                   (123_457, 16), (99_991, 19)])
def test_staged_sizes_and_ranks(psi, n):
    st = run_case(psi, n, 1, "bf16", steps=2, mode=STAGED)
    st.check()
    assert st.mismatches == 0, st


def test_staged_ring_wraps():
    # 3,000,017 elements over 4 ranks: ~1465 tiles, ~10 per CTA, 4 stages
    st = run_case(3_000_017, 4, 2, "fp16", steps=2, mode=STAGED, loss_scale=1024.0, sigma=1e-3)
    st.check()
    assert st.mismatches == 0, st


def test_staged_overflow_and_clip():
    inject = [(1, 5, 4_321, INF), (2, 0, 199_999, NAN)]
    st = run_case(200_000, 8, 1, "fp16", steps=4, mode=STAGED, loss_scale=65536.0, sigma=1e-3,
                  inject=inject, hyper_kw=dict(max_norm=0.05))
    st.check()
    assert st.mismatches == 0, st


def test_staged_argument_checks():
    def refused(psi, n, stage, flags, align=8):
        h = B.zero_init_partition(psi, n, stage, B.ZERO_BF16, align, flags)
        P = B.zero_partition_info(h)[0]
        rows = 1 if stage == 3 else n
        grads = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        params = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(rows)]
        k = n if stage == 0 else (2 if flags else 1)
        master, m, v = (torch.zeros(k * P, device="cuda") for _ in range(3))
        try:
            with pytest.raises(B.ZeroError):
                B.zero_step(h, grads, params, master, m, v, B.hyper(mode=STAGED))
        finally:
            B.zero_destroy(h)

    db = B.ZERO_F_DOUBLE_BUFFER
    refused(4096, 20, 1, db)          # two stages do not fit
    refused(4096, 4, 0, 0)            # stage 0
    refused(4096, 4, 1, 0)            # not double-buffered
    refused(1001, 3, 2, db, align=1)  # psi_pad 1002: not a multiple of 8


def test_staged_refuses_host_gradients():
    # pinned host rows are readable by plain loads (the AUTO path takes them)
    # but the staged step's bulk copies read device memory only: refused
    # before any launch
    psi, n = 4096, 2
    h = B.zero_init_partition(psi, n, 1, B.ZERO_BF16, 8, B.ZERO_F_DOUBLE_BUFFER)
    P = B.zero_partition_info(h)[0]
    host = torch.zeros((n, P), dtype=torch.bfloat16, pin_memory=True)
    params = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    master, m, v = (torch.zeros(2 * P, device="cuda") for _ in range(3))
    try:
        with pytest.raises(B.ZeroError, match="device memory"):
            B.zero_step(h, [host[r] for r in range(n)], params, master, m, v, B.hyper(mode=STAGED))
    finally:
        B.zero_destroy(h)


def test_staged_wait_that_runs_out_is_reported_and_changes_nothing():
    # A held tile (no copy issued for CTA 0's second tile) makes that CTA's
    # bounded waits run out after ~2 s.  The step is skipped -- state,
    # replicas, t and the loss scale unchanged -- and the status reports
    # ZERO_ETIMEOUT until zero_set_scaler.  A twin run without the held step
    # ends bit-identical.
    from _parity import bits16, bits32
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    psi, n = 1_000_003, 4
    g = torch.Generator(device="cuda")
    g.manual_seed(17)
    width = (psi + 8 * n - 1) // (8 * n) * (8 * n)        # psi_pad: 16-byte aligned rows
    grads = [(torch.randn((n, width), generator=g, device="cuda") * 1e-2).to(torch.bfloat16) for _ in range(2)]
    master0 = torch.randn(psi, generator=g, device="cuda") * 0.02
    hyp = B.hyper(mode=STAGED, weight_decay=0.01)

    def make():
        b = RankBuffers(psi, n, 1, "bf16", double_buffer=True)
        mv, _, _ = b.state(0)
        mv[:psi].copy_(master0)
        b.params[:, :b.psi_pad].copy_(mv.to(torch.bfloat16).unsqueeze(0).expand(n, b.psi_pad))
        b.set_scaler(256.0, 0, 0)
        return b

    def rows(k, b):
        return [grads[k][r, :b.psi_pad] for r in range(n)]

    twin = make()
    twin.step(hyp, rows(0, twin))
    twin.step(hyp, rows(1, twin))
    torch.cuda.synchronize()

    buf = make()
    buf.step(hyp, rows(0, buf))
    torch.cuda.synchronize()
    slot = buf.status()["state_slot"]
    before = [bits32(x) for x in buf.state(slot)] + [bits16(buf.params)]
    B.zero_debug_hold_staged(buf.h, 1)
    buf.step(hyp, rows(1, buf))
    torch.cuda.synchronize()
    with pytest.raises(B.ZeroError, match="ZERO_ETIMEOUT") as ei:
        B.zero_get_status(buf.h)
    st = ei.value.result
    assert st["error"] == 1 and st["overflow"] == 1 and st["applied"] == 0
    assert st["steps_applied"] == 1 and st["loss_scale"] == 256.0 and st["state_slot"] == slot
    after = [bits32(x) for x in buf.state(slot)] + [bits16(buf.params)]
    for x, y in zip(before, after):
        assert np.array_equal(x, y)
    # clear the error word, run the step again: identical to the twin
    buf.set_scaler(256.0, 1, slot)
    buf.step(hyp, rows(1, buf))
    s1, s2 = buf.status(), twin.status()
    assert s1["steps_applied"] == s2["steps_applied"] == 2 and s1["error"] == 0
    for x, y in zip(buf.state(s1["state_slot"]), twin.state(s2["state_slot"])):
        assert np.array_equal(bits32(x), bits32(y))
    assert np.array_equal(bits16(buf.params), bits16(twin.params))
    buf.close()
    twin.close()
