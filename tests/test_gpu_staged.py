"""The staged speculative step (inputs through shared memory by bulk copies)
against the oracle, element by element.

Sizes cover: no full tile (tail only), whole tiles and a tail, more tiles
per CTA than pipeline stages (the stage ring wraps), N from 1 to 19 (the
largest N whose two stages fit), overflow, clipping (the speculative redo),
and the argument checks that refuse the mode.
"""

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
