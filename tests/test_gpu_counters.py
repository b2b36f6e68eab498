"""Exact counters of zero_bytes_moved through the C ABI.

* Model-state bytes per rank and communication elements per step at every
  stage and several (psi, N), against the oracle's closed forms; the
  figures the ZeRO pages print (toy model 10.21 / 2.79 / 1.56 / 0.32 MB at
  N = 32, the 7.5B and 13B tables, the 7.5B communication) from a handle
  alone.
* The resident region of ZeRO-3 persistence (zero_set_persistent), and
  the ZeRO-3 schedule setting it from a persistence layout.
* The algorithmic HBM bytes of every kind of call: the byte sizes of the
  buffers the call must read and write, once each.
"""

import json
import os
from fractions import Fraction
from decimal import Decimal

import pytest
import torch

import oracle as O
from zero_partitioned_mixed_gb300 import _binding as B
from zero_partitioned_mixed_gb300 import persistence as PL
from zero_partitioned_mixed_gb300 import synth as S
from zero_partitioned_mixed_gb300.buffers import RankBuffers
from zero_partitioned_mixed_gb300.schedule import Zero3Schedule

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_tables.json")


def _close_to_printed(value: Fraction, printed: str) -> bool:
    decimals = max(0, -Decimal(printed).as_tuple().exponent)
    return abs(value - Fraction(printed)) <= Fraction(1, 2 * 10 ** decimals)


def _counters(psi, n, stage, align=8):
    h = B.zero_init_partition(psi, n, stage, B.ZERO_BF16, align, 0)
    try:
        return B.zero_bytes_moved(h)
    finally:
        B.zero_destroy(h)


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
@pytest.mark.parametrize("psi,n,align", [(637_824, 32, 8), (5, 2, 2), (1_000, 3, 1), (124_439_808, 8, 8),
                                         (1 << 20, 64, 8), (6_738_415_616, 8, 8)])
def test_counters_every_stage(psi, n, align, stage):
    b = _counters(psi, n, stage, align)
    part = O.partition(psi, n, align)
    P = part.psi_pad
    assert (b["psi"], b["psi_pad"], b["shard"], b["n_ranks"], b["stage"]) == (psi, P, part.shard, n, stage)
    assert b["model_state_bytes_per_rank"] == O.model_state_bytes(P, n, stage)
    assert b["comm_elems_paper"] == O.comm_elems_paper(P, stage)
    assert b["comm_elems_ring"] == O.comm_elems_ring(P, n, stage)
    assert (b["hbm_read_bytes"], b["hbm_write_bytes"], b["hbm_read_total"], b["hbm_write_total"]) == (0, 0, 0, 0)


def test_counters_print_the_page_figures():
    with open(GOLDEN) as f:
        tables = json.load(f)
    checked = 0
    for row in tables["model_state"]:
        if row["n"] > B.ZERO_MAX_RANKS:
            continue        # the library simulates at most 64 ranks
        b = _counters(row["psi"], row["n"], row["stage"], row.get("align", 8))
        assert b["model_state_bytes_per_rank"] == O.model_state_bytes(b["psi_pad"], row["n"], row["stage"])
        assert _close_to_printed(Fraction(b["model_state_bytes_per_rank"], row["unit_bytes"]), row["printed"]), row
        checked += 1
    assert checked >= 20
    # the toy model's row of the simulation README, exactly: 10.21 / 2.79 / 1.56 / 0.32 MB
    got = [round(_counters(637_824, 32, s)["model_state_bytes_per_rank"] / 1e6, 2) for s in range(4)]
    assert got == [10.21, 2.79, 1.56, 0.32]
    for row in tables["comm_paper_bytes"]:
        b = _counters(row["psi"], 8, row["stage"])
        assert _close_to_printed(Fraction(2 * b["comm_elems_paper"], 10 ** 9), row["printed_gb"]), row


@pytest.mark.parametrize("psi,n", [(637_824, 32), (124_439_808, 8), (1_000, 3)])
def test_persistent_region_counters(psi, n):
    h = B.zero_init_partition(psi, n, 3, B.ZERO_BF16, 8, 0)
    P = O.partition(psi, n, 8).psi_pad
    try:
        for p0 in (P, 0, P - 1_000, P // 2 + 3, P - 1):
            B.zero_set_persistent(h, p0)
            b = B.zero_bytes_moved(h)
            pers = P - p0
            assert b["model_state_bytes_per_rank"] == O.model_state_bytes_persistent(P, pers, n)
            assert b["comm_elems_paper"] == O.comm_elems_persistent(P, pers)
            assert b["comm_elems_ring"] == O.comm_elems_ring_persistent(P, pers, n)
        with pytest.raises(B.ZeroError):
            B.zero_set_persistent(h, P + 1)
    finally:
        B.zero_destroy(h)
    h2 = B.zero_init_partition(psi, n, 2, B.ZERO_BF16, 8, 0)
    try:
        with pytest.raises(B.ZeroError):
            B.zero_set_persistent(h2, 0)
    finally:
        B.zero_destroy(h2)


def test_schedule_reports_its_resident_region():
    # GPT-2 small under the guide's threshold of 1e5: the schedule tells the
    # handle where its resident region starts
    n = 8
    lay = PL.persistent_layout(S.gpt2_small_shapes(), 100_000)
    buf = RankBuffers(lay.psi, n, 3, "bf16", double_buffer=False)
    P = buf.psi_pad
    p0 = lay.persistent_from(P)
    Zero3Schedule(buf, PL.tensor_buckets(lay, P), prefetch=False, persistent_from=p0)
    b = buf.bytes_moved()
    assert 0 < P - p0 < P
    assert b["model_state_bytes_per_rank"] == O.model_state_bytes_persistent(P, P - p0, n)
    assert b["comm_elems_paper"] == O.comm_elems_persistent(P, P - p0)
    buf.close()


# ---------------------------------------------------------------- HBM bytes per call
def _nbytes(rows, count, elem):
    return rows * count * elem


class Calls:
    """Runs calls on small buffers and checks each call's HBM counters and the running totals."""

    def __init__(self, buf):
        self.buf = buf
        self.tot = (0, 0)

    def expect(self, read, write):
        b = self.buf.bytes_moved()
        assert (b["hbm_read_bytes"], b["hbm_write_bytes"]) == (read, write)
        self.tot = (self.tot[0] + read, self.tot[1] + write)
        assert (b["hbm_read_total"], b["hbm_write_total"]) == self.tot


PSI, N = 20_000, 4


def _one_shot(stage, mode, double_buffer):
    buf = RankBuffers(PSI, N, stage, "bf16", double_buffer=double_buffer)
    buf.grads[:, :PSI].normal_(0, 1e-2)
    P = buf.psi_pad
    G = _nbytes(N, P, 2)                        # the N gradient rows
    R = _nbytes(N, P, 2)                        # the N 16-bit replicas
    S1 = _nbytes(3, P, 4)                       # master, m, v (one slot)
    W = _nbytes(1, P, 4)                        # the fp32 averaged gradient between two passes
    return buf, P, G, R, S1, W


@pytest.mark.parametrize("stage", [1, 2])
def test_hbm_bytes_one_shot_steps(stage):
    for mode in (B.ZERO_MODE_SPECULATIVE, B.ZERO_MODE_SPECULATIVE_STAGED, B.ZERO_MODE_TWO_PASS_WS,
                 B.ZERO_MODE_TWO_PASS_REREAD):
        spec = mode in (B.ZERO_MODE_SPECULATIVE, B.ZERO_MODE_SPECULATIVE_STAGED)
        buf, P, G, R, S1, W = _one_shot(stage, mode, spec)
        c = Calls(buf)
        for _ in range(2):
            buf.step(B.hyper(mode=mode))
            if spec:           # one pass: gradients and state in, state and replicas out
                c.expect(G + S1, S1 + R)
            elif mode == B.ZERO_MODE_TWO_PASS_WS:   # the averaged gradient goes through the workspace
                c.expect(G + W + S1, W + S1 + R)
            else:              # the second pass reduces the gradients again
                c.expect(2 * G + S1, S1 + R)
        buf.close()


def test_hbm_bytes_stage0():
    buf, P, G, R, S1, W = _one_shot(0, B.ZERO_MODE_AUTO, False)
    c = Calls(buf)
    buf.step(B.hyper())
    c.expect(G + W + N * S1, W + N * S1 + R)   # N full replicas of the state
    buf.close()


@pytest.mark.parametrize("spec", [True, False])
def test_hbm_bytes_zero3_step(spec):
    buf = RankBuffers(PSI, N, 3, "bf16", double_buffer=spec)
    P = buf.psi_pad
    c = Calls(buf)
    hyp = B.hyper(mode=B.ZERO_MODE_AUTO)
    buckets = [(0, 8_008), (8_008, 8_009), (8_009, P)]
    outs = [torch.zeros(P + 8, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    grads = [torch.zeros(P + 8, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    for (a, b) in buckets:
        L = b - a
        buf.gather(a, b, outs)
        c.expect(_nbytes(1, L, 2), _nbytes(N, L, 2))          # the shard's range to N ranks
    for (a, b) in reversed(buckets):
        L = b - a
        buf.gather(a, b, outs)
        c.expect(_nbytes(1, L, 2), _nbytes(N, L, 2))
        buf.reduce_scatter(a, b, grads, hyp)
        if spec:   # N gradient rows and the state in; the state and the 16-bit shard out
            c.expect(_nbytes(N, L, 2) + _nbytes(3, L, 4), _nbytes(3, L, 4) + _nbytes(1, L, 2))
        else:      # N gradient rows in; the averaged gradient out to the workspace
            c.expect(_nbytes(N, L, 2), _nbytes(1, L, 4))
    buf.step(hyp)
    if spec:
        c.expect(0, 0)                                          # the update was fused into the buckets
    else:
        c.expect(_nbytes(1, P, 4) + _nbytes(3, P, 4), _nbytes(3, P, 4) + _nbytes(1, P, 2))
    buf.close()


@pytest.mark.parametrize("spec", [True, False])
def test_hbm_bytes_zero2_buckets(spec):
    buf = RankBuffers(PSI, N, 2, "bf16", double_buffer=spec)
    P = buf.psi_pad
    c = Calls(buf)
    hyp = B.hyper()
    cb = [torch.zeros(P + 8, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    for (a, b) in [(12_000, P), (0, 12_000)]:
        L = b - a
        buf.reduce_scatter(a, b, cb, hyp)
        if spec:   # the bucket's update and its all-gather into the N replicas are fused here
            c.expect(_nbytes(N, L, 2) + _nbytes(3, L, 4), _nbytes(3, L, 4) + _nbytes(N, L, 2))
        else:
            c.expect(_nbytes(N, L, 2), _nbytes(1, L, 4))
    buf.finish_bucketed_step(hyp)
    if spec:
        c.expect(0, 0)
    else:
        c.expect(_nbytes(1, P, 4) + _nbytes(3, P, 4), _nbytes(3, P, 4) + _nbytes(N, P, 2))
    buf.close()


@pytest.mark.parametrize("bits", [8, 4])
def test_hbm_bytes_zeropp(bits):
    buf = RankBuffers(PSI, N, 3, "bf16", double_buffer=True)
    P = buf.psi_pad
    c = Calls(buf)
    a, b = 0, P
    L = b - a
    nb = (L + O.Q_BLOCK - 1) // O.Q_BLOCK
    codes = [torch.zeros(L + 16, dtype=torch.uint8, device="cuda") for _ in range(N)]
    scales = [torch.zeros(2 * nb, dtype=torch.float32, device="cuda") for _ in range(N)]
    B.zero_gather_bucket_q8(buf.h, a, b, buf.params, codes, scales)
    c.expect(_nbytes(1, L, 2), N * (L + 8 * nb))              # INT8 codes and a (scale, lo) pair per block
    B.zero_reduce_scatter_bucket_q(buf.h, a, b, bits, codes, scales, buf.master, buf.m, buf.v, buf.params,
                                   B.hyper())
    c.expect(N * (L * bits // 8 + 8 * nb) + _nbytes(3, L, 4), _nbytes(3, L, 4) + _nbytes(1, L, 2))
    buf.step(B.hyper())
    c.expect(0, 0)
    buf.close()


@pytest.mark.parametrize("spec", [True, False])
def test_hbm_bytes_fused_reduce_scatter_gather(spec):
    # one call: the reduce-scatter of one bucket and the gather of another,
    # counted as the two parts' bytes together (one launch when 8-aligned,
    # two calls otherwise)
    buf = RankBuffers(PSI, N, 3, "bf16", double_buffer=spec)
    P = buf.psi_pad
    c = Calls(buf)
    hyp = B.hyper()
    grads = [torch.zeros(P + 8, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    outs = [torch.zeros(P + 8, dtype=torch.bfloat16, device="cuda") for _ in range(N)]

    def rs_bytes(L):
        if spec:
            return _nbytes(N, L, 2) + _nbytes(3, L, 4), _nbytes(3, L, 4) + _nbytes(1, L, 2)
        return _nbytes(N, L, 2), _nbytes(1, L, 4)

    for (a, b), (ga, gb) in (((12_000, P), (8_000, 12_000)), ((8_001, 12_000), (0, 8_001)), ((0, 8_001), (0, 0))):
        buf.reduce_scatter_gather(a, b, grads, hyp, ga, gb, outs)
        r, w = rs_bytes(b - a)
        c.expect(r + _nbytes(1, gb - ga, 2), w + _nbytes(N, gb - ga, 2))
    buf.step(hyp)
    if spec:
        c.expect(0, 0)
    else:
        c.expect(_nbytes(1, P, 4) + _nbytes(3, P, 4), _nbytes(3, P, 4) + _nbytes(1, P, 2))
    buf.close()
