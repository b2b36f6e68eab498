"""Pins for the CPU oracle: each test checks it against something other than
itself -- numbers the ZeRO pages print, closed forms, IEEE-defined
rounding vectors, brute force on tiny inputs and a high-precision
re-evaluation of Adam -- so that a dropped term, a wrong sign or index, or
a transposed operand in the oracle fails at least one of them."""

import json
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_tables.json")


def _tables():
    with open(GOLDEN) as f:
        return json.load(f)


def _close_to_printed(value: Fraction, printed: str) -> bool:
    d = Decimal(printed)
    decimals = max(0, -d.as_tuple().exponent)
    half = Fraction(1, 2 * 10 ** decimals)
    return abs(value - Fraction(printed)) <= half


# ---------------------------------------------------------------- partition
@pytest.mark.parametrize("align", [1, 2, 8])
@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_partition_brute_force(n, align):
    for psi in range(0, 65):
        p = O.partition(psi, n, align)
        unit = n * align
        # smallest multiple of N*align that is >= psi, found by search
        want = 0
        while want < psi:
            want += unit
        assert p.psi_pad == want
        assert p.shard * n == p.psi_pad
        owner = [-1] * p.psi_pad
        for r, (off, real) in enumerate(zip(p.offsets, p.real)):
            assert off == r * p.shard
            for i in range(off, off + p.shard):
                assert owner[i] == -1
                owner[i] = r
            assert real == sum(1 for i in range(off, off + p.shard) if i < psi)
        assert all(o >= 0 for o in owner)
        assert sum(p.real) == psi


def test_partition_toy_numbers():
    p = O.partition(637824, 32, 8)
    assert (p.psi_pad, p.shard) == (637952, 19936)
    assert p.real[-1] == 637824 - 31 * 19936 == 19808


# ---------------------------------------------------------------- accounting
def test_model_state_tables_printed_on_pages():
    for row in _tables()["model_state"]:
        psi = row["psi"]
        if row.get("padded"):
            psi = O.partition(psi, row["n"], row["align"]).psi_pad
        b = O.model_state_bytes(psi, row["n"], row["stage"])
        assert _close_to_printed(Fraction(b, row["unit_bytes"]), row["printed"]), row


def test_unpadded_toy_would_not_print_156():
    # The padding reading: without it ZeRO-2 at N = 32 would print 1.55 MB.
    b = O.model_state_bytes(637824, 32, 2)
    assert not _close_to_printed(Fraction(b, 10 ** 6), "1.56")


def test_bytes_per_param_at_32():
    for row in _tables()["bytes_per_param_at_n32"]:
        b = O.model_state_bytes(32 * 1000, 32, row["stage"])
        assert _close_to_printed(Fraction(b, 32 * 1000), row["printed"]), row


def test_table1_model_sizes_fit_32gb():
    for row in _tables()["fits_32gb_table1"]:
        assert O.model_state_bytes(row["psi"], row["n"], row["stage"]) <= row["capacity_bytes"]


def test_exact_formulas_on_integers():
    for n in (1, 2, 4, 8, 64):
        psi = n * 1000
        assert O.model_state_bytes(psi, n, 0) == 16 * psi
        assert O.model_state_bytes(psi, n, 1) * n == 4 * psi * n + 12 * psi
        assert O.model_state_bytes(psi, n, 2) * n == 2 * psi * n + 14 * psi
        assert O.model_state_bytes(psi, n, 3) * n == 16 * psi
    # at N = 1 every stage holds everything
    assert len({O.model_state_bytes(800, 1, s) for s in range(4)}) == 1


def test_comm_ring_printed():
    for row in _tables()["comm_ring_per_psi"]:
        n, psi = row["n"], row["n"] * 10 ** 6
        if row["model"] == "ring":
            e = O.comm_elems_ring(psi, n, row["stage"])
        else:
            e = O.comm_elems_ring_allreduce_zero1(psi, n)
        assert _close_to_printed(Fraction(e, psi), row["printed"]), row


def test_comm_paper_printed():
    for row in _tables()["comm_paper_bytes"]:
        e = O.comm_elems_paper(row["psi"], row["stage"])
        gb = Fraction(2 * e, 10 ** 9)
        assert _close_to_printed(gb, row["printed_gb"])
        assert _close_to_printed(gb / 50, row["printed_s_at_50gbs"])
    # 1.5x for stage 3 against the DP baseline (ZeRO summary Sec. 7)
    assert Fraction(O.comm_elems_paper(10, 3), O.comm_elems_paper(10, 0)) == Fraction(3, 2)


def test_ring_stage3_cell_is_the_documented_gap():
    row = _tables()["not_reproduced"][0]
    e = O.comm_elems_ring(32 * 10 ** 6, 32, 3)
    assert not _close_to_printed(Fraction(e, 32 * 10 ** 6), "2.89"), row
    assert Fraction(e, 32 * 10 ** 6) == Fraction(93, 32)


# ---------------------------------------------------------------- 16-bit rounding
FP16_VECTORS = [
    # (fp32 value, expected binary16 bits), from the IEEE 754 binary16 layout
    (1.0, 0x3C00), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
    (65504.0, 0x7BFF), (65519.99609375, 0x7BFF), (65520.0, 0x7C00),
    (1e10, 0x7C00), (-1e10, 0xFC00),
    (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000),            # tie -> even (zero)
    (3 * 2.0 ** -25, 0x0002),                              # tie -> even (2 ulp)
    (1 + 2.0 ** -11, 0x3C00), (1 + 3 * 2.0 ** -11, 0x3C02),  # ties
    (1 + 2.0 ** -11 + 2.0 ** -20, 0x3C01),                 # above the tie
    (2.0 ** -14, 0x0400), (2.0 ** -14 - 2.0 ** -24, 0x03FF),
]
BF16_VECTORS = [
    (1.0, 0x3F80), (-1.0, 0xBF80), (0.0, 0x0000), (-0.0, 0x8000),
    (1 + 2.0 ** -8, 0x3F80), (1 + 3 * 2.0 ** -8, 0x3F82), (1 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),
    (3.4028234663852886e38, 0x7F80),                       # above bf16 max -> inf
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),
    (2.0 ** -149, 0x0000), (2.0 ** -133, 0x0001),
    (float("inf"), 0x7F80), (float("-inf"), 0xFF80),
]


def test_rne16_fp16_vectors():
    x = np.array([v for v, _ in FP16_VECTORS], np.float32)
    got = O.rne16(x, O.FP16)
    assert [int(b) for b in got] == [b for _, b in FP16_VECTORS]


def test_rne16_bf16_vectors():
    x = np.array([v for v, _ in BF16_VECTORS], np.float32)
    got = O.rne16(x, O.BF16)
    assert [int(b) for b in got] == [b for _, b in BF16_VECTORS]
    nan = O.rne16(np.array([np.nan], np.float32), O.BF16)[0]
    assert (int(nan) & 0x7F80) == 0x7F80 and (int(nan) & 0x007F) != 0


def test_widen16_exact_roundtrip():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    for dt in (O.FP16, O.BF16):
        w = O.widen16(bits, dt)
        finite = np.isfinite(w)
        back = O.rne16(w[finite], dt)
        assert np.array_equal(back, bits[finite])
    # spot values from the formats' definitions
    assert O.widen16(np.array([0x3C00], np.uint16), O.FP16)[0] == 1.0
    assert O.widen16(np.array([0x0001], np.uint16), O.FP16)[0] == 2.0 ** -24
    assert O.widen16(np.array([0x3F80], np.uint16), O.BF16)[0] == 1.0


# ---------------------------------------------------------------- hand-worked tiny case
def _bits(vals, dt):
    return O.rne16(np.array(vals, np.float32), dt)


def _tiny_grads(dt):
    g0 = [1, 2, -1, 0.5, 4, 0, 0, 0]
    g1 = [3, 2, -3, -2.5, 0, 0, 0, 0]
    return np.stack([_bits(g0, dt), _bits(g1, dt)])


@pytest.mark.parametrize("dt", [O.FP16, O.BF16])
@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_tiny_case_by_hand(stage, dt):
    # psi = 5, N = 2, align = 2: psi_pad = 8, shard 4, offsets [0, 4], real [4, 1].
    # sums [4, 4, -4, -2, 4] -> g_hat = sums / 2 = [2, 2, -2, -1, 2]; |g_hat|^2 = 17.
    # Adam t = 1, lr = 2^-6, b1 = 0.5, b2 = 0.75, eps = 0: every update is
    # lr * sign(g_hat), all exact in fp32 and in both 16-bit formats.
    part = O.partition(5, 2, 2)
    assert (part.psi_pad, part.shard, part.offsets, part.real) == (8, 4, (0, 4), (4, 1))
    h = O.Hyper(lr=2.0 ** -6, beta1=0.5, beta2=0.75, eps=0.0)
    p0 = [0.5, 0.25, 0.0, -0.5, 1.0]
    st = O.init_state(stage, dt, part, np.array(p0, np.float32))
    buckets = [(0, 3), (3, 8)] if stage == 3 else None
    new, res = O.step(st, _tiny_grads(dt), h, buckets)
    want = np.array([0.484375, 0.234375, 0.015625, -0.484375, 0.984375], np.float32)
    assert res.applied and not res.overflow
    assert res.norm == math.sqrt(17.0)
    master = new.master[0] if stage == 0 else new.master
    assert np.array_equal(master[:5], want)
    assert np.all(master[5:] == 0)
    qs = new.params if stage == 3 else new.params[0]
    assert np.array_equal(O.widen16(qs[:5], dt), want)
    if stage != 3:
        assert np.array_equal(new.params[0], new.params[1])
    else:
        # the gathers hand every rank the owners' 16-bit values of the bucket
        before = O.rne16(np.array(p0 + [0, 0, 0], np.float32), dt)
        assert np.array_equal(res.gathered_fwd[0][1], before[0:3])
        assert np.array_equal(res.gathered_bwd[1][0], before[3:8])


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_padding_gradients_are_ignored(stage):
    # The padding [psi, psi_pad) of every gradient row is read as zero and
    # the padding of master, m, v and the 16-bit copies stays zero: finite
    # garbage there changes nothing (the tiny case, psi = 5 of psi_pad = 8).
    part = O.partition(5, 2, 2)
    h = O.Hyper(lr=2.0 ** -6, beta1=0.5, beta2=0.75, eps=0.0)
    p0 = np.array([0.5, 0.25, 0.0, -0.5, 1.0], np.float32)
    buckets = [(0, 3), (3, 8)] if stage == 3 else None
    clean = _tiny_grads(O.FP16)
    dirty = clean.copy()
    dirty[:, 5:] = _bits([0.75, -3.0, 1.5], O.FP16)
    a, _ = O.step(O.init_state(stage, O.FP16, part, p0), clean, h, buckets)
    b, _ = O.step(O.init_state(stage, O.FP16, part, p0), dirty, h, buckets)
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v), (a.params, b.params)):
        assert x.tobytes() == y.tobytes()
    mb = b.master if stage != 0 else b.master[0]
    assert np.all(mb[5:8] == 0) and np.all((b.m if stage != 0 else b.m[0])[5:8] == 0)
    qb = b.params if stage == 3 else b.params[0]
    assert np.all(qb[5:8] == 0)


@pytest.mark.parametrize("stage", [1, 2, 3])
def test_loss_scale_divides_out(stage):
    # Loss scaling: gradients computed at scale 2^10 and unscaled by 2^10 give
    # the hand-worked result exactly (powers of two: every product is exact).
    part = O.partition(5, 2, 2)
    h = O.Hyper(lr=2.0 ** -6, beta1=0.5, beta2=0.75, eps=0.0)
    p0 = [0.5, 0.25, 0.0, -0.5, 1.0]
    st = O.init_state(stage, O.BF16, part, np.array(p0, np.float32), loss_scale=1024.0)
    g = np.stack([_bits(np.array([1, 2, -1, 0.5, 4, 0, 0, 0]) * 1024, O.BF16),
                  _bits(np.array([3, 2, -3, -2.5, 0, 0, 0, 0]) * 1024, O.BF16)])
    new, res = O.step(st, g, h, [(0, 8)] if stage == 3 else None)
    assert res.norm == math.sqrt(17.0)
    want = np.array([0.484375, 0.234375, 0.015625, -0.484375, 0.984375], np.float32)
    assert np.array_equal(new.master[:5], want)
    assert new.loss_scale == 1024.0


# ---------------------------------------------------------------- equivalence
def _random_case(seed, psi, n, dt, scale=1.0, sigma=1e-2):
    rng = np.random.default_rng(seed)
    part = O.partition(psi, n, 8)
    master = rng.normal(0, 0.02, psi).astype(np.float32)
    m = rng.normal(0, 1e-4, psi).astype(np.float32)
    v = np.abs(rng.normal(0, 1e-6, psi)).astype(np.float32)
    grads = []
    for _ in range(3):
        g = np.zeros((n, part.psi_pad), np.float32)
        g[:, :psi] = rng.normal(0, sigma, (n, psi)) * scale
        grads.append(O.rne16(g, dt))
    return part, master, m, v, grads


@pytest.mark.parametrize("dt", [O.FP16, O.BF16])
def test_all_stages_identical(dt):
    # "zero-stages-simulation" README: every stage produced identical trained weights.
    n, psi = 4, 1001
    part, master, m, v, grads = _random_case(1, psi, n, dt)
    h = O.Hyper(lr=1e-3, weight_decay=0.1, max_norm=0.05)
    finals = []
    for stage in range(4):
        st = O.init_state(stage, dt, part, master, m, v)
        for k in range(3):
            buckets = [(0, 96), (96, 640), (640, part.psi_pad)] if stage == 3 else None
            st, res = O.step(st, grads[k], h, buckets)
            assert res.applied
        finals.append(st)
    ref = finals[1]
    for st in finals:
        mm = st.master[0] if st.stage == 0 else st.master
        assert np.array_equal(mm.view(np.uint32), ref.master.view(np.uint32))
        q = st.params if st.stage == 3 else st.params[0]
        assert np.array_equal(q, ref.params[0])
    s0 = finals[0]
    for r in range(n):
        assert np.array_equal(s0.master[r], s0.master[0])
        assert np.array_equal(s0.m[r], s0.m[0])
        assert np.array_equal(s0.params[r], s0.params[0])


def test_all_reduce_is_reduce_scatter_then_all_gather():
    # CMU 11-868 notes, exercise 3: all-reduce == reduce-scatter + all-gather.
    rng = np.random.default_rng(7)
    part = O.partition(77, 4, 2)
    g = [rng.normal(0, 1, part.psi_pad).astype(np.float32) for _ in range(4)]
    ar = O.all_reduce_mean(g, 4, 8.0)
    ag = O.all_gather(O.reduce_scatter_mean(g, part, 8.0))
    for r in range(4):
        assert np.array_equal(ar[r], ag)


def test_replicas_equal_cast_of_master():
    part, master, m, v, grads = _random_case(3, 333, 3, O.BF16)
    st = O.init_state(2, O.BF16, part, master, m, v)
    for k in range(3):
        st, _ = O.step(st, grads[k], O.Hyper())
        for r in range(3):
            assert np.array_equal(st.params[r], O.rne16(st.master, O.BF16))


# ---------------------------------------------------------------- Adam closed forms
def test_adam_step1_is_lr_times_sign():
    # Step 1 of Adam with eps = 0 moves every weight by lr * sign(g) (Kingma & Ba).
    # Dyadic inputs keep every fp32 operation exact; b1 != 1 - b1 and b2 != 1 - b2
    # so a swapped coefficient would show.
    rng = np.random.default_rng(11)
    k = 4096
    g = (rng.integers(1, 64, k) * rng.choice([-1, 1], k)).astype(np.float32) * np.float32(2.0 ** -10)
    p0 = (rng.integers(-512, 512, k)).astype(np.float32) * np.float32(2.0 ** -9)
    for b1, b2 in ((0.75, 0.9375), (0.5, 0.75), (0.875, 0.984375)):
        sc = O.step_scalars(O.Hyper(lr=2.0 ** -7, beta1=b1, beta2=b2, eps=0.0), 1)
        p1, m1, v1 = O.adam_update(p0, np.zeros(k, np.float32), np.zeros(k, np.float32), g, sc)
        assert np.array_equal(p1, p0 - np.float32(2.0 ** -7) * np.sign(g))
        assert np.array_equal(m1, np.float32(1 - b1) * g)
        assert np.array_equal(v1, np.float32(1 - b2) * g * g)


def test_zero_gradient_only_decays():
    sc = O.step_scalars(O.Hyper(lr=1e-2, weight_decay=0.5, eps=1e-8), 3)
    p0 = np.linspace(-1, 1, 101).astype(np.float32)
    z = np.zeros_like(p0)
    p1, m1, v1 = O.adam_update(p0, z, z, z, sc)
    assert np.array_equal(p1, p0 * np.float32(1 - 1e-2 * np.float32(0.5)))
    assert not np.any(m1) and not np.any(v1)


def _hp_adam(p, m, v, g, h, t):
    """Kingma & Ba AdamW in 60-digit decimal arithmetic, textbook form:
    p <- p(1 - lr wd); m <- b1 m + (1-b1) g; v <- b2 v + (1-b2) g^2;
    p <- p - lr * (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps)."""
    getcontext().prec = 60
    D = lambda x: Decimal(float(np.float32(x)))
    lr, b1, b2, eps, wd = D(h.lr), D(h.beta1), D(h.beta2), D(h.eps), D(h.weight_decay)
    p, m, v, g = Decimal(float(p)), Decimal(float(m)), Decimal(float(v)), Decimal(float(g))
    p = p * (1 - lr * wd)
    m = b1 * m + (1 - b1) * g
    v = b2 * v + (1 - b2) * g * g
    mhat = m / (1 - b1 ** t)
    vhat = v / (1 - b2 ** t)
    upd = lr * mhat / (vhat.sqrt() + eps)
    return p - upd, m, v, upd


def test_adam_against_high_precision():
    rng = np.random.default_rng(5)
    u = 2.0 ** -24
    for t in (1, 2, 7, 1000):
        h = O.Hyper(lr=3e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.05)
        sc = O.step_scalars(h, t)
        k = 300
        p = rng.normal(0, 0.02, k).astype(np.float32)
        m = rng.normal(0, 1e-3, k).astype(np.float32)
        v = np.abs(rng.normal(0, 1e-5, k)).astype(np.float32)
        g = rng.normal(0, 1e-2, k).astype(np.float32)
        p1, m1, v1 = O.adam_update(p, m, v, g, sc)
        for i in range(k):
            pe, me, ve, upd = _hp_adam(p[i], m[i], v[i], g[i], h, t)
            ulp_p = float(np.spacing(np.abs(np.float32(pe))))
            assert abs(Decimal(float(p1[i])) - pe) <= Decimal(2 * ulp_p) + abs(upd) * Decimal(16 * u)
            mag_m = abs(Decimal(float(np.float32(h.beta1))) * Decimal(float(m[i]))) + abs(Decimal(float(g[i])) / 10)
            assert abs(Decimal(float(m1[i])) - me) <= mag_m * Decimal(4 * u)
            assert abs(Decimal(float(v1[i])) - ve) <= abs(ve) * Decimal(4 * u) + Decimal(float(g[i]) ** 2) * Decimal(4 * u)


# ---------------------------------------------------------------- overflow / norm / clip
@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_overflow_skips_step_and_halves_scale(stage, bad):
    part, master, m, v, grads = _random_case(9, 200, 4, O.FP16, scale=1024.0)
    st = O.init_state(stage, O.FP16, part, master, m, v, loss_scale=1024.0)
    st.t = 5
    g = grads[0].copy()
    g[2, 123] = O.rne16(np.array([bad], np.float32), O.FP16)[0]
    new, res = O.step(st, g, O.Hyper())
    assert res.overflow and not res.applied
    assert new.loss_scale == 512.0 and new.t == 5
    for a, b in ((new.master, st.master), (new.m, st.m), (new.v, st.v), (new.params, st.params)):
        assert a.tobytes() == b.tobytes()


def test_overflow_in_padding_is_ignored_and_scale_floor():
    part = O.partition(10, 2, 8)
    st = O.init_state(1, O.FP16, part, np.ones(10, np.float32), loss_scale=1.0)
    g = np.zeros((2, part.psi_pad), np.uint16)
    g[1, 12] = 0x7C00  # +inf in padding: ignored
    new, res = O.step(st, g, O.Hyper(eps=1e-8))
    assert res.applied
    g[1, 3] = 0x7C00
    new2, res2 = O.step(new, g, O.Hyper())
    assert res2.overflow and new2.loss_scale == 1.0


def test_norm_of_constant_gradient():
    # all-equal averaged gradient c over psi = 64 elements: norm = |c| * 8
    part = O.partition(64, 4, 8)
    g = np.full((4, part.psi_pad), O.rne16(np.array([-0.375], np.float32), O.FP16)[0], np.uint16)
    st = O.init_state(2, O.FP16, part, np.zeros(64, np.float32))
    _, res = O.step(st, g, O.Hyper(eps=1e-8))
    assert res.norm == 0.375 * 8


def test_rank_sum_is_left_to_right_from_positive_zero():
    # The reduction order the pages leave open is fixed here as ranks 0..N-1,
    # each addition rounded in fp32, starting from +0.  Two cases checkable by
    # hand pin it: 1e8 - 1e8 + 1 is 1 left to right, but 0 right to left
    # (1 - 1e8 rounds to -1e8 in fp32); and -0 + -0 from +0 is +0, while
    # starting from the first rank would keep -0.
    s = O.rank_sum([np.array([1e8], np.float32), np.array([-1e8], np.float32), np.array([1.0], np.float32)])
    assert s.dtype == np.float32 and s[0] == np.float32(1.0)
    z = O.rank_sum([np.array([-0.0], np.float32), np.array([-0.0], np.float32)])
    assert z[0] == 0.0 and not np.signbit(z[0])


def _nearest_f32(x):
    # the fp32 value nearest the rational x, ties to even mantissa, found
    # among the neighbours of its double approximation (exact arithmetic)
    from fractions import Fraction
    d = np.float32(float(x))
    cands = [np.nextafter(d, np.float32(-np.inf)), d, np.nextafter(d, np.float32(np.inf))]
    return min(cands, key=lambda c: (abs(Fraction(float(c)) - x), int(np.float32(c).view(np.uint32)) & 1))


def test_unscale_is_one_rounded_division():
    # g_hat = s / f32(N * scale): one division, rounded once.  With N = 3 and
    # scale = 1000 (not powers of two) dividing by N and then by the scale
    # rounds twice, and these sums are ones where that changes the result.
    from fractions import Fraction
    s = np.array([41.32598114013672, 1042.513427734375, -128.53466796875], np.float32)
    got = O.unscale(s, 3, 1000.0)
    want = [_nearest_f32(Fraction(float(x)) / 3000) for x in s]
    assert got.dtype == np.float32 and [float(x) for x in got] == [float(x) for x in want]


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_norm_accumulates_in_double(stage):
    # One rank, g_hat = [2^26, 1, 1, 1, 1] (exact in bf16): the sum of squares
    # 2^52 + 4 is exact in fp64 (spacing 1 there) but 2^52 in fp32 (spacing
    # 2^29), so the norm is sqrt(2^52 + 4), not 2^26.
    part = O.partition(5, 1, 1)
    g = O.rne16(np.array([[2.0 ** 26, 1, 1, 1, 1]], np.float32), O.BF16)
    st = O.init_state(stage, O.BF16, part, np.zeros(5, np.float32))
    _, res = O.step(st, g, O.Hyper(eps=1e-8), [(0, 5)] if stage == 3 else None)
    assert res.norm == math.sqrt(2.0 ** 52 + 4) and res.norm != 2.0 ** 26


@pytest.mark.parametrize("stage", [1, 3])
@pytest.mark.parametrize("x", [2.0 ** 100, 2.0 ** -130])
def test_norm_squares_beyond_fp32_range(stage, x):
    # One rank, bf16 g_hat = [x, x, x, x]: the squares 2^200 and 2^-260 lie
    # outside fp32 (overflow, underflow) but are exact in fp64, so the norm
    # is exactly 2x.
    part = O.partition(4, 1, 1)
    g = O.rne16(np.full((1, 4), x, np.float32), O.BF16)
    assert np.array_equal(O.widen16(g, O.BF16), np.full((1, 4), x, np.float32))
    st = O.init_state(stage, O.BF16, part, np.zeros(4, np.float32))
    with np.errstate(over="ignore"):            # the fp32 g * g of the update is inf
        _, res = O.step(st, g, O.Hyper(eps=1e-8), [(0, 4)] if stage == 3 else None)
    assert res.norm == 2 * x


@pytest.mark.parametrize("stage", [1, 3])
def test_norm_sums_each_shard_left_to_right(stage):
    # Each owner adds its shard's squares in order, in fp64.  One rank,
    # bf16 g_hat = [1, 2^-27 x 16]: every square 2^-54 is below half an ulp
    # of 1, so each addition after the first rounds back to 1 and the norm
    # is exactly 1.  Adding the small squares first (pairwise or several
    # accumulators) gives 1 + 2^-50 and a norm above 1.
    part = O.partition(17, 1, 1)
    g = O.rne16(np.array([[1.0] + [2.0 ** -27] * 16], np.float32), O.BF16)
    assert np.array_equal(O.widen16(g, O.BF16)[0][1:], np.full(16, 2.0 ** -27, np.float32))
    st = O.init_state(stage, O.BF16, part, np.zeros(17, np.float32))
    _, res = O.step(st, g, O.Hyper(eps=1e-8), [(0, 17)] if stage == 3 else None)
    assert res.norm == 1.0


def test_clip_scales_gradient_to_max_norm():
    part, master, m, v, grads = _random_case(13, 500, 2, O.FP16)
    h_free = O.Hyper(beta1=0.75, eps=1e-8)
    st = O.init_state(2, O.FP16, part, master)
    _, res = O.step(st, grads[0], h_free)
    norm = res.norm
    assert res.clip is None
    h_clip = O.Hyper(beta1=0.75, eps=1e-8, max_norm=norm / 4)
    new, res2 = O.step(st, grads[0], h_clip)
    assert res2.clip is not None
    c = float(np.float32(norm / 4)) / (norm + 1e-6)   # max_norm / (norm + 1e-6)
    assert abs(float(res2.clip) - c) <= 2.0 ** -24 * c
    # m after step 1 from m = 0 is (1 - b1) * c * g_hat: its norm is 0.25 * c * norm
    m_norm = float(np.sqrt(np.sum(new.m.astype(np.float64) ** 2)))
    assert abs(m_norm - 0.25 * c * norm) <= 1e-6 * m_norm
    # max_norm above the norm: no clipping
    _, res3 = O.step(st, grads[0], O.Hyper(beta1=0.75, eps=1e-8, max_norm=norm * 2))
    assert res3.clip is None


# ---------------------------------------------------------------- ZeRO++ quantizer
def test_quantizer_is_lossless_on_its_grid():
    # values lo + k*s with k in [0, 255] (k = 0 and 255 present, s dyadic):
    # scale = 255 s / 255 = s exactly and every code is k exactly
    rng = np.random.default_rng(21)
    s, lo = 2.0 ** -6, -1.5
    k = rng.integers(0, 256, 1000)
    k[:2] = [0, 255]
    x = (lo + k * s).astype(np.float32)
    codes, scale, l0 = O.quantize_blocks(x, 8, block=1000)
    assert scale[0] == np.float32(s) and l0[0] == np.float32(lo)
    assert np.array_equal(codes, k.astype(np.uint8))
    assert np.array_equal(O.dequantize_blocks(codes, scale, l0, block=1000), x)
    # 4-bit: 16 levels
    k4 = rng.integers(0, 16, 300)
    k4[:2] = [0, 15]
    x4 = (0.25 + k4 * 2.0 ** -3).astype(np.float32)
    c4, s4, l4 = O.quantize_blocks(x4, 4, block=300)
    assert np.array_equal(c4, k4.astype(np.uint8)) and s4[0] == np.float32(0.125)


def _rint_even(q):
    # nearest integer to the rational q, ties to even
    return round(q)


def test_quantizer_code_is_one_division_by_the_scale():
    # The notes name zero-point block quantization and give no formula, so the
    # oracle takes the plain definition: code = rint((x - lo) / scale), the
    # subtraction and the division each one fp32 operation rounded once.
    # Forming 1 / scale once per block and multiplying by it rounds
    # differently for values near the middle between two levels; the blocks
    # here are made of such values (lo = 0, so x - lo is exact) and their
    # codes are worked out in exact rational arithmetic.
    from fractions import Fraction
    rng = np.random.default_rng(41)
    for bits in (8, 4):
        qmax = (1 << bits) - 1
        hi = np.float32(rng.uniform(0.5, 2.0))
        s = _nearest_f32(Fraction(float(hi)) / qmax)
        inv = _nearest_f32(Fraction(qmax) / Fraction(float(hi)))
        vals, want, differ = [], [], 0
        for k in range(qmax):
            mid = np.float32((k + 0.5) * float(s))
            for step in (-2, -1, 0, 1, 2):
                x = mid
                for _ in range(abs(step)):
                    x = np.nextafter(x, np.float32(np.inf if step > 0 else -np.inf))
                fx = Fraction(float(x))
                code = min(qmax, max(0, _rint_even(Fraction(float(_nearest_f32(fx / Fraction(float(s))))))))
                short = min(qmax, max(0, _rint_even(Fraction(float(_nearest_f32(fx * Fraction(float(inv))))))))
                if code != short and len(vals) < 254:
                    vals.append(x)
                    want.append(code)
                    differ += 1
        assert differ >= 3, differ
        block = np.array([0.0, hi] + vals, np.float32)
        codes, scale, lo = O.quantize_blocks(block, bits, block=block.size)
        assert scale[0] == s and lo[0] == 0.0
        assert list(codes[:2]) == [0, qmax]
        assert [int(c) for c in codes[2:]] == want


def test_quantizer_error_bound_and_order():
    rng = np.random.default_rng(22)
    x = rng.normal(0, 3, 5000).astype(np.float32)
    for bits in (8, 4):
        codes, scale, lo = O.quantize_blocks(x, bits)
        xq = O.dequantize_blocks(codes, scale, lo)
        k = np.arange(x.size) // O.Q_BLOCK
        ulp = np.spacing(np.abs(x).max()).astype(np.float64)
        assert np.all(np.abs(xq.astype(np.float64) - x) <= scale[k] / 2 + 4 * ulp)
        for b in range(scale.size):
            blk = slice(b * O.Q_BLOCK, (b + 1) * O.Q_BLOCK)
            xb, cb = x[blk], codes[blk]
            assert cb[np.argmin(xb)] == 0 and cb[np.argmax(xb)] == (1 << bits) - 1
            order = np.argsort(xb, kind="stable")
            assert np.all(np.diff(cb[order].astype(int)) >= 0)      # codes are monotone
    assert (O.quantize_blocks(x, 8)[0].size, O.quantize_blocks(x, 8)[1].size) == (5000, 20)


def test_quantizer_constant_block_and_nan():
    c, s, l = O.quantize_blocks(np.full(10, 0.375, np.float32), 8)
    assert s[0] == 0 and not np.any(c) and np.all(O.dequantize_blocks(c, s, l) == 0.375)
    x = np.ones(300, np.float32)
    x[5] = np.nan
    c, s, l = O.quantize_blocks(x, 8)
    assert np.all(np.isnan(O.dequantize_blocks(c, s, l)[:256]))   # the NaN poisons its block
    assert np.all(O.dequantize_blocks(c, s, l)[256:] == 1.0)


def test_int4_packing():
    assert list(O.pack_int4(np.array([1, 2, 15, 0], np.uint8))) == [0x21, 0x0F]
    c = np.random.default_rng(3).integers(0, 16, 301).astype(np.uint8)
    assert np.array_equal(O.unpack_int4(O.pack_int4(c), 301), c)


@pytest.mark.parametrize("bits", [8, 4])
def test_quantized_reduce_scatter_equals_plain_on_grid_gradients(bits):
    # gradients whose every quantization block spans at most 2^bits levels of a
    # dyadic grid are exchanged losslessly: the ZeRO++ step equals ZeRO-3's
    rng = np.random.default_rng(23)
    n, psi = 3, 700
    part = O.partition(psi, n, 8)
    buckets = [(0, 256), (256, 520), (520, part.psi_pad)]
    master = rng.normal(0, 0.02, psi).astype(np.float32)
    levels = (1 << bits) - 1
    g = np.zeros((n, part.psi_pad), np.float32)
    for r in range(n):
        for (a, b) in buckets:
            for k0 in range(a, b, O.Q_BLOCK):
                k1 = min(b, k0 + O.Q_BLOCK)
                q = rng.integers(0, levels + 1, k1 - k0)
                q[:2] = [0, levels]
                g[r, k0:k1] = (q - levels // 2) * 2.0 ** -10
    g[:, psi:] = 0
    gb = O.rne16(g, O.BF16)
    assert np.array_equal(O.widen16(gb, O.BF16), g)
    h = O.Hyper(weight_decay=0.1)
    st = O.init_state(3, O.BF16, part, master)
    bg = [gb[:, a:b] for (a, b) in buckets]
    want, r1 = O.step_stage3(st, bg, buckets, h)
    got, r2 = O.step_stage3_quantized(st, bg, buckets, h, bits)
    assert np.array_equal(want.master, got.master) and np.array_equal(want.params, got.params)
    assert r1.norm == r2.norm


def test_quantized_gather_reproduces_grid_weights():
    # a shard whose blocks hold at most 256 grid levels is gathered exactly
    rng = np.random.default_rng(24)
    q = rng.integers(0, 256, 600)
    for k0 in range(0, 600, O.Q_BLOCK):
        q[k0:k0 + 2] = [0, 255]                  # every block spans the full 256 levels
    w = O.rne16(((q - 128) * 2.0 ** -9).astype(np.float32), O.BF16)
    outs, view = O.quantized_gather(w, 0, 600, O.BF16, 4)
    assert len(outs) == 4 and np.array_equal(view, w)


# ---------------------------------------------------------------- ZeRO-3 param_persistence_threshold
def test_persistent_layout_against_a_sort_key():
    # "ZeRO Stage 1/2/3" guide, ZeRO-3 config: params with fewer elements than
    # the threshold stay replicated.  The layout is the stable partition
    # "partitioned first, persistent last": the same order as sorting by the
    # key (is_small, model index), which the oracle does not compute.
    rng = np.random.default_rng(11)
    for trial in range(200):
        k = int(rng.integers(0, 12))
        sizes = [int(x) for x in rng.integers(1, 40, k)]
        thr = int(rng.integers(0, 45))
        order, p0, psi = O.persistent_layout(sizes, thr)
        want = sorted(range(k), key=lambda i: (sizes[i] < thr, i))
        assert order == want
        assert psi == sum(sizes)
        assert p0 == sum(s for s in sizes if s >= thr)
        # the region [p0, psi) is exactly the small tensors
        pos = 0
        for i in order:
            assert (pos >= p0) == (sizes[i] < thr)
            pos += sizes[i]


def test_persistent_threshold_is_strict_and_degenerate_cases():
    sizes = [100, 99, 101, 100]
    order, p0, psi = O.persistent_layout(sizes, 100)
    assert order == [0, 2, 3, 1] and p0 == 301 and psi == 400   # exactly 100 stays partitioned
    assert O.persistent_layout(sizes, 0) == ([0, 1, 2, 3], 400, 400)       # nothing persistent
    assert O.persistent_layout(sizes, 10 ** 9) == ([0, 1, 2, 3], 0, 400)   # everything persistent
    assert O.persistent_layout([], 5) == ([], 0, 0)


def test_guide_threshold_on_the_model_lists():
    # threshold 1e5 (the guide's value).  GPT-2 small: every bias and layer
    # norm is persistent -- per layer 2*768 (ln_1) + 2304 + 768 + 2*768 (ln_2)
    # + 3072 + 768 = 9984, times 12, plus ln_f 2*768 = 121,344 elements in 98
    # tensors.  Llama-7B: the 65 RMSNorm weights of 4096 = 266,240.
    from zero_partitioned_mixed_gb300 import synth as S
    for shapes, n_pers, psi_pers in ((S.gpt2_small_shapes(), 98, 121_344), (S.llama7b_shapes(), 65, 266_240)):
        sizes = [S.numel(s) for _, s in shapes]
        order, p0, psi = O.persistent_layout(sizes, 100_000)
        assert psi - p0 == psi_pers
        assert sum(1 for i in order if sizes[i] < 100_000) == n_pers


def test_persistent_comm_and_memory_endpoints():
    # No persistent tensor: ZeRO-3's 3 Psi and (4+K) Psi / N.  Every tensor
    # persistent: the forward/backward gathers vanish and the refresh is one
    # all-gather, so the communication is ZeRO-2's 2 Psi, and the memory is
    # ZeRO-2's plus the 16-bit owner shards kept as the refresh's source.
    for psi, n in ((637_952, 32), (124_439_808, 8), (6_738_415_616 + 0, 8)):
        pp = O.partition(psi, n, 8).psi_pad
        assert O.comm_elems_persistent(pp, 0) == O.comm_elems_paper(pp, 3)
        assert O.comm_elems_persistent(pp, pp) == O.comm_elems_paper(pp, 2)
        assert O.comm_elems_persistent(pp, 1000) == 3 * pp - 1000
        assert O.model_state_bytes_persistent(pp, 0, n) == O.model_state_bytes(pp, n, 3)
        assert O.model_state_bytes_persistent(pp, pp, n) == O.model_state_bytes(pp, n, 2) + 2 * pp // n
        # the ring model at the same ends: ZeRO-3's and ZeRO-2's (N-1)/N counts
        assert O.comm_elems_ring_persistent(pp, 0, n) == O.comm_elems_ring(pp, n, 3)
        assert O.comm_elems_ring_persistent(pp, pp, n) == O.comm_elems_ring(pp, n, 2)
        # in between: (N-1)/N of each of the four collectives, summed exactly
        from fractions import Fraction
        k = Fraction(n - 1, n)
        exact = 2 * k * (pp - 1000) + k * pp + k * 1000
        assert O.comm_elems_ring_persistent(pp, 1000, n) == math.floor(exact)


@pytest.mark.parametrize("dt", [O.FP16, O.BF16])
def test_persistence_moves_no_value(dt):
    # persistence changes where 16-bit copies live, not what the step computes:
    # three steps equal stage 1's bit for bit; the persistent copies equal the
    # cast of the new master over [p0, psi_pad); an overflowed step keeps them.
    n, psi = 4, 1001
    part, master, m, v, grads = _random_case(5, psi, n, dt)
    pp = part.psi_pad
    p0 = 640
    buckets = [(0, 96), (96, 640), (640, 900), (900, pp)]
    h = O.Hyper(lr=1e-3, weight_decay=0.1, max_norm=0.05)
    s3 = O.init_state(3, dt, part, master, m, v)
    s1 = O.init_state(1, dt, part, master, m, v)
    for k in range(3):
        g = grads[k].copy()
        if k == 1:
            g[2, 700] = O.rne16(np.array([np.inf], np.float32), dt)[0]
        s3, res, reps = O.step_stage3_persistent(s3, [g[:, a:b] for (a, b) in buckets], buckets, h, p0)
        s1, res1 = O.step(s1, g, h)
        assert res.overflow == res1.overflow == (k == 1)
        assert np.array_equal(s3.master.view(np.uint32), s1.master.view(np.uint32))
        assert np.array_equal(s3.params, s1.params[0])
        assert len(reps) == n and all(np.array_equal(x, O.rne16(s3.master, dt)[p0:pp]) for x in reps)
        assert len(res.gathered_fwd) == len(res.gathered_bwd) == 2
        assert np.array_equal(res.gathered_bwd[1][3], res.gathered_fwd[1][0])
    with pytest.raises(ValueError):
        O.step_stage3_persistent(s3, [grads[0][:, 0:700], grads[0][:, 700:pp]], [(0, 700), (700, pp)], h, p0)
