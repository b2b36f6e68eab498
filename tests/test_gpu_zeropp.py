"""ZeRO++ quantized exchanges on the GPU vs the oracle: block quantizer and
dequantizer (INT8 / INT4, both 16-bit formats, ragged sizes), the INT8
quantized ZeRO-3 gather, and ZeRO-3 steps whose reduce-scatter consumes the
ranks' quantized gradients (speculative and two-pass, overflow)."""

import numpy as np
import pytest
import torch

import oracle as O
from _parity import bits16, bits32
from zero_partitioned_mixed_gb300 import _binding as B
from zero_partitioned_mixed_gb300 import synth as S
from zero_partitioned_mixed_gb300.buffers import RankBuffers

pytestmark = pytest.mark.gpu
ZDT = {"fp16": B.ZERO_FP16, "bf16": B.ZERO_BF16}


def _nb(count):
    return (count + O.Q_BLOCK - 1) // O.Q_BLOCK


def _codes_buf(count, bits):
    nbytes = count if bits == 8 else (count + 1) // 2
    return torch.zeros(max(16, (nbytes + 15) // 16 * 16), dtype=torch.uint8, device="cuda")


def _quantize_gpu(x16, dtype, bits):
    n = x16.numel()
    codes = _codes_buf(n, bits)
    scales = torch.zeros(max(2, 2 * _nb(n)), dtype=torch.float32, device="cuda")
    B.zero_quantize_blocks(ZDT[dtype], bits, x16, n, codes, scales)
    return codes, scales


def _oracle_codes(x_bits, dtype, bits):
    codes, scale, lo = O.quantize_blocks(O.widen16(x_bits, dtype), bits)
    packed = codes if bits == 8 else O.pack_int4(codes)
    return packed, scale, lo


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("count", [1, 7, 255, 256, 257, 4096, 100_003])
def test_quantize_and_dequantize_match_oracle(dtype, bits, count):
    g = torch.Generator(device="cuda")
    g.manual_seed(count * 7 + bits)
    x = torch.empty(max(8, (count + 7) // 8 * 8), dtype=S.torch_dtype(dtype), device="cuda")
    x[:count] = (torch.randn(count, generator=g, device="cuda") * 3).to(x.dtype)
    x[count:] = 0
    if count > 300:
        x[256:512] = x[300]                     # a constant block: scale 0
    codes, scales = _quantize_gpu(x[:count], dtype, bits)
    xb = bits16(x[:count])
    packed, scale, lo = _oracle_codes(xb, dtype, bits)
    got = codes.cpu().numpy()[:packed.size]
    assert np.array_equal(got, packed)
    sc = scales.cpu().numpy()[:2 * _nb(count)]
    assert np.array_equal(sc[0::2].view(np.uint32), scale.view(np.uint32))
    assert np.array_equal(sc[1::2].view(np.uint32), lo.view(np.uint32))
    out = torch.zeros_like(x)
    B.zero_dequantize_blocks(ZDT[dtype], bits, codes, scales, count, out)
    want = O.rne16(O.dequantize_blocks(O.quantize_blocks(O.widen16(xb, dtype), bits)[0], scale, lo), dtype)
    assert np.array_equal(bits16(out[:count]), want)


def _near_midpoint_blocks(dtype, bits, n_blocks, seed):
    # 256-element blocks [0, hi, x, ...] of 16-bit values x for which
    # rint(x / scale) and rint(x * (1 / scale)) give different codes: the
    # values near the middle between two levels that tell the plain division
    # from a reciprocal multiply.  Found by enumerating every positive finite
    # 16-bit value below hi.
    qmax = np.float32((1 << bits) - 1)
    top = 0x7C00 if dtype == "fp16" else 0x7F80
    allv = O.widen16(np.arange(1, top, dtype=np.uint16), dtype)
    rng = np.random.default_rng(seed)
    his = allv[(allv > 0.25) & (allv < 4.0)]
    blocks, differing = [], 0
    for hi in rng.permutation(his):
        x = allv[allv < hi]
        with np.errstate(over="ignore"):
            d = x[np.rint(x / np.float32(hi / qmax)) != np.rint(x * np.float32(qmax / hi))]
        if d.size == 0:
            continue
        fill = rng.choice(x, 254 - d.size) if d.size < 254 else np.zeros(0, np.float32)
        blk = np.concatenate([[np.float32(0), hi], d[:254], fill]).astype(np.float32)
        blocks.append(blk)
        differing += min(d.size, 254)
        if len(blocks) == n_blocks:
            break
    return np.concatenate(blocks), differing


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("bits", [8, 4])
def test_quantizer_divides_by_the_scale(dtype, bits):
    x, differing = _near_midpoint_blocks(dtype, bits, 64, 3 + bits)
    assert differing >= 40
    xb = O.rne16(x, dtype)
    assert np.array_equal(O.widen16(xb, dtype), x)
    dev = torch.from_numpy(xb.view(np.int16)).cuda().view(S.torch_dtype(dtype))
    codes, scales = _quantize_gpu(dev, dtype, bits)
    packed, scale, lo = _oracle_codes(xb, dtype, bits)
    assert np.array_equal(codes.cpu().numpy()[:packed.size], packed)
    sc = scales.cpu().numpy()[:2 * _nb(x.size)]
    assert np.array_equal(sc[0::2].view(np.uint32), scale.view(np.uint32))


def _same_floats(got, want):
    # bit-equal, or NaN on both sides (a NaN's payload is not part of the format)
    g, w = np.asarray(got, np.float32), np.asarray(want, np.float32)
    both_nan = np.isnan(g) & np.isnan(w)
    return bool(np.all(both_nan | (g.view(np.uint32) == w.view(np.uint32))))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("bits", [8, 4])
def test_quantizer_special_blocks(dtype, bits):
    # blocks that the kernels leave to the clamped division (a NaN, +-inf, a
    # range that overflows, a scale below 2^-100 from bf16 subnormals) and
    # blocks at the edges of the screened path (constant +-0, fp16
    # subnormals), each beside ordinary ones, in a buffer with a ragged end
    rng = np.random.default_rng(5 + bits)
    base = lambda: rng.normal(0, 1, 256).astype(np.float32)
    blocks = [base()]
    b = base(); b[17] = np.nan; blocks.append(b)
    b = base(); b[3] = np.inf; blocks.append(b)
    b = base(); b[200] = -np.inf; blocks.append(b)
    big = np.float32(60000.0 if dtype == "fp16" else 3.0e38)
    b = base(); b[0] = big; b[1] = -big; blocks.append(b)
    tiny = np.float32(2.0 ** -24 if dtype == "fp16" else 2.0 ** -133)
    blocks.append((rng.integers(0, 4, 256) * tiny).astype(np.float32))
    blocks.append(np.zeros(256, np.float32))
    b = np.zeros(256, np.float32); b[::2] = -0.0; blocks.append(b)
    blocks.append(base()[:77])
    xb = O.rne16(np.concatenate(blocks), dtype)
    count = xb.size
    dev = torch.zeros(max(8, (count + 7) // 8 * 8), dtype=S.torch_dtype(dtype), device="cuda")
    dev[:count].copy_(torch.from_numpy(xb.view(np.int16)).view(S.torch_dtype(dtype)))
    codes, scales = _quantize_gpu(dev[:count], dtype, bits)
    with np.errstate(over="ignore"):            # hi - lo overflows in one block
        packed, scale, lo = _oracle_codes(xb, dtype, bits)
    assert np.array_equal(codes.cpu().numpy()[:packed.size], packed)
    sc = scales.cpu().numpy()[:2 * _nb(count)]
    assert _same_floats(sc[0::2], scale) and _same_floats(sc[1::2], lo)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("a,b", [(0, 70_000), (1024, 1032), (13, 5_013), (256, 257)])
def test_quantized_gather_matches_oracle(a, b, dt):
    psi, n = 80_000, 4
    buf = RankBuffers(psi, n, 3, dt)
    P = buf.psi_pad
    td = S.torch_dtype(dt)
    buf.params[:P].copy_((torch.randn(P, device="cuda") * 0.02).to(td))
    L = b - a
    codes = [_codes_buf(L, 8) for _ in range(n)]
    scales = [torch.zeros(2 * _nb(L), dtype=torch.float32, device="cuda") for _ in range(n)]
    B.zero_gather_bucket_q8(buf.h, a, b, buf.params, codes, scales)
    outs, view = O.quantized_gather(bits16(buf.params[:P]), a, b, dt, n)
    for r in range(n):
        c, s, l = outs[r]
        assert np.array_equal(codes[r].cpu().numpy()[:L], c)
        sc = scales[r].cpu().numpy()
        assert np.array_equal(sc[0::2], s) and np.array_equal(sc[1::2], l)
        deq = torch.zeros(max(8, (L + 7) // 8 * 8), dtype=td, device="cuda")
        B.zero_dequantize_blocks(ZDT[dt], 8, codes[r], scales[r], L, deq)
        assert np.array_equal(bits16(deq[:L]), view)
    assert buf.bytes_moved()["hbm_write_bytes"] == n * (L + 8 * _nb(L))
    buf.close()


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("double_buffer", [True, False])
@pytest.mark.parametrize("psi,n,align,cuts", [
    (150_001, 4, 8, [40_000, 40_013, 99_999]),
    # psi_pad = 31,910 is not a multiple of 8: with two state slots the
    # second starts off a vector boundary, so even the 8-aligned buckets
    # must take the element-wise path
    (31_910, 5, 2, [13_520, 16_280, 24_864]),
])
def test_quantized_reduce_scatter_step_matches_oracle(bits, double_buffer, psi, n, align, cuts):
    dt = "bf16"
    part = O.partition(psi, n, align)
    P = part.psi_pad
    edges = [0] + cuts + [P]
    buckets = list(zip(edges, edges[1:]))
    buf = RankBuffers(psi, n, 3, dt, align=align, double_buffer=double_buffer)
    g = torch.Generator(device="cuda")
    g.manual_seed(bits)
    master = torch.randn(psi, generator=g, device="cuda") * 0.02
    st = O.init_state(3, dt, part, master.cpu().numpy())
    mv, _, _ = buf.state(0)
    mv.copy_(torch.from_numpy(st.master))
    buf.params[:P].copy_(torch.from_numpy(st.params.view(np.int16)).view(torch.bfloat16))
    hb, ho = B.hyper(weight_decay=0.05), O.Hyper(weight_decay=0.05)
    for step in range(3):
        grads = torch.zeros((n, buf.stride), dtype=torch.bfloat16, device="cuda")
        grads[:, :psi] = (torch.randn((n, psi), generator=g, device="cuda") * 1e-2).to(torch.bfloat16)
        if step == 1:
            grads[2, psi // 2 + 3] = float("inf")
        gb = bits16(grads)
        for (a, b) in reversed(buckets):
            L = b - a
            codes, scales = [], []
            for r in range(n):
                src = torch.zeros(max(8, (L + 7) // 8 * 8), dtype=torch.bfloat16, device="cuda")
                src[:L].copy_(grads[r, a:b])
                c, s = _quantize_gpu(src[:L], dt, bits)
                codes.append(c)
                scales.append(s)
            B.zero_reduce_scatter_bucket_q(buf.h, a, b, bits, codes, scales, buf.master, buf.m, buf.v,
                                           buf.params, hb)
        buf.step(hb)
        st, res = O.step_stage3_quantized(st, [gb[:, a:b] for (a, b) in buckets], buckets, ho, bits)
        s = buf.status()
        assert bool(s["overflow"]) == res.overflow == (step == 1)
        assert s["steps_applied"] == st.t
        if res.applied:
            assert abs(s["grad_norm"] - res.norm) <= 1e-5 * res.norm
        gm, gmm, gv = buf.state(s["state_slot"])
        assert np.array_equal(bits32(gm), st.master.view(np.uint32))
        assert np.array_equal(bits32(gmm), st.m.view(np.uint32))
        assert np.array_equal(bits32(gv), st.v.view(np.uint32))
        assert np.array_equal(bits16(buf.params[:P]), st.params)
    buf.close()


def test_quantized_calls_reject_bad_arguments():
    x = torch.zeros(64, dtype=torch.float16, device="cuda")
    with pytest.raises(B.ZeroError):
        B.zero_quantize_blocks(B.ZERO_FP16, 3, x, 64, x, x)
    with pytest.raises(B.ZeroError):
        B.zero_quantize_blocks(B.ZERO_FP16, 8, x.view(-1)[1:], 8, x, x)
    buf = RankBuffers(1024, 2, 2, "fp16")
    with pytest.raises(B.ZeroError):
        B.zero_gather_bucket_q8(buf.h, 0, 8, buf.params, [x, x], [x, x])
    buf.close()


@pytest.mark.parametrize("bits", [8, 4])
def test_zeropp_step_at_scale(bits):
    # psi = 2^24 + 13 over 8 ranks in 4 buckets: the quantized gather's
    # launches reach its full chunk count and the reduce-scatter a full
    # grid; every code, scale, state element and shard element is compared
    psi, n, dt = (1 << 24) + 13, 8, "bf16"
    part = O.partition(psi, n, 8)
    P = part.psi_pad
    cut = P // 4 // 8 * 8
    buckets = [(0, cut), (cut, 2 * cut), (2 * cut, 3 * cut + 5), (3 * cut + 5, P)]
    buf = RankBuffers(psi, n, 3, dt, double_buffer=True)
    g = torch.Generator(device="cuda")
    g.manual_seed(31 + bits)
    master = torch.randn(psi, generator=g, device="cuda") * 0.02
    st = O.init_state(3, dt, part, master.cpu().numpy())
    buf.state(0)[0].copy_(torch.from_numpy(st.master))
    buf.params[:P].copy_(torch.from_numpy(st.params.view(np.int16)).view(torch.bfloat16))
    hb, ho = B.hyper(weight_decay=0.1), O.Hyper(weight_decay=0.1)
    # the forward gather of every bucket, INT8, against the oracle's
    shard_bits = bits16(buf.params[:P])
    for (a, b) in buckets:
        L = b - a
        codes = [_codes_buf(L, 8) for _ in range(n)]
        scales = [torch.zeros(2 * _nb(L), dtype=torch.float32, device="cuda") for _ in range(n)]
        B.zero_gather_bucket_q8(buf.h, a, b, buf.params, codes, scales)
        outs, _ = O.quantized_gather(shard_bits, a, b, dt, n)
        for r in (0, n - 1):
            c, s, l = outs[r]
            assert np.array_equal(codes[r].cpu().numpy()[:L], c)
            sc = scales[r].cpu().numpy()
            assert np.array_equal(sc[0::2].view(np.uint32), s.view(np.uint32))
            assert np.array_equal(sc[1::2].view(np.uint32), l.view(np.uint32))
    # one step whose reduce-scatter takes the ranks' quantized gradients
    grads = torch.zeros((n, buf.stride), dtype=torch.bfloat16, device="cuda")
    grads[:, :psi] = (torch.randn((n, psi), generator=g, device="cuda") * 1e-2).to(torch.bfloat16)
    gb = bits16(grads)
    for (a, b) in reversed(buckets):
        L = b - a
        codes, scales = [], []
        for r in range(n):
            src = torch.zeros(max(8, (L + 7) // 8 * 8), dtype=torch.bfloat16, device="cuda")
            src[:L].copy_(grads[r, a:b])
            c, s = _quantize_gpu(src[:L], dt, bits)
            codes.append(c)
            scales.append(s)
        B.zero_reduce_scatter_bucket_q(buf.h, a, b, bits, codes, scales, buf.master, buf.m, buf.v, buf.params, hb)
    buf.step(hb)
    st, res = O.step_stage3_quantized(st, [gb[:, a:b] for (a, b) in buckets], buckets, ho, bits)
    s = buf.status()
    assert not s["overflow"] and not res.overflow and s["steps_applied"] == 1
    assert abs(s["grad_norm"] - res.norm) <= 1e-5 * res.norm
    gm, gmm, gv = buf.state(s["state_slot"])
    assert np.array_equal(bits32(gm), st.master.view(np.uint32))
    assert np.array_equal(bits32(gmm), st.m.view(np.uint32))
    assert np.array_equal(bits32(gv), st.v.view(np.uint32))
    assert np.array_equal(bits16(buf.params[:P]), st.params)
    buf.close()


@pytest.mark.parametrize("bits", [8, 4])
def test_quantized_reduce_scatter_extreme_scales(bits):
    # bf16 gradient blocks whose scales lie above 2^100, in the subnormal
    # range (bf16 subnormals), near 2^60 and ordinary, in one bucket of three
    # ranks: the dequantized sums, the fp32 squares of the update (which
    # overflow) and the norm (summed in fp64 there); every state element
    # and the norm against the oracle
    psi, n, dt = 256 * 12 + 77, 3, "bf16"
    part = O.partition(psi, n, 8)
    P = part.psi_pad
    rng = np.random.default_rng(40 + bits)
    mags = np.array([2.0 ** 110, 2.0 ** -130, 2.0 ** 60, 1.0, 2.0 ** 100, 2.0 ** -120,
                     1e-3, 2.0 ** 110, 1.0, 2.0 ** -130, 1.0, 2.0 ** 50, 1.0])
    g = rng.normal(0, 1, (n, psi)) * np.repeat(mags, 256)[:psi]
    gbits = np.zeros((n, P), np.uint16)
    gbits[:, :psi] = O.rne16(g.astype(np.float32), dt)
    buf = RankBuffers(psi, n, 3, dt)
    master = (rng.normal(0, 0.02, psi)).astype(np.float32)
    st = O.init_state(3, dt, part, master)
    buf.state(0)[0].copy_(torch.from_numpy(st.master))
    buf.params[:P].copy_(torch.from_numpy(st.params.view(np.int16)).view(torch.bfloat16))
    hb, ho = B.hyper(), O.Hyper()
    dev = torch.from_numpy(gbits.view(np.int16)).cuda().view(torch.bfloat16)
    codes, scales = [], []
    for r in range(n):
        c, s = _quantize_gpu(dev[r, :P], dt, bits)
        codes.append(c)
        scales.append(s)
    assert float(scales[0][0].item()) > 2.0 ** 100
    B.zero_reduce_scatter_bucket_q(buf.h, 0, P, bits, codes, scales, buf.master, buf.m, buf.v, buf.params, hb)
    buf.step(hb)
    with np.errstate(over="ignore", invalid="ignore"):
        st, res = O.step_stage3_quantized(st, [gbits], [(0, P)], ho, bits)
    s = buf.status()
    assert bool(s["overflow"]) == res.overflow
    if res.applied:
        assert abs(s["grad_norm"] - res.norm) <= 1e-5 * res.norm
    gm, gmm, gv = buf.state(s["state_slot"])
    assert np.array_equal(bits32(gm), st.master.view(np.uint32))
    assert np.array_equal(bits32(gmm), st.m.view(np.uint32))
    assert np.array_equal(bits32(gv), st.v.view(np.uint32))
    assert np.array_equal(bits16(buf.params[:P]), st.params)
    buf.close()
