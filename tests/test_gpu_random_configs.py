"""Seeded random configurations against the oracle, element by element.

Each case draws a stage, a rank count, a dtype, a mode, a ragged psi and
alignment, a bucket layout (stage 3, or stage 2 reduced during backward),
whether the ZeRO-3 backward runs through the fused reduce-scatter + gather,
a loss scale, an overflow at a random step, rank and index, and clipping;
then runs three steps through the C ABI and compares every element of the
state, the replicas or shard and the gathered rows with the oracle.  The
draws are fixed by the seed, so a failing case reproduces.
"""

import numpy as np
import pytest

from _parity import run_case

pytestmark = pytest.mark.gpu

INF, NAN = float("inf"), float("nan")


def _buckets(rng, pp, align_to):
    """A random tiling of [0, pp) into 1..6 buckets; boundaries on multiples of align_to."""
    k = int(rng.integers(1, 7))
    cuts = sorted(set(int(c) // align_to * align_to for c in rng.integers(1, max(2, pp), k - 1)))
    cuts = [c for c in cuts if 0 < c < pp]
    edges = [0] + cuts + [pp]
    return [(a, b) for a, b in zip(edges, edges[1:]) if b > a]


def _case(seed):
    rng = np.random.default_rng(seed)
    stage = int(rng.choice([0, 1, 2, 3]))
    n = int(rng.choice([1, 2, 3, 4, 5, 8, 13]))
    dtype = str(rng.choice(["fp16", "bf16"]))
    align = int(rng.choice([1, 2, 8]))
    psi = int(rng.integers(1, 60_000))
    unit = n * align
    pp = (psi + unit - 1) // unit * unit
    double_buffer = stage != 0 and bool(rng.integers(0, 2))
    # stage 2 reduced during backward has no re-read mode
    bucketed = stage == 3 or (stage == 2 and bool(rng.integers(0, 2)))
    mode = 0
    if stage in (1, 2):
        mode = int(rng.choice([0, 1] + ([] if bucketed else [2]) + ([3] if double_buffer else [])))
    buckets, fused = None, False
    if bucketed:
        buckets = _buckets(rng, pp, int(rng.choice([1, 8])))
        fused = stage == 3 and bool(rng.integers(0, 2))
    loss_scale = float(rng.choice([1.0, 8.0, 1000.0, 65536.0]))
    sigma = float(rng.choice([1e-3, 1e-2]))
    inject = []
    if rng.integers(0, 3) == 0 and psi > 0:
        inject = [(int(rng.integers(0, 3)), int(rng.integers(0, n)), int(rng.integers(0, psi)),
                   float(rng.choice([INF, -INF, NAN])))]
    hyper_kw = {"weight_decay": float(rng.choice([0.0, 0.1]))}
    if rng.integers(0, 3) == 0:
        hyper_kw["max_norm"] = float(rng.choice([1e-3, 10.0]))   # clipping on, or a bound never reached
    return dict(psi=psi, n=n, stage=stage, dtype=dtype, align=align, mode=mode, double_buffer=double_buffer,
                buckets=buckets, fused=fused, loss_scale=loss_scale, sigma=sigma,
                inject=inject, hyper_kw=hyper_kw, seed=seed)


@pytest.mark.parametrize("seed", range(200))
def test_random_configuration_matches_oracle(seed):
    c = _case(seed)
    # bucketed steps cannot re-read their gradients: clipping there needs a
    # two-pass mode (the library refuses a speculative one), which AUTO picks
    if c["buckets"] is not None and "max_norm" in c["hyper_kw"]:
        c["mode"] = 0
    st = run_case(c["psi"], c["n"], c["stage"], c["dtype"], steps=3, align=c["align"], mode=c["mode"],
                  double_buffer=c["double_buffer"], loss_scale=c["loss_scale"], hyper_kw=c["hyper_kw"],
                  buckets=c["buckets"], inject=c["inject"], sigma=c["sigma"], seed=c["seed"], fused=c["fused"])
    st.check()
    if "max_norm" not in c["hyper_kw"]:
        assert st.mismatches == 0, (c, st)


def _quantize_rows(rows, L, dt, bits):
    import torch
    from zero_partitioned_mixed_gb300 import _binding as B
    nb = (L + 255) // 256
    codes, scales = [], []
    for src in rows:
        c = torch.zeros(max(16, (L + 15) // 16 * 16), dtype=torch.uint8, device="cuda")
        s = torch.zeros(max(2, 2 * nb), dtype=torch.float32, device="cuda")
        B.zero_quantize_blocks(B.ZERO_BF16 if dt == "bf16" else B.ZERO_FP16, bits, src, L, c, s)
        codes.append(c)
        scales.append(s)
    return codes, scales


@pytest.mark.parametrize("seed", range(60))
def test_random_zeropp_step_matches_oracle(seed):
    # ZeRO-3 steps whose reduce-scatter takes the ranks' quantized gradients,
    # at random shapes, bucket layouts, code widths and modes, with overflow
    import torch

    import oracle as O
    from _parity import bits16, bits32
    from zero_partitioned_mixed_gb300 import _binding as B
    from zero_partitioned_mixed_gb300 import synth as S
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.choice([1, 2, 3, 4, 5, 8]))
    align = int(rng.choice([1, 2, 8]))
    psi = int(rng.integers(1, 40_000))
    dt = str(rng.choice(["fp16", "bf16"]))
    bits = int(rng.choice([8, 4]))
    db = bool(rng.integers(0, 2))
    part = O.partition(psi, n, align)
    P = part.psi_pad
    buckets = _buckets(rng, P, int(rng.choice([1, 8])))
    buf = RankBuffers(psi, n, 3, dt, align=align, double_buffer=db)
    td = S.torch_dtype(dt)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    master = torch.randn(psi, generator=g, device="cuda") * 0.02
    st = O.init_state(3, dt, part, master.cpu().numpy())
    buf.state(0)[0].copy_(torch.from_numpy(st.master))
    buf.params[:P].copy_(torch.from_numpy(st.params.view(np.int16)).view(td))
    hb, ho = B.hyper(weight_decay=0.05), O.Hyper(weight_decay=0.05)
    bad_step = int(rng.integers(0, 4))
    for step in range(3):
        grads = torch.zeros((n, max(8, (P + 7) // 8 * 8)), dtype=td, device="cuda")
        grads[:, :psi] = (torch.randn((n, psi), generator=g, device="cuda") * 1e-2).to(td)
        if step == bad_step:
            grads[int(rng.integers(0, n)), int(rng.integers(0, psi))] = float("inf")
        gb = bits16(grads)
        for (a, b) in reversed(buckets):
            L = b - a
            rows = []
            for r in range(n):
                src = torch.zeros(max(8, (L + 7) // 8 * 8), dtype=td, device="cuda")
                src[:L].copy_(grads[r, a:b])
                rows.append(src[:L])
            codes, scales = _quantize_rows(rows, L, dt, bits)
            B.zero_reduce_scatter_bucket_q(buf.h, a, b, bits, codes, scales, buf.master, buf.m, buf.v,
                                           buf.params, hb)
        buf.step(hb)
        st, res = O.step_stage3_quantized(st, [gb[:, a:b] for (a, b) in buckets], buckets, ho, bits)
        s = buf.status()
        assert bool(s["overflow"]) == res.overflow and s["steps_applied"] == st.t
        if res.applied:
            assert abs(s["grad_norm"] - res.norm) <= 1e-5 * res.norm
        gm, gmm, gv = buf.state(s["state_slot"])
        assert np.array_equal(bits32(gm), st.master.view(np.uint32))
        assert np.array_equal(bits32(gmm), st.m.view(np.uint32))
        assert np.array_equal(bits32(gv), st.v.view(np.uint32))
        assert np.array_equal(bits16(buf.params[:P]), st.params)
    buf.close()


@pytest.mark.parametrize("seed", range(120))
def test_random_shapes_write_nothing_outside_their_buffers(seed):
    # every buffer a call touches sits between sentinel bands; random stages,
    # shapes, modes (the staged one included), bucket layouts, fused or
    # separate ZeRO-3 backward, ZeRO++ calls; two steps, one with an overflow
    import torch

    from test_gpu_guard_bands import Guarded
    from zero_partitioned_mixed_gb300 import _binding as B
    rng = np.random.default_rng(2000 + seed)
    G = Guarded()
    stage = int(rng.choice([0, 1, 2, 3]))
    n = int(rng.choice([1, 2, 3, 4, 5, 8, 19]))
    align = int(rng.choice([1, 2, 8]))
    psi = int(rng.integers(1, 30_000))
    db = stage != 0 and bool(rng.integers(0, 2))
    dt, td = (B.ZERO_BF16, torch.bfloat16) if rng.integers(0, 2) else (B.ZERO_FP16, torch.float16)
    h = B.zero_init_partition(psi, n, stage, dt, align, B.ZERO_F_DOUBLE_BUFFER if db else 0)
    P = B.zero_partition_info(h)[0]
    rows = n if stage == 0 else (2 if db else 1)
    master, m, v = (G.tensor(rows * P, torch.float32) for _ in range(3))
    master[:psi].normal_(0, 0.02)
    hyp_kw = {"max_norm": 1e-3} if rng.integers(0, 3) == 0 else {}
    try:
        for step in range(2):
            inf_at = int(rng.integers(0, psi)) if step == 1 else -1
            if stage in (0, 1, 2) and not (stage == 2 and rng.integers(0, 2)):
                # stage 0 keeps g_hat in the workspace: AUTO or the workspace two-pass mode
                modes = [0, 1] if stage == 0 else (
                    [0, 1, 2] + ([3] if db else []) + ([4] if db and P % 8 == 0 and n <= 19 else []))
                mode = int(rng.choice(modes))
                grads = [G.tensor(P, td) for _ in range(n)]
                params = [G.tensor(P, td) for _ in range(n)]
                for gr in grads:
                    gr[:psi].copy_(torch.randn(psi, device="cuda").mul_(1e-2))
                if inf_at >= 0:
                    grads[0][inf_at] = float("inf")
                B.zero_step(h, grads, params, master, m, v, B.hyper(mode=mode, **hyp_kw))
            elif stage == 2:
                params = [G.tensor(P, td) for _ in range(n)]
                for (a, b) in reversed(_buckets(rng, P, int(rng.choice([1, 8])))):
                    L = b - a
                    gr = [G.tensor(L, td) for _ in range(n)]
                    for t in gr:
                        t.copy_(torch.randn(L, device="cuda").mul_(1e-2))
                    if a <= inf_at < b:
                        gr[0][inf_at - a] = float("inf")
                    B.zero_reduce_scatter_bucket_replicas(h, a, b, gr, master, m, v, params, B.hyper(**hyp_kw))
                B.zero_step(h, None, params, master, m, v, B.hyper(**hyp_kw))
            else:
                shard = G.tensor(P, td)
                back = list(reversed(_buckets(rng, P, int(rng.choice([1, 8])))))
                fused = bool(rng.integers(0, 2))
                quant = int(rng.choice([0, 0, 8, 4]))
                out0 = [G.tensor(back[0][1] - back[0][0], td) for _ in range(n)]
                B.zero_gather_bucket(h, back[0][0], back[0][1], shard, out0)
                for k, (a, b) in enumerate(back):
                    L = b - a
                    gr = [G.tensor(L, td) for _ in range(n)]
                    for t in gr:
                        t.copy_(torch.randn(L, device="cuda").mul_(1e-2))
                    if a <= inf_at < b:
                        gr[0][inf_at - a] = float("inf")
                    nxt = back[k + 1] if k + 1 < len(back) else None
                    if quant:
                        nb = (L + 255) // 256
                        codes = [G.tensor(L if quant == 8 else (L + 1) // 2, torch.uint8) for _ in range(n)]
                        scales = [G.tensor(2 * nb, torch.float32) for _ in range(n)]
                        for r in range(n):
                            B.zero_quantize_blocks(dt, quant, gr[r], L, codes[r], scales[r])
                        B.zero_reduce_scatter_bucket_q(h, a, b, quant, codes, scales, master, m, v, shard,
                                                       B.hyper(**hyp_kw))
                        if nxt:
                            qc = [G.tensor(nxt[1] - nxt[0], torch.uint8) for _ in range(n)]
                            qs = [G.tensor(2 * ((nxt[1] - nxt[0] + 255) // 256), torch.float32) for _ in range(n)]
                            B.zero_gather_bucket_q8(h, nxt[0], nxt[1], shard, qc, qs)
                    elif fused and nxt:
                        outs = [G.tensor(nxt[1] - nxt[0], td) for _ in range(n)]
                        B.zero_reduce_scatter_gather_bucket(h, a, b, gr, master, m, v, shard, B.hyper(**hyp_kw),
                                                            nxt[0], nxt[1], outs)
                    else:
                        B.zero_reduce_scatter_bucket(h, a, b, gr, master, m, v, shard, B.hyper(**hyp_kw))
                        if nxt:
                            outs = [G.tensor(nxt[1] - nxt[0], td) for _ in range(n)]
                            B.zero_gather_bucket(h, nxt[0], nxt[1], shard, outs)
                B.zero_step(h, None, [shard], master, m, v, B.hyper(**hyp_kw))
        torch.cuda.synchronize()
        G.check()
    finally:
        B.zero_destroy(h)
