"""ZeRO-3 with param_persistence_threshold through Zero3Schedule, against the
oracle: small tensors laid out last keep N resident 16-bit copies, are never
gathered per bucket, are reduce-scattered after backward and refreshed after
each update.  Final states, shards, resident copies and what the forward
callbacks see must match the oracle bit for bit, with and without prefetch,
and replayed from a CUDA graph."""

import numpy as np
import pytest
import torch

import oracle as O
from _parity import bits16, bits32
from zero_partitioned_mixed_gb300 import _binding as B
from zero_partitioned_mixed_gb300.buffers import RankBuffers
from zero_partitioned_mixed_gb300.persistence import persistent_layout, tensor_buckets
from zero_partitioned_mixed_gb300.schedule import Zero3Schedule

pytestmark = pytest.mark.gpu

N = 4
THRESHOLD = 300


def _shapes():
    d, ffn, vocab, ctx = 64, 256, 500, 128
    out = [("wte", (vocab, d)), ("wpe", (ctx, d))]
    for i in range(3):
        out += [(f"h{i}.ln_1.w", (d,)), (f"h{i}.ln_1.b", (d,)), (f"h{i}.attn.w", (3 * d, d)),
                (f"h{i}.attn.b", (3 * d,)), (f"h{i}.proj.w", (d, d)), (f"h{i}.proj.b", (d,)),
                (f"h{i}.ln_2.w", (d,)), (f"h{i}.ln_2.b", (d,)), (f"h{i}.fc.w", (ffn, d)),
                (f"h{i}.fc.b", (ffn,)), (f"h{i}.fc2.w", (d, ffn)), (f"h{i}.fc2.b", (d,))]
    out += [("ln_f.w", (d,)), ("ln_f.b", (d,)), ("odd", (37,))]
    return out


def _setup(threshold, seed=3):
    lay = persistent_layout(_shapes(), threshold)
    psi = lay.psi
    part = O.partition(psi, N, 8)
    P = part.psi_pad
    buckets = tensor_buckets(lay, P)
    buf = RankBuffers(psi, N, 3, "bf16", double_buffer=True)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    master = torch.randn(psi, generator=g, device="cuda") * 0.02
    st = O.init_state(3, "bf16", part, master.cpu().numpy())
    mv, _, _ = buf.state(0)
    mv.copy_(torch.from_numpy(st.master))
    buf.params[:P].copy_(torch.from_numpy(st.params.view(np.int16)).view(torch.bfloat16))
    steps = []
    for k in range(3):
        gr = torch.zeros((N, P), dtype=torch.bfloat16, device="cuda")
        gr[:, :psi] = (torch.randn((N, psi), generator=g, device="cuda") * 1e-2).to(torch.bfloat16)
        if k == 1:
            gr[2, lay.p0 + 5] = float("inf")          # an overflow inside the persistent region
        steps.append(gr)
    lmax = max(b - a for a, b in buckets)
    gb = [torch.zeros((N, max(8, (lmax + 7) // 8 * 8)), dtype=torch.bfloat16, device="cuda")
          for _ in buckets]
    return lay, part, buckets, buf, st, steps, gb


def _load(steps, k, buckets, gb):
    for i, (a, b) in enumerate(buckets):
        gb[i][:, :b - a].copy_(steps[k][:, a:b])


@pytest.mark.parametrize("prefetch,graph", [(False, False), (True, False), (True, True)])
def test_persistent_schedule_matches_oracle(prefetch, graph):
    lay, part, buckets, buf, st, steps, gb = _setup(THRESHOLD)
    P = part.psi_pad
    p0 = lay.persistent_from(P)
    assert 0 < p0 < lay.psi and lay.n_persistent == 3 * 8 + 3
    sched = Zero3Schedule(buf, buckets, prefetch=prefetch, persistent_from=p0)
    fwd_seen = []

    def fwd(i, rows):
        a, b = buckets[i]
        assert b <= p0
        fwd_seen.append((i, [bits16(rows[r][:b - a]) for r in range(N)],
                         [bits16(x[:P - p0]) for x in sched.resident_rows()]))

    grads = lambda i: [gb[i][r] for r in range(N)]
    g = None
    for k in range(3):
        _load(steps, k, buckets, gb)
        if graph and k == 1:
            g = sched.capture(B.hyper(weight_decay=0.01), grads)
        if g is not None:
            g.replay()
        else:
            sched.step(B.hyper(weight_decay=0.01), grads, forward=None if graph else fwd)
    torch.cuda.synchronize()
    # the oracle, step by step
    ho = O.Hyper(weight_decay=0.01)
    gbits = [bits16(s) for s in steps]
    ost = st
    fwd_want = []
    for k in range(3):
        before = ost.params.copy()
        reps_before = [before[p0:P]] * N
        ost, res, reps = O.step_stage3_persistent(ost, [gbits[k][:, a:b] for (a, b) in buckets], buckets, ho, p0)
        assert res.overflow == (k == 1)
        gathered = [i for i, (a, b) in enumerate(buckets) if b <= p0]
        fwd_want += [(i, res.gathered_fwd[j], reps_before) for j, i in enumerate(gathered)]
    s = buf.status()
    m, mm, vv = buf.state(s["state_slot"])
    assert np.array_equal(bits32(m), ost.master.view(np.uint32))
    assert np.array_equal(bits32(mm), ost.m.view(np.uint32))
    assert np.array_equal(bits32(vv), ost.v.view(np.uint32))
    assert np.array_equal(bits16(buf.params)[:P], ost.params)
    res_rows = sched.resident_rows()
    for r in range(N):
        assert np.array_equal(bits16(res_rows[r][:P - p0]), reps[r])
    assert s["steps_applied"] == 2 and s["overflow"] == 0
    if not graph:
        assert len(fwd_seen) == len(fwd_want)
        for (i, rows, res_now), (j, want_rows, want_res) in zip(fwd_seen, fwd_want):
            assert i == j
            for r in range(N):
                assert np.array_equal(rows[r], want_rows[r])
                assert np.array_equal(res_now[r], want_res[r])
    buf.close()


def test_threshold_zero_is_plain_zero3():
    # nothing persistent: no resident copies, every tensor gathered
    lay, part, buckets, buf, st, steps, gb = _setup(0)
    assert lay.p0 == lay.psi and lay.n_persistent == 0
    sched = Zero3Schedule(buf, buckets, prefetch=True, persistent_from=lay.persistent_from(part.psi_pad))
    assert sched.resident is None and len(sched.gathered) == len(buckets)
    for k in range(3):
        _load(steps, k, buckets, gb)
        sched.step(B.hyper(), lambda i: [gb[i][r] for r in range(N)])
    torch.cuda.synchronize()
    ost = st
    for k in range(3):
        ost, _ = O.step_stage3(ost, [bits16(steps[k])[:, a:b] for (a, b) in buckets], buckets, O.Hyper())
    m, _, _ = buf.state(buf.status()["state_slot"])
    assert np.array_equal(bits32(m), ost.master.view(np.uint32))
    buf.close()


def test_all_persistent():
    # every tensor below the threshold: no gather at all during the passes
    lay, part, buckets, buf, st, steps, gb = _setup(10 ** 9)
    assert lay.p0 == 0 and buckets == [(0, part.psi_pad)]
    sched = Zero3Schedule(buf, buckets, prefetch=True, persistent_from=lay.persistent_from(part.psi_pad))
    assert sched.gathered == []
    _load(steps, 0, buckets, gb)
    sched.step(B.hyper(), lambda i: [gb[i][r] for r in range(N)])
    torch.cuda.synchronize()
    ost, res, reps = O.step_stage3_persistent(st, [bits16(steps[0])], buckets, O.Hyper(), 0)
    for r in range(N):
        assert np.array_equal(bits16(sched.resident_rows()[r][:part.psi_pad]), reps[r])
    buf.close()


def test_straddling_bucket_is_refused():
    lay, part, buckets, buf, st, steps, gb = _setup(THRESHOLD)
    with pytest.raises(ValueError):
        Zero3Schedule(buf, [(0, lay.p0 + 8), (lay.p0 + 8, part.psi_pad)], persistent_from=lay.p0)
    buf.close()
