"""ZeRO-3 schedule: gathers prefetched one bucket ahead on a side stream, and
the whole step captured into a CUDA graph and replayed.  Both must give the
same bits as the plain sequential schedule (and the oracle)."""

import numpy as np
import pytest
import torch

import oracle as O
from _parity import bits16, bits32
from zero_partitioned_mixed_gb300 import _binding as B
from zero_partitioned_mixed_gb300.buffers import RankBuffers
from zero_partitioned_mixed_gb300.schedule import Zero3Schedule

pytestmark = pytest.mark.gpu

PSI, N = 300_001, 4


def _setup(double_buffer=True):
    part = O.partition(PSI, N, 8)
    P = part.psi_pad
    buckets = [(0, 70_000), (70_000, 70_008), (70_008, 190_000), (190_000, 190_003), (190_003, P)]
    buf = RankBuffers(PSI, N, 3, "bf16", double_buffer=double_buffer)
    g = torch.Generator(device="cuda")
    g.manual_seed(99)
    master = torch.randn(PSI, generator=g, device="cuda") * 0.02
    st = O.init_state(3, "bf16", part, master.cpu().numpy())
    mv, _, _ = buf.state(0)
    mv.copy_(torch.from_numpy(st.master))
    buf.params[:P].copy_(torch.from_numpy(st.params.view(np.int16)).view(torch.bfloat16))
    # fixed per-bucket gradient buffers (the caller's backward would fill them)
    grads = torch.zeros((N, buf.stride), dtype=torch.bfloat16, device="cuda")
    grads[:, :PSI] = (torch.randn((N, PSI), generator=g, device="cuda") * 1e-2).to(torch.bfloat16)
    gb = []
    for (a, b) in buckets:
        t = torch.zeros((N, max(8, (b - a + 7) // 8 * 8)), dtype=torch.bfloat16, device="cuda")
        t[:, :b - a].copy_(grads[:, a:b])
        gb.append(t)
    return part, buckets, buf, st, grads, gb


def _state(buf):
    s = buf.status()
    m, mm, vv = buf.state(s["state_slot"])
    return bits32(m), bits32(mm), bits32(vv), bits16(buf.params), s


@pytest.mark.parametrize("double_buffer", [True, False])
def test_prefetch_matches_sequential_and_oracle(double_buffer):
    h = B.hyper(weight_decay=0.01)
    results = []
    # sequential, side-stream prefetch, and backward gathers fused into the reduce-scatters
    for prefetch, fuse in ((False, False), (True, False), (False, True), (True, True)):
        part, buckets, buf, st, grads, gb = _setup(double_buffer)
        sched = Zero3Schedule(buf, buckets, prefetch=prefetch, fuse=fuse)
        seen = []

        def fwd(i, rows):
            a, b = buckets[i]
            seen.append(all(torch.equal(rows[r][:b - a], buf.params[a:b]) for r in range(N)))

        for _ in range(3):
            sched.step(h, lambda i: [gb[i][r] for r in range(N)], forward=fwd, backward=fwd)
        torch.cuda.synchronize()
        assert all(seen) and len(seen) == 3 * 2 * len(buckets)
        results.append(_state(buf))
        buf.close()
    for other in results[1:]:
        for x, y in zip(results[0][:4], other[:4]):
            assert np.array_equal(x, y)
    # and the oracle
    part, buckets, buf, st, grads, gb = _setup(double_buffer)
    gbits = bits16(grads)
    ho = O.Hyper(weight_decay=0.01)
    for _ in range(3):
        st, _ = O.step_stage3(st, [gbits[:, a:b] for (a, b) in buckets], buckets, ho)
    assert np.array_equal(results[1][0], st.master.view(np.uint32))
    assert np.array_equal(results[1][3][:part.psi_pad], st.params)
    buf.close()


@pytest.mark.parametrize("fuse", [False, True])
def test_cuda_graph_replay_matches_eager(fuse):
    h = B.hyper(weight_decay=0.01)
    # eager: 4 steps
    part, buckets, buf, st, grads, gb = _setup()
    sched = Zero3Schedule(buf, buckets, prefetch=True, fuse=fuse)
    for _ in range(4):
        sched.step(h, lambda i: [gb[i][r] for r in range(N)])
    torch.cuda.synchronize()
    want = _state(buf)
    buf.close()
    # one eager warm-up step, capture one step, replay it three times
    part, buckets, buf, st, grads, gb = _setup()
    sched = Zero3Schedule(buf, buckets, prefetch=True, fuse=fuse)
    sched.step(h, lambda i: [gb[i][r] for r in range(N)])
    g = sched.capture(h, lambda i: [gb[i][r] for r in range(N)])
    torch.cuda.synchronize()
    s = buf.status()
    assert s["steps_applied"] == 1            # capture recorded the step but ran nothing
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    got = _state(buf)
    assert got[4]["steps_applied"] == 4 and got[4]["state_slot"] == want[4]["state_slot"]
    for x, y in zip(want[:4], got[:4]):
        assert np.array_equal(x, y)
    buf.close()


def test_stage1_step_captures_and_replays():
    # the speculative one-shot step (three launches) in a graph
    buf_e = RankBuffers(100_000, 8, 1, "fp16")
    buf_g = RankBuffers(100_000, 8, 1, "fp16")
    torch.manual_seed(1)
    for b in (buf_e, buf_g):
        b.master[:100_000].copy_(torch.linspace(-0.1, 0.1, 100_000, device="cuda"))
        b.params[:, :100_000].copy_(b.master[:100_000].to(torch.float16))
    g = (torch.randn((8, buf_e.stride), device="cuda") * 1e-2).to(torch.float16)
    g[:, 100_000:] = 0
    rows = [g[r] for r in range(8)]
    h = B.hyper(max_norm=0.5)
    for _ in range(3):
        buf_e.step(h, rows)
    buf_g.step(h, rows)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            buf_g.step(h, rows)
    torch.cuda.current_stream().wait_stream(s)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    for x, y in ((buf_e.master, buf_g.master), (buf_e.params, buf_g.params)):
        assert torch.equal(x.view(torch.int16) if x.dtype != torch.float32 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype != torch.float32 else y.view(torch.int32))
    assert buf_e.status()["steps_applied"] == buf_g.status()["steps_applied"] == 3
    buf_e.close(); buf_g.close()
