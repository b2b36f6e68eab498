"""Out-of-bounds writes would show as changed guard bands.

Every buffer the kernels touch is carved out of a larger allocation with
4 KiB sentinel regions before and after it, filled with a bit pattern.
After steps of every stage and mode (vector and element-wise paths,
ragged sizes, overflow and clipping, ZeRO-3 and ZeRO++ buckets) the
sentinels must be unchanged.  (A stand-in for a memory checker.)
"""

import pytest
import torch

from zero_partitioned_mixed_gb300 import _binding as B

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side
PATTERN = 0x5A


class Guarded:
    def __init__(self):
        self.allocs = []

    def tensor(self, numel, dtype):
        esz = torch.empty((), dtype=dtype).element_size()
        g = GUARD // esz
        raw = torch.empty(numel + 2 * g, dtype=dtype, device="cuda")
        raw.view(torch.uint8).fill_(PATTERN)
        inner = raw[g:g + numel]
        inner.zero_()
        self.allocs.append((raw, g, numel))
        return inner

    def check(self):
        for raw, g, numel in self.allocs:
            b = raw.view(torch.uint8)
            esz = raw.element_size()
            head, tail = b[:g * esz], b[(g + numel) * esz:]
            assert bool((head == PATTERN).all()) and bool((tail == PATTERN).all()), "guard band overwritten"


def _round8(x):
    return (x + 7) // 8 * 8


@pytest.mark.parametrize("psi,n,align", [(100_003, 8, 8), (1001, 3, 1), (5, 2, 2), (64, 1, 8)])
@pytest.mark.parametrize("stage,mode,db", [(0, 0, False), (1, 3, True), (2, 1, False), (2, 2, False),
                                           (2, 3, True)])
def test_no_writes_outside_buffers_stages_0_to_2(psi, n, align, stage, mode, db):
    G = Guarded()
    dt = B.ZERO_BF16
    h = B.zero_init_partition(psi, n, stage, dt, align, B.ZERO_F_DOUBLE_BUFFER if db else 0)
    P = B.zero_partition_info(h)[0]
    grads = [G.tensor(P, torch.bfloat16) for _ in range(n)]
    params = [G.tensor(P, torch.bfloat16) for _ in range(n)]
    rows = n if stage == 0 else (2 if db else 1)
    master, m, v = (G.tensor(rows * P, torch.float32) for _ in range(3))
    torch.manual_seed(psi)
    for g in grads:
        g[:psi].copy_(torch.randn(psi, device="cuda").mul_(1e-2))
    master[:psi].normal_(0, 0.02)
    if stage != 0:
        for r in range(n):
            params[r].copy_(master[:P].to(torch.bfloat16))
    # a plain step, a step that clips (speculative: redone), a step that overflows
    for k, hyp in enumerate([B.hyper(mode=mode), B.hyper(mode=mode, max_norm=1e-3),
                             B.hyper(mode=mode, max_norm=1e-3)]):
        if k == 2:
            grads[0][min(3, psi - 1)] = float("inf")
        B.zero_step(h, grads, params, master, m, v, hyp)
    torch.cuda.synchronize()
    G.check()
    B.zero_destroy(h)


@pytest.mark.parametrize("db", [True, False])
def test_no_writes_outside_buffers_stage3_and_zeropp(db):
    G = Guarded()
    psi, n = 70_001, 4
    h = B.zero_init_partition(psi, n, 3, B.ZERO_FP16, 8, B.ZERO_F_DOUBLE_BUFFER if db else 0)
    P = B.zero_partition_info(h)[0]
    shard = G.tensor(P, torch.float16)
    master, m, v = (G.tensor((2 if db else 1) * P, torch.float32) for _ in range(3))
    master[:psi].normal_(0, 0.02)
    shard.copy_(master[:P].to(torch.float16))
    buckets = [(0, 30_000), (30_000, 30_005), (30_005, 61_000), (61_000, P)]
    hyp = B.hyper()
    for step in range(2):
        for (a, b) in buckets:
            L = b - a
            outs = [G.tensor(L, torch.float16) for _ in range(n)]
            B.zero_gather_bucket(h, a, b, shard, outs)
            codes = [G.tensor(L, torch.uint8) for _ in range(n)]
            scales = [G.tensor(2 * ((L + 255) // 256), torch.float32) for _ in range(n)]
            B.zero_gather_bucket_q8(h, a, b, shard, codes, scales)
            deq = G.tensor(L, torch.float16)
            B.zero_dequantize_blocks(B.ZERO_FP16, 8, codes[0], scales[0], L, deq)
        for (a, b) in reversed(buckets):
            L = b - a
            g = [G.tensor(L, torch.float16) for _ in range(n)]
            for t in g:
                t.copy_(torch.randn(L, device="cuda").mul_(1e-2))
            if step == 0:
                B.zero_reduce_scatter_bucket(h, a, b, g, master, m, v, shard, hyp)
            else:
                codes = [G.tensor((L + 1) // 2, torch.uint8) for _ in range(n)]
                scales = [G.tensor(2 * ((L + 255) // 256), torch.float32) for _ in range(n)]
                for r in range(n):
                    B.zero_quantize_blocks(B.ZERO_FP16, 4, g[r], L, codes[r], scales[r])
                B.zero_reduce_scatter_bucket_q(h, a, b, 4, codes, scales, master, m, v, shard, hyp)
        B.zero_step(h, None, [shard], master, m, v, hyp)
    torch.cuda.synchronize()
    G.check()
    B.zero_destroy(h)


@pytest.mark.parametrize("psi,n", [(100_003, 8), (5, 2), (64, 1), (300_000, 19)])
def test_no_writes_outside_buffers_staged_step(psi, n):
    G = Guarded()
    h = B.zero_init_partition(psi, n, 1, B.ZERO_FP16, 8, B.ZERO_F_DOUBLE_BUFFER)
    P = B.zero_partition_info(h)[0]
    grads = [G.tensor(P, torch.float16) for _ in range(n)]
    params = [G.tensor(P, torch.float16) for _ in range(n)]
    master, m, v = (G.tensor(2 * P, torch.float32) for _ in range(3))
    torch.manual_seed(psi)
    for g in grads:
        g[:psi].copy_(torch.randn(psi, device="cuda").mul_(1e-2))
    master[:psi].normal_(0, 0.02)
    for r in range(n):
        params[r].copy_(master[:P].to(torch.float16))
    mode = B.ZERO_MODE_SPECULATIVE_STAGED
    for k, hyp in enumerate([B.hyper(mode=mode), B.hyper(mode=mode, max_norm=1e-3),
                             B.hyper(mode=mode, max_norm=1e-3)]):
        if k == 2:
            grads[n - 1][min(3, psi - 1)] = float("inf")
        B.zero_step(h, grads, params, master, m, v, hyp)
    torch.cuda.synchronize()
    G.check()
    B.zero_destroy(h)


@pytest.mark.parametrize("db", [True, False])
@pytest.mark.parametrize("n", [2, 8])
def test_no_writes_outside_buffers_fused_backward(db, n):
    # ZeRO-3 backward through zero_reduce_scatter_gather_bucket: one launch for
    # 8-aligned bucket pairs, two calls otherwise; guarded gradient rows,
    # gather outputs, shard and state
    G = Guarded()
    psi = 70_001
    h = B.zero_init_partition(psi, n, 3, B.ZERO_BF16, 8, B.ZERO_F_DOUBLE_BUFFER if db else 0)
    P = B.zero_partition_info(h)[0]
    shard = G.tensor(P, torch.bfloat16)
    master, m, v = (G.tensor((2 if db else 1) * P, torch.float32) for _ in range(3))
    master[:psi].normal_(0, 0.02)
    shard.copy_(master[:P].to(torch.bfloat16))
    # step 0: 8-aligned buckets (each pair one launch); step 1: unaligned ones (two calls)
    layouts = [[(0, 30_000), (30_000, 30_008), (30_008, 61_000), (61_000, P)],
               [(0, 30_000), (30_000, 30_005), (30_005, 61_000), (61_000, P)]]
    hyp = B.hyper()
    for step in range(2):
        back = list(reversed(layouts[step]))
        first = back[0]
        B.zero_gather_bucket(h, first[0], first[1], shard, [G.tensor(first[1] - first[0], torch.bfloat16)
                                                          for _ in range(n)])
        for k, (a, b) in enumerate(back):
            L = b - a
            g = [G.tensor(L, torch.bfloat16) for _ in range(n)]
            for t in g:
                t.copy_(torch.randn(L, device="cuda").mul_(1e-2))
            if k + 1 < len(back):
                ga, gb = back[k + 1]
                outs = [G.tensor(gb - ga, torch.bfloat16) for _ in range(n)]
                B.zero_reduce_scatter_gather_bucket(h, a, b, g, master, m, v, shard, hyp, ga, gb, outs)
            else:
                B.zero_reduce_scatter_bucket(h, a, b, g, master, m, v, shard, hyp)
        B.zero_step(h, None, [shard], master, m, v, hyp)
    torch.cuda.synchronize()
    G.check()
    B.zero_destroy(h)
