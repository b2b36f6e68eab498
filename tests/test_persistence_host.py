"""Host logic of parameter persistence (no GPU): the package's flat layout
and buckets agree with the oracle's layout on the model lists and on
random lists."""

import numpy as np

import oracle as O
from zero_partitioned_mixed_gb300 import synth as S
from zero_partitioned_mixed_gb300.persistence import persistent_layout, tensor_buckets


def _check(shapes, thr, n=8):
    lay = persistent_layout(shapes, thr)
    sizes = [S.numel(s) for _, s in shapes]
    order, p0, psi = O.persistent_layout(sizes, thr)
    assert list(lay.order) == order and lay.p0 == p0 and lay.psi == psi
    pos = 0
    for i in order:
        assert lay.ranges[shapes[i][0]] == (pos, pos + sizes[i])
        pos += sizes[i]
    pp = O.partition(psi, n, 8).psi_pad if psi else 0
    bk = tensor_buckets(lay, pp)
    if pp:
        assert bk[0][0] == 0 and bk[-1][1] == pp
        assert all(bk[i][1] == bk[i + 1][0] for i in range(len(bk) - 1))
        b0 = lay.persistent_from(pp)
        assert all(not (a < b0 < b) for a, b in bk)
    return lay, bk


def test_model_lists_at_the_guide_threshold():
    lay, bk = _check(S.gpt2_small_shapes(), 100_000)
    assert lay.n_persistent == 98 and lay.psi_persistent == 121_344 and len(bk) == 148 - 98 + 1
    lay, bk = _check(S.llama7b_shapes(), 100_000)
    assert lay.n_persistent == 65 and lay.psi_persistent == 266_240 and len(bk) == 291 - 65 + 1


def test_random_lists():
    rng = np.random.default_rng(2)
    for _ in range(100):
        k = int(rng.integers(1, 15))
        shapes = [(f"t{i}", (int(rng.integers(1, 50)),)) for i in range(k)]
        _check(shapes, int(rng.integers(0, 60)), n=int(rng.integers(1, 5)))
