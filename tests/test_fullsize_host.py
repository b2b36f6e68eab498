"""The full-size checker's per-chunk work on the CPU: chunks of a step the
oracle itself computed pass with no mismatch and the oracle's norm, and a
planted one-ulp error, a wrong replica or a changed state is found."""

import math

import numpy as np

import oracle as O
from _fullsize import Tally, _check_chunk


def _case(psi=1_000, n=4, seed=3):
    rng = np.random.default_rng(seed)
    part = O.partition(psi, n, 8)
    master = rng.normal(0, 0.02, psi).astype(np.float32)
    m = rng.normal(0, 1e-4, psi).astype(np.float32)
    v = np.abs(rng.normal(0, 1e-6, psi)).astype(np.float32)
    st = O.init_state(1, O.BF16, part, master, m, v, loss_scale=8.0)
    g = np.zeros((n, part.psi_pad), np.float32)
    g[:, :psi] = rng.normal(0, 1e-2, (n, psi)) * 8.0
    gb = O.rne16(g, O.BF16)
    h = O.Hyper(weight_decay=0.1)
    new, res = O.step(st, gb, h)
    return part, st, new, res, gb, h


def _run(part, st, new, res, gb, h, chunk, params=None, digest=False):
    tal = Tally()
    P = part.psi_pad
    params = new.params if params is None else params
    sc = O.step_scalars(h, 1)
    for s in range(0, P, chunk):
        e = min(P, s + chunk)
        tal.merge(_check_chunk(s, part.psi, part.shard, part.n_ranks, O.BF16, gb[:, s:e],
                               [st.master[s:e], st.m[s:e], st.v[s:e]], [new.master[s:e], new.m[s:e], new.v[s:e]],
                               params[:, s:e], 8.0, sc, None, digest))
    return tal


def test_oracle_step_passes_in_any_chunking():
    part, st, new, res, gb, h = _case()
    for chunk in (part.psi_pad, 256, 100, 7):
        tal = _run(part, st, new, res, gb, h, chunk)
        assert tal.mismatches == 0 and not tal.bad
        assert tal.compared == (3 + part.n_ranks) * part.psi_pad
        assert math.isclose(tal.norm(part.n_ranks), res.norm, rel_tol=1e-12)


def test_planted_errors_are_found():
    part, st, new, res, gb, h = _case()
    bad = new.copy()
    bad.m[123] = np.nextafter(bad.m[123], np.float32(1))
    tal = _run(part, st, bad, res, gb, h, 256)
    assert tal.mismatches == 1 and tal.max_ulp32 == 1
    q = new.params.copy()
    q[2, 999] ^= 1
    tal = _run(part, st, new, res, gb, h, 256, params=q)
    assert tal.mismatches == 1 and tal.max_ulp16 == 1
    # a non-finite gradient is seen as an overflow
    g2 = gb.copy()
    g2[1, 500] = O.rne16(np.array([np.inf], np.float32), O.BF16)[0]
    out = _check_chunk(0, part.psi, part.shard, part.n_ranks, O.BF16, g2, None, None, None, 8.0, None, None,
                       False)
    assert out["bad"]


def test_digests_tell_changed_state():
    part, st, new, res, gb, h = _case()
    a = _run(part, st, new, res, gb, h, 128, digest=True)
    b = _run(part, st, new, res, gb, h, 128, digest=True)
    assert a.digests == b.digests and len(a.digests) == (3 + part.n_ranks) * ((part.psi_pad + 127) // 128)
    changed = new.copy()
    changed.v[7] = np.float32(0.5)
    c = Tally()
    P = part.psi_pad
    for s in range(0, P, 128):
        e = min(P, s + 128)
        c.merge(_check_chunk(s, part.psi, part.shard, part.n_ranks, O.BF16, None, None,
                             [changed.master[s:e], changed.m[s:e], changed.v[s:e]], changed.params[:, s:e],
                             8.0, None, None, True))
    assert c.digests != a.digests
