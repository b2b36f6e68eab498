"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch each one.  A pin set that lets a dropped term, a wrong sign or index,
or a swapped operand through would not pin the oracle."""

import math

import numpy as np
import pytest

import oracle
import oracle.zero_oracle as Z
import test_oracle_pins as pins


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(Z, name, fn)
    monkeypatch.setattr(oracle, name, fn, raising=False)
    monkeypatch.setattr(pins.O, name, fn, raising=False)


PIN_RUNS = [
    (pins.test_partition_brute_force, dict(n=3, align=2)),
    (pins.test_partition_toy_numbers, {}),
    (pins.test_model_state_tables_printed_on_pages, {}),
    (pins.test_exact_formulas_on_integers, {}),
    (pins.test_comm_ring_printed, {}),
    (pins.test_comm_paper_printed, {}),
    (pins.test_rne16_fp16_vectors, {}),
    (pins.test_rne16_bf16_vectors, {}),
    (pins.test_tiny_case_by_hand, dict(stage=1, dt="fp16")),
    (pins.test_tiny_case_by_hand, dict(stage=3, dt="bf16")),
    (pins.test_tiny_case_by_hand, dict(stage=0, dt="fp16")),
    (pins.test_loss_scale_divides_out, dict(stage=2)),
    (pins.test_padding_gradients_are_ignored, dict(stage=1)),
    (pins.test_padding_gradients_are_ignored, dict(stage=3)),
    (pins.test_all_stages_identical, dict(dt="bf16")),
    (pins.test_all_reduce_is_reduce_scatter_then_all_gather, {}),
    (pins.test_adam_step1_is_lr_times_sign, {}),
    (pins.test_zero_gradient_only_decays, {}),
    (pins.test_adam_against_high_precision, {}),
    (pins.test_overflow_skips_step_and_halves_scale, dict(stage=1, bad=np.inf)),
    (pins.test_overflow_skips_step_and_halves_scale, dict(stage=3, bad=np.nan)),
    (pins.test_norm_of_constant_gradient, {}),
    (pins.test_rank_sum_is_left_to_right_from_positive_zero, {}),
    (pins.test_unscale_is_one_rounded_division, {}),
    (pins.test_norm_accumulates_in_double, dict(stage=0)),
    (pins.test_norm_accumulates_in_double, dict(stage=2)),
    (pins.test_clip_scales_gradient_to_max_norm, {}),
    (pins.test_norm_sums_each_shard_left_to_right, dict(stage=1)),
    (pins.test_norm_squares_beyond_fp32_range, dict(stage=1, x=2.0 ** 100)),
    (pins.test_replicas_equal_cast_of_master, {}),
    (pins.test_quantizer_is_lossless_on_its_grid, {}),
    (pins.test_quantizer_error_bound_and_order, {}),
    (pins.test_quantizer_code_is_one_division_by_the_scale, {}),
    (pins.test_quantizer_constant_block_and_nan, {}),
    (pins.test_int4_packing, {}),
    (pins.test_quantized_reduce_scatter_equals_plain_on_grid_gradients, dict(bits=8)),
    (pins.test_persistent_layout_against_a_sort_key, {}),
    (pins.test_persistent_threshold_is_strict_and_degenerate_cases, {}),
    (pins.test_persistent_comm_and_memory_endpoints, {}),
    (pins.test_persistence_moves_no_value, dict(dt="fp16")),
    (pins.test_unpadded_toy_would_not_print_156, {}),
    (pins.test_bytes_per_param_at_32, {}),
    (pins.test_table1_model_sizes_fit_32gb, {}),
    (pins.test_ring_stage3_cell_is_the_documented_gap, {}),
    (pins.test_widen16_exact_roundtrip, {}),
    (pins.test_overflow_in_padding_is_ignored_and_scale_floor, {}),
    (pins.test_quantized_gather_reproduces_grid_weights, {}),
    (pins.test_guide_threshold_on_the_model_lists, {}),
]


def _caught() -> list:
    failed = []
    for fn, kw in PIN_RUNS:
        try:
            fn(**kw)
        except (AssertionError, ValueError, IndexError, ZeroDivisionError) as e:
            failed.append(fn.__name__)
    return failed


# ---------------------------------------------------------------- mutants
orig_adam = Z.adam_update
orig_scalars = Z.step_scalars
orig_rank_sum = Z.rank_sum
orig_unscale = Z.unscale
orig_partition = Z.partition
orig_rne16 = Z.rne16
orig_msb = Z.model_state_bytes
orig_clip = Z.clip_factor
orig_norm_shards = Z._norm_from_shards
orig_skip = Z._skip
orig_quant = Z.quantize_blocks
orig_dequant = Z.dequantize_blocks
orig_pack4 = Z.pack_int4


def adam_swapped_beta(p, m, v, g, sc):
    sc2 = Z.StepScalars(sc.a1, sc.b2, sc.b1, sc.a2, sc.eps, sc.dfac, sc.step_size, sc.bc2s)
    return orig_adam(p, m, v, g, sc2)


def adam_no_decay(p, m, v, g, sc):
    sc2 = Z.StepScalars(sc.b1, sc.b2, sc.a1, sc.a2, sc.eps, np.float32(1.0), sc.step_size, sc.bc2s)
    return orig_adam(p, m, v, g, sc2)


def adam_wrong_sign(p, m, v, g, sc):
    sc2 = Z.StepScalars(sc.b1, sc.b2, sc.a1, sc.a2, sc.eps, sc.dfac, -sc.step_size, sc.bc2s)
    return orig_adam(p, m, v, g, sc2)


def adam_eps_inside_sqrt(p, m, v, g, sc):
    p = np.asarray(p, np.float32) * sc.dfac
    m = sc.b1 * np.asarray(m, np.float32) + sc.a1 * np.asarray(g, np.float32)
    v = sc.b2 * np.asarray(v, np.float32) + sc.a2 * (np.asarray(g, np.float32) ** 2)
    den = np.sqrt(v + sc.eps) / sc.bc2s
    return (p - sc.step_size * (m / den)).astype(np.float32), m.astype(np.float32), v.astype(np.float32)


def scalars_no_bias_correction(h, t):
    s = orig_scalars(h, t)
    return Z.StepScalars(s.b1, s.b2, s.a1, s.a2, s.eps, s.dfac, np.float32(h.lr), np.float32(1.0))


def scalars_t_off_by_one(h, t):
    return orig_scalars(h, t + 1)


def rank_sum_drops_last(gs):
    return orig_rank_sum(list(gs)[:-1]) if len(gs) > 1 else orig_rank_sum(gs)


def unscale_forgets_scale(s, n, scale):
    return orig_unscale(s, n, 1.0)


def unscale_forgets_n(s, n, scale):
    return orig_unscale(s, 1, scale)


def partition_off_by_one(psi, n, align=8):
    p = orig_partition(psi, n, align)
    offs = tuple(o + (1 if i else 0) for i, o in enumerate(p.offsets))
    return Z.Partition(p.psi, p.n_ranks, p.align, p.psi_pad, p.shard, offs, p.real)


def partition_no_padding(psi, n, align=8):
    p = orig_partition(psi, n, align)
    shard = -(-psi // n) if psi else 0
    offs = tuple(r * shard for r in range(n))
    real = tuple(max(0, min(psi - o, shard)) for o in offs)
    return Z.Partition(psi, n, align, shard * n, shard, offs, real)


def rne16_truncates(x, dtype):
    if dtype == Z.BF16:
        u = np.asarray(x, np.float32).view(np.uint32)
        return (u >> np.uint32(16)).astype(np.uint16)
    return orig_rne16(x, dtype)


def msb_drops_grad_term(psi, n, stage, k=12):
    if stage == 2:
        return 2 * psi + (k * psi) // n
    return orig_msb(psi, n, stage, k)


def clip_wrong_comparison(norm, max_norm):
    if Z._f32(max_norm) <= 0.0:
        return None
    c = Z._f32(max_norm) / (norm + 1e-6)
    return np.float32(c) if c > 1.0 else None


def norm_wrong_shard_index(shards, part):
    total = 0.0
    for r, real in enumerate(part.real):
        x = np.asarray(shards[(r + 1) % part.n_ranks][:real], np.float64)
        total += float(np.sum(x * x))
    return math.sqrt(total)


def skip_keeps_scale(state):
    return state.copy()


def quant_qmax_off_by_one(x, bits, block=Z.Q_BLOCK):
    x = np.asarray(x, np.float32)
    codes, scale, lo = orig_quant(x, bits, block)
    scale = scale * np.float32(((1 << bits) - 1) / (1 << bits))
    k = np.arange(x.size) // block
    q = np.where(scale[k] != 0, np.rint((x - lo[k]) / np.where(scale[k] != 0, scale[k], 1)), 0)
    return np.clip(q, 0, (1 << bits) - 1).astype(np.uint8), scale, lo


def quant_floor(x, bits, block=Z.Q_BLOCK):
    x = np.asarray(x, np.float32)
    codes, scale, lo = orig_quant(x, bits, block)
    k = np.arange(x.size) // block
    q = np.where(scale[k] != 0, np.floor((x - lo[k]) / np.where(scale[k] != 0, scale[k], 1) - 0.25), 0)
    return np.clip(q, 0, (1 << bits) - 1).astype(np.uint8), scale, lo


def quant_multiplies_by_inverse(x, bits, block=Z.Q_BLOCK):
    # codes from (x - lo) * f32((2^bits - 1) / (hi - lo)) instead of (x - lo) / scale
    x = np.asarray(x, np.float32)
    codes, scale, lo = orig_quant(x, bits, block)
    qmax = np.float32((1 << bits) - 1)
    out = np.zeros(x.size, np.uint8)
    for b in range(scale.size):
        blk = x[b * block:(b + 1) * block]
        if scale[b] == 0:
            continue
        with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
            inv = qmax / np.float32(np.float32(blk.max() + np.float32(0)) - lo[b])
            q = np.rint((blk - lo[b]) * inv)
        q = np.where(np.isnan(q), 0, q)
        out[b * block:(b + 1) * block] = np.clip(q, 0, qmax).astype(np.uint8)
    return out, scale, lo


def dequant_forgets_lo(codes, scale, lo, block=Z.Q_BLOCK):
    return orig_dequant(codes, scale, np.zeros_like(lo), block)


def pack4_swapped_nibbles(codes):
    c = np.asarray(codes, np.uint8)
    if c.size % 2:
        c = np.concatenate([c, np.zeros(1, np.uint8)])
    return (c[1::2] & 0x0F) | ((c[0::2] & 0x0F) << 4)


def persist_threshold_inclusive(sizes, threshold):
    # "<=" instead of "<": a tensor of exactly the threshold becomes persistent
    big = [i for i, n in enumerate(sizes) if n > threshold]
    small = [i for i, n in enumerate(sizes) if n <= threshold]
    return big + small, sum(sizes[i] for i in big), sum(sizes)


def persist_small_first(sizes, threshold):
    # the region placed at the front instead of the end
    big = [i for i, n in enumerate(sizes) if not n < threshold]
    small = [i for i, n in enumerate(sizes) if n < threshold]
    return small + big, sum(sizes[i] for i in small), sum(sizes)


def persist_comm_no_refresh(psi, psi_pers):
    return 2 * (psi - psi_pers) + psi


def persist_ring_no_refresh(psi, psi_pers, n_ranks):
    return (n_ranks - 1) * (3 * psi - 2 * psi_pers) // n_ranks


def persist_msb_no_replicas(psi, psi_pers, n_ranks, k=12):
    return ((4 + k) * psi) // n_ranks


def persist_step_stale_replicas(state, bucket_grads, buckets, h, p0):
    # the persistent copies left at the values before the update
    pp = state.part.psi_pad
    old = [state.params[p0:pp].copy() for _ in range(state.part.n_ranks)]
    out, res = Z.step_stage3(state, bucket_grads, buckets, h)
    return out, res, old


def rank_sum_reversed(grads_f32):
    s = np.zeros(np.asarray(grads_f32[0]).shape, np.float32)
    for g in reversed(list(grads_f32)):
        s = s + np.asarray(g, np.float32)
    return s


def rank_sum_from_first_rank(grads_f32):
    gs = [np.asarray(g, np.float32) for g in grads_f32]
    s = gs[0].copy()
    for g in gs[1:]:
        s = s + g
    return s


def update_shards_with_padding(state, ghat_shards, h, norm):
    # each owner updates its whole shard, padding included
    part = state.part
    c = Z.clip_factor(norm, h.max_norm)
    sc = Z.step_scalars(h, state.t + 1)
    out = state.copy()
    for r, off in enumerate(part.offsets):
        gr = np.asarray(ghat_shards[r][:part.shard], np.float32)
        if c is not None:
            gr = gr * c
        sl = slice(off, off + part.shard)
        p, m, v = Z.adam_update(state.master[sl], state.m[sl], state.v[sl], gr, sc)
        out.master[sl], out.m[sl], out.v[sl] = p, m, v
    out.t = state.t + 1
    return out, c


def skip_without_floor(state):
    out = state.copy()
    out.loss_scale = state.loss_scale / 2.0
    return out


def unscale_two_roundings(s, n_ranks, loss_scale):
    return ((np.asarray(s, np.float32) / np.float32(n_ranks)) / np.float32(loss_scale)).astype(np.float32)


def norm_shards_in_fp32(ghat_shards, part):
    total = np.float32(0.0)
    for r, real in enumerate(part.real):
        x = np.asarray(ghat_shards[r][:real], np.float32)
        total = np.float32(total + np.sum(x * x, dtype=np.float32))
    return math.sqrt(float(total))


def norm_shards_pairwise(ghat_shards, part):
    # numpy's own summation order (several accumulators, then pairwise)
    total = 0.0
    for r, real in enumerate(part.real):
        x = np.asarray(ghat_shards[r][:real], np.float64)
        total = total + float(np.sum(x * x))
    return math.sqrt(total)


def norm_full_in_fp32(ghat, part):
    total = np.float32(0.0)
    for off, real in zip(part.offsets, part.real):
        x = np.asarray(ghat[off:off + real], np.float32)
        total = np.float32(total + np.sum(x * x, dtype=np.float32))
    return math.sqrt(float(total))


MUTANTS = [
    ("adam_update", adam_swapped_beta),
    ("adam_update", adam_no_decay),
    ("adam_update", adam_wrong_sign),
    ("adam_update", adam_eps_inside_sqrt),
    ("step_scalars", scalars_no_bias_correction),
    ("step_scalars", scalars_t_off_by_one),
    ("rank_sum", rank_sum_drops_last),
    ("rank_sum", rank_sum_reversed),
    ("rank_sum", rank_sum_from_first_rank),
    ("_norm_from_shards", norm_shards_in_fp32),
    ("_norm_from_shards", norm_shards_pairwise),
    ("grad_norm", norm_full_in_fp32),
    ("unscale", unscale_forgets_scale),
    ("unscale", unscale_forgets_n),
    ("unscale", unscale_two_roundings),
    ("partition", partition_off_by_one),
    ("partition", partition_no_padding),
    ("rne16", rne16_truncates),
    ("model_state_bytes", msb_drops_grad_term),
    ("clip_factor", clip_wrong_comparison),
    ("_norm_from_shards", norm_wrong_shard_index),
    ("_skip", skip_keeps_scale),
    ("_skip", skip_without_floor),
    ("_update_shards", update_shards_with_padding),
    ("quantize_blocks", quant_qmax_off_by_one),
    ("quantize_blocks", quant_floor),
    ("quantize_blocks", quant_multiplies_by_inverse),
    ("dequantize_blocks", dequant_forgets_lo),
    ("pack_int4", pack4_swapped_nibbles),
    ("persistent_layout", persist_threshold_inclusive),
    ("persistent_layout", persist_small_first),
    ("comm_elems_persistent", persist_comm_no_refresh),
    ("comm_elems_ring_persistent", persist_ring_no_refresh),
    ("model_state_bytes_persistent", persist_msb_no_replicas),
    ("step_stage3_persistent", persist_step_stale_replicas),
]


def test_unmutated_oracle_passes_every_pin():
    assert _caught() == []


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_each_planted_mistake_is_caught(monkeypatch, name, mutant):
    _patch(monkeypatch, name, mutant)
    assert _caught(), f"no pin catches the mutant {mutant.__name__}"
