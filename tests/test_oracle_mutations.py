"""Planted mistakes: each plausible bug in the oracle must trip at least one pin.

Every mutant below is planted in the oracle module on the CPU (monkeypatch) and
the compact pin set ``pin_failures`` is run against it; an unmutated oracle
passes every pin, each mutant fails at least one.
"""
import math

import numpy as np
import pytest

import oracle
import oracle.mla_oracle as om
import test_oracle_pins as pins
from brute_force import partial_brute

_orig_attend = om.attend


def _pin_brute(base):
    rng = np.random.default_rng(5)
    q, kv, bt, sl = pins.tiny_case(rng, [0, 3, 9, 21], heads=2, num_parts=3, dk=10,
                                   page_size=4)
    for r in range(3):
        out, lse = oracle.decode_partial(q, kv, bt, sl, r, 3, 0.41, base, page_size=4,
                                         d_v=6)
        bo, bl = partial_brute(q.tolist(), kv.tolist(), bt.tolist(), sl.tolist(), r, 3,
                               0.41, 6, 4, base2=bool(base))
        np.testing.assert_allclose(out, np.array(bo), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse, np.array(bl), rtol=1e-10, atol=1e-12)


def _pin_full_dims():
    pins.test_partial_matches_brute_force_full_dims()


def _pin_closed_forms():
    pins.test_single_token_returns_its_value_and_score()
    pins.test_equal_scores_average_the_values()
    pins.test_equal_values_return_that_value()
    pins.test_zero_query_gives_uniform_weights()


def _pin_partitions():
    pins.test_merging_partials_gives_unpartitioned_result(3)
    pins.test_partition_owning_nothing_is_exactly_neutral()
    pins.test_base2_lse_is_natural_times_log2e()


def _pin_combine():
    for base in (0, 1):
        pins.test_combine_matches_brute_force(base)
    pins.test_combine_single_finite_lse_selects_its_partial()
    pins.test_combine_all_empty_is_neutral()


def _pin_formats():
    pins.test_e4m3_decode_matches_torch_on_every_pattern()
    pins.test_fp8_partial_matches_brute_force()


def _pin_append():
    import test_oracle_append as ap
    ap.test_e4m3_encode_round_trips_every_finite_code()
    ap.test_e4m3_encode_ties_go_to_the_even_code()
    ap.test_e4m3_encode_saturates_at_448()
    ap.test_e4m3_encode_matches_torch_float8_in_range()
    ap.test_append_writes_the_row_bits_and_nothing_else()
    for n in (2, 3, 8):
        ap.test_partition_appends_together_equal_one_unpartitioned_append(n)
    ap.test_e4m3_append_stores_torchs_cast_of_x_over_scale()
    ap.test_rows_with_a_bad_page_are_counted_and_not_written()
    ap.test_decode_after_append_attends_to_the_new_row()


def _pin_meta():
    import test_oracle_dcp_meta as dm
    for n in (1, 2, 3, 8):
        dm.test_local_lengths_count_the_owned_tokens(n)
    dm.test_table_recovers_the_page_assignment()
    dm.test_bad_requests_are_counted_and_padded()
    for r, P in [(0, 1), (1, 2), (2, 4), (5, 8)]:
        dm.test_decode_over_the_compact_pool_is_the_partition(r, P)


def _pin_causal():
    import test_oracle_causal as tc
    tc.test_one_query_token_is_the_single_token_decode()
    for T, P in [(2, 1), (3, 2), (4, 8), (8, 3)]:
        tc.test_query_token_i_sees_the_first_L_minus_T_plus_i_plus_1_tokens(T, P)
    tc.test_partitions_merge_to_the_unpartitioned_causal_result()
    tc.test_query_tokens_that_see_nothing_are_neutral()


PINS = [lambda: _pin_brute(0), lambda: _pin_brute(1), _pin_full_dims, _pin_closed_forms,
        _pin_partitions, _pin_combine, _pin_formats, _pin_append, _pin_meta, _pin_causal]


def pin_failures() -> int:
    bad = 0
    for pin in PINS:
        try:
            pin()
        except Exception:  # an assertion, or a mutant that no longer runs
            bad += 1
    return bad


# ---------------------------------------------------------------- the mutants

def _blocked_owner(seq_len, num_parts, part_id):
    per = -(-seq_len // num_parts)
    return np.arange(part_id * per, min(seq_len, (part_id + 1) * per), dtype=np.int64)


def _off_by_one_owner(seq_len, num_parts, part_id):
    return np.arange(part_id + 1, seq_len, num_parts, dtype=np.int64)


def _swapped_page_row(kv_bits, bt_row, tokens, page_size):
    pages = np.asarray(bt_row)[tokens % page_size % len(bt_row)].astype(np.int64)
    return kv_bits[pages, tokens // page_size % page_size]


def _identity_placement(kv_bits, bt_row, tokens, page_size):
    return kv_bits[(tokens // page_size).astype(np.int64), tokens % page_size]


def _drop_rope(q, k, sm_scale, d_v=om.D_V):
    keep = d_v if q.shape[1] > d_v else q.shape[1] - 2
    return _orig_attend(q[:, :keep], k[:, :keep], sm_scale, d_v)


def _value_from_tail(q, k, sm_scale, d_v=om.D_V):
    out, lse = _orig_attend(q, k, sm_scale, d_v)
    if k.shape[0] == 0:
        return out, lse
    s = sm_scale * (q @ k.T)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    return (w @ k[:, -d_v:]) / w.sum(axis=1, keepdims=True), lse


def _lse_without_scale(q, k, sm_scale, d_v=om.D_V):
    out, lse = _orig_attend(q, k, sm_scale, d_v)
    if k.shape[0] == 0:
        return out, lse
    s = q @ k.T
    mu = s.max(axis=1)
    return out, mu + np.log(np.exp(s - mu[:, None]).sum(axis=1))


def _normalised_over_heads(q, k, sm_scale, d_v=om.D_V):
    if k.shape[0] == 0:
        return _orig_attend(q, k, sm_scale, d_v)
    s = sm_scale * (q @ k.T)
    w = np.exp(s - s.max())
    out = (w @ k[:, :d_v]) / w.sum(axis=0).sum()
    return out, s.max() + np.log(w.sum(axis=1))


def _zero_lse_when_empty(q, k, sm_scale, d_v=om.D_V):
    out, lse = _orig_attend(q, k, sm_scale, d_v)
    return out, (np.zeros_like(lse) if k.shape[0] == 0 else lse)


def _base2_divides(lse_natural, lse_base):
    return lse_natural if lse_base == 0 else lse_natural / om.LOG2E


def _combine_wrong_sign(partials, lses, lse_base=0):
    lam = om.lse_to_natural(lses, lse_base)
    big = lam.max(axis=0)
    w = np.where(np.isfinite(lam), np.exp(big[None] - lam), 0.0)
    z = w.sum(axis=0)
    return (w[..., None] * partials).sum(axis=0) / z[..., None], om.lse_to_base(
        big + np.log(z), lse_base)


def _combine_unnormalised(partials, lses, lse_base=0):
    lam = om.lse_to_natural(lses, lse_base)
    big = lam.max(axis=0)
    safe = np.where(np.isfinite(big), big, 0.0)
    w = np.where(np.isfinite(lam), np.exp(lam - safe[None]), 0.0)
    z = w.sum(axis=0)
    lse = np.where(np.isfinite(big), safe + np.log(np.where(z > 0, z, 1)), -np.inf)
    return (w[..., None] * partials).sum(axis=0), om.lse_to_base(lse, lse_base)


def _e4m3_bias8(bits):
    return om.e4m3_to_f64(bits) / 2.0


def _e4m3_encode_variant(x, tie_up=False, truncate=False, saturate=True):
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    vals, codes = om._e4m3_finite_table()
    a = np.abs(x)
    hi = np.minimum(np.searchsorted(vals, a, side="left"), len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - vals[lo], vals[hi] - a
    if truncate:
        pick_hi = np.zeros_like(a, dtype=bool)
    elif tie_up:
        pick_hi = dhi <= dlo
    else:
        pick_hi = (dhi < dlo) | ((dhi == dlo) & ((codes[hi] & 1) == 0))
    c = np.where(pick_hi, codes[hi], codes[lo])
    c = np.where(vals[hi] == a, codes[hi], c)
    c = np.where(a >= vals[-1], codes[-1] if saturate else 0x7F, c)
    c = np.where((a == vals[-1]), codes[-1], c)
    return (c | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


_orig_append = om.kv_append


def _append_ignores_owner(kv, bt, pos, new, part_id, num_parts, *a, **k):
    return _orig_append(kv, bt, pos, new, 0, 1, *a, **k)


def _append_row_off_by_one(kv, bt, pos, new, part_id, num_parts, *a, **k):
    pos = np.where(np.asarray(pos) >= 0, np.asarray(pos) + 1, pos)
    return _orig_append(kv, bt, pos, new, part_id, num_parts, *a, **k)


def _append_scale_multiplies(kv, bt, pos, new, part_id, num_parts, kv_dtype="bf16",
                             kv_scale=1.0, **k):
    return _orig_append(kv, bt, pos, new, part_id, num_parts, kv_dtype, 1.0 / kv_scale, **k)


_orig_meta = om.dcp_local_metadata


def _meta_ignores_extra(seq_lens, idx, r2t, part_id, num_parts, extra_tokens=0, **k):
    return _orig_meta(seq_lens, idx, r2t, part_id, num_parts, 0, **k)


def _meta_page_of_token_i(seq_lens, idx, r2t, part_id, num_parts, extra_tokens=0, max_pages=1,
                          pad_value=0, page_size=64):
    g, loc, table, bad = _orig_meta(seq_lens, idx, r2t, part_id, num_parts, extra_tokens,
                                    max_pages, pad_value, page_size)
    r2t = np.asarray(r2t)
    for b in range(len(loc)):
        for i in range(-(-int(loc[b]) // page_size)):
            if table[b, i] != pad_value and i < r2t.shape[1] and r2t[int(idx[b]), i] >= 0:
                table[b, i] = r2t[int(idx[b]), i] // page_size
    return g, loc, table, bad


def _local_len_off_by_one(seq_len, num_parts, part_id):
    return seq_len // num_parts + (1 if part_id <= seq_len % num_parts else 0)


def _causal_variant(shift=0, no_bound=False, reverse=False):
    def f(q_bits, kv_bits, block_table, seq_lens, part_id, num_parts, sm_scale,
          lse_base=om.LSE_NATURAL, kv_dtype="bf16", kv_scale=1.0, page_size=64, requests=None,
          d_v=om.D_V):
        q_bits = np.asarray(q_bits)
        T = q_bits.shape[1]
        rows = range(len(seq_lens)) if requests is None else list(requests)
        outs, lses = [], []
        for b in rows:
            ob, lb = [], []
            for i in range(T):
                ii = T - 1 - i if reverse else i
                vis = int(seq_lens[b]) if no_bound else max(0, int(seq_lens[b]) - T + ii + 1 + shift)
                toks = om.owned_tokens(vis, num_parts, part_id)
                k = om.dequant_rows(om.gather_rows(kv_bits, block_table[b], toks, page_size),
                                    kv_dtype, kv_scale)
                o, l = om.attend(om.bf16_to_f64(q_bits[b, i]), k, sm_scale, d_v)
                ob.append(o)
                lb.append(om.lse_to_base(l, lse_base))
            outs.append(np.stack(ob))
            lses.append(np.stack(lb))
        return np.stack(outs), np.stack(lses)
    return f


MUTANTS = {
    "causal bound dropped": ("decode_partial_causal", _causal_variant(no_bound=True)),
    "causal bound one token late": ("decode_partial_causal", _causal_variant(shift=1)),
    "query tokens in reverse order": ("decode_partial_causal", _causal_variant(reverse=True)),
    "metadata ignores the draft tokens": ("dcp_local_metadata", _meta_ignores_extra),
    "metadata page of token i, not 64 i": ("dcp_local_metadata", _meta_page_of_token_i),
    "local length off by one": ("local_len", _local_len_off_by_one),
    "e4m3 encode truncates": ("f32_to_e4m3", lambda x: _e4m3_encode_variant(x, truncate=True)),
    "e4m3 ties away from zero": ("f32_to_e4m3", lambda x: _e4m3_encode_variant(x, tie_up=True)),
    "e4m3 no saturation": ("f32_to_e4m3", lambda x: _e4m3_encode_variant(x, saturate=False)),
    "append ignores the owner rule": ("kv_append", _append_ignores_owner),
    "append one row off": ("kv_append", _append_row_off_by_one),
    "append multiplies by the scale": ("kv_append", _append_scale_multiplies),
    "blocked owner rule": ("owned_tokens", _blocked_owner),
    "owner off by one": ("owned_tokens", _off_by_one_owner),
    "page / row swapped": ("gather_rows", _swapped_page_row),
    "block table ignored": ("gather_rows", _identity_placement),
    "rope dims dropped from the score": ("attend", _drop_rope),
    "value taken from the tail dims": ("attend", _value_from_tail),
    "lse without sm_scale": ("attend", _lse_without_scale),
    "softmax normalised over heads": ("attend", _normalised_over_heads),
    "empty partition lse = 0": ("attend", _zero_lse_when_empty),
    "base-2 conversion inverted": ("lse_to_base", _base2_divides),
    "combine weight sign flipped": ("lse_combine", _combine_wrong_sign),
    "combine not normalised": ("lse_combine", _combine_unnormalised),
    "e4m3 exponent bias 8": ("e4m3_to_f64", _e4m3_bias8),
}


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(om, name, fn)
    monkeypatch.setattr(oracle, name, fn)


def test_unmutated_oracle_passes_every_pin():
    assert pin_failures() == 0


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(monkeypatch, mutant):
    name, fn = MUTANTS[mutant]
    _patch(monkeypatch, name, fn)
    assert pin_failures() >= 1, f"no pin caught: {mutant}"
