"""Pins of the fp64 oracle against things other than itself.

* number formats against torch's own bf16 / float8_e4m3fn conversions;
* attention against the independent pure-Python brute force (tests/brute_force.py)
  on tiny inputs, reduced and full (576/512) dims, every P in {1,2,3,4,8};
* closed forms: one token, equal scores, equal values, zero query;
* partition invariants: merging the P partials gives the unpartitioned result,
  partitions that own nothing give exactly (0, -inf), base 2 == base e * log2 e;
* combine: brute force, identity at P = 1, equal LSEs give the mean, a single
  finite LSE selects its partial, a common shift moves only the merged LSE.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from brute_force import attend_brute, bf16, combine_brute, partial_brute
from casebits import bits, case_bits

RTOL = 1e-11


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    return bits(torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16))


def tiny_case(rng, lens, heads, num_parts, dk=12, page_size=4, extra_pages=3):
    need = [(L + page_size - 1) // page_size for L in lens]
    pool = sum(need) + extra_pages
    perm = rng.permutation(pool)
    bt = np.zeros((len(lens), max(1, max(need))), dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off:off + n]
        off += n
    q = to_bf16_bits(rng.standard_normal((len(lens), 1, heads, dk)))
    kv = to_bf16_bits(rng.standard_normal((pool, page_size, dk)))
    return q, kv, bt, np.array(lens, dtype=np.int32)


# ------------------------------------------------------------------ formats

def test_bf16_decode_matches_torch_on_every_pattern():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(allbits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64)
    np.testing.assert_array_equal(oracle.bf16_to_f64(allbits), ref.numpy())


def test_e4m3_decode_matches_torch_on_every_pattern():
    allbits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(allbits.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.e4m3_to_f64(allbits), ref)


def test_e4m3_special_values():
    dec = oracle.e4m3_to_f64(np.array([0x7E, 0x08, 0x01, 0x80, 0x00, 0x38, 0xFE, 0x07],
                                      dtype=np.uint8))
    assert dec.tolist() == [448.0, 2.0 ** -6, 2.0 ** -9, -0.0, 0.0, 1.0, -448.0,
                            7 / 8 * 2.0 ** -6]
    assert np.isnan(oracle.e4m3_to_f64(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


# ------------------------------------------------------------------ brute force

@pytest.mark.parametrize("num_parts", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("base", [0, 1])
def test_partial_matches_brute_force_reduced_dims(num_parts, base):
    rng = np.random.default_rng(100 + num_parts)
    lens = [0, 1, 5, 17, 40]
    q, kv, bt, sl = tiny_case(rng, lens, heads=3, num_parts=num_parts)
    for r in range(num_parts):
        out, lse = oracle.decode_partial(q, kv, bt, sl, r, num_parts, 0.37, base,
                                         page_size=4, d_v=8)
        bo, bl = partial_brute(q.tolist(), kv.tolist(), bt.tolist(), sl.tolist(), r,
                               num_parts, 0.37, 8, 4, base2=bool(base))
        np.testing.assert_allclose(out, np.array(bo), rtol=RTOL, atol=1e-13)
        np.testing.assert_allclose(lse, np.array(bl), rtol=RTOL, atol=1e-13)


def test_partial_matches_brute_force_full_dims():
    case = workloads.make_decode_case("tiny_full", 2, [40, 23], num_parts=3, seed=7)
    q, kv, bt, sl = case_bits(case)
    for r in range(3):
        out, lse = oracle.decode_partial(q, kv, bt, sl, r, 3, case.sm_scale, 0)
        bo, bl = partial_brute(q.tolist(), kv.tolist(), bt.tolist(), sl.tolist(), r, 3,
                               case.sm_scale, 512, 64)
        np.testing.assert_allclose(out, np.array(bo), rtol=RTOL, atol=1e-13)
        np.testing.assert_allclose(lse, np.array(bl), rtol=RTOL, atol=1e-13)


def test_fp8_partial_matches_brute_force():
    case = workloads.make_decode_case("tiny_fp8", 2, [37, 64], kv_dtype="e4m3",
                                      num_parts=2, seed=3)
    q, kv, bt, sl = case_bits(case)

    def dec(x):  # torch's own e4m3 conversion, then the per-tensor scale
        t = torch.tensor([int(x)], dtype=torch.uint8).view(torch.float8_e4m3fn)
        return float(t.to(torch.float64)) * case.kv_scale

    for r in range(2):
        out, lse = oracle.decode_partial(q, kv, bt, sl, r, 2, case.sm_scale, 0,
                                         kv_dtype="e4m3", kv_scale=case.kv_scale)
        bo, bl = partial_brute(q.tolist(), kv.tolist(), bt.tolist(), sl.tolist(), r, 2,
                               case.sm_scale, 512, 64, decode=dec)
        np.testing.assert_allclose(out, np.array(bo), rtol=RTOL, atol=1e-13)
        np.testing.assert_allclose(lse, np.array(bl), rtol=RTOL, atol=1e-13)


# ------------------------------------------------------------------ closed forms

def _single_page_case(rows_f32: np.ndarray, q_f32: np.ndarray):
    """One request whose cache is exactly ``rows`` (bf16-representable)."""
    n = rows_f32.shape[0]
    kv = np.zeros((1, 64, rows_f32.shape[1]), dtype=np.float32)
    kv[0, :n] = rows_f32
    return (to_bf16_bits(q_f32[None, None, None, :]), to_bf16_bits(kv),
            np.zeros((1, 1), dtype=np.int32), np.array([n], dtype=np.int32))


def test_single_token_returns_its_value_and_score():
    rng = np.random.default_rng(1)
    row = oracle.bf16_to_f64(to_bf16_bits(rng.standard_normal(576)))
    qv = oracle.bf16_to_f64(to_bf16_bits(rng.standard_normal(576)))
    q, kv, bt, sl = _single_page_case(row[None].astype(np.float32), qv.astype(np.float32))
    out, lse = oracle.decode_full(q, kv, bt, sl, 0.25)
    np.testing.assert_array_equal(out[0, 0], row[:512])
    assert lse[0, 0] == pytest.approx(0.25 * math.fsum(qv * row), rel=1e-14)


def test_equal_scores_average_the_values():
    """q is zero on the latent dims and the rows share their rope part, so every
    score is the same: out = mean of the 512 latent dims, lse = s + ln n."""
    rng = np.random.default_rng(2)
    n = 37
    rows = rng.standard_normal((n, 576)).astype(np.float32)
    rows[:, 512:] = rows[0, 512:]
    qv = np.zeros(576, dtype=np.float32)
    qv[512:] = rng.standard_normal(64)
    q, kv, bt, sl = _single_page_case(rows, qv)
    out, lse = oracle.decode_full(q, kv, bt, sl, 0.5)
    r64 = oracle.bf16_to_f64(kv[0, :n])
    q64 = oracle.bf16_to_f64(q[0, 0, 0])
    np.testing.assert_allclose(out[0, 0], r64[:, :512].mean(axis=0), rtol=1e-12, atol=1e-14)
    s = 0.5 * math.fsum(q64 * r64[0])
    assert lse[0, 0] == pytest.approx(s + math.log(n), rel=1e-13)


def test_equal_values_return_that_value():
    rng = np.random.default_rng(3)
    n = 50
    rows = rng.standard_normal((n, 576)).astype(np.float32)
    rows[:, :512] = rows[0, :512]
    q, kv, bt, sl = _single_page_case(rows, rng.standard_normal(576).astype(np.float32))
    out, _ = oracle.decode_full(q, kv, bt, sl, 1.0)
    np.testing.assert_allclose(out[0, 0], oracle.bf16_to_f64(kv[0, 0, :512]), rtol=1e-13)


def test_zero_query_gives_uniform_weights():
    rng = np.random.default_rng(4)
    n = 29
    rows = rng.standard_normal((n, 576)).astype(np.float32)
    q, kv, bt, sl = _single_page_case(rows, np.zeros(576, dtype=np.float32))
    out, lse = oracle.decode_full(q, kv, bt, sl, 0.7)
    np.testing.assert_allclose(out[0, 0], oracle.bf16_to_f64(kv[0, :n, :512]).mean(axis=0),
                               rtol=1e-12, atol=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(n), rel=1e-14)


# ------------------------------------------------------------------ partitions

@pytest.mark.parametrize("num_parts", [2, 3, 4, 8])
def test_merging_partials_gives_unpartitioned_result(num_parts):
    case = workloads.make_decode_case("merge", 4, [0, 1, 3, 7, 130, 300], seed=11,
                                      num_parts=num_parts)
    q, kv, bt, sl = case_bits(case)
    full_o, full_l = oracle.decode_full(q, kv, bt, sl, case.sm_scale)
    parts = [oracle.decode_partial(q, kv, bt, sl, r, num_parts, case.sm_scale, 0)
             for r in range(num_parts)]
    mo, ml = oracle.lse_combine(np.stack([p[0] for p in parts]),
                                np.stack([p[1] for p in parts]), 0)
    np.testing.assert_allclose(mo, full_o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ml, full_l, rtol=1e-12, atol=0)


def test_partition_owning_nothing_is_exactly_neutral():
    case = workloads.make_decode_case("empty", 3, [1, 3, 5, 7, 0], num_parts=8, seed=5)
    q, kv, bt, sl = case_bits(case)
    for r in range(8):
        for base in (0, 1):
            out, lse = oracle.decode_partial(q, kv, bt, sl, r, 8, case.sm_scale, base)
            for b, L in enumerate(sl):
                if r >= L:
                    assert np.all(out[b] == 0.0) and np.all(np.isneginf(lse[b]))
                else:
                    assert np.all(np.isfinite(lse[b]))


def test_base2_lse_is_natural_times_log2e():
    case = workloads.make_decode_case("base", 4, [77, 1, 0], num_parts=2, seed=6)
    q, kv, bt, sl = case_bits(case)
    for r in range(2):
        o_e, l_e = oracle.decode_partial(q, kv, bt, sl, r, 2, case.sm_scale, 0)
        o_2, l_2 = oracle.decode_partial(q, kv, bt, sl, r, 2, case.sm_scale, 1)
        np.testing.assert_array_equal(o_e, o_2)
        fin = np.isfinite(l_e)
        np.testing.assert_allclose(l_2[fin], l_e[fin] / math.log(2.0), rtol=1e-15)
        assert np.array_equal(np.isneginf(l_2), ~fin)


def test_placement_of_pages_does_not_matter():
    """Moving every logical page to another physical page (and the block table
    with it) leaves the result bit-identical."""
    case = workloads.make_decode_case("perm", 4, [200, 64, 9], num_parts=2, seed=8,
                                      pool_pages=12)
    q, kv, bt, sl = case_bits(case)
    rng = np.random.default_rng(0)
    perm = rng.permutation(kv.shape[0])          # new physical slot of each page
    kv2 = np.empty_like(kv)
    kv2[perm] = kv
    bt2 = perm[bt]
    for r in range(2):
        a = oracle.decode_partial(q, kv, bt, sl, r, 2, case.sm_scale, 0)
        b = oracle.decode_partial(q, kv2, bt2, sl, r, 2, case.sm_scale, 0)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------------------------ combine

def _combine_inputs(seed, P=5, T=3, H=2, D=6, empties=((0, 1), (2, 0), (2, 3))):
    rng = np.random.default_rng(seed)
    parts = oracle.bf16_to_f64(to_bf16_bits(rng.standard_normal((P, T, H, D))))
    lses = rng.normal(5, 3, (P, T, H)).astype(np.float32).astype(np.float64)
    for t, p in empties:
        parts[p, t] = 0.0
        lses[p, t] = -np.inf
    return parts, lses


@pytest.mark.parametrize("base", [0, 1])
def test_combine_matches_brute_force(base):
    parts, lses = _combine_inputs(9)
    out, lse = oracle.lse_combine(parts, lses, base)
    P, T, H, D = parts.shape
    for t in range(T):
        for h in range(H):
            bo, bl = combine_brute(parts[:, t, h].tolist(), lses[:, t, h].tolist(),
                                   base2=bool(base))
            np.testing.assert_allclose(out[t, h], bo, rtol=RTOL, atol=1e-14)
            assert lse[t, h] == pytest.approx(bl, rel=1e-13)


def test_combine_single_partition_is_identity():
    parts, lses = _combine_inputs(10, P=1, empties=((1, 0),))
    out, lse = oracle.lse_combine(parts, lses, 0)
    np.testing.assert_allclose(out, parts[0], rtol=1e-15)
    np.testing.assert_array_equal(lse, lses[0])


def test_combine_equal_lses_take_the_mean():
    parts, _ = _combine_inputs(11, empties=())
    lses = np.full(parts.shape[:3], 2.5)
    out, lse = oracle.lse_combine(parts, lses, 0)
    np.testing.assert_allclose(out, parts.mean(axis=0), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, 2.5 + math.log(parts.shape[0]), rtol=1e-14)


def test_combine_single_finite_lse_selects_its_partial():
    parts, lses = _combine_inputs(12, empties=())
    lses[:] = -np.inf
    lses[3] = 1.25
    out, lse = oracle.lse_combine(parts, lses, 1)
    np.testing.assert_array_equal(out, parts[3])
    np.testing.assert_array_equal(lse, lses[3])


def test_combine_shift_moves_only_the_lse():
    parts, lses = _combine_inputs(13)
    o1, l1 = oracle.lse_combine(parts, lses, 0)
    o2, l2 = oracle.lse_combine(parts, lses + 7.0, 0)
    np.testing.assert_allclose(o2, o1, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(l2, l1 + 7.0, rtol=1e-14)


def test_combine_all_empty_is_neutral():
    parts, lses = _combine_inputs(14, empties=())
    parts[:, 1] = 0.0
    lses[:, 1] = -np.inf
    out, lse = oracle.lse_combine(parts, lses, 0)
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    assert np.all(np.isfinite(out))


def test_brute_force_bf16_decoder_is_exact():
    """The brute force's own bf16 decode agrees with torch on sampled patterns."""
    for b in [0, 1, 0x3F80, 0xBF80, 0x7F7F, 0x0001, 0x8000, 0x4049]:
        t = torch.from_numpy(np.array([b], dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
        assert bf16(b) == float(t.to(torch.float64))
    assert attend_brute([0.0], [], 1.0, 1) == ([0.0], float("-inf"))
