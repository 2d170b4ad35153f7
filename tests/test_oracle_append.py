"""Pins of the oracle's write side: the e4m3 encoder (OCP FP8: nearest value,
ties to even, saturation at 448) and the KV append (placement, owner filter,
untouched rows), each checked against something other than its own formula:
every code's round trip, the midpoints, torch's float8 cast, the union of the
partitions, and attention over the appended cache.
"""
import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import tiny_case


def _finite_codes():
    c = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_to_f64(c)
    keep = ~np.isnan(v)
    return c[keep], v[keep]


def test_e4m3_encode_round_trips_every_finite_code():
    codes, vals = _finite_codes()
    assert len(codes) == 254
    np.testing.assert_array_equal(oracle.f32_to_e4m3(vals.astype(np.float32)), codes)


def test_e4m3_encode_ties_go_to_the_even_code():
    for sign in (1.0, -1.0):
        vals = np.sort(oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8)))  # 0 .. 448
        lo, hi = vals[:-1], vals[1:]
        mid = (lo + hi) / 2  # exact in fp32: at most 5 significant bits
        got = oracle.f32_to_e4m3((sign * mid).astype(np.float32))
        low_code = oracle.f32_to_e4m3((sign * lo).astype(np.float32))
        high_code = oracle.f32_to_e4m3((sign * hi).astype(np.float32))
        even = np.where((low_code & 1) == 0, low_code, high_code)
        np.testing.assert_array_equal(got, even)
        # one fp32 step either side of the midpoint goes to the nearer value
        below = np.nextafter(mid.astype(np.float32), np.float32(0))
        above = np.nextafter(mid.astype(np.float32), np.float32(np.inf))
        np.testing.assert_array_equal(oracle.f32_to_e4m3(sign * below), low_code)
        np.testing.assert_array_equal(oracle.f32_to_e4m3(sign * above), high_code)


def test_e4m3_encode_saturates_at_448():
    x = np.array([448, 460, 464, 500, 1e30, np.inf], dtype=np.float32)
    np.testing.assert_array_equal(oracle.f32_to_e4m3(x), np.full(6, 0x7E, np.uint8))
    np.testing.assert_array_equal(oracle.f32_to_e4m3(-x), np.full(6, 0xFE, np.uint8))
    assert oracle.f32_to_e4m3(np.float32(-0.0)) == 0x80
    assert oracle.f32_to_e4m3(np.float32(2.0 ** -10)) == 0x00   # half the smallest: to even
    assert oracle.f32_to_e4m3(np.float32(1.5 * 2.0 ** -10)) == 0x01


def test_e4m3_encode_matches_torch_float8_in_range():
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(50000, generator=g) * 100, torch.randn(50000, generator=g) * 0.01,
                   (torch.rand(20000, generator=g) - 0.5) * 2 * 2.0 ** -6]).clamp(-448, 448)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.f32_to_e4m3(x.numpy()), ref)


def _append_case(rng, num_pages=12, batch=5, dk=576):
    kv = rng.integers(0, 1 << 16, size=(num_pages, 64, dk)).astype(np.uint16)
    bt = np.stack([rng.permutation(num_pages)[:4] for _ in range(batch)]).astype(np.int32)
    new = (rng.standard_normal((batch, dk)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return kv, bt, new


def test_append_writes_the_row_bits_and_nothing_else():
    rng = np.random.default_rng(0)
    kv, bt, new = _append_case(rng)
    pos = np.array([0, 63, 64, 200, -1], dtype=np.int32)
    out, bad = oracle.kv_append(kv, bt, pos, new, 0, 1)
    assert bad == 0
    expect = kv.copy()
    for b, t in enumerate(pos):
        if t >= 0:
            expect[bt[b, t // 64], t % 64] = new[b]
    np.testing.assert_array_equal(out, expect)
    assert not np.shares_memory(out, kv)


@pytest.mark.parametrize("num_parts", [2, 3, 8])
def test_partition_appends_together_equal_one_unpartitioned_append(num_parts):
    rng = np.random.default_rng(num_parts)
    kv, bt, new = _append_case(rng, batch=6)
    pos = rng.integers(0, 256, size=6).astype(np.int32)
    whole, _ = oracle.kv_append(kv, bt, pos, new, 0, 1)
    step = kv
    written = 0
    for r in range(num_parts):
        nxt, _ = oracle.kv_append(step, bt, pos, new, r, num_parts)
        written += int((nxt != step).any(axis=2).sum())
        step = nxt
    np.testing.assert_array_equal(step, whole)
    # and each partition wrote only the rows it owns
    for r in range(num_parts):
        part, _ = oracle.kv_append(kv, bt, pos, new, r, num_parts)
        changed = {(int(p), int(i)) for p, i in zip(*np.nonzero((part != kv).any(axis=2)))}
        owned = {(int(bt[b, t // 64]), int(t % 64)) for b, t in enumerate(pos) if t % num_parts == r}
        assert changed <= owned


def test_e4m3_append_stores_torchs_cast_of_x_over_scale():
    rng = np.random.default_rng(7)
    _, bt, new = _append_case(rng)
    kv = np.zeros((12, 64, 576), dtype=np.uint8)
    scale = np.float32(4.0 / 448)
    pos = np.array([5, 70, 129, 191, 250], dtype=np.int32)
    out, _ = oracle.kv_append(kv, bt, pos, new, 0, 1, kv_dtype="e4m3", kv_scale=float(scale))
    x = torch.from_numpy((new.astype(np.uint32) << 16).view(np.float32))
    ref = (x / torch.tensor(scale)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for b, t in enumerate(pos):
        np.testing.assert_array_equal(out[bt[b, t // 64], t % 64], ref[b])


def test_rows_with_a_bad_page_are_counted_and_not_written():
    rng = np.random.default_rng(9)
    kv, bt, new = _append_case(rng)
    bt[1, 1] = 99          # past the pool
    pos = np.array([3, 100, 64 * 4 + 1, -5, 10], dtype=np.int32)  # request 2: past the table
    out, bad = oracle.kv_append(kv, bt, pos, new, 0, 1)
    assert bad == 2
    assert (out[bt[0, 0], 3] == new[0]).all() and (out[bt[4, 0], 10] == new[4]).all()
    assert int((out != kv).any(axis=2).sum()) == 2


def test_decode_after_append_attends_to_the_new_row():
    """Appending token L then decoding L + 1 tokens equals attention over the
    L old rows and the new row put side by side directly."""
    rng = np.random.default_rng(11)
    # tables sized for one more token (64 -> 65 opens a second page)
    q, kv, bt, sl1 = tiny_case(rng, [38, 65, 6], heads=3, num_parts=1, dk=576, page_size=64)
    sl = sl1 - 1
    new = (rng.standard_normal((3, 576)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kv2, _ = oracle.kv_append(kv, bt, sl.astype(np.int32), new, 0, 1)
    out, lse = oracle.decode_full(q, kv2, bt, sl + 1, 0.07)
    for b, L in enumerate(sl):
        old = oracle.dequant_rows(oracle.gather_rows(kv, bt[b], np.arange(L), 64), "bf16", 1.0)
        k = np.concatenate([old, oracle.bf16_to_f64(new[b])[None]], axis=0)
        ro, rl = oracle.attend(oracle.bf16_to_f64(q[b, 0]), k, 0.07)
        np.testing.assert_allclose(out[b], ro, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[b], rl, rtol=1e-12, atol=1e-12)
