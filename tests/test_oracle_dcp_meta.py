"""Pins of the oracle's DCP rank metadata: local lengths by literal
enumeration, the page table recovering a known page assignment, every bad
case counted, and a decode over the rank's compact pool equal to the
partition of the global cache."""
import numpy as np
import pytest

import oracle
from dcp_local import compact_pool
from test_oracle_pins import tiny_case


@pytest.mark.parametrize("num_parts", [1, 2, 3, 8])
def test_local_lengths_count_the_owned_tokens(num_parts):
    lens = np.array([0, 1, 2, 7, 8, 9, 63, 64, 65, 200, 131072], dtype=np.int32)
    for extra in (0, 3):
        tot = np.zeros(len(lens), dtype=np.int64)
        for r in range(num_parts):
            g, loc, _, bad = oracle.dcp_local_metadata(lens, np.zeros(len(lens), np.int32),
                                                       np.zeros((1, 1 << 18), np.int32), r,
                                                       num_parts, extra, max_pages=4096)
            assert bad == 0
            np.testing.assert_array_equal(g, lens + extra)
            want = [sum(1 for t in range(L + extra) if t % num_parts == r) if L < 300 else
                    len(range(r, L + extra, num_parts)) for L in lens]
            np.testing.assert_array_equal(loc, want)
            tot += loc
        np.testing.assert_array_equal(tot, lens + extra)


def test_table_recovers_the_page_assignment():
    rng = np.random.default_rng(1)
    q, kv, bt, sl = tiny_case(rng, [5, 64, 65, 300, 0], heads=2, num_parts=1, dk=576, page_size=64)
    for r, P in [(0, 1), (1, 2), (3, 4)]:
        pool, r2t, pages, local = compact_pool(kv, bt, sl, r, P, rng)
        order = rng.permutation(len(sl)).astype(np.int32)      # request -> row of req_to_token
        r2t_perm = np.zeros_like(r2t)
        r2t_perm[order] = r2t
        g, loc, table, bad = oracle.dcp_local_metadata(sl, order, r2t_perm, r, P, max_pages=8,
                                                       pad_value=-1)
        assert bad == 0
        np.testing.assert_array_equal(loc, local)
        for b in range(len(sl)):
            np.testing.assert_array_equal(table[b, :len(pages[b])], pages[b])
            assert (table[b, len(pages[b]):] == -1).all()


def test_bad_requests_are_counted_and_padded():
    r2t = np.arange(2 * 256, dtype=np.int32).reshape(2, 256)
    r2t[1, 64] = -1                                        # a negative slot
    r2t[0, 128] += 3                                       # a slot inside a page
    lens = np.array([-5, 100, 100, 1000, 200, 150, 128], dtype=np.int32)
    idx = np.array([0, 5, 1, 0, 0, 0, 0], dtype=np.int32)  # request 1: no such pool row
    g, loc, table, bad = oracle.dcp_local_metadata(lens, idx, r2t, 0, 1, max_pages=3, pad_value=9)
    # -5: negative; idx 5: outside; request 2: slot -1 on its second page;
    # 1000 tokens: 16 pages > 3; 200 tokens: 4 pages > 3; 150 tokens: its
    # third page starts at a slot that is not a page's first (128 tokens
    # stop short of it and are fine)
    assert bad == 6
    assert loc[0] == 0 and (table[[0, 1, 3, 4]] == 9).all()
    assert table[2, 0] == r2t[1, 0] // 64 and table[2, 1] == 9 and table[2, 2] == 9
    assert list(table[5]) == [0, 1, 9] and list(table[6]) == [0, 1, 9]


@pytest.mark.parametrize("r,P", [(0, 1), (1, 2), (2, 4), (5, 8)])
def test_decode_over_the_compact_pool_is_the_partition(r, P):
    rng = np.random.default_rng(10 + r)
    q, kv, bt, sl = tiny_case(rng, [1, 40, 64, 129, 500, 0], heads=3, num_parts=P, dk=576,
                              page_size=64)
    pool, r2t, _, _ = compact_pool(kv, bt, sl, r, P, rng)
    _, loc, table, bad = oracle.dcp_local_metadata(sl, np.arange(len(sl), dtype=np.int32), r2t, r, P,
                                                   max_pages=16)
    assert bad == 0
    lo, ll = oracle.decode_partial(q, pool, table, loc, 0, 1, 0.07, 1)
    go, gl = oracle.decode_partial(q, kv, bt, sl, r, P, 0.07, 1)
    np.testing.assert_allclose(lo, go, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(np.isneginf(ll), np.isneginf(gl))
    np.testing.assert_allclose(ll[np.isfinite(ll)], gl[np.isfinite(gl)], rtol=0, atol=1e-12)
