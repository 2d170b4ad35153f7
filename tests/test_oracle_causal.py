"""Pins of the oracle's multi-token (causal) decode: one query token reduces
to the single-token decode; query token i equals a single-token decode of
length L - T + i + 1; merging the partitions gives the unpartitioned result;
query tokens that see nothing are exactly neutral."""
import numpy as np
import pytest

import oracle
from test_oracle_pins import tiny_case, to_bf16_bits


def _case(rng, lens, T, heads=3, P=1):
    q, kv, bt, sl = tiny_case(rng, lens, heads=heads, num_parts=P, dk=576, page_size=64)
    qT = to_bf16_bits(rng.standard_normal((len(lens), T, heads, 576)))
    return qT, kv, bt, sl


def test_one_query_token_is_the_single_token_decode():
    rng = np.random.default_rng(0)
    q, kv, bt, sl = _case(rng, [1, 70, 300], T=1)
    for r, P in [(0, 1), (1, 3)]:
        co, cl = oracle.decode_partial_causal(q, kv, bt, sl, r, P, 0.09, 1)
        so, slse = oracle.decode_partial(q, kv, bt, sl, r, P, 0.09, 1)
        np.testing.assert_array_equal(co[:, 0], so)
        np.testing.assert_array_equal(cl[:, 0], slse)


@pytest.mark.parametrize("T,P", [(2, 1), (3, 2), (4, 8), (8, 3)])
def test_query_token_i_sees_the_first_L_minus_T_plus_i_plus_1_tokens(T, P):
    rng = np.random.default_rng(T * 10 + P)
    lens = [T, 9, 64, 130, 500]
    q, kv, bt, sl = _case(rng, lens, T=T, P=P)
    for r in range(P):
        co, cl = oracle.decode_partial_causal(q, kv, bt, sl, r, P, 0.09, 0)
        for i in range(T):
            li = (sl - T + i + 1).astype(np.int32)
            so, slse = oracle.decode_partial(np.ascontiguousarray(q[:, i:i + 1]), kv, bt, li, r, P,
                                             0.09, 0)
            np.testing.assert_allclose(co[:, i], so, rtol=0, atol=1e-14)
            np.testing.assert_array_equal(cl[:, i], slse)


def test_partitions_merge_to_the_unpartitioned_causal_result():
    rng = np.random.default_rng(5)
    T, P = 4, 4
    q, kv, bt, sl = _case(rng, [6, 100, 255], T=T, P=P)
    full_o, full_l = oracle.decode_partial_causal(q, kv, bt, sl, 0, 1, 0.05, 0)
    parts = [oracle.decode_partial_causal(q, kv, bt, sl, r, P, 0.05, 0) for r in range(P)]
    po = np.stack([p[0] for p in parts])
    pl = np.stack([p[1] for p in parts])
    mo, ml = oracle.lse_combine(po, pl, 0)
    np.testing.assert_allclose(mo, full_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, full_l, rtol=0, atol=1e-12)


def test_query_tokens_that_see_nothing_are_neutral():
    rng = np.random.default_rng(6)
    T, P = 4, 8
    q, kv, bt, sl = _case(rng, [2, 4], T=T, P=P)
    for r in range(P):
        co, cl = oracle.decode_partial_causal(q, kv, bt, sl, r, P, 0.1, 0)
        for b, L in enumerate(sl):
            for i in range(T):
                vis = max(0, int(L) - T + i + 1)
                if oracle.local_len(vis, P, r) == 0:
                    assert (co[b, i] == 0).all() and np.isneginf(cl[b, i]).all()
