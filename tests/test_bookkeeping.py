"""Round-robin partition bookkeeping, pinned exactly.

The two properties are the ones the decode-layout test of sglang pull 33926
(test snippet ``TestDcpDecodeLayout``) asserts for P in {1,2,3,4,8} and
L in 0..40: the per-rank lengths sum to the global length, and one decode step
grows exactly one rank, namely rank (L-1) mod P.
"""
import os

import numpy as np
import pytest

import oracle

SIZES = [1, 2, 3, 4, 8]
LENS = list(range(0, 41))
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dcp_local_lens.txt")


def test_ranks_partition_the_global_length():
    for p in SIZES:
        for L in LENS:
            assert sum(oracle.local_len(L, p, r) for r in range(p)) == L


def test_newest_token_is_owned_by_exactly_one_rank():
    for p in SIZES:
        for L in LENS[1:]:
            grew = [oracle.local_len(L, p, r) - oracle.local_len(L - 1, p, r)
                    for r in range(p)]
            assert sum(grew) == 1
            assert grew[(L - 1) % p] == 1


@pytest.mark.parametrize("p", SIZES + [5, 6, 7, 16])
def test_owned_tokens_match_literal_enumeration(p):
    for L in list(range(0, 70)) + [131071, 131072]:
        for r in range(p):
            lit = [t for t in range(L) if t % p == r] if L < 1000 else None
            got = oracle.owned_tokens(L, p, r)
            assert len(got) == oracle.local_len(L, p, r)
            if lit is not None:
                assert got.tolist() == lit
            else:
                assert np.all(got % p == r) and np.all(np.diff(got) == p)


def test_owned_tokens_cover_every_token_once():
    for p in SIZES:
        for L in LENS:
            toks = np.concatenate([oracle.owned_tokens(L, p, r) for r in range(p)])
            assert sorted(toks.tolist()) == list(range(L))


def test_golden_local_lengths():
    """The stored table (written by golden/make_golden.py from the oracle) must
    still satisfy the page's two properties, and the oracle must reproduce it."""
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    seen = 0
    for p_s, L_s, *lens in rows:
        p, L = int(p_s), int(L_s)
        lens = [int(x) for x in lens]
        assert len(lens) == p and sum(lens) == L
        assert lens == [oracle.local_len(L, p, r) for r in range(p)]
        seen += 1
    assert seen == len(SIZES) * len(LENS)
