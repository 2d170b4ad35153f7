"""GPU parity of several query tokens per request (multi-token prediction /
target verify) on the tensor-core kernel: every row against the oracle's
causal decode (query token i of T sees the owned tokens t < L - T + i + 1),
rows that see nothing exactly (0, -inf), requests split across SMs, and the
all-partition call with its merge."""
import numpy as np
import pytest
import torch

import mla_paged_decode_gb300 as mla
import oracle
import workloads
from casebits import case_bits, subcase_bits
from gpu_helpers import FP8_ATOL, assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_decode_gb300 import build
    build.build()
    mla.load_library()


def _neutral_rows(out, lse, lens, T, P, r):
    o, l = out.detach().cpu(), lse.detach().cpu()
    for b, L in enumerate(lens):
        for i in range(T):
            if oracle.local_len(max(0, L - T + i + 1), P, r) == 0:
                assert torch.all(o[b, i].view(torch.int16) == 0), (b, i)
                assert torch.all(torch.isneginf(l[b, i])), (b, i)


CASES = [
    # heads, T, lens, num_parts, kv dtype
    (16, 2, [2, 65, 300, 1000], 1, "bf16"),
    (16, 4, [1, 3, 5, 64, 129, 2000], 8, "bf16"),      # L < T: rows that see nothing
    (64, 2, [2, 70, 4097, 31], 2, "bf16"),             # one 64-row group per query token
    (32, 3, [3, 500, 90, 7], 4, "bf16"),               # groups straddle query tokens
    (128, 2, [800, 2, 65], 1, "bf16"),
    (8, 8, [8, 9, 200, 63], 2, "bf16"),
    (16, 4, [4, 900, 70, 1], 4, "e4m3"),
    (32, 2, [3, 500, 90, 7], 3, "bf16"),               # strided gather: rows y0 + kP of a page
    (16, 3, [1, 2, 5, 300, 130], 6, "e4m3"),
    (64, 4, [4, 5, 64, 65, 66, 2000], 5, "bf16"),      # row bounds at page edges, in slots
    (16, 2, [1, 700, 1025], 7, "e4m3"),
    (16, 2, [3, 500, 90, 7], 12, "bf16"),              # owner mask: gather 4, keep 1 of 3
]


@pytest.mark.parametrize("heads,T,lens,num_parts,kv_dtype", CASES)
def test_causal_rows_match_the_oracle(heads, T, lens, num_parts, kv_dtype):
    case = workloads.make_decode_case(f"mtp_h{heads}_t{T}", heads, lens, seed=heads * T,
                                      device="cuda", kv_dtype=kv_dtype, num_parts=num_parts,
                                      tail_poison=True, q_len=T,
                                      pool_pages=sum((L + 63) // 64 for L in lens) + 3)
    q, kv, bt, sl = case_bits(case)
    B = case.batch
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table, case.kv_scale)
    atol = FP8_ATOL if kv_dtype == "e4m3" else 2e-2
    for r in range(num_parts):
        for base in (0, 1):
            out = torch.full((B, T, heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
            lse = torch.full((B, T, heads), float("nan"), dtype=torch.float32, device="cuda")
            mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, r, num_parts,
                               case.sm_scale, base, out, lse, kv_scale=case.kv_scale, workspace=ws)
            ro, rl = oracle.decode_partial_causal(q, kv, bt, sl, r, num_parts, case.sm_scale, base,
                                                  kv_dtype=kv_dtype, kv_scale=case.kv_scale)
            assert_out_close(out, ro, atol=atol, what=f"part {r} base {base}")
            assert_lse_close(lse, rl, base, what=f"part {r}")
            _neutral_rows(out, lse, lens, T, num_parts, r)
    assert mla.check_workspace(ws) == 0


def test_a_long_causal_request_split_across_ctas():
    case = workloads.make_decode_case("mtp_long", 64, [150000, 9], seed=8, device="cuda", q_len=2)
    q, kv, bt, sl = case_bits(case)
    out = torch.empty(2, 2, 64, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(2, 2, 64, dtype=torch.float32, device="cuda")
    mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, 0, 1,
                       case.sm_scale, 0, out, lse)
    ro, rl = oracle.decode_partial_causal(q, kv, bt, sl, 0, 1, case.sm_scale, 0)
    assert_out_close(out, ro, what="long causal")
    assert_lse_close(lse, rl, 0, what="long causal")


@pytest.mark.parametrize("T,num_parts", [(2, 8), (4, 4), (3, 3), (2, 7)])
def test_all_partitions_call_with_several_query_tokens(T, num_parts):
    lens = [1, 2, T + 3, 700, 5000]
    case = workloads.make_decode_case("mtp_dcp", 16, lens, seed=T, device="cuda", q_len=T,
                                      num_parts=num_parts)
    q, kv, bt, sl = case_bits(case)
    out_lse = torch.empty(len(lens), T, 16, dtype=torch.float32, device="cuda")
    out, _, parts, plses = mla.decode_dcp(case.q, case.kv_pages, case.block_table, case.seq_lens,
                                          num_parts, case.sm_scale, 1, out_lse=out_lse)
    for r in range(num_parts):
        ro, rl = oracle.decode_partial_causal(q, kv, bt, sl, r, num_parts, case.sm_scale, 1)
        assert_out_close(parts[r], ro, what=f"partition {r}")
        assert_lse_close(plses[r], rl, 1, what=f"partition {r}")
        _neutral_rows(parts[r], plses[r], lens, T, num_parts, r)
    fo, fl = oracle.decode_partial_causal(q, kv, bt, sl, 0, 1, case.sm_scale, 1)
    assert_out_close(out, fo, what="merged")
    assert_lse_close(out_lse, fl, 1, what="merged")


def test_two_query_tokens_on_the_32k_batch_every_request():
    """The 32K-context batch with two query tokens per request (two 64-row
    groups per request, the layout whose groups walk the same pages side by
    side), every request against the oracle, 8 at a time."""
    case = workloads.config_long32k(device="cuda", q_len=2)
    B = case.batch
    out = torch.full((B, 2, 64, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, 2, 64), float("nan"), dtype=torch.float32, device="cuda")
    mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, 0, 1,
                       case.sm_scale, 0, out, lse)
    for i in range(0, B, 8):
        sel = list(range(i, i + 8))
        q, kv, bt, sl = subcase_bits(case, sel)
        ro, rl = oracle.decode_partial_causal(q, kv, bt, sl, 0, 1, case.sm_scale, 0)
        assert_out_close(out[sel], ro, what=f"requests {sel[0]}..{sel[-1]}")
        assert_lse_close(lse[sel], rl, 0, what=f"requests {sel[0]}..{sel[-1]}")


def test_sixteen_query_tokens_at_128_heads():
    """The widest request: 16 query tokens x 128 heads = 2048 rows, 32 head
    groups walking the same pages side by side (and a request shorter than
    16 tokens, whose first rows see nothing)."""
    lens = [3000, 9, 700]
    case = workloads.make_decode_case("mtp16", 128, lens, seed=16, device="cuda", q_len=16,
                                      tail_poison=True,
                                      pool_pages=sum((L + 63) // 64 for L in lens) + 3)
    q, kv, bt, sl = case_bits(case)
    B = case.batch
    out = torch.full((B, 16, 128, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, 16, 128), float("nan"), dtype=torch.float32, device="cuda")
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table)
    mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, 0, 1,
                       case.sm_scale, 1, out, lse, workspace=ws)
    assert mla.check_workspace(ws) == 0
    ro, rl = oracle.decode_partial_causal(q, kv, bt, sl, 0, 1, case.sm_scale, 1)
    assert_out_close(out, ro, what="16 tokens x 128 heads")
    assert_lse_close(lse, rl, 1, what="16 tokens x 128 heads")
    _neutral_rows(out, lse, lens, 16, 1, 0)
