"""GPU parity of mla_decode_dcp (all partitions in one call, then their merge):
every partition's (out, lse) against the oracle's partition, the merged
result against the unpartitioned oracle, the merge against mla_lse_combine of
the returned partials (bit for bit), and the full-size DCP workload: every
partition of 20 of its 64 requests (the four short ones among them).
"""
import numpy as np
import pytest
import torch

import mla_paged_decode_gb300 as mla
import oracle
import workloads
from casebits import case_bits
from gpu_helpers import (FP8_ATOL, assert_lse_close, assert_neutral, assert_out_close,
                         check_requests, run_partial)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_decode_gb300 import build
    build.build()
    mla.load_library()


CASES = [
    # heads, lens, num_parts, kv dtype
    (16, [1, 3, 5, 7, 300, 1025, 0], 8, "bf16"),
    (64, [64, 200, 1000, 4097, 1], 4, "bf16"),
    (128, [700, 65, 2, 0], 2, "bf16"),
    (32, [77, 3000, 9], 1, "bf16"),
    (16, [40, 999, 3], 3, "bf16"),            # P in {3, 5, 6, 7}: the strided gather, one launch
    (64, [1300, 5, 4097, 70], 5, "bf16"),
    (16, [333, 6, 65, 0], 6, "bf16"),
    (32, [2049, 7, 700], 7, "bf16"),
    (16, [40, 999, 3], 3, "e4m3"),            # e4m3, the strided gather too
    (64, [700, 2, 1500], 7, "e4m3"),
    (64, [1500, 33, 640, 0], 4, "e4m3"),
    (16, [1, 2, 3, 900, 2049], 8, "e4m3"),
    (128, [3000, 1, 700, 64], 8, "bf16"),     # two head groups of every partition, one launch
    (128, [1100, 2, 90], 3, "e4m3"),          # the same through the strided gather
    (96, [5000, 129], 1, "bf16"),             # one partition through mla_decode_dcp
]


@pytest.mark.parametrize("heads,lens,num_parts,kv_dtype", CASES)
@pytest.mark.parametrize("base", [0, 1])
def test_partitions_and_merge_match_the_oracle(heads, lens, num_parts, kv_dtype, base):
    case = workloads.make_decode_case(f"dcp_h{heads}_p{num_parts}", heads, lens, seed=heads + num_parts,
                                      device="cuda", kv_dtype=kv_dtype, num_parts=num_parts,
                                      tail_poison=True,
                                      pool_pages=sum((L + 63) // 64 for L in lens) + 3)
    B = case.batch
    ws = mla.make_dcp_workspace(case.q, case.kv_pages, case.block_table, num_parts, case.kv_scale)
    out_lse = torch.full((B, 1, heads), float("nan"), dtype=torch.float32, device="cuda")
    out, _, parts, plses = mla.decode_dcp(case.q, case.kv_pages, case.block_table, case.seq_lens,
                                          num_parts, case.sm_scale, base, out_lse=out_lse,
                                          kv_scale=case.kv_scale, workspace=ws)
    assert mla.check_workspace(ws) == 0
    q, kv, bt, sl = case_bits(case)
    atol = FP8_ATOL if kv_dtype == "e4m3" else 2e-2
    for r in range(num_parts):
        ro, rl = oracle.decode_partial(q, kv, bt, sl, r, num_parts, case.sm_scale, base,
                                       kv_dtype=kv_dtype, kv_scale=case.kv_scale)
        assert_out_close(parts[r], ro[:, None], atol=atol, what=f"partition {r}")
        assert_lse_close(plses[r], rl[:, None], base, what=f"partition {r}")
        assert_neutral(parts[r], plses[r], [b for b in range(B) if oracle.local_len(int(sl[b]), num_parts, r) == 0])
    fo, fl = oracle.decode_full(q, kv, bt, sl, case.sm_scale, base, kv_dtype=kv_dtype,
                                kv_scale=case.kv_scale)
    nz = [b for b in range(B) if sl[b] > 0]
    assert_out_close(out[nz], fo[nz][:, None], atol=atol, what="merged")
    assert_lse_close(out_lse[nz], fl[nz][:, None], base, what="merged")
    assert_neutral(out, out_lse, [b for b in range(B) if sl[b] == 0])
    # the merge is mla_lse_combine of the returned partials, bit for bit
    again = torch.empty_like(out)
    again_lse = torch.empty_like(out_lse)
    mla.lse_combine(parts.view(num_parts, B, heads, 512), plses.view(num_parts, B, heads), num_parts,
                    again.view(B, heads, 512), lse_base=base, out_lse=again_lse.view(B, heads))
    assert torch.equal(again.view(torch.int16), out.view(torch.int16))
    assert torch.equal(again_lse, out_lse)


def test_full_size_dcp8_in_one_call():
    case = workloads.config_dcp8(device="cuda")
    B, H = case.batch, case.heads
    ws = mla.make_dcp_workspace(case.q, case.kv_pages, case.block_table, 8)
    out, _, parts, plses = mla.decode_dcp(case.q, case.kv_pages, case.block_table, case.seq_lens,
                                          8, case.sm_scale, 1, workspace=ws)
    assert mla.check_workspace(ws) == 0
    long_ = list(range(0, 60, 4)) + [59]   # 16 of the 60 long requests
    short = [60, 61, 62, 63]               # L = 1, 3, 5, 7
    lens = case.seq_lens.cpu().tolist()
    for r in range(8):
        check_requests(oracle, case, parts[r], plses[r], r, 1, long_ + short, chunk=4,
                       what=f"dcp8 partition {r}")
        assert_neutral(parts[r], plses[r], [b for b in short if r >= lens[b]])
    out_lse = torch.empty(B, 1, H, dtype=torch.float32, device="cuda")
    out2, _, _, _ = mla.decode_dcp(case.q, case.kv_pages, case.block_table, case.seq_lens, 8,
                                   case.sm_scale, 1, workspace=ws, out_lse=out_lse)
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    check_requests(oracle, case, out, out_lse, 0, 1, long_ + short, num_parts=1, chunk=4,
                   what="dcp8 merged vs unpartitioned")
    # partition 3 computed alone agrees with its slice of the fused launch
    alone, alone_lse = run_partial(case, 3, 1)
    assert_out_close(parts[3], alone.float().cpu().numpy().astype(np.float64), what="fused vs alone")
    # fp32 sums split at other boundaries: base-2 lse ~16 agrees to a few 1e-4
    assert torch.allclose(plses[3], alone_lse, atol=2e-3, rtol=0)


def test_one_partition_call_equals_the_partial_bit_for_bit():
    """mla_decode_dcp with one partition runs mla_decode_partial's kernels
    and a combine of one partial, which returns it unchanged: its partition
    output and its merged output both equal mla_decode_partial's bits."""
    case = workloads.make_decode_case("dcp_one", 64, [5000, 33, 1, 0, 2049], seed=41,
                                      device="cuda", pool_pages=120)
    B = case.batch
    out_lse = torch.empty(B, 1, 64, dtype=torch.float32, device="cuda")
    out, _, parts, plses = mla.decode_dcp(case.q, case.kv_pages, case.block_table, case.seq_lens,
                                          1, case.sm_scale, 1, out_lse=out_lse)
    ref_out, ref_lse = run_partial(case, 0, 1)
    for o, l in ((parts[0], plses[0]), (out, out_lse)):
        assert torch.equal(o.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(l, ref_lse)
