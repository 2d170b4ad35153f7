"""GPU parity of mla_kv_append with the oracle's write side: bit-exact cache
bytes (bf16 copies; e4m3 codes of fp32(x) / kv_scale, nearest even,
saturated), the owner filter of each partition, skipped rows with a bad page,
and a decode over the appended cache.
"""
import numpy as np
import pytest
import torch

import mla_paged_decode_gb300 as mla
import oracle
import workloads
from casebits import bits, case_bits
from gpu_helpers import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_decode_gb300 import build
    build.build()
    mla.load_library()


def _new_rows(batch, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(batch, 576, generator=g) * scale).to(torch.bfloat16).cuda()


def _case(kv_dtype, seed, batch=9):
    # lengths 0..., tables with room for the appended token
    lens = [0, 1, 63, 64, 65, 127, 128, 300, 5][:batch]
    return workloads.make_decode_case(f"append_{kv_dtype}", 16, [L + 1 for L in lens], seed=seed,
                                      device="cuda", kv_dtype=kv_dtype,
                                      pool_pages=sum((L + 64) // 64 for L in lens) + 4)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("num_parts", [1, 2, 4])
def test_append_matches_the_oracle_bit_for_bit(kv_dtype, num_parts):
    case = _case(kv_dtype, seed=num_parts)
    B = case.batch
    pos = (case.seq_lens - 1).clone()
    pos[3] = -1                                   # skipped request
    new = _new_rows(B, seed=10 + num_parts, scale=3.0 if kv_dtype == "e4m3" else 1.0)
    if kv_dtype == "e4m3":                        # past 448 * scale: saturates
        new[2, :8] = torch.tensor([1e4, -1e4, 0.0, -0.0, 1e-6, -1e-6, 7.5, -7.5]).to(torch.bfloat16)
    kv_bits, bt = bits(case.kv_pages), case.block_table.cpu().numpy()
    expect = kv_bits
    for r in range(num_parts):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        mla.kv_append(new, case.kv_pages, case.block_table, pos, r, num_parts,
                      kv_scale=case.kv_scale, error_word=err)
        expect, bad = oracle.kv_append(expect, bt, pos.cpu().numpy(), bits(new), r, num_parts,
                                       kv_dtype, case.kv_scale)
        torch.cuda.synchronize()
        assert bad == 0 and int(err.item()) == 0
        np.testing.assert_array_equal(bits(case.kv_pages), expect, err_msg=f"after partition {r}")


def test_bad_page_rows_are_skipped_and_reported():
    case = _case("bf16", seed=5)
    bt = case.block_table.clone()
    bt[1, 0] = case.num_pages + 7                 # request 1 appends at t = 1: page 0
    pos = (case.seq_lens - 1).clone()
    pos[4] = 64 * bt.shape[1]                     # past the table
    new = _new_rows(case.batch, seed=2)
    before = bits(case.kv_pages)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.kv_append(new, case.kv_pages, bt, pos, 0, 1, error_word=err)
    expect, bad = oracle.kv_append(before, bt.cpu().numpy(), pos.cpu().numpy(), bits(new), 0, 1)
    torch.cuda.synchronize()
    assert bad == 2 and int(err.item()) == 1
    np.testing.assert_array_equal(bits(case.kv_pages), expect)
    # without an error word the same rows are skipped silently
    mla.kv_append(new, case.kv_pages, bt, pos, 0, 1)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(case.kv_pages), expect)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_decode_after_append_matches_the_oracle(kv_dtype):
    """Append token L, then decode L + 1 tokens in two partitions."""
    case = _case(kv_dtype, seed=21)
    old = case.seq_lens - 1
    new = _new_rows(case.batch, seed=4)
    mla.kv_append(new, case.kv_pages, case.block_table, old, 0, 1, kv_scale=case.kv_scale)
    q, kv, bt, lens = case_bits(case)
    atol = 6e-2 if kv_dtype == "e4m3" else 2e-2
    for r in range(2):
        out = torch.empty(case.batch, 1, 16, 512, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(case.batch, 1, 16, dtype=torch.float32, device="cuda")
        mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, r, 2,
                           case.sm_scale, 0, out, lse, kv_scale=case.kv_scale)
        ro, rl = oracle.decode_partial(q, kv, bt, lens, r, 2, case.sm_scale, 0, kv_dtype=kv_dtype,
                                       kv_scale=case.kv_scale)
        assert_out_close(out, ro[:, None], atol=atol, what=f"part {r}")
        assert_lse_close(lse, rl[:, None], 0, what=f"part {r}")


def test_full_size_append_changes_exactly_the_target_rows():
    case = workloads.config_long32k(device="cuda")
    before = case.kv_pages.clone()
    pos = case.seq_lens - 1                       # rewrite each request's last token
    new = _new_rows(case.batch, seed=8)
    mla.kv_append(new, case.kv_pages, case.block_table, pos, 0, 1)
    changed = (case.kv_pages.view(torch.int16) != before.view(torch.int16)).any(dim=2).nonzero()
    bt = case.block_table.cpu().numpy()
    target = {(int(bt[b, t // 64]), int(t % 64)) for b, t in enumerate(pos.cpu().tolist())}
    assert {(int(p), int(r)) for p, r in changed.cpu().tolist()} <= target
    for b, t in enumerate(pos.cpu().tolist()):
        assert torch.equal(case.kv_pages[bt[b, t // 64], t % 64].view(torch.int16),
                           new[b].view(torch.int16))
