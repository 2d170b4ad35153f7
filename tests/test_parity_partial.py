"""GPU parity of mla_decode_partial against the fp64 oracle.

Small cases are compared element by element on every request and partition;
the full-size workloads (the configuration the bench times, in the same launch
configuration) on every request of the 32K-context and e4m3 batches and on
every partition of 20 of the 64 requests of the eight-partition batch (the
four short ones among them), which the oracle computes a few requests at a
time, plus the properties that hold at any size (finite outputs, exact
neutral pairs).
"""
import numpy as np
import pytest
import torch

import mla_paged_decode_gb300 as mla
import oracle
import workloads
from casebits import case_bits
from gpu_helpers import (FP8_ATOL, assert_lse_close, assert_neutral, assert_out_close,
                         check_requests, oracle_partial_sub, run_partial)

# the long requests of the eight-partition batch checked at full size, then
# its four short ones (L = 1, 3, 5, 7)
DCP8_LONG = list(range(0, 60, 4)) + [59]
DCP8_SHORT = [60, 61, 62, 63]

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_decode_gb300 import build
    build.build()
    mla.load_library()


def _check_all(case, bases=(0, 1), atol=None):
    q, kv, bt, lens = case_bits(case)
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table, case.kv_scale)
    for r in range(case.num_parts):
        for base in bases:
            out, lse = run_partial(case, r, base, workspace=ws)
            ro, rl = oracle.decode_partial(q, kv, bt, lens, r, case.num_parts, case.sm_scale,
                                           base, kv_dtype=case.kv_dtype, kv_scale=case.kv_scale)
            what = f"{case.name} part {r} base {base}"
            assert_out_close(out, ro[:, None], **({"atol": atol} if atol else {}), what=what)
            assert_lse_close(lse, rl[:, None], base, what=what)
            empties = [b for b in range(case.batch) if oracle.local_len(int(lens[b]), case.num_parts, r) == 0]
            assert_neutral(out, lse, empties)
    assert mla.check_workspace(ws) == 0


def test_small_config_partials_then_combine():
    case = workloads.config_small(device="cuda")
    _check_all(case)
    q, kv, bt, lens = case_bits(case)
    for base in (0, 1):
        parts = [run_partial(case, r, base) for r in range(2)]
        P = torch.stack([o.view(1, 16, 512) for o, _ in parts])     # [P, T=1, H, D]
        L = torch.stack([l.view(1, 16) for _, l in parts])
        merged = torch.empty(1, 16, 512, dtype=torch.bfloat16, device="cuda")
        merged_lse = torch.empty(1, 16, dtype=torch.float32, device="cuda")
        mla.lse_combine(P, L, 2, merged, lse_base=base, out_lse=merged_lse)
        fo, fl = oracle.decode_full(q, kv, bt, lens, case.sm_scale, base)
        assert_out_close(merged, fo, what=f"merged base {base}")
        assert_lse_close(merged_lse, fl, base, what=f"merged base {base}")


SHAPES = [
    # heads, lens, num_parts, kv dtype
    (16, [0, 1, 63, 64, 65, 129, 300], 1, "bf16"),
    (64, [5, 64, 200, 1000, 0, 4097], 1, "bf16"),
    (1, [77, 3000, 2], 2, "bf16"),
    (32, [1, 2, 3, 8, 130, 999], 3, "bf16"),
    (16, [1, 3, 5, 7, 511, 1025], 8, "bf16"),
    (128, [700, 64, 1, 0], 2, "bf16"),
    (64, [1500, 33, 0, 640], 4, "e4m3"),
    (128, [900, 1, 65], 1, "e4m3"),
    (16, [300, 17], 5, "e4m3"),
    (16, [1, 3, 5, 7, 511, 1025], 8, "e4m3"),
    (128, [2000, 97, 40, 0], 2, "e4m3"),
    (48, [64, 96, 31, 2049], 1, "e4m3"),
    (80, [300, 900, 1], 2, "e4m3"),
    (80, [700, 5], 1, "bf16"),
    (128, [1300, 64, 1, 0, 511], 1, "bf16"),   # one page per tile, two head groups
    (1, [77, 3000, 2, 65], 1, "bf16"),
    (7, [129, 2, 1000], 1, "bf16"),
    # P in {3, 5, 6, 7}, one query token: the strided gather (rows y0 + kP of each page)
    (64, [1, 63, 64, 65, 3000], 6, "e4m3"),
    (128, [2049, 7, 640], 7, "e4m3"),
    (64, [1300, 5, 4097, 70], 5, "bf16"),
    (16, [1, 2, 3, 4, 5, 6, 7, 64, 65, 2000], 7, "bf16"),
    (128, [700, 64, 1, 0, 191, 192, 193], 3, "bf16"),   # two head groups; page-edge lengths
    # other P not dividing 8: gather partition r mod gcd(P, 8), drop other owners' tokens
    (16, [1, 3, 5, 7, 511, 1025, 2049], 16, "bf16"),  # gather 8, keep 1 of 2
    (32, [300, 2049, 17, 0], 6, "bf16"),              # gather 2, keep 1 of 3
    (64, [700, 65, 1300], 12, "e4m3"),                # gather 4, keep 1 of 3
    (16, [40, 999, 3, 70], 17, "bf16"),               # 17 / 1 > 16: the CUDA-core kernel
]


@pytest.mark.parametrize("heads,lens,num_parts,kv_dtype", SHAPES)
def test_random_shapes_with_poisoned_tails(heads, lens, num_parts, kv_dtype):
    """Unused rows of the last page and all unowned pages hold NaN: they must
    never reach an output."""
    case = workloads.make_decode_case(f"h{heads}_p{num_parts}_{kv_dtype}", heads, lens,
                                      num_parts=num_parts, kv_dtype=kv_dtype, seed=heads + num_parts,
                                      device="cuda", tail_poison=True, pool_pages=sum(
                                          (L + 63) // 64 for L in lens) + 3)
    _check_all(case, atol=FP8_ATOL if kv_dtype == "e4m3" else None)


def test_many_short_requests():
    """600 requests of 1..300 tokens: every CTA walks several requests, and
    many of them end mid-tile."""
    lens = [int(x) for x in torch.randint(1, 301, (600,), generator=torch.Generator().manual_seed(3))]
    case = workloads.make_decode_case("many_short", 16, lens, seed=3, device="cuda",
                                      tail_poison=True, pool_pages=sum((L + 63) // 64 for L in lens) + 3)
    _check_all(case, bases=(0,))


@pytest.mark.parametrize("num_parts,kv_dtype", [(1, "bf16"), (2, "bf16"), (3, "bf16"), (8, "e4m3")])
def test_requests_sharing_cache_pages(num_parts, kv_dtype):
    """Block tables that alias physical pages, as a shared prompt prefix
    does: requests 1 and 2 reuse request 0's first 40 and 39 pages, and
    request 3 maps both of its logical pages to one physical page."""
    lens = [3000, 3100, 2600, 128, 700]
    case = workloads.make_decode_case("shared", 64, lens, seed=61, device="cuda",
                                      kv_dtype=kv_dtype, num_parts=num_parts)
    bt = case.block_table
    bt[1, :40] = bt[0, :40]
    bt[2, :39] = bt[0, :39]
    bt[3, 1] = bt[3, 0]
    _check_all(case, bases=(0,), atol=FP8_ATOL if kv_dtype == "e4m3" else None)


def test_single_request_spread_over_every_cta():
    """One long request: every CTA holds a split, the last one merges them."""
    case = workloads.make_decode_case("one_long", 64, [150000], seed=21, device="cuda")
    out, lse = run_partial(case, 0, 0)
    ro, rl = oracle_partial_sub(oracle, case, [0], 0, 0)
    assert_out_close(out, ro[:, None], what="one long request")
    assert_lse_close(lse, rl[:, None], 0)


def test_long32k_full_size_every_request():
    case = workloads.config_long32k(device="cuda")
    out, lse = run_partial(case, 0, 0)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    check_requests(oracle, case, out, lse, 0, 0, range(case.batch), what="long32k")


def test_dcp8_full_size_partials_and_combine():
    case = workloads.config_dcp8(device="cuda")
    B, H = case.batch, case.heads
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table)
    outs = torch.empty(8, B, 1, H, 512, dtype=torch.bfloat16, device="cuda")
    lses = torch.empty(8, B, 1, H, dtype=torch.float32, device="cuda")
    for r in range(8):
        run_partial(case, r, 1, workspace=ws, out=outs[r], lse=lses[r])
    assert mla.check_workspace(ws) == 0
    lens = case.seq_lens.cpu().tolist()
    for r in range(8):
        check_requests(oracle, case, outs[r], lses[r], r, 1, DCP8_LONG + DCP8_SHORT, chunk=4,
                       what=f"dcp8 part {r}")
        assert_neutral(outs[r], lses[r], [b for b in DCP8_SHORT if r >= lens[b]])
    merged = torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device="cuda")
    merged_lse = torch.empty(B, 1, H, dtype=torch.float32, device="cuda")
    mla.lse_combine(outs.view(8, B, H, 512), lses.view(8, B, H), 8, merged.view(B, H, 512),
                    lse_base=1, out_lse=merged_lse.view(B, H))
    check_requests(oracle, case, merged, merged_lse, 0, 1, DCP8_LONG + DCP8_SHORT, num_parts=1,
                   chunk=4, what="dcp8 merged vs unpartitioned")


def test_fp8_full_size_every_request():
    case = workloads.config_fp8(device="cuda")
    out, lse = run_partial(case, 0, 0)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    check_requests(oracle, case, out, lse, 0, 0, range(case.batch), atol=FP8_ATOL, what="fp8")


def test_outputs_are_deterministic_and_placement_free():
    case = workloads.make_decode_case("det", 64, [5000, 77, 12000], seed=4, device="cuda",
                                      num_parts=2, pool_pages=400)
    a = run_partial(case, 1, 0)
    b = run_partial(case, 1, 0)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])
    perm = torch.randperm(case.num_pages, generator=torch.Generator().manual_seed(1)).cuda()
    kv2 = torch.empty_like(case.kv_pages)
    kv2[perm] = case.kv_pages
    bt2 = perm[case.block_table.long()].to(torch.int32)
    moved = workloads.DecodeCase(case.name, case.q, kv2, bt2, case.seq_lens, case.kv_dtype,
                                 case.kv_scale, case.sm_scale, case.num_parts)
    c = run_partial(moved, 1, 0)
    assert torch.equal(a[0].view(torch.int16), c[0].view(torch.int16))
    assert torch.equal(a[1], c[1])


def test_bounds_are_checked_in_the_kernel():
    """An out-of-range page index and an over-long length are skipped and
    reported, never dereferenced."""
    case = workloads.make_decode_case("bounds", 16, [130, 64], seed=2, device="cuda")
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table)
    run_partial(case, 0, 0, workspace=ws)
    assert mla.check_workspace(ws) == 0
    bad = case.block_table.clone()
    bad[0, 1] = case.num_pages + 1000
    broken = workloads.DecodeCase(case.name, case.q, case.kv_pages, bad, case.seq_lens,
                                  case.kv_dtype, case.kv_scale, case.sm_scale, 1)
    run_partial(broken, 0, 0, workspace=ws)
    assert mla.check_workspace(ws) == -9
    too_long = case.seq_lens.clone()
    too_long[1] = 64 * case.block_table.shape[1] + 1
    broken = workloads.DecodeCase(case.name, case.q, case.kv_pages, case.block_table, too_long,
                                  case.kv_dtype, case.kv_scale, case.sm_scale, 1)
    run_partial(broken, 0, 0, workspace=ws)
    assert mla.check_workspace(ws) == -9
    run_partial(case, 0, 0, workspace=ws)
    assert mla.check_workspace(ws) == 0


def test_multi_token_query_is_rejected_off_the_tensor_core_path():
    """Several query tokens run on the tensor-core kernel only; with P = 17
    (17 / gcd(17, 8) > 16: the CUDA-core kernel) the call is refused before
    launching."""
    case = workloads.config_small(device="cuda")
    q2 = torch.zeros(1, 2, 16, 576, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1, 2, 16, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 2, 16, dtype=torch.float32, device="cuda")
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table)
    with pytest.raises(mla.MlaError) as e:
        mla.decode_partial(q2, case.kv_pages, case.block_table, case.seq_lens, 0, 17,
                           case.sm_scale, 0, out, lse, workspace=ws)
    assert e.value.status == -2


def test_many_back_to_back_calls_never_time_out_and_stay_identical():
    """Pipeline races (a lost or aliased barrier phase) would show up as a
    timeout reported in the workspace or as differing outputs."""
    case = workloads.config_long32k(device="cuda", batch=32, pool_pages=17000, seed=3)
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table)
    ref_out, ref_lse = run_partial(case, 0, 0, workspace=ws)
    out = torch.empty_like(ref_out)
    lse = torch.empty_like(ref_lse)
    for _ in range(300):
        mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, 0, 1,
                           case.sm_scale, 0, out, lse, workspace=ws)
    assert mla.check_workspace(ws) == 0
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse, ref_lse)


@pytest.mark.parametrize("num_parts", [1, 2])
def test_growing_scores_take_the_rescale_path(num_parts):
    """The rope dims of the keys grow along the sequence, so a later tile's
    maximum exceeds the running maximum by far more than 2^8 and O must be
    rescaled; the values (latent dims) keep their N(0, 1) scale."""
    case = workloads.make_decode_case("growing", 64, [2000, 700, 129], seed=12, device="cuda",
                                      num_parts=num_parts)
    bt = case.block_table.cpu()
    kv = case.kv_pages.float()
    for b, L in enumerate(case.seq_lens.cpu().tolist()):
        for i in range((L + 63) // 64):
            kv[int(bt[b, i]), :, 512:] *= 1.0 + 1.5 * i
    case.kv_pages = kv.to(torch.bfloat16)
    _check_all(case)


@pytest.mark.parametrize("num_parts", [1, 4])
@pytest.mark.parametrize("q_shift", [16, -24])
def test_fp8_query_far_outside_f16_range(q_shift, num_parts):
    """An e4m3 cache runs its MMAs on e4m3 operands: Q is rescaled by a power of
    two and split into two e4m3 terms, so a query of magnitude 2^16 (past the
    e4m3 maximum) or 2^-24 (far below its subnormals) gives the same
    attention as the unscaled one; sm_scale carries the opposite power so
    that the scores are ordinary."""
    case = workloads.make_decode_case("fp8_qshift", 64, [700, 65, 1300], seed=30 + q_shift,
                                      device="cuda", kv_dtype="e4m3", num_parts=num_parts)
    case.q = (case.q.float() * 2.0 ** q_shift).to(torch.bfloat16)
    case.sm_scale = case.sm_scale * 2.0 ** -q_shift
    _check_all(case, bases=(0,), atol=FP8_ATOL)


@pytest.mark.parametrize("num_parts", [1, 3])
def test_fp8_cache_of_subnormal_codes(num_parts):
    """Every cached code has a zero exponent field: OCP e4m3 subnormals,
    (m / 8) * 2^-6 times the scale.  With a scale of 64 they are ordinary
    keys and values, and the kernel's e4m3 MMAs must take them as stored; a
    flush to zero anywhere would show in the relative-norm bound, which
    holds for outputs of any magnitude."""
    case = workloads.make_decode_case("fp8_subnormal", 64, [700, 65, 1300], seed=41,
                                      device="cuda", kv_dtype="e4m3", num_parts=num_parts)
    case.kv_pages &= 0x87
    case.kv_scale = 64.0
    _check_all(case, bases=(0, 1), atol=FP8_ATOL)


@pytest.mark.parametrize("num_parts", [1, 3])
def test_fp8_attention_sink_with_a_long_tail(num_parts):
    """Each request's first token scores 10 nats above all the others, so
    every other weight is e^-10 (about 2^-14.4) of the maximum, yet the
    20,000-token tail holds nearly half of the softmax mass.  P enters the
    e4m3 MMAs as two terms; weights that small must keep a value (its lo
    term is e5m2) or the output collapses onto the first token's row."""
    case = workloads.make_decode_case("fp8_sink", 64, [20000, 3000], seed=52, device="cuda",
                                      kv_dtype="e4m3", num_parts=num_parts)
    kv = case.kv_pages.clone()
    kv[:, :, 512:] = 0                       # rope codes: +0, so every score is 0 ...
    bt = case.block_table.cpu()
    for b in range(case.batch):
        kv[int(bt[b, 0]), 0, 512:] = 0x78    # ... but token 0's: e4m3 code of 256
    case.kv_pages = kv
    q = torch.zeros_like(case.q, dtype=torch.float32)
    q[..., 512:] = 10.0 / (case.sm_scale * 64 * 256.0 * case.kv_scale)
    case.q = q.to(torch.bfloat16)
    _check_all(case, bases=(0,), atol=FP8_ATOL)
