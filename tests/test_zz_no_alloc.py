"""The allocation-free decode entry point, called through the C ABI.

Some callers cannot call cudaMalloc (runtimes that own all of HBM, decode
loops that cannot take an allocation's device synchronisation, C hosts with
no allocator).  mla_decode_partial_noalloc serves them from scratch built into
the library.  This checks, on two calls in a row (the second one finds the
first one's leftovers in the shared scratch), that its outputs match those of
mla_decode_partial (bitwise: the same kernels run), and that a batch beyond
the built-in limit is refused without a launch.  The file is named so that pytest
collects it last.
"""
import ctypes

import pytest
import torch

import mla_paged_decode_gb300 as mla
import workloads
from gpu_helpers import FP8_ATOL, assert_lse_close, assert_out_close, run_partial

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_decode_gb300 import build
    build.build()
    lib = mla.load_library()
    fn = lib.mla_decode_partial_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, i32, i32, ctypes.c_float, i32, vp, vp,
                   ctypes.POINTER(mla.DecodeDesc), vp]
    fn.restype = i32
    return lib


def _call(lib, case, part_id, base, out, lse):
    d = mla.DecodeDesc(batch=case.batch, num_heads=case.heads, q_len=1, head_dim_qk=576,
                       head_dim_v=512, page_size=64, num_pages=case.num_pages,
                       max_pages_per_seq=case.block_table.shape[1],
                       kv_dtype=0 if case.kv_dtype == "bf16" else 1, kv_scale=case.kv_scale)
    stream = torch.cuda.current_stream().cuda_stream
    return lib.mla_decode_partial_noalloc(
        case.q.data_ptr(), case.kv_pages.data_ptr(), case.block_table.data_ptr(),
        case.seq_lens.data_ptr(), part_id, case.num_parts, case.sm_scale, base,
        out.data_ptr(), lse.data_ptr(), ctypes.byref(d), stream)


# a gather of 64/P rows per page; the strided gather; an e4m3 cache alone and gathered
@pytest.mark.parametrize("num_parts,kv_dtype", [(2, "bf16"), (3, "bf16"), (1, "e4m3"), (4, "e4m3")])
def test_noalloc_matches_the_workspace_entry_point_twice_in_a_row(lib, num_parts, kv_dtype):
    case = workloads.make_decode_case("noalloc", 64, [5000, 77, 12000, 1, 0], num_parts=num_parts,
                                      seed=31, device="cuda", pool_pages=400, kv_dtype=kv_dtype)
    for call, (part_id, base) in enumerate([(0, 0), (1 % num_parts, 1)]):
        ref_out, ref_lse = run_partial(case, part_id, base)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _call(lib, case, part_id, base, out, lse) == 0
        torch.cuda.synchronize()
        ref = ref_out.double().cpu().numpy()
        assert_out_close(out, ref, **({"atol": FP8_ATOL} if kv_dtype == "e4m3" else {}),
                         what=f"no-alloc call {call}")
        assert_lse_close(lse, ref_lse.double().cpu().numpy(), base, what=f"no-alloc call {call}")
        # the same tensor-core kernels on the same grid (the no-alloc grid is
        # capped at 152 CTAs: with more SMs the split points differ)
        if torch.cuda.get_device_properties(0).multi_processor_count <= 152:
            assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), call
            assert torch.equal(lse, ref_lse), call


def test_noalloc_refuses_batches_beyond_its_scratch(lib):
    case = workloads.make_decode_case("noalloc_big", 64, [64] * 8193, seed=1, device="cuda")
    out = torch.zeros(case.batch, 1, 64, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(case.batch, 1, 64, dtype=torch.float32, device="cuda")
    assert _call(lib, case, 0, 0, out, lse) == -5
    assert torch.all(out == 0) and torch.all(lse == 0)
