"""The C-ABI library: it loads, exports every function include/*.h declares, and
rejects bad arguments on the host before anything reaches a GPU.

None of these calls launches work: every one fails argument validation first,
so they run on machines without a GPU.
"""
import ctypes
import glob
import os
import re

import pytest

import mla_paged_decode_gb300 as mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"\b(mla_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(mla.library_path()):
        from mla_paged_decode_gb300 import build
        build.build()
    return mla.load_library()


def test_header_declares_the_two_operations():
    names = declared_functions()
    assert "mla_decode_partial" in names and "mla_lse_combine" in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exported_symbols_are_c_linkage():
    out = os.popen(f"nm -D --defined-only {mla.library_path()}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def _desc(**kw):
    base = dict(batch=2, num_heads=16, q_len=1, head_dim_qk=576, head_dim_v=512, page_size=64,
                num_pages=8, max_pages_per_seq=4, kv_dtype=0, kv_scale=1.0)
    base.update(kw)
    return mla.DecodeDesc(**base)


FAKE = 1 << 20  # a 256-aligned non-null address that is never dereferenced


def _partial(lib, d, *, part_id=0, num_parts=1, lse_base=0, sm_scale=0.1, q=FAKE, ws=FAKE,
             ws_bytes=1 << 40):
    return lib.mla_decode_partial(q, FAKE, FAKE, FAKE, part_id, num_parts, sm_scale, lse_base,
                                  FAKE, FAKE, ctypes.byref(d) if d is not None else None,
                                  ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q_len=17), -2), (dict(q_len=0), -2), (dict(head_dim_qk=512), -2),
    (dict(head_dim_v=576), -2), (dict(page_size=32), -2), (dict(num_heads=0), -2),
    (dict(num_heads=129), -2), (dict(num_pages=0), -2), (dict(max_pages_per_seq=0), -2),
    (dict(batch=-1), -2), (dict(kv_dtype=7), -6), (dict(kv_dtype=1, kv_scale=0.0), -6),
    (dict(kv_dtype=1, kv_scale=float("nan")), -6),
])
def test_bad_descriptor_is_rejected(lib, kw, code):
    assert _partial(lib, _desc(**kw)) == code


def test_bad_partition_is_rejected(lib):
    for part_id, num_parts in [(0, 0), (-1, 2), (2, 2), (5, 4)]:
        assert _partial(lib, _desc(), part_id=part_id, num_parts=num_parts) == -3


def test_bad_enum_and_scale_are_rejected(lib):
    assert _partial(lib, _desc(), lse_base=2) == -6
    assert _partial(lib, _desc(), sm_scale=float("inf")) == -6


def test_null_and_misaligned_pointers_are_rejected(lib):
    assert _partial(lib, None) == -1
    assert _partial(lib, _desc(), q=0) == -1
    assert _partial(lib, _desc(), ws=0) == -1
    assert _partial(lib, _desc(), q=FAKE + 2) == -4
    assert _partial(lib, _desc(), ws=FAKE + 16) == -4


def test_empty_batch_is_a_no_op(lib):
    assert _partial(lib, _desc(batch=0), q=0, ws=0) == 0


def test_workspace_size_is_sane(lib):
    d = _desc(batch=64, num_heads=64)
    n = lib.mla_decode_workspace_size(ctypes.byref(d), 152)
    assert n > 0 and n % 256 == 0
    assert lib.mla_decode_workspace_size(ctypes.byref(_desc(q_len=17)), 152) == 0
    assert lib.mla_decode_workspace_size(None, 152) == 0
    more = lib.mla_decode_workspace_size(ctypes.byref(d), 304)
    assert more > n


def test_combine_rejects_bad_arguments(lib):
    def call(num_parts=2, **kw):
        base = dict(num_tokens=4, num_heads=16, head_dim=512, lse_base=0, out_lse=None)
        base.update(kw)
        d = mla.CombineDesc(**base)
        return lib.mla_lse_combine(FAKE, FAKE, num_parts, FAKE, ctypes.byref(d), None)
    assert call(num_parts=0) == -3
    assert call(num_parts=100000) == -3
    assert call(head_dim=12) == -2
    assert call(head_dim=0) == -2
    assert call(num_heads=0) == -2
    assert call(lse_base=3) == -6
    assert call(num_tokens=0) == 0
    assert lib.mla_lse_combine(0, FAKE, 2, FAKE, ctypes.byref(mla.CombineDesc(
        num_tokens=1, num_heads=1, head_dim=8, lse_base=0, out_lse=None)), None) == -1


def test_status_strings(lib):
    for code in range(-10, 1):
        assert lib.mla_status_string(code)
    assert lib.mla_version() >= 100


def test_python_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 16, 576, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mla.decode_partial(q, q, q, q, 0, 1, 0.1, 0, q, q)


def _append(lib, d, *, part_id=0, num_parts=1, kv_new=FAKE, kv=FAKE, err=None):
    return lib.mla_kv_append(kv_new, kv, FAKE, FAKE, part_id, num_parts,
                             ctypes.byref(d) if d is not None else None, err, None)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim_qk=512), -2), (dict(page_size=128), -2), (dict(num_pages=0), -2),
    (dict(max_pages_per_seq=0), -2), (dict(batch=-3), -2), (dict(kv_dtype=2), -6),
    (dict(kv_dtype=1, kv_scale=-1.0), -6), (dict(kv_dtype=1, kv_scale=float("inf")), -6),
])
def test_append_rejects_a_bad_cache_descriptor(lib, kw, code):
    assert _append(lib, _desc(**kw)) == code


def test_append_ignores_the_query_fields_of_the_descriptor(lib):
    # q_len, num_heads and head_dim_v describe a query, not the cache: a
    # descriptor with other values still gets as far as the pointer checks
    assert _append(lib, _desc(q_len=3, num_heads=0, head_dim_v=1), kv_new=0) == -1


def test_append_rejects_bad_partition_pointers_and_alignment(lib):
    for part_id, num_parts in [(0, 0), (3, 3), (-1, 1)]:
        assert _append(lib, _desc(), part_id=part_id, num_parts=num_parts) == -3
    assert _append(lib, None) == -1
    assert _append(lib, _desc(), kv_new=0) == -1
    assert _append(lib, _desc(), kv=0) == -1
    assert _append(lib, _desc(), kv_new=FAKE + 8) == -4
    assert _append(lib, _desc(), kv=FAKE + 4) == -4
    assert _append(lib, _desc(), err=FAKE + 2) == -4
    assert _append(lib, _desc(batch=0), kv_new=0, kv=0) == 0


def _dcp(lib, d, *, num_parts=2, partials=FAKE, out=FAKE, out_lse=None, ws=FAKE, ws_bytes=1 << 40):
    return lib.mla_decode_dcp(FAKE, FAKE, FAKE, FAKE, num_parts, 0.1, 0, partials, FAKE, out,
                              out_lse, ctypes.byref(d) if d is not None else None, ws, ws_bytes,
                              None)


def test_dcp_rejects_bad_arguments(lib):
    assert _dcp(lib, _desc(q_len=17)) == -2
    assert _dcp(lib, _desc(), num_parts=0) == -3
    assert _dcp(lib, _desc(), num_parts=257) == -3
    assert _dcp(lib, None) == -1
    assert _dcp(lib, _desc(), partials=0) == -1
    assert _dcp(lib, _desc(), out=FAKE + 8) == -4
    assert _dcp(lib, _desc(), out_lse=FAKE + 2) == -4
    assert _dcp(lib, _desc(batch=0), partials=0, out=0, ws=0) == 0


def test_dcp_workspace_covers_every_partition(lib):
    d = _desc(batch=64, num_heads=16)
    one = lib.mla_decode_workspace_size(ctypes.byref(d), 152)
    eight = lib.mla_decode_dcp_workspace_size(ctypes.byref(d), 8, 152)
    assert eight > one and eight % 256 == 0
    assert lib.mla_decode_dcp_workspace_size(ctypes.byref(d), 0, 152) == 0


def _meta(lib, part_id=0, num_parts=2, seq=FAKE, out=FAKE, err=None, **kw):
    base = dict(batch=4, num_req_slots=8, req_to_token_width=256, max_pages_per_seq=4,
                extra_tokens=0, pad_value=0, page_size=64)
    base.update(kw)
    d = mla.DcpMetaDesc(**base)
    return lib.mla_dcp_local_metadata(seq, FAKE, FAKE, part_id, num_parts, ctypes.byref(d), out,
                                      FAKE, FAKE, err, None)


def test_dcp_metadata_rejects_bad_arguments(lib):
    assert _meta(lib, num_parts=0) == -3
    assert _meta(lib, part_id=2) == -3
    assert _meta(lib, page_size=32) == -2
    assert _meta(lib, num_req_slots=0) == -2
    assert _meta(lib, max_pages_per_seq=0) == -2
    assert _meta(lib, extra_tokens=-1) == -6
    assert _meta(lib, seq=0) == -1
    assert _meta(lib, out=FAKE + 2) == -4
    assert _meta(lib, err=FAKE + 1) == -4
    assert _meta(lib, batch=0, seq=0, out=0) == 0


def test_several_query_tokens_need_the_tensor_core_path(lib):
    # num_parts / gcd(num_parts, 8) > 16 runs the CUDA-core kernel, which
    # takes one query token (17 / 1, 136 / 8); 3 and 48 / 8 stay on the tensor cores
    assert _partial(lib, _desc(q_len=2), part_id=0, num_parts=17) == -2
    assert _partial(lib, _desc(q_len=2), part_id=5, num_parts=136) == -2
    assert _dcp(lib, _desc(q_len=4), num_parts=17) == -2


def test_selftest_rejects_bad_arguments(lib):
    lib.mla_selftest_bounded_wait.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    assert lib.mla_selftest_bounded_wait(None, 10**6, None) == -1
    assert lib.mla_selftest_bounded_wait(FAKE + 16, 10**6, None) == -4
    assert lib.mla_selftest_bounded_wait(FAKE, 10, None) == -6
    assert lib.mla_selftest_bounded_wait(FAKE, 2 * 10**8, None) == -6


def test_arch_gate_takes_sm103_only(lib):
    """The kernels are built for sm_103a: every other compute capability of the
    family or around it is refused (MLA_ERR_DEVICE before any launch)."""
    lib.mla_arch_supported.argtypes = [ctypes.c_int, ctypes.c_int]
    assert lib.mla_arch_supported(10, 3) == 1
    for major, minor in [(10, 0), (10, 1), (10, 2), (11, 0), (12, 0), (12, 1), (9, 0), (8, 9)]:
        assert lib.mla_arch_supported(major, minor) == 0, (major, minor)


def test_a_valid_call_without_a_gpu_returns_an_error():
    """With every argument valid, a machine without a usable GPU gets a
    status, not a crash (the device query fails before any launch)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("the fake pointers must never reach a real launch")
    lib = mla.load_library() if os.path.exists(mla.library_path()) else None
    if lib is None:
        pytest.skip("library not built")
    st = _partial(lib, _desc())
    assert st in (-7, -8), st   # MLA_ERR_CUDA or MLA_ERR_DEVICE
