"""Python binding of the GB300 MLA paged-decode C ABI (include/mla_decode.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``_lib/libmla_decode.so``.  PyTorch supplies device memory and the
current stream.  If the library is not built, every call raises: there is no
CPU fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

__all__ = [
    "MlaError", "LSE_NATURAL", "LSE_BASE2", "decode_partial", "lse_combine",
    "workspace_size", "make_workspace", "check_workspace", "library_path", "load_library",
    "decode_partial_noalloc",
]

LSE_NATURAL = 0
LSE_BASE2 = 1
KV_BF16 = 0
KV_E4M3 = 1
_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libmla_decode.so")
_lib = None
_lock = threading.Lock()


class MlaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


class DecodeDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("q_len", ctypes.c_int32), ("head_dim_qk", ctypes.c_int32),
                ("head_dim_v", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("kv_scale", ctypes.c_float)]


class CombineDesc(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("lse_base", ctypes.c_int32),
                ("out_lse", ctypes.c_void_p)]


def library_path() -> str:
    return _LIB_PATH


class DcpMetaDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_req_slots", ctypes.c_int32),
                ("req_to_token_width", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("extra_tokens", ctypes.c_int32), ("pad_value", ctypes.c_int32),
                ("page_size", ctypes.c_int32)]


def load_library():
    """Loads the built library (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is not built; run `python -m mla_paged_decode_gb300.build`")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.mla_decode_partial.argtypes = [vp, vp, vp, vp, i32, i32, f32, i32, vp, vp,
                                           ctypes.POINTER(DecodeDesc), vp, sz, vp]
        lib.mla_decode_partial.restype = i32
        lib.mla_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeDesc), i32]
        lib.mla_decode_workspace_size.restype = sz
        lib.mla_decode_check_workspace.argtypes = [vp, vp]
        lib.mla_decode_check_workspace.restype = i32
        lib.mla_decode_dcp.argtypes = [vp, vp, vp, vp, i32, f32, i32, vp, vp, vp, vp,
                                       ctypes.POINTER(DecodeDesc), vp, sz, vp]
        lib.mla_decode_dcp.restype = i32
        lib.mla_decode_dcp_workspace_size.argtypes = [ctypes.POINTER(DecodeDesc), i32, i32]
        lib.mla_decode_dcp_workspace_size.restype = sz
        lib.mla_dcp_local_metadata.argtypes = [vp, vp, vp, i32, i32, ctypes.POINTER(DcpMetaDesc),
                                               vp, vp, vp, vp, vp]
        lib.mla_dcp_local_metadata.restype = i32
        lib.mla_kv_append.argtypes = [vp, vp, vp, vp, i32, i32, ctypes.POINTER(DecodeDesc), vp, vp]
        lib.mla_kv_append.restype = i32
        lib.mla_lse_combine.argtypes = [vp, vp, i32, vp, ctypes.POINTER(CombineDesc), vp]
        lib.mla_lse_combine.restype = i32
        lib.mla_status_string.argtypes = [i32]
        lib.mla_status_string.restype = ctypes.c_char_p
        lib.mla_last_cuda_error.argtypes = []
        lib.mla_last_cuda_error.restype = ctypes.c_char_p
        lib.mla_version.argtypes = []
        lib.mla_version.restype = i32
        lib.mla_selftest_bounded_wait.argtypes = [vp, ctypes.c_int64, vp]
        lib.mla_selftest_bounded_wait.restype = i32
        _lib = lib
        return lib


def _check(status: int):
    if status != 0:
        lib = load_library()
        msg = lib.mla_status_string(status).decode()
        if status == -7:
            msg += ": " + lib.mla_last_cuda_error().decode()
        raise MlaError(status, msg)


def _on(device):
    """The device context for a call: nothing to switch when it is current
    (the switch costs a few microseconds, felt by small decodes)."""
    if torch.cuda.current_device() == device.index:
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _stream_ptr(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def _kv_dtype_code(kv_pages: torch.Tensor) -> int:
    if kv_pages.dtype == torch.bfloat16:
        return KV_BF16
    if kv_pages.dtype in (torch.uint8, torch.float8_e4m3fn):
        return KV_E4M3
    raise TypeError(f"kv_pages must be bf16 or e4m3 bytes, got {kv_pages.dtype}")


_DESCS: dict = {}


def _decode_desc(q, kv_pages, block_table, kv_scale) -> DecodeDesc:
    """The call's size descriptor, built once per distinct set of shapes (the
    library only reads it during the call)."""
    key = (q.shape, kv_pages.shape, kv_pages.dtype, block_table.shape, float(kv_scale))
    d = _DESCS.get(key)
    if d is None:
        d = _make_decode_desc(q, kv_pages, block_table, kv_scale)
        if len(_DESCS) > 256:
            _DESCS.clear()
        _DESCS[key] = d
    return d


def _make_decode_desc(q, kv_pages, block_table, kv_scale) -> DecodeDesc:
    if q.dim() != 4:
        raise ValueError("q must be [B, q_len, H, 576]")
    B, q_len, H, dqk = q.shape
    if kv_pages.dim() != 3:
        raise ValueError("kv_pages must be [num_pages, page_size, 576]")
    return DecodeDesc(batch=B, num_heads=H, q_len=q_len, head_dim_qk=dqk, head_dim_v=512,
                      page_size=kv_pages.shape[1], num_pages=kv_pages.shape[0],
                      max_pages_per_seq=block_table.shape[1] if block_table.dim() == 2 else 0,
                      kv_dtype=_kv_dtype_code(kv_pages), kv_scale=float(kv_scale))


def workspace_size(q: torch.Tensor, kv_pages: torch.Tensor, block_table: torch.Tensor,
                   kv_scale: float = 1.0) -> int:
    d = _decode_desc(q, kv_pages, block_table, kv_scale)
    with torch.cuda.device(q.device):
        n = load_library().mla_decode_workspace_size(ctypes.byref(d), 0)
    if n == 0:
        raise MlaError(-2, "cannot size a workspace for these shapes")
    return n


def make_workspace(q, kv_pages, block_table, kv_scale: float = 1.0) -> torch.Tensor:
    """A zero-filled workspace for these shapes on q's device."""
    return torch.zeros(workspace_size(q, kv_pages, block_table, kv_scale), dtype=torch.uint8,
                       device=q.device)


def _need(t: torch.Tensor, name: str, dtypes, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def decode_partial(q, kv_pages, block_table, seq_lens, part_id: int, num_parts: int,
                   sm_scale: float, lse_base: int, out, lse, *, kv_scale: float = 1.0,
                   workspace: torch.Tensor | None = None, stream=None):
    """mla_decode_partial on torch tensors (see include/mla_decode.h).

    q bf16 [B,1,H,576]; kv_pages bf16 [pages,64,576] or uint8/float8_e4m3fn;
    block_table int32 [B,max_pages]; seq_lens int32 [B] (global lengths);
    out bf16 [B,1,H,512] and lse fp32 [B,1,H] are written in place.
    """
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("decode_partial runs on CUDA tensors only")
    _need(q, "q", (torch.bfloat16,), dev)
    _need(kv_pages, "kv_pages", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn), dev)
    _need(block_table, "block_table", (torch.int32,), dev)
    _need(seq_lens, "seq_lens", (torch.int32,), dev)
    _need(out, "out", (torch.bfloat16,), dev)
    _need(lse, "lse", (torch.float32,), dev)
    d = _decode_desc(q, kv_pages, block_table, kv_scale)
    if seq_lens.numel() != d.batch or block_table.dim() != 2 or block_table.shape[0] != d.batch:
        raise ValueError("seq_lens / block_table do not match the batch")
    if out.numel() != d.batch * d.q_len * d.num_heads * 512 or lse.numel() != d.batch * d.q_len * d.num_heads:
        raise ValueError("out must be [B,1,H,512] and lse [B,1,H]")
    if workspace is None:
        workspace = make_workspace(q, kv_pages, block_table, kv_scale)
    _need(workspace, "workspace", (torch.uint8,), dev)
    with _on(dev):
        st = load_library().mla_decode_partial(
            q.data_ptr(), kv_pages.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(),
            int(part_id), int(num_parts), float(sm_scale), int(lse_base), out.data_ptr(),
            lse.data_ptr(), ctypes.byref(d), workspace.data_ptr(), workspace.numel(),
            _stream_ptr(stream, dev))
    _check(st)
    return out, lse


def kv_append(kv_new, kv_pages, block_table, positions, part_id: int = 0, num_parts: int = 1, *,
              kv_scale: float = 1.0, error_word=None, stream=None):
    """mla_kv_append on torch tensors (see include/mla_decode.h).

    kv_new bf16 [B, 576] (or [B, 1, 576]): each request's new token row;
    positions int32 [B]: its global index (the length before the append;
    negative skips the request).  Row positions[b] is written into kv_pages
    (bf16, or uint8/float8_e4m3fn quantised with kv_scale) in place, if
    partition part_id of num_parts owns it.  error_word: optional int32 [1]
    device tensor that receives bit 0 for a row whose page entry is out of
    range (that row is skipped).
    """
    dev = kv_pages.device
    if dev.type != "cuda":
        raise ValueError("kv_append runs on CUDA tensors only")
    _need(kv_new, "kv_new", (torch.bfloat16,), dev)
    _need(kv_pages, "kv_pages", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn), dev)
    _need(block_table, "block_table", (torch.int32,), dev)
    _need(positions, "positions", (torch.int32,), dev)
    if kv_pages.dim() != 3 or block_table.dim() != 2:
        raise ValueError("kv_pages must be [num_pages, 64, 576] and block_table [B, max_pages]")
    B = positions.numel()
    if kv_new.numel() != B * 576 or kv_new.shape[-1] != 576 or block_table.shape[0] != B:
        raise ValueError("kv_new must be [B, 576] and block_table [B, max_pages] for B positions")
    if error_word is not None:
        _need(error_word, "error_word", (torch.int32,), dev)
    d = DecodeDesc(batch=B, num_heads=1, q_len=1, head_dim_qk=576, head_dim_v=512,
                   page_size=kv_pages.shape[1], num_pages=kv_pages.shape[0],
                   max_pages_per_seq=block_table.shape[1], kv_dtype=_kv_dtype_code(kv_pages),
                   kv_scale=float(kv_scale))
    with _on(dev):
        st = load_library().mla_kv_append(
            kv_new.data_ptr(), kv_pages.data_ptr(), block_table.data_ptr(), positions.data_ptr(),
            int(part_id), int(num_parts), ctypes.byref(d),
            error_word.data_ptr() if error_word is not None else None, _stream_ptr(stream, dev))
    _check(st)
    return kv_pages


def make_dcp_workspace(q, kv_pages, block_table, num_parts: int, kv_scale: float = 1.0):
    """A zero-filled workspace for decode_dcp over num_parts partitions."""
    d = _decode_desc(q, kv_pages, block_table, kv_scale)
    with torch.cuda.device(q.device):
        n = load_library().mla_decode_dcp_workspace_size(ctypes.byref(d), int(num_parts), 0)
    if n == 0:
        raise MlaError(-2, "cannot size a workspace for these shapes")
    return torch.zeros(n, dtype=torch.uint8, device=q.device)


def decode_dcp(q, kv_pages, block_table, seq_lens, num_parts: int, sm_scale: float,
               lse_base: int, *, partials=None, partial_lses=None, out=None, out_lse=None,
               kv_scale: float = 1.0, workspace=None, stream=None):
    """mla_decode_dcp: every partition's (out, lse) and their merge in one call.

    Returns (out [B,1,H,512], out_lse [B,1,H] or None, partials [P,B,1,H,512],
    partial_lses [P,B,1,H]); the output tensors are allocated when not given.
    """
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("decode_dcp runs on CUDA tensors only")
    _need(q, "q", (torch.bfloat16,), dev)
    _need(kv_pages, "kv_pages", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn), dev)
    _need(block_table, "block_table", (torch.int32,), dev)
    _need(seq_lens, "seq_lens", (torch.int32,), dev)
    d = _decode_desc(q, kv_pages, block_table, kv_scale)
    B, T, H, P = d.batch, d.q_len, d.num_heads, int(num_parts)
    if seq_lens.numel() != B or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("seq_lens / block_table do not match the batch")
    if partials is None:
        partials = torch.empty(P, B, T, H, 512, dtype=torch.bfloat16, device=dev)
    if partial_lses is None:
        partial_lses = torch.empty(P, B, T, H, dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty(B, T, H, 512, dtype=torch.bfloat16, device=dev)
    _need(partials, "partials", (torch.bfloat16,), dev)
    _need(partial_lses, "partial_lses", (torch.float32,), dev)
    _need(out, "out", (torch.bfloat16,), dev)
    if partials.numel() != P * B * T * H * 512 or partial_lses.numel() != P * B * T * H:
        raise ValueError("partials must be [P,B,q_len,H,512] and partial_lses [P,B,q_len,H]")
    if out.numel() != B * T * H * 512:
        raise ValueError("out must be [B,q_len,H,512]")
    if out_lse is not None:
        _need(out_lse, "out_lse", (torch.float32,), dev)
        if out_lse.numel() != B * T * H:
            raise ValueError("out_lse must be [B,q_len,H]")
    if workspace is None:
        workspace = make_dcp_workspace(q, kv_pages, block_table, P, kv_scale)
    _need(workspace, "workspace", (torch.uint8,), dev)
    with _on(dev):
        st = load_library().mla_decode_dcp(
            q.data_ptr(), kv_pages.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(), P,
            float(sm_scale), int(lse_base), partials.data_ptr(), partial_lses.data_ptr(),
            out.data_ptr(), out_lse.data_ptr() if out_lse is not None else None, ctypes.byref(d),
            workspace.data_ptr(), workspace.numel(), _stream_ptr(stream, dev))
    _check(st)
    return out, out_lse, partials, partial_lses


def dcp_local_metadata(seq_lens, req_pool_indices, req_to_token, part_id: int, num_parts: int,
                       *, max_pages: int, extra_tokens: int = 0, pad_value: int = 0,
                       global_lens=None, local_lens=None, block_table=None, error_word=None,
                       stream=None):
    """mla_dcp_local_metadata: a DCP rank's global and local lengths and its
    rank-local page table [B, max_pages], built on the device (into the given
    buffers when passed, so a captured graph can keep reading them).
    Returns (global_lens, local_lens, block_table)."""
    dev = seq_lens.device
    if dev.type != "cuda":
        raise ValueError("dcp_local_metadata runs on CUDA tensors only")
    _need(seq_lens, "seq_lens", (torch.int32,), dev)
    _need(req_pool_indices, "req_pool_indices", (torch.int32,), dev)
    _need(req_to_token, "req_to_token", (torch.int32,), dev)
    B = seq_lens.numel()
    if req_pool_indices.numel() != B or req_to_token.dim() != 2:
        raise ValueError("req_pool_indices must be [B] and req_to_token [slots, width]")
    global_lens = global_lens if global_lens is not None else torch.empty(B, dtype=torch.int32, device=dev)
    local_lens = local_lens if local_lens is not None else torch.empty(B, dtype=torch.int32, device=dev)
    block_table = block_table if block_table is not None else torch.empty(
        B, int(max_pages), dtype=torch.int32, device=dev)
    for t, n in ((global_lens, "global_lens"), (local_lens, "local_lens"), (block_table, "block_table")):
        _need(t, n, (torch.int32,), dev)
    if global_lens.numel() != B or local_lens.numel() != B or block_table.numel() != B * int(max_pages):
        raise ValueError("output buffers do not match the batch and max_pages")
    if error_word is not None:
        _need(error_word, "error_word", (torch.int32,), dev)
    d = DcpMetaDesc(batch=B, num_req_slots=req_to_token.shape[0],
                    req_to_token_width=req_to_token.shape[1], max_pages_per_seq=int(max_pages),
                    extra_tokens=int(extra_tokens), pad_value=int(pad_value), page_size=64)
    with _on(dev):
        st = load_library().mla_dcp_local_metadata(
            seq_lens.data_ptr(), req_pool_indices.data_ptr(), req_to_token.data_ptr(), int(part_id),
            int(num_parts), ctypes.byref(d), global_lens.data_ptr(), local_lens.data_ptr(),
            block_table.data_ptr(), error_word.data_ptr() if error_word is not None else None,
            _stream_ptr(stream, dev))
    _check(st)
    return global_lens, local_lens, block_table


def check_workspace(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the kernel's bounds
    status: 0, or -9 if a block-table entry or a length was out of bounds."""
    with torch.cuda.device(workspace.device):
        st = load_library().mla_decode_check_workspace(workspace.data_ptr(),
                                                       _stream_ptr(stream, workspace.device))
    if st not in (0, -9):
        _check(st)
    return st


def selftest_bounded_wait(workspace: torch.Tensor, timeout_ns: int, stream=None) -> None:
    """mla_selftest_bounded_wait: two warps wait on barriers that nothing
    completes; the waits give up (after timeout_ns, and on the abort flag)
    and report MLA_ERR_TIMEOUT in the workspace's error word."""
    with torch.cuda.device(workspace.device):
        _check(load_library().mla_selftest_bounded_wait(
            workspace.data_ptr(), int(timeout_ns), _stream_ptr(stream, workspace.device)))


def lse_combine(partials, lses, num_parts: int, out, *, lse_base: int = LSE_NATURAL,
                out_lse=None, stream=None):
    """mla_lse_combine: partials bf16 [P,T,H,D], lses fp32 [P,T,H] -> out bf16 [T,H,D]."""
    dev = partials.device
    if dev.type != "cuda":
        raise ValueError("lse_combine runs on CUDA tensors only")
    _need(partials, "partials", (torch.bfloat16,), dev)
    _need(lses, "lses", (torch.float32,), dev)
    _need(out, "out", (torch.bfloat16,), dev)
    if partials.dim() != 4 or partials.shape[0] != num_parts:
        raise ValueError("partials must be [num_parts, T, H, D]")
    P, T, H, D = partials.shape
    if lses.numel() != P * T * H or out.numel() != T * H * D:
        raise ValueError("lses must be [P,T,H] and out [T,H,D]")
    if out_lse is not None:
        _need(out_lse, "out_lse", (torch.float32,), dev)
        if out_lse.numel() != T * H:
            raise ValueError("out_lse must be [T,H]")
    d = CombineDesc(num_tokens=T, num_heads=H, head_dim=D, lse_base=int(lse_base),
                    out_lse=out_lse.data_ptr() if out_lse is not None else None)
    with _on(dev):
        st = load_library().mla_lse_combine(partials.data_ptr(), lses.data_ptr(), int(num_parts),
                                            out.data_ptr(), ctypes.byref(d), _stream_ptr(stream, dev))
    _check(st)
    return out


def decode_partial_noalloc(q, kv_pages, block_table, seq_lens, part_id: int, num_parts: int,
                           sm_scale: float, lse_base: int, out, lse, *, kv_scale: float = 1.0,
                           stream=None):
    """mla_decode_partial_noalloc: the same call without a workspace, for
    callers that cannot allocate device memory (see include/mla_decode.h).
    It uses scratch built into the library, shared by every call: calls that
    may overlap on the GPU must be serialised by the caller."""
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("decode_partial_noalloc runs on CUDA tensors only")
    _need(q, "q", (torch.bfloat16,), dev)
    _need(kv_pages, "kv_pages", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn), dev)
    _need(block_table, "block_table", (torch.int32,), dev)
    _need(seq_lens, "seq_lens", (torch.int32,), dev)
    _need(out, "out", (torch.bfloat16,), dev)
    _need(lse, "lse", (torch.float32,), dev)
    d = _decode_desc(q, kv_pages, block_table, kv_scale)
    lib = load_library()
    fn = lib.mla_decode_partial_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, i32, i32, ctypes.c_float, i32, vp, vp,
                   ctypes.POINTER(DecodeDesc), vp]
    fn.restype = i32
    with _on(dev):
        st = fn(q.data_ptr(), kv_pages.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(),
                int(part_id), int(num_parts), float(sm_scale), int(lse_base), out.data_ptr(),
                lse.data_ptr(), ctypes.byref(d), _stream_ptr(stream, dev))
    _check(st)
    return out, lse
