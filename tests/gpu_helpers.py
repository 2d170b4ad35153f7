"""Helpers of the GPU parity tests: run the library, fetch only what the oracle
needs, and compare with the tolerances of the decode-partial contract.

Tolerances (bf16 outputs): max |gpu - oracle| <= 2e-2 and
||gpu - oracle||_2 / ||oracle||_2 <= 1e-2; LSE: |gpu - oracle| <= 5e-3 in natural
log (a base-2 LSE is converted first); e4m3 KV: max abs <= 6e-2 against the
oracle fed the same dequantised values.  Positions where the oracle's LSE is
-inf must be -inf on the GPU too, with out exactly 0.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import mla_paged_decode_gb300 as mla
from casebits import bits, subcase_bits  # noqa: F401

OUT_ATOL = 2e-2
OUT_REL = 1e-2
LSE_ATOL = 5e-3
FP8_ATOL = 6e-2


def run_partial(case, part_id, lse_base=0, workspace=None, out=None, lse=None):
    B, H = case.batch, case.heads
    dev = case.q.device
    out = out if out is not None else torch.full((B, 1, H, 512), float("nan"),
                                                 dtype=torch.bfloat16, device=dev)
    lse = lse if lse is not None else torch.full((B, 1, H), float("nan"), dtype=torch.float32,
                                                 device=dev)
    if workspace is None:
        workspace = mla.make_workspace(case.q, case.kv_pages, case.block_table, case.kv_scale)
    mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, part_id,
                       case.num_parts, case.sm_scale, lse_base, out, lse,
                       kv_scale=case.kv_scale, workspace=workspace)
    return out, lse


def oracle_partial_sub(oracle, case, requests, part_id, lse_base=0, num_parts=None):
    q, kv, bt, lens = subcase_bits(case, requests)
    return oracle.decode_partial(q, kv, bt, lens, part_id,
                                 case.num_parts if num_parts is None else num_parts,
                                 case.sm_scale, lse_base, kv_dtype=case.kv_dtype,
                                 kv_scale=case.kv_scale)


def to_natural(lse: np.ndarray, base: int) -> np.ndarray:
    return lse * math.log(2.0) if base == 1 else lse


def assert_out_close(gpu_out, ref, atol=OUT_ATOL, rel=OUT_REL, what=""):
    g = gpu_out.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    nref = np.linalg.norm(ref)
    assert err.max() <= atol, f"{what}: max abs err {err.max():.3e} > {atol}"
    if nref > 0:
        r = np.linalg.norm(g - ref) / nref
        assert r <= rel, f"{what}: rel err {r:.3e} > {rel}"
    return float(err.max())


def assert_lse_close(gpu_lse, ref, base, atol=LSE_ATOL, what=""):
    g = gpu_lse.detach().cpu().numpy().astype(np.float64).reshape(ref.shape)
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(g), ninf), f"{what}: -inf pattern differs"
    if (~ninf).any():
        e = np.abs(to_natural(g[~ninf], base) - to_natural(ref[~ninf], base))
        assert np.all(np.isfinite(g[~ninf])), f"{what}: non-finite lse"
        assert e.max() <= atol, f"{what}: lse err {e.max():.3e} > {atol}"


def assert_neutral(gpu_out, gpu_lse, mask_rows):
    """Rows (requests) in mask_rows must be exactly (0, -inf)."""
    o = gpu_out.detach().cpu()
    l = gpu_lse.detach().cpu()
    for b in mask_rows:
        assert torch.all(o[b].view(torch.int16) == 0), f"request {b}: out not exactly 0"
        assert torch.all(torch.isneginf(l[b])), f"request {b}: lse not -inf"


def check_requests(oracle, case, out, lse, part_id, lse_base, requests, atol=OUT_ATOL,
                   num_parts=None, chunk=8, what=""):
    """Every request in `requests` against the oracle, `chunk` requests at a
    time (only their pages leave the GPU, so host memory stays bounded).
    out / lse are the GPU results for the whole batch ([B, 1, H, 512] and
    [B, 1, H]); returns the largest absolute output error seen."""
    worst = 0.0
    requests = list(requests)
    for i in range(0, len(requests), chunk):
        sel = requests[i:i + chunk]
        ro, rl = oracle_partial_sub(oracle, case, sel, part_id, lse_base, num_parts=num_parts)
        w = f"{what} requests {sel[0]}..{sel[-1]}"
        worst = max(worst, assert_out_close(out[sel], ro[:, None], atol=atol, what=w))
        assert_lse_close(lse[sel], rl[:, None], lse_base, what=w)
    return worst
