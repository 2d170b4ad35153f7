"""Marshalling helpers shared by the tests: torch tensors -> raw numpy bits."""
from __future__ import annotations

import numpy as np
import torch


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.uint8:
        return t.numpy()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def case_bits(case):
    """(q_bits, kv_bits, block_table, seq_lens) of a workloads.DecodeCase."""
    return (bits(case.q), bits(case.kv_pages), case.block_table.cpu().numpy(),
            case.seq_lens.cpu().numpy())


def oracle_partial(oracle, case, part_id, lse_base=0, requests=None):
    q, kv, bt, lens = case_bits(case)
    return oracle.decode_partial(q, kv, bt, lens, part_id, case.num_parts, case.sm_scale,
                                 lse_base, kv_dtype=case.kv_dtype, kv_scale=case.kv_scale,
                                 requests=requests)
