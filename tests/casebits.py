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


def subcase_bits(case, requests):
    """Oracle inputs for a subset of requests: only their pages leave the GPU."""
    bt = case.block_table.cpu().numpy()
    lens = case.seq_lens.cpu().numpy()
    pages, new_bt = [], np.zeros((len(requests), bt.shape[1]), dtype=np.int64)
    for i, b in enumerate(requests):
        n = (int(lens[b]) + 63) // 64
        new_bt[i, :n] = np.arange(len(pages), len(pages) + n)
        pages.extend(bt[b, :n].tolist())
    if not pages:
        pages = [0]
    idx = torch.tensor(pages, dtype=torch.long, device=case.kv_pages.device)
    kv_sub = bits(case.kv_pages.index_select(0, idx))
    q_sub = bits(case.q[list(requests)])
    return q_sub, kv_sub, new_bt, lens[list(requests)]
