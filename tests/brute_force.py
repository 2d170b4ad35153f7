"""Pure-Python brute force for tiny cases, written independently of the oracle.

It decodes bf16 with ``struct``, enumerates owned tokens by literally testing
``t % P == r``, and sums with ``math.fsum``.  It exists only to pin the oracle.
"""
from __future__ import annotations

import math
import struct


def bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def attend_brute(q: list[float], keys: list[list[float]], sm_scale: float, d_v: int):
    """Returns (out list[d_v], natural lse) by the textbook definition."""
    if not keys:
        return [0.0] * d_v, float("-inf")
    scores = [sm_scale * math.fsum(a * b for a, b in zip(q, k)) for k in keys]
    top = max(scores)
    weights = [math.exp(s - top) for s in scores]
    total = math.fsum(weights)
    out = [math.fsum(w * k[c] for w, k in zip(weights, keys)) / total for c in range(d_v)]
    return out, top + math.log(total)


def partial_brute(q_bits, kv_bits, block_table, seq_lens, part_id, num_parts, sm_scale,
                  d_v, page_size, base2=False, decode=None):
    """q_bits [B][1][H][dk] ints, kv_bits [pages][page_size][dk] ints."""
    decode = decode or bf16
    outs, lses = [], []
    for b, seq_len in enumerate(seq_lens):
        toks = [t for t in range(int(seq_len)) if t % num_parts == part_id]
        keys = []
        for t in toks:
            page = int(block_table[b][t // page_size])
            keys.append([decode(x) for x in kv_bits[page][t % page_size]])
        per_head_out, per_head_lse = [], []
        for h in range(len(q_bits[b][0])):
            q = [bf16(x) for x in q_bits[b][0][h]]
            o, l = attend_brute(q, keys, sm_scale, d_v)
            if base2 and l != float("-inf"):
                l = l / math.log(2.0)
            per_head_out.append(o)
            per_head_lse.append(l)
        outs.append(per_head_out)
        lses.append(per_head_lse)
    return outs, lses


def combine_brute(partials, lses, base2=False):
    """partials [P][D] floats and lses [P] for ONE output row."""
    nat = [l * math.log(2.0) if (base2 and l != float("-inf")) else l for l in lses]
    live = [(o, l) for o, l in zip(partials, nat) if l != float("-inf")]
    if not live:
        return [0.0] * len(partials[0]), float("-inf")
    top = max(l for _, l in live)
    w = [math.exp(l - top) for _, l in live]
    total = math.fsum(w)
    out = [math.fsum(wi * o[c] for wi, (o, _) in zip(w, live)) / total
           for c in range(len(partials[0]))]
    lse = top + math.log(total)
    if base2:
        lse = lse / math.log(2.0)
    return out, lse
