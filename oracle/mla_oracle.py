"""Plain fp64 CPU oracle for MLA absorbed paged decode over round-robin
decode-context-parallel (DCP) partitions, and for the LSE-weighted combine.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
baseline leg call this module; the product path never does, and this module
imports nothing from the product package.  It computes the plain definition
(two-pass max-then-sum softmax over every owned token, fp64, numpy matmul as a
library step) with no blocking, splitting or online rescaling.

Sources, by page and section:

* sglang pull 33926 (trtllm_mla decode path gains DCP):
  - "功能与动机" (motivation): token t is owned by rank t mod P, and for a
    single-token decode the rank-local slice is exactly the causally visible
    prefix, so no mask is applied.
  - code snippet ``_get_dcp_local_max_seq_len``: local length
    L // P + (r < L % P).
  - "实现拆解" (implementation) step 3: a rank that owns no tokens returns the
    neutral pair (0, -inf) (``fixup_zero_kv_rows``); the FP8 KV path exists.
  - "实现拆解" step 4: producers emit the LSE in base 2 or base e, and the
    conversion happens at the merge site.
* sglang pull 33364 ([Attention][DCP] Add symm_a2a ...), "Modifications",
  kernel 4 ``wait_lse_combine_kernel``: the LSE-weighted softmax reduction over
  all ranks' partial outputs.

Readings where the pages are silent (each also listed in the design notes):

* of the 576 query/key dims the first 512 are the latent (also the value) and
  the last 64 the rope part;
* the LSE includes ``sm_scale``: lse = log sum_j exp(sm_scale * q.k_j);
* FP8 rows dequantise as e4m3 value x per-tensor ``kv_scale`` (OCP e4m3:
  bias 7, no infinities, S.1111.111 is NaN);
* the combine of partitions that are all empty is (0, -inf), never NaN.
"""
from __future__ import annotations

import numpy as np

D_QK = 576
D_V = 512
PAGE_SIZE = 64
LOG2E = 1.4426950408889634   # log2(e)
LN2 = 0.6931471805599453     # ln(2)
LSE_NATURAL = 0
LSE_BASE2 = 1


# ------------------------------------------------------------ partition rule

def local_len(seq_len: int, num_parts: int, part_id: int) -> int:
    """Number of tokens partition ``part_id`` owns out of ``seq_len``
    (pull 33926, ``_get_dcp_local_max_seq_len``: L // P + (r < L % P),
    without the clamp to 1 that only served that kernel's scheduler)."""
    return seq_len // num_parts + (1 if part_id < seq_len % num_parts else 0)


def dcp_local_metadata(seq_lens, req_pool_indices, req_to_token, part_id: int, num_parts: int,
                       extra_tokens: int = 0, max_pages: int = 1, pad_value: int = 0,
                       page_size: int = 64):
    """A DCP rank's decode metadata (sglang pull 33926,
    ``_apply_dcp_cuda_graph_metadata``: global and rank-local lengths written
    once per step into capture-stable buffers, then the page table rebuilt
    over the rank's own slice).  Global lengths are L_b + extra_tokens (the
    draft tokens of a target-verify step); local lengths are n_r(L); the
    rank-local page table over the rank's compact pool maps local page i of
    request b to the pool page holding its local token 64 i:
    req_to_token[req_pool_indices[b], 64 i] // 64, for i < ceil(n / 64), and
    pad_value after.  A request is counted bad (and its whole table row is
    pad_value) if its global length is negative (local length 0), its pool
    index is outside req_to_token, its pages do not fit max_pages or the
    width of req_to_token; a token slot that is negative, or not the first
    slot of a pool page (a page table can only describe a pool that holds a
    request's local tokens in whole pages), gives pad_value for that page and
    also counts the request.  Returns (global, local, table, bad)."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    r2t = np.asarray(req_to_token)
    B = len(seq_lens)
    glob = (seq_lens + extra_tokens).astype(np.int32)
    loc = np.zeros(B, dtype=np.int32)
    table = np.full((B, max_pages), pad_value, dtype=np.int32)
    bad = 0
    for b in range(B):
        L = int(glob[b])
        if L < 0:
            bad += 1
            continue
        loc[b] = local_len(L, num_parts, part_id)
        req = int(req_pool_indices[b])
        npages = -(-int(loc[b]) // page_size)
        if req < 0 or req >= r2t.shape[0] or npages > max_pages or \
                (npages > 0 and (npages - 1) * page_size >= r2t.shape[1]):
            bad += 1
            continue
        neg = False
        for i in range(npages):
            slot = int(r2t[req, i * page_size])
            if slot < 0 or slot % page_size != 0:
                neg = True
            else:
                table[b, i] = slot // page_size
        bad += int(neg)
    return glob, loc, table, bad


def owned_tokens(seq_len: int, num_parts: int, part_id: int) -> np.ndarray:
    """Global 0-based token indices t < seq_len with t mod P == part_id
    (pull 33926, motivation: round-robin owner rule)."""
    return np.arange(part_id, seq_len, num_parts, dtype=np.int64)


# ------------------------------------------------------------ number formats

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly (bf16 is the top half of
    an IEEE binary32)."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):        # NaN patterns stay NaN
        return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(bits: np.ndarray) -> np.ndarray:
    """OCP FP8 e4m3 bit patterns (uint8) -> float64.

    sign = bit 7, exponent = bits 6..3 (bias 7), mantissa = bits 2..0.
    exponent 0 is subnormal: m/8 * 2^-6; otherwise (1 + m/8) * 2^(e-7).
    0x7F and 0xFF are NaN; there are no infinities.
    """
    b = np.asarray(bits).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & ((b & 0x7) == 7), np.nan, mag)
    return sign * mag


def _e4m3_finite_table():
    """The 127 non-negative finite e4m3 values, ascending, with their codes."""
    codes = np.arange(0x7F, dtype=np.uint8)          # 0x00 .. 0x7E (0x7F is NaN)
    return e4m3_to_f64(codes), codes


def f32_to_e4m3(x) -> np.ndarray:
    """fp32 values -> OCP e4m3 codes (uint8): the nearest representable value,
    ties to the even code (mantissa bit 0 clear), magnitudes beyond the
    largest finite value 448 saturate to +-448, the sign is kept (so -0 and
    negative values that round to zero give 0x80).  NaN inputs are not
    defined here.  Exact: every fp32 input, e4m3 value and midpoint is exact
    in fp64 (the write path of sglang pull 33926, implementation step 3:
    the FP8 cache stores the quantised latent with one per-tensor scale)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    vals, codes = _e4m3_finite_table()
    a = np.abs(x)
    hi = np.searchsorted(vals, a, side="left")       # first value >= a
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo = a - vals[lo]
    dhi = vals[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((codes[hi] & 1) == 0))
    c = np.where(a >= vals[-1], codes[-1], np.where(pick_hi, codes[hi], codes[lo]))
    c = np.where(vals[hi] == a, codes[hi], c)
    return (c | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def kv_append(kv_bits: np.ndarray, block_table: np.ndarray, positions: np.ndarray,
              new_bits: np.ndarray, part_id: int, num_parts: int, kv_dtype: str = "bf16",
              kv_scale: float = 1.0, page_size: int = PAGE_SIZE):
    """Writes each request's new latent row (bf16 bits [576]) into the paged
    cache at global token positions[b] (the request's length before the
    append), if positions[b] >= 0 and partition ``part_id`` owns that token
    (positions[b] mod P == part_id: under DCP each rank writes only its own
    tokens, sglang pull 33926, implementation step 4).  An e4m3 cache stores
    f32_to_e4m3(fp32(x) / fp32(kv_scale)), the division in fp32 like the
    kernel's.  A row whose page entry lies outside the table or the pool is
    skipped and counted.  Returns (new cache, number of skipped rows); the
    input cache is not modified."""
    out = np.array(kv_bits, copy=True)
    bt = np.asarray(block_table)
    num_pages, max_pages = out.shape[0], bt.shape[1]
    bad = 0
    for b in range(len(positions)):
        t = int(positions[b])
        if t < 0 or t % num_parts != part_id:
            continue
        lp = t // page_size
        if lp >= max_pages:
            bad += 1
            continue
        pg = int(bt[b, lp])
        if pg < 0 or pg >= num_pages:
            bad += 1
            continue
        row = np.asarray(new_bits[b], dtype=np.uint16)
        if kv_dtype == "bf16":
            out[pg, t % page_size] = row
        else:
            x = (row.astype(np.uint32) << 16).view(np.float32)
            out[pg, t % page_size] = f32_to_e4m3(x / np.float32(kv_scale))
    return out, bad


# ------------------------------------------------------------ paged gather

def gather_rows(kv_bits: np.ndarray, block_table_row: np.ndarray, tokens: np.ndarray,
                page_size: int) -> np.ndarray:
    """Raw cache rows of global tokens ``tokens``:
    kv_pages[block_table[t // page_size], t % page_size, :]."""
    pages = np.asarray(block_table_row)[tokens // page_size].astype(np.int64)
    return kv_bits[pages, tokens % page_size]


def dequant_rows(raw: np.ndarray, kv_dtype: str, kv_scale: float) -> np.ndarray:
    if kv_dtype == "bf16":
        return bf16_to_f64(raw)
    if kv_dtype == "e4m3":
        return e4m3_to_f64(raw) * float(kv_scale)
    raise ValueError(kv_dtype)


# ------------------------------------------------------------ attention

def attend(q: np.ndarray, k: np.ndarray, sm_scale: float, d_v: int = D_V):
    """Softmax attention of H query rows over n cached rows, fp64.

    q: [H, 576], k: [n, 576]; the value of row j is k[j, :512] (``d_v``
    leading dims; reduced dims are used only by the tests).
    Returns (out [H, 512], lse [H]) with the natural-log LSE of the scaled
    scores; n == 0 gives the neutral pair (0, -inf) (pull 33926, step 3).
    """
    heads = q.shape[0]
    if k.shape[0] == 0:
        return np.zeros((heads, d_v)), np.full(heads, -np.inf)
    v = k[:, :d_v]
    s = sm_scale * (q @ k.T)                      # [H, n]
    mu = s.max(axis=1, keepdims=True)
    w = np.exp(s - mu)
    z = w.sum(axis=1, keepdims=True)
    out = (w @ v) / z
    lse = mu[:, 0] + np.log(z[:, 0])
    return out, lse


def lse_to_base(lse_natural: np.ndarray, lse_base: int) -> np.ndarray:
    """Express a natural-log LSE in the requested base (pull 33926, step 4);
    -inf stays -inf."""
    if lse_base == LSE_NATURAL:
        return lse_natural
    if lse_base == LSE_BASE2:
        return lse_natural * LOG2E
    raise ValueError(lse_base)


def lse_to_natural(lse: np.ndarray, lse_base: int) -> np.ndarray:
    if lse_base == LSE_NATURAL:
        return np.asarray(lse, dtype=np.float64)
    if lse_base == LSE_BASE2:
        return np.asarray(lse, dtype=np.float64) * LN2
    raise ValueError(lse_base)


def decode_partial(q_bits: np.ndarray, kv_bits: np.ndarray, block_table: np.ndarray,
                   seq_lens, part_id: int, num_parts: int, sm_scale: float,
                   lse_base: int = LSE_NATURAL, kv_dtype: str = "bf16",
                   kv_scale: float = 1.0, page_size: int = 64, requests=None,
                   d_v: int = D_V):
    """Partition ``part_id`` of ``num_parts``: attention of every request's
    query over the global tokens it owns.

    q_bits: uint16 [B, 1, H, 576] (bf16); kv_bits: uint16 [pages, 64, 576]
    (bf16) or uint8 (e4m3); block_table: int [B, max_pages]; seq_lens: global
    lengths.  ``requests`` restricts the work to a subset of batch rows.
    Returns out [B', H, 512] and lse [B', H] (requested base), fp64.
    """
    if np.asarray(q_bits).shape[1] != 1:
        raise ValueError("single-token decode only (q_len == 1)")
    rows = range(len(seq_lens)) if requests is None else list(requests)
    outs, lses = [], []
    for b in rows:
        toks = owned_tokens(int(seq_lens[b]), num_parts, part_id)
        k = dequant_rows(gather_rows(kv_bits, block_table[b], toks, page_size),
                         kv_dtype, kv_scale)
        q = bf16_to_f64(q_bits[b, 0])
        o, l = attend(q, k, sm_scale, d_v)
        outs.append(o)
        lses.append(lse_to_base(l, lse_base))
    return np.stack(outs), np.stack(lses)


def decode_partial_causal(q_bits: np.ndarray, kv_bits: np.ndarray, block_table: np.ndarray,
                          seq_lens, part_id: int, num_parts: int, sm_scale: float,
                          lse_base: int = LSE_NATURAL, kv_dtype: str = "bf16",
                          kv_scale: float = 1.0, page_size: int = 64, requests=None,
                          d_v: int = D_V):
    """Several query tokens per request (q_len = T: multi-token prediction /
    target verify).  The cache already holds the T new tokens (the KV length
    of a target-verify step is the prefix plus the draft tokens, sglang pull
    33926's metadata code), so query token i of request b is global token
    L_b - T + i and attends causally: to the tokens the partition owns among
    t < L_b - T + i + 1.  A query token with none gets (0, -inf).

    q_bits: uint16 [B, T, H, 576].  Returns out [B', T, H, 512] and lse
    [B', T, H] (requested base), fp64.
    """
    q_bits = np.asarray(q_bits)
    T = q_bits.shape[1]
    rows = range(len(seq_lens)) if requests is None else list(requests)
    outs, lses = [], []
    for b in rows:
        ob, lb = [], []
        for i in range(T):
            vis = max(0, int(seq_lens[b]) - T + i + 1)
            toks = owned_tokens(vis, num_parts, part_id)
            k = dequant_rows(gather_rows(kv_bits, block_table[b], toks, page_size),
                             kv_dtype, kv_scale)
            o, l = attend(bf16_to_f64(q_bits[b, i]), k, sm_scale, d_v)
            ob.append(o)
            lb.append(lse_to_base(l, lse_base))
        outs.append(np.stack(ob))
        lses.append(np.stack(lb))
    return np.stack(outs), np.stack(lses)


def decode_full(q_bits, kv_bits, block_table, seq_lens, sm_scale, lse_base=LSE_NATURAL,
                **kw):
    """The unpartitioned result: every token < L attended (P = 1)."""
    return decode_partial(q_bits, kv_bits, block_table, seq_lens, 0, 1, sm_scale,
                          lse_base, **kw)


# ------------------------------------------------------------ LSE combine

def lse_combine(partials: np.ndarray, lses: np.ndarray, lse_base: int = LSE_NATURAL):
    """LSE-weighted merge of P partial results (pull 33364, Modifications,
    kernel 4), with the base converted at the merge site (pull 33926, step 4).

    partials: fp64 [P, ..., D]; lses: [P, ...] in base ``lse_base``.
    For each output row: M = max_p lse_p, w_p = exp(lse_p - M),
    out = sum_p w_p o_p / sum_p w_p, lse = M + log sum_p w_p.
    Rows whose partitions are all (0, -inf) give (0, -inf).
    """
    lam = lse_to_natural(lses, lse_base)
    big = lam.max(axis=0)
    finite = np.isfinite(big)
    safe = np.where(finite, big, 0.0)
    w = np.where(np.isfinite(lam), np.exp(lam - safe[None]), 0.0)
    z = w.sum(axis=0)
    num = (w[..., None] * partials).sum(axis=0)
    out = np.where(finite[..., None], num / np.where(finite, z, 1.0)[..., None], 0.0)
    lse = np.where(finite, safe + np.log(np.where(finite, z, 1.0)), -np.inf)
    return out, lse_to_base(lse, lse_base)
