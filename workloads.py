"""Seeded synthetic inputs for MLA absorbed paged decode and the LSE combine.

This module is the only code shared by the fp64 oracle side and the CUDA side:
it draws the random tensors (query, paged latent KV pool, block tables, sequence
lengths, combine partials) and holds none of the attention arithmetic.  The FP8
cache is produced the way a KV-append step would produce it (per-tensor scale
= amax / 448, round-to-nearest via torch's float8_e4m3fn cast); reading it back
is each side's own business.

Workloads (shapes of the decode-context-parallel pages' setting; no dataset is
involved and no trained weights exist here, all values are N(0, 1)):

* ``config_small``     B=1,  H=16,  L=300, pool of 5 pages, P=2 (then combine)
* ``config_long32k``   B=64, H=64,  L ~ U{4096..32768}, pool 40k pages, P=1
* ``config_dcp8``      B=64, H=16,  60 x 131072 + {1,3,5,7}, P=8 (then combine)
* ``config_fp8``       B=128, H=128, e4m3 KV, L ~ lognormal(median 8192, sigma 1)
                       clipped to [1024, 65536], P=1
* ``combine_case``     P=8 partials, T tokens, H=16, D=512, lse ~ N(5, 3),
                       one partition per token set to (0, -inf)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAGE_SIZE = 64
D_QK = 576          # 512 latent + 64 rope
D_V = 512           # latent part of each cached row
SM_SCALE_192 = 1.0 / math.sqrt(192.0)

# one sub-stream per tensor so that changing one shape never reshuffles another
_SUB = {"q": 1, "kv": 2, "lens": 3, "perm": 4, "part": 5, "lse": 6, "empty": 7}


def _gen(seed: int, what: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1009 + _SUB[what])
    return g


@dataclass
class DecodeCase:
    """One decode batch: a global paged cache and the global sequence lengths."""
    name: str
    q: torch.Tensor            # bf16 [B, 1, H, 576]
    kv_pages: torch.Tensor     # bf16 [num_pages, 64, 576], or uint8 e4m3 bits
    block_table: torch.Tensor  # int32 [B, max_pages]; logical page -> physical page
    seq_lens: torch.Tensor     # int32 [B], global lengths
    kv_dtype: str              # "bf16" or "e4m3"
    kv_scale: float            # per-tensor dequant scale (1.0 for bf16)
    sm_scale: float
    num_parts: int
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def heads(self) -> int:
        return self.q.shape[2]

    @property
    def num_pages(self) -> int:
        return self.kv_pages.shape[0]


def pages_for(seq_len: int) -> int:
    return (seq_len + PAGE_SIZE - 1) // PAGE_SIZE


def uniform_lens(batch: int, lo: int, hi: int, seed: int) -> list[int]:
    g = _gen(seed, "lens", "cpu")
    return torch.randint(lo, hi + 1, (batch,), generator=g).tolist()


def lognormal_lens(batch: int, median: float, sigma: float, lo: int, hi: int,
                   seed: int) -> list[int]:
    g = _gen(seed, "lens", "cpu")
    z = torch.randn(batch, generator=g, dtype=torch.float64)
    lens = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
    return [int(x) for x in lens.tolist()]


def _randn_bf16(shape, gen, device, chunk_rows: int = 4096) -> torch.Tensor:
    """N(0,1) rounded to bf16, drawn in slabs along dim 0 to bound temporaries."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        out[s:e] = torch.randn((e - s,) + tuple(shape[1:]), generator=gen,
                               device=device).to(torch.bfloat16)
    return out


def _randn_e4m3(shape, gen, device, chunk_rows: int = 4096):
    """N(0,1) quantised to e4m3 with one per-tensor scale (amax / 448)."""
    x = torch.empty(shape, dtype=torch.float32, device=device)
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        x[s:e] = torch.randn((e - s,) + tuple(shape[1:]), generator=gen, device=device)
    amax = float(x.abs().max().item())
    scale = amax / 448.0
    bits = torch.empty(shape, dtype=torch.uint8, device=device)
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        bits[s:e] = (x[s:e] / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    del x
    return bits, scale


def make_decode_case(name: str, heads: int, seq_lens: list[int], *,
                     pool_pages: int | None = None, kv_dtype: str = "bf16",
                     num_parts: int = 1, sm_scale: float = SM_SCALE_192,
                     seed: int = 0, device="cpu", tail_poison: bool = False,
                     pad_value: int = 0, q_len: int = 1) -> DecodeCase:
    """Build a paged decode batch.

    Each request's ceil(L/64) pages are drawn without replacement from a
    shuffled pool, so the block table is a random permutation of physical
    pages.  ``tail_poison`` fills the unused rows of every request's last page
    (and every page no request owns) with NaN bit patterns: a correct kernel
    never lets them reach its output.  Block-table entries past a request's
    last page hold ``pad_value``.  ``q_len`` query tokens per request (the
    last q_len tokens of each length) give q [B, q_len, H, 576].
    """
    batch = len(seq_lens)
    need = [pages_for(L) for L in seq_lens]
    total = sum(need)
    num_pages = max(total, pool_pages or 0, 1)
    perm = torch.randperm(num_pages, generator=_gen(seed, "perm", "cpu"))
    width = max(1, max(need) if need else 1)
    bt = torch.full((batch, width), pad_value, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n

    q = _randn_bf16((batch, q_len, heads, D_QK), _gen(seed, "q", device), device)
    if kv_dtype == "bf16":
        kv = _randn_bf16((num_pages, PAGE_SIZE, D_QK), _gen(seed, "kv", device), device)
        kv_scale = 1.0
    elif kv_dtype == "e4m3":
        kv, kv_scale = _randn_e4m3((num_pages, PAGE_SIZE, D_QK), _gen(seed, "kv", device),
                                   device)
    else:
        raise ValueError(kv_dtype)

    if tail_poison:
        nan_bits = 0x7FC0 if kv_dtype == "bf16" else 0x7F
        view = kv.view(torch.int16) if kv_dtype == "bf16" else kv
        used = torch.zeros(num_pages, dtype=torch.bool)
        for b, L in enumerate(seq_lens):
            n = need[b]
            if n:
                used[bt[b, :n].long()] = True
                rem = L - (n - 1) * PAGE_SIZE
                if rem < PAGE_SIZE:
                    view[int(bt[b, n - 1]), rem:] = nan_bits
        unused = (~used).nonzero().flatten()
        if unused.numel():
            view[unused.to(view.device)] = nan_bits

    return DecodeCase(name=name, q=q, kv_pages=kv, block_table=bt.to(device),
                      seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
                      kv_dtype=kv_dtype, kv_scale=kv_scale, sm_scale=sm_scale,
                      num_parts=num_parts, meta={"seed": seed})


# ---------------------------------------------------------------- named workloads

def config_small(device="cpu", seed: int = 0, **kw) -> DecodeCase:
    """B=1, H=16, L=300 (5 pages, the last holds 44 rows), P=2."""
    return make_decode_case("small_b1_h16_l300_p2", 16, [300], pool_pages=5,
                            num_parts=2, seed=seed, device=device, **kw)


def config_long32k(device="cpu", seed: int = 0, batch: int = 64, pool_pages: int = 40000,
                   **kw) -> DecodeCase:
    """B=64, H=64, L ~ U{4096..32768}, 40k-page pool, P=1."""
    lens = uniform_lens(batch, 4096, 32768, seed)
    return make_decode_case("long32k_b64_h64_bf16", 64, lens, pool_pages=pool_pages,
                            num_parts=1, seed=seed, device=device, **kw)


def config_dcp8(device="cpu", seed: int = 0, long_len: int = 131072,
                n_long: int = 60, **kw) -> DecodeCase:
    """B=64, H=16, 60 requests at 131072 plus L in {1,3,5,7}, P=8."""
    lens = [long_len] * n_long + [1, 3, 5, 7]
    return make_decode_case("dcp8_b64_h16_131k", 16, lens, num_parts=8, seed=seed,
                            device=device, **kw)


def config_fp8(device="cpu", seed: int = 0, batch: int = 128, **kw) -> DecodeCase:
    """B=128, H=128, e4m3 KV with a per-tensor scale, lognormal lengths, P=1."""
    lens = lognormal_lens(batch, 8192.0, 1.0, 1024, 65536, seed)
    return make_decode_case("fp8_b128_h128_lognormal", 128, lens, kv_dtype="e4m3",
                            num_parts=1, seed=seed, device=device, **kw)


@dataclass
class CombineCase:
    partials: torch.Tensor   # bf16 [P, T, H, D]
    lses: torch.Tensor       # fp32 [P, T, H]
    empty_part: torch.Tensor  # int64 [T]: the partition set to (0, -inf) per token


def combine_case(tokens: int, num_parts: int = 8, heads: int = 16, dim: int = D_V,
                 seed: int = 0, device="cpu", lse_mean: float = 5.0,
                 lse_std: float = 3.0, empty_per_token: int = 1) -> CombineCase:
    """Partials ~ N(0,1) bf16, lse ~ N(5, 3) fp32; per token, ``empty_per_token``
    partitions (chosen at random) hold the neutral pair (0, -inf)."""
    partials = _randn_bf16((num_parts, tokens, heads, dim), _gen(seed, "part", device),
                           device)
    lses = (torch.randn((num_parts, tokens, heads), generator=_gen(seed, "lse", "cpu"),
                        dtype=torch.float32) * lse_std + lse_mean).to(device)
    ge = _gen(seed, "empty", "cpu")
    empty = torch.zeros(tokens, dtype=torch.int64)
    for t in range(tokens):
        chosen = torch.randperm(num_parts, generator=ge)[:empty_per_token]
        empty[t] = chosen[0] if empty_per_token else -1
        for p in chosen.tolist():
            partials[p, t] = 0
            lses[p, t] = float("-inf")
    return CombineCase(partials=partials, lses=lses, empty_part=empty)
