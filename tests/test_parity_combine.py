"""GPU parity of mla_lse_combine against the fp64 oracle on the standalone
combine workload: P = 8 partials, T in {1, 8, 16, 32, 64, 128}, H = 16,
D = 512, lse ~ N(5, 3), one partition per token set to (0, -inf), LSE given
in natural log, converted to base 2, and raw values read as base 2."""
import math

import numpy as np
import pytest
import torch

import mla_paged_decode_gb300 as mla
import oracle
import workloads
from casebits import bits
from gpu_helpers import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_decode_gb300 import build
    build.build()
    mla.load_library()


def _run(partials, lses, base):
    P, T, H, D = partials.shape
    out = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    out_lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    mla.lse_combine(partials, lses, P, out, lse_base=base, out_lse=out_lse)
    return out, out_lse


@pytest.mark.parametrize("tokens", [1, 8, 16, 32, 64, 128])
def test_combine_matches_oracle(tokens):
    c = workloads.combine_case(tokens, device="cuda", seed=tokens)
    parts64 = oracle.bf16_to_f64(bits(c.partials))
    lam = c.lses.cpu().numpy().astype(np.float64)
    # (i) natural-log LSE
    out, ol = _run(c.partials, c.lses, 0)
    ro, rl = oracle.lse_combine(parts64, lam, 0)
    assert_out_close(out, ro, what=f"T={tokens} natural")
    assert_lse_close(ol, rl, 0, what=f"T={tokens} natural")
    # (ii) the same LSE expressed in base 2 must give the same merge
    lam2 = (c.lses * math.log2(math.e)).contiguous()
    out2, ol2 = _run(c.partials, lam2, 1)
    ro2, rl2 = oracle.lse_combine(parts64, lam2.cpu().numpy().astype(np.float64), 1)
    assert_out_close(out2, ro2, what=f"T={tokens} base2 converted")
    assert_lse_close(ol2, rl2, 1, what=f"T={tokens} base2 converted")
    assert_out_close(out2, ro, what=f"T={tokens} base2 vs natural")
    # (iii) the raw values read as base-2 LSEs
    out3, ol3 = _run(c.partials, c.lses, 1)
    ro3, rl3 = oracle.lse_combine(parts64, lam, 1)
    assert_out_close(out3, ro3, what=f"T={tokens} raw base2")
    assert_lse_close(ol3, rl3, 1, what=f"T={tokens} raw base2")


def test_all_empty_rows_are_neutral_and_p1_is_identity():
    c = workloads.combine_case(4, device="cuda", seed=3)
    c.partials[:, 2] = 0
    c.lses[:, 2] = float("-inf")
    out, ol = _run(c.partials, c.lses, 0)
    assert torch.all(out[2].view(torch.int16) == 0) and torch.isneginf(ol[2]).all()
    assert torch.isfinite(out.float()).all()
    one = workloads.combine_case(5, num_parts=1, device="cuda", seed=4, empty_per_token=0)
    out1, ol1 = _run(one.partials, one.lses, 1)
    assert torch.equal(out1.view(torch.int16), one.partials[0].view(torch.int16))
    assert torch.equal(ol1, one.lses[0])


def test_combine_large_head_dim_and_many_parts():
    c = workloads.combine_case(3, num_parts=37, heads=5, dim=1024, device="cuda", seed=9,
                               empty_per_token=3)
    out, ol = _run(c.partials, c.lses, 0)
    ro, rl = oracle.lse_combine(oracle.bf16_to_f64(bits(c.partials)),
                                c.lses.cpu().numpy().astype(np.float64), 0)
    assert_out_close(out, ro)
    assert_lse_close(ol, rl, 0)
