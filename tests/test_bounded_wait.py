"""Failure detection without a GPU fault: the kernels' bounded waits, run on
barriers that nothing completes, give up, report MLA_ERR_TIMEOUT through the
workspace, and leave the context usable."""
import time

import pytest
import torch

import mla_paged_decode_gb300 as mla
import workloads
from gpu_helpers import run_partial

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_decode_gb300 import build
    build.build()
    mla.load_library()


def test_a_wait_that_nothing_completes_gives_up_and_reports():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    timeout_ns = 20_000_000  # 20 ms
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    mla.selftest_bounded_wait(ws, timeout_ns)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    word = int(ws[:4].view(torch.int32).item())
    assert word & 4, hex(word)                       # the timeout bit
    assert word & (1 << 8) and word & (1 << 9), hex(word)  # both warps left their waits
    # warp 0 waited out its limit; warp 1 (limit 200 ms) left on the abort flag
    assert 0.015 < elapsed < 0.15, elapsed
    with pytest.raises(mla.MlaError) as e:
        mla.check_workspace(ws)                      # MLA_ERR_TIMEOUT; the word is then cleared
    assert e.value.status == -10
    assert int(ws[:4].view(torch.int32).item()) == 0


def test_the_context_stays_usable_after_a_timeout():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    mla.selftest_bounded_wait(ws, 1_000_000)
    torch.cuda.synchronize()
    case = workloads.make_decode_case("after_timeout", 16, [300, 65], seed=3, device="cuda")
    out, lse = run_partial(case, 0, 0)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
