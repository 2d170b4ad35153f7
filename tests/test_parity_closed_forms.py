"""GPU results on inputs whose attention has a closed form.

Each case fixes the answer by the mathematics alone (no oracle involved):
- a zero query gives every owned token the weight 1, so the output is the
  plain mean of the owned value rows and the LSE is exactly ln n_r, the
  count the owner rule gives (sglang pull 33926, "Decode layout": token t
  of a request lives on partition t mod P);
- a query that is zero on the latent dims, against keys that share their
  rope dims, gives one common score s, so the output is again the mean and
  the LSE is s + ln n_r (the latent-first, rope-last reading of the
  576-dim key);
- a request of one token returns that token's value row bit for bit and
  its own score as the LSE;
- value rows that are all the same vector c return c, whatever the scores.

The LSE bound of the zero-query case, 1e-5, is tight enough that a token
dropped or counted twice (ln(n +- 1) - ln n >= 1 / (n + 1)) fails it for
every length used here.
"""
import math

import numpy as np
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


def owned_tokens(L: int, P: int, r: int) -> list[int]:
    return list(range(r, L, P))


def owned_rows(case, b: int, r: int) -> torch.Tensor:
    """fp64 [n, 576]: the cached rows of request b's tokens owned by partition r."""
    t = torch.tensor(owned_tokens(int(case.seq_lens[b]), case.num_parts, r), dtype=torch.long)
    if t.numel() == 0:
        return torch.zeros(0, 576, dtype=torch.float64)
    pages = case.block_table[b].cpu().long()[t // 64]
    rows = case.kv_pages[pages.to(case.kv_pages.device), (t % 64).to(case.kv_pages.device)].cpu()
    if case.kv_dtype == "e4m3":
        return rows.view(torch.float8_e4m3fn).to(torch.float64) * case.kv_scale
    return rows.to(torch.float64)


def _natural(lse: torch.Tensor) -> np.ndarray:
    return lse.detach().float().cpu().numpy().astype(np.float64)


def _check_uniform(case, ws, score_of_request, lse_tol):
    """Every owned token has the same score: out = mean of the value rows,
    lse = score + ln n_r; a partition with no token returns (0, -inf)."""
    for r in range(case.num_parts):
        out, lse = run_partial(case, r, 0, workspace=ws)
        o = out.float().cpu().numpy().astype(np.float64)
        l = _natural(lse)
        for b in range(case.batch):
            rows = owned_rows(case, b, r)
            n = rows.shape[0]
            if n == 0:
                assert np.all(o[b] == 0.0) and np.all(np.isneginf(l[b])), f"part {r} req {b}"
                continue
            mean = rows[:, :512].mean(0).numpy()
            err = np.abs(o[b, 0] - mean[None, :]).max()
            assert err <= 1e-2 + 2 ** -8 * np.abs(mean).max(), f"part {r} req {b}: out err {err:.3e}"
            want = score_of_request(b) + math.log(n)
            lerr = np.abs(l[b, 0] - want).max()
            assert lerr <= lse_tol, f"part {r} req {b} n {n}: lse err {lerr:.3e}"


UNIFORM_CASES = [
    (16, [1, 63, 64, 65, 1000], 1, "bf16"),
    (64, [4097, 130, 7], 3, "bf16"),
    (16, [700, 65, 1300, 2], 8, "bf16"),
    (64, [1000, 333], 2, "e4m3"),
    (32, [2049, 5], 6, "e4m3"),
]


@pytest.mark.parametrize("heads,lens,num_parts,kv_dtype", UNIFORM_CASES)
def test_zero_query_gives_the_mean_and_ln_n(heads, lens, num_parts, kv_dtype):
    case = workloads.make_decode_case("q0", heads, lens, seed=51, device="cuda",
                                      kv_dtype=kv_dtype, num_parts=num_parts, tail_poison=True)
    case.q.zero_()
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table, case.kv_scale)
    _check_uniform(case, ws, lambda b: 0.0, 1e-5)
    assert mla.check_workspace(ws) == 0


@pytest.mark.parametrize("heads,lens,num_parts,kv_dtype", UNIFORM_CASES)
def test_scores_from_the_rope_dims_alone(heads, lens, num_parts, kv_dtype):
    case = workloads.make_decode_case("rope", heads, lens, seed=52, device="cuda",
                                      kv_dtype=kv_dtype, num_parts=num_parts)
    case.q[..., :512] = 0
    case.kv_pages[:, :, 512:] = case.kv_pages[0, 0, 512:].clone()  # one rope vector everywhere
    rope = owned_rows(case, 0, 0)[0, 512:] if int(case.seq_lens[0]) else None
    q = case.q.cpu().to(torch.float64)

    def score(b):  # the same for every head only if q's rope part is; take head 0 and check all
        s = case.sm_scale * (q[b, 0, :, 512:] @ rope)
        return s.numpy()

    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table, case.kv_scale)
    _check_uniform(case, ws, score, 2e-4)


def test_one_token_returns_its_row():
    case = workloads.make_decode_case("one", 64, [1, 1, 1, 1], seed=53, device="cuda")
    out, lse = run_partial(case, 0, 0)
    q = case.q.cpu().to(torch.float64)
    for b in range(case.batch):
        row = case.kv_pages[int(case.block_table[b, 0])][0]
        assert torch.equal(out[b, 0].view(torch.int16), row[:512].expand(64, 512).view(torch.int16))
        s = case.sm_scale * (q[b, 0] @ row.cpu().to(torch.float64))
        assert np.abs(_natural(lse[b, 0]) - s.numpy()).max() <= 1e-3


@pytest.mark.parametrize("num_parts,kv_dtype", [(1, "bf16"), (3, "bf16"), (8, "bf16"), (1, "e4m3")])
def test_equal_value_rows_return_that_row(num_parts, kv_dtype):
    case = workloads.make_decode_case("vconst", 64, [5000, 77, 1025], seed=54, device="cuda",
                                      kv_dtype=kv_dtype, num_parts=num_parts)
    case.kv_pages[:, :, :512] = case.kv_pages[0, 0, :512].clone()
    c = owned_rows(case, 0, 0)[0, :512].numpy()
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table, case.kv_scale)
    for r in range(num_parts):
        out, _ = run_partial(case, r, 0, workspace=ws)
        o = out.float().cpu().numpy().astype(np.float64)
        err = np.abs(o[:, 0] - c[None, None, :]).max()
        assert err <= 2 ** -8 * np.abs(c).max(), f"part {r}: err {err:.3e}"


def test_zero_query_through_the_all_partition_call():
    """The same closed form for mla_decode_dcp's merged output over all P
    partitions: the mean over every token, lse = ln L."""
    lens = [4097, 1, 3, 700]
    case = workloads.make_decode_case("q0dcp", 16, lens, seed=55, device="cuda", num_parts=8)
    case.q.zero_()
    out, out_lse, _, _ = mla.decode_dcp(case.q, case.kv_pages, case.block_table, case.seq_lens, 8,
                                        case.sm_scale, 0,
                                        out_lse=torch.empty(len(lens), 1, 16, dtype=torch.float32,
                                                            device="cuda"))
    o = out.float().cpu().numpy().astype(np.float64)
    one = workloads.DecodeCase(case.name, case.q, case.kv_pages, case.block_table, case.seq_lens,
                               case.kv_dtype, case.kv_scale, case.sm_scale, 1)
    for b, L in enumerate(lens):
        mean = owned_rows(one, b, 0)[:, :512].mean(0).numpy()
        assert np.abs(o[b, 0] - mean[None, :]).max() <= 1e-2
        assert np.abs(_natural(out_lse[b, 0]) - math.log(L)).max() <= 1e-5
