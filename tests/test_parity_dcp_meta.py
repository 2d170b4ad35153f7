"""GPU parity of mla_dcp_local_metadata (a DCP rank's lengths and page table,
built on the device) and of decoding a rank's compact pool with it: the
metadata bit for bit against the oracle, the rank's decode bit for bit
against the partition of the global cache, and both captured in a CUDA graph
that keeps working as the lengths change between replays."""
import numpy as np
import pytest
import torch

import mla_paged_decode_gb300 as mla
import oracle
import workloads
from casebits import bits, case_bits
from dcp_local import compact_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_decode_gb300 import build
    build.build()
    mla.load_library()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("num_parts,extra", [(1, 0), (2, 0), (3, 2), (8, 0), (8, 5)])
def test_metadata_matches_the_oracle(num_parts, extra):
    rng = np.random.default_rng(num_parts + extra)
    B, width, slots = 37, 4096, 50
    lens = rng.integers(0, 3000, size=B).astype(np.int32)
    lens[:4] = [0, 1, num_parts - 1, 64 * num_parts]
    idx = rng.integers(0, slots - 1, size=B).astype(np.int32)
    # a pool in whole pages: slot = 64 * (a random page) + the token's row
    pages = rng.integers(0, 1 << 14, size=(slots, width // 64)).astype(np.int32)
    r2t = (64 * np.repeat(pages, 64, axis=1) + np.tile(np.arange(64, dtype=np.int32), width // 64))
    r2t = np.ascontiguousarray(r2t.astype(np.int32))
    lens[5], idx[6], r2t[idx[7], 0] = -3, slots + 2, -1       # the bad cases
    lens[8], idx[8] = 300 * num_parts, slots - 1              # and a slot inside a page
    r2t[slots - 1, 128] += 5
    for r in range(num_parts):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        g, loc, tab = mla.dcp_local_metadata(_dev(lens), _dev(idx), _dev(r2t), r, num_parts,
                                             max_pages=40, extra_tokens=extra, pad_value=-1,
                                             error_word=err)
        og, ol, ot, bad = oracle.dcp_local_metadata(lens, idx, r2t, r, num_parts, extra, 40, -1)
        np.testing.assert_array_equal(g.cpu().numpy(), og)
        np.testing.assert_array_equal(loc.cpu().numpy(), ol)
        np.testing.assert_array_equal(tab.cpu().numpy(), ot)
        assert (int(err.item()) != 0) == (bad > 0)


def test_metadata_flags_a_slot_inside_a_page():
    # two requests of 200 tokens (4 local pages each) over a pool in whole
    # pages; then the same with one fault only: request 1's second local page
    # starting one slot into a page
    aligned = np.ascontiguousarray((np.arange(2 * 256, dtype=np.int32) + 64 * 7).reshape(2, 256))
    faulted = aligned.copy()
    faulted[1, 64] += 1
    lens, idx = np.array([200, 200], np.int32), np.array([0, 1], np.int32)
    for r2t, fault in ((aligned, False), (faulted, True)):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        _, _, tab = mla.dcp_local_metadata(_dev(lens), _dev(idx), _dev(r2t), 0, 1, max_pages=4,
                                           pad_value=-1, error_word=err)
        _, _, ot, bad = oracle.dcp_local_metadata(lens, idx, r2t, 0, 1, 0, 4, -1)
        np.testing.assert_array_equal(tab.cpu().numpy(), ot)
        assert bad == int(fault) and (int(err.item()) != 0) == fault
        assert (ot[1, 1] == -1) == fault and list(ot[0]) == [7, 8, 9, 10]


@pytest.mark.parametrize("kv_dtype,heads,num_parts", [("bf16", 16, 8), ("bf16", 64, 2),
                                                       ("bf16", 128, 4), ("e4m3", 16, 4),
                                                       ("e4m3", 64, 2), ("e4m3", 128, 8)])
def test_rank_decode_equals_the_global_partition_bit_for_bit(kv_dtype, heads, num_parts):
    lens = [1, 7, 64 * num_parts, 3000, 129, 0, 20000]
    case = workloads.make_decode_case("rank", heads, lens, seed=heads, device="cuda",
                                      kv_dtype=kv_dtype, num_parts=num_parts)
    q, kv, bt, sl = case_bits(case)
    rng = np.random.default_rng(3)
    for r in range(num_parts):
        pool, r2t, _, _ = compact_pool(kv, bt, sl, r, num_parts, rng)
        pool_t = _dev(pool).view(torch.bfloat16 if kv_dtype == "bf16" else torch.uint8)
        _, loc, tab = mla.dcp_local_metadata(case.seq_lens, _dev(np.arange(len(lens), dtype=np.int32)),
                                             _dev(r2t), r, num_parts, max_pages=bt.shape[1])
        out_l = torch.empty(len(lens), 1, heads, 512, dtype=torch.bfloat16, device="cuda")
        lse_l = torch.empty(len(lens), 1, heads, dtype=torch.float32, device="cuda")
        mla.decode_partial(case.q, pool_t, tab, loc, 0, 1, case.sm_scale, 1, out_l, lse_l,
                           kv_scale=case.kv_scale)
        out_g = torch.empty_like(out_l)
        lse_g = torch.empty_like(lse_l)
        mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, r, num_parts,
                           case.sm_scale, 1, out_g, lse_g, kv_scale=case.kv_scale)
        assert torch.equal(out_l.view(torch.int16), out_g.view(torch.int16)), f"partition {r}"
        assert torch.equal(lse_l, lse_g), f"partition {r}"


def test_metadata_and_rank_decode_replay_in_a_cuda_graph():
    P, r, heads = 4, 1, 16
    lens = [900, 64, 3, 5000]
    case = workloads.make_decode_case("graph_rank", heads, [L + 300 for L in lens], seed=9,
                                      device="cuda", num_parts=P)
    q, kv, bt, sl_full = case_bits(case)
    pool, r2t, _, _ = compact_pool(kv, bt, sl_full, r, P, np.random.default_rng(4))
    pool_t, r2t_t = _dev(pool).view(torch.bfloat16), _dev(r2t)
    idx = _dev(np.arange(4, dtype=np.int32))
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")   # the step's lengths, updated in place
    g = torch.empty(4, dtype=torch.int32, device="cuda")
    loc = torch.empty_like(g)
    tab = torch.empty(4, bt.shape[1], dtype=torch.int32, device="cuda")
    out = torch.empty(4, 1, heads, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(4, 1, heads, dtype=torch.float32, device="cuda")
    ws = mla.make_workspace(case.q, pool_t, tab)
    s = torch.cuda.Stream()

    def step(stream):
        mla.dcp_local_metadata(seq, idx, r2t_t, r, P, max_pages=bt.shape[1], global_lens=g,
                               local_lens=loc, block_table=tab, stream=stream)
        mla.decode_partial(case.q, pool_t, tab, loc, 0, 1, case.sm_scale, 0, out, lse,
                           workspace=ws, stream=stream)

    with torch.cuda.stream(s):
        step(s)                      # first call outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step(s)
    for extra in (0, 17, 250):
        seq.copy_(torch.tensor(lens, dtype=torch.int32) + extra)
        graph.replay()
        torch.cuda.synchronize()
        ro, rl = oracle.decode_partial(q, kv, bt, np.array(lens, dtype=np.int32) + extra, r, P,
                                       case.sm_scale, 0)
        assert np.abs(out.float().cpu().numpy()[:, 0] - ro).max() <= 2e-2
        assert np.abs(lse.cpu().numpy()[:, 0] - rl).max() <= 5e-3
