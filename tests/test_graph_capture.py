"""Both calls are capture-stable: no host sync, no allocation, caller-owned
buffers.  Captured into a CUDA graph and replayed, they give the same bits as
eager calls (the DCP pages test their combine with and without graphs)."""
import pytest
import torch

import mla_paged_decode_gb300 as mla
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_decode_gb300 import build
    build.build()
    mla.load_library()


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_decode_partials_and_combine_replay_bit_identical(kv_dtype):
    case = workloads.make_decode_case("graph", 64, [3000, 65, 1, 900], num_parts=2, seed=5,
                                      device="cuda", kv_dtype=kv_dtype)
    B, H = case.batch, case.heads
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table, case.kv_scale)
    outs = torch.empty(2, B, 1, H, 512, dtype=torch.bfloat16, device="cuda")
    lses = torch.empty(2, B, 1, H, dtype=torch.float32, device="cuda")
    merged = torch.empty(B, H, 512, dtype=torch.bfloat16, device="cuda")

    def step(stream):
        for r in range(2):
            mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, r, 2,
                               case.sm_scale, 1, outs[r], lses[r], kv_scale=case.kv_scale,
                               workspace=ws, stream=stream)
        mla.lse_combine(outs.view(2, B, H, 512), lses.view(2, B, H), 2, merged, lse_base=1,
                        stream=stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.synchronize()
    eager = (outs.clone(), lses.clone(), merged.clone())
    outs.zero_(); lses.zero_(); merged.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (outs, lses, merged)):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                           b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16))
    assert mla.check_workspace(ws) == 0
