"""The library's first launches on a device, made from several host threads
at once: each kernel's shared-memory limit is raised once per device under a
lock, so every thread's call launches and all of them agree bit for bit.
Run in a fresh process, so that these are the process's first launches."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, threading
sys.path.insert(0, ROOT)
import torch
import mla_paged_decode_gb300 as mla
import workloads
mla.load_library()
torch.cuda.init()
case = workloads.make_decode_case("threads", 64, [3000, 65, 1, 900], num_parts=3, seed=9,
                                  device="cuda")
B, H = case.batch, case.heads
N = 8
outs = [torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
lses = [torch.empty(B, 1, H, dtype=torch.float32, device="cuda") for _ in range(N)]
wss = [mla.make_workspace(case.q, case.kv_pages, case.block_table) for _ in range(N)]
streams = [torch.cuda.Stream() for _ in range(N)]
torch.cuda.synchronize()
errors = []
start = threading.Barrier(N)

def run(i):
    try:
        torch.cuda.set_device(0)
        start.wait()
        # kernels of three variants, first launched here: the strided gather
        # (P = 3), one partition (P = 1) and the all-partition call (P = 2)
        mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, i % 3, 3,
                           case.sm_scale, 0, outs[i], lses[i], workspace=wss[i], stream=streams[i])
        mla.decode_dcp(case.q, case.kv_pages, case.block_table, case.seq_lens, 2 if i % 2 else 1,
                       case.sm_scale, 0, stream=streams[i])
    except Exception as e:  # reported to the parent
        errors.append(repr(e))

threads = [threading.Thread(target=run, args=(i,)) for i in range(N)]
for t in threads:
    t.start()
for t in threads:
    t.join()
torch.cuda.synchronize()
assert not errors, errors
for i in range(N):
    assert mla.check_workspace(wss[i]) == 0
    j = i % 3
    assert torch.equal(outs[i].view(torch.int16), outs[j].view(torch.int16)), i
    assert torch.equal(lses[i], lses[j]), i
print("threads ok")
"""


def test_first_launches_from_eight_threads():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_decode_gb300 import build
    build.build()
    r = subprocess.run([sys.executable, "-c", CHILD.replace("ROOT", repr(ROOT))],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok" in r.stdout
