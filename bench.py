"""Benchmark of the MLA absorbed paged-decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one ``mla_decode_partial`` call (P = 1) over the 32K-context batch:
B = 64 requests, H = 64 heads, L ~ U{4096..32768}, bf16 latent KV in a
40,000-page pool, page size 64.  It reads ~1.36 GB of KV per step, far more
than the 129 MB L2, so no flush is needed between steps.  Prints one JSON line:
tokens/s (one new token per request per step), KV GB/s and its fraction of
the measured HBM copy peak, the end-to-end figure through the C ABI with host
buffers, the fp64 CPU oracle timed on the host cores, and SM clocks sampled
from before the warm-up to after the timed region (the GPU kept under the
same load throughout).  At one GPU the line also carries, under "configs",
the same record for the other workloads, measured in the same process: the
small two-partition case (B=1, H=16, L=300, P=2), the eight-partition DCP
batch (B=64, H=16, 60 x 131072 + {1, 3, 5, 7}), the e4m3 batch (B=128,
H=128) and the standalone LSE combine (P=8, T up to 128).

N > 1 (torchrun, one process per GPU): every rank runs its own replica of the
workload (the method's partitions are emulated on one GPU; there is no
exchange), time is the max over ranks, value the sum over ranks.

``--impl reference`` times the fp64 CPU oracle instead (rank 0 only): each
step is one DCP partition (1 of 64) of one request of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MLA decode tokens/s and KV-read HBM GB/s (fraction of roofline) on 1 GB300"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
ROW_BYTES = {"bf16": 576 * 2, "e4m3": 576}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_partial_long32k_traffic.txt")
DCP8_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_dcp_dcp8_traffic.txt")
FP8_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_partial_fp8_traffic.txt")
SMALL_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_dcp_small_traffic.txt")
COMBINE_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "lse_combine_t128_traffic.txt")


# ---------------------------------------------------------------- distributed helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    """Maximum of a per-rank float over all ranks (identity at world 1)."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate(ms_per_rank_max: float, steps: int, units_per_step_per_rank: int, world: int):
    """Whole-job throughput: units of all ranks / the slowest rank's time."""
    secs = ms_per_rank_max / 1e3
    return units_per_step_per_rank * steps * world / secs


# ---------------------------------------------------------------- measurement helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Dense bf16 peak for the secondary (tensor) fraction: the burst figure
    of the measured file, else the recipe's fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


_COMMENT = re.compile(r"/\*.*?\*/|//[^\n]*", re.S)


def code_tokens(text: str) -> str:
    """C++/CUDA source with its comments removed and its whitespace collapsed:
    what the compiler sees of it (the sources carry no `//` or `/*` inside
    string literals)."""
    return " ".join(_COMMENT.sub(" ", text).split())


def kernel_digest(sources=None) -> str:
    """Digest of the kernel sources' code (comments and layout left out): the
    named files of csrc/ (those one kernel and its launch are built from),
    else all of them."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_paged_decode_gb300", "csrc")
    names = sorted(sources) if sources else sorted(
        n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh")))
    for name in names:
        with open(os.path.join(csrc, name)) as f:
            h.update((name + "\n" + code_tokens(f.read())).encode())
    return h.hexdigest()[:16]


def recorded_traffic(path=TRAFFIC_FILE):
    """DRAM bytes per launch from a committed ncu summary under profiles/, if
    it was taken on the current sources of that kernel (its `sources` line
    names them; else None)."""
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if "=" in line and not line.startswith("#"):
            k, v = line.strip().split("=", 1)
            kv[k.strip()] = v.strip()
    sources = [s.strip() for s in kv.get("sources", "").split(",") if s.strip()]
    if kv.get("kernel_digest") != kernel_digest(sources or None):
        return None
    try:
        return int(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background.

    Started before the warm-up: wait_first() returns once nvidia-smi has
    written its first sample (taken before any load, so stop() leaves it
    out), and the caller then keeps the GPU under the step's load from
    before the warm-up until after the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 50):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            uuid = None
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", str(period_ms)]
        if uuid:
            cmd[1:1] = ["-i", uuid]
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def wait_first(self, timeout_s: float = 5.0) -> bool:
        """True once the first sample line is on disk (False on timeout)."""
        if self.proc is None:
            return False
        t_end = time.perf_counter() + timeout_s
        while time.perf_counter() < t_end:
            self.out.flush()
            try:
                with open(self.path) as f:
                    if f.read().count("\n") >= 1:
                        return True
            except OSError:
                pass
            if self.proc.poll() is not None:
                return False
            time.sleep(0.01)
        return False

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = open(self.path).read().splitlines()
        for line in lines[1:]:  # the first sample was taken before the load
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "nvidia-smi every 50 ms while the GPU runs this step: %.2f s of the "
                          "same steps before the warm-up, the warm-up, the timed region and "
                          "%.2f s of the same steps after it" % (LOAD_BEFORE_S, LOAD_AFTER_S)}


def gpu_setup(world: int, rank: int, local: int):
    """This rank's device and current stream, the process group, and the
    in-tree library (built by rank 0, or by any rank that finds it missing)."""
    import mla_paged_decode_gb300 as mla
    from mla_paged_decode_gb300 import build
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    if rank == 0 or not os.path.exists(mla.library_path()):
        build.build()
    barrier(world)
    mla.load_library()
    return mla, dev, torch.cuda.current_stream(dev)


def timed_steps(step, steps: int, warmup: int, world: int, dev, stream, sample_clocks=False,
                side_streams=(), tail=None):
    """`warmup` untimed calls of step(), then exactly `steps` timed ones,
    bracketed by a barrier and a synchronize on both sides and timed with CUDA
    events on `stream` (which side streams wait for before their first copy;
    `tail` runs after the last step, inside the region).  Returns the
    milliseconds (max over ranks) and the clock record (or None).

    With sample_clocks, nvidia-smi samples from before the warm-up until after
    the timed region; untimed runs of the same step before the warm-up and
    after the region keep the GPU under this load long enough for samples
    even when the region itself lasts a few milliseconds."""
    clocks = None
    if sample_clocks:
        clocks = ClockSampler(dev.index)
        clocks.wait_first()
        _load(step, LOAD_BEFORE_S, dev)
    for _ in range(warmup):
        step()
    if tail:
        tail()
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for st in side_streams:
        st.wait_event(e0)
    for _ in range(steps):
        step()
    if tail:
        tail()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    info = None
    if clocks:
        _load(step, LOAD_AFTER_S, dev)
        info = clocks.stop()
    return max_over_ranks(e0.elapsed_time(e1), world, dev), info


LOAD_BEFORE_S = 0.4   # untimed runs of the step around a clock-sampled region
LOAD_AFTER_S = 0.2


def _load(step, seconds: float, dev):
    """Runs step() for about `seconds` (untimed), in batches of 8 calls."""
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        for _ in range(8):
            step()
        torch.cuda.synchronize(dev)


GRAPH_CALLS = 20  # calls captured in one graph


def graph_time(call, dev, stream, steps: int) -> float:
    """Milliseconds for `steps` calls of call(stream) replayed from CUDA
    graphs of GRAPH_CALLS calls each (3 replays of warm-up first)."""
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for _ in range(GRAPH_CALLS):
            call(cap)
    stream.wait_stream(cap)
    replays = max(1, steps // GRAPH_CALLS)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) * steps / (replays * GRAPH_CALLS)


def e2e_times(op, host_in, outputs, args, world, dev, stream):
    """End-to-end timing of a call through the public API with host buffers.

    host_in: the step's inputs as pinned host tensors; outputs: device
    tensors shaped like the step's results; op(inp, out) enqueues the call on
    `stream` with device inputs `inp` and outputs `out` (dicts by the same
    names).  Every step copies its inputs in from pinned host memory and reads
    its results back.  Timed twice: serially on one stream, and as a serving
    loop runs it (device inputs and outputs double-buffered, step i's inputs
    copied in on one copy stream while step i - 1 computes, its results read
    back on another while step i + 1 computes; the last read-back is inside
    the region).  Returns (pipelined ms, serial ms, H2D bytes, D2H bytes) per
    `args.steps` steps; the results of both loops must agree bit for bit."""
    def dev_like(t):
        return torch.empty(t.shape, dtype=t.dtype, device=dev)

    def host_like(t):
        return torch.empty(t.shape, dtype=t.dtype).pin_memory()

    d_in = {k: dev_like(v) for k, v in host_in.items()}
    d_out = {k: dev_like(v) for k, v in outputs.items()}
    h_out = {k: host_like(v) for k, v in outputs.items()}

    def serial_step():
        for k, v in host_in.items():
            d_in[k].copy_(v, non_blocking=True)
        op(d_in, d_out)
        for k, v in h_out.items():
            v.copy_(d_out[k], non_blocking=True)

    with torch.cuda.stream(stream):
        serial_ms, _ = timed_steps(serial_step, args.steps, max(3, args.warmup), world, dev, stream)

    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = [dict(inp={k: dev_like(v) for k, v in host_in.items()},
                 out={k: dev_like(v) for k, v in outputs.items()},
                 host={k: host_like(v) for k, v in outputs.items()},
                 ev_in=torch.cuda.Event(), ev_done=torch.cuda.Event(), ev_out=torch.cuda.Event())
            for _ in range(2)]
    for bb in bufs:  # so that the first waits on them are satisfied
        bb["ev_done"].record(stream)
        bb["ev_out"].record(stream)
    it = [0]

    def pipelined_step():
        bb = bufs[it[0] % 2]
        it[0] += 1
        h2d_s.wait_event(bb["ev_done"])        # the call that last read these inputs
        with torch.cuda.stream(h2d_s):
            for k, v in host_in.items():
                bb["inp"][k].copy_(v, non_blocking=True)
        bb["ev_in"].record(h2d_s)
        stream.wait_event(bb["ev_in"])
        stream.wait_event(bb["ev_out"])         # the read-back of this buffer's last results
        op(bb["inp"], bb["out"])
        bb["ev_done"].record(stream)
        d2h_s.wait_event(bb["ev_done"])
        with torch.cuda.stream(d2h_s):
            for k, v in bb["host"].items():
                v.copy_(bb["out"][k], non_blocking=True)
        bb["ev_out"].record(d2h_s)

    def drain():  # the last results are read back inside the timed region
        for bb in bufs:
            stream.wait_event(bb["ev_out"])

    pipe_ms, _ = timed_steps(pipelined_step, args.steps, max(3, args.warmup), world, dev, stream,
                             side_streams=(h2d_s, d2h_s), tail=drain)
    torch.cuda.synchronize(dev)
    for bb in bufs:
        for k, v in h_out.items():
            a, b = bb["host"][k], v
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), k
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in outputs.values())
    return pipe_ms, serial_ms, h2d, d2h


E2E_NOTE = ("inputs copied from pinned host memory and results read back every step; the KV "
            "cache stays resident in HBM. pipelined_value: copies double-buffered on two copy "
            "streams, overlapping the neighbouring steps' computation (a serving loop); "
            "serial_value: every copy and the call in sequence on one stream; value: the "
            "faster of the two (mode)")


def e2e_record(units_per_step, args, world, pipe_ms, serial_ms, h2d, d2h, unit, what):
    """The e2e key: the faster of the pipelined and serial loops as `value`
    (a latency-bound step gains nothing from the copy streams and pays their
    bookkeeping), both reported."""
    pipe = aggregate(pipe_ms, args.steps, units_per_step, world)
    serial = aggregate(serial_ms, args.steps, units_per_step, world)
    return {"value": max(pipe, serial), "unit": unit,
            "mode": "pipelined" if pipe >= serial else "serial",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined_value": pipe, "serial_value": serial, "note": what + ": " + E2E_NOTE}


def cpu_baseline(case, seconds: float):
    """The fp64 oracle, as it stands, on whole requests of the same workload
    until ``seconds`` of CPU time have passed."""
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from casebits import subcase_bits
    done, spent = 0, 0.0
    tokens = 0
    while spent < seconds and done < case.batch:
        q, kv, bt, lens = subcase_bits(case, [done])
        t0 = time.perf_counter()
        oracle.decode_partial(q, kv, bt, lens, 0, 1, case.sm_scale, 0, kv_dtype=case.kv_dtype,
                              kv_scale=case.kv_scale)
        spent += time.perf_counter() - t0
        tokens += int(lens[0])
        done += 1
    return {"value": done / spent, "unit": "tokens/s", "cores": _oracle_threads(),
            "kind": "oracle",
            "sample": f"first {done} of {case.batch} requests of the same batch "
                      f"({tokens} cached tokens, all {case.heads} heads), fp64 numpy, "
                      f"{spent:.1f} s"}


def _oracle_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads", 1) for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ---------------------------------------------------------------- the two arms

def run_ours(args, world, rank, local):
    """The headline line; at one GPU it also carries, under "configs", the
    same record for each of the other workloads (the small two-partition
    case, the eight-partition DCP batch, the e4m3 batch and the standalone
    combine), measured in the same process."""
    mla, dev, stream = gpu_setup(world, rank, local)
    line = measure_decode(args, world, rank, mla, dev, stream)
    if world == 1 and not args.no_configs:
        sub = argparse.Namespace(**vars(args))
        sub.steps = min(max(args.steps, 20), 200)
        sub.cpu_seconds = min(args.cpu_seconds, 6.0)
        configs = {}
        for measure in (measure_small, measure_dcp8, measure_fp8, measure_combine):
            torch.cuda.empty_cache()
            sub.batch = 128 if measure is measure_fp8 else 64  # each workload's own batch
            rec = measure(sub, world, rank, mla, dev, stream)
            configs[rec["config"]["workload"]] = rec
        line["configs"] = configs
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_decode(args, world, rank, mla, dev, stream):
    """One mla_decode_partial call (P = 1) over the 32K-context batch per step."""
    case = workloads.config_long32k(device=dev, seed=args.seed, batch=args.batch,
                                    pool_pages=args.pool_pages)
    if args.batch != 64 or args.pool_pages != 40000:
        case.name += f"_b{args.batch}_pool{args.pool_pages}"
    B, H = case.batch, case.heads
    kv_bytes = int(case.seq_lens.sum().item()) * ROW_BYTES[case.kv_dtype]
    out = torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, 1, H, dtype=torch.float32, device=dev)
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table)

    def step():
        mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, 0, 1,
                           case.sm_scale, 0, out, lse, workspace=ws, stream=stream)

    ms_max, clock_info = timed_steps(step, args.steps, args.warmup, world, dev, stream,
                                     sample_clocks=True)
    assert mla.check_workspace(ws) == 0

    # The same calls replayed from a CUDA graph (reported separately): the
    # host's launch work leaves the timed region.
    graph_ms = graph_time(lambda st: mla.decode_partial(
        case.q, case.kv_pages, case.block_table, case.seq_lens, 0, 1, case.sm_scale, 0, out, lse,
        workspace=ws, stream=st), dev, stream, args.steps)
    graph_ms_max = max_over_ranks(graph_ms, world, dev)
    assert mla.check_workspace(ws) == 0

    # end to end through the C ABI with host buffers: pinned H2D inputs, D2H results
    def e2e_op(inp, o):
        mla.decode_partial(inp["q"], case.kv_pages, inp["bt"], inp["sl"], 0, 1, case.sm_scale, 0,
                           o["out"], o["lse"], workspace=ws, stream=stream)

    e_ms_max, e_serial_ms, h2d, d2h = e2e_times(
        e2e_op, {"q": case.q.cpu().pin_memory(), "bt": case.block_table.cpu().pin_memory(),
                 "sl": case.seq_lens.cpu().pin_memory()}, {"out": out, "lse": lse},
        args, world, dev, stream)

    value = aggregate(ms_max, args.steps, B, world)
    avg_launch_s = ms_max / 1e3 / args.steps
    peak, peak_kind = measured_peaks()
    achieved = kv_bytes / avg_launch_s / 1e9
    flops = float(case.seq_lens.sum().item()) * H * (2 * 576 + 2 * 512)
    tflops = flops / avg_launch_s / 1e12
    tpeak, tpeak_kind = measured_bf16_tflops()
    traffic = recorded_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": case.name, "batch": B, "heads": H, "q_len": 1,
                   "seq_lens": "uniform 4096..32768 (seed %d)" % args.seed,
                   "mean_seq_len": kv_bytes / ROW_BYTES[case.kv_dtype] / B,
                   "page_size": 64, "pool_pages": case.num_pages, "num_parts": 1,
                   "kv_dtype": "bf16", "kv_bytes_per_step": kv_bytes,
                   "l2": "inputs larger than L2: %.2f GB of KV read per step, no flush" % (kv_bytes / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "kv_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "frac_of_8tbs": achieved / 8000.0,
                     "traffic": traffic,
                     "kernel": "mla_decode_partial: decode kernel + split merge, timed "
                               "together per call (CUDA events on the launching stream)",
                     # secondary: algorithmic flops of the real heads (QK^T over 576 dims,
                     # PV over 512) against the dense bf16 peak; the padding of the
                     # score MMA to 64 rows is not counted
                     "tensor_tflops": tflops, "tensor_peak_tflops": tpeak,
                     "tensor_frac": tflops / tpeak, "tensor_peak_source": tpeak_kind},
        "e2e": e2e_record(B, args, world, e_ms_max, e_serial_ms, h2d, d2h, "tokens/s",
                          "q, block table and lengths in, out and lse back"),
        "graph": {"value": aggregate(graph_ms_max, args.steps, B, world), "unit": "tokens/s",
                  "ms_per_step": graph_ms_max / args.steps, "calls_per_graph": GRAPH_CALLS,
                  "note": "the same calls replayed from CUDA graphs (not the headline)"},
        # each mla_decode_partial call launches the decode kernel and the split merge
        "gpu_launches": 2 * args.steps,
        "clocks": clock_info,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, args.cpu_seconds)
    return line


def run_reference(args, world, rank):
    """The fp64 CPU oracle as it stands, one DCP partition (1 of 64) of one
    request per step, on the host cores."""
    if rank != 0:
        return
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from casebits import subcase_bits
    # the same seeded batch as the GPU arm (drawn on the GPU when there is one,
    # so both arms see identical values); only the sampled pages reach the host
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = workloads.config_long32k(device=gen_dev, seed=args.seed)
    P = 64
    B = case.batch
    subs = {}

    def step(i):
        b, r = (i // P) % B, i % P
        if b not in subs:
            subs.clear()
            subs[b] = subcase_bits(case, [b])
        q, kv, bt, lens = subs[b]
        oracle.decode_partial(q, kv, bt, lens, r, P, case.sm_scale, 0)

    for i in range(args.warmup):
        step(i)
    spent = 0.0
    for i in range(args.steps):
        b = (i // P) % B
        if b not in subs:
            subs.clear()
            subs[b] = subcase_bits(case, [b])
        t0 = time.perf_counter()
        step(i)
        spent += time.perf_counter() - t0
    value = (args.steps / P) / spent
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": spent * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": case.name, "batch": B, "heads": case.heads, "page_size": 64,
                   "num_parts": 1, "seq_lens": "uniform 4096..32768 (seed %d)" % args.seed},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _oracle_threads(),
                         "kind": "oracle",
                         "sample": "each step: one round-robin partition (1 of 64) of one "
                                   "request, all heads; tokens/s counts 1/64 token per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _append_subcache(case_bits_, B):
    """The pages the append touches, copied into a compact cache (oracle sample)."""
    kv, bt, pos = case_bits_
    pages = [int(bt[b, int(pos[b]) // 64]) for b in range(B)]
    uniq = sorted(set(pages))
    remap = {p: i for i, p in enumerate(uniq)}
    small = kv[uniq]
    sbt = np.zeros((B, bt.shape[1]), dtype=np.int32)
    for b in range(B):
        sbt[b, int(pos[b]) // 64] = remap[pages[b]]
    return small, sbt


def run_append(args, world, rank, local):
    """--op kv_append: one new cache row per request of the headline batch
    (each request's last token rewritten, so its table needs no new page)."""
    mla, dev, stream = gpu_setup(world, rank, local)
    case = workloads.config_long32k(device=dev, seed=args.seed, batch=args.batch,
                                    pool_pages=args.pool_pages)
    B = case.batch
    pos = (case.seq_lens - 1).contiguous()
    g = torch.Generator().manual_seed(args.seed + 1)
    new = torch.randn(B, 576, generator=g).to(torch.bfloat16).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        mla.kv_append(new, case.kv_pages, case.block_table, pos, 0, 1, error_word=err,
                      stream=stream)

    ms, clock_info = timed_steps(step, args.steps, args.warmup, world, dev, stream,
                                 sample_clocks=True)
    assert int(err.item()) == 0
    # end to end: the new rows and positions from pinned host memory, the error word back
    def e2e_op(inp, o):
        mla.kv_append(inp["new"], case.kv_pages, case.block_table, inp["pos"], 0, 1,
                      error_word=o["err"], stream=stream)

    e_ms, e_serial_ms, h2d, d2h = e2e_times(
        e2e_op, {"new": new.cpu().pin_memory(), "pos": pos.cpu().pin_memory()},
        {"err": torch.zeros(1, dtype=torch.int32, device=dev)}, args, world, dev, stream)
    per_s = ms / 1e3 / args.steps
    byts = B * (1152 + 1152 + 8)   # new row read, cache row written, position + table entry
    peak, peak_kind = measured_peaks()
    line = {
        "metric": "KV append: new cache rows per second (one per request), 1 GB300",
        "value": aggregate(ms, args.steps, B, world), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "kv_append_" + case.name, "batch": B, "kv_dtype": "bf16",
                   "positions": "each request's last token", "pool_pages": case.num_pages,
                   "l2": "no flush: 147 KB per step, latency-bound"},
        "roofline": {"bound": "hbm", "achieved": byts / per_s / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": byts / per_s / 1e9 / peak, "peak_source": peak_kind,
                     "traffic": None,
                     "kernel": "mla_kv_append (one launch per step); far below the HBM roof: "
                               "a launch-latency-bound write of B rows"},
        "e2e": e2e_record(B, args, world, e_ms, e_serial_ms, h2d, d2h, "rows/s",
                          "the new rows and positions in, the error word back"),
        "gpu_launches": args.steps,
        "clocks": clock_info,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        import oracle
        kv_b = case.kv_pages.view(torch.int16).cpu().numpy().view(np.uint16)
        bt = case.block_table.cpu().numpy()
        small, sbt = _append_subcache((kv_b, bt, pos.cpu().numpy()), B)
        new_b = new.view(torch.int16).cpu().numpy().view(np.uint16)
        spent, calls = 0.0, 0
        while spent < min(args.cpu_seconds, 5.0):
            a = time.perf_counter()
            oracle.kv_append(small, sbt, pos.cpu().numpy(), new_b, 0, 1)
            spent += time.perf_counter() - a
            calls += 1
        line["cpu_baseline"] = {"value": calls * B / spent, "unit": "rows/s", "cores": 1,
                                "kind": "oracle",
                                "sample": f"{calls} appends of the {B} rows into a compact copy "
                                          f"of the {len(small)} touched pages, {spent:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def _print_line(make):
    """Runs one op's measurement and prints its line (rank 0)."""
    def run(args, world, rank, local):
        mla, dev, stream = gpu_setup(world, rank, local)
        line = make(args, world, rank, mla, dev, stream)
        if rank == 0:
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
    return run


def measure_dcp8(args, world, rank, mla, dev, stream):
    """--op dcp8: the decode-context-parallel workload (B=64, H=16, P=8; 60
    requests of 131072 tokens and four of 1, 3, 5, 7) as one mla_decode_dcp
    call per step: every partition's (out, lse) and their combine."""
    case = workloads.config_dcp8(device=dev, seed=args.seed, n_long=args.n_long)
    if args.n_long != 60:
        case.name += f"_long{args.n_long}"
    B, H, P = case.batch, case.heads, case.num_parts
    kv_bytes = int(case.seq_lens.sum().item()) * ROW_BYTES[case.kv_dtype]
    ws = mla.make_dcp_workspace(case.q, case.kv_pages, case.block_table, P)
    parts = torch.empty(P, B, 1, H, 512, dtype=torch.bfloat16, device=dev)
    plse = torch.empty(P, B, 1, H, dtype=torch.float32, device=dev)
    out = torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device=dev)
    out_lse = torch.empty(B, 1, H, dtype=torch.float32, device=dev)

    def step(q=case.q, bt=case.block_table, sl=case.seq_lens):
        mla.decode_dcp(q, case.kv_pages, bt, sl, P, case.sm_scale, 1, partials=parts,
                       partial_lses=plse, out=out, out_lse=out_lse, workspace=ws, stream=stream)

    ms, clock_info = timed_steps(step, args.steps, args.warmup, world, dev, stream,
                                 sample_clocks=True)
    assert mla.check_workspace(ws) == 0
    def e2e_op(inp, o):
        mla.decode_dcp(inp["q"], case.kv_pages, inp["bt"], inp["sl"], P, case.sm_scale, 1,
                       partials=parts, partial_lses=plse, out=o["out"], out_lse=o["lse"],
                       workspace=ws, stream=stream)

    e_ms, e_serial_ms, h2d, d2h = e2e_times(
        e2e_op, {"q": case.q.cpu().pin_memory(), "bt": case.block_table.cpu().pin_memory(),
                 "sl": case.seq_lens.cpu().pin_memory()}, {"out": out, "lse": out_lse},
        args, world, dev, stream)
    per_s = ms / 1e3 / args.steps
    peak, peak_kind = measured_peaks()
    tpeak, tpeak_kind = measured_bf16_tflops()
    flops = float(case.seq_lens.sum().item()) * H * (2 * 576 + 2 * 512)
    line = {
        "metric": "MLA decode tokens/s and KV-read HBM GB/s (fraction of roofline) on 1 GB300",
        "value": aggregate(ms, args.steps, B, world), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": case.name, "batch": B, "heads": H, "q_len": 1, "num_parts": P,
                   "seq_lens": "60 x 131072 + {1, 3, 5, 7}", "page_size": 64,
                   "pool_pages": case.num_pages, "kv_dtype": "bf16", "kv_bytes_per_step": kv_bytes,
                   "l2": "inputs larger than L2: %.2f GB of KV read per step, no flush" % (kv_bytes / 1e9),
                   "parallelism": "DCP partitions emulated on one GPU"},
        "roofline": {"bound": "hbm", "achieved": kv_bytes / per_s / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": kv_bytes / per_s / 1e9 / peak,
                     "peak_source": peak_kind, "frac_of_8tbs": kv_bytes / per_s / 1e9 / 8000.0,
                     "traffic": recorded_traffic(DCP8_TRAFFIC_FILE),
                     "kernel": "mla_decode_dcp: one decode launch over the 8 partitions and "
                               "one split merge with the LSE combine fused, timed together "
                               "per call",
                     "tensor_tflops": flops / per_s / 1e12, "tensor_peak_tflops": tpeak,
                     "tensor_frac": flops / per_s / 1e12 / tpeak, "tensor_peak_source": tpeak_kind},
        "e2e": e2e_record(B, args, world, e_ms, e_serial_ms, h2d, d2h, "tokens/s",
                          "q, block table and lengths in, the result and its lse back"),
        "gpu_launches": 2 * args.steps,
        "clocks": clock_info,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        import oracle
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from casebits import subcase_bits
        spent, tokens, done = 0.0, 0, 0
        while spent < args.cpu_seconds and done < B:
            q, kv, bt, lens = subcase_bits(case, [done])
            a = time.perf_counter()
            for r in range(P):
                oracle.decode_partial(q, kv, bt, lens, r, P, case.sm_scale, 1)
            spent += time.perf_counter() - a
            tokens += int(lens[0])
            done += 1
        line["cpu_baseline"] = {"value": done / spent, "unit": "tokens/s", "cores": _oracle_threads(),
                                "kind": "oracle",
                                "sample": f"all {P} partitions of the first {done} of {B} requests "
                                          f"({tokens} cached tokens), fp64 numpy, {spent:.1f} s"}
    return line


run_dcp8 = _print_line(measure_dcp8)


def measure_fp8(args, world, rank, mla, dev, stream):
    """--op fp8: the e4m3-cache workload (B=128, H=128, lognormal lengths with
    median 8192, per-tensor scale, P=1) through mla_decode_partial.  Its
    roofline is the tensor pipe: the MMAs run on e4m3 operands, the cache's
    raw rows with Q and P each as two fp8 terms (so every product is two
    MMAs, and the executed MMA flops are twice the algorithmic ones); the
    two 64-head groups of a request walk its pages side by side on two SMs,
    so the second read of a page is served by L2."""
    case = workloads.config_fp8(device=dev, seed=args.seed, batch=args.batch)
    if args.batch != 128:
        case.name += f"_b{args.batch}"
    B, H = case.batch, case.heads
    n_tok = int(case.seq_lens.sum().item())
    kv_bytes = n_tok * ROW_BYTES[case.kv_dtype]
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table, case.kv_scale)
    out = torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, 1, H, dtype=torch.float32, device=dev)

    def step(q=case.q, bt=case.block_table, sl=case.seq_lens):
        mla.decode_partial(q, case.kv_pages, bt, sl, 0, 1, case.sm_scale, 0, out, lse,
                           kv_scale=case.kv_scale, workspace=ws, stream=stream)

    ms, clock_info = timed_steps(step, args.steps, args.warmup, world, dev, stream,
                                 sample_clocks=True)
    assert mla.check_workspace(ws) == 0
    def e2e_op(inp, o):
        mla.decode_partial(inp["q"], case.kv_pages, inp["bt"], inp["sl"], 0, 1, case.sm_scale, 0,
                           o["out"], o["lse"], kv_scale=case.kv_scale, workspace=ws, stream=stream)

    e_ms, e_serial_ms, h2d, d2h = e2e_times(
        e2e_op, {"q": case.q.cpu().pin_memory(), "bt": case.block_table.cpu().pin_memory(),
                 "sl": case.seq_lens.cpu().pin_memory()}, {"out": out, "lse": lse},
        args, world, dev, stream)
    per_s = ms / 1e3 / args.steps
    peak, peak_kind = measured_peaks()
    bpeak, bpeak_kind = measured_bf16_tflops()
    # dense e4m3 peak: the measured bf16 figure times the nominal fp8 / bf16
    # ratio (4.5 / 2.25 PFLOP/s)
    tpeak = 2.0 * bpeak
    flops = float(n_tok) * H * (2 * 576 + 2 * 512)
    tflops = flops / per_s / 1e12
    line = {
        "metric": "MLA decode tokens/s and KV-read HBM GB/s (fraction of roofline) on 1 GB300",
        "value": aggregate(ms, args.steps, B, world), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": case.name, "batch": B, "heads": H, "q_len": 1, "num_parts": 1,
                   "seq_lens": "lognormal, median 8192, sigma 1, clipped to [1024, 65536] (seed %d)"
                               % args.seed,
                   "page_size": 64, "pool_pages": case.num_pages, "kv_dtype": "e4m3",
                   "kv_bytes_per_step": kv_bytes,
                   "l2": "%.2f GB of e4m3 KV per step (more than L2); the two 64-head groups "
                         "of a request read it side by side, the second read from L2"
                         % (kv_bytes / 1e9),
                   "parallelism": "single GPU"},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": tpeak,
                     "unit": "TFLOP/s", "frac": tflops / tpeak,
                     "peak_source": bpeak_kind + " bf16 x 2 (nominal e4m3 / bf16 ratio)",
                     "traffic": recorded_traffic(FP8_TRAFFIC_FILE),
                     "kernel": "mla_decode_partial on an e4m3 cache: decode kernel + split merge, "
                               "timed together per call (e4m3 MMAs on the raw cache rows; real "
                               "heads' flops, QK^T over 576 dims and PV over 512)",
                     "mma_tflops": 2.0 * tflops, "mma_frac": 2.0 * tflops / tpeak,
                     "mma_note": "Q and P enter the MMAs as two fp8 terms each (hi + lo), so "
                                 "the MMAs execute twice the algorithmic flops",
                     "hbm_achieved_gbs": kv_bytes / per_s / 1e9, "hbm_peak_gbs": peak,
                     "hbm_frac": kv_bytes / per_s / 1e9 / peak, "hbm_peak_source": peak_kind},
        "e2e": e2e_record(B, args, world, e_ms, e_serial_ms, h2d, d2h, "tokens/s",
                          "q, block table and lengths in, the result and its lse back"),
        "gpu_launches": 2 * args.steps,
        "clocks": clock_info,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, args.cpu_seconds)
    return line


run_fp8 = _print_line(measure_fp8)


def _line(args, world, ms, units, unit, config, roofline, e2e, launches, clock_info,
          metric="MLA decode tokens/s and KV-read HBM GB/s (fraction of roofline) on 1 GB300"):
    """The JSON line's common keys for `units` processed per step per rank."""
    return {"metric": metric, "value": aggregate(ms, args.steps, units, world), "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
            "roofline": roofline, "e2e": e2e, "gpu_launches": launches, "clocks": clock_info}


def _hbm_roofline(kv_bytes, ms, steps, kernel):
    peak, peak_kind = measured_peaks()
    gbs = kv_bytes / (ms / 1e3 / steps) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
            "peak_source": peak_kind, "frac_of_8tbs": gbs / 8000.0, "traffic": None,
            "kernel": kernel}


def run_dcp_parts(args, world, rank, local):
    """--op dcp --parts P: the 32K-context batch (B=64, H=64, bf16) as P
    round-robin partitions and their merge, one mla_decode_dcp call per step
    (the tensor-core kernel: one launch for all partitions when P > 1 divides 8
    or P is 3, 5, 6 or 7 (the strided gather), else one launch per partition:
    P = 1 the single-partition kernel, larger P the owner mask when
    P / gcd(P, 8) <= 16, else the CUDA-core kernel).  KV GB/s counts each
    cached row once."""
    mla, dev, stream = gpu_setup(world, rank, local)
    P = args.parts
    case = workloads.config_long32k(device=dev, seed=args.seed, batch=args.batch,
                                    pool_pages=args.pool_pages)
    B, H = case.batch, case.heads
    kv_bytes = int(case.seq_lens.sum().item()) * ROW_BYTES[case.kv_dtype]
    ws = mla.make_dcp_workspace(case.q, case.kv_pages, case.block_table, P)
    parts = torch.empty(P, B, 1, H, 512, dtype=torch.bfloat16, device=dev)
    plse = torch.empty(P, B, 1, H, dtype=torch.float32, device=dev)
    out = torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device=dev)

    def step():
        mla.decode_dcp(case.q, case.kv_pages, case.block_table, case.seq_lens, P, case.sm_scale,
                       0, partials=parts, partial_lses=plse, out=out, workspace=ws, stream=stream)

    ms, clock_info = timed_steps(step, args.steps, args.warmup, world, dev, stream,
                                 sample_clocks=True)
    assert mla.check_workspace(ws) == 0

    def e2e_op(inp, o):
        mla.decode_dcp(inp["q"], case.kv_pages, inp["bt"], inp["sl"], P, case.sm_scale, 0,
                       partials=parts, partial_lses=plse, out=o["out"], out_lse=o["lse"],
                       workspace=ws, stream=stream)

    e_ms, e_serial_ms, h2d, d2h = e2e_times(
        e2e_op, {"q": case.q.cpu().pin_memory(), "bt": case.block_table.cpu().pin_memory(),
                 "sl": case.seq_lens.cpu().pin_memory()},
        {"out": out, "lse": torch.empty(B, 1, H, dtype=torch.float32, device=dev)},
        args, world, dev, stream)
    g = math.gcd(P, 8)
    one_launch = 1 < P <= 8
    path = ("mla_decode_partial's kernels on the one partition, then the combine (a copy)"
            if P == 1 else "one launch for all partitions" if 8 % P == 0 else
            "one launch for all partitions, strided gather (rows y0 + kP of each page)"
            if one_launch else
            "one launch per partition, owner mask over the gather of partition r mod %d" % g
            if P // g <= 16 else "the CUDA-core kernel, one launch per partition")
    line = _line(args, world, ms, B, "tokens/s",
                 {"workload": "long32k_b64_h64_bf16_p%d" % P, "batch": B, "heads": H, "q_len": 1,
                  "num_parts": P, "path": path, "kv_bytes_per_step": kv_bytes,
                  "l2": "inputs larger than L2: %.2f GB of KV per step" % (kv_bytes / 1e9),
                  "parallelism": "DCP partitions emulated on one GPU"},
                 _hbm_roofline(kv_bytes, ms, args.steps,
                               "mla_decode_dcp: every partition's decode and the merge, timed "
                               "together per call (rows gathered P / gcd(P, 8) times when P > 8 "
                               "does not divide 8)"),
                 e2e_record(B, args, world, e_ms, e_serial_ms, h2d, d2h, "tokens/s",
                            "q, block table and lengths in, the merged result and its lse back"),
                 # the decode (+ its split merge) per partition launch, then the combine
                 (2 if one_launch else 2 * P + 1) * args.steps, clock_info)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_mtp(args, world, rank, local):
    """--op mtp --q-len T: T query tokens per request (multi-token prediction
    or target verify) on the 32K-context lengths, B=64, H=64, P=1; query token
    i attends to the tokens before L - T + i + 1.  One 64-row group per query
    token, each on its own SM; the groups of a request walk its pages side by
    side, so HBM serves each page once and L2 the other groups' reads.  KV
    GB/s counts each cached row once."""
    mla, dev, stream = gpu_setup(world, rank, local)
    T = args.q_len
    case = workloads.config_long32k(device=dev, seed=args.seed, q_len=T)
    B, H = case.batch, case.heads
    kv_bytes = int(case.seq_lens.sum().item()) * ROW_BYTES[case.kv_dtype]
    ws = mla.make_workspace(case.q, case.kv_pages, case.block_table)
    out = torch.empty(B, T, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, T, H, dtype=torch.float32, device=dev)

    def step():
        mla.decode_partial(case.q, case.kv_pages, case.block_table, case.seq_lens, 0, 1,
                           case.sm_scale, 0, out, lse, workspace=ws, stream=stream)

    ms, clock_info = timed_steps(step, args.steps, args.warmup, world, dev, stream,
                                 sample_clocks=True)
    assert mla.check_workspace(ws) == 0

    def e2e_op(inp, o):
        mla.decode_partial(inp["q"], case.kv_pages, inp["bt"], inp["sl"], 0, 1, case.sm_scale, 0,
                           o["out"], o["lse"], workspace=ws, stream=stream)

    e_ms, e_serial_ms, h2d, d2h = e2e_times(
        e2e_op, {"q": case.q.cpu().pin_memory(), "bt": case.block_table.cpu().pin_memory(),
                 "sl": case.seq_lens.cpu().pin_memory()}, {"out": out, "lse": lse},
        args, world, dev, stream)
    groups = -(-T * H // 64)
    line = _line(args, world, ms, B * T, "query tokens/s",
                 {"workload": "long32k_b64_h64_bf16_q%d" % T, "batch": B, "heads": H, "q_len": T,
                  "num_parts": 1, "row_groups_per_request": groups, "kv_bytes_per_step": kv_bytes,
                  "l2": "inputs larger than L2: %.2f GB of KV per step" % (kv_bytes / 1e9),
                  "parallelism": "single GPU"},
                 _hbm_roofline(kv_bytes, ms, args.steps,
                               "mla_decode_partial with %d query tokens: decode kernel + split "
                               "merge; bytes = the KV once (%d 64-row groups read it side by "
                               "side)" % (T, groups)),
                 e2e_record(B * T, args, world, e_ms, e_serial_ms, h2d, d2h, "query tokens/s",
                            "q (all query tokens), block table and lengths in, out and lse back"),
                 2 * args.steps, clock_info)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_combine(args, world, rank, mla, dev, stream):
    """--op combine: mla_lse_combine alone on the micro-benchmark shapes (P=8,
    H=16, D=512, T in {1, 8, 16, 32, 64, 128} tokens; partials N(0, 1) bf16,
    lse N(5, 3), one partition per token holding the neutral pair), each
    call replayed from CUDA graphs so that the small launches are timed on
    the device.  value: GB/s at T = 128; every T in `points`.  e2e: the
    T = 128 call with its partials and lses copied in from pinned host
    memory and its result read back, every step."""
    P, H, D = 8, 16, 512
    points = []
    for T in args.tokens:
        c = workloads.combine_case(T, num_parts=P, heads=H, dim=D, seed=args.seed, device=dev)
        out = torch.empty(T, H, D, dtype=torch.bfloat16, device=dev)
        out_lse = torch.empty(T, H, dtype=torch.float32, device=dev)

        def call(st, c=c, out=out, out_lse=out_lse):
            mla.lse_combine(c.partials, c.lses, P, out, lse_base=mla.LSE_NATURAL,
                            out_lse=out_lse, stream=st)

        for _ in range(args.warmup):
            call(stream)
        torch.cuda.synchronize(dev)
        ms = max_over_ranks(graph_time(call, dev, stream, args.steps), world, dev)
        us = ms * 1e3 / args.steps
        nbytes = c.partials.numel() * 2 + c.lses.numel() * 4 + out.numel() * 2 + out_lse.numel() * 4
        points.append({"tokens": T, "us_per_call": us, "gbs": nbytes / us / 1e3,
                       "bytes_per_call": nbytes})
    # the clock record: the same call eagerly, sampled around its region
    _, clock_info = timed_steps(lambda: call(stream), args.steps, args.warmup, world, dev, stream,
                                sample_clocks=True)

    # end to end at the last T through the C ABI with host buffers
    def e2e_op(inp, o):
        mla.lse_combine(inp["partials"], inp["lses"], P, o["out"], lse_base=mla.LSE_NATURAL,
                        out_lse=o["lse"], stream=stream)

    e_ms, e_serial_ms, h2d, d2h = e2e_times(
        e2e_op, {"partials": c.partials.cpu().pin_memory(), "lses": c.lses.cpu().pin_memory()},
        {"out": out, "lse": out_lse}, args, world, dev, stream)
    peak, peak_kind = measured_peaks()
    top = points[-1]
    line = {
        "metric": "MLA LSE combine GB/s (P=8, H=16, D=512) on 1 GB300",
        "value": top["gbs"] * world, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": top["us_per_call"] / 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "combine_p8_h16_d512", "points": points,
                   "timing": "CUDA graphs of %d calls, replayed" % GRAPH_CALLS,
                   "l2": "no flush: 19 MB per call at T = 128 stays in L2 (an upper bound "
                         "on the HBM rate)"},
        "roofline": {"bound": "hbm", "achieved": top["gbs"], "peak": peak, "unit": "GB/s",
                     "frac": top["gbs"] / peak, "peak_source": peak_kind,
                     "traffic": recorded_traffic(COMBINE_TRAFFIC_FILE),
                     "kernel": "lse_combine_kernel at T = 128 (latency-bound below)"},
        "e2e": e2e_record(top["bytes_per_call"] / 1e9, args, world, e_ms, e_serial_ms, h2d, d2h,
                          "GB/s", "partials and lses in, the merged out and lse back (GB/s "
                          "counts the combine's own bytes)"),
        "gpu_launches": args.steps * len(points),
        "clocks": clock_info,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        import oracle
        pb = c.partials.view(torch.int16).cpu().numpy().view(np.uint16)
        parts64 = oracle.bf16_to_f64(pb)
        lses64 = c.lses.cpu().numpy().astype(np.float64)
        spent, calls = 0.0, 0
        while spent < min(args.cpu_seconds, 3.0):
            a = time.perf_counter()
            oracle.lse_combine(parts64, lses64, oracle.LSE_NATURAL)
            spent += time.perf_counter() - a
            calls += 1
        line["cpu_baseline"] = {"value": top["bytes_per_call"] * calls / spent / 1e9,
                                "unit": "GB/s", "cores": _oracle_threads(), "kind": "oracle",
                                "sample": f"{calls} fp64 combines of the T = 128 case (8 x 128 x "
                                          f"16 rows of 512), {spent:.1f} s; GB/s counts the "
                                          f"kernel's bf16 / fp32 bytes"}
    return line


run_combine = _print_line(measure_combine)


def measure_small(args, world, rank, mla, dev, stream):
    """The small case: B=1, H=16, L=300, bf16, its two round-robin partitions
    and their combine as one mla_decode_dcp call per step (one decode launch
    for both partitions, one merge-and-combine launch).  Latency-bound: 345.6
    KB of KV."""
    case = workloads.config_small(device=dev, seed=args.seed)
    B, H, P = case.batch, case.heads, case.num_parts
    kv_bytes = int(case.seq_lens.sum().item()) * ROW_BYTES[case.kv_dtype]
    ws = mla.make_dcp_workspace(case.q, case.kv_pages, case.block_table, P)
    parts = torch.empty(P, B, 1, H, 512, dtype=torch.bfloat16, device=dev)
    plse = torch.empty(P, B, 1, H, dtype=torch.float32, device=dev)
    out = torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device=dev)
    out_lse = torch.empty(B, 1, H, dtype=torch.float32, device=dev)

    def step(q=case.q, bt=case.block_table, sl=case.seq_lens):
        mla.decode_dcp(q, case.kv_pages, bt, sl, P, case.sm_scale, 0, partials=parts,
                       partial_lses=plse, out=out, out_lse=out_lse, workspace=ws, stream=stream)

    ms, clock_info = timed_steps(step, args.steps, args.warmup, world, dev, stream,
                                 sample_clocks=True)
    assert mla.check_workspace(ws) == 0
    def e2e_op(inp, o):
        mla.decode_dcp(inp["q"], case.kv_pages, inp["bt"], inp["sl"], P, case.sm_scale, 0,
                       partials=parts, partial_lses=plse, out=o["out"], out_lse=o["lse"],
                       workspace=ws, stream=stream)

    e_ms, e_serial_ms, h2d, d2h = e2e_times(
        e2e_op, {"q": case.q.cpu().pin_memory(), "bt": case.block_table.cpu().pin_memory(),
                 "sl": case.seq_lens.cpu().pin_memory()}, {"out": out, "lse": out_lse},
        args, world, dev, stream)
    roof = _hbm_roofline(kv_bytes, ms, args.steps,
                         "mla_decode_dcp with P = 2: one decode launch for both partitions and "
                         "one merge-and-combine launch, timed together per call; latency-bound "
                         "(345.6 KB of KV, L2-resident across steps)")
    roof["traffic"] = recorded_traffic(SMALL_TRAFFIC_FILE)
    line = _line(args, world, ms, B, "tokens/s",
                 {"workload": case.name, "batch": B, "heads": H, "q_len": 1, "num_parts": P,
                  "seq_lens": "300", "page_size": 64, "pool_pages": case.num_pages,
                  "kv_dtype": "bf16", "kv_bytes_per_step": kv_bytes,
                  "l2": "no flush: 345.6 KB of KV stays in L2 (a latency measurement)",
                  "parallelism": "DCP partitions emulated on one GPU"},
                 roof,
                 e2e_record(B, args, world, e_ms, e_serial_ms, h2d, d2h, "tokens/s",
                            "q, block table and lengths in, the merged result and its lse back"),
                 2 * args.steps, clock_info)
    line["us_per_step"] = ms * 1e3 / args.steps
    # the same calls replayed from CUDA graphs: the device time of a step
    # whose eager launches are partly bound by the host
    graph_ms = max_over_ranks(graph_time(lambda st: mla.decode_dcp(
        case.q, case.kv_pages, case.block_table, case.seq_lens, P, case.sm_scale, 0,
        partials=parts, partial_lses=plse, out=out, out_lse=out_lse, workspace=ws, stream=st),
        dev, stream, args.steps), world, dev)
    line["graph"] = {"value": aggregate(graph_ms, args.steps, B, world), "unit": "tokens/s",
                     "us_per_step": graph_ms * 1e3 / args.steps, "calls_per_graph": GRAPH_CALLS,
                     "note": "the same calls replayed from CUDA graphs (device time)"}
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        import oracle
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from casebits import case_bits
        q, kv, bt, lens = case_bits(case)
        spent, calls = 0.0, 0
        while spent < min(args.cpu_seconds, 3.0):
            a = time.perf_counter()
            po, pl = zip(*[oracle.decode_partial(q, kv, bt, lens, r, P, case.sm_scale, 0)
                           for r in range(P)])
            oracle.lse_combine(np.stack(po), np.stack(pl), oracle.LSE_NATURAL)
            spent += time.perf_counter() - a
            calls += 1
        line["cpu_baseline"] = {"value": calls * B / spent, "unit": "tokens/s",
                                "cores": _oracle_threads(), "kind": "oracle",
                                "sample": f"{calls} steps of the whole case (both partitions "
                                          f"and the combine, fp64 numpy), {spent:.1f} s"}
    return line


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=["decode", "small", "dcp8", "fp8", "kv_append", "combine",
                                     "dcp", "mtp"],
                    default="decode",
                    help="decode (the headline; at one GPU its line also carries the small, "
                         "dcp8, fp8 and combine records under \"configs\"), small (B=1, H=16, "
                         "L=300, P=2), dcp8 (the 8-partition DCP workload in one "
                         "mla_decode_dcp call), fp8 (the e4m3-cache workload), combine, dcp "
                         "--parts P, mtp --q-len T, or the KV append of one row per request")
    ap.add_argument("--no-configs", action="store_true",
                    help="decode: the headline record alone, without the other workloads")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--parts", type=int, default=3, help="partitions for --op dcp")
    ap.add_argument("--q-len", type=int, default=2, help="query tokens per request for --op mtp")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="requests per step (default: the workload's own, 64 for decode and "
                         "128 for fp8; smaller only for profiling)")
    ap.add_argument("--pool-pages", type=int, default=40000,
                    help="cache pool size in pages (40000 = the headline workload)")
    ap.add_argument("--n-long", type=int, default=60,
                    help="dcp8: requests of 131072 tokens (60 = the workload; fewer only for profiling)")
    ap.add_argument("--tokens", type=lambda s: [int(x) for x in s.split(",")],
                    default=[1, 8, 16, 32, 64, 128],
                    help="combine: token counts (the last one is the line's value)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.batch is None:
        args.batch = 128 if args.op == "fp8" else 64
    world, rank, local = dist_env()
    if args.op == "kv_append":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the append's CPU oracle is reported as cpu_baseline of --op kv_append"}))
            return
        run_append(args, world, rank, local)
    elif args.op in ("dcp", "mtp"):
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the oracle of these workloads is the decode op's reference arm"}))
            return
        (run_dcp_parts if args.op == "dcp" else run_mtp)(args, world, rank, local)
    elif args.op == "small":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the small case's CPU oracle is reported as cpu_baseline of --op small"}))
            return
        _print_line(measure_small)(args, world, rank, local)
    elif args.op == "combine":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the combine's oracle is pinned in tests/test_oracle_pins.py"}))
            return
        run_combine(args, world, rank, local)
    elif args.op == "fp8":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the fp8 workload's CPU oracle is reported as cpu_baseline of --op fp8"}))
            return
        run_fp8(args, world, rank, local)
    elif args.op == "dcp8":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the DCP workload's CPU oracle is reported as cpu_baseline of --op dcp8"}))
            return
        run_dcp8(args, world, rank, local)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
