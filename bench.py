#!/usr/bin/env python3
"""Benchmark of the DSA decode step on GB300: queries/s at batch 64 x 8K context.

Workload (the BF16 decode configuration): 64 requests with contexts drawn
uniformly from [2048, 8192], one query token each, index_topk 2048, 64 e4m3
indexer heads x 128 with fp32 per-token key scales, 16 MLA heads over a bf16
576-wide latent cache in 64-token pages under random block tables. Inputs are
seeded synthetic tensors (inputs.make_config("decode")).

One step = one pass of the whole hot path through the C ABI (dsa_decode_step:
lightning indexer -> radix top-k -> sparse MLA + split combine), captured once
in a CUDA graph and replayed. Between timed steps a 256 MiB buffer is written
to flush L2 (outside the timed events). Under torchrun every rank runs its own
replica of the workload (data-parallel over requests, no collective in the
path); `value` counts the queries of all ranks over the slowest rank's time.

`e2e` is the same throughput through the C ABI with host buffers: two micro-batches
of the decode workload take turns, each step's inputs copied host->device from
page-locked memory while the other micro-batch's step runs, and each step's O and
LSE written to page-locked host memory by its kernels; every copy is inside the
timed region. `e2e.serial` is one step at a time with its copies on its own
critical path (the latency of a single step with host buffers).

`--impl reference` times the float64 CPU oracle on this host's cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from dsa_sparse_attention_02_gb300 import _lib, inputs, runner  # noqa: E402

METRIC = "DSA decode queries/s at batch 64×ctx 8K; achieved HBM GB/s vs GB300 peak"
WORKLOAD = ("decode: batch 64, context ~U[2048,8192], 1 query token, index_topk 2048, "
            "64 e4m3 indexer heads x 128 (+fp32 per-token key scale), 16 MLA heads, "
            "bf16 576-wide latent KV, 64-token pages, random block tables")
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
E4M3_PER_BF16 = 2.0          # nominal dense e4m3 : bf16 tensor rate on this part (4.5 : 2.25 PFLOP/s)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration step lines")
    ap.add_argument("--only-config", choices=list(inputs.CONFIG_NAMES), default=None,
                    help="run just --warmup + --steps steps of one configuration (no graph, no flush; for "
                         "profiler launch lists) and print its step time")
    ap.add_argument("--hist", action="store_true",
                    help="with --only-config: the full layer through dsa_decode_step_hist")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers

def algorithmic_bytes(wl):
    """Bytes the step must move at least: every index key (128 e4m3 + 4 B scale) of every
    request, and every selected 576-wide bf16 latent row (1152 B)."""
    idx_bytes = int(wl.seq_lens.astype(np.int64).sum()) * (128 + 4)
    _, pos = _positions(wl)
    selected = int(np.minimum(pos + 1, wl.topk).sum())
    return idx_bytes, selected * 576 * 2, selected


def _positions(wl):
    req = np.repeat(np.arange(wl.B), wl.n_q)
    pos = np.concatenate([np.arange(L - n, L) for L, n in zip(wl.seq_lens, wl.n_q)])
    return req, pos


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_bf16_tflops():
    try:
        with open(PEAKS_PATH) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


# The sources that decide what a kernel does and how it is launched: its own file,
# the shared device headers and the host entry points that configure the launch.
KERNEL_SOURCES = {"sparse_mla_kernel": ["sparse_mla.cu"], "indexer_kernel": ["indexer.cu"],
                  "topk_kernel": ["topk.cu"]}
SHARED_SOURCES = ["api.cu", "common.cuh", "kernels.cuh", "ptx.cuh"]


def kernel_source_hash(kernel=None):
    """Hash of every CUDA source (kernel None) or of one kernel's sources."""
    csrc = os.path.join(ROOT, "dsa_sparse_attention_02_gb300", "csrc")
    files = sorted(os.listdir(csrc)) if kernel is None else sorted(KERNEL_SOURCES[kernel] + SHARED_SOURCES)
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def load_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if taken on the kernel's
    current sources."""
    try:
        with open(TRAFFIC_PATH) as f:
            t = json.load(f)
        if t["kernels"][kernel].get("source_hash") != kernel_source_hash(kernel):
            return None
        return t["kernels"][kernel]["dram_bytes_per_launch"]
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- reference arm

def oracle_step_time(wl, nq, reps_min_s):
    """Runs the oracle over `nq` queries of the workload repeatedly for >= reps_min_s;
    returns seconds per query."""
    import oracle
    ts = list(range(min(nq, wl.T)))
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.dsa_step(wl, ts=ts)
        n += len(ts)
        el = time.perf_counter() - t0
        if el >= reps_min_s:
            return el / n


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True,
                             timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def oracle_one_thread(name, budget_s=4.0):
    """Oracle queries/s of configuration `name` with every BLAS pool held to one thread (a
    fresh interpreter, since the pools size themselves when numpy loads)."""
    code = ("import sys, time; sys.path.insert(0, %r)\n"
            "import oracle\n"
            "from dsa_sparse_attention_02_gb300 import inputs\n"
            "wl = inputs.make_config(%r)\n"
            "ts = list(range(wl.T)); n = 0; t0 = time.perf_counter()\n"
            "while time.perf_counter() - t0 < %f:\n"
            "    oracle.dsa_step(wl, ts=ts); n += len(ts)\n"
            "print(n / (time.perf_counter() - t0))\n") % (ROOT, name, budget_s)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, "-c", code], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                             text=True, env=env, timeout=300)
        return float(out.stdout.strip().splitlines()[-1])
    except Exception:
        return None


def cpu_baseline(wl, budget_s=12.0):
    import oracle  # noqa: F401  (the oracle is the baseline)
    sec_per_q = oracle_step_time(wl, wl.T, budget_s)
    return {"value": 1.0 / sec_per_q, "unit": "queries/s", "cores": os.cpu_count(), "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"float64 numpy oracle (indexer, top-k, attention) over all {wl.T} queries of the "
                      f"decode workload, repeated for >= {budget_s:.0f} s; BLAS threads = host cores"}


def run_reference(args, rank, world, budget=90.0):
    """The reference arm: the float64 oracle on this host's cores, rank 0 only, each
    step a sample of the decode workload's queries sized so that the whole run takes
    about `budget` seconds."""
    if rank != 0:
        return
    wl = inputs.make_config("decode")
    per_q = oracle_step_time(wl, 2, min(1.0, budget / 10))     # calibration
    nq = int(max(1, min(wl.T, budget / max(1, args.steps + args.warmup) / per_q)))
    for _ in range(args.warmup):
        oracle_step_time(wl, nq, 0.0)
    import oracle
    ts = list(range(nq))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.dsa_step(wl, ts=ts)
    el = time.perf_counter() - t0
    value = nq * args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded PCG64)",
            "config": {"workload": WORKLOAD, "queries_per_step": nq},
            "cpu_baseline": {"value": value, "unit": "queries/s", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"{nq} of the 64 queries per step (float64 numpy oracle)"},
            "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm

def replica_seed(rank):
    """Seed of rank `rank`'s replica of the decode workload: every rank draws its own
    requests (data-parallel over requests; no rank reads another's data)."""
    return inputs.CONFIG_SEEDS["decode"] + 1000 * rank


def aggregate_over_ranks(units, ms, dist=None, device="cpu"):
    """Whole-job throughput of a data-parallel run: the units that all ranks processed
    divided by the slowest rank's time. `units` and `ms` are this rank's; returns
    (units per second over all ranks, the maximum of `ms` over ranks)."""
    if dist is None:
        return units / (ms / 1000.0), ms
    t_ms = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    t_units = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(t_ms, op=dist.ReduceOp.MAX)
    dist.all_reduce(t_units, op=dist.ReduceOp.SUM)
    ms_max = float(t_ms.item())
    return float(t_units.item()) / (ms_max / 1000.0), ms_max


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.only_config:
        run_one_config(args.only_config, args.warmup, args.steps, dev, hist=args.hist)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    wl = inputs.make_config("decode", seed=replica_seed(rank))
    dw = runner.DeviceWorkload(wl, dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    # warm-up (eager), then capture one step in a CUDA graph
    for _ in range(args.warmup):
        dw.step()
    torch.cuda.synchronize()
    if dw.check_error() != 0:
        raise SystemExit("device error during warm-up")
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        dw.step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        dw.step()
    for _ in range(3):
        flush.fill_(1)
        graph.replay()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            graph.replay()
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if dist:
        dist.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = float(sum(step_ms))
    if dw.check_error() != 0:
        raise SystemExit("device error during the timed steps")
    value, total_ms = aggregate_over_ranks(wl.T * args.steps, total_ms, dist, dev)
    ms_per_step = total_ms / args.steps

    # ---- end to end through the public API with host buffers
    if dist:
        dist.barrier()
    # `value`: two micro-batches taking turns, each step's input copy overlapping the
    # other's step (throughput, like `value`); `serial`: one step at a time, each copy
    # and output write on the step's own critical path (latency of one step)
    serial = measure_e2e(dw, graph, flush, stream, max(20, min(args.steps, 200)))
    serial["value"], serial["ms_per_step"] = aggregate_over_ranks(wl.T, serial["ms_per_step"], dist, dev)
    dw_b = runner.DeviceWorkload(wl, dev)
    pipe = measure_e2e_pipelined(dw, dw_b, stream, max(10, min(args.steps, 100)))
    del dw_b
    torch.cuda.empty_cache()
    pipe_value, pipe_ms = aggregate_over_ranks(wl.T, pipe["ms_per_step"], dist, dev)
    e2e = {"value": pipe_value, "unit": "queries/s", "h2d_bytes_per_step": pipe["h2d_bytes_per_step"],
           "d2h_bytes_per_step": pipe["d2h_bytes_per_step"], "ms_per_step": pipe_ms, "steps": pipe["steps"],
           "scheme": pipe["scheme"], "serial": serial}
    # ---- per-kernel breakdown for the roofline of the dominant kernel
    comp = measure_components(dw, flush, stream, max(20, min(args.steps, 200)))
    # ---- next row beyond the step: the cache update (timed alone; not part of `value`)
    append = measure_cache_append(dw, flush, stream, max(20, min(args.steps, 100)))
    int8_attend = measure_int8_attend(dw, flush, stream, max(20, min(args.steps, 100)))
    fp8_attend = measure_int8_attend(dw, flush, stream, max(20, min(args.steps, 100)), kv_dtype=_lib.DSA_E4M3)
    prep = measure_indexer_prep(dw, flush, stream, max(20, min(args.steps, 100)))
    idx_prefill = measure_indexer_prefill(flush, stream, max(10, min(args.steps, 30)), dev)
    bounded = measure_bounded_step(dw, flush, stream, max(20, min(args.steps, 100)))
    hist_steps = measure_hist_steps(flush, stream, max(10, min(args.steps, 30)), dev)
    configs = {} if args.no_configs else {
        c: measure_config(c, flush, stream, max(10, min(args.steps, 30)), dev) for c in ("tiny", "mtp", "prefill", "longctx")}

    idx_b, lat_b, selected = algorithmic_bytes(wl)
    peak, peak_kind = load_peaks()
    attn_gbs = lat_b / (comp["attend_ms"] / 1000.0) / 1e9
    step_gbs = (idx_b + lat_b) / (ms_per_step / 1000.0) / 1e9
    launches_per_step = 4           # indexer, top-k, sparse MLA split, combine
    line = {
        "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3+bf16", "data": "synthetic (seeded PCG64, decode configuration)",
        "config": {"workload": WORKLOAD, "queries_per_step_per_gpu": wl.T,
                   "l2": "flushed between timed steps (256 MiB write outside the events)",
                   "timed": "CUDA-graph replay of dsa_decode_step, CUDA events per step",
                   "step_ms_p10_p50_p90": [float(np.percentile(step_ms, q)) for q in (10, 50, 90)],
                   "wall_s_timed_region": wall},
        "hbm": {"algorithmic_bytes_per_step": idx_b + lat_b, "index_key_bytes": idx_b,
                "selected_latent_bytes": lat_b, "achieved_gbs": step_gbs,
                "frac_of_peak": step_gbs / peak, "peak_gbs": peak, "peak_kind": peak_kind,
                "frac_of_8tbs_nominal": step_gbs / 8000.0},
        "roofline": {"kernel": "sparse MLA attend (split kernel + combine)", "bound": "hbm",
                     "achieved": attn_gbs, "peak": peak, "unit": "GB/s", "frac": attn_gbs / peak,
                     "peak_kind": peak_kind, "algorithmic_bytes_per_launch": lat_b,
                     "avg_launch_ms": comp["attend_ms"],
                     "traffic": load_traffic("sparse_mla_kernel")},
        "components_ms": comp,
        "next_rows": {"cache_append": append, "int8_latent_attend": int8_attend, "indexer_prep": prep,
                      "bounded_scoring": bounded, "indexer_histogram": hist_steps},
        "e4m3_latent_attend": fp8_attend,
        "configs": configs,
        "indexer_prefill": idx_prefill,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
        line["cpu_baseline"]["tiny_one_thread_queries_per_s"] = oracle_one_thread("tiny")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_one_config(name, warmup, steps, device, hist=False):
    """Eager steps of one configuration, for profilers: warmup + steps calls of the whole
    step (every layer; the full layer through dsa_decode_step_hist with hist), then a
    device-error check and one JSON line with the mean time."""
    wl = inputs.make_config(name)
    dw = runner.DeviceWorkload(wl, device, hist=hist)
    for _ in range(warmup):
        dw.step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        dw.step()
    e1.record()
    torch.cuda.synchronize()
    if dw.check_error() != 0:
        raise SystemExit(f"device error in the {name} steps")
    print(json.dumps({"config": name, "steps": steps, "ms_per_step_eager": e0.elapsed_time(e1) / max(1, steps)}))


def measure_e2e(dw, graph, flush, stream, n):
    """Same metric with per-step host inputs and outputs, all inside the timed events:
    the step's inputs copied host->device from page-locked memory (geometry, indexer q,
    scales and weights in one copy; the MLA query, which only the attention reads, in a
    second copy on a side stream that overlaps the indexer and top-k), then the step
    (dsa_decode_step_wait_q: its attention waits for the MLA query's copy) with O and
    LSE in page-locked host memory, which the attention and combine kernels write
    directly (device->host over the chip-to-chip link, overlapping their own work). The
    input copies are dsa_stage_copy; the whole is one CUDA graph per step."""
    host_in = dw.inputs.detach().cpu().pin_memory()
    host_out = torch.empty(dw.outputs.shape, dtype=dw.outputs.dtype, pin_memory=True)
    h2d = host_in.numel() * host_in.element_size()
    d2h = host_out.numel() * host_out.element_size()
    off = dw.inputs_mla_q_offset
    side = torch.cuda.Stream()
    fork, q_ready = torch.cuda.Event(), torch.cuda.Event()
    # the step's arguments with every layer's O and LSE at the same offsets of host_out
    base, hbase = dw.outputs.data_ptr(), host_out.data_ptr()
    host_args = []
    for a in dw.args:
        ha = _lib.dsa_step_args_t.from_buffer_copy(a)
        ha.out = hbase + (a.out - base)
        ha.lse = hbase + (a.lse - base)
        host_args.append(ha)

    def enqueue():
        cur = torch.cuda.current_stream()
        fork.record(cur)
        side.wait_event(fork)
        with torch.cuda.stream(side):
            _lib.dsa_stage_copy(dw.inputs[off:], host_in[off:], h2d - off)
            q_ready.record(side)
        _lib.dsa_stage_copy(dw.inputs, host_in, off)
        for i, a in enumerate(host_args):
            if i == 0:
                _lib.dsa_decode_step_wait_q(a, q_ready, dw.ws)
            else:
                _lib.dsa_decode_step(a, dw.ws)

    warm = torch.cuda.Stream()
    warm.wait_stream(stream)
    with torch.cuda.stream(warm):
        enqueue()
    stream.wait_stream(warm)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        enqueue()
    ms = []
    for i in range(n):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    avg = sum(ms) / len(ms)
    # the host copy of the outputs is the device step's, bit for bit
    dw.step()
    torch.cuda.synchronize()
    if dw.check_error() != 0 or not torch.equal(host_out, dw.outputs.cpu()):
        raise SystemExit("end-to-end outputs differ from the device step's")
    return {"value": dw.wl.T / (avg / 1000.0), "unit": "queries/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": avg,
            "copies": ("dsa_stage_copy (an SM copy kernel) from page-locked host memory: the indexer's inputs and "
                       "the MLA query (overlapping the indexer and top-k) in; O and LSE written to page-locked host "
                       "memory by the attention and combine kernels")}


def measure_e2e_pipelined(dwa, dwb, stream, n_pairs):
    """The end-to-end step with two independent micro-batches (two decode workloads of
    the same shape, each with its own caches, inputs and page-locked host buffers)
    taking turns: while one micro-batch's step runs, the other's inputs are copied
    host->device (dsa_stage_copy on a side stream); each step waits for its own inputs,
    and its O and LSE reach page-locked host memory from the kernels. Every step's
    input copy and output write is inside the timed region (one event pair around the
    first inputs' copy and n_pairs graph replays of two steps each). No L2 flush: each
    step reads its own micro-batch's 193 MB, and the two alternate, so a step finds
    little of its data in the 126 MB L2."""
    dws = (dwa, dwb)
    host_in = [d.inputs.detach().cpu().pin_memory() for d in dws]
    host_out = [torch.empty(d.outputs.shape, dtype=d.outputs.dtype, pin_memory=True) for d in dws]
    h2d = host_in[0].numel() * host_in[0].element_size()
    d2h = host_out[0].numel() * host_out[0].element_size()
    host_args = []
    for d, ho in zip(dws, host_out):
        base, hbase = d.outputs.data_ptr(), ho.data_ptr()
        lst = []
        for a in d.args:
            ha = _lib.dsa_step_args_t.from_buffer_copy(a)
            ha.out = hbase + (a.out - base)
            ha.lse = hbase + (a.lse - base)
            lst.append(ha)
        host_args.append(lst)
    side = torch.cuda.Stream()
    fork, b_in, a_done, join = (torch.cuda.Event() for _ in range(4))

    def step(x):
        for a in host_args[x]:
            _lib.dsa_decode_step(a, dws[x].ws)

    def pair():
        # A's inputs are on the device (copied at the end of the previous pair); B's are
        # copied while A runs, and A's next ones while B runs
        cur = torch.cuda.current_stream()
        fork.record(cur)
        side.wait_event(fork)
        with torch.cuda.stream(side):
            _lib.dsa_stage_copy(dwb.inputs, host_in[1], h2d)
            b_in.record(side)
        step(0)
        a_done.record(cur)
        cur.wait_event(b_in)
        step(1)
        with torch.cuda.stream(side):
            side.wait_event(a_done)
            _lib.dsa_stage_copy(dwa.inputs, host_in[0], h2d)
            join.record(side)
        cur.wait_event(join)

    warm = torch.cuda.Stream()
    warm.wait_stream(stream)
    with torch.cuda.stream(warm):
        pair()
    stream.wait_stream(warm)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pair()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    _lib.dsa_stage_copy(dwa.inputs, host_in[0], h2d, stream)
    for _ in range(n_pairs):
        g.replay()
    e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / (2 * n_pairs)
    for x, d in enumerate(dws):
        d.step()
        torch.cuda.synchronize()
        if d.check_error() != 0 or not torch.equal(host_out[x], d.outputs.cpu()):
            raise SystemExit("pipelined end-to-end outputs differ from the device step's")
    return {"ms_per_step": ms, "queries_per_s": dwa.wl.T / (ms / 1000.0), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": 2 * n_pairs,
            "scheme": ("two micro-batches of the decode workload taking turns; each step's inputs copied by "
                       "dsa_stage_copy while the other micro-batch's step runs; O and LSE written to page-locked "
                       "host memory by the kernels; one event pair around all steps; no L2 flush (the two "
                       "micro-batches' 193 MB working sets alternate)")}


def measure_indexer_prefill(flush, stream, n, device):
    """The lightning indexer alone on the prefill workload (2048 queries at positions
    14336..16383 of one 16384-token request, 64 e4m3 heads x 128): a contraction, so
    it is read against the e4m3 tensor rate, taken as the measured bf16 rate times
    the nominal e4m3/bf16 ratio. Algorithmic work: 2 x 128 x heads flops per causal
    (query, key) pair."""
    wl = inputs.make_config("prefill")
    dw = runner.DeviceWorkload(wl, device)
    g = dw.geom
    stride = int(-(-wl.max_seq_len // 64) * 64)
    scores = torch.empty(wl.T, stride, dtype=torch.float32, device=device)
    ws = _lib.workspace(_lib.dsa_indexer_scores_workspace_size(g), device)

    def launch():
        _lib.dsa_indexer_scores(g, dw.qk_dtype, dw.q_idx, dw.q_scale, dw.w, dw.idx_k, dw.idx_k_scale,
                                scores, ws)

    for _ in range(3):
        launch()
    torch.cuda.synchronize()
    if _lib.dsa_get_error(ws) != 0:
        raise SystemExit("device error in the prefill indexer")
    total = 0.0
    for i in range(n):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        e1.synchronize()
        total += e0.elapsed_time(e1)
    ms = total / n
    _, pos = _positions(wl)
    flops = 2.0 * 128 * int(dw.w.shape[1]) * float((pos.astype(np.int64) + 1).sum())
    bf16, kind = load_bf16_tflops()
    peak = bf16 * E4M3_PER_BF16
    achieved = flops / (ms / 1000.0) / 1e12
    return {"ms": ms, "queries": wl.T, "context": int(wl.max_seq_len), "algorithmic_tflop": flops / 1e12,
            "achieved_tflops": achieved, "peak_tflops": peak, "frac": achieved / peak,
            "peak_kind": f"{kind} bf16 x {E4M3_PER_BF16:g} (nominal e4m3/bf16 ratio)", "bound": "tensor"}


def measure_components(dw, flush, stream, n):
    """Average device time of each entry point of the step, launched alone with the
    GPU kept busy (a sleep kernel) while the host enqueues, L2 flushed before each."""
    wl = dw.wl
    g = dw.geom
    stride = int(-(-wl.max_seq_len // 64) * 64)
    scores = torch.empty(wl.T, stride, dtype=torch.float32, device=dw.device)
    idx = torch.empty(wl.T, wl.topk, dtype=torch.int32, device=dw.device)
    lay = dw.layers[0]
    ws = _lib.workspace(max(_lib.dsa_topk_workspace_size(g, wl.topk),
                            _lib.dsa_sparse_mla_attend_workspace_size(g, lay.q.shape[1], wl.topk)),
                        dw.device)
    acc = {"indexer_ms": 0.0, "topk_ms": 0.0, "attend_ms": 0.0}
    for i in range(n):
        flush.fill_(i & 0xFF)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        torch.cuda._sleep(400_000)
        ev[0].record(stream)
        _lib.dsa_indexer_scores(g, dw.qk_dtype, dw.q_idx, dw.q_scale, dw.w, dw.idx_k, dw.idx_k_scale,
                                scores, ws)
        ev[1].record(stream)
        _lib.dsa_topk(g, scores, wl.topk, idx, ws)
        ev[2].record(stream)
        flush.fill_((i + 1) & 0xFF)
        torch.cuda._sleep(400_000)
        ev3 = torch.cuda.Event(enable_timing=True)
        ev3.record(stream)
        _lib.dsa_sparse_mla_attend(g, lay.kv_dtype, lay.q, lay.kv, idx, wl.topk, wl.sm_scale, lay.out,
                                   lay.lse, ws)
        ev[3].record(stream)
        ev[3].synchronize()
        acc["indexer_ms"] += ev[0].elapsed_time(ev[1])
        acc["topk_ms"] += ev[1].elapsed_time(ev[2])
        acc["attend_ms"] += ev3.elapsed_time(ev[3])
    return {k: v / n for k, v in acc.items()}


def measure_cache_append(dw, flush, stream, n):
    """Device time of dsa_cache_append (the cache-update row), launched alone with the
    GPU kept busy while the host enqueues, L2 flushed before each: (a) the decode
    batch's 64 new tokens into its bf16 latent and e4m3 index caches, (b) a 2048-token
    prefill chunk into e4m3 latent and index caches. Algorithmic bytes: the new rows
    read (1152 + 256 B per token) and the cache rows written."""
    wl = dw.wl
    dev = dw.device
    rng = np.random.default_rng(99)

    def bits(shape):
        x = rng.standard_normal(shape).astype(np.float32)
        return torch.from_numpy((x.view(np.uint32) >> 16).astype(np.uint16).view(np.int16)).to(dev)

    ws = _lib.workspace(256, dev)
    cases = {}
    lay = dw.layers[0]
    cases["decode_64_tokens_bf16_latent"] = (
        dw.geom, lay.kv_dtype, bits((wl.T, 576)), lay.kv, bits((wl.T, 128)), wl.T * (1152 + 256 + 1152 + 132))
    L, m = 4096, 2048
    P = L // 64
    seq = torch.tensor([L], dtype=torch.int32, device=dev)
    cu = torch.tensor([0, m], dtype=torch.int32, device=dev)
    bt = torch.from_numpy(rng.permutation(P).astype(np.int32).reshape(1, P)).to(dev)
    g2 = _lib.Geometry(seq, cu, bt, num_pages=P, max_seq_len=L, T=m)
    kv2 = torch.zeros(P, 64 * 656, dtype=torch.uint8, device=dev)
    ik2 = torch.zeros(P, 64, 128, dtype=torch.uint8, device=dev)
    is2 = torch.zeros(P, 64, dtype=torch.float32, device=dev)
    cases["prefill_2048_tokens_e4m3_latent"] = (g2, _lib.DSA_E4M3, bits((m, 576)), kv2, bits((m, 128)),
                                                m * (1152 + 256 + 656 + 132))
    out = {}
    for name, (g, kvd, kv_new, kv, k_new, nbytes) in cases.items():
        ik, isc = (dw.idx_k, dw.idx_k_scale) if g is dw.geom else (ik2, is2)
        tot = 0.0
        for i in range(n):
            flush.fill_(i & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(200_000)
            a.record(stream)
            _lib.dsa_cache_append(g, kvd, kv_new, kv, _lib.DSA_E4M3, k_new, ik, isc, ws)
            b.record(stream)
            b.synchronize()
            tot += a.elapsed_time(b)
        ms = tot / n
        out[name] = {"ms": ms, "algorithmic_bytes": nbytes, "achieved_gbs": nbytes / (ms / 1000.0) / 1e9}
    return out


def measure_indexer_prep(dw, flush, stream, n):
    """Device time of dsa_indexer_prepare (the indexer-preparation row), launched alone
    with the GPU kept busy while the host enqueues, L2 flushed before each: (a) the
    decode batch's 64 tokens x 64 indexer heads, keys into its e4m3 index cache, (b) a
    2048-token prefill chunk. Algorithmic bytes: bf16 q and k read (256 B per head and
    per key), e4m3 codes and fp32 scales written (132 B each), the RoPE table rows of
    the tokens' positions read (256 B per token)."""
    import types
    wl = dw.wl
    dev = dw.device
    ws = _lib.workspace(256, dev)
    hi = int(wl.q_idx.shape[1])

    def dev_bits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

    cases = {}
    pi = inputs.make_prep_inputs(wl, hi=hi, rope_dim=64, seed=7)
    cases["decode_64_tokens_64_heads"] = (dw.geom, pi, dw.idx_k, dw.idx_k_scale, wl.T)
    L, m = 4096, 2048
    P = L // 64
    rng = np.random.default_rng(98)
    seq = torch.tensor([L], dtype=torch.int32, device=dev)
    cu = torch.tensor([0, m], dtype=torch.int32, device=dev)
    bt = torch.from_numpy(rng.permutation(P).astype(np.int32).reshape(1, P)).to(dev)
    g2 = _lib.Geometry(seq, cu, bt, num_pages=P, max_seq_len=L, T=m)
    pi2 = inputs.make_prep_inputs(types.SimpleNamespace(n_q=np.array([m]), max_seq_len=L), hi=hi, rope_dim=64, seed=8)
    cases["prefill_2048_tokens_64_heads"] = (g2, pi2, torch.zeros(P, 64, 128, dtype=torch.uint8, device=dev),
                                             torch.zeros(P, 64, dtype=torch.float32, device=dev), m)
    out = {}
    for name, (g, p, kc, ks, T) in cases.items():
        q_in, k_in = dev_bits(p.q_in), dev_bits(p.k_in)
        cos, sin = torch.from_numpy(p.rope_cos).to(dev), torch.from_numpy(p.rope_sin).to(dev)
        gm, bt_ = torch.from_numpy(p.ln_gamma).to(dev), torch.from_numpy(p.ln_beta).to(dev)
        q_out = torch.empty(T, hi, 128, dtype=torch.uint8, device=dev)
        q_scale = torch.empty(T, hi, dtype=torch.float32, device=dev)
        nbytes = T * (hi * (256 + 132) + 256 + 132 + 256)
        tot = 0.0
        for i in range(n):
            flush.fill_(i & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(200_000)
            a.record(stream)
            _lib.dsa_indexer_prepare(g, hi, p.rope_dim, q_in, k_in, cos, sin, gm, bt_, p.ln_eps, q_out, q_scale,
                                     kc, ks, ws)
            b.record(stream)
            b.synchronize()
            tot += a.elapsed_time(b)
        ms = tot / n
        out[name] = {"ms": ms, "algorithmic_bytes": nbytes, "achieved_gbs": nbytes / (ms / 1000.0) / 1e9}
    return out


def measure_bounded_step(dw, flush, stream, n, rows=16):
    """The decode step through dsa_decode_step_bounded with a score budget of `rows`
    queries (64 / rows ranges, each scored and reduced before the next), captured in
    a CUDA graph and replayed like the main step; its score workspace against the
    unbounded step's."""
    wl = dw.wl
    dev = dw.device
    row_bytes = (-(-wl.max_seq_len // 64) * 64) * 4
    budget = rows * row_bytes
    a0 = dw.args[0]
    ws = _lib.workspace(max([_lib.dsa_decode_step_bounded_workspace_size(a0, budget)] +
                            [_lib.dsa_decode_step_workspace_size(a) for a in dw.args[1:]]), dev)

    def enqueue():
        for a in dw.args:
            _lib.dsa_decode_step_bounded(a, budget, ws)

    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        enqueue()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        enqueue()
    tot = 0.0
    for i in range(n):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(200_000)
        a.record(stream)
        g.replay()
        b.record(stream)
        b.synchronize()
        tot += a.elapsed_time(b)
    return {"budget_rows": rows, "ranges": -(-wl.T // rows), "ms_per_step": tot / n,
            "score_workspace_bytes": budget, "unbounded_score_workspace_bytes": wl.T * row_bytes}


CONFIG_LINES = {
    "tiny": "batch 2, contexts 200 and 256, 1 query, index_topk 64, 4 bf16 indexer heads, bf16 latent",
    "mtp": ("FP8-latent MTP verify: batch 32, context ~U[4096,16384], 4 causal queries per request, "
            "index_topk 2048, 64 e4m3 indexer heads, e4m3 latent records, two layers (IndexShare)"),
    "prefill": ("chunked prefill: 1 request, 16384 cached tokens, 2048 queries at positions 14336..16383, "
                "index_topk 2048, 64 e4m3 indexer heads, bf16 latent"),
    "longctx": ("long-context decode: batch 8, context 131072, 1 query, index_topk 2048, 64 e4m3 indexer "
                "heads (1% of key rows duplicated: exact score ties), bf16 latent"),
}


def latent_row_bytes(kv_dtype):
    return 576 * 2 if kv_dtype == "bf16" else 656


def measure_config(name, flush, stream, n, device, oracle_budget_s=3.0):
    """One whole step (every layer, through dsa_decode_step, captured in a CUDA graph) of
    configuration `name`, timed like the headline step; its algorithmic bytes (index keys,
    and the selected latent rows per query, and their union per request) and, for the
    prefill, flops; the oracle's time per query on a sample of the same workload."""
    import oracle
    wl = inputs.make_config(name)
    dw = runner.DeviceWorkload(wl, device)
    for _ in range(3):
        dw.step()
    torch.cuda.synchronize()
    if dw.check_error() != 0:
        raise SystemExit(f"device error in the {name} step")
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        dw.step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        dw.step()
    ms = []
    for i in range(n):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    step_ms = statistics.median(ms)
    req, pos = _positions(wl)
    idx = dw.idx.cpu().numpy()
    idx_key_bytes = int(wl.seq_lens.astype(np.int64).sum()) * (128 + 4 if wl.qk_dtype == "e4m3" else 256)
    per_token_rows = int((idx >= 0).sum())
    union_rows = sum(len(np.unique(idx[req == b][idx[req == b] >= 0])) for b in range(wl.B))
    lat_tok = sum(per_token_rows * latent_row_bytes(L.kv_dtype) for L in wl.layers)
    lat_union = sum(union_rows * latent_row_bytes(L.kv_dtype) for L in wl.layers)
    peak, kind = load_peaks()
    out = {"workload": CONFIG_LINES[name], "queries": wl.T, "layers": len(wl.layers), "ms": step_ms,
           "queries_per_s": wl.T / (step_ms / 1000.0),
           "index_key_bytes": idx_key_bytes, "selected_latent_bytes_per_token": lat_tok,
           "selected_latent_bytes_union_per_request": lat_union,
           "algorithmic_bytes": idx_key_bytes + lat_tok,
           "achieved_gbs": (idx_key_bytes + lat_tok) / (step_ms / 1000.0) / 1e9,
           "frac_of_peak": (idx_key_bytes + lat_tok) / (step_ms / 1000.0) / 1e9 / peak,
           "achieved_gbs_union_bytes": (idx_key_bytes + lat_union) / (step_ms / 1000.0) / 1e9,
           "peak_gbs": peak, "peak_kind": kind}
    if name == "prefill":
        idx_flops = 2.0 * 128 * wl.Hi * float((pos.astype(np.int64) + 1).sum())
        att_flops = 2.0 * (576 + 512) * wl.heads * float(np.minimum(pos + 1, wl.topk).sum()) * len(wl.layers)
        bf16, bkind = load_bf16_tflops()
        out.update({"indexer_tflop": idx_flops / 1e12, "attention_tflop": att_flops / 1e12,
                    "achieved_tflops": (idx_flops + att_flops) / (step_ms / 1000.0) / 1e12,
                    "tensor_peak_tflops_e4m3": bf16 * E4M3_PER_BF16, "tensor_peak_kind": bkind,
                    "bound": "tensor (indexer) + L2 gather (attention)"})
    # the oracle on a bounded sample of the same workload
    nq = 1 if name in ("longctx", "prefill") else min(wl.T, 4)
    sec = oracle_step_time(wl, nq, oracle_budget_s)
    out["oracle"] = {"queries_per_s": 1.0 / sec, "sample_queries": nq, "cores": os.cpu_count(),
                     "sample": f"the first {nq} queries of the workload, repeated for >= {oracle_budget_s:.0f} s"}
    del dw
    torch.cuda.empty_cache()
    return out


def measure_hist_steps(flush, stream, n, device, names=("decode", "prefill")):
    """The step through dsa_decode_step_hist (the top-k's first radix digit counted by
    the indexer) on the decode and chunked-prefill workloads, captured and replayed like
    the headline step (median of n), with the number of segments whose histogram the
    top-k rejected (0: every selection used the indexer's counts)."""
    out = {}
    for name in names:
        wl = inputs.make_config(name)
        dw = runner.DeviceWorkload(wl, device, hist=True)
        for _ in range(3):
            dw.step()
        torch.cuda.synchronize()
        if dw.check_error() != 0:
            raise SystemExit(f"device error in the {name} step with histograms")
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            dw.step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            dw.step()
        ms = []
        for i in range(n):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
        out[name] = {"ms": statistics.median(ms), "rejected_segments": int(dw.ws[:8].view(torch.int32)[1])}
        del dw, g
        torch.cuda.empty_cache()
    out["entry_point"] = "dsa_decode_step_hist (opt-in; dsa_decode_step, timed above, counts the digit in the top-k)"
    return out


def measure_int8_attend(dw, flush, stream, n, kv_dtype=None):
    """Device time of dsa_sparse_mla_attend over an int8 (next row f4) or, with
    kv_dtype=DSA_E4M3, an e4m3 latent record cache: the decode workload's bf16 latent
    cache re-encoded as records by dsa_cache_append (every row, as one request with an
    identity block table), then attended with the step's own selection. Algorithmic
    bytes: the selected 656-byte records."""
    kv_dtype = _lib.DSA_I8 if kv_dtype is None else kv_dtype
    wl = dw.wl
    dev = dw.device
    lay = dw.layers[0]
    P = wl.num_pages
    rows = P * 64
    seq = torch.tensor([rows], dtype=torch.int32, device=dev)
    cu = torch.tensor([0, rows], dtype=torch.int32, device=dev)
    bt = torch.arange(P, dtype=torch.int32, device=dev).view(1, P)
    g_all = _lib.Geometry(seq, cu, bt, num_pages=P, max_seq_len=rows, T=rows)
    kv8 = torch.empty(P, 64 * 656, dtype=torch.uint8, device=dev)
    ws = _lib.workspace(max(256, _lib.dsa_sparse_mla_attend_workspace_size(dw.geom, lay.q.shape[1], wl.topk)), dev)
    _lib.dsa_cache_append(g_all, kv_dtype, lay.kv.view(rows, 576), kv8, _lib.DSA_E4M3, None, None, None, ws)
    dw.step()
    torch.cuda.synchronize()
    _, pos = _positions(wl)
    selected = int(np.minimum(pos + 1, wl.topk).sum())
    out = torch.empty_like(lay.out)
    lse = torch.empty_like(lay.lse)
    tot = 0.0
    for i in range(n):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(400_000)
        a.record(stream)
        _lib.dsa_sparse_mla_attend(dw.geom, kv_dtype, lay.q, kv8, dw.idx, wl.topk, wl.sm_scale, out, lse, ws)
        b.record(stream)
        b.synchronize()
        tot += a.elapsed_time(b)
    ms = tot / n
    nbytes = selected * 656
    return {"ms": ms, "algorithmic_bytes": nbytes, "achieved_gbs": nbytes / (ms / 1000.0) / 1e9,
            "cache": ("the decode cache re-encoded as int8 records (per-128 amax/127 scales, bf16 RoPE)"
                      if kv_dtype == _lib.DSA_I8 else
                      "the decode cache re-encoded as e4m3 records (per-128 amax/448 scales, bf16 RoPE)")}


if __name__ == "__main__":
    main()
