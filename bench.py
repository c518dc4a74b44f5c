"""Throughput of the mbarrier/TMA tile pipeline on one GB300 (or N, one per rank).

One step = one pass of the whole hot path over one batch of input:
  * tile_copy   fp16 16384 x 16384 (512 MiB), 128 x 64 tiles, seeded uniform[-1, 1)
  * tile_rowsum bf16 8192 x 65536 (1 GiB), 64 x 256 tiles, seeded normal(0, 1)
Metric: achieved HBM GB/s = algorithmic bytes (copy: read + write of the
matrix; row sum: read of the matrix + write of the fp32 sums) / device time,
1 GB = 1e9 B.  Inputs are far larger than the 129 MB L2, so no flush is needed
between steps.

Default (--impl mbtile) prints one JSON line on rank 0.  --impl reference times
the CPU oracle (the plain restatement used by the tests) on a bounded sample of
the same workload.  --sweep prints one extra line per stage / warp / CTA point.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

COPY = dict(name="copy", dtype="f16", M=16384, N=16384, tile_m=128, tile_n=64,
            dist="uniform", seed=1003)
ROWSUM = dict(name="rowsum", dtype="bf16", M=8192, N=65536, tile_m=64, tile_n=256,
              dist="normal", seed=1004)
ESIZE = {"f16": 2, "bf16": 2, "f32": 4}
# The ragged fp32 12289 x 8191 and fp16 24577 x 16383 workloads, stored with a 16-byte row
# pitch (--only --config).
RAGGED = {
    "5a": dict(name="5a", dtype="f32", M=12289, N=8191, tile_m=128, tile_n=32, dist="uniform",
               seed=1005),
    "5b": dict(name="5b", dtype="f16", M=24577, N=16383, tile_m=128, tile_n=64,
               dist="uniform", seed=1006),
}
FALLBACK_HBM_GBS = 6800.0
MODE_NAME = {0: "default", 1: "bulk tensor stores", 2: "LSU stores"}
GRAPH_CHUNK = 50   # steps per captured CUDA graph

# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture
# of each kernel on the full-size workload, keyed by the SHA-256 of the kernel
# code it was taken on (kernel_source_sha); reported only while that code is
# unchanged.
NCU_TRAFFIC: dict = {
    "copy": {"src_sha": "012614f4d8ee5b8b", "bytes_per_launch": 536938240 + 485307136},
    "rowsum": {"src_sha": "012614f4d8ee5b8b", "bytes_per_launch": 1073840384 + 2676736},
}

def copy_bytes(c=COPY):
    return 2 * c["M"] * c["N"] * ESIZE[c["dtype"]]


def rowsum_bytes(c=ROWSUM):
    return c["M"] * c["N"] * ESIZE[c["dtype"]] + 4 * c["M"]


def kernel_source_sha() -> str:
    """Hash of the code (comments and blank lines left out, so that editing a
    comment keeps the key) of the files that hold the copy and row-sum
    kernels (the other kernels live in their own headers)."""
    h = hashlib.sha256()
    for f in ("mbtile_kernels.cu", "internal.h"):
        with open(os.path.join(ROOT, "mbarrier_async_tile_gb300", "csrc", f)) as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples: list[tuple[float, list[str]]] = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside and self.samples:
            # timed region shorter than the sampling period: nearest samples
            near = sorted(self.samples, key=lambda ts: abs(ts[0] - (t0 + t1) / 2))[:3]
            inside, window = [s for _, s in near], "nearest"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        mx = [num(s[2]) for s in inside if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4)
                          if len(s) > 5 + i and s[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "window": window}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def make_inputs(device):
    import synthetic

    x3 = synthetic.make_matrix(COPY["M"], COPY["N"], COPY["dtype"], COPY["dist"],
                               COPY["seed"], draw_on=str(device))
    d3 = torch.empty_like(x3)
    x4 = synthetic.make_matrix(ROWSUM["M"], ROWSUM["N"], ROWSUM["dtype"], ROWSUM["dist"],
                               ROWSUM["seed"], draw_on=str(device))
    o4 = torch.empty(ROWSUM["M"], dtype=torch.float32, device=device)
    return x3, d3, x4, o4


def host_cores() -> int:
    return len(os.sched_getaffinity(0))


def oracle_blocks_parallel(jobs, pool) -> float:
    """Run independent oracle calls (closures over disjoint row blocks) on a
    thread pool; the oracle's C loops release the GIL.  Returns the
    wall-clock seconds."""
    t = time.perf_counter()
    for f in [pool.submit(j) for j in jobs]:
        f.result()
    return time.perf_counter() - t


def host_memcpy_gbs(nbytes: int = 256 << 20) -> float:
    """Context: a plain single-thread memcpy of nbytes on the host, read +
    write bytes over the best of 3."""
    import ctypes

    a = torch.ones(nbytes, dtype=torch.uint8)
    b = torch.empty_like(a)
    best = float("inf")
    for _ in range(3):
        t = time.perf_counter()
        ctypes.memmove(b.data_ptr(), a.data_ptr(), nbytes)
        best = min(best, time.perf_counter() - t)
    return 2 * nbytes / best / 1e9


def cpu_baseline(x3, d3, x4, o4, budget_s: float = 12.0) -> dict:
    """Time the CPU oracle, as it stands, on a bounded sample of the same
    workload: row blocks of both matrices in proportion to their bytes, first
    on one host core (about budget_s / 2 of CPU time), then on all host
    cores (disjoint row blocks on as many threads, about budget_s / 2 of wall
    time).  The GPU's outputs on every sampled row are checked against the
    oracle's."""
    import oracle

    oracle.build()
    cores = host_cores()
    blk3, blk4 = 256, ROWSUM["tile_m"]
    state = {}
    checks = {"mismatches": 0, "worst": 0.0}

    def next_block():
        """(job, check, bytes) of the next row block, or None when both
        matrices are exhausted."""
        r3, r4 = state["r3"], state["r4"]
        take_copy = r3 < COPY["M"] and (state["b3"] <= state["b4"] or r4 >= ROWSUM["M"])
        if take_copy:
            src = x3[r3:r3 + blk3].cpu()
            want = torch.empty_like(src)
            got = d3[r3:r3 + blk3].cpu()
            state["r3"] += blk3
            nbytes = 2 * src.numel() * src.element_size()
            state["b3"] += nbytes

            def check():
                checks["mismatches"] += int((got.view(torch.int16) != want.view(torch.int16)).sum())
            return (lambda: oracle.copy(src, want)), check, nbytes
        if r4 < ROWSUM["M"]:
            src = x4[r4:r4 + blk4].cpu()
            got = o4[r4:r4 + blk4].cpu().double()
            res = {}
            state["r4"] += blk4
            nbytes = src.numel() * src.element_size() + 4 * src.shape[0]
            state["b4"] += nbytes

            def job():
                res["ref"], res["sq"] = oracle.rowsum(src, with_sumsq=True)

            def check():
                err = ((got - res["ref"]).abs() / torch.maximum(res["ref"].abs(),
                                                                res["sq"].sqrt())).max().item()
                checks["worst"] = max(checks["worst"], err)
            return job, check, nbytes
        return None

    # one core, from the first row of both matrices
    state.update(r3=0, r4=0, b3=0, b4=0)
    t1 = 0.0
    bytes1 = 0
    while t1 < budget_s / 2:
        blk = next_block()
        if blk is None:
            break
        job, check, nbytes = blk
        t = time.perf_counter()
        job()
        t1 += time.perf_counter() - t
        check()
        bytes1 += nbytes
    rows1 = (state["r3"], state["r4"])
    # all cores, again from the first row: rounds of `cores` blocks
    state.update(r3=0, r4=0, b3=0, b4=0)
    tn = 0.0
    bytesn = 0
    with concurrent.futures.ThreadPoolExecutor(max_workers=cores) as pool:
        while tn < budget_s / 2:
            blocks = [b for b in (next_block() for _ in range(cores)) if b is not None]
            if not blocks:
                break
            tn += oracle_blocks_parallel([b[0] for b in blocks], pool)
            for _, check, nbytes in blocks:
                check()
                bytesn += nbytes
    one = bytes1 / t1 / 1e9 if t1 > 0 else None
    alln = bytesn / tn / 1e9 if tn > 0 else None
    return {
        "value": round(alln if alln is not None else one, 4), "unit": "GB/s",
        "cores": cores if alln is not None else 1, "kind": "oracle",
        "sample": (f"row blocks of {blk3} (copy) / {blk4} (row sum) rows, in proportion "
                   f"to their bytes: on 1 core {rows1[0]} of {COPY['M']} copy rows and "
                   f"{rows1[1]} of {ROWSUM['M']} row-sum rows ({bytes1 / 1e9:.3f} GB "
                   f"algorithmic, {t1:.2f} s); on {cores} cores, one block per thread, "
                   f"{state['r3']} and {state['r4']} rows ({bytesn / 1e9:.3f} GB, "
                   f"{tn:.2f} s)"),
        "single_core": {"value": round(one, 4) if one else None, "unit": "GB/s", "cores": 1},
        "host_memcpy_gbs_1_thread": round(host_memcpy_gbs(), 2),
        "parity_on_sample": {"copy_mismatched_elements": checks["mismatches"],
                             "rowsum_worst_scaled_error": checks["worst"]},
    }


def bench_gpu(args, rank, world):
    import mbarrier_async_tile_gb300 as mbt

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    mbt.tile_device_info()  # loads the library, fails loudly if it is missing
    x3, d3, x4, o4 = make_inputs(dev)
    main = torch.cuda.current_stream()
    side = (torch.cuda.Stream(), torch.cuda.Stream())

    def run_pass(two_streams: bool, record: bool):
        """Warm up, then time args.steps steps.  One stream: copy then row sum,
        per-kernel events on it.  Two streams: each operation on its own
        stream (independent calls, so one kernel's tail overlaps the next
        one's start).  Returns (total ms, mean copy ms, mean rowsum ms)."""
        s_copy, s_rowsum = side if two_streams else (main, main)

        def step(ev=None):
            if ev is not None:
                ev[0].record(s_copy)
            mbt.tile_copy(x3, d3, COPY["tile_m"], COPY["tile_n"], args.copy_stages,
                          store_mode=args.store_mode, stream=s_copy)
            if ev is not None:
                ev[1].record(s_copy)
                ev[2].record(s_rowsum)
            mbt.tile_rowsum(x4, o4, ROWSUM["tile_m"], ROWSUM["tile_n"], args.rowsum_stages,
                            stream=s_rowsum)
            if ev is not None:
                ev[3].record(s_rowsum)

        def fork():
            s_copy.wait_stream(main)
            s_rowsum.wait_stream(main)

        def join():
            main.wait_stream(s_copy)
            main.wait_stream(s_rowsum)

        fork()
        for _ in range(args.warmup):
            step()
        join()
        code, info = mbt.tile_status(main)
        if code != 0:
            raise RuntimeError(f"pipeline status {code} {info}")
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
               for _ in range(args.steps)] if record else [None] * args.steps
        barrier(world)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(main)
        fork()
        for k in range(args.steps):
            step(evs[k])
        join()
        end.record(main)
        torch.cuda.synchronize()
        barrier(world)
        code, info = mbt.tile_status(main)
        if code != 0:
            raise RuntimeError(f"pipeline status {code} {info}")
        ms_c = ms_r = None
        if record:
            ms_c = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
            ms_r = sum(e[2].elapsed_time(e[3]) for e in evs) / args.steps
        return start.elapsed_time(end), ms_c, ms_r

    def run_kernel_pass(which: str):
        """Time args.steps back-to-back launches of one kernel on the main
        stream, twice: with one event pair around the whole series (the mean
        launch duration, gaps between launches included: the roofline's
        figure) and with an event pair around each launch (each launch then
        also pays its own start-up, which back-to-back launches overlap with
        the previous launch's tail).  Returns (ms back to back, ms per event
        pair, (best, median) of the event pairs).  In the one-stream pass a
        row sum starts while L2 still writes back the dirty lines the copy
        before it left (up to ~126 MB), so that pass charges part of the
        copy's writes to the row sum; here every launch follows one of its
        own kind (steady state)."""
        def launch():
            if which == "copy":
                mbt.tile_copy(x3, d3, COPY["tile_m"], COPY["tile_n"], args.copy_stages,
                              store_mode=args.store_mode, stream=main)
            else:
                mbt.tile_rowsum(x4, o4, ROWSUM["tile_m"], ROWSUM["tile_n"], args.rowsum_stages,
                                stream=main)

        def check():
            code, info = mbt.tile_status(main)
            if code != 0:
                raise RuntimeError(f"pipeline status {code} {info}")

        for _ in range(args.warmup):
            launch()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        start.record(main)
        for _ in range(args.steps):
            launch()
        end.record(main)
        torch.cuda.synchronize()
        barrier(world)
        check()
        ms_b2b = reduce_max(start.elapsed_time(end) / args.steps, world)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        for a, b in evs:
            a.record(main)
            launch()
            b.record(main)
        torch.cuda.synchronize()
        barrier(world)
        check()
        per = [a.elapsed_time(b) for a, b in evs]
        ms_pairs = reduce_max(sum(per) / len(per), world)
        pairs_stats = (reduce_max(min(per), world), reduce_max(statistics.median(per), world))
        return ms_b2b, ms_pairs, pairs_stats

    def copy_on(stream):
        mbt.tile_copy(x3, d3, COPY["tile_m"], COPY["tile_n"], args.copy_stages,
                      store_mode=args.store_mode, stream=stream)

    def rowsum_on(stream):
        mbt.tile_rowsum(x4, o4, ROWSUM["tile_m"], ROWSUM["tile_n"], args.rowsum_stages,
                        stream=stream)

    def graphed(chunk_body, steps: int):
        """CUDA graphs that together replay `steps` steps: chunk_body(origin,
        n) launches n steps from the capturing stream `origin` (forking to
        and joining back from side streams itself).  Returns a function that
        replays them on the current stream."""
        full, rem = divmod(steps, GRAPH_CHUNK)
        graphs = []
        cap = torch.cuda.Stream()
        cap.wait_stream(main)
        chunk_body(cap, 1)   # outside the capture: the library's workspace for cap
        torch.cuda.synchronize()
        for n, times in ((GRAPH_CHUNK, full), (rem, 1)):
            if n == 0 or times == 0:
                continue
            g = torch.cuda.CUDAGraph()
            cap.wait_stream(main)
            with torch.cuda.graph(g, stream=cap):
                chunk_body(cap, n)
            graphs.append((g, times))

        def replay():
            for g, times in graphs:
                for _ in range(times):
                    g.replay()
        return replay

    def time_graphed(replay) -> float:
        """Mean ms per step of the replayed graphs (one event pair around all
        of them), after one untimed replay of the whole set."""
        replay()
        torch.cuda.synchronize()
        code, info = mbt.tile_status(main)
        if code != 0:
            raise RuntimeError(f"pipeline status {code} {info}")
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        start.record(main)
        replay()
        end.record(main)
        torch.cuda.synchronize()
        barrier(world)
        code, info = mbt.tile_status(main)
        if code != 0:
            raise RuntimeError(f"pipeline status {code} {info}")
        return reduce_max(start.elapsed_time(end), world)

    def kernel_chunk(which):
        def body(origin, n):
            for _ in range(n):
                (copy_on if which == "copy" else rowsum_on)(origin)
        return body

    def step_chunk(two_streams):
        def body(origin, n):
            s_copy, s_rowsum = side if two_streams else (origin, origin)
            s_copy.wait_stream(origin)
            s_rowsum.wait_stream(origin)
            for _ in range(n):
                copy_on(s_copy)
                rowsum_on(s_rowsum)
            origin.wait_stream(s_copy)
            origin.wait_stream(s_rowsum)
        return body

    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    t0 = time.time()
    # per-kernel passes: steady-state launch durations for the roofline,
    # launched one by one from the host (back to back, and with an event pair
    # around each launch), then replayed from CUDA graphs
    ms_copy_stream, ms_copy_pairs, copy_pairs_stats = run_kernel_pass("copy")
    ms_rowsum_stream, ms_rowsum_pairs, rowsum_pairs_stats = run_kernel_pass("rowsum")
    ms_copy_graph = time_graphed(graphed(kernel_chunk("copy"), args.steps)) / args.steps
    ms_rowsum_graph = time_graphed(graphed(kernel_chunk("rowsum"), args.steps)) / args.steps
    # sequential passes: both operations on one stream, then again with
    # per-kernel events (which add gaps, so they do not time value_one_stream)
    ms_seq, _, _ = run_pass(False, False)
    _, ms_copy_seq, ms_rowsum_seq = run_pass(False, True)
    # the headline pass: the steps launched from the host, then the same
    # steps replayed from CUDA graphs
    if args.streams == 2:
        ms_total_stream, _, _ = run_pass(True, False)
    else:
        ms_total_stream = ms_seq
    ms_total_graph = time_graphed(graphed(step_chunk(args.streams == 2), args.steps))
    graph = args.launch == "graph"
    ms_copy = ms_copy_graph if graph else ms_copy_stream
    ms_rowsum = ms_rowsum_graph if graph else ms_rowsum_stream
    ms_total = ms_total_graph if graph else ms_total_stream
    t1 = time.time()
    # every workload configuration and the stage sweep, each point
    # in its own clock window
    sweep = flat = None
    read_ref = None if args.no_read_ref else read_reference(dev, clocks)
    # the same at the row-sum workload's size (the same per-launch ramp and tail)
    read_same = (None if args.no_read_ref else
                 read_reference(dev, clocks, nbytes=ROWSUM["M"] * ROWSUM["N"] * ESIZE[ROWSUM["dtype"]]))
    if not args.no_sweep:
        theo = mbt.tile_device_info()["hbm_gbs_theoretical"]
        sweep = config_sweep(dev, clocks, measured_peak()[0], theo,
                             read_peak=read_ref["gbs"] if read_ref else None,
                             read_at_size=not args.no_read_ref)
        flat = flat_points(dev, clocks, measured_peak()[0],
                           read_peak=read_ref["gbs"] if read_ref else None)
    time.sleep(0.15)
    clocks.stop()
    step_bytes = copy_bytes() + rowsum_bytes()
    value_one_stream = aggregate_gbs(step_bytes, args.steps, world, reduce_max(ms_seq, world))
    ms_max = reduce_max(ms_total, world)
    value = aggregate_gbs(step_bytes, args.steps, world, ms_max)
    value_other_launch = aggregate_gbs(step_bytes, args.steps, world, reduce_max(
        ms_total_stream if graph else ms_total_graph, world))

    # end to end through the public API with host buffers
    e2e = bench_e2e(args, mbt, x3, x4, world)

    peak, peak_kind = measured_peak()
    kernels = {
        "copy": {"ms": round(ms_copy, 4), "bytes": copy_bytes(),
                 "gbs": round(copy_bytes() / ms_copy / 1e6, 1),
                 "ms_host_launched": round(ms_copy_stream, 4),
                 "gbs_host_launched": round(copy_bytes() / ms_copy_stream / 1e6, 1),
                 "ms_event_pairs": round(ms_copy_pairs, 4),
                 "gbs_event_pairs": round(copy_bytes() / ms_copy_pairs / 1e6, 1),
                 "ms_event_pairs_best": round(copy_pairs_stats[0], 4),
                 "ms_event_pairs_median": round(copy_pairs_stats[1], 4),
                 "ms_in_one_stream_step": round(ms_copy_seq, 4),
                 "stages": args.copy_stages, "tile": [COPY["tile_m"], COPY["tile_n"]]},
        "rowsum": {"ms": round(ms_rowsum, 4), "bytes": rowsum_bytes(),
                   "gbs": round(rowsum_bytes() / ms_rowsum / 1e6, 1),
                   "ms_host_launched": round(ms_rowsum_stream, 4),
                   "gbs_host_launched": round(rowsum_bytes() / ms_rowsum_stream / 1e6, 1),
                   "ms_event_pairs": round(ms_rowsum_pairs, 4),
                   "gbs_event_pairs": round(rowsum_bytes() / ms_rowsum_pairs / 1e6, 1),
                   "ms_event_pairs_best": round(rowsum_pairs_stats[0], 4),
                   "ms_event_pairs_median": round(rowsum_pairs_stats[1], 4),
                   "ms_in_one_stream_step": round(ms_rowsum_seq, 4),
                   "stages": args.rowsum_stages, "tile": [ROWSUM["tile_m"], ROWSUM["tile_n"]]},
    }
    dom_name = "copy" if ms_copy >= ms_rowsum else "rowsum"
    dom = kernels[dom_name]
    traffic = None
    entry = NCU_TRAFFIC.get(dom_name)
    if entry and entry.get("src_sha") == kernel_source_sha():
        traffic = entry["bytes_per_launch"]
    roofline = {"bound": "hbm", "kernel": f"mbt_{dom_name}_kernel",
                "achieved": dom["gbs"], "peak": peak, "unit": "GB/s",
                "frac": round(dom["gbs"] / peak, 4), "traffic": traffic,
                "peak_source": f"{peak_kind} hbm_gbs (copy read+write)",
                "timing": ((f"{args.steps} launches of the kernel replayed from CUDA graphs "
                            f"of {GRAPH_CHUNK} launches" if graph else
                            f"{args.steps} launches of the kernel from the host") +
                           ", back to back on one stream, one CUDA event pair around all "
                           "of them: mean per launch, gaps included; kernels.*."
                           "ms_host_launched: the same launches from the host; kernels.*."
                           "ms_event_pairs: host launches with an event pair around each "
                           "(mean; _best and _median of the same launches); "
                           "kernels.*.ms_in_one_stream_step: the two kernels alternating "
                           "on one stream, where each inherits the other's L2 write-back"),
                "read_peak": read_ref,
                "frac_of_read_peak": (round(dom["gbs"] / read_ref["gbs"], 4)
                                      if dom_name == "rowsum" and read_ref else None),
                "rowsum_frac_of_read_peak": (round(kernels["rowsum"]["gbs"] / read_ref["gbs"], 4)
                                             if read_ref else None),
                "read_same_size": read_same,
                "rowsum_frac_of_read_same_size": (round(kernels["rowsum"]["gbs"] / read_same["gbs"], 4)
                                                  if read_same else None)}
    out = {
        "metric": "achieved HBM GB/s (read+write) for pipelined tile copy + rowsum",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 copy + bf16->f32 rowsum", "data": "synthetic (seeded, drawn on device)",
        "config": {"workload": ("tile_copy fp16 16384x16384 tile 128x64 + tile_rowsum "
                                "bf16 8192x65536 tile 64x256"),
                   "copy_stages": args.copy_stages, "rowsum_stages": args.rowsum_stages,
                   "copy_store_mode": args.store_mode,
                   "streams": ("copy and rowsum each on its own stream (independent calls, "
                               "so the kernels overlap); value_one_stream: both on one stream"
                               if args.streams == 2 else "one stream"),
                   "launch": (f"steps replayed from CUDA graphs of {GRAPH_CHUNK} steps each "
                              "(captured once before the timed region)" if graph else
                              "each call launched from the host"),
                   "l2": "inputs (512 MiB, 1 GiB) larger than L2; no flush",
                   "parallelism": f"independent replica per GPU x{world}"},
        "frac_of_peak": round(value / world / peak, 4),
        "value_one_stream": round(value_one_stream, 1),
        ("value_host_launched" if graph else "value_graph_replay"): round(value_other_launch, 1),
        "kernels": kernels,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks.summary(t0, t1),
    }
    if sweep is not None:
        out["sweep"] = sweep
        out["sweep_note"] = (
            "every workload configuration (1, 2: latency; 3: copy at 1/2/3/4/6 "
            "stages with LSU and bulk stores; 4: row and column sums at 2/3/4 stages with a "
            "caller's workspace, and the plain calls with the library's own; 5a/5b: copy, "
            "row sum, column sum and fused copy + row sum at 3 stages), each timed by "
            f"replaying CUDA graphs of its calls for about {POINT_TARGET_S} s on one stream "
            "(ms = mean per launch, gaps included; ms_host_launched: 20 host launches back "
            "to back), clocks sampled during its replays, output checked on the device "
            "before timing; frac = gbs / measured hbm_gbs")
    if flat is not None:
        out["flat_points"] = flat
        out["flat_note"] = (
            "the 1-D bulk-copy kernels (row pitches that are not a multiple of 16 bytes, "
            "and row sums of rows of at most 64 bytes), dense matrices: each point checked "
            f"on the device, then launched from the host back to back for about "
            f"{POINT_TARGET_S} s between one event pair (no graph), clocks sampled in that "
            "window; windows = the plan's bulk-copy windows (row pieces or groups of rows)")
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(x3, d3, x4, o4, args.cpu_budget)
    return out


def bench_e2e(args, mbt, x3, x4, world):
    """Same metric through the host-buffer C-ABI calls: every step runs
    tile_copy_host on the fp16 matrix and tile_rowsum_host on the bf16 matrix,
    both in pinned host memory; each call copies its input in, runs the tile
    pipeline and copies the result out, slab by slab with the three
    overlapped, and returns when the result is in host memory.  With
    args.e2e_threads == 2 the two calls of a step run on two host threads
    (independent calls; the copy's device-to-host traffic then shares the
    link with the row sum's host-to-device traffic).  Host wall-clock time,
    max over ranks."""
    import threading

    steps = max(1, min(args.steps, args.e2e_steps))
    h3 = torch.empty(x3.shape, dtype=x3.dtype, pin_memory=True)
    h3.copy_(x3)
    h4 = torch.empty(x4.shape, dtype=x4.dtype, pin_memory=True)
    h4.copy_(x4)
    r3 = torch.empty_like(h3, pin_memory=True)
    r4 = torch.empty(x4.shape[0], dtype=torch.float32, pin_memory=True)

    def run_copy():
        mbt.tile_copy_host(h3, r3, COPY["tile_m"], COPY["tile_n"], args.copy_stages,
                           store_mode=args.store_mode)

    def run_rowsum():
        mbt.tile_rowsum_host(h4, r4, ROWSUM["tile_m"], ROWSUM["tile_n"], args.rowsum_stages)

    def step():
        if args.e2e_threads == 2:
            t = threading.Thread(target=run_copy)
            t.start()
            run_rowsum()
            t.join()
        else:
            run_copy()
            run_rowsum()

    step()   # warm-up: staging sets allocated, plans cached
    if not torch.equal(r3.view(torch.int16), h3.view(torch.int16)):
        raise RuntimeError("tile_copy_host result differs from its input")
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    ms = reduce_max((time.perf_counter() - t0) * 1e3, world)
    value = aggregate_gbs(copy_bytes() + rowsum_bytes(), steps, world, ms)
    h2d = h3.numel() * h3.element_size() + h4.numel() * h4.element_size()
    d2h = r3.numel() * r3.element_size() + r4.numel() * r4.element_size()
    link = link_rates(x3.device)
    bound = link_bound_gbs(h2d, d2h, copy_bytes() + rowsum_bytes(), link)
    return {"value": round(value, 1), "unit": "GB/s", "steps": steps,
            "api": "tile_copy_host + tile_rowsum_host (host buffers, pinned)",
            "host_threads": args.e2e_threads,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "link": link, "link_bound": round(bound, 1),
            "frac_of_link_bound": round(value / world / bound, 4),
            "link_note": ("link_bound: the step's algorithmic bytes over the shortest time "
                          "the link allows for its host-to-device and device-to-host bytes: "
                          "all device-to-host traffic overlapped with host-to-device traffic "
                          "at the rates both directions reach together, the rest of the "
                          "host-to-device traffic alone")}


def link_rates(device, nbytes: int = 512 << 20) -> dict:
    """GB/s of pinned-host <-> device copies of nbytes (best of 3): each
    direction alone, then both at once on two streams (each direction's own
    rate while the other runs)."""
    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=device)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def best_ms(run):
        best = float("inf")
        for _ in range(3):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            torch.cuda.synchronize()
            run(ev)
            torch.cuda.synchronize()
            best = min(best, run.ms(ev))
        return best

    def one(dst, src, stream):
        def run(ev):
            ev[0].record(stream)
            with torch.cuda.stream(stream):
                dst.copy_(src, non_blocking=True)
            ev[1].record(stream)
        run.ms = lambda ev: ev[0].elapsed_time(ev[1])
        return run

    h2d = nbytes / best_ms(one(d_a, h_in, s1)) / 1e6
    d2h = nbytes / best_ms(one(h_out, d_b, s2)) / 1e6
    both = {}
    for _ in range(3):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        torch.cuda.synchronize()
        ev[0].record(s1)
        ev[2].record(s2)
        with torch.cuda.stream(s1):
            d_a.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_b, non_blocking=True)
        ev[1].record(s1)
        ev[3].record(s2)
        torch.cuda.synchronize()
        hb = nbytes / ev[0].elapsed_time(ev[1]) / 1e6
        db = nbytes / ev[2].elapsed_time(ev[3]) / 1e6
        if hb + db > both.get("h2d_gbs", 0) + both.get("d2h_gbs", 0):
            both = {"h2d_gbs": round(hb, 1), "d2h_gbs": round(db, 1)}
    return {"h2d_gbs": round(h2d, 1), "d2h_gbs": round(d2h, 1), "both": both,
            "bytes": nbytes}


def link_bound_gbs(h2d: int, d2h: int, alg: int, link: dict) -> float:
    """Throughput bound of a step that moves h2d bytes in and d2h bytes out:
    the out-going bytes overlapped with in-coming ones at the rates both
    directions reach together, the remainder of either direction alone."""
    hb, db = link["both"]["h2d_gbs"] * 1e9, link["both"]["d2h_gbs"] * 1e9
    if d2h / db <= h2d / hb:
        t = d2h / db + (h2d - hb * d2h / db) / (link["h2d_gbs"] * 1e9)
    else:
        t = h2d / hb + (d2h - db * h2d / hb) / (link["d2h_gbs"] * 1e9)
    return alg / t / 1e9


def bench_only(args):
    """Run one kernel ``args.steps`` times on the first ``args.rows`` rows of
    its workload (for profiling a smaller case under ncu), and print its GB/s."""
    import mbarrier_async_tile_gb300 as mbt
    import synthetic

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.only == "read":
        # the read reference on a buffer of --rows MiB (default 1024)
        nbytes = (args.rows or 1024) << 20
        buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        out = torch.empty(1, dtype=torch.int32, device=dev)
        fn = lambda: mbt.tile_read_checksum(buf, out)  # noqa: E731
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(args.steps):
            fn()
        e.record()
        torch.cuda.synchronize()
        ms = s.elapsed_time(e) / args.steps
        print(json.dumps({"only": "read", "bytes": nbytes, "ms": round(ms, 4),
                          "gbs": round(nbytes / ms / 1e6, 1)}), flush=True)
        return
    c = ROWSUM if args.only in ("rowsum", "colsum") else COPY
    if args.config:
        c = RAGGED[args.config]
    rows = args.rows or c["M"]
    cols = args.cols or c["N"] - args.trim_cols
    ld = synthetic.pitched_ld(cols, c["dtype"]) if args.config else cols
    x = synthetic.make_matrix(rows, cols, c["dtype"], c["dist"], c["seed"], ld=ld,
                              draw_on=str(dev))[:, :cols]
    def like_x():
        return torch.empty(rows, ld, dtype=x.dtype, device=dev)[:, :cols]

    if args.only == "copy_rowsum":
        y = like_x()
        o = torch.empty(rows, dtype=torch.float32, device=dev)
        ws = torch.zeros(1 << 22, dtype=torch.uint8, device=dev)
        fn = lambda: mbt.tile_copy_rowsum(x, y, o, c["tile_m"], c["tile_n"],  # noqa: E731
                                          args.copy_stages, workspace=ws)
        nbytes = 2 * x.numel() * x.element_size() + 4 * rows
    elif args.only == "copy":
        y = like_x()
        fn = lambda: mbt.tile_copy(x, y, c["tile_m"], c["tile_n"], args.copy_stages,  # noqa: E731
                                   consumer_warps=args.consumer_warps,
                                   ctas_per_sm=args.ctas_per_sm, max_ctas=args.max_ctas,
                                   store_mode=args.store_mode)
        nbytes = 2 * x.numel() * x.element_size()
    elif args.only == "colsum":
        y = torch.empty(cols, dtype=torch.float32, device=dev)
        ws = torch.zeros(1 << 22, dtype=torch.uint8, device=dev)
        fn = lambda: mbt.tile_colsum(x, y, c["tile_m"], c["tile_n"], args.rowsum_stages,  # noqa: E731
                                     consumer_warps=args.consumer_warps,
                                     ctas_per_sm=args.ctas_per_sm, max_ctas=args.max_ctas,
                                     workspace=ws)
        nbytes = x.numel() * x.element_size() + 4 * cols
    else:
        y = torch.empty(rows, dtype=torch.float32, device=dev)
        ws = torch.zeros(1 << 22, dtype=torch.uint8, device=dev)
        fn = lambda: mbt.tile_rowsum(x, y, c["tile_m"], c["tile_n"], args.rowsum_stages,  # noqa: E731
                                     consumer_warps=args.consumer_warps,
                                     ctas_per_sm=args.ctas_per_sm, max_ctas=args.max_ctas,
                                     workspace=ws)
        nbytes = x.numel() * x.element_size() + 4 * rows
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        fn()
    e.record()
    torch.cuda.synchronize()
    code, info = mbt.tile_status()
    if code != 0:
        raise RuntimeError(f"pipeline status {code} {info}")
    ms = s.elapsed_time(e) / args.steps
    print(json.dumps({"only": args.only, "rows": rows, "cols": cols, "ms": round(ms, 4),
                      "gbs": round(nbytes / ms / 1e6, 1)}), flush=True)


# Every workload configuration (lesson shapes 1-2, streaming 3-4, ragged 5a-5b), each point timed in its own window
# with the SM clocks sampled there.  (config, op, dtype, M, N, tile_m, tile_n,
# stages, extra) -- extra: store_mode for copies, "caller" / "library" for the
# sums' workspace.
CONFIG_POINTS = (
    [("1", "copy", "f16", 256, 128, 128, 64, 1, {}),
     ("2", "copy", "f16", 128, 512, 128, 64, 3, {"consumer_warps": 3, "max_ctas": 1})]
    + [("3", "copy", "f16", 16384, 16384, 128, 64, st, {"store_mode": mode})
       for mode in (2, 1) for st in (1, 2, 3, 4, 6)]
    + [("4", op, "bf16", 8192, 65536, 64, 256, st, {"workspace": "caller"})
       for op in ("rowsum", "colsum") for st in (2, 3, 4)]
    + [("4", op, "bf16", 8192, 65536, 64, 256, 2, {"workspace": "library"})
       for op in ("rowsum", "colsum")]
    + [(cfg, op, dt, M, N, tm, tn, 3, extra)
       for cfg, dt, M, N, tm, tn in (("5a", "f32", 12289, 8191, 128, 32),
                                     ("5b", "f16", 24577, 16383, 128, 64))
       for op, extra in (("copy", {"store_mode": 2}), ("copy", {"store_mode": 1}),
                         ("rowsum", {"workspace": "caller"}),
                         ("rowsum", {"workspace": "library"}),
                         ("colsum", {"workspace": "caller"}),
                         ("colsum", {"workspace": "library"}),
                         ("copy_rowsum", {"workspace": "library"}))]
)
CONFIG_SEEDS = {"1": 1001, "2": 1002, "3": 1003, "4": 1004, "5a": 1005, "5b": 1006}
CONFIG_DIST = {"4": "normal"}
POINT_TARGET_S = 0.25     # device time of each point's timed graph replays


# The 1-D bulk-copy path: row pitches that are not a multiple of 16 bytes (a
# 2-D tensor map cannot describe them) and row sums of rows of at most 64
# bytes.  (op, dtype, M, N, tile_m, tile_n, stages); every matrix dense.
FLAT_POINTS = (
    ("rowsum", "bf16", 4096, 65535, 64, 256, 2),     # 131,070-byte rows, in pieces
    ("rowsum", "f16", 24577, 16383, 128, 64, 2),     # 32,766-byte rows, one a window
    ("rowsum", "f16", 4194304, 63, 128, 64, 2),      # 126-byte rows, lane groups
    ("rowsum", "bf16", 8000000, 16, 64, 256, 2),     # 32-byte rows, one thread a row
    ("copy", "f16", 24577, 16383, 128, 64, 3),       # one contiguous byte array
)
FLAT_SEED = 1007


def flat_points(dev, clocks, peak: float, read_peak: float | None = None,
                target_s: float = POINT_TARGET_S) -> list:
    """Each FLAT_POINTS entry: run once and checked on the device (copies bit
    for bit, row sums on 64 sampled rows against a float64 sum within 1e-5 of
    max(|sum|, sqrt(sum of squares))), 20 launches to size the timed run,
    then launches from the host back to back for about `target_s` between one
    event pair on a side stream, with the SM clocks sampled in that window.
    A point that raises is recorded with its error and the next one runs."""
    import mbarrier_async_tile_gb300 as mbt
    import synthetic

    side = torch.cuda.Stream()
    points = []
    for op, dt, M, N, tm, tn, st in FLAT_POINTS:
        rec = {"op": op, "dtype": dt, "shape": [M, N], "ld": N, "tile": [tm, tn],
               "stages": st}
        x = y = o = call = None
        try:
            es = ESIZE[dt]
            x = synthetic.make_matrix(M, N, dt, "uniform", FLAT_SEED, draw_on=str(dev))
            if op == "copy":
                y = torch.full_like(x, float("nan"))
                nbytes = 2 * M * N * es

                def call(s, x=x, y=y):
                    mbt.tile_copy(x, y, tm, tn, st, stream=s)
            else:
                o = torch.full((M,), float("nan"), dtype=torch.float32, device=dev)
                nbytes = M * N * es + 4 * M

                def call(s, x=x, o=o):
                    mbt.tile_rowsum(x, o, tm, tn, st, stream=s)
            plan = mbt.tile_plan_device(mbt.OP_COPY if op == "copy" else mbt.OP_ROWSUM,
                                        M, N, tm, tn, st, x.dtype)
            side.wait_stream(torch.cuda.current_stream())
            call(side)
            code, info = mbt.tile_status(side)
            if code != 0:
                raise RuntimeError(f"pipeline status {code} {info}")
            if op == "copy":
                iv = torch.int32 if es == 4 else torch.int16
                ok = torch.equal(y.view(iv), x.view(iv))
            else:
                g = torch.Generator().manual_seed(5)
                idx = torch.randperm(M, generator=g)[:64].to(dev)
                part = x.index_select(0, idx).double()
                ref = part.sum(1)
                scale = torch.maximum(ref.abs(), part.pow(2).sum(1).sqrt())
                ok = bool(((o[idx].double() - ref).abs() <= 1e-5 * scale).all())
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for _ in range(3):
                call(side)
            e0.record(side)
            for _ in range(20):
                call(side)
            e1.record(side)
            torch.cuda.synchronize()
            n = max(20, int(target_s / max(e0.elapsed_time(e1) / 20 / 1e3, 1e-6)))
            t0 = time.time()
            e0.record(side)
            for _ in range(n):
                call(side)
            e1.record(side)
            torch.cuda.synchronize()
            t1 = time.time()
            code, info = mbt.tile_status(side)
            if code != 0:
                raise RuntimeError(f"pipeline status {code} {info}")
            ms = e0.elapsed_time(e1) / n
            gbs = nbytes / ms / 1e6
            c = clocks.summary(t0, t1)
            rec.update(bytes=nbytes, ms=round(ms, 4), gbs=round(gbs, 1),
                       frac=round(gbs / peak, 4),
                       frac_of_read_peak=(round(gbs / read_peak, 4)
                                          if read_peak and op == "rowsum" else None),
                       grid=plan["grid"], threads=plan["threads"],
                       stage_bytes=plan["stage_bytes"], windows=plan["num_tiles"],
                       launches_timed=n, parity_ok=bool(ok),
                       clocks={"sm_mhz": c.get("sm_mhz"), "sm_max_mhz": c.get("sm_max_mhz"),
                               "reasons": c.get("reasons"), "samples": c.get("samples")})
        except Exception as e:   # recorded; the other points and the line go on
            rec["error"] = f"{type(e).__name__}: {e}"[:300]
        del x, y, o, call      # the closure holds the tensors too
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        points.append(rec)
    return points


READ_REF_BYTES = 4 << 30   # the read reference's buffer: far larger than L2


def read_reference(dev, clocks, target_s: float = POINT_TARGET_S,
                   nbytes: int = READ_REF_BYTES) -> dict:
    """The read-only ceiling of this device for the reductions: GB/s of
    tile_read_checksum (one pass of 16-byte loads over an nbytes buffer, every
    32-bit word folded into an XOR checksum), replayed from a CUDA graph of 10
    launches for about `target_s`, one event pair around the replays, with
    the clocks sampled meanwhile."""
    import mbarrier_async_tile_gb300 as mbt

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.empty(1, dtype=torch.int32, device=dev)
    side.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        mbt.tile_read_checksum(buf, out, stream=side)
    torch.cuda.synchronize()
    n = 10
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(n):
            mbt.tile_read_checksum(buf, out, stream=side)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(side):
        e0.record(side)
        graph.replay()
        e1.record(side)
    torch.cuda.synchronize()
    reps = max(3, int(target_s / max(e0.elapsed_time(e1) / 1e3, 1e-6)) + 1)
    t0 = time.time()
    with torch.cuda.stream(side):
        e0.record(side)
        for _ in range(reps):
            graph.replay()
        e1.record(side)
    torch.cuda.synchronize()
    t1 = time.time()
    ms = e0.elapsed_time(e1) / (reps * n)
    del graph, buf
    torch.cuda.empty_cache()
    c = clocks.summary(t0, t1)
    return {"gbs": round(nbytes / ms / 1e6, 1), "ms": round(ms, 4),
            "bytes": nbytes, "kernel": "mbt_read_checksum_kernel",
            "what": (f"tile_read_checksum: one pass of 16-byte loads over a {nbytes >> 20} MiB "
                     "device buffer (XOR of every 32-bit word), graph replay, mean per launch"),
            "launches_timed": reps * n,
            "clocks": {"sm_mhz": c.get("sm_mhz"), "sm_max_mhz": c.get("sm_max_mhz"),
                       "reasons": c.get("reasons"), "samples": c.get("samples")}}


def config_sweep(dev, clocks, peak: float, theo: float, target_s: float = POINT_TARGET_S,
                 select=None, read_peak: float | None = None, read_at_size: bool = False):
    """Time every CONFIG_POINTS entry (or those `select` keeps) on one side
    stream: the calls captured in a CUDA graph (20 launches, 200 for the
    latency-bound lesson shapes), replayed until about `target_s` of device
    time, one event pair around the replays (mean per launch, gaps included);
    then 20 launches from the host, back to back.  The SM clocks sampled
    during each point's replays go with it.  Each point's output is checked
    once on the device first (copies bit for bit, sums on sampled rows or
    columns against a float64 reduction within 1e-5 of max(|sum|, sqrt(sum
    of squares))).  With `read_at_size`, each row or column sum is also
    compared with the read reference over as many bytes as the sum reads
    (measured once per size: a short launch pays the same ramp-up and tail).
    Returns the list of point records."""
    import mbarrier_async_tile_gb300 as mbt
    import synthetic

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    out_points = []
    cache = {}
    read_at = {}   # bytes -> read reference GB/s at that size

    def matrix(cfg, dt, M, N):
        key = (cfg, dt, M, N)
        if key not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            ld = synthetic.pitched_ld(N, dt) if cfg in ("5a", "5b") else N
            x = synthetic.make_matrix(M, N, dt, CONFIG_DIST.get(cfg, "uniform"),
                                      CONFIG_SEEDS[cfg], ld=ld, draw_on=str(dev))
            cache[key] = (x, ld)
        return cache[key]

    def check_status(what):
        code, info = mbt.tile_status(side)
        if code != 0:
            raise RuntimeError(f"{what}: pipeline status {code} {info}")

    def sums_ok(got, x, dim, g):
        n = x.shape[1 - dim]
        idx = torch.randperm(n, generator=g)[:64].to(dev)
        part = x.index_select(1 - dim, idx).double()
        ref = part.sum(dim)
        scale = torch.maximum(ref.abs(), part.pow(2).sum(dim).sqrt())
        return bool(((got[idx].double() - ref).abs() <= 1e-5 * scale).all())

    for (cfg, op, dt, M, N, tm, tn, st, extra) in CONFIG_POINTS:
        if select is not None and not select(cfg, op, st, extra):
            continue
        x, ld = matrix(cfg, dt, M, N)
        xs = x[:, :N]
        es = ESIZE[dt]
        ws_kind = extra.get("workspace")
        kw = {k: v for k, v in extra.items() if k != "workspace"}
        y = torch.empty_like(x)[:, :N] if op in ("copy", "copy_rowsum") else None
        o = torch.empty(N if op == "colsum" else M, dtype=torch.float32, device=dev) \
            if op != "copy" else None
        ws = None
        if ws_kind == "caller":
            need = (mbt.tile_colsum_workspace_bytes if op == "colsum"
                    else mbt.tile_rowsum_workspace_bytes)(M, N, tm, tn, st, xs.dtype, ld_src=ld)
            ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
        if op == "copy":
            call = lambda s: mbt.tile_copy(xs, y, tm, tn, st, stream=s, **kw)  # noqa: E731
            nbytes = 2 * M * N * es
        elif op == "rowsum":
            call = lambda s: mbt.tile_rowsum(xs, o, tm, tn, st, workspace=ws,  # noqa: E731
                                             stream=s, **kw)
            nbytes = M * N * es + 4 * M
        elif op == "colsum":
            call = lambda s: mbt.tile_colsum(xs, o, tm, tn, st, workspace=ws,  # noqa: E731
                                             stream=s, **kw)
            nbytes = M * N * es + 4 * N
        else:
            call = lambda s: mbt.tile_copy_rowsum(xs, y, o, tm, tn, st, stream=s,  # noqa: E731
                                                  **kw)
            nbytes = 2 * M * N * es + 4 * M
        latency = cfg in ("1", "2")
        n_graph = 200 if latency else 20
        # once, checked (this also plans, and allocates the library's workspace)
        if y is not None:
            y.fill_(float("nan"))
        # inputs, poison and workspace were written on the current stream
        side.wait_stream(torch.cuda.current_stream())
        call(side)
        torch.cuda.synchronize()
        check_status(f"config {cfg} {op}")
        g = torch.Generator().manual_seed(5)
        ok = True
        if y is not None:
            iv = torch.int32 if es == 4 else torch.int16
            ok = ok and torch.equal(y.contiguous().view(iv), xs.contiguous().view(iv))
        if op in ("rowsum", "copy_rowsum"):
            ok = ok and sums_ok(o, xs, 1, g)
        if op == "colsum":
            ok = ok and sums_ok(o, xs, 0, g)
        # host-launched, back to back
        for _ in range(3):
            call(side)
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_host = 200 if latency else 20
        torch.cuda.synchronize()
        h0.record(side)
        for _ in range(n_host):
            call(side)
        h1.record(side)
        torch.cuda.synchronize()
        check_status(f"config {cfg} {op}")
        ms_host = h0.elapsed_time(h1) / n_host
        # graph replays
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for _ in range(n_graph):
                call(side)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(side):
            e0.record(side)
            graph.replay()
            e1.record(side)
        torch.cuda.synchronize()
        reps = max(3, int(target_s / max(e0.elapsed_time(e1) / 1e3, 1e-6)) + 1)
        t0 = time.time()
        with torch.cuda.stream(side):
            e0.record(side)
            for _ in range(reps):
                graph.replay()
            e1.record(side)
        torch.cuda.synchronize()
        t1 = time.time()
        check_status(f"config {cfg} {op}")
        ms = e0.elapsed_time(e1) / (reps * n_graph)
        del graph
        rec = {"config": cfg, "op": op, "dtype": dt, "shape": [M, N], "ld": ld,
               "tile": [tm, tn], "stages": st}
        if "store_mode" in extra:
            rec["store"] = MODE_NAME[extra["store_mode"]]
        if ws_kind:
            rec["workspace"] = ws_kind
        if "max_ctas" in extra:
            rec["ctas"] = extra["max_ctas"]
            rec["consumer_warps"] = extra["consumer_warps"]
        rec["bytes"] = nbytes
        if latency:
            rec["us_per_call"] = round(ms * 1e3, 3)
            rec["us_per_call_host_launched"] = round(ms_host * 1e3, 3)
        else:
            gbs = nbytes / ms / 1e6
            rec.update(ms=round(ms, 4), gbs=round(gbs, 1), frac=round(gbs / peak, 4),
                       frac_theoretical=round(gbs / theo, 4) if theo else None,
                       frac_of_read_peak=(round(gbs / read_peak, 4)
                                          if read_peak and op in ("rowsum", "colsum") else None),
                       ms_host_launched=round(ms_host, 4),
                       gbs_host_launched=round(nbytes / ms_host / 1e6, 1))
        rec["launches_timed"] = reps * n_graph
        rec["parity_ok"] = bool(ok)
        c = clocks.summary(t0, t1)
        if read_at_size and not latency and op in ("rowsum", "colsum"):
            rb = (M * N * es + 15) // 16 * 16
            if rb not in read_at:
                read_at[rb] = read_reference(dev, clocks, target_s, rb)["gbs"]
            rec["read_same_size_gbs"] = read_at[rb]
            rec["frac_of_read_same_size"] = round(rec["gbs"] / read_at[rb], 4)
        rec["clocks"] = {"sm_mhz": c.get("sm_mhz"), "sm_max_mhz": c.get("sm_max_mhz"),
                         "reasons": c.get("reasons"), "samples": c.get("samples")}
        out_points.append(rec)
    cache.clear()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out_points


def bench_configs(args):
    """One JSON line per configuration point (see config_sweep) and per
    1-D bulk-copy point (flat_points), then the denominators."""
    import mbarrier_async_tile_gb300 as mbt

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, peak_kind = measured_peak()
    theo = mbt.tile_device_info()["hbm_gbs_theoretical"]
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    try:
        ref = read_reference(dev, clocks)
        print(json.dumps({"read_reference": ref}), flush=True)
        for rec in config_sweep(dev, clocks, peak, theo, read_peak=ref["gbs"]):
            print(json.dumps(rec), flush=True)
        for rec in flat_points(dev, clocks, peak, read_peak=ref["gbs"]):
            print(json.dumps({"flat": rec}), flush=True)
    finally:
        clocks.stop()
    print(json.dumps({"peak_gbs": peak, "peak_source": peak_kind,
                      "theoretical_gbs": round(theo, 1)}), flush=True)


def bench_sweep(args):
    """One line per (op, stages, consumer warps, CTAs per SM) point."""
    import mbarrier_async_tile_gb300 as mbt

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    x3, d3, x4, o4 = make_inputs(dev)
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device=dev)
    reps = 20

    def timeit(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        torch.cuda.synchronize()
        assert mbt.tile_status()[0] == 0
        return s.elapsed_time(e) / reps

    for st in args.sweep_stages:
        for w in args.sweep_warps:
            for cps in args.sweep_ctas:
                try:
                    ms = timeit(lambda: mbt.tile_copy(x3, d3, COPY["tile_m"], COPY["tile_n"], st,
                                                      consumer_warps=w, ctas_per_sm=cps,
                                                      store_mode=args.store_mode))
                    print(json.dumps({"sweep": "copy", "store_mode": args.store_mode,
                                      "stages": st, "consumer_warps": w,
                                      "ctas_per_sm": cps, "ms": round(ms, 4),
                                      "gbs": round(copy_bytes() / ms / 1e6, 1)}), flush=True)
                except mbt.MbtError as exc:
                    print(json.dumps({"sweep": "copy", "stages": st, "consumer_warps": w,
                                      "ctas_per_sm": cps, "error": str(exc)}), flush=True)
                if st < 2 or st > 6:
                    continue
                try:
                    ms = timeit(lambda: mbt.tile_rowsum(x4, o4, ROWSUM["tile_m"], ROWSUM["tile_n"],
                                                        st, consumer_warps=w, ctas_per_sm=cps,
                                                        workspace=ws))
                    print(json.dumps({"sweep": "rowsum", "stages": st, "consumer_warps": w,
                                      "ctas_per_sm": cps, "ms": round(ms, 4),
                                      "gbs": round(rowsum_bytes() / ms / 1e6, 1)}), flush=True)
                except mbt.MbtError as exc:
                    print(json.dumps({"sweep": "rowsum", "stages": st, "consumer_warps": w,
                                      "ctas_per_sm": cps, "error": str(exc)}), flush=True)


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def bench_reference(args):
    """Time the CPU oracle as it stands on the host's cores: each step is one
    bounded sample of the workload (row blocks of both matrices in
    proportion to their bytes), split into disjoint row blocks that run on
    as many host threads as there are cores."""
    import oracle
    import synthetic

    oracle.build()
    cores = host_cores()
    rows3, rows4 = 32 * cores, 8 * cores   # 1 + 1 MiB of input per thread per step
    x3 = synthetic.make_matrix(rows3, COPY["N"], COPY["dtype"], COPY["dist"], COPY["seed"])
    x4 = synthetic.make_matrix(rows4, ROWSUM["N"], ROWSUM["dtype"], ROWSUM["dist"],
                               ROWSUM["seed"])
    d3 = torch.empty_like(x3)
    jobs = []
    for i in range(cores):
        a3, a4 = slice(32 * i, 32 * (i + 1)), slice(8 * i, 8 * (i + 1))
        jobs.append(lambda a3=a3, a4=a4: (oracle.copy(x3[a3], d3[a3]), oracle.rowsum(x4[a4])))

    with concurrent.futures.ThreadPoolExecutor(max_workers=cores) as pool:
        for _ in range(args.warmup):
            oracle_blocks_parallel(jobs, pool)
        sec = 0.0
        for _ in range(args.steps):
            sec += oracle_blocks_parallel(jobs, pool)
    if not torch.equal(d3.view(torch.int16), x3.view(torch.int16)):
        raise RuntimeError("oracle copy differs from its input")
    nbytes = 2 * x3.numel() * 2 + x4.numel() * 2 + 4 * rows4
    value = nbytes * args.steps / sec / 1e9
    sample = (f"each step: oracle copy of {rows3} rows of the fp16 16384x16384 matrix and "
              f"oracle row sum of {rows4} rows of the bf16 8192x65536 matrix "
              f"({nbytes / 1e6:.1f} MB algorithmic), split over {cores} host threads")
    return {
        "impl": "reference",
        "metric": "achieved HBM GB/s (read+write) for pipelined tile copy + rowsum",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sec / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 copy + bf16->f64 rowsum", "data": "synthetic (seeded)",
        "config": {"workload": ("tile_copy fp16 16384x16384 tile 128x64 + tile_rowsum "
                                "bf16 8192x65536 tile 64x256 (row-block sample per step)")},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
def aggregate_gbs(step_bytes: int, steps: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: every rank processed `steps` steps of `step_bytes`
    (independent replicas); the job took the slowest rank's time."""
    return world * step_bytes * steps / (ms_max / 1e3) / 1e9


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.distributed.get_backend() == "nccl" else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mbtile", "reference"], default="mbtile")
    ap.add_argument("--streams", type=int, default=2, choices=[1, 2])
    ap.add_argument("--launch", choices=["graph", "host"], default="graph",
                    help="time steps replayed from CUDA graphs (default) or launched "
                         "call by call from the host; the other is reported beside it")
    ap.add_argument("--copy-stages", type=int, default=3)
    ap.add_argument("--rowsum-stages", type=int, default=2)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-threads", type=int, default=2, choices=(1, 2),
                    help="host threads running the two host-buffer calls of an e2e step")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--all-configs", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="leave the per-configuration sweep out of the default line")
    ap.add_argument("--no-read-ref", action="store_true",
                    help="leave the read-bandwidth reference out of the default line")
    ap.add_argument("--only", choices=["copy", "rowsum", "copy_rowsum", "colsum", "read"])
    ap.add_argument("--config", choices=sorted(RAGGED),
                    help="--only: one of the ragged workloads (pitched rows) instead of "
                         "the bench workload")
    ap.add_argument("--trim-cols", type=int, default=0,
                    help="--only: drop this many columns (an odd count gives a dense matrix "
                         "whose rows are not a multiple of 16 bytes: the 1-D bulk-copy path)")
    ap.add_argument("--store-mode", type=int, default=0, choices=[0, 1, 2])
    ap.add_argument("--rows", type=int, default=0)
    ap.add_argument("--cols", type=int, default=0,
                    help="--only: columns of the matrix (dense rows; a pitch that is not a "
                         "multiple of 16 bytes takes the 1-D bulk-copy kernels)")
    ap.add_argument("--consumer-warps", type=int, default=0)
    ap.add_argument("--ctas-per-sm", type=int, default=0)
    ap.add_argument("--max-ctas", type=int, default=0)
    ap.add_argument("--sweep-stages", type=int, nargs="*", default=[1, 2, 3, 4, 6])
    ap.add_argument("--sweep-warps", type=int, nargs="*", default=[3, 4, 7])
    ap.add_argument("--sweep-ctas", type=int, nargs="*", default=[1, 2, 0])
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(bench_reference(args)), flush=True)
        return 0
    if args.sweep:
        bench_sweep(args)
        return 0
    if args.only:
        bench_only(args)
        return 0
    if args.all_configs:
        bench_configs(args)
        return 0
    if world > 1:
        torch.distributed.init_process_group(
            backend="nccl" if torch.cuda.is_available() else "gloo")
    out = bench_gpu(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
