#!/usr/bin/env python3
"""Benchmark of the EXL3 trellis linear on one GB300 (or N replicas).

Workload (decode rows at the 27B shapes): K = 5120, 4-bit trellis codes, 16
rows of FP16 activations. One step is one q/k/v group call (N = 6144 + 1024 +
1024: one rotation launch and one linear launch) followed by one single call on
a 5120 x 5120 weight: the whole hot path (rotation, weight stream, decode, MMA,
split-K combine, output rotation) over one batch. The timed K steps replay from
one CUDA graph.

Metric: weight-stream GB/s (packed code bytes of every weight the step reads /
step time), with µs per call alongside. Weights cycle through enough distinct
copies that every step streams from HBM (> 4x the 129 MB L2). The CPU oracle
is timed on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

K = 5120
BITS = 4
ROWS = 16
QKV = (6144, 1024, 1024)
O_N = 5120
L2_BYTES = 129 * 1024 * 1024
METRIC = "EXL3 linear \u00b5s/call & weight-stream GB/s vs HBM roofline, rows 1/16/64/128"


def packed_bytes(Kk, N, bits):
    return Kk * N * bits // 8


STEP_WEIGHT_BYTES = sum(packed_bytes(K, n, BITS) for n in QKV) + packed_bytes(K, O_N, BITS)
STEP_WORKLOAD = ("decode rows at 27B shapes: q/k/v group (6144+1024+1024) + single 5120x5120, K=5120, "
                 "4-bit, 16 rows FP16")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        loaded = [v for v in sm if smax and v > 0.3 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, ws: int, device) -> float:
    """Max of a float over ranks (the slowest rank's time decides)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job(ms_local: float, steps: int, ws: int, device) -> tuple[float, float]:
    """Whole-job throughput of N replicas: every rank streams STEP_WEIGHT_BYTES
    per step, and the slowest rank's time over the timed steps decides.
    Returns (max ms over ranks, GB/s of all ranks together)."""
    ms_max = reduce_max(ms_local, ws, device)
    sec_per_step = ms_max / 1e3 / steps
    return ms_max, ws * STEP_WEIGHT_BYTES / sec_per_step / 1e9


# ---------------------------------------------------------------------------- CPU oracle leg

def _step_blocks():
    """The headline step's 128-column blocks in order: (member, N, block) for
    the q/k/v group's three weights and the single 5120 x 5120 weight."""
    return [(m, n, b) for m, n in enumerate(QKV + (O_N,)) for b in range(n // 128)]


def _step_inputs():
    """The step's four weights and x as rank 0 of the GPU arm draws them, in
    the oracle's FP64 form."""
    import numpy as np

    import oracle
    import synth
    seed = 1000
    members = []
    for m, n in enumerate(QKV + (O_N,)):
        members.append((synth.codes(seed, K, n, BITS, m), synth.suh(seed, K, m).astype(np.float64),
                        synth.svh(seed, n, m).astype(np.float64)))
    x = synth.as_f64(synth.activations(seed, ROWS, K, "f16"), "f16")
    oracle.lib()
    return members, x


def _oracle_block(inp, i):
    """The oracle as it stands on block i of the step (one call, its rotation included)."""
    import oracle
    members, x = inp
    m, n, b = _step_blocks()[i]
    codes, suh, svh = members[m]
    oracle.linear(codes, K, 128, BITS, suh, svh[128 * b:128 * b + 128], x, tile_row_stride=(n // 16) * 8 * BITS,
                  col_from=128 * b)


_W = {}


def _oracle_worker_init():
    _W["inp"] = _step_inputs()


def _oracle_worker_block(i):
    _oracle_block(_W["inp"], i)
    return i


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def oracle_sample(seconds_budget: float = 12.0):
    """Time the CPU oracle as it stands on two bounded samples of the headline
    step: one core walking the step's 128-column blocks in order (one oracle
    call per block), and every host core on the whole step (its 104 blocks
    spread over a pool of spawned worker processes, each running the
    single-threaded oracle on one block at a time)."""
    import multiprocessing as mp

    inp = _step_inputs()
    nblk = len(_step_blocks())
    times = []
    t_end = time.perf_counter() + seconds_budget / 2
    while True:
        t0 = time.perf_counter()
        _oracle_block(inp, len(times) % nblk)
        times.append(time.perf_counter() - t0)
        if (time.perf_counter() > t_end and len(times) >= 8) or len(times) >= nblk:
            break
    sec1 = statistics.median(times)
    gbs1 = packed_bytes(K, 128, BITS) / sec1 / 1e9
    cores = host_cores()
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_oracle_worker_init) as pool:
        pool.map(_oracle_worker_block, range(cores))  # warm: every worker has its inputs
        ptimes = []
        t_end = time.perf_counter() + seconds_budget / 2
        while True:
            t0 = time.perf_counter()
            pool.map(_oracle_worker_block, range(nblk), chunksize=1)
            ptimes.append(time.perf_counter() - t0)
            if time.perf_counter() > t_end or len(ptimes) >= 20:
                break
    secp = statistics.median(ptimes)
    gbsp = STEP_WEIGHT_BYTES / secp / 1e9
    return {"value": round(gbsp, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"the whole step (q/k/v group + 5120x5120, {ROWS} rows), its {nblk} column blocks spread over "
                      f"{cores} spawned processes each running the FP64 single-thread C oracle; median of "
                      f"{len(ptimes)} steps ({secp * 1e3:.1f} ms per step)",
            "single_core": {"value": round(gbs1, 5), "unit": "GB/s", "cores": 1,
                            "sample": f"the step's first {len(times)} 128-column blocks, {ROWS} rows, one core, "
                                      f"one oracle call each; median {sec1 * 1e3:.1f} ms per block"}}


def step_config(ws: int) -> dict:
    """The workload keys both arms report (the GPU arm adds how it times)."""
    return {"workload": STEP_WORKLOAD, "K": K, "bits": BITS, "rows": ROWS, "weights_per_step_bytes": STEP_WEIGHT_BYTES,
            "parallelism": f"replicas x{ws}"}


def run_reference(args):
    """The oracle as it stands, timed on the host's cores, on the headline
    step's workload: the same weights and x as rank 0 of the GPU arm, walked
    one 128-column block per oracle call through the step's 104 blocks (q, k,
    v, then the 5120 x 5120 weight; every block has the same K, so each is a
    fair sample of the step), as many blocks per step as keep the whole run at
    about 2000 calls."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp = _step_inputs()
    blocks = _step_blocks()
    per_step = max(1, min(len(blocks), 2000 // max(1, args.steps + args.warmup)))
    pos = [0]

    def step():
        for _ in range(per_step):
            _oracle_block(inp, pos[0] % len(blocks))
            pos[0] += 1

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    sec = (time.perf_counter() - t0) / args.steps
    gbs = per_step * packed_bytes(K, 128, BITS) / sec / 1e9
    sample = (f"{per_step} of the step's {len(blocks)} 128-column blocks per step (q/k/v group then the 5120x5120 "
              f"weight, in turn), {ROWS} rows; FP64 single-thread C oracle, one call per block")
    cfg = step_config(ws)
    cfg["l2"] = "n/a (host)"
    cfg["timing"] = "host wall clock over K steps after W warm-up steps"
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu": cpu_model(),
                             "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------- GPU leg

def run_gpu(args):
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build_library()
    import exl3_trellis_quantized_rot_gb300 as tfx
    import synth

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)

    # weights: enough distinct copies of the step's four weights to exceed 4x L2
    copies = max(2, -(-4 * L2_BYTES // STEP_WEIGHT_BYTES))

    def up(seed, N, member):
        codes = synth.codes(seed, K, N, BITS, member)
        t = torch.from_numpy(codes.view(np.int32)).to(dev)
        su = torch.from_numpy(synth.suh(seed, K, member).view(np.int16)).to(dev)
        sv = torch.from_numpy(synth.svh(seed, N, member).view(np.int16)).to(dev)
        return t, su, sv, N

    base = [up(1000 + rank, N, m) for m, N in enumerate(QKV)] + [up(1000 + rank, O_N, 3)]
    sets = []
    for c in range(copies):
        ws_c = []
        for (t, su, sv, N) in base:
            wc = tfx.Weight(t.clone(), su, sv, K, N, BITS, tfx.F16)  # same codes, distinct memory
            tfx.reserve(wc, 128, stream)
            ws_c.append(wc)
        sets.append(ws_c)
    x = torch.from_numpy(synth.activations(1000 + rank, ROWS, K, "f16")).to(dev)
    # the four outputs are consecutive slices of one buffer: one D2H copy per step
    y_all = torch.empty(ROWS * (sum(QKV) + O_N), dtype=torch.float16, device=dev)
    offs = np.cumsum([0] + [ROWS * n for n in QKV + (O_N,)])
    ys = [y_all[offs[i]:offs[i + 1]].view(ROWS, n) for i, n in enumerate(QKV)]
    yo = y_all[offs[3]:offs[4]].view(ROWS, O_N)

    def step(i, xin=x, rows=ROWS):
        q, k, v, o = sets[i % copies]
        tfx.group([q, k, v], xin[:rows], rows, [y[:rows] for y in ys], stream)
        tfx.linear(o, xin[:rows], rows, yo[:rows], stream)

    def capture(fn, n):
        """A CUDA graph of fn(0) .. fn(n-1) on the bench stream (the calls allocate nothing)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(i)
        return g

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # the timed region: exactly K steps, replayed from one CUDA graph (one
    # launch per kernel, no host work between them), weights resident in HBM
    n0 = tfx.launch_count()
    g_steps = capture(step, args.steps)
    launches = tfx.launch_count() - n0  # kernels of the library recorded into the timed graph
    g_steps.replay()  # untimed: first replay after instantiation
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # keep the GPU busy while the sampler starts, so the samples see the load
        t_end = time.perf_counter() + 0.5
        while time.perf_counter() < t_end:
            g_steps.replay()
            torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        g_steps.replay()
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    clocks = clk.summary()
    ms = start.elapsed_time(stop)
    ms_max, value = whole_job(ms, args.steps, ws, dev)
    sec_per_step = ms_max / 1e3 / args.steps
    del g_steps

    # roofline of the step. The ALU (decode) peak is measured here, in this run,
    # by the library's decode-rate probe: the decode rule plus one MMA per tile
    # at full occupancy on words from shared memory, no global traffic; best
    # of 5 timed launches on the bench stream.
    probe_w, probe_f = tfx.decode_rate(BITS, 4000)
    sink = torch.empty(probe_f, dtype=torch.float32, device=dev)
    probe_ms = []
    for i in range(6):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        tfx.decode_rate(BITS, 4000, sink, stream)
        b.record(stream)
        torch.cuda.synchronize()
        if i:
            probe_ms.append(a.elapsed_time(b))
    dec_peak = probe_w / (min(probe_ms) / 1e3) / 1e9

    def alg_bytes(Ns):
        # packed codes + x read + svh + y written
        return sum(packed_bytes(K, n, BITS) + 2 * ROWS * K + 2 * n + 2 * ROWS * n for n in Ns)

    # achieved over the whole timed step: two calls, each a rotation launch and
    # a linear launch; all of the step's time is charged to the linear kernels,
    # so this is a lower bound of the linear kernel's own rate
    hbm_achieved = (alg_bytes(QKV) + alg_bytes([O_N])) / sec_per_step / 1e9
    peak, peak_kind = load_peaks()
    dec_weights = sum(K * n for n in QKV) + K * O_N
    dec_achieved = dec_weights / sec_per_step / 1e9
    traffic = None
    tp = os.path.join(ROOT, "profiles", "linear_kernel_traffic.json")
    if os.path.exists(tp):
        d = json.load(open(tp))
        if d.get("kernel_source_sha256") == kernel_source_hash():
            traffic = d.get("bytes_per_launch_decode_rows_step")

    # end to end through the public API: every step copies its x from pinned
    # host memory to the device, runs the two calls and copies all four outputs
    # back to pinned host memory. The copies run on a second stream, double
    # buffered, so that step i's outputs travel back and step i+1's x travels in
    # while step i+1 (resp. step i) computes, the way a serving engine overlaps
    # transfers with compute; the K steps (and every copy) replay from one CUDA
    # graph and sit inside the timed region.
    copy_stream = torch.cuda.Stream(device=dev)
    xh = x.cpu().pin_memory()
    xds = [torch.empty_like(x) for _ in range(2)]
    ybufs = [torch.empty_like(y_all) for _ in range(2)]
    yhs = [torch.empty(y_all.numel(), dtype=torch.float16).pin_memory() for _ in range(2)]

    def views(buf):
        return ([buf[offs[i]:offs[i + 1]].view(ROWS, n) for i, n in enumerate(QKV)],
                buf[offs[3]:offs[4]].view(ROWS, O_N))

    yviews = [views(bf) for bf in ybufs]

    def e2e_steps(n_steps):
        ev = lambda: torch.cuda.Event()  # noqa: E731
        ev_h = [ev() for _ in range(n_steps)]
        ev_c = [ev() for _ in range(n_steps)]
        ev_d = [ev() for _ in range(n_steps)]
        fork = ev()
        fork.record(stream)
        copy_stream.wait_event(fork)
        with torch.cuda.stream(copy_stream):
            xds[0].copy_(xh, non_blocking=True)
            ev_h[0].record(copy_stream)
        for i in range(n_steps):
            bsel = i % 2
            stream.wait_event(ev_h[i])
            if i >= 2:
                stream.wait_event(ev_d[i - 2])  # outputs of step i-2 are on the host: reuse the buffer
            q, k, v, o = sets[i % copies]
            ysb, yob = yviews[bsel]
            tfx.group([q, k, v], xds[bsel], ROWS, ysb, stream)
            tfx.linear(o, xds[bsel], ROWS, yob, stream)
            ev_c[i].record(stream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < n_steps:
                    if i >= 1:
                        copy_stream.wait_event(ev_c[i - 1])  # x buffer (i+1)%2 was read by step i-1
                    xds[(i + 1) % 2].copy_(xh, non_blocking=True)
                    ev_h[i + 1].record(copy_stream)
                copy_stream.wait_event(ev_c[i])
                yhs[bsel].copy_(ybufs[bsel], non_blocking=True)
                ev_d[i].record(copy_stream)
        stream.wait_event(ev_d[n_steps - 1])  # join: the last outputs are on the host

    e2e_steps(3)
    torch.cuda.synchronize()
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        e2e_steps(args.steps)
    g_e2e.replay()
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g_e2e.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), ws, dev)
    e2e_value = ws * STEP_WEIGHT_BYTES / (e2e_ms / 1e3 / args.steps) / 1e9
    del g_e2e

    # per-shape µs/call (extra detail): each a CUDA graph of back-to-back calls
    # cycling through the weight copies
    detail = {}
    if not args.no_detail:

        def time_calls(fn, n_calls):
            for i in range(3):
                fn(i)
            torch.cuda.synchronize()
            g = capture(fn, n_calls)
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) * 1e3 / n_calls

        n_calls = 200
        for rows in (1, 7, 16):
            xr_ = x[:rows]
            detail[f"qkv_group_rows{rows}_us"] = round(time_calls(
                lambda i, xr_=xr_, rows=rows: tfx.group(sets[i % copies][:3], xr_, rows, [y[:rows] for y in ys], stream),
                n_calls), 3)
            detail[f"single_5120_rows{rows}_us"] = round(time_calls(
                lambda i, xr_=xr_, rows=rows: tfx.linear(sets[i % copies][3], xr_, rows, yo[:rows], stream),
                n_calls), 3)

        # layer chaining: the q/k/v group, then o_proj (K = 6144, N = 5120) on
        # q's output, at 16 rows: one by one, and as one tfx_exl3_chain with
        # and without programmatic dependent launch between the kernels
        o6 = []
        ocodes = torch.from_numpy(synth.codes(1500 + rank, 6144, O_N, BITS).view(np.int32)).to(dev)
        osu = torch.from_numpy(synth.suh(1500 + rank, 6144).view(np.int16)).to(dev)
        osv = torch.from_numpy(synth.svh(1500 + rank, O_N).view(np.int16)).to(dev)
        for c in range(copies):
            wc = tfx.Weight(ocodes.clone() if c else ocodes, osu, osv, 6144, O_N, BITS, tfx.F16)
            tfx.reserve(wc, 128, stream)
            o6.append(wc)
        yo6 = torch.empty((ROWS, O_N), dtype=torch.float16, device=dev)

        def unchained(i):
            q, k, v, _ = sets[i % copies]
            tfx.group([q, k, v], x, ROWS, ys, stream)
            tfx.linear(o6[i % copies], ys[0], ROWS, yo6, stream)

        def chained(i, pdl):
            q, k, v, _ = sets[i % copies]
            tfx.chain([([q, k, v], x, ys), ([o6[i % copies]], ys[0], [yo6])], ROWS, pdl=pdl, stream=stream)

        detail["chain_qkv_o_rows16_unchained_us"] = round(time_calls(unchained, n_calls), 3)
        detail["chain_qkv_o_rows16_pdl_off_us"] = round(time_calls(lambda i: chained(i, 0), n_calls), 3)
        detail["chain_qkv_o_rows16_pdl_on_us"] = round(time_calls(lambda i: chained(i, 1), n_calls), 3)
        detail["chain_qkv_o_rows16_pdl_auto_us"] = round(time_calls(lambda i: chained(i, 2), n_calls), 3)
        del o6, ocodes

        # mid rows on the 5120x5120 weight (same copies, reserved for 128 rows)
        x128 = torch.from_numpy(synth.activations(2000 + rank, 128, K, "f16")).to(dev)
        y128 = torch.empty((128, O_N), dtype=torch.float16, device=dev)
        for rows in (64, 128):
            us = time_calls(lambda i, rows=rows: tfx.linear(sets[i % copies][3], x128[:rows], rows, y128[:rows], stream),
                            n_calls)
            detail[f"single_5120_rows{rows}_us"] = round(us, 3)
            detail[f"single_5120_rows{rows}_tflops"] = round(2 * rows * K * O_N / us / 1e6, 1)

        # gate+up group (K = 5120, N = 17408 each, BF16 activations) at mid rows and a 4096-row chunk
        GU = 17408
        gu_bytes = 2 * packed_bytes(K, GU, BITS)
        gu_copies = max(2, -(-4 * L2_BYTES // gu_bytes))
        gbase = []
        for m in range(2):
            codes = synth.codes(3000 + rank, K, GU, BITS, m)
            gbase.append((torch.from_numpy(codes.view(np.int32)).to(dev),
                          torch.from_numpy(synth.suh(3000 + rank, K, m).view(np.int16)).to(dev),
                          torch.from_numpy(synth.svh(3000 + rank, GU, m).view(np.int16)).to(dev)))
        gsets = []
        for c in range(gu_copies):
            pair = []
            for (t, su, sv) in gbase:
                wc = tfx.Weight(t.clone() if c else t, su, sv, K, GU, BITS, tfx.BF16)
                tfx.reserve(wc, 128, stream)
                pair.append(wc)
            gsets.append(pair)
        xb = torch.from_numpy(synth.activations(3000 + rank, 128, K, "bf16").view(np.int16)).to(dev).view(torch.bfloat16)
        gys = [torch.empty((128, GU), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        for rows in (1, 16, 64, 128):
            us = time_calls(lambda i, rows=rows: tfx.group(gsets[i % gu_copies], xb[:rows], rows,
                                                           [y[:rows] for y in gys], stream), 40)
            detail[f"gate_up_rows{rows}_us"] = round(us, 3)
            detail[f"gate_up_rows{rows}_GBps"] = round(gu_bytes / us / 1e3, 1)
            detail[f"gate_up_rows{rows}_tflops"] = round(2 * rows * K * 2 * GU / us / 1e6, 1)
        del gsets

        # bit-width sweep: 5120 x 5120 at 1..8 bits, rows 1 and 64, packed bytes per second
        for bits in range(1, 9):
            wb = packed_bytes(K, O_N, bits)
            ncop = max(2, -(-4 * L2_BYTES // wb))
            codes = torch.from_numpy(synth.codes(5000 + bits, K, O_N, bits).view(np.int32)).to(dev)
            su = torch.from_numpy(synth.suh(5000 + bits, K).view(np.int16)).to(dev)
            sv = torch.from_numpy(synth.svh(5000 + bits, O_N).view(np.int16)).to(dev)
            bws = []
            for c in range(ncop):
                wc = tfx.Weight(codes.clone() if c else codes, su, sv, K, O_N, bits, tfx.F16)
                tfx.reserve(wc, 64, stream)
                bws.append(wc)
            for rows in (1, 64):
                us = time_calls(lambda i, rows=rows: tfx.linear(bws[i % ncop], x128[:rows], rows, y128[:rows], stream),
                                n_calls)
                detail[f"bits{bits}_5120_rows{rows}_us"] = round(us, 3)
                detail[f"bits{bits}_5120_rows{rows}_GBps"] = round(wb / us / 1e3, 1)
            del bws, codes

        # LM head, 6-bit, K = 5120, N = 248,320: the full head, the view of its first
        # 98,304 columns, and 64-block views (the last 64 blocks, and distinct 64-block
        # views of the same head cycled so that every call streams from HBM)
        HN, HB = 248320, 6
        hcodes = torch.from_numpy(synth.codes(6000, K, HN, HB).view(np.int32)).to(dev)
        hsu = torch.from_numpy(synth.suh(6000, K).view(np.int16)).to(dev)
        hsv = torch.from_numpy(synth.svh(6000, HN).view(np.int16)).to(dev)
        head = tfx.Weight(hcodes, hsu, hsv, K, HN, HB, tfx.F16)
        tfx.reserve(head, 16, stream)
        first = tfx.columns(head, 0, 98304)
        tfx.reserve(first, 16, stream)
        keep = HN - 240128 - 7904
        packs = []
        for j in range(4):
            pv = [tfx.columns(head, 0, 98304), tfx.columns(head, 240128, 8192)]
            for v in pv:
                tfx.reserve(v, 16, stream)
            packs.append(pv)
        yp_ = torch.empty((16, 98304 + keep), dtype=torch.float16, device=dev)
        tails = []
        for j in range(8):
            tv = tfx.columns(head, 240128 - j * 8192 * 3, 8192)
            tfx.reserve(tv, 16, stream)
            tails.append(tv)
        yh_ = torch.empty((16, HN), dtype=torch.float16, device=dev)
        yf_ = torch.empty((16, 98304), dtype=torch.float16, device=dev)
        yt_ = torch.empty((16, 8192), dtype=torch.float16, device=dev)
        for rows in (1, 8, 16):
            for name, fn, nbytes in (
                    ("full", lambda i, rows=rows: tfx.linear(head, x[:rows], rows, yh_[:rows], stream),
                     packed_bytes(K, HN, HB)),
                    ("first98304", lambda i, rows=rows: tfx.linear(first, x[:rows], rows, yf_[:rows], stream),
                     packed_bytes(K, 98304, HB)),
                    ("last64blocks", lambda i, rows=rows: tfx.linear(tails[i % len(tails)], x[:rows], rows,
                                                                     yt_[:rows], stream),
                     packed_bytes(K, 8192, HB)),
                    ("packed_spans", lambda i, rows=rows: tfx.pack_spans(packs[i % len(packs)], x[:rows],
                                                                         yp_[:rows], [0, 7904], rows, stream),
                     packed_bytes(K, 98304 + 8192, HB))):
                us = time_calls(fn, 20)
                detail[f"lm_head_{name}_rows{rows}_us"] = round(us, 3)
                detail[f"lm_head_{name}_rows{rows}_GBps"] = round(nbytes / us / 1e3, 1)
        del head, first, tails, packs, hcodes
        # trellis encoder: a seeded Gaussian 1024 x 1024 weight (4096 tiles,
        # std 1.155, the decode rule's value spread) on the value grid; per bit
        # width the GPU's tiles/s and the decoded weights' mean squared error
        EK = EN = 1024
        rng_e = np.random.default_rng(9000 + rank)
        tg = np.clip(np.rint(rng_e.normal(0.0, 1.155, (EK, EN)) * 128), -1024, 1023).astype(np.int16)
        t_tg = torch.from_numpy(tg).to(dev)
        for eb in range(1, 9):
            scr = torch.empty(tfx.encode_scratch_bytes(EK, EN, eb), dtype=torch.uint8, device=dev)
            tfx.encode(t_tg, eb, scratch=scr, stream=stream)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            _, err = tfx.encode(t_tg, eb, scratch=scr, stream=stream)
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            tiles = (EK // 16) * (EN // 16)
            detail[f"encode_bits{eb}_tiles_per_s"] = round(tiles / (ms / 1e3), 1)
            detail[f"encode_bits{eb}_mse"] = round(float(err.sum()) / (EK * EN) / 128 ** 2, 6)
            del scr
        del t_tg

        gate = tfx.Weight(gbase[0][0], gbase[0][1], gbase[0][2], K, GU, BITS, tfx.BF16)
        tfx.reserve(gate, 4096, stream)
        x4k = torch.from_numpy(synth.activations(4000 + rank, 4096, K, "bf16").view(np.int16)).to(dev).view(torch.bfloat16)
        y4k = torch.empty((4096, GU), dtype=torch.bfloat16, device=dev)
        us = time_calls(lambda i: tfx.linear(gate, x4k, 4096, y4k, stream), 5)
        detail["gate_rows4096_us"] = round(us, 1)
        detail["gate_rows4096_tflops"] = round(2 * 4096 * K * GU / us / 1e6, 1)
        torch.cuda.synchronize()

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        cpu = oracle_sample()
        if not args.no_detail:
            # the encoder's CPU oracle on a bounded sample: 4 tiles of the same
            # kind of weight at 4 bits, one core
            import oracle
            rng_c = np.random.default_rng(9100)
            tgc = np.clip(np.rint(rng_c.normal(0.0, 1.155, (32, 32)) * 128), -1024, 1023).astype(np.int16)
            t0 = time.perf_counter()
            oracle.encode(tgc, 32, 32, 4)
            detail["encode_bits4_cpu_oracle_tiles_per_s"] = round(4 / (time.perf_counter() - t0), 3)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(sec_per_step * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {**step_config(ws),
                       "l2": f"weights cycled through {copies} distinct copies "
                             f"({copies * STEP_WEIGHT_BYTES / 1e6:.0f} MB > 4x L2)",
                       "timing": "K steps replayed from one CUDA graph, CUDA events on the launching stream"},
            "us_per_step": round(sec_per_step * 1e6, 3),
            "detail": detail,
            "roofline": {"bound": "alu", "achieved": round(dec_achieved, 1), "peak": round(dec_peak, 1),
                         "unit": "G decoded weights/s", "frac": round(dec_achieved / dec_peak, 4), "traffic": traffic,
                         "kernel": "linear_warp_kernel<4,2,2> (decode rows; q/k/v group folded through global slabs "
                                   "and the combine kernel, 5120x5120 in its clusters), group + single call",
                         "timing": "whole timed step (rotation and combine launches included) per step",
                         "peak_source": f"measured in this run: tfx_exl3_debug_decode_rate probe ({probe_w / 1e9:.2f} "
                                        f"G weights per launch, best of 5 launches, {min(probe_ms) * 1e3:.1f} us)",
                         "hbm": {"achieved": round(hbm_achieved, 1), "peak": peak, "unit": "GB/s",
                                 "frac": round(hbm_achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs"}},
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": xh.numel() * 2,
                    "d2h_bytes_per_step": yhs[0].numel() * 2,
                    "how": "x copied in and all outputs copied out every step on a second stream, "
                           "double buffered and overlapped with compute, replayed from one CUDA graph"},
            "gpu_launches": int(launches),  # counted by the library while the K timed steps were captured
            "clocks": clocks,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_case(args):
    """A few calls of one workload on cuda:0 and nothing else (the command the
    ncu captures under profiles/ run): 'qkv_group_rows16' (q/k/v group,
    K = 5120, 4-bit, 16 rows), 'single_5120_rows16' (5120 x 5120, 4-bit, 16
    rows), 'lm_head_rows1' (5120 x 248,320, 6-bit, 1 row), 'gate_rows128'
    (5120 x 17408, 4-bit, 128 rows: the tensor-core kernel), 'encode_b4' (the
    trellis encoder, 1024 x 1024 at 4 bits) or 'decode_rate' (the decode-rate
    probe)."""
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build_library()
    import exl3_trellis_quantized_rot_gb300 as tfx
    import synth
    dev = torch.device("cuda", 0)

    def weight(seed, N, bits, member=0, copies=1):
        codes = torch.from_numpy(synth.codes(seed, K, N, bits, member).view(np.int32)).to(dev)
        su = torch.from_numpy(synth.suh(seed, K, member).view(np.int16)).to(dev)
        sv = torch.from_numpy(synth.svh(seed, N, member).view(np.int16)).to(dev)
        out = []
        for c in range(copies):
            w = tfx.Weight(codes.clone() if c else codes, su, sv, K, N, bits, tfx.F16)
            tfx.reserve(w, 16)
            out.append(w)
        return out

    x = torch.from_numpy(synth.activations(7, 128, K, "f16")).to(dev)
    if args.case == "encode_b4":
        # the trellis encoder on a seeded Gaussian 1024 x 1024 weight at 4 bits
        rng_e = np.random.default_rng(9000)
        tg = np.clip(np.rint(rng_e.normal(0.0, 1.155, (1024, 1024)) * 128), -1024, 1023).astype(np.int16)
        t_tg = torch.from_numpy(tg).to(dev)
        for i in range(2):
            words, err = tfx.encode(t_tg, 4)
        ys = [err.float()]
    elif args.case == "decode_rate":
        # the decode-rate probe (the ALU roofline of the bench line)
        nw, nf = tfx.decode_rate(BITS, 4000)
        sink = torch.empty(nf, dtype=torch.float32, device=dev)
        for i in range(3):
            tfx.decode_rate(BITS, 4000, sink)
        ys = [sink]
    elif args.case == "gate_rows128":
        ws_ = weight(8, 17408, BITS, copies=3)
        for w in ws_:
            tfx.reserve(w, 128)
        for i in range(6):
            ys = [tfx.linear(ws_[i % 3], x)]
    elif args.case == "qkv_group_rows16":
        ms = [weight(7, n, BITS, m, copies=6) for m, n in enumerate(QKV)]
        for i in range(20):
            ys = tfx.group([ms[0][i % 6], ms[1][i % 6], ms[2][i % 6]], x[:16])
    elif args.case == "single_5120_rows16":
        ws_ = weight(7, O_N, BITS, copies=8)
        for i in range(20):
            ys = [tfx.linear(ws_[i % 8], x[:16])]
    else:
        head = weight(6000, 248320, 6)[0]
        for i in range(4):
            ys = [tfx.linear(head, x[:1])]
    torch.cuda.synchronize()
    print(args.case, "ok", float(ys[0].float().abs().mean()))
    return 0


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("exl3_kernels.cuh", "exl3_host.cu", "exl3_bits.cu"):
        h.update(open(os.path.join(ROOT, "exl3_trellis_quantized_rot_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--no-detail", action="store_true", help="skip the per-row-count detail timings")
    ap.add_argument("--case", choices=["qkv_group_rows16", "single_5120_rows16", "lm_head_rows1", "gate_rows128",
                                       "encode_b4", "decode_rate"],
                    help="run a few calls of one workload and exit (for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.case:
        return run_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
