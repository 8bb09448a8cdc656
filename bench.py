"""Benchmark of the GB300 low-bit product library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-rows]
                    [--rows-only stream|decode|prefill]

Headline workload (the decode GEMV the metric is quoted on): Q2_0_g64 GEMV, 4096 x 4096 weights,
batch 1, q8_0 activations.  One step = one pass of the decode hot path over one token: q8_0
quantization of x [1][4096] followed by the GEMV of that activation against R = 64 distinct
4096 x 4096 weight matrices (302 MB of packed weights, more than the 129 MB L2, so every step
streams its weights from HBM), issued as one grouped call (lb_gemv_q2_0_g64_grouped: the 64
matrices share the activation, like q|k|v or gate|up).  The step is captured once in a CUDA graph
and replayed.  The same 64 GEMVs issued as 64 single-matrix launches are reported beside it.

value       packed-weight bytes streamed per second (whole job, all ranks), weights resident in HBM
e2e         the same metric through the public API with the token's activation copied from pinned
            host memory and the step's outputs copied back, inside the timed region
roofline    the dominant kernel (the GEMV) against the measured HBM copy bandwidth
cpu_baseline the CPU oracle, as it stands, on a bounded sample of the same workload
rows        the other hot-path rows (batch 8, Q1_0 / Q2_0_g64 Qwen3-8B-shaped token, planar
            BitNet-2B4T token with its bf16 head), each measured the same way, outside the timed
            region of the headline number

Under torchrun (N > 1) every rank runs its own replica of the workload (the path shards by
rows with no exchange, so no data-path collective is used); the timed region is bracketed by a
barrier and the max time over ranks is taken.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import re
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode GEMV packed-weight GB/s (% HBM peak); prefill GEMM int8 TOPS (% peak)"
WORKLOAD = "Q2_0_g64 GEMV 4096x4096, batch 1, q8_0 activations (N(0,1)), codes -1/0/+1 at 31/38/31 %"
N_ROT = 64
ROWS_K = 4096
ROWS_N = 4096


def scale_stride(K, qk):
    """Row stride of the repacked scale plane (K/QK rounded up to a multiple of 8)."""
    return (K // qk + 7) // 8 * 8


def q2_bytes(N, K):
    return N * (K // 64) * 18


def q1_bytes(N, K):
    return N * (K // 128) * 18


def trit_bytes(N, K):
    """Planar ternary weights: one 16-byte {pos, neg} beat per 64 columns of a row."""
    return N * (K // 64) * 16


def bf16_bytes(N, K):
    return N * K * 2


def peaks(tensor: bool = False):
    """HBM GB/s (or, with tensor=True, dense bf16 TFLOP/s burst) and whether it was measured."""
    key, fallback = ("bf16_tflops", 1900.0) if tensor else ("hbm_gbs", 6800.0)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p[key]), "measured"
    except Exception:
        return fallback, "fallback"


# ---------------------------------------------------------------------------------------------
# distributed plumbing (barrier + max over ranks only)
# ---------------------------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix=f"lb_clocks_rank{self.index}_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if not self.proc:
            out["reasons"] = ["nvidia-smi unavailable"]
            return out
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if sm:
            out.update(sm_mhz=statistics.median(sm), sm_max_mhz=max(mx), samples=len(sm))
        out["reasons"] = sorted(reasons)
        return out


# ---------------------------------------------------------------------------------------------
# profile summary: DRAM traffic of the dominant kernel, valid only for the source it measured
# ---------------------------------------------------------------------------------------------
def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for name in ("lb_stream.cuh", "lb_gemv_q.cuh", "lb_gemv_q2.cu", "lb_common.cuh"):
        with open(os.path.join(ROOT, "bit_matvec_lb_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(path_name: str):
    path = os.path.join(ROOT, "profiles", path_name)
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.]+)\s+source_sha:\s*([0-9a-f]+)", text)
    if not m or m.group(2) != kernel_source_sha():
        return None
    return float(m.group(1))


# ---------------------------------------------------------------------------------------------
# CPU oracle baseline (bounded sample, all host cores, rows split across threads)
# ---------------------------------------------------------------------------------------------
def oracle_gbs(blocks_np: np.ndarray, q, dx, budget_s: float, qk: int = 64, threads=None):
    import oracle
    fn = oracle.q2_0_g64_product if qk == 64 else oracle.q1_0_product
    cores = threads or len(os.sched_getaffinity(0))
    N = blocks_np.shape[0]
    chunks = [blocks_np[i:i + max(1, N // cores)] for i in range(0, N, max(1, N // cores))]
    fn(blocks_np[:8], q, dx, want_isum=False)  # build / warm
    done_rows = 0
    t0 = time.perf_counter()
    reps = 0
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        while True:
            list(ex.map(lambda c: fn(c, q, dx, want_isum=False), chunks))
            reps += 1
            done_rows += N
            if time.perf_counter() - t0 >= budget_s:
                break
    dt = time.perf_counter() - t0
    K = q.shape[1]
    nbytes = done_rows * (K // qk) * 18
    return nbytes / dt / 1e9, cores, reps, dt


# ---------------------------------------------------------------------------------------------
# GPU workload helpers
# ---------------------------------------------------------------------------------------------
class Graph:
    """Capture a sequence of library calls once and replay it."""

    def __init__(self, fn, stream):
        import torch
        self.g = torch.cuda.CUDAGraph()
        self.stream = stream
        with torch.cuda.stream(stream):
            fn()  # warm (also sets kernel attributes outside capture)
        torch.cuda.synchronize()
        with torch.cuda.graph(self.g, stream=stream):
            fn()

    def replay(self):
        self.g.replay()


def time_graph(graph: Graph, reps: int, warm: int = 3) -> float:
    """Average ms per replay, CUDA events on the capture stream."""
    import torch
    for _ in range(warm):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(graph.stream):
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def read_probe(stream, nbytes: int = 1 << 30, reps: int = 10):
    """Read-only HBM bandwidth in this process: torch's sum over a 1 GiB buffer (a library
    kernel, reads only), beside the measured copy peak that the roofline divides by."""
    import torch
    try:
        buf = torch.ones(nbytes // 4, dtype=torch.float32, device="cuda")
        with torch.cuda.stream(stream):
            for _ in range(3):
                buf.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                buf.sum()
            e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        del buf
        return {"GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                "what": "torch.sum over 1 GiB fp32 (read only), CUDA events, same process"}
    except Exception as e:  # the probe is context; it never fails the bench line
        return {"error": f"{type(e).__name__}: {e}"[:200]}


def make_q2_weights(N, K, seed, device="cuda"):
    """Random Q2_0_g64 weights in the repacked layout (code plane + fp16 scale plane)."""
    import synth
    codes = synth.device_q2_codes_packed(N * K // 4, seed, device=device)
    scales = synth.device_fp16_scales(N * scale_stride(K, 64), seed + 7919, device=device)
    return codes, scales


def make_q1_weights(N, K, seed, device="cuda"):
    import synth
    bits = synth.device_bytes(N * K // 8, seed, device=device)
    scales = synth.device_fp16_scales(N * scale_stride(K, 128), seed + 7919, device=device)
    return bits, scales


def headline(lb, args, dist, out):
    import torch
    import synth
    import oracle

    N, K = ROWS_N, ROWS_K
    stream = torch.cuda.Stream()
    # weights: AoS source blocks generated on the device, split by the library's repack
    W = []
    for r in range(N_ROT):
        aos_codes = synth.device_q2_codes_packed(N * K // 4, seed=1000 * (dist.rank + 1) + r)
        aos_scales = synth.device_fp16_scales(N * K // 64, seed=2000 * (dist.rank + 1) + r)
        aos = torch.empty((N * K // 64, 18), dtype=torch.uint8, device="cuda")
        aos[:, 0:2] = aos_scales.view(torch.uint8).view(-1, 2)
        aos[:, 2:] = aos_codes.view(-1, 16)
        codes = torch.empty(N * K // 4, dtype=torch.uint8, device="cuda")
        scales = torch.empty(N * scale_stride(K, 64), dtype=torch.int16, device="cuda")
        lb.lb_repack_q2_0_g64(aos, N, K, codes, scales)
        W.append((codes, scales, aos if r == 0 else None))
    torch.cuda.synchronize()
    x_np = synth.activations(1, K, seed=1)
    x = torch.from_numpy(x_np).cuda()
    q = torch.empty((1, K), dtype=torch.int8, device="cuda")
    d = torch.empty((1, K // 32), dtype=torch.int16, device="cuda")
    Y = torch.empty((N_ROT, 1, N), dtype=torch.float32, device="cuda")

    group = [(W[r][0], W[r][1], Y[r], None, N) for r in range(N_ROT)]

    def step():
        lb.lb_quantize_q8_0(x, q, d, 1, K, stream=stream)
        lb.lb_gemv_q2_0_g64_grouped(group, q, d, K, 1, stream=stream)

    def gemvs_only():
        lb.lb_gemv_q2_0_g64_grouped(group, q, d, K, 1, stream=stream)

    def gemvs_single():
        for r in range(N_ROT):
            lb.lb_gemv_q2_0_g64(W[r][0], W[r][1], q, d, Y[r], None, N, K, 1, stream=stream)

    g_step = Graph(step, stream)
    g_gemv = Graph(gemvs_only, stream)

    # sanity: sampled rows of copy 0 against the oracle (outside any timed region)
    torch.cuda.synchronize()
    blocks0 = W[0][2].cpu().numpy().reshape(N, K // 64, 18)
    q_ref, d_ref = oracle.quantize_q8_0(x_np)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    rows = np.arange(0, N, 257)
    ref = oracle.q2_0_g64_product(blocks0[rows], q_ref, d_ref, want_isum=False)
    err = np.abs(Y[0].cpu().numpy()[:, rows].astype(np.float64) - ref.y_exact)
    assert np.all(err <= ref.tolerance()), "GPU output outside the oracle bound"

    # ---- timed region (the warm-up follows the clock sampler's start-up pause, so the GPU is
    #      not idle when the first timed step begins) ----
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(args.steps):
            g_step.replay()
        e1.record()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = dist.max(e0.elapsed_time(e1) / args.steps)
    step_bytes = N_ROT * q2_bytes(N, K)
    value = step_bytes * dist.world / (ms * 1e-3) / 1e9

    # ---- roofline: the grouped GEMV launch alone, average duration over the same graph ----
    hbm, peak_kind = peaks()
    ms_gemv = time_graph(g_gemv, reps=max(50, args.steps // 4))
    # weights and scales of 64 matrices + the q8_0 activation + 64 output rows
    alg_bytes = N_ROT * (q2_bytes(N, K) + 4 * N) + (K + K // 16)
    achieved = alg_bytes / (ms_gemv * 1e-3) / 1e9
    ms_single = time_graph(Graph(gemvs_single, stream), reps=max(20, args.steps // 20)) / N_ROT
    traffic = profiled_traffic("stream_gemv_q2_0_g64_4096x4096_b1.md")
    probe = read_probe(stream)

    # ---- e2e: pinned host activation in, outputs out, every step ----
    # Two buffer sets alternate between steps: while step i computes on `stream`, a copy stream
    # reads step i-1's outputs back and uploads step i+1's activation (each step still moves its
    # own activation in and its own outputs out; events order every reuse of a buffer).
    x_host = torch.from_numpy(x_np).pin_memory()
    y_host = [torch.empty((N_ROT, 1, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    xs = [x, torch.empty_like(x)]
    Ys = [Y, torch.empty_like(Y)]
    qs2 = [q, torch.empty_like(q)]
    ds2 = [d, torch.empty_like(d)]

    def step_set(b):
        def f():
            lb.lb_quantize_q8_0(xs[b], qs2[b], ds2[b], 1, K, stream=stream)
            lb.lb_gemv_q2_0_g64_grouped([(W[r][0], W[r][1], Ys[b][r], None, N)
                                         for r in range(N_ROT)], qs2[b], ds2[b], K, 1,
                                        stream=stream)
        return f
    g_sets = [Graph(step_set(0), stream), Graph(step_set(1), stream)]
    cstream = torch.cuda.Stream()
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]
    ev_h2d = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        with torch.cuda.stream(cstream):
            for b in range(2):
                xs[b].copy_(x_host, non_blocking=True)
                ev_h2d[b].record(cstream)
                ev_d2h[b].record(cstream)
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(stream):
                stream.wait_event(ev_h2d[b])
                stream.wait_event(ev_d2h[b])
                g_sets[b].replay()
                ev_comp[b].record(stream)
            with torch.cuda.stream(cstream):
                cstream.wait_event(ev_comp[b])
                y_host[b].copy_(Ys[b], non_blocking=True)
                ev_d2h[b].record(cstream)
                xs[b].copy_(x_host, non_blocking=True)  # the activation of step i + 2
                ev_h2d[b].record(cstream)
        stream.wait_stream(cstream)

    e2e_steps = max(20, args.steps // 4)
    e2e_run(3)
    torch.cuda.synchronize()
    dist.barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        f0.record()
    e2e_run(e2e_steps)
    with torch.cuda.stream(stream):
        f1.record()
    torch.cuda.synchronize()
    ms_e2e = dist.max(f0.elapsed_time(f1) / e2e_steps)
    # the last step's outputs came back intact
    last = (e2e_steps - 1) & 1
    assert np.array_equal(y_host[last].numpy(), Ys[last].cpu().numpy())

    out.update({
        "value": round(value, 2), "ms_per_step": round(ms, 5),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": traffic,
                     "peak_kind": peak_kind,
                     "kernel": "stream_gemv_kernel<Q2_0_g64, B=1> (64-matrix grouped launch)",
                     "alg_bytes_per_launch": alg_bytes, "avg_launch_us": round(ms_gemv * 1e3, 3)},
        "e2e": {"value": round(step_bytes * dist.world / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(x_host.numel() * 4),
                "d2h_bytes_per_step": int(y_host[0].numel() * 4),
                "pipelined": "two buffer sets; copies of neighbouring steps overlap compute"},
        "clocks": clocks,
        "gpu_launches": int(args.steps * 2),
        "pct_hbm": round(100 * value / dist.world / hbm, 2),
        "read_probe": dict(probe, **({"gemv_launch_frac": round(achieved / probe["GB/s"], 4)}
                                     if "GB/s" in probe else {})),
        "single_launch": {"GB/s": round(q2_bytes(N, K) / (ms_single * 1e-3) / 1e9, 1),
                          "us_per_gemv": round(ms_single * 1e3, 3),
                          "note": "the same 64 GEMVs as 64 single-matrix launches (PDL-chained)"},
    })

    if dist.rank == 0:
        q_ref2 = q_ref
        gbs, cores, reps, dt = oracle_gbs(blocks0[:512], q_ref2, d_ref, budget_s=args.cpu_budget)
        gbs1, _, reps1, dt1 = oracle_gbs(blocks0[:64], q_ref2, d_ref,
                                         budget_s=max(1.0, args.cpu_budget / 4), threads=1)
        out["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                               "kind": "oracle",
                               "sample": f"rows 0..511 of one 4096x4096 Q2_0_g64 matrix, batch 1, "
                                         f"rows split over {cores} threads, {reps} passes in "
                                         f"{dt:.1f} s",
                               "single_thread": {"value": round(gbs1, 4), "unit": "GB/s",
                                                 "cores": 1,
                                                 "sample": f"rows 0..63, {reps1} passes in "
                                                           f"{dt1:.1f} s"}}
    del W, g_step, g_gemv
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------------------------
# other rows of the hot path (outside the headline timed region)
# ---------------------------------------------------------------------------------------------
def rows_measure(lb, out, which: str = "all"):
    import torch
    import synth
    stream = torch.cuda.Stream()
    rows = {}
    if which == "stream":
        rows_stream(lb, rows, stream)
    if which in ("all", "decode"):
        rows_stream(lb, rows, stream)
        rows_decode(lb, rows, stream)
        rows_dequant(lb, rows, stream)
        rows_base3(lb, rows, stream)
    if which in ("all", "prefill"):
        rows_prefill(lb, rows, stream)
        rows_tensor_rates(rows)
    out["rows"] = rows


def rows_stream(lb, rows, stream):
    import torch
    import synth
    hbm, _ = peaks()

    # (0) one token, the other two formats: 64 distinct 4096 x 4096 matrices per grouped launch
    #     (rotated past L2), quantizer + GEMV per step, beside the Q2_0_g64 headline
    probe = read_probe(stream)
    N, K = ROWS_N, ROWS_K
    x1 = torch.from_numpy(synth.activations(1, K, seed=1)).cuda()
    q1 = torch.empty((1, K), dtype=torch.int8, device="cuda")
    d1 = torch.empty((1, K // 32), dtype=torch.int16, device="cuda")
    s1 = torch.empty((1,), dtype=torch.float32, device="cuda")
    Y1 = torch.empty((N_ROT, 1, N), dtype=torch.float32, device="cuda")
    for fmt in ("q1_0", "planar"):
        if fmt == "q1_0":
            W1 = [make_q1_weights(N, K, 51_000 + r) for r in range(N_ROT)]
            wbytes = q1_bytes(N, K)
            grp = [(W1[r][0], W1[r][1], Y1[r], None, N) for r in range(N_ROT)]

            def quant():
                lb.lb_quantize_q8_0(x1, q1, d1, 1, K, stream=stream)

            def gemv():
                lb.lb_gemv_q1_0_grouped(grp, q1, d1, K, 1, stream=stream)
            act = K + K // 16
        else:
            W1 = [synth.device_trit_planes(N, K, 52_000 + r) for r in range(N_ROT)]
            wbytes = trit_bytes(N, K)
            grp = [(W1[r], 0.02, Y1[r], None, N) for r in range(N_ROT)]

            def quant():
                lb.lb_quantize_i8_absmax(x1, q1, s1, 1, K, stream=stream)

            def gemv():
                lb.lb_gemv_trit_planes_grouped(grp, q1, s1, K, 1, stream=stream)
            act = K + 4

        def step1():
            quant()
            gemv()
        ms = time_graph(Graph(step1, stream), reps=50)
        ms_g = time_graph(Graph(gemv, stream), reps=50)
        gbs = N_ROT * wbytes / (ms * 1e-3) / 1e9
        launch = (N_ROT * (wbytes + 4 * N) + act) / (ms_g * 1e-3) / 1e9
        rows[f"{fmt}_4096x4096_b1"] = {
            "GB/s": round(gbs, 1), "pct_hbm": round(100 * gbs / hbm, 1),
            "launch_GB/s": round(launch, 1), "launch_pct_hbm": round(100 * launch / hbm, 1),
            "launch_frac_of_read_probe": (round(launch / probe["GB/s"], 4)
                                          if "GB/s" in probe else None),
            "weights_per_step": f"{N_ROT} distinct {N}x{K} matrices, {N_ROT * wbytes} B"}
        del W1, grp
        torch.cuda.empty_cache()


def rows_decode(lb, rows, stream):
    import torch
    import synth
    hbm, _ = peaks()

    # (1) config 2 at batch 8
    N, K, B = ROWS_N, ROWS_K, 8
    W = [make_q2_weights(N, K, 50_000 + r) for r in range(N_ROT)]
    x = torch.from_numpy(synth.activations(B, K, seed=1)).cuda()
    q = torch.empty((B, K), dtype=torch.int8, device="cuda")
    d = torch.empty((B, K // 32), dtype=torch.int16, device="cuda")
    Y = torch.empty((N_ROT, B, N), dtype=torch.float32, device="cuda")

    group8 = [(W[r][0], W[r][1], Y[r], None, N) for r in range(N_ROT)]

    def step_b8():
        lb.lb_quantize_q8_0(x, q, d, B, K, stream=stream)
        lb.lb_gemv_q2_0_g64_grouped(group8, q, d, K, B, stream=stream)
    ms = time_graph(Graph(step_b8, stream), reps=50)
    gbs = N_ROT * q2_bytes(N, K) / (ms * 1e-3) / 1e9
    rows["q2_0_g64_4096x4096_b8"] = {"GB/s": round(gbs, 1), "pct_hbm": round(100 * gbs / hbm, 1),
                                     "us_per_gemv": round(ms * 1e3 / N_ROT, 3)}
    del W, Y
    torch.cuda.empty_cache()

    # (2) Qwen3-8B-shaped decode token, Q1_0 and Q2_0_g64, batch 1 (252 GEMVs in 144 grouped
    #     launches and 144 quantizations, 36 layers)
    for fmt in ("q2_0_g64", "q1_0"):
        make = make_q2_weights if fmt == "q2_0_g64" else make_q1_weights
        grouped = (lb.lb_gemv_q2_0_g64_grouped if fmt == "q2_0_g64"
                   else lb.lb_gemv_q1_0_grouped)
        nbytes = q2_bytes if fmt == "q2_0_g64" else q1_bytes
        layers = []
        total = 0
        for layer in range(synth.QWEN3_8B_LAYERS):
            proj = []
            for p, (name, n, k) in enumerate(synth.QWEN3_8B_PROJ):
                proj.append((make(n, k, synth.proj_seed(60_000, layer, p)), n, k))
                total += nbytes(n, k)
            layers.append(proj)
        xs = {k: torch.from_numpy(synth.activations(1, k, seed=k)).cuda() for k in (4096, 12288)}
        qs = {k: torch.empty((1, k), dtype=torch.int8, device="cuda") for k in (4096, 12288)}
        ds = {k: torch.empty((1, k // 32), dtype=torch.int16, device="cuda") for k in (4096, 12288)}
        ybufs = [torch.empty(12288, dtype=torch.float32, device="cuda") for _ in range(7)]
        # q|k|v and gate|up read the same activation: one grouped call each
        groups = [(0, 1, 2), (3,), (4, 5), (6,)]

        def token():
            for proj in layers:
                for gi, members in enumerate(groups):
                    k = proj[members[0]][2]
                    # every group reads a new activation (attention input, attention output,
                    # FFN input, FFN mid), quantized just before it
                    lb.lb_quantize_q8_0(xs[k], qs[k], ds[k], 1, k, stream=stream)
                    mats = [(proj[i][0][0], proj[i][0][1], ybufs[i], None, proj[i][1])
                            for i in members]
                    grouped(mats, qs[k], ds[k], k, 1, stream=stream)
        ms = time_graph(Graph(token, stream), reps=20)
        gbs = total / (ms * 1e-3) / 1e9
        rows[f"qwen3_8b_token_{fmt}_b1"] = {"GB/s": round(gbs, 1), "pct_hbm": round(100 * gbs / hbm, 1),
                                            "ms_per_token": round(ms, 4), "bytes": total,
                                            "launches": 36 * 8}
        del layers
        torch.cuda.empty_cache()

    # (3) BitNet-2B4T-shaped token: planar body (210 GEMVs) + bf16 head 128256x2560, B=1 and 8
    body = []
    body_bytes = 0
    for layer in range(synth.BITNET_2B4T_LAYERS):
        for p, (name, n, k) in enumerate(synth.BITNET_2B4T_PROJ):
            planes = synth.device_trit_planes(n, k, synth.proj_seed(70_000, layer, p))
            body.append((planes, n, k))
            body_bytes += trit_bytes(n, k)
    HN, HK = synth.BITNET_HEAD
    head = synth.device_bytes(bf16_bytes(HN, HK), 80_000).view(torch.int16)
    head = (head & 0x3FFF) | 0x3C00  # finite bf16 patterns
    for B in (1, 8):
        x = torch.from_numpy(synth.activations(B, 6912, seed=2)).cuda()
        xq = {k: (torch.empty((B, k), dtype=torch.int8, device="cuda"),
                  torch.empty((B,), dtype=torch.float32, device="cuda")) for k in (2560, 6912)}
        xh = torch.from_numpy(synth.activations(B, HK, seed=3)).cuda()
        ybs = [torch.empty((B, 6912), dtype=torch.float32, device="cuda") for _ in range(7)]
        yh = torch.empty((B, HN), dtype=torch.float32, device="cuda")
        x2560 = x[:, :2560].contiguous()
        groups = [(0, 1, 2), (3,), (4, 5), (6,)]

        def token_bitnet():
            for layer in range(synth.BITNET_2B4T_LAYERS):
                proj = body[7 * layer: 7 * layer + 7]
                for gi, members in enumerate(groups):
                    k = proj[members[0]][2]
                    src = x2560 if k == 2560 else x  # a new activation for every group
                    lb.lb_quantize_i8_absmax(src, xq[k][0], xq[k][1], B, k, stream=stream)
                    mats = [(proj[i][0], 0.02, ybs[i], None, proj[i][1]) for i in members]
                    lb.lb_gemv_trit_planes_grouped(mats, xq[k][0], xq[k][1], k, B,
                                                   stream=stream)
            lb.lb_gemv_bf16(head, xh, yh, HN, HK, B, stream=stream)

        def head_only():
            lb.lb_gemv_bf16(head, xh, yh, HN, HK, B, stream=stream)

        ms = time_graph(Graph(token_bitnet, stream), reps=20)
        ms_head = time_graph(Graph(head_only, stream), reps=20)
        tot = body_bytes + bf16_bytes(HN, HK)
        rows[f"bitnet_2b4t_token_b{B}"] = {
            "GB/s": round(tot / (ms * 1e-3) / 1e9, 1), "pct_hbm": round(100 * tot / (ms * 1e-3) / 1e9 / hbm, 1),
            "ms_per_token": round(ms, 4), "bytes": tot,
            "head_GB/s": round(bf16_bytes(HN, HK) / (ms_head * 1e-3) / 1e9, 1),
            "body_GB/s": round(body_bytes / ((ms - ms_head) * 1e-3) / 1e9, 1)}


def rows_dequant(lb, rows, stream):
    import torch
    import synth
    hbm, _ = peaks()
    # (6) load-time dequantization, HBM-bound: 16 distinct 4096 x 4096 matrices per pass
    #     (> L2), Q2_0_g64 and planar, to fp32 and bf16, each into its own output buffer (so
    #     the written bytes leave the L2 too); bytes = packed weights + scales read + outputs
    #     written
    N, K, R = ROWS_N, ROWS_K, 16
    Wq = [make_q2_weights(N, K, 96_000 + r) for r in range(R)]
    Wt = [synth.device_trit_planes(N, K, 97_000 + r) for r in range(R)]
    for fmt, esz in ((lb.OUT_F32, 4), (lb.OUT_BF16, 2)):
        outs = [torch.empty((N, K), dtype=torch.float32 if esz == 4 else torch.int16,
                            device="cuda") for _ in range(R)]
        name = "f32" if esz == 4 else "bf16"

        def q2pass():
            for (c, s), out in zip(Wq, outs):
                lb.lb_dequantize_q2_0_g64(c, s, N, K, fmt, out, stream=stream)

        def tpass():
            for t, out in zip(Wt, outs):
                lb.lb_dequantize_trit_planes(t, 0.02, N, K, fmt, out, stream=stream)
        for label, fn, wbytes in (("q2_0_g64", q2pass, q2_bytes(N, K) + N * scale_stride(K, 64) * 2 - N * (K // 64) * 2),
                                  ("trit_planes", tpass, trit_bytes(N, K))):
            ms = time_graph(Graph(fn, stream), reps=20) / R
            gbs = (wbytes + N * K * esz) / (ms * 1e-3) / 1e9
            rows[f"dequant_{label}_4096x4096_{name}"] = {
                "GB/s": round(gbs, 1), "pct_hbm": round(100 * gbs / hbm, 1),
                "us_per_matrix": round(ms * 1e3, 2)}
        del outs
    del Wq, Wt
    torch.cuda.empty_cache()


def rows_base3(lb, rows, stream):
    import torch
    import synth
    hbm, _ = peaks()
    # (7) base-3 packing (five trits per byte) against the planar layout on the same trits:
    #     8 distinct 16384 x 8192 ternary matrices per pass (> L2), per-token int8 activations,
    #     1 and 8 tokens; GB/s counts each layout's own packed bytes
    N, K, R = 16384, 8192, 8
    planes = [synth.device_trit_planes(N, K, 98_000 + r) for r in range(R)]
    packed = []
    for t in planes:
        b3 = torch.empty((N, lb.base3_row_bytes(K)), dtype=torch.uint8, device="cuda")
        lb.lb_pack_base3(t, N, K, b3, stream=stream)
        packed.append(b3)
    torch.cuda.synchronize()
    pbytes, bbytes = N * K // 4, N * lb.base3_row_bytes(K)
    out = {}
    for B in (1, 8):
        x = torch.from_numpy(synth.activations(B, K, seed=5)).cuda()
        q = torch.empty((B, K), dtype=torch.int8, device="cuda")
        xs = torch.empty((B,), dtype=torch.float32, device="cuda")
        lb.lb_quantize_i8_absmax(x, q, xs, B, K)
        y = torch.empty((B, N), dtype=torch.float32, device="cuda")

        def b3pass():
            for w in packed:
                lb.lb_gemv_base3(w, 0.02, q, xs, y, None, N, K, B, stream=stream)

        def plpass():
            for w in planes:
                lb.lb_gemv_trit_planes(w, 0.02, q, xs, y, None, N, K, B, stream=stream)
        ms3 = time_graph(Graph(b3pass, stream), reps=20) / R
        msp = time_graph(Graph(plpass, stream), reps=20) / R
        out[f"b{B}"] = {"base3_us": round(ms3 * 1e3, 2), "planar_us": round(msp * 1e3, 2),
                        "base3_GB/s": round(bbytes / (ms3 * 1e-3) / 1e9, 1),
                        "planar_GB/s": round(pbytes / (msp * 1e-3) / 1e9, 1),
                        "base3_pct_hbm": round(100 * bbytes / (ms3 * 1e-3) / 1e9 / hbm, 1),
                        "planar_time_over_base3": round(msp / ms3, 3)}
    out["bytes_per_matrix"] = {"base3": bbytes, "planar": pbytes}
    rows["base3_vs_planar_16384x8192"] = out
    del planes, packed
    torch.cuda.empty_cache()


def rows_tensor_rates(rows):
    """Dense instruction rates of the tensor-core forms an exact prefill GEMM could use, measured
    on this GPU by the probe library (one CTA per SM, operands resident, back-to-back MMAs)."""
    import ctypes
    from bit_matvec_lb_gb300 import build as lbbuild
    try:
        probe = ctypes.CDLL(lbbuild.PROBE_LIB)
    except OSError as e:
        rows["tensor_rates_probe"] = {"unavailable": str(e)}
        return
    probe.lbp_tensor_rates.restype = ctypes.c_int
    probe.lbp_tensor_rates.argtypes = [ctypes.POINTER(ctypes.c_double)]
    r = (ctypes.c_double * 4)()
    st = probe.lbp_tensor_rates(r)
    tflops, _ = peaks(tensor=True)
    names = ["tcgen05_f16_m128n256k16", "tcgen05_f8f6f4_e4m3_m128n256k32",
             "mma_sync_f16_m16n8k16", "mma_sync_s8_m16n8k32"]
    rows["tensor_rates_probe"] = {
        "status": st,
        **{n: {"TFLOP/s": round(v / 1e12, 1), "frac_of_bf16_peak": round(v / 1e12 / tflops, 3)}
           for n, v in zip(names, r)},
        "note": "dense 2MNK per MMA, one CTA per SM, zero operands resident; the exact GEMMs run "
                "kind::f16 (the integer kinds are not available), so its rate and the measured "
                "cuBLAS bf16 figure are the prefill denominators"}


def rows_prefill(lb, rows, stream):
    import torch
    import synth
    # (4) Qwen3-8B-shaped prefill: 512 tokens through one layer's seven projections, Q1_0 and
    #     Q2_0_g64 (q8_0 quantization of the three distinct activations + seven GEMMs per pass)
    M = synth.PREFILL_M
    tflops, _ = peaks(tensor=True)
    xs = {k: torch.from_numpy(synth.activations(M, k, seed=10 + k)).cuda() for k in (4096, 12288)}
    qs = {k: torch.empty((M, k), dtype=torch.int8, device="cuda") for k in (4096, 12288)}
    ds = {k: torch.empty((M, k // 32), dtype=torch.int16, device="cuda") for k in (4096, 12288)}
    ws = torch.empty(lb.lb_gemm_workspace_bytes(M, 12288), dtype=torch.uint8, device="cuda")
    ops = 2 * M * sum(n * k for _, n, k in synth.QWEN3_8B_PROJ)
    # q|k|v and gate|up read the same activation: one grouped GEMM each
    groups = [(0, 1, 2), (3,), (4, 5), (6,)]
    for fmt in ("q2_0_g64", "q1_0"):
        make = make_q2_weights if fmt == "q2_0_g64" else make_q1_weights
        gemm = lb.lb_gemm_q2_0_g64_grouped if fmt == "q2_0_g64" else lb.lb_gemm_q1_0_grouped
        proj = [(make(n, k, synth.proj_seed(90_000, 0, i)), n, k)
                for i, (_, n, k) in enumerate(synth.QWEN3_8B_PROJ)]
        ys = [torch.empty((M, n), dtype=torch.float32, device="cuda") for _, n, _ in proj]

        def layer():
            # one q8_0 per group: attention input, attention output, FFN input, FFN mid
            for members in groups:
                k = proj[members[0]][2]
                lb.lb_quantize_q8_0(xs[k], qs[k], ds[k], M, k, stream=stream)
                gemm([(proj[i][0][0], proj[i][0][1], ys[i], proj[i][1]) for i in members],
                     qs[k], ds[k], M, k, ws, stream=stream)
        ms = time_graph(Graph(layer, stream), reps=20)
        tops = ops / (ms * 1e-3) / 1e12
        rows[f"qwen3_8b_prefill_m512_{fmt}"] = {
            "TOPS": round(tops, 1), "pct_tensor_peak": round(100 * tops / tflops, 1),
            "ms_per_layer": round(ms, 4), "int8_equivalent_ops": ops,
            "peak": f"{tflops} TFLOP/s dense bf16/f16 tensor (measured cuBLAS), the rate of the "
                    f"exact f16 tensor-core path the GEMM runs on"}
        del proj, ys
        torch.cuda.empty_cache()

    # (5) BitNet-2B4T-shaped prefill, planar ternary: 512 tokens through one layer's seven
    #     projections (per-token int8 quantization of the three distinct activations + the
    #     GEMMs; q|k|v and gate|up grouped)
    bproj = [(synth.device_trit_planes(n, k, synth.proj_seed(95_000, 0, i)), n, k)
             for i, (_, n, k) in enumerate(synth.BITNET_2B4T_PROJ)]
    bks = sorted({k for _, _, k in bproj})
    bx = {k: torch.from_numpy(synth.activations(M, k, seed=20 + k)).cuda() for k in bks}
    bq = {k: (torch.empty((M, k), dtype=torch.int8, device="cuda"),
              torch.empty((M,), dtype=torch.float32, device="cuda")) for k in bks}
    bws = torch.empty(lb.lb_gemm_trit_workspace_bytes(M, max(bks)), dtype=torch.uint8,
                      device="cuda")
    bys = [torch.empty((M, n), dtype=torch.float32, device="cuda") for _, n, _ in bproj]
    bops = 2 * M * sum(n * k for _, n, k in synth.BITNET_2B4T_PROJ)

    def layer_planar():
        # quantizer that also writes the GEMM's operand tiles, then the GEMM from them
        for members in groups:
            k = bproj[members[0]][2]
            lb.lb_quantize_i8_absmax_tiles(bx[k], bq[k][0], bq[k][1], M, k, bws, stream=stream)
            lb.lb_gemm_trit_planes_grouped_tiles(
                [(bproj[i][0], 0.02, bys[i], None, bproj[i][1]) for i in members],
                bq[k][1], M, k, bws, stream=stream)

    def layer_planar_prologue():
        # the same layer with the plain quantizer and the GEMM's own activation prologue
        for members in groups:
            k = bproj[members[0]][2]
            lb.lb_quantize_i8_absmax(bx[k], bq[k][0], bq[k][1], M, k, stream=stream)
            lb.lb_gemm_trit_planes_grouped(
                [(bproj[i][0], 0.02, bys[i], None, bproj[i][1]) for i in members],
                bq[k][0], bq[k][1], M, k, bws, stream=stream)
    ms = time_graph(Graph(layer_planar, stream), reps=20)
    ms_p = time_graph(Graph(layer_planar_prologue, stream), reps=20)
    tops = bops / (ms * 1e-3) / 1e12
    rows["bitnet_2b4t_prefill_m512_planar"] = {
        "TOPS": round(tops, 1), "pct_tensor_peak": round(100 * tops / tflops, 1),
        "ms_per_layer": round(ms, 4), "int8_equivalent_ops": bops,
        "TOPS_with_prologue_launch": round(bops / (ms_p * 1e-3) / 1e12, 1),
        "peak": f"{tflops} TFLOP/s dense bf16/f16 tensor (measured cuBLAS), the rate of the "
                f"exact f16 tensor-core path the GEMM runs on"}
    for i, (name, n, k) in enumerate(synth.BITNET_2B4T_PROJ):
        def one(i=i, n=n, k=k):
            lb.lb_gemm_trit_planes_grouped([(bproj[i][0], 0.02, bys[i], None, n)],
                                           bq[k][0], bq[k][1], M, k, bws, stream=stream)
        ms1 = time_graph(Graph(one, stream), reps=50)
        rows["bitnet_2b4t_prefill_m512_planar"][f"{name}_TOPS"] = round(
            2 * M * n * k / (ms1 * 1e-3) / 1e12, 1)
    del bproj, bys
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands
# ---------------------------------------------------------------------------------------------
def reference_arm(args, dist, base):
    if dist.rank != 0:
        return None
    import oracle
    import synth
    N, K = 512, ROWS_K
    blocks = synth.q2_0_blocks(N, K, seed=0)
    q, dx = oracle.quantize_q8_0(synth.activations(1, K, seed=1))
    cores = len(os.sched_getaffinity(0))
    chunks = [blocks[i:i + max(1, N // cores)] for i in range(0, N, max(1, N // cores))]

    def one():
        with cf.ThreadPoolExecutor(max_workers=cores) as ex:
            list(ex.map(lambda c: oracle.q2_0_g64_product(c, q, dx, want_isum=False), chunks))
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = (time.perf_counter() - t0) / args.steps
    value = q2_bytes(N, K) / dt / 1e9
    sample = f"rows 0..{N - 1} of a 4096x4096 Q2_0_g64 matrix per step, batch 1, {cores} threads"
    base.update({"impl": "reference", "value": round(value, 4), "ms_per_step": round(dt * 1e3, 3),
                 "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                                  "kind": "oracle", "sample": sample},
                 "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                         "d2h_bytes_per_step": 0}})
    return base


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true")
    ap.add_argument("--rows-only", choices=["stream", "decode", "prefill"], default=None,
                    help="skip the headline; run (and print) only these rows")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    dist = Dist()
    base = {"metric": METRIC, "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8",
            "data": "synthetic (seeded; random weights of the stated shapes and distributions)",
            "config": {"workload": WORKLOAD, "weights_per_step": f"{N_ROT} distinct 4096x4096 "
                       f"matrices, {N_ROT * q2_bytes(ROWS_N, ROWS_K)} B (> 129 MB L2)",
                       "l2": "inputs larger than L2 (weight rotation)",
                       "parallelism": f"replicas x{dist.world}"}}
    if args.impl == "reference":
        line = reference_arm(args, dist, base)
        if line:
            print(json.dumps(line))
        dist.close()
        return

    import torch
    import bit_matvec_lb_gb300 as lb
    if dist.world == 1:
        torch.cuda.set_device(0)
    lb.load()
    if args.rows_only:
        out = {}
        rows_measure(lb, out, args.rows_only)
        print(json.dumps(out))
        dist.close()
        return
    out = dict(base)
    headline(lb, args, dist, out)
    if dist.rank == 0 and dist.world == 1 and not args.no_rows:
        rows_measure(lb, out)
    if dist.rank == 0:
        print(json.dumps(out))
    dist.close()


if __name__ == "__main__":
    main()
