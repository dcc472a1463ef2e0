#!/usr/bin/env python3
"""Benchmark of the ROCmFP2 decode GEMV (the headline workload) on GB300.

Workload: ROCmFP2 weights [M=14336, K=4096] (Student-t(5) x 0.02 with 1% of
columns x8, seed 1), fp32 activations ~ N(0,1); one step = one rfp2_gemv call
on batch 1 (a single kernel: Q8_1 activation quantize fused into the GEMV).  The metric is packed
weight bytes per second (18,350,080 bytes per call).

Timing: W warm-up steps, then exactly K steps, captured as CUDA graphs of back
to back calls and timed with CUDA events on the capture stream.  Consecutive
calls rotate over enough copies of the packed weights that the working set is
more than 4x the L2 (each copy is re-read only after >500 MB of other reads).
SM clocks and throttle reasons are sampled with nvidia-smi during the run.

Also reported in the same JSON line: that kernel against the HBM roofline, the
GEMV on pre-quantized activations, batch 4, the end-to-end figure through the public API with host
buffers (activations H2D and outputs D2H inside the timed region), and the
CPU oracle timed on a bounded sample on the host cores (cpu_baseline).

``--impl reference`` times the CPU oracle alone (the reference arm).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

M_DEC, K_DEC = 14336, 4096
WEIGHT_BYTES = M_DEC * K_DEC // 32 * 10
L2_BYTES = 129 * 1024 * 1024
METRIC = "ROCmFP2 GEMV packed-weight GB/s (% HBM peak); prefill GEMM TOPS (% peak)"
WORKLOAD = ("rocmfp2 decode GEMV 14336x4096, batch 1, fp32 activations quantized in the call "
            "(Student-t(5)*0.02 weights, 41 outlier columns x8, seed 1)")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured (MEASURED_PEAKS.json)"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback (no MEASURED_PEAKS.json)"}


# ---------------------------------------------------------------------------
# clocks


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if ts < t0 - 0.2 or ts > t1 + 0.2:
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# multi-rank aggregation (replicas: every rank runs the same workload)


def max_over_ranks(value: float, device) -> float:
    """Largest `value` over the ranks of the default process group (the
    slowest replica's time), or `value` itself without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_step: int, ms_per_step_max: float, world: int) -> float:
    """Whole-job throughput: the bytes all replicas processed per step over
    the slowest replica's step time."""
    return world * bytes_per_step / (ms_per_step_max * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# ncu traffic figure (only while the kernel sources are those it was taken on)

GEMV_SOURCES = ["gemv.cu", "gemv_core.cuh", "rfp2_decode.cuh", "common.cuh", "quantize.cuh"]


def gemv_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in GEMV_SOURCES:
        with open(os.path.join(ROOT, "gemm_rocmfp2_mul_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic():
    """dram read+write bytes per GEMV launch from the committed ncu summary,
    or None if the kernel sources changed since that capture."""
    path = os.path.join(ROOT, "profiles", "gemv_stream_decode_14336x4096_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256") != gemv_source_hash():
            return None
        return int(kv["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# GPU arm


def _graph_time_ms(torch, fn, calls: int, reps: int = 1):
    """Capture `calls` invocations of fn(i) in one CUDA graph; return the
    per-call time (ms) of `reps` replays timed with events on the stream."""
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn(0)  # prime outside capture (library init, smem attributes)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(calls):
                fn(i)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / (calls * reps), g, stream


def run_gpu(args):
    import torch
    import gemm_rocmfp2_mul_gb300 as gl
    from synth import decode_gemv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    gl.build()
    gl.lib()
    peaks = load_peaks()

    # ---- data (untimed): synthetic weights packed on the GPU, copies for L2 rotation
    w = decode_gemv(N=4)
    Wd = torch.from_numpy(w["W"]).cuda()
    P = gl.rfp2_pack_weights(Wd)
    del Wd
    torch.cuda.synchronize()
    # the weights are written once, before any timed call: each call may
    # stream its weights while the previous call is still running
    gl.rfp2_set_weight_prefetch(True)
    copies = max(4, -(-4 * L2_BYTES // WEIGHT_BYTES))
    copies = 1 << (copies - 1).bit_length()
    Pc = torch.empty((copies,) + tuple(P.shape), dtype=torch.uint8, device="cuda")
    Pc[:] = P
    x1 = torch.from_numpy(w["x"][:1]).cuda()
    x4 = torch.from_numpy(w["x"][:4]).cuda()
    y1 = torch.empty((1, M_DEC), dtype=torch.float32, device="cuda")
    y4 = torch.empty((4, M_DEC), dtype=torch.float32, device="cuda")
    ws1 = torch.empty(gl.rfp2_gemv_workspace_bytes(1, K_DEC), dtype=torch.uint8, device="cuda")
    ws4 = torch.empty(gl.rfp2_gemv_workspace_bytes(4, K_DEC), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step1(i):
        gl.rfp2_gemv(Pc[i % copies], M_DEC, K_DEC, x1, y=y1, workspace=ws1, dev_status=st)

    def step4(i):
        gl.rfp2_gemv(Pc[i % copies], M_DEC, K_DEC, x4, y=y4, workspace=ws4, dev_status=st)

    q1, d1 = gl.rfp2_quantize_act(x1)

    def kern1(i):
        gl.rfp2_gemv_q8(Pc[i % copies], M_DEC, K_DEC, q1, d1, y=y1, dev_status=st)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)

    # ---- warm-up: W steps (plus a short clock ramp of the same calls)
    G = min(args.steps, 1000)
    _, gw, sw = _graph_time_ms(torch, step1, max(args.warmup, 3))
    t_ramp = time.time()
    while time.time() - t_ramp < 1.0:
        gw.replay()
    torch.cuda.synchronize()

    # ---- timed: exactly K steps (graphs of G calls + one remainder graph)
    full, rem = divmod(args.steps, G)
    ms_g, gg, sg = _graph_time_ms(torch, step1, G)
    graphs = [(gg, sg)] * full
    if rem:
        _, gr, sr = _graph_time_ms(torch, step1, rem)
        graphs.append((gr, sr))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    main_stream = sg
    with torch.cuda.stream(main_stream):
        start.record(main_stream)
        for g_, s_ in graphs:
            g_.replay()
        end.record(main_stream)
    end.synchronize()
    torch.cuda.synchronize()
    t1 = time.time()
    total_ms = start.elapsed_time(end)
    total_ms = max_over_ranks(total_ms, "cuda")
    ms_per_step = total_ms / args.steps
    value = aggregate_gbs(WEIGHT_BYTES, ms_per_step, world)

    # ---- the GEMV kernel alone (roofline) and batch 4
    kreps = max(1, 5000 // G)
    ms_k, _, _ = _graph_time_ms(torch, kern1, G, reps=kreps)
    ms_b4, _, _ = _graph_time_ms(torch, step4, G, reps=kreps)
    clocks.stop()
    clk = clocks.summary(t_ramp, time.time())
    status = int(st.item())

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(torch, gl, w, Pc, copies, args.steps)
    del Pc
    torch.cuda.empty_cache()

    # ---- the other rows of the hot path on their own workloads
    global CPU_ROWS
    CPU_ROWS = not (args.no_cpu_baseline or rank != 0)
    sec = {} if args.no_secondary else secondary(torch, gl, peaks)
    cpu_sec = {}
    if CPU_ROWS:
        cpu_sec["decode_batch4"] = cpu_decode_batch4()

    # one launch per step (the batch-1 GEMV quantizes x itself), so the
    # kernel's average launch duration is the graph-timed per-step time
    achieved = WEIGHT_BYTES / (ms_per_step * 1e-3) / 1e9
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "i8",
        "data": "synthetic",
        "config": {
            "workload": WORKLOAD,
            "M": M_DEC, "K": K_DEC, "batch": 1,
            "bytes_per_step": WEIGHT_BYTES,
            "l2": f"inputs larger than L2: {copies} rotating weight copies "
                  f"({copies * WEIGHT_BYTES / 1e6:.0f} MB > 129 MB L2)",
            "timing": f"CUDA graphs of {G} back-to-back calls, CUDA events on the capture stream",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "gemv_stream_kernel<1,4,true> (activations quantized in-kernel, weights streamed by bulk async copies)",
            "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": args.traffic if args.traffic is not None else measured_traffic(),
            "peak_source": peaks["source"] + " hbm_gbs",
            "us_per_launch": round(ms_per_step * 1e3, 3),
        },
        "secondary": dict({
            "decode_batch4": {
                "workload": "same weights, batch 4 through rfp2_gemv (int8 dp4a path, quantize "
                            "fused, one launch)",
                "value": round(WEIGHT_BYTES / (ms_b4 * 1e-3) / 1e9, 1), "unit": "GB/s",
                "us_per_call": round(ms_b4 * 1e3, 3),
                "frac_of_hbm_peak": round(WEIGHT_BYTES / (ms_b4 * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            },
            "call_us_batch1": round(ms_per_step * 1e3, 3),
            "gemv_q8_prequantized_us": round(ms_k * 1e3, 3),
        }, **sec),
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk,
        "dev_status": status,
    }
    for key, row in cpu_sec.items():
        if key in out["secondary"]:
            out["secondary"][key]["cpu_oracle"] = row
    if rank == 0:
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def _graph_us(torch, fn, calls, reps):
    ms, _, _ = _graph_time_ms(torch, fn, calls, reps)
    return ms * 1e3


def _sec_moe(torch, gl, peaks, reps=3):
    """MoE bulk-expert GEMV: 256 experts of 768 x 2048, 16 tokens, top-8."""
    from synth import moe_expert_weights, moe_gemv
    E, M, K, T, top_k = 256, 768, 2048, 16, 8
    w = moe_gemv(E=E, M=M, K=K, T=T, top_k=top_k, seed=2, experts=False)
    copies = 3
    Pc = torch.empty((copies, E, M, K // 32, 10), dtype=torch.uint8, device="cuda")
    for e in range(E):
        gl.rfp2_pack_weights(torch.from_numpy(moe_expert_weights(2, E, M, K, e)).cuda(), out=Pc[0, e])
    for c in range(1, copies):
        Pc[c] = Pc[0]
    ids = torch.from_numpy(w["ids"]).cuda()
    x = torch.from_numpy(w["x"]).cuda()
    y = torch.empty((T, top_k, M), dtype=torch.float32, device="cuda")
    ws = torch.empty(gl.rfp2_moe_workspace_bytes(T, top_k, K), dtype=torch.uint8, device="cuda")
    touched = len(set(w["ids"].ravel().tolist()))
    nbytes = touched * M * K // 32 * 10
    cpu = None
    if CPU_ROWS:
        import oracle
        ids_h = w["ids"]
        ex = sorted(set(ids_h.ravel().tolist()))[:4]
        Pe = {e: oracle.rfp2_pack(moe_expert_weights(2, E, M, K, e)[:64]) for e in ex}
        pairs = [(t, j) for t in range(T) for j in range(top_k) if int(ids_h[t, j]) in Pe]

        def moe_step():
            q, d = oracle.quantize_act(w["x"])
            for t, j in pairs:
                oracle.rfp2_gemv(Pe[int(ids_h[t, j])], 64, K, q[t:t + 1], d[t:t + 1])

        cpu = cpu_row(moe_step, len(ex) * 64 * K // 32 * 10, "GB/s (touched experts' packed bytes)",
                      f"quantize 16 tokens + {len(pairs)} (token, slot) GEMVs over 64 rows of "
                      f"{len(ex)} touched experts per step")
    us = _graph_us(torch, lambda i: gl.rfp2_moe_gemv(Pc[i % copies], E, M, K, ids, x, y=y,
                                                     workspace=ws), 200, reps)
    del Pc, ids, x, y, ws
    torch.cuda.empty_cache()
    return {"moe_gemv": {
        "workload": f"256 experts x ROCmFP2 [768, 2048], 16 tokens, top-8 ({touched} experts "
                    f"touched), seed 2; {copies} copies of all experts rotate",
        "value": round(nbytes / us / 1e3, 1), "unit": "GB/s (touched experts' packed bytes)",
        "us_per_call": round(us, 2), "bytes_per_call": nbytes,
        "frac_of_hbm_peak": round(nbytes / us / 1e3 / peaks["hbm_gbs"], 4),
        **({"cpu_oracle": cpu} if cpu else {})}}


def _sec_hfp4(torch, gl, peaks, reps=3):
    """HFP4G32 GEMV 8192 x 8192, batch 1 and 8."""
    from synth import hfp4_gemv
    out = {}
    w = hfp4_gemv(N=8)
    M, K = w["W"].shape
    P = gl.hfp4_pack_weights(torch.from_numpy(w["W"]).cuda())
    copies = 16
    Pc = torch.empty((copies,) + tuple(P.shape), dtype=torch.uint8, device="cuda")
    Pc[:] = P
    Ph = None
    if CPU_ROWS:
        import oracle
        Ph = oracle.hfp4_pack(w["W"][:256])
    for N in (1, 8):
        x = torch.from_numpy(w["x"][:N].copy()).cuda()
        y = torch.empty((N, M), dtype=torch.float32, device="cuda")
        ws = torch.empty(gl.hfp4_gemv_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
        us = _graph_us(torch, lambda i: gl.hfp4_gemv(Pc[i % copies], M, K, x, y=y, workspace=ws),
                       200, reps)
        out[f"hfp4_gemv_batch{N}"] = {
            "workload": f"HFP4G32 [8192, 8192] N(0, 0.02^2) seed 4, batch {N}; {copies} copies rotate",
            "value": round(P.numel() / us / 1e3, 1), "unit": "GB/s (packed bytes)",
            "us_per_call": round(us, 2), "bytes_per_call": int(P.numel()),
            "frac_of_hbm_peak": round(P.numel() / us / 1e3 / peaks["hbm_gbs"], 4)}
        if Ph is not None:
            import oracle
            xh = w["x"][:N].copy()
            out[f"hfp4_gemv_batch{N}"]["cpu_oracle"] = cpu_row(
                lambda: oracle.hfp4_gemv(Ph, 256, K, xh), Ph.size, "GB/s (packed bytes)",
                f"GEMV over 256 of {M} rows at batch {N} per step")
    del P, Pc
    torch.cuda.empty_cache()
    return out


def _sec_gemm(torch, gl, peaks, hfp4=False, reps=3):
    """Prefill GEMM 17408 x 5120 x 2048 tokens (weight decode to bf16 included),
    ROCmFP2 or (hfp4=True) HFP4G32 weights."""
    import numpy as np
    from synth import prefill_gemm
    w = prefill_gemm()
    M, K = w["W"].shape
    N = w["X"].shape[0]
    Wd = torch.from_numpy(w["W"]).cuda()
    P = gl.hfp4_pack_weights(Wd) if hfp4 else gl.rfp2_pack_weights(Wd)
    del Wd
    X = torch.from_numpy(w["X"].view(np.int16)).cuda()
    Y = torch.empty((N, M), dtype=torch.float32, device="cuda")
    if hfp4:
        ws = torch.empty(gl.hfp4_gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
        fn = lambda i: gl.hfp4_gemm(P, M, K, X, Y=Y, workspace=ws)
    else:  # decoded inside the GEMM: no workspace
        ws = None
        fn = lambda i: gl.rfp2_gemm(P, M, K, X, Y=Y)
    us = _graph_us(torch, fn, 20, reps)
    tflops = 2.0 * M * K * N / us / 1e6
    fmt = "HFP4G32" if hfp4 else "ROCmFP2"
    cpu = None
    if CPU_ROWS:
        import oracle
        if hfp4:
            Po = oracle.hfp4_pack(w["W"][:4])
            gstep = lambda: oracle.hfp4_gemm(Po, 4, K, w["X"])
        else:
            Po = oracle.rfp2_pack(w["W"][:4])
            gstep = lambda: oracle.rfp2_gemm(Po, 4, K, w["X"])
        cpu = cpu_row(gstep, 2.0 * 4 * N * K, "TFLOP/s",
                      f"4 of {M} weight rows x {N} tokens x K = {K} per step", scale=1e12)
    yardstick = None
    if not hfp4:
        # cuBLAS bf16 on bf16 weights of the same shape and spread, already
        # expanded (bf16 output): a library reference, not this path
        Wexp = (torch.randn((M, K), generator=torch.Generator(device="cuda").manual_seed(3),
                            device="cuda") * 0.015).to(torch.bfloat16)
        Xb = X.view(torch.bfloat16)
        Yb = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
        yus = _graph_us(torch, lambda i: torch.matmul(Xb, Wexp.t(), out=Yb), 20, reps)
        yardstick = {"cublas_bf16_us": round(yus, 1),
                     "cublas_bf16_tflops": round(2.0 * M * K * N / yus / 1e6, 1),
                     "what": "torch.matmul (cuBLAS) bf16 x bf16 -> bf16 on bf16 weights of "
                             "the same shape and spread, no decode"}
        del Wexp, Xb, Yb
    del P, X, Y, ws
    torch.cuda.empty_cache()
    return {("hfp4_prefill_gemm" if hfp4 else "prefill_gemm"): {
        "workload": f"{fmt} [17408, 5120] N(0, 0.015^2) x bf16 [2048, 5120] (0.5% x20), seed 3",
        "value": round(tflops, 1), "unit": "TFLOP/s (2*M*N*K, weight decode included)",
        "us_per_call": round(us, 1),
        "frac_of_bf16_peak": round(tflops / peaks["bf16_tflops"], 4),
        "frac_of_bf16_sustained": round(tflops / peaks["bf16_tflops_sustained"], 4),
        "bound": "tensor", "peak_source": peaks["source"] + " bf16_tflops (cuBLAS bf16)",
        **({"yardstick": yardstick} if yardstick else {}),
        **({"cpu_oracle": cpu} if cpu else {})}}


def _sec_verify(torch, gl, peaks, reps=3):
    """Verify batches of 32 and 128 tokens on the decode weights (tensor-core
    GEMV on Q8_1 activations, weights expanded once per call)."""
    from synth import decode_gemv
    out = {}
    w = decode_gemv(N=1)
    M, K = w["W"].shape
    P = gl.rfp2_pack_weights(torch.from_numpy(w["W"]).cuda())
    copies = 8
    Pc = torch.empty((copies,) + tuple(P.shape), dtype=torch.uint8, device="cuda")
    Pc[:] = P
    Po = _oracle_sample(128)[1] if CPU_ROWS else None
    for N in (32, 128):
        xh = np.random.default_rng(N).standard_normal((N, K)).astype(np.float32)
        x = torch.from_numpy(xh).cuda()
        y = torch.empty((N, M), dtype=torch.float32, device="cuda")
        ws = torch.empty(gl.rfp2_gemv_batched_workspace_bytes(M, K, N), dtype=torch.uint8,
                         device="cuda")
        us = _graph_us(torch, lambda i: gl.rfp2_gemv_batched(Pc[i % copies], M, K, x, y=y,
                                                             workspace=ws), 50, reps)
        out[f"verify_batch{N}"] = {
            "workload": f"ROCmFP2 decode weights [14336, 4096] (seed 1), {N} tokens N(0,1); "
                        f"{copies} copies rotate",
            "value": round(P.numel() / us / 1e3, 1), "unit": "GB/s (packed bytes)",
            "tflops": round(2.0 * M * K * N / us / 1e6, 1),
            "us_per_call": round(us, 2), "bytes_per_call": int(P.numel())}
        if Po is not None:
            import oracle

            def vstep(xh=xh):
                q, d = oracle.quantize_act(xh)
                oracle.rfp2_gemv(Po, 128, K, q, d)

            out[f"verify_batch{N}"]["cpu_oracle"] = cpu_row(
                vstep, Po.size, "GB/s (packed bytes)",
                f"quantize {N} tokens + GEMV over 128 of {M} rows per step")
    del P, Pc
    torch.cuda.empty_cache()
    return out


def _sec_decode(torch, gl, peaks, N=1, reps=3):
    """The decode GEMV alone (batch N through rfp2_gemv), the headline
    workload's kernel in a graph of back-to-back calls over rotating copies."""
    from synth import decode_gemv
    w = decode_gemv(N=max(N, 1))
    P = gl.rfp2_pack_weights(torch.from_numpy(w["W"]).cuda())
    torch.cuda.synchronize()
    gl.rfp2_set_weight_prefetch(True)  # weights written once, before the timed calls
    copies = max(4, -(-4 * L2_BYTES // WEIGHT_BYTES))
    copies = 1 << (copies - 1).bit_length()
    Pc = torch.empty((copies,) + tuple(P.shape), dtype=torch.uint8, device="cuda")
    Pc[:] = P
    x = torch.from_numpy(w["x"][:N].copy()).cuda()
    y = torch.empty((N, M_DEC), dtype=torch.float32, device="cuda")
    ws = torch.empty(gl.rfp2_gemv_workspace_bytes(N, K_DEC), dtype=torch.uint8, device="cuda")
    us = _graph_us(torch, lambda i: gl.rfp2_gemv(Pc[i % copies], M_DEC, K_DEC, x, y=y,
                                                 workspace=ws), 200, reps)
    del P, Pc
    torch.cuda.empty_cache()
    return {f"decode_batch{N}_alone": {
        "workload": f"ROCmFP2 decode weights [14336, 4096] (seed 1), batch {N}; {copies} copies rotate",
        "value": round(WEIGHT_BYTES / us / 1e3, 1), "unit": "GB/s (packed bytes)",
        "us_per_call": round(us, 3),
        "frac_of_hbm_peak": round(WEIGHT_BYTES / us / 1e3 / peaks["hbm_gbs"], 4)}}


def _sec_nvfp4(torch, gl, peaks, reps=3):
    """Block-scaled FP4 (NVFP4) prefill GEMM 17408 x 5120 x 2048 tokens on the
    FP4 tensor cores.  The weights convert once (exactly) to the NVFP4 image,
    like packing; the per-token activation quantization is inside the timed
    call.  The conversion is timed on its own."""
    from synth import prefill_gemm
    w = prefill_gemm()
    M, K = w["W"].shape
    N = w["X"].shape[0]
    Wd = torch.from_numpy(w["W"]).cuda()
    P = gl.rfp2_pack_weights(Wd)
    del Wd
    Wnv = gl.rfp2_to_nvfp4(P, M, K)
    X = torch.from_numpy(w["X"].view(np.int16)).cuda()
    Y = torch.empty((N, M), dtype=torch.float32, device="cuda")
    ws = torch.empty(gl.rfp2_gemm_nvfp4_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    us = _graph_us(torch, lambda i: gl.rfp2_gemm_nvfp4(Wnv, M, K, X, Y=Y, workspace=ws), 20, reps)
    conv_us = _graph_us(torch, lambda i: gl.rfp2_to_nvfp4(P, M, K, out=Wnv), 20, reps)
    tflops = 2.0 * M * K * N / us / 1e6
    # nominal dense FP4 : bf16 = 13.5 : 2.25 on this GPU, applied to the measured bf16 peak
    fp4_peak = peaks["bf16_tflops"] * 6.0
    Yb = gl.rfp2_gemm(P, M, K, X)
    torch.cuda.synchronize()
    dev_bf16 = float((torch.linalg.vector_norm(Y - Yb, dim=1) /
                      torch.linalg.vector_norm(Yb, dim=1)).max())
    cpu = None
    if CPU_ROWS:
        import oracle
        Po = oracle.rfp2_pack(w["W"][:4])
        wc, wsb = oracle.rfp2_to_nvfp4(Po, 4, K)
        xf = (w["X"].astype(np.uint32) << 16).view(np.float32)

        def nstep():
            xc, xs, gg = oracle.nvfp4_quant_act(xf)
            oracle.nvfp4_gemm(wc, wsb, 4, K, xc, xs, gg)

        cpu = cpu_row(nstep, 2.0 * 4 * N * K, "TFLOP/s",
                      f"quantize {N} tokens + 4 of {M} weight rows x {N} tokens x K = {K} per step",
                      scale=1e12)
    del P, Wnv, X, Y, ws, Yb
    torch.cuda.empty_cache()
    return {"nvfp4_prefill_gemm": dict({
        "workload": f"ROCmFP2 [17408, 5120] N(0, 0.015^2) as its exact NVFP4 image x bf16 [2048, 5120] "
                    f"(0.5% x20) quantized to NVFP4 per call, seed 3",
        "value": round(tflops, 1), "unit": "TFLOP/s (2*M*N*K, activation quantization included)",
        "us_per_call": round(us, 1),
        "frac_of_fp4_peak": round(tflops / fp4_peak, 4),
        "peak_source": "measured bf16 peak (MEASURED_PEAKS.json) x 6 (nominal dense fp4 : bf16)",
        "weight_conversion_us": round(conv_us, 1),
        "max_rel_diff_vs_bf16_gemm": round(dev_bf16, 5),
        "bound": "tensor"}, **({"cpu_oracle": cpu} if cpu else {}))}


SECONDARY_ROWS = {
    "decode1": lambda torch, gl, peaks, reps=3: _sec_decode(torch, gl, peaks, 1, reps),
    "decode4": lambda torch, gl, peaks, reps=3: _sec_decode(torch, gl, peaks, 4, reps),
    "verify": _sec_verify,
    "moe": _sec_moe,
    "hfp4": _sec_hfp4,
    "gemm": lambda torch, gl, peaks, reps=3: _sec_gemm(torch, gl, peaks, False, reps),
    "hgemm": lambda torch, gl, peaks, reps=3: _sec_gemm(torch, gl, peaks, True, reps),
    "nvfp4": _sec_nvfp4,
}


def secondary(torch, gl, peaks):
    """The other rows of the hot path, each on its own synthetic workload, in
    CUDA graphs of back-to-back calls over weight copies larger than L2."""
    out = {}
    for name, fn in SECONDARY_ROWS.items():
        if not name.startswith("decode"):
            out.update(fn(torch, gl, peaks))
    return out


def run_only(args):
    """One secondary row alone (one graph replay), for profiler captures."""
    import torch
    import gemm_rocmfp2_mul_gb300 as gl
    torch.cuda.set_device(0)
    gl.build()
    gl.lib()
    out = SECONDARY_ROWS[args.only](torch, gl, load_peaks(), reps=1)
    print(json.dumps(out), flush=True)


def run_e2e(torch, gl, w, Pc, copies, steps, C=32):
    """Same metric through the public API with the activations in pinned host
    memory: each step copies its x H2D, runs rfp2_gemv and copies its y D2H.
    Steps go in chunks of C: the C input copies of a chunk (their own device
    buffers) on one stream, one event, the chunk's C GEMVs back to back on
    the compute stream, one event, the C output copies on a third stream.
    Two sets of buffers let one chunk's copies overlap the neighbouring
    chunks' GEMVs, as in a serving loop taking independent requests C at a
    time.  Only the first GEMV of a chunk waits for an event; the others keep
    the programmatic overlap with the GEMV before them.  Measured per step
    with the GEMV at 6.4 us a call: an event wait before every GEMV (two or
    eight buffers) 12.3 us; chunks of 8 / 16 / 32 steps 7.8 / 7.3 / 7.2 us."""
    NB = 2 * C
    x_h = [torch.from_numpy(w["x"][:1].copy()).pin_memory() for _ in range(NB)]
    y_h = [torch.empty((1, M_DEC), dtype=torch.float32).pin_memory() for _ in range(NB)]
    x_d = [torch.empty((1, K_DEC), dtype=torch.float32, device="cuda") for _ in range(NB)]
    y_d = [torch.empty((1, M_DEC), dtype=torch.float32, device="cuda") for _ in range(NB)]
    ws = [torch.empty(gl.rfp2_gemv_workspace_bytes(1, K_DEC), dtype=torch.uint8, device="cuda")
          for _ in range(NB)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def steps_graph(n):
        s_comp = torch.cuda.current_stream()
        ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}
        for j in range(n // C):
            h = j % 2
            bufs = range(h * C, h * C + C)
            # the chunk's buffers were last read by chunk j - 2's GEMVs
            s_in.wait_stream(s_comp) if j < 2 else s_in.wait_event(ev["comp"][h])
            with torch.cuda.stream(s_in):
                for b in bufs:
                    x_d[b].copy_(x_h[b], non_blocking=True)
                ev["in"][h].record(s_in)
            s_comp.wait_event(ev["in"][h])
            if j >= 2:
                s_comp.wait_event(ev["out"][h])  # chunk j - 2's outputs copied out
            for k, b in enumerate(bufs):
                gl.rfp2_gemv(Pc[(j * C + k) % copies], M_DEC, K_DEC, x_d[b], y=y_d[b], workspace=ws[b])
            ev["comp"][h].record(s_comp)
            s_out.wait_event(ev["comp"][h])
            with torch.cuda.stream(s_out):
                for b in bufs:
                    y_h[b].copy_(y_d[b], non_blocking=True)
                ev["out"][h].record(s_out)
        s_comp.wait_stream(s_in)
        s_comp.wait_stream(s_out)

    G = max(C, min(steps, 1000) // C * C)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        gl.rfp2_gemv(Pc[0], M_DEC, K_DEC, x_d[0], y=y_d[0], workspace=ws[0])  # library init
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            steps_graph(G)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // G)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
    end.synchronize()
    ms = start.elapsed_time(end) / (G * reps)
    return {"value": round(WEIGHT_BYTES / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": 1 * K_DEC * 4, "d2h_bytes_per_step": 1 * M_DEC * 4,
            "us_per_step": round(ms * 1e3, 3),
            "pipelining": f"chunks of {C} steps, {NB} buffers; H2D, GEMV and D2H on three "
                          f"streams ordered by one event per chunk and stream"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)


_DECODE_W = None


def _oracle_sample(rows: int):
    """The oracle's own packing of `rows` evenly spaced rows of the decode
    weights (preparation, untimed) and the batch-1 activations."""
    global _DECODE_W
    import oracle
    from synth import decode_gemv
    if _DECODE_W is None:
        _DECODE_W = decode_gemv(N=8)
    w = _DECODE_W
    idx = np.linspace(0, M_DEC - 1, rows).astype(np.int64)
    P = oracle.rfp2_pack(w["W"][idx])
    return oracle, P, w["x"][:1].copy(), idx


def host_threads() -> int:
    """Cores of this process's CPU affinity set."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _timed_threads(step, threads: int, seconds: float):
    """Run step() repeatedly on `threads` host threads for about `seconds`
    (the oracle's ctypes calls release the GIL); returns (total steps,
    elapsed seconds)."""
    from concurrent.futures import ThreadPoolExecutor
    t0 = time.perf_counter()
    deadline = t0 + seconds

    def worker(_):
        n = 0
        while True:
            step()
            n += 1
            if time.perf_counter() >= deadline:
                return n

    with ThreadPoolExecutor(threads) as ex:
        counts = list(ex.map(worker, range(threads)))
    return sum(counts), time.perf_counter() - t0


# whether the secondary rows also time the oracle on a sample of their data
CPU_ROWS = False
CPU_ROW_SECONDS = 2.0


def cpu_row(step, bytes_or_flops: float, unit: str, sample: str, scale: float = 1e9) -> dict:
    """The oracle's rate on one secondary workload: step() on every core of
    the affinity set for CPU_ROW_SECONDS."""
    T = host_threads()
    n, dt = _timed_threads(step, T, CPU_ROW_SECONDS)
    return {"value": round(n * bytes_or_flops / dt / scale, 6), "unit": unit, "cores": T,
            "kind": "oracle", "sample": f"{sample}; {n} steps in {dt:.1f} s"}


def cpu_decode_batch4():
    orc, P, x, idx = _oracle_sample(512)
    x4 = _DECODE_W["x"][:4].copy()

    def step():
        q, d = orc.quantize_act(x4)
        orc.rfp2_gemv(P, 512, K_DEC, q, d)

    return cpu_row(step, 512 * K_DEC // 32 * 10, "GB/s",
                   f"quantize 4 tokens + GEMV over 512 of {M_DEC} rows per step")


def cpu_baseline(seconds: float, rows: int = 512):
    """The oracle (plain single-threaded C, fp64 dots) on a bounded sample of
    the same workload: quantize x + GEMV over `rows` sampled weight rows, on
    one core and then on every core of the affinity set (one independent copy
    of the step per thread); scaled to packed-weight GB/s."""
    orc, P, x, idx = _oracle_sample(rows)

    def step():
        q, d = orc.quantize_act(x)
        orc.rfp2_gemv(P, rows, K_DEC, q, d)

    per = rows * K_DEC // 32 * 10
    n1, dt1 = _timed_threads(step, 1, seconds / 3)
    T = host_threads()
    nT, dtT = _timed_threads(step, T, 2 * seconds / 3)
    return {"value": round(nT * per / dtT / 1e9, 6), "unit": "GB/s", "cores": T,
            "kind": "oracle", "single_core_value": round(n1 * per / dt1 / 1e9, 6),
            "sample": f"quantize x + GEMV over {rows} of {M_DEC} decode rows per step; "
                      f"{n1} steps on 1 core in {dt1:.1f} s, {nT} steps on {T} cores in {dtT:.1f} s"}


def run_reference(args):
    """Reference arm: the CPU oracle on the host cores, exactly K steps after W
    warm-up steps; each step is quantize + GEMV over a row sample sized so the
    whole run stays within --ref-seconds (a minute by default)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    orc, P, x, idx = _oracle_sample(64)
    t0 = time.perf_counter()
    q, d = orc.quantize_act(x)
    orc.rfp2_gemv(P, 64, K_DEC, q, d)
    per_row = (time.perf_counter() - t0) / 64
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    # the oracle packs its sample (about 2 ms a row): keep that preparation short
    rows = int(min(2048, max(8, host_threads() * budget / max(per_row, 1e-9))))
    orc, P, x, idx = _oracle_sample(rows)
    T = host_threads()
    # every step: quantize x + GEMV over the sampled rows, the rows split over
    # the host cores (contiguous ranges, one oracle call per core)
    cuts = [rows * i // T for i in range(T + 1)]
    parts = [np.ascontiguousarray(P[cuts[i]:cuts[i + 1]]) for i in range(T)]
    from concurrent.futures import ThreadPoolExecutor
    pool = ThreadPoolExecutor(T)

    def step():
        q, d = orc.quantize_act(x)
        list(pool.map(lambda p: orc.rfp2_gemv(p, p.shape[0], K_DEC, q, d) if p.shape[0] else None,
                      parts))

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    pool.shutdown()
    value = args.steps * rows * K_DEC // 32 * 10 / dt / 1e9
    sample = (f"each step = quantize x + GEMV over {rows} of {M_DEC} rows split over {T} cores "
              f"({dt:.1f} s total)")
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_DEC, "K": K_DEC, "batch": 1,
                   "reference": "CPU oracle (plain C, fp64), bounded row sample"},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": T, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the MoE, HFP4 and prefill GEMM measurements")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="time budget of the reference arm's K + W steps")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per GEMV launch from an ncu capture of this kernel")
    ap.add_argument("--only", choices=sorted(SECONDARY_ROWS),
                    help="time one secondary row alone (for profiler captures) and exit")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
