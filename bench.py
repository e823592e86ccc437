#!/usr/bin/env python
"""Benchmark of the decode quant + quantized-linear path (one JSON line).

Headline workload - the INT8 W8A8 M-sweep on two DeepSeek-V4 linears:
(K=4096, N=1024) and (K=1024, N=32768), M in {1,2,3,4,7,8,9,16,32,64};
X bf16 ~ N(0,1) with 0.1% x50 outliers, W int8 uniform [-127,127], per-channel
scales U[1e-3,1e-2].  One step = for every (linear, M): the standalone
per-token quant, the standalone W8A8 GEMM on its output, and the fused
quant + GEMM.  Throughput = algorithmic bytes of the step / step time (GB/s).

Timing: device-resident inputs, each op group captured once as a CUDA graph
and replayed; CUDA events on the launching stream; W warm-up steps, then K
timed steps between a barrier + synchronize.  Every call reads its own copy
of the weights and a step reads 720 MB of weights (> 2x the 129 MB L2), so
each call streams its weights from HBM.  Activations stay L2-hot, as they
would right after the producing kernel in a decode step.

Also reported: per-call microseconds and GB/s for every (op, linear, M); the
other workloads (FP8 group quant with packed UE8M0 scales, the block-scaled
einsum in both scale formats, the fp32-scale + repack control, the MoE
expert chain); an end-to-end number through the public API with host
buffers; the roofline of the dominant kernel; the CPU oracle on the host's
cores; SM clocks sampled during the timed region.

`--impl reference` times the CPU oracle (the reference arm) on the same
workload, metric and unit.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs/call & GB/s per quantized linear vs M=1..64; % of GB300 HBM/tensor peak"
UNIT = "GB/s"
MS = [1, 2, 3, 4, 7, 8, 9, 16, 32, 64]
LINEARS = [(4096, 1024), (1024, 32768)]
SEED = 0x5EED0000


# ---------------------------------------------------------------- algorithmic bytes
def bytes_quant(M, K):
    return 2 * M * K + M * K + 4 * M


def bytes_gemm(M, K, N):
    return N * K + 4 * N + M * K + 4 * M + 2 * M * N


def bytes_fused(M, K, N):
    return N * K + 4 * N + 2 * M * K + 2 * M * N


def step_bytes():
    return sum(bytes_quant(M, K) + bytes_gemm(M, K, N) + bytes_fused(M, K, N) for K, N in LINEARS for M in MS)


def bytes_group_quant(T, G, D):
    Ta = (T + 3) // 4 * 4
    return 2 * T * G * D + T * G * D + 4 * G * ((D // 128 + 3) // 4) * Ta


def bytes_einsum(T, G, D, N):
    Ta = (T + 3) // 4 * 4
    P = (D // 128 + 3) // 4
    return G * D * N + 4 * G * (D // 128) * (N // 128) + T * G * D + 4 * G * P * Ta + 2 * T * G * N


# ---------------------------------------------------------------- peaks
def max_over_ranks(x, dist, device):
    """The largest of every rank's x: the job takes as long as its slowest rank."""
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(bytes_per_step_per_rank, ms_per_step, world):
    """GB/s of the whole job: every rank (an independent replica) moves its own step's bytes in the
    slowest rank's step time."""
    return world * bytes_per_step_per_rank / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


ENGINES = [(0, "mma_sync_f16_m16n8k16"), (1, "mma_sync_e4m3_m16n8k32"), (2, "mma_sync_s8_m16n8k32"),
           (3, "tcgen05_f16_128x256x16"), (4, "tcgen05_f8f6f4_128x256x32"), (5, "tcgen05_f16_128x64x16"),
           (6, "tcgen05_f8f6f4_128x16x32")]


def engine_peaks(torch, dev):
    """Measured throughput (TFLOP/s, TOPS for s8) of each matrix engine the kernels use, from
    libfq_peaks.so: mma.sync with 8 warps x 4 CTAs per SM and 8 independent chains a warp; tcgen05 with
    one issuing thread per SM.  Each kernel is sized to run ~1 ms and timed with CUDA events."""
    import ctypes
    from fp8_dynamic_quant_gb300 import build as fqbuild
    if not os.path.exists(fqbuild.PEAKS_LIB):
        return None
    L = ctypes.CDLL(fqbuild.PEAKS_LIB)
    L.fq_peak_run.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                              ctypes.POINTER(ctypes.c_double), ctypes.c_void_p, ctypes.c_void_p]
    L.fq_peak_run.restype = ctypes.c_int
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sink = torch.zeros(256, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for kind, name in ENGINES:
        ctas = sms * 4 if kind <= 2 else sms
        ops = ctypes.c_double(0)

        def run(iters):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            rc = L.fq_peak_run(kind, iters, ctas, ctypes.c_void_p(stream.cuda_stream), ctypes.byref(ops),
                               ctypes.c_void_p(err.data_ptr()), ctypes.c_void_p(sink.data_ptr()))
            b.record()
            torch.cuda.synchronize()
            if rc != 0:
                raise RuntimeError("fq_peak_run(%d) failed: %d" % (kind, rc))
            return a.elapsed_time(b)
        iters = 64
        run(iters)
        ms = run(iters)
        iters = max(64, int(iters * 1.0 / max(ms, 1e-3)))       # about 1 ms
        run(iters)
        ms = min(run(iters) for _ in range(3))
        out[name] = round(ops.value / (ms * 1e-3) / 1e12, 1)
    if int(err.item()) != 0:
        return None
    out["unit"] = "TFLOP/s (s8: TOPS), measured on this GPU"
    return out


def traffic_for(kernel_key, sources):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d:
        return None
    h = hashlib.sha256()
    for s in sources:
        h.update(open(os.path.join(ROOT, s), "rb").read())
    return d["dram_bytes_per_launch"] if d.get("source_sha256") == h.hexdigest() else None


def library_schedules(fn, torch):
    """Runs fn() once with FQ_DEBUG_SCHEDULE=1 and returns the schedule the
    library reported for each W8A8 call, in call order (read from its stderr)."""
    import tempfile
    sys.stderr.flush()
    saved = os.dup(2)
    old = os.environ.get("FQ_DEBUG_SCHEDULE")
    with tempfile.TemporaryFile(mode="w+") as tmp:
        os.dup2(tmp.fileno(), 2)
        os.environ["FQ_DEBUG_SCHEDULE"] = "1"
        try:
            fn()
            torch.cuda.synchronize()
        finally:
            sys.stderr.flush()
            os.dup2(saved, 2)
            os.close(saved)
            if old is None:
                del os.environ["FQ_DEBUG_SCHEDULE"]
            else:
                os.environ["FQ_DEBUG_SCHEDULE"] = old
        tmp.seek(0)
        lines = [l for l in tmp.read().splitlines() if l.startswith("fq: ")]
    return [l.split("schedule=")[1].split()[0] for l in lines]


# ---------------------------------------------------------------- clocks
class ClockSampler:
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [l for (t, l) in self.lines if t0 <= t <= t1 + 0.15]
        if not rows:
            rows = [l for (_, l) in self.lines]
        if not rows:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- the fq arm
def run_fq(args, rank, world, local_rank):
    import torch
    import fp8_dynamic_quant_gb300 as fq
    from fp8_dynamic_quant_gb300 import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    fq.lib()  # fail loudly if the library is missing
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 132 * 2 ** 20)
    hbm_peak, bf16_peak, peak_src = measured_peaks()

    def bf(a):
        import numpy as np
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    # ---------------- headline workload buffers
    n_copies = {}
    W, SW = {}, {}
    for (K, N) in LINEARS:
        wbytes = K * N
        n_copies[(K, N)] = max(20, -(-2 * l2 // wbytes) + 1)
        W[(K, N)] = [synth.uniform_int8_device((N, K), SEED + 100 * i + K + N, dev) for i in range(n_copies[(K, N)])]
        SW[(K, N)] = [synth.uniform_f32_device((N,), 1e-3, 1e-2, SEED + 7 + 100 * i + N, dev)
                      for i in range(n_copies[(K, N)])]
    X, XQ, SX, Y, YF = {}, {}, {}, {}, {}
    for (K, N) in LINEARS:
        for M in MS:
            X[(K, N, M)] = bf(synth.activations(M, K, SEED + 1000 + M + K))
            XQ[(K, N, M)] = torch.empty((M, K), dtype=torch.int8, device=dev)
            SX[(K, N, M)] = torch.empty((M,), dtype=torch.float32, device=dev)
            Y[(K, N, M)] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            YF[(K, N, M)] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws_bytes = max(fq.workspace_bytes(fq.OP_W8A8_QUANT_LINEAR, 64, K, N) for (K, N) in LINEARS)
    ws_bytes = max(ws_bytes, fq.workspace_bytes(fq.OP_FP8_GROUP_EINSUM, 256, 4096, 1024, 8))
    ws = fq.new_workspace(ws_bytes, dev)

    def call_quant(K, N, M):
        fq.dynamic_quant_int8(X[(K, N, M)], XQ[(K, N, M)], SX[(K, N, M)])

    def call_gemm(K, N, M, c):
        fq.w8a8_linear(XQ[(K, N, M)], SX[(K, N, M)], W[(K, N)][c], SW[(K, N)][c], y=Y[(K, N, M)], ws=ws)

    def call_fused(K, N, M, c):
        fq.w8a8_quant_linear(X[(K, N, M)], W[(K, N)][c], SW[(K, N)][c], y=YF[(K, N, M)], ws=ws)

    # launches per fused call, as the library reports its own schedule choice
    # (FQ_DEBUG_SCHEDULE): "dp224+quant" is one launch, anything else a quant
    # launch plus a GEMM launch
    fused_sched = library_schedules(lambda: [call_fused(K, N, M, 10 + i) for (K, N) in LINEARS
                                             for i, M in enumerate(MS)], torch)
    fused_n = {key: (1 if "dp224+quant" in sched else 2) for key, sched in
               zip([(K, N, M) for (K, N) in LINEARS for M in MS], fused_sched)}

    def fused_launches(M, K, N):
        return fused_n[(K, N, M)]

    small, big = LINEARS
    groups = [
        ("quant", lambda: [call_quant(K, N, M) for (K, N) in LINEARS for M in MS],
         sum(bytes_quant(M, K) for (K, N) in LINEARS for M in MS), 2 * len(MS)),
        ("gemm_K4096_N1024", lambda: [call_gemm(*small, M, i) for i, M in enumerate(MS)],
         sum(bytes_gemm(M, *small) for M in MS), len(MS)),
        ("gemm_K1024_N32768", lambda: [call_gemm(*big, M, i) for i, M in enumerate(MS)],
         sum(bytes_gemm(M, *big) for M in MS), len(MS)),
        ("fused_K4096_N1024", lambda: [call_fused(*small, M, 10 + i) for i, M in enumerate(MS)],
         sum(bytes_fused(M, *small) for M in MS), sum(fused_launches(M, *small) for M in MS)),
        ("fused_K1024_N32768", lambda: [call_fused(*big, M, 10 + i) for i, M in enumerate(MS)],
         sum(bytes_fused(M, *big) for M in MS), sum(fused_launches(M, *big) for M in MS)),
    ]
    launches_per_step = sum(g[3] for g in groups)

    # eager warm-up of every call (lazy host-side set-up), then capture
    for _, fn, _, _ in groups:
        fn()
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(dev)
    graphs = []
    for name, fn, nbytes, nl in groups:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn()
        graphs.append((name, g, nbytes, nl))
    torch.cuda.synchronize()

    def step(evs=None):
        for i, (_, g, _, _) in enumerate(graphs):
            if evs is not None:
                evs[i].record()
            g.replay()
        if evs is not None:
            evs[len(graphs)].record()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()

    K_steps = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)] for _ in range(K_steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    w0 = time.time()
    t_start.record()
    for k in range(K_steps):
        step(evs[k])
    t_end.record()
    torch.cuda.synchronize()
    w1 = time.time()
    if dist is not None:
        dist.barrier()
    time.sleep(0.15)
    clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    if dist is not None:
        total_ms = max_over_ranks(total_ms, dist, dev)
    group_ms = [sum(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(K_steps)) / K_steps for i in range(len(graphs))]
    ms_per_step = total_ms / K_steps
    sb = step_bytes()
    value = whole_job_value(sb, ms_per_step, world)

    group_report = {}
    for (name, _, nbytes, nl), ms in zip(graphs, group_ms):
        gbps = nbytes / (ms * 1e-3) / 1e9
        group_report[name] = {"us_per_step": round(ms * 1e3, 2), "launches": nl, "GBps": round(gbps, 1),
                              "frac_hbm": round(gbps / hbm_peak, 3)}

    # roofline of the dominant kernel: the W8A8 GEMM on the (K=1024, N=32768) linear
    dom_ms = group_ms[2]
    dom_bytes_per_launch = groups[2][2] / len(MS)
    achieved = dom_bytes_per_launch / (dom_ms * 1e-3 / len(MS)) / 1e9
    big_sched = library_schedules(lambda: [call_gemm(*big, M, i) for i, M in enumerate(MS)], torch)
    kern = {"dp224": "w8a8_gemm_kernel<MT,14> (224-row tiles)", "umma": "w8a8_umma_kernel (tcgen05)",
            "streamk": "w8a8_gemm_kernel<MT,8> (stream-K)", "cluster4": "w8a8_cluster_kernel"}
    ran = []
    for sch, M in zip(big_sched, MS):
        name = kern.get(sch, sch)
        if not ran or ran[-1][0] != name:
            ran.append([name, []])
        ran[-1][1].append(M)
    roofline = {"kernel": "W8A8 GEMM on (K=1024, N=32768), M in 1..64: " +
                          "; ".join("%s at M=%s" % (n, ",".join(map(str, ms))) for n, ms in ran),
                "bound": "hbm",
                "achieved": round(achieved, 1), "peak": hbm_peak, "peak_source": peak_src + " hbm_gbs",
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 3),
                "traffic": traffic_for("w8a8_gemm_kernel@K1024xN32768",
                                       ["fp8_dynamic_quant_gb300/csrc/gemm_w8a8.cu",
                                        "fp8_dynamic_quant_gb300/csrc/fq_common.cuh"]),
                "algorithmic_bytes_per_launch": int(dom_bytes_per_launch),
                "avg_launch_us": round(dom_ms * 1e3 / len(MS), 3)}

    out = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K_steps,
           "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
           "config": workload_config(),
           "timing": "op groups captured as CUDA graphs, replayed; CUDA events on the launching stream",
           "parallelism": "replicas" if world > 1 else "single GPU",
           "gpu_launches": launches_per_step * K_steps,
           "groups": group_report, "roofline": roofline}
    clk = clocks.summary(w0, w1)
    out["clocks"] = clk

    if rank == 0:
        out["engine_peaks"] = engine_peaks(torch, dev)
        ep = out["engine_peaks"] or {}
        # compute term of the roofline kernel: 2MNK per launch against the engine it runs on
        ops = sum(2.0 * M * big[0] * big[1] for M in MS) / len(MS)
        eng = ep.get("mma_sync_f16_m16n8k16")
        roofline["compute"] = {"ops_per_launch": ops, "engine": "mma.sync f16 (M<=16) / tcgen05 kind::f16 (M=32,64); "
                               "peak: the mma.sync f16 one (the lower)",
                               "engine_peak_tflops": eng,
                               "achieved_tflops": round(ops / (dom_ms * 1e-3 / len(MS)) / 1e12, 2),
                               "frac": round(ops / (dom_ms * 1e-3 / len(MS)) / 1e12 / eng, 4) if eng else None}
    if rank == 0 and not args.no_extras:
        out["per_call"] = per_call_breakdown(fq, torch, dev, W, SW, X, XQ, SX, Y, YF, ws, hbm_peak)
        out["other_configs"] = other_configs(fq, synth, torch, dev, bf, l2, hbm_peak)
        out["e2e"] = e2e(fq, torch, dev, W, SW, X, ws, args)
    else:
        out["e2e"] = e2e(fq, torch, dev, W, SW, X, ws, args) if rank == 0 else None
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    return out


def time_graph(torch, fn, reps=3, calls=1):
    """Capture fn() in a CUDA graph and return microseconds per call (median of reps replays)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        fn()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3 / calls)
    return statistics.median(ts)


def time_eager(torch, fn, calls, reps=3):
    """Microseconds per call of `calls` eager calls issued back to back (fn issues them), CUDA events
    on the current stream, median of reps: the launch floor the graph series hides."""
    fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3 / calls)
    return statistics.median(ts)


def per_call_breakdown(fq, torch, dev, W, SW, X, XQ, SX, Y, YF, ws, hbm_peak):
    """Microseconds and GB/s per call for every (op, linear, M), each call on a different weight copy:
    CUDA-graph replays (the *_us series) and the same calls issued eagerly (*_eager_us)."""
    res = {}
    for (K, N) in LINEARS:
        nc = len(W[(K, N)])
        key = "K%d_N%d" % (K, N)
        res[key] = {"M": MS, "quant_us": [], "gemm_us": [], "fused_us": [], "gemm_GBps": [], "fused_GBps": [],
                    "gemm_frac_hbm": [], "fused_frac_hbm": [], "quant_eager_us": [], "gemm_eager_us": [],
                    "fused_eager_us": [], "weight_copies_per_graph": nc}
        for M in MS:
            R = 16
            tq = time_graph(torch, lambda: [fq.dynamic_quant_int8(X[(K, N, M)], XQ[(K, N, M)], SX[(K, N, M)])
                                            for _ in range(R)], calls=R)
            tg = time_graph(torch, lambda: [fq.w8a8_linear(XQ[(K, N, M)], SX[(K, N, M)], W[(K, N)][c], SW[(K, N)][c],
                                                           y=Y[(K, N, M)], ws=ws) for c in range(nc)], calls=nc)
            tf = time_graph(torch, lambda: [fq.w8a8_quant_linear(X[(K, N, M)], W[(K, N)][c], SW[(K, N)][c],
                                                                 y=YF[(K, N, M)], ws=ws) for c in range(nc)], calls=nc)
            eq = time_eager(torch, lambda: [fq.dynamic_quant_int8(X[(K, N, M)], XQ[(K, N, M)], SX[(K, N, M)])
                                            for _ in range(R)], R)
            eg = time_eager(torch, lambda: [fq.w8a8_linear(XQ[(K, N, M)], SX[(K, N, M)], W[(K, N)][c], SW[(K, N)][c],
                                                           y=Y[(K, N, M)], ws=ws) for c in range(nc)], nc)
            ef = time_eager(torch, lambda: [fq.w8a8_quant_linear(X[(K, N, M)], W[(K, N)][c], SW[(K, N)][c],
                                                                 y=YF[(K, N, M)], ws=ws) for c in range(nc)], nc)
            res[key]["quant_eager_us"].append(round(eq, 2))
            res[key]["gemm_eager_us"].append(round(eg, 2))
            res[key]["fused_eager_us"].append(round(ef, 2))
            gb = bytes_gemm(M, K, N) / (tg * 1e-6) / 1e9
            fb = bytes_fused(M, K, N) / (tf * 1e-6) / 1e9
            res[key]["quant_us"].append(round(tq, 2))
            res[key]["gemm_us"].append(round(tg, 2))
            res[key]["fused_us"].append(round(tf, 2))
            res[key]["gemm_GBps"].append(round(gb, 1))
            res[key]["fused_GBps"].append(round(fb, 1))
            res[key]["gemm_frac_hbm"].append(round(gb / hbm_peak, 3))
            res[key]["fused_frac_hbm"].append(round(fb / hbm_peak, 3))
    return res


def other_configs(fq, synth, torch, dev, bf, l2, hbm_peak):
    import numpy as np
    res = {}
    # --- FP8 per-128 group quant with packed UE8M0 scales, G=8, D=4096
    G, D = 8, 4096
    fp8q = {}
    for T in [1, 3, 4, 17, 128, 4096]:
        copies = max(1, -(-2 * l2 // (2 * T * G * D)))
        copies = min(copies, 8)
        xs = [bf(synth.group_activations(T, G, D, SEED + 2 + c)) for c in range(copies)]
        xq = torch.empty((T, G, D), dtype=torch.float8_e4m3fn, device=dev)
        st = torch.empty((G, 8, (T + 3) // 4 * 4), dtype=torch.int32, device=dev)
        R = max(copies, 8)
        us = time_graph(torch, lambda: [fq.quant_fp8_group_ue8m0_packed(xs[i % copies], xq, st) for i in range(R)],
                        calls=R)
        gb = bytes_group_quant(T, G, D) / (us * 1e-6) / 1e9
        fp8q[str(T)] = {"us": round(us, 2), "GBps": round(gb, 1), "frac_hbm": round(gb / hbm_peak, 3)}
        del xs
    res["fp8_group_quant_ue8m0_packed_G8_D4096"] = fp8q
    # --- per-token INT8 quant at a size where HBM matters: M=16384, K=4096 (201 MB moved)
    M, K = 16384, 4096
    xs = [bf(synth.activations(M, K, SEED + 9 + c)) for c in range(2)]
    xq = torch.empty((M, K), dtype=torch.int8, device=dev)
    sx = torch.empty((M,), dtype=torch.float32, device=dev)
    us = time_graph(torch, lambda: [fq.dynamic_quant_int8(xs[i % 2], xq, sx) for i in range(4)], calls=4)
    gb = bytes_quant(M, K) / (us * 1e-6) / 1e9
    res["int8_quant_M16384_K4096"] = {"us": round(us, 2), "GBps": round(gb, 1), "frac_hbm": round(gb / hbm_peak, 3)}
    del xs
    # --- block-scaled FP8 einsum (wo_a-like), W [8, 4096, 1024], both scale formats; and the repack control
    N = 1024
    ncp = max(2, -(-2 * l2 // (G * D * N)) + 1)
    wq, sw = [], []
    for c in range(ncp):
        w = torch.randn((G, N, D), generator=torch.Generator(device=dev).manual_seed(SEED + 50 + c),
                        device=dev, dtype=torch.float32) * 0.02
        a, b = fq.quantize_weight_fp8_block(w)
        wq.append(a)
        sw.append(b)
        del w
    ein = {}
    for T in [1, 4, 16, 64, 256]:
        x = bf(synth.group_activations(T, G, D, SEED + 3 + T))
        xq8, st = fq.quant_fp8_group_ue8m0_packed(x)
        _, s32 = fq.quant_fp8_group_fp32(x)
        y = torch.empty((T, G, N), dtype=torch.bfloat16, device=dev)
        wsz = fq.new_workspace(fq.workspace_bytes(fq.OP_FP8_GROUP_EINSUM, T, D, N, G), dev)
        tp = time_graph(torch, lambda: [fq.fp8_group_einsum(xq8, st, fq.SCALE_UE8M0_PACKED, wq[c], sw[c], y=y, ws=wsz)
                                        for c in range(ncp)], calls=ncp)
        tf = time_graph(torch, lambda: [fq.fp8_group_einsum(xq8, s32, fq.SCALE_FP32, wq[c], sw[c], y=y, ws=wsz)
                                        for c in range(ncp)], calls=ncp)
        # decode-step A/B: producer writes packed scales directly, vs fp32 scales + separate repack
        xqa = torch.empty_like(xq8)
        sta = torch.empty_like(st)
        s32a = torch.empty_like(s32)
        t_direct = time_graph(torch, lambda: [(fq.quant_fp8_group_ue8m0_packed(x, xqa, sta),
                                               fq.fp8_group_einsum(xqa, sta, fq.SCALE_UE8M0_PACKED, wq[c], sw[c],
                                                                   y=y, ws=wsz)) for c in range(ncp)], calls=ncp)
        t_control = time_graph(torch, lambda: [(fq.quant_fp8_group_fp32(x, xqa, s32a), fq.pack_scales_ue8m0(s32a, sta),
                                                fq.fp8_group_einsum(xqa, sta, fq.SCALE_UE8M0_PACKED, wq[c], sw[c],
                                                                    y=y, ws=wsz)) for c in range(ncp)], calls=ncp)
        nbytes = bytes_einsum(T, G, D, N)
        gb = nbytes / (tp * 1e-6) / 1e9
        flops = 2.0 * T * G * D * N
        ein[str(T)] = {"packed_us": round(tp, 2), "fp32_us": round(tf, 2), "GBps": round(gb, 1),
                       "frac_hbm": round(gb / hbm_peak, 3), "TFLOPs": round(flops / (tp * 1e-6) / 1e12, 1),
                       "quant_plus_einsum_us": round(t_direct, 2),
                       "control_quant_fp32_repack_einsum_us": round(t_control, 2)}
    res["fp8_group_einsum_G8_D4096_N1024"] = ein
    del wq, sw
    # --- RMSNorm fused with the INT8 per-token / FP8 per-group quant, K = 4096
    K = 4096
    gam = bf(synth.activations(1, K, SEED + 60)[0])
    rq = {}
    for M in [1, 4, 16, 64, 16384]:
        copies = max(1, min(8, -(-2 * l2 // (2 * M * K))))
        xs = [bf(synth.activations(M, K, SEED + 61 + c)) for c in range(copies)]
        xq = torch.empty((M, K), dtype=torch.int8, device=dev)
        sx = torch.empty((M,), dtype=torch.float32, device=dev)
        x8 = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
        s8 = torch.empty((1, (K // 128 + 3) // 4, (M + 3) // 4 * 4), dtype=torch.int32, device=dev)
        R = max(copies, 8)
        ui = time_graph(torch, lambda: [fq.rmsnorm_quant_int8(xs[i % copies], gam, 1e-6, xq, sx) for i in range(R)],
                        calls=R)
        uf = time_graph(torch, lambda: [fq.rmsnorm_quant_fp8_ue8m0_packed(xs[i % copies], gam, 1e-6, x8, s8)
                                        for i in range(R)], calls=R)
        bi = 3 * M * K + 2 * K + 4 * M
        bfp = 3 * M * K + 2 * K + 4 * s8.numel()
        rq[str(M)] = {"int8_us": round(ui, 2), "int8_GBps": round(bi / (ui * 1e-6) / 1e9, 1),
                      "fp8_us": round(uf, 2), "fp8_GBps": round(bfp / (uf * 1e-6) / 1e9, 1),
                      "int8_frac_hbm": round(bi / (ui * 1e-6) / 1e9 / hbm_peak, 3)}
        del xs
    res["rmsnorm_quant_K4096"] = rq
    # --- 32-element block-scaled FP8 (MXFP8-like): producer and tensor-core block-scaled linear
    mxr = {}
    for (K, N) in LINEARS:
        ncp = max(2, -(-2 * l2 // (K * N)) + 1)
        wl = []
        for c in range(ncp):
            wb = (torch.randn((N, K), generator=torch.Generator(device=dev).manual_seed(SEED + 80 + c), device=dev)
                  * 0.02).to(torch.bfloat16)
            wl.append(fq.quant_mxfp8(wb))
            del wb
        row = {}
        for M in [1, 4, 16, 64, 128]:
            xb = bf(synth.activations(M, K, SEED + 81 + M))
            qx, sxb = fq.quant_mxfp8(xb)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            wsm = fq.new_workspace(fq.workspace_bytes(fq.OP_MXFP8_LINEAR, M, K, N), dev)
            us = time_graph(torch, lambda: [fq.mxfp8_linear(qx, sxb, wl[c][0], wl[c][1], y=y, ws=wsm)
                                            for c in range(ncp)], calls=ncp)
            nbytes = N * K + N * K // 32 + M * K + M * K // 32 + 2 * M * N
            row[str(M)] = {"us": round(us, 2), "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                           "frac_hbm": round(nbytes / (us * 1e-6) / 1e9 / hbm_peak, 3)}
        mxr["linear_K%d_N%d" % (K, N)] = row
        del wl
    M, K = 16384, 4096
    xs = [bf(synth.activations(M, K, SEED + 90 + c)) for c in range(2)]
    q8 = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    sfb = torch.empty(((M + 127) // 128, K // 128, 512), dtype=torch.uint8, device=dev)
    us = time_graph(torch, lambda: [fq.quant_mxfp8(xs[i % 2], q8, sfb) for i in range(4)], calls=4)
    nbytes = 3 * M * K + M * K // 32
    mxr["quant_M16384_K4096"] = {"us": round(us, 2), "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                                 "frac_hbm": round(nbytes / (us * 1e-6) / 1e9 / hbm_peak, 3)}
    del xs
    res["mxfp8_block32"] = mxr
    # --- expert-local M_e sweep of the grouped W8A8 linear: 16 experts of M_e rows each
    Ex = 16
    me_res = {}
    for (K, N, name) in [(4096, 4096, "W13_K4096_N4096"), (2048, 4096, "W2_K2048_N4096")]:
        wg = synth.uniform_int8_device((Ex, N, K), SEED + 70 + K, dev)
        swg = synth.uniform_f32_device((Ex, N), 1e-3, 1e-2, SEED + 71 + K, dev)
        row = {}
        for Me in [1, 2, 4, 8, 16, 32, 64, 96, 127, 128, 129, 160, 192, 256]:
            R = Ex * Me
            xg = synth.uniform_int8_device((R, K), SEED + 72 + Me, dev)
            sg = synth.uniform_f32_device((R,), 1e-3, 1e-2, SEED + 73 + Me, dev)
            offs = torch.arange(0, R + 1, Me, dtype=torch.int32, device=dev)
            yg = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
            wsg = fq.new_workspace(fq.workspace_bytes(fq.OP_W8A8_GROUPED_LINEAR, R, K, N, Ex), dev)
            us = time_graph(torch, lambda: fq.w8a8_grouped_linear(xg, sg, offs, wg, swg, y=yg, ws=wsg), reps=3,
                            calls=1)
            nbytes = Ex * N * K + 4 * Ex * N + R * K + 4 * R + 2 * R * N
            row[str(Me)] = {"us": round(us, 1), "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                            "TOPS": round(2.0 * R * N * K / (us * 1e-6) / 1e12, 1)}
            del xg, yg, wsg
        me_res[name] = row
        del wg, swg
    res["grouped_w8a8_Me_sweep_16_experts"] = me_res
    torch.cuda.empty_cache()
    # --- MoE expert chain: 256 tokens, hidden 4096, 256 experts, top-8 Zipf(1.1), intermediate 2048
    T, topk, E, H, I = 256, 8, 256, 4096, 2048
    c = synth.moe_case(T, topk, E, H, I, SEED + 4, with_weights=False)
    Wd = synth.moe_weights_device(E, H, I, SEED + 4, dev)
    x = bf(c["x"])
    ids = torch.from_numpy(c["topk_ids"]).to(dev)
    tw = torch.from_numpy(c["topk_w"]).to(dev)
    bufs = fq.MoEBuffers(T, topk, E, H, I, dev)
    us = time_graph(torch, lambda: fq.moe_forward(x, ids, tw, Wd["w13"], Wd["sw13"], Wd["w2"], Wd["sw2"], bufs=bufs),
                    reps=5)
    touched = int(np.unique(c["topk_ids"]).size)
    R = T * topk
    wbytes = touched * (2 * I * H + H * I + 4 * (2 * I + H))
    abytes = (3 * T * H + 4 * T) + 2 * R * H + (R * H + 2 * R * 2 * I) + (2 * R * 2 * I + R * I) + \
        (R * I + 2 * R * H) + (2 * R * H + 2 * T * H)
    gb = (wbytes + abytes) / (us * 1e-6) / 1e9
    res["moe_chain_T256_E256_top8"] = {"us": round(us, 1), "touched_experts": touched, "GBps": round(gb, 1),
                                       "frac_hbm": round(gb / hbm_peak, 3),
                                       "algorithmic_bytes": int(wbytes + abytes)}
    del Wd, bufs
    torch.cuda.empty_cache()
    return res


def e2e(fq, torch, dev, W, SW, X, ws, args):
    """The headline step through the public API with host buffers.  Every step
    copies all of its inputs from one pinned host staging buffer to the device
    (one copy), makes the step's 60 public-API calls on views of that buffer,
    and reads all of their results back into one pinned host buffer (one
    copy): what a serving loop that stages a batch does.  The inputs are the
    quant's and the fused op's bf16 activations and the linear's int8
    activations with their scales (host data: the quant's results)."""
    ALIGN = 256  # every view starts on a 256-byte boundary (the kernels need 16)

    def layout(items):
        off, views = 0, {}
        for key, nbytes in items:
            views[key] = (off, nbytes)
            off += -(-nbytes // ALIGN) * ALIGN
        return views, off

    ins, outs = [], []
    for (K, N) in LINEARS:
        for M in MS:
            k = (K, N, M)
            ins += [(k + ("x",), 2 * M * K), (k + ("xq",), M * K), (k + ("sx",), 4 * M), (k + ("x3",), 2 * M * K)]
            outs += [(k + ("xq",), M * K), (k + ("sx",), 4 * M), (k + ("y",), 2 * M * N), (k + ("yf",), 2 * M * N)]
    vin, nin = layout(ins)
    vout, nout = layout(outs)
    h2d = sum(n for _, n in ins)
    d2h = sum(n for _, n in outs)
    hin = torch.zeros(nin, dtype=torch.uint8).pin_memory()
    hout = torch.zeros(nout, dtype=torch.uint8).pin_memory()
    din = torch.zeros(nin, dtype=torch.uint8, device=dev)
    dout = torch.zeros(nout, dtype=torch.uint8, device=dev)

    def view(buf, views, key, dtype, shape):
        off, nbytes = views[key]
        return buf[off:off + nbytes].view(dtype).view(shape)

    # host inputs: the activations, and the int8 quant of them for the linear
    for (K, N) in LINEARS:
        for M in MS:
            k = (K, N, M)
            x = X[k]
            xq, sx = fq.dynamic_quant_int8(x)
            view(hin, vin, k + ("x",), torch.bfloat16, (M, K)).copy_(x.cpu())
            view(hin, vin, k + ("x3",), torch.bfloat16, (M, K)).copy_(x.cpu())
            view(hin, vin, k + ("xq",), torch.int8, (M, K)).copy_(xq.cpu())
            view(hin, vin, k + ("sx",), torch.float32, (M,)).copy_(sx.cpu())
    calls = []
    for (K, N) in LINEARS:
        for i, M in enumerate(MS):
            k = (K, N, M)
            calls.append((i, K, N, M,
                          view(din, vin, k + ("x",), torch.bfloat16, (M, K)),
                          view(din, vin, k + ("xq",), torch.int8, (M, K)),
                          view(din, vin, k + ("sx",), torch.float32, (M,)),
                          view(din, vin, k + ("x3",), torch.bfloat16, (M, K)),
                          view(dout, vout, k + ("xq",), torch.int8, (M, K)),
                          view(dout, vout, k + ("sx",), torch.float32, (M,)),
                          view(dout, vout, k + ("y",), torch.bfloat16, (M, N)),
                          view(dout, vout, k + ("yf",), torch.bfloat16, (M, N))))

    def one_step():
        din.copy_(hin, non_blocking=True)
        for (i, K, N, M, x, xq, sx, x3, oq, os_, y, yf) in calls:
            fq.dynamic_quant_int8(x, oq, os_)
            fq.w8a8_linear(xq, sx, W[(K, N)][i], SW[(K, N)][i], y=y, ws=ws)
            fq.w8a8_quant_linear(x3, W[(K, N)][10 + i], SW[(K, N)][10 + i], y=yf, ws=ws)
        hout.copy_(dout, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(3):
        one_step()
    n = max(50, min(400, args.steps // 10))
    t0 = time.perf_counter()
    for _ in range(n):
        one_step()
    dt = (time.perf_counter() - t0) / n
    return {"value": round(step_bytes() / dt / 1e9, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(dt * 1e3, 3), "steps": n,
            "how": "eager public-API calls (60 a step) on views of one device buffer; every step one H2D copy "
                   "of all its inputs from a pinned host staging buffer and one D2H copy of all its results, "
                   "inside the timed loop, wall clock"}


# ---------------------------------------------------------------- the oracle (CPU baseline / reference arm)
BLAS_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                    "NUMEXPR_NUM_THREADS", "VECLIB_MAXIMUM_THREADS")


def oracle_workload(path):
    """Writes the headline step's oracle inputs (numpy arrays) to `path` (.npz)."""
    import numpy as np
    from fp8_dynamic_quant_gb300 import synth
    arrs = {}
    for (K, N) in LINEARS:
        arrs["w_%d_%d" % (K, N)] = synth.uniform_int8((N, K), SEED + K + N)
        arrs["sw_%d_%d" % (K, N)] = synth.channel_scales(N, SEED + 7 + N)
        for M in MS:
            arrs["x_%d_%d" % (K, M)] = synth.activations(M, K, SEED + 1000 + M + K)
    np.savez(path, **arrs)


def oracle_calls(path):
    """The headline step as a list of oracle calls (label, fn, algorithmic bytes), inputs read from `path`."""
    import numpy as np
    from oracle import int8 as oi8
    a = np.load(path)
    calls = []
    for (K, N) in LINEARS:
        w, sw = a["w_%d_%d" % (K, N)], a["sw_%d_%d" % (K, N)]
        for M in MS:
            x = a["x_%d_%d" % (K, M)]
            q, s = oi8.dynamic_quant_int8(x)
            calls.append(("quant", (lambda x=x: oi8.dynamic_quant_int8(x)), bytes_quant(M, K)))
            calls.append(("gemm", (lambda q=q, s=s, w=w, sw=sw: oi8.w8a8_linear(q, s, w, sw)), bytes_gemm(M, K, N)))
            calls.append(("fused", (lambda x=x, w=w, sw=sw: oi8.w8a8_quant_linear(x, w, sw)), bytes_fused(M, K, N)))
    return calls


def _oracle_proc(path, start, rounds, seconds, barrier, results):
    """One single-threaded oracle process: `rounds` rounds, each starting at the shared barrier and
    running oracle calls round-robin (from call `start`) for at least `seconds`."""
    calls = oracle_calls(path)
    i = start
    out = []
    for _ in range(rounds):
        barrier.wait()
        t0 = time.perf_counter()
        b = n = 0
        while True:
            _, fn, nb = calls[i % len(calls)]
            fn()
            b += nb
            n += 1
            i += 1
            if time.perf_counter() - t0 >= seconds:
                break
        out.append((b, n, time.perf_counter() - t0))
    results.put(out)


def oracle_rate(workers, rounds, seconds):
    """Runs the oracle in `workers` spawned processes, each with one BLAS thread, for `rounds` rounds
    of about `seconds` each.  Returns per-round (bytes, calls, wall seconds) summed over the workers;
    a round's wall time is its slowest worker's."""
    import multiprocessing
    import tempfile
    ctx = multiprocessing.get_context("spawn")      # no fork after CUDA is up
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "oracle_inputs.npz")
        oracle_workload(path)
        saved = {v: os.environ.get(v) for v in BLAS_THREAD_VARS}
        for v in BLAS_THREAD_VARS:
            os.environ[v] = "1"
        try:
            barrier = ctx.Barrier(workers)
            results = ctx.Queue()
            ncalls = 3 * len(LINEARS) * len(MS)
            procs = [ctx.Process(target=_oracle_proc, args=(path, (k * 7) % ncalls, rounds, seconds, barrier,
                                                            results)) for k in range(workers)]
            for p in procs:
                p.start()
            per = [results.get() for _ in procs]
            for p in procs:
                p.join()
        finally:
            for v, val in saved.items():
                if val is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = val
    return [(sum(w[r][0] for w in per), sum(w[r][1] for w in per), max(w[r][2] for w in per))
            for r in range(rounds)]


def cpu_baseline(budget_s=20.0):
    """The oracle as it stands on the host cores, over a bounded sample of the headline step: once
    single-threaded, once in one single-threaded process per core.  The headline object is the
    all-cores run; the single-thread run is reported beside it."""
    ncpu = os.cpu_count() or 1
    (b1, n1, t1), = oracle_rate(1, 1, 0.4 * budget_s)
    (bn, nn, tn), = oracle_rate(ncpu, 1, 0.6 * budget_s)
    return {"value": round(bn / tn / 1e9, 4), "unit": UNIT, "cores": ncpu, "kind": "oracle",
            "sample": "%d oracle calls cycling over the 60 calls of one headline step (quant, GEMM, fused per "
                      "linear and M) in %d single-threaded processes (one per core), %.1f s wall" % (nn, ncpu, tn),
            "single_thread": {"value": round(b1 / t1 / 1e9, 4), "unit": UNIT, "cores": 1,
                              "sample": "%d oracle calls in one process with one BLAS thread, %.1f s" % (n1, t1)}}


def workload_config():
    """The `config` object of the bench line, the same for both arms."""
    return {"workload": "INT8 W8A8 M-sweep: per-token quant, W8A8 GEMM and fused quant+GEMM on "
                        "(K=4096,N=1024) and (K=1024,N=32768), M in {1,2,3,4,7,8,9,16,32,64}",
            "linears": [list(l) for l in LINEARS], "M": MS,
            "bytes_per_step": step_bytes(),
            "l2": "each call reads its own weight copy; %d MB of weights per step (> 2x the 126 MB L2) so every "
                  "call streams weights from HBM; activations L2-hot" %
                  (sum(K * N for (K, N) in LINEARS) * 20 // 2 ** 20)}


def run_reference(args):
    """Reference arm: the CPU oracle in one single-threaded process per host core, each step a bounded
    round of the headline workload's oracle calls."""
    ncpu = os.cpu_count() or 1
    budget_total = float(os.environ.get("FQ_REF_BUDGET_S", "120"))
    per_step = max(0.05, budget_total / max(1, args.steps + args.warmup))
    rounds = oracle_rate(ncpu, args.warmup + args.steps, per_step)[args.warmup:]
    tot_b = sum(r[0] for r in rounds)
    dt = sum(r[2] for r in rounds)
    calls = sum(r[1] for r in rounds)
    v = tot_b / dt / 1e9
    sample = ("each step: oracle calls of the headline sweep round-robin for >= %.3f s in %d single-threaded "
              "processes (one per core); %d timed calls" % (per_step, ncpu, calls))
    return {"metric": METRIC, "value": round(v, 4), "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / max(1, args.steps), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic", "impl": "reference",
            "config": workload_config(),
            "timing": "host wall clock per round; rounds start together at a process barrier",
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": ncpu, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_profile_case(name):
    """Run one op of the workload a few times, untimed, as a target for a profiler.

    gemm_K1024_N32768 / gemm_K4096_N1024: the W8A8 GEMM once per M of the sweep,
    each call on its own weight copy; fused_K1024_N32768: the fused quant + GEMM
    the same way; einsum_T<T>: the block-scaled FP8 einsum
    (G=8, D=4096, N=1024) three times; int8_quant_M16384: the per-token quant
    at M=16384, K=4096 twice; rmsnorm_quant_M16384: RMSNorm + INT8 quant at
    M=16384, K=4096 twice; mxfp8_K4096_N1024 / mxfp8_K1024_N32768: the
    32-element block-scaled linear at M=16 three times on one weight set;
    fp8_group_quant_T4096: the group quant with packed UE8M0 scales at T=4096,
    G=8, D=4096 twice.  Prints one status line."""
    import torch
    import fp8_dynamic_quant_gb300 as fq
    from fp8_dynamic_quant_gb300 import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fq.lib()

    def bf(a):
        import numpy as np
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    launches = 0
    if name.startswith("gemm_"):
        K, N = {"gemm_K1024_N32768": (1024, 32768), "gemm_K4096_N1024": (4096, 1024)}[name]
        ws = fq.new_workspace(fq.workspace_bytes(fq.OP_W8A8_LINEAR, 64, K, N), dev)
        for i, M in enumerate(MS):
            w = synth.uniform_int8_device((N, K), SEED + 100 * i + K + N, dev)
            sw = synth.uniform_f32_device((N,), 1e-3, 1e-2, SEED + 7 + 100 * i + N, dev)
            xq, sx = fq.dynamic_quant_int8(bf(synth.activations(M, K, SEED + 1000 + M + K)))
            fq.w8a8_linear(xq, sx, w, sw, ws=ws)
            launches += 1
    elif name == "fused_K1024_N32768":
        K, N = 1024, 32768
        ws = fq.new_workspace(fq.workspace_bytes(fq.OP_W8A8_QUANT_LINEAR, 64, K, N), dev)
        for i, M in enumerate(MS):
            w = synth.uniform_int8_device((N, K), SEED + 100 * i + K + N, dev)
            sw = synth.uniform_f32_device((N,), 1e-3, 1e-2, SEED + 7 + 100 * i + N, dev)
            fq.w8a8_quant_linear(bf(synth.activations(M, K, SEED + 1000 + M + K)), w, sw, ws=ws)
            launches += 1
    elif name.startswith("einsum_T"):
        T, G, D, N = int(name[len("einsum_T"):]), 8, 4096, 1024
        w = torch.randn((G, N, D), generator=torch.Generator(device=dev).manual_seed(SEED + 50),
                        device=dev, dtype=torch.float32) * 0.02
        wq, sw = fq.quantize_weight_fp8_block(w)
        del w
        xq8, st = fq.quant_fp8_group_ue8m0_packed(bf(synth.group_activations(T, G, D, SEED + 3 + T)))
        for _ in range(3):
            fq.fp8_group_einsum(xq8, st, fq.SCALE_UE8M0_PACKED, wq, sw)
            launches += 1
    elif name == "int8_quant_M16384":
        x = bf(synth.activations(16384, 4096, SEED + 9))
        for _ in range(2):
            fq.dynamic_quant_int8(x)
            launches += 1
    elif name == "rmsnorm_quant_M16384":
        x = bf(synth.activations(16384, 4096, SEED + 61))
        gam = bf(synth.activations(1, 4096, SEED + 60)[0])
        for _ in range(2):
            fq.rmsnorm_quant_int8(x, gam, 1e-6)
            launches += 1
    elif name.startswith("mxfp8_"):
        K, N = {"mxfp8_K4096_N1024": (4096, 1024), "mxfp8_K1024_N32768": (1024, 32768)}[name]
        wb = (torch.randn((N, K), generator=torch.Generator(device=dev).manual_seed(SEED + 80), device=dev) * 0.02).to(
            torch.bfloat16)
        wq, wsf = fq.quant_mxfp8(wb)
        del wb
        qx, sxb = fq.quant_mxfp8(bf(synth.activations(16, K, SEED + 81 + 16)))
        ws = fq.new_workspace(fq.workspace_bytes(fq.OP_MXFP8_LINEAR, 16, K, N), dev)
        for _ in range(3):
            fq.mxfp8_linear(qx, sxb, wq, wsf, ws=ws)
            launches += 1
    elif name == "fp8_group_quant_T4096":
        x = bf(synth.group_activations(4096, 8, 4096, SEED + 2))
        for _ in range(2):
            fq.quant_fp8_group_ue8m0_packed(x)
            launches += 1
    else:
        raise SystemExit("unknown profile case: " + name)
    torch.cuda.synchronize()
    st_, word = fq.device_error()
    print(json.dumps({"profile_case": name, "op_calls": launches, "device_error": int(word)}))
    return 0 if st_ == 0 else 1


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["fq", "reference"], default="fq")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-call table, other configs and e2e")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--profile-case", default=None,
                    help="run one op of the workload untimed (a profiler target) and exit; prints no bench line")
    args = ap.parse_args()
    if args.profile_case:
        return run_profile_case(args.profile_case)
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)))
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group(backend="nccl")
    out = run_fq(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))
    return 0


if __name__ == "__main__":
    sys.exit(main())
