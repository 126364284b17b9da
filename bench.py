"""Benchmark of the quantized small-batch matvec on GB300.

Metric: effective weight bandwidth (algorithmic weight bytes / time, GB/s)
and microseconds per call, for the small-batch Q4_K matvec M = 17408,
K = 5120 at 1, 2, 4, 8 and 16 tokens; one step = one call at each of those
token counts.  Effective bandwidth = weight bytes / kernel time is the pages'
own measure ("Running GLM-5.3 on Two 8-GPU AMD W7900D Machines", paragraph
under the constraint table of "A faster kernel can still leave the full
chain slower").

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Inputs are synthetic and seeded (N(0, 0.02) weights quantized on the GPU by
the library's quantizer, N(0, 1) activations).  Weights rotate over 12
replicas (600 MB, > 4x the 129 MB L2), one replica per step, so every call
streams from HBM.
Each call is the library's matvec with a caller workspace (qmv_splitk_run,
which picks one split for this shape and, above 4 tokens, quantizes the
activations once into the workspace).  Timed region: exactly --steps steps,
each the replay of a captured one-step graph, CUDA events on the launching
stream.  `e2e` repeats the steps through the public API with the
activations copied in from pinned host memory and the outputs copied back,
every step (two device buffer sets, each copy direction on its own stream, so
that a step's copies overlap its neighbours' matvecs).  `--impl reference` times the CPU oracle on a bounded sample of
the same workload on the host cores.  Under torchrun (N > 1) every rank runs
the same single-GPU workload (replicas: nothing in the path is sharded), the
time is the maximum over ranks and the value sums the ranks' bytes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "µs/call and effective weight GB/s (fraction of GB300 HBM peak), 1–64 tokens"
WORKLOAD = "q4_k_matvec_17408x5120"
FMT, M, K = 1, 17408, 5120
NTOKS = (1, 2, 4, 8, 16)
REPLICAS = 12
BYTES_PER_CALL = M * (K // 256) * 144
KERNEL_SOURCES = ("moe_matvec_gb300/csrc/qmv_dense.cuh", "moe_matvec_gb300/csrc/qmv_core.cuh",
                  "moe_matvec_gb300/csrc/common.cuh", "moe_matvec_gb300/csrc/qmv_dense_inst.cuh",
                  "moe_matvec_gb300/csrc/qmv_api.cu", "moe_matvec_gb300/csrc/qmv_mma.cuh",
                  "moe_matvec_gb300/csrc/qmv_mma_q4_k.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "qmv_dense_q4_k_traffic.json")


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def recorded_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except OSError:
        return None
    if rec.get("kernel_hash") != kernel_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.tmp.name)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                for nm, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# distributed plumbing (replicas only)
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(times_ms, bytes_per_rank):
    """Whole-job throughput: all ranks' bytes over the slowest rank's time."""
    t = max(times_ms)
    return sum(bytes_per_rank) / (t * 1e-3) / 1e9, t


def gather_floats(value: float, world: int):
    if world == 1:
        return [value]
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    out = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(out, t)
    return [float(o.item()) for o in out]


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------
# CPU baseline (the oracle, as it stands)
# --------------------------------------------------------------------------

def oracle_sample(rows: int, seed: int = 4242):
    import oracle
    from moe_matvec_gb300 import synth
    w = synth.weights(seed, rows, K)
    Wn = oracle.quantize(FMT, w)
    xs = {n: synth.activations(seed + n, n, K) for n in NTOKS}
    return Wn, xs


def time_oracle(Wn, xs, threads: int):
    import oracle
    t0 = time.perf_counter()
    for n in NTOKS:
        oracle.qmv(FMT, Wn, xs[n], K, nthreads=threads)
    return time.perf_counter() - t0


def cpu_baseline(budget_s: float = 12.0):
    """The oracle on the host cores: whole passes over a row sample of the
    workload (all rows when a pass is short), repeated until about budget_s
    seconds of CPU work."""
    threads = os.cpu_count() or 1
    Wn, xs = oracle_sample(64)
    t = time_oracle(Wn, xs, threads)
    rows = int(min(M, max(64, 64 * budget_s / max(t, 1e-6))))
    Wn, xs = oracle_sample(rows)
    passes, t = 0, 0.0
    while t < budget_s or passes == 0:
        t += time_oracle(Wn, xs, threads)
        passes += 1
    sample_bytes = rows * (K // 256) * 144 * len(NTOKS) * passes
    return {"value": sample_bytes / t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} of {M} rows, n_tok in {list(NTOKS)}, {passes} pass(es) ({t:.1f} s)"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    threads = os.cpu_count() or 1
    # per-step sample sized so that warmup + steps finish in about two minutes
    Wn, xs = oracle_sample(16)
    t16 = time_oracle(Wn, xs, threads)
    per_step = 100.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(M, 16 * per_step / max(t16, 1e-6))))
    Wn, xs = oracle_sample(rows)
    for _ in range(args.warmup):
        time_oracle(Wn, xs, threads)
    t = 0.0
    for _ in range(args.steps):
        t += time_oracle(Wn, xs, threads)
    step_bytes = rows * (K // 256) * 144 * len(NTOKS)
    value = step_bytes * args.steps / t / 1e9
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8xint8->int32, f32",
            "data": "synthetic", "config": {"workload": WORKLOAD, "n_tok": list(NTOKS), "format": "Q4_K"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{rows} of {M} rows per step, n_tok in {list(NTOKS)}"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from moe_matvec_gb300 import api, synth
    api.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)

    # weights: N(0, 0.02) drawn on the GPU, quantized by the library, replicated
    g = torch.Generator(device=dev)
    g.manual_seed(1001 + rank)
    w = torch.randn((M, K), generator=g, device=dev, dtype=torch.float32) * 0.02
    W0 = api.quantize_weights(FMT, w)
    del w
    Ws = [W0] + [W0.clone() for _ in range(REPLICAS - 1)]
    # the step's inputs and outputs as views of two contiguous buffers, so the
    # end-to-end run moves each step's inputs and results with one copy each
    x_all = torch.cat([torch.from_numpy(synth.activations(1010 + n, n, K)) for n in NTOKS]).to(dev)
    y_all = torch.empty((sum(NTOKS), M), device=dev)
    offs = [int(v) for v in np.cumsum([0] + list(NTOKS))]
    xs = {n: x_all[offs[i]:offs[i + 1]] for i, n in enumerate(NTOKS)}
    ys = {n: y_all[offs[i]:offs[i + 1]] for i, n in enumerate(NTOKS)}
    # the library's matvec with a caller workspace (qmv_splitk_run; one split
    # for this shape): above 4 tokens it quantizes the activations once
    splits = {n: api.splitk_choose(FMT, M, K, n) for n in NTOKS}
    wss = {n: torch.empty(max(16, api.splitk_workspace_fast_bytes(M, K, n, splits[n])), dtype=torch.uint8,
                          device=dev) for n in NTOKS}
    torch.cuda.synchronize()

    def matvec(W, n, s):
        api.splitk_run(FMT, W, xs[n], M, K, n_split=splits[n], ws=wss[n], out=ys[n], stream=s)

    def step(r, s):
        for n in NTOKS:
            matvec(Ws[r % REPLICAS], n, s)

    # one graph per replica, each one whole step on that replica; step i of
    # the run replays graph i mod REPLICAS, so exactly --steps steps are timed
    # after exactly --warmup untimed ones, every step streaming from HBM
    with torch.cuda.stream(stream):
        for r in range(REPLICAS):          # eager warm-up (also builds everything)
            step(r, stream)
    stream.synchronize()
    graphs = []
    for r in range(REPLICAS):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step(r, stream)
        graphs.append(gr)
    steps = args.steps
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % REPLICAS].replay()
    stream.synchronize()

    # measured issue rates of the pipes (denominators of the ALU roofline)
    pipe_rates = api.measure_pipes(stream)

    # per-token-count graphs for the per-call breakdown
    per_n = {}
    for n in NTOKS:
        gn = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gn, stream=stream):
            for r in range(REPLICAS):
                matvec(Ws[r], n, stream)
        with torch.cuda.stream(stream):
            gn.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        nrep = 50
        stream.synchronize()
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(nrep):
                gn.replay()
        e1.record(stream)
        e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (nrep * REPLICAS)
        per_n[str(n)] = {"us_per_call": round(us, 3), "gbs": round(BYTES_PER_CALL / (us * 1e-6) / 1e9, 1)}
        # the same calls as back-to-back eager launches through the binding
        # (host launch cost included): the per-call cost a graph amortizes
        neager = 10
        stream.synchronize()
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(neager):
                for r in range(REPLICAS):
                    matvec(Ws[r], n, stream)
        e1.record(stream)
        e1.synchronize()
        per_n[str(n)]["us_per_call_eager"] = round(e0.elapsed_time(e1) * 1e3 / (neager * REPLICAS), 3)

    # timed region
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.25)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for i in range(steps):
                graphs[(args.warmup + i) % REPLICAS].replay()
        e1.record(stream)
        e1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    step_bytes = BYTES_PER_CALL * len(NTOKS)
    value, tmax = aggregate(gather_floats(ms, world), [step_bytes * steps] * world)
    # one matvec kernel per call, plus the activation quantizer where the call
    # quantizes once: above 4 tokens on this shape (one split, 17408 rows); the
    # ncu launch list of the step shows the same kernels
    launches = steps * sum(2 if n > 4 else 1 for n in NTOKS)

    extra = None
    if not args.no_extra:
        extra = run_extra(torch, api, synth, stream, dev, measured_peaks()[0]["hbm_gbs"])

    # e2e: public API with host buffers, eager launches; every step copies its
    # inputs in from pinned host memory (one copy) and reads its results back
    # (one copy).  Two device buffer sets and one stream per copy direction
    # let step i's copies overlap the matvecs of its neighbours, as a serving
    # loop would run them.
    xh = x_all.cpu().pin_memory()
    yh = [torch.empty((sum(NTOKS), M)).pin_memory() for _ in range(2)]
    xb = [x_all, torch.empty_like(x_all)]
    yb = [y_all, torch.empty_like(y_all)]
    views = [({n: xb[b][offs[i]:offs[i + 1]] for i, n in enumerate(NTOKS)},
              {n: yb[b][offs[i]:offs[i + 1]] for i, n in enumerate(NTOKS)}) for b in range(2)]
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "out", "back")}
    e2e_steps = max(REPLICAS, min(steps, 2000))
    barrier(world)
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    h2d.wait_event(a0)
    d2h.wait_event(a0)
    for i in range(e2e_steps):
        b = i % 2
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(ev["out"][b])        # step i - 2 has read xb[b]
            xb[b].copy_(xh, non_blocking=True)
            ev["in"][b].record(h2d)
        stream.wait_event(ev["in"][b])
        if i >= 2:
            stream.wait_event(ev["back"][b])        # step i - 2's results are out of yb[b]
        xv, yv = views[b]
        for n in NTOKS:
            api.splitk_run(FMT, Ws[i % REPLICAS], xv[n], M, K, n_split=splits[n], ws=wss[n], out=yv[n],
                           stream=stream)
        ev["out"][b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev["out"][b])
            yh[b].copy_(yb[b], non_blocking=True)
            ev["back"][b].record(d2h)
    stream.wait_event(ev["back"][(e2e_steps - 1) % 2])
    stream.wait_event(ev["back"][(e2e_steps - 2) % 2])
    a1.record(stream)
    a1.synchronize()
    barrier(world)
    e2e_ms = a0.elapsed_time(a1)
    e2e_value, _ = aggregate(gather_floats(e2e_ms, world), [step_bytes * e2e_steps] * world)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peaks, peak_kind = measured_peaks()
    achieved = step_bytes * steps / (ms * 1e-3) / 1e9
    # The 8- and 16-token calls are not bound by HBM.  They run on the tensor
    # cores (mma.sync, f16 operands holding the integer codes): their useful
    # multiply-adds (M K n) against the measured mma.sync rate per SM per clock
    # x SMs x the SM clock sampled during the timed region.  For comparison,
    # the floor of a dp4a kernel (one dp4a per 4 weights per token at the
    # measured dp4a rate) and the call time relative to it.
    clk_summary = clk.summary()
    sm_mhz = clk_summary.get("sm_mhz") or peaks.get("sm_max_mhz", 2070.0)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    mma_peak = 2.0 * pipe_rates["mma_sync_f16_mac"] * nsm * sm_mhz * 1e6   # FLOP/s
    dp4a_peak = pipe_rates["dp4a"] * nsm * sm_mhz * 1e6                     # dp4a/s
    roof_alu = {"bound": "tensor", "pipe": "mma.sync m16n8k16 f16 -> f32", "unit": "TFLOP/s",
                "peak": round(mma_peak / 1e12, 2),
                "peak_kind": "measured (qmv_measure_pipes mma.sync f16 MAC per SM per clock x SMs x sampled SM "
                             "clock)",
                "kernel": "qmv_mma_q4k_kernel<8 / 16 token slots>", "per_n": {}}
    for n in (8, 16):
        us = per_n[str(n)]["us_per_call"]
        a = 2.0 * M * K * n / (us * 1e-6)
        floor_us = M * K * n / 4 / dp4a_peak * 1e6
        roof_alu["per_n"][str(n)] = {"achieved": round(a / 1e12, 3), "frac": round(a / mma_peak, 4),
                                     "dp4a_floor_us": round(floor_us, 2),
                                     "dp4a_floor_over_call": round(floor_us / us, 3)}
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": recorded_traffic(),
            "peak_kind": peak_kind,
            "kernel": "qmv_dense_kernel<Q4_K> (1, 2, 4 tokens), qmv_mma_q4k_kernel (8, 16 tokens)",
            "algorithmic_bytes_per_launch": BYTES_PER_CALL}
    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": tmax / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8xint8->int32, f32",
            "data": "synthetic N(0,0.02) weights quantized on GPU, N(0,1) activations",
            "config": {"workload": WORKLOAD, "format": "Q4_K", "M": M, "K": K, "n_tok": list(NTOKS),
                       "l2": f"weights rotate over {REPLICAS} replicas ({REPLICAS * BYTES_PER_CALL / 1e6:.0f} MB "
                             "> 4x L2), inputs larger than L2", "timing": "CUDA graph replay, CUDA events",
                       "parallelism": f"replicas x{world}"},
            "us_per_call": per_n, "roofline": roof,
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": sum(n * K * 4 for n in NTOKS),
                    "d2h_bytes_per_step": sum(n * M * 4 for n in NTOKS),
                    "ms_per_step": e2e_ms / e2e_steps},
            "gpu_launches": launches, "clocks": clk_summary, "roofline_alu": roof_alu,
            "pipe_rates_per_sm_clk": {k: round(v, 2) for k, v in pipe_rates.items()}}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if extra is not None:
        line["workloads"] = extra          # last: the long block of the other configurations
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------------------------
# the other workloads (parity-test configurations), timed the same way
# --------------------------------------------------------------------------

def _graph_us(torch, stream, calls, reps=20):
    """µs per call of `calls` (callables launching on `stream`) replayed as one
    CUDA graph `reps` times, after an eager pass and a warm replay."""
    with torch.cuda.stream(stream):
        for c in calls:
            c()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in calls:
            c()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * len(calls))


def _replicas(torch, api, fmt, M, K, nbytes_min, dev, seed):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    w = torch.randn((M, K), generator=g, device=dev, dtype=torch.float32) * 0.02
    W0 = api.quantize_weights(fmt, w)
    del w
    rb = M * api.row_bytes(fmt, K)
    n = max(1, -(-nbytes_min // rb))
    return [W0] + [W0.clone() for _ in range(n - 1)], rb


def run_extra(torch, api, synth, stream, dev, peak):
    """µs/call and effective weight GB/s of every other configuration: the
    Q8_0 GEMV, the IQ4_XS, Q5_K, Q6_K, Q8_G128, F16 and F32 matvecs, split-K
    (LM head and long K), the MoE
    decode layer, the router + top-k step in front of it, sibling matvecs
    sharing x and the matvec with a residual add.  Weight sets
    rotate over replicas totalling > 2 x L2 (the LM head alone is > 6 x L2);
    MoE calls rotate over 16 routing draws."""
    out = {}
    l2x2 = 2 * 135 * 2 ** 20

    def line(bytes_per_call, us):
        gbs = bytes_per_call / (us * 1e-6) / 1e9
        return {"us_per_call": round(us, 3), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}

    dense = [("q8_0_gemv_4096x4096", 0, 4096, 4096, (1,)),
             ("iq4_xs_6144x2048", 2, 6144, 2048, (1, 4, 8)),
             ("iq4_xs_2048x6144", 2, 2048, 6144, (1, 4, 8)),
             ("q5_k_17408x5120", 3, 17408, 5120, (1, 4, 16)),
             ("q6_k_17408x5120", 4, 17408, 5120, (1, 4, 16)),
             ("q8_g128_lm_head_151936x5120", 6, 151936, 5120, (1, 4, 16)),
             ("f16_17408x5120", 7, 17408, 5120, (1, 4, 16)),
             ("f32_4096x4096", 8, 4096, 4096, (1, 4, 16))]
    for i, (name, fmt, M, K, ns) in enumerate(dense):
        Ws, rb = _replicas(torch, api, fmt, M, K, l2x2, dev, 2000 + i)
        res = {}
        for n in ns:
            x = torch.from_numpy(synth.activations(3000 + n, n, K)).to(dev)
            y = torch.empty((n, M), device=dev)
            S = api.splitk_choose(fmt, M, K, n)
            ws = torch.empty(max(16, api.splitk_workspace_fast_bytes(M, K, n, S)), dtype=torch.uint8, device=dev)
            calls = [(lambda W=W: api.splitk_run(fmt, W, x, M, K, n_split=S, ws=ws, out=y, stream=stream))
                     for W in Ws]
            r = line(rb, _graph_us(torch, stream, calls))
            r["n_split"] = S
            res[str(n)] = r
        out[name] = {"format": ["Q8_0", "Q4_K", "IQ4_XS", "Q5_K", "Q6_K", "Q8_G64", "Q8_G128", "F16", "F32"][fmt],
                     "bytes_per_call": rb, "replicas": len(Ws),
                     "n_tok": res}
        del Ws

    splitk = [("splitk_q8_0_151936x5120", 151936, 5120, 2), ("splitk_q8_0_512x65536", 512, 65536, None)]
    for i, (name, M, K, reps_min) in enumerate(splitk):
        Ws, rb = _replicas(torch, api, 0, M, K, l2x2, dev, 2100 + i)
        res = {}
        for n in (1, 2, 4, 8, 16):
            x = torch.from_numpy(synth.activations(3100 + n, n, K)).to(dev)
            y = torch.empty((n, M), device=dev)
            S = api.splitk_choose(0, M, K, n)
            ws = torch.empty(max(16, api.splitk_workspace_fast_bytes(M, K, n, S)), dtype=torch.uint8, device=dev)
            calls = [(lambda W=W: api.splitk_run(0, W, x, M, K, n_split=S, ws=ws, out=y, stream=stream))
                     for W in Ws]
            r = line(rb, _graph_us(torch, stream, calls, reps=10 if rb > 2 ** 28 else 20))
            r["n_split"] = S
            res[str(n)] = r
        out[name] = {"format": "Q8_0", "bytes_per_call": rb, "replicas": len(Ws), "n_tok": res}
        del Ws

    c = synth.MOE_CASE
    g = torch.Generator(device=dev)
    g.manual_seed(2200)
    H, F, E = c.hidden, c.ffn, c.n_experts
    wg = torch.empty((E, 2 * F, api.row_bytes(c.fmt_gate_up, H)), dtype=torch.uint8, device=dev)
    wd = torch.empty((E, H, api.row_bytes(c.fmt_down, F)), dtype=torch.uint8, device=dev)
    for e in range(E):
        wg[e] = api.quantize_weights(c.fmt_gate_up, torch.randn((2 * F, H), generator=g, device=dev) * 0.02)
        wd[e] = api.quantize_weights(c.fmt_down, torch.randn((H, F), generator=g, device=dev) * 0.02)
    ex = api.moe_experts(E, H, F, c.fmt_gate_up, c.fmt_down, wg, wd)
    per_expert = wg[0].numel() + wd[0].numel()
    res = {}
    for n in c.n_toks:
        sets = [synth.routing(2300 + 17 * n + k, n, E, c.top_k) for k in range(16)]
        ids = [torch.from_numpy(a).to(dev) for a, _ in sets]
        gates = [torch.from_numpy(b).to(dev) for _, b in sets]
        x = torch.from_numpy(synth.activations(2400 + n, n, H)).to(dev)
        y = torch.empty((n, H), device=dev)
        ws = torch.empty(api.moe_workspace_bytes(ex, n, c.top_k), dtype=torch.uint8, device=dev)
        calls = [(lambda k=k: api.moe_run(ex, ids[k], gates[k], x, ws=ws, out=y, stream=stream))
                 for k in range(len(sets))]
        us = _graph_us(torch, stream, calls)
        distinct = sum(len(np.unique(a)) for a, _ in sets) / len(sets)
        r = line(distinct * per_expert, us)
        r["distinct_experts"] = round(distinct, 2)
        res[str(n)] = r
    out["moe_128x_top8_h4096_f1536"] = {"format": "gate/up IQ4_XS, down Q4_K", "bytes_per_expert": per_expert,
                                        "routing_draws": 16, "n_tok": res}

    # the same layer for prompt-sized batches on the tensor cores
    # (moe_qmv_prefill_run): tokens / s, effective weight GB/s of the touched
    # experts and tensor-core TFLOP/s (2 x multiply-adds of the contraction)
    res = {}
    macs_per_slot = 2 * F * H + H * F
    for n in (512, 2048):
        sets = [synth.routing(2350 + 17 * n + k, n, E, c.top_k) for k in range(2)]
        ids = [torch.from_numpy(a).to(dev) for a, _ in sets]
        gates = [torch.from_numpy(b).to(dev) for _, b in sets]
        x = torch.from_numpy(synth.activations(2450 + n, n, H)).to(dev)
        y = torch.empty((n, H), device=dev)
        ws = torch.empty(api.moe_prefill_workspace_bytes(ex, n, c.top_k), dtype=torch.uint8, device=dev)
        calls = [(lambda k=k: api.moe_prefill_run(ex, ids[k], gates[k], x, ws=ws, out=y, stream=stream))
                 for k in range(len(sets))]
        us = _graph_us(torch, stream, calls, reps=5)
        distinct = sum(len(np.unique(a)) for a, _ in sets) / len(sets)
        r = line(distinct * per_expert, us)
        r["tokens_per_s"] = round(n / (us * 1e-6), 1)
        r["tensor_tflops"] = round(2.0 * n * c.top_k * macs_per_slot / (us * 1e-6) / 1e12, 2)
        res[str(n)] = r
    out["moe_prefill_128x_top8_h4096_f1536"] = {"format": "gate/up IQ4_XS, down Q4_K", "kernel": "tcgen05 f16",
                                                "bytes_per_expert": per_expert, "n_tok": res}
    del wg, wd

    # router + top-k producing those ids / gates: a Q8_0 router of 128
    # experts over hidden 4096, softmax gating, top-8; router replicas > 2 x L2
    Ws, rb = _replicas(torch, api, 0, E, H, l2x2, dev, 2500)
    res = {}
    for n in c.n_toks:
        x = torch.from_numpy(synth.activations(2600 + n, n, H)).to(dev)
        lg = torch.empty((n, E), dtype=torch.float32, device=dev)
        ri = torch.empty((n, c.top_k), dtype=torch.int32, device=dev)
        rg = torch.empty((n, c.top_k), dtype=torch.float32, device=dev)
        calls = [(lambda W=W: api.route_run(0, W, x, E, H, c.top_k, api.GATING_SOFTMAX, logits=lg, ids=ri, gates=rg,
                                            stream=stream)) for W in Ws]
        res[str(n)] = line(rb, _graph_us(torch, stream, calls))
    out["router_q8_0_128x4096_top8"] = {"format": "Q8_0", "gating": "softmax", "bytes_per_call": rb,
                                        "replicas": len(Ws), "n_tok": res}
    del Ws

    # sibling matvecs sharing x (q / k / v shapes, Q4_K, hidden 5120), against
    # the same three matrices as separate calls
    Hs = 5120
    shapes = [(5120, 2700), (1024, 2701), (1024, 2702)]
    tot_rows = sum(Ms for Ms, _ in shapes)
    sets = [_replicas(torch, api, 1, Ms, Hs, l2x2 * Ms // tot_rows, dev, sd) for Ms, sd in shapes]
    reps = min(len(w) for w, _ in sets)
    rb = sum(b for _, b in sets)
    res = {}
    for n in (1, 4, 16):
        x = torch.from_numpy(synth.activations(2710 + n, n, Hs)).to(dev)
        ys = [torch.empty((n, Ms), device=dev) for Ms, _ in shapes]
        ws = torch.empty(max(16, api.act_q8_bytes(Hs, n)), dtype=torch.uint8, device=dev)
        fused = [(lambda i=i: api.run_siblings([(1, sets[j][0][i], shapes[j][0]) for j in range(3)], x, Hs,
                                               outs=ys, ws=ws, stream=stream)) for i in range(reps)]
        wss = [torch.empty(max(16, api.splitk_workspace_fast_bytes(Ms, Hs, n, 1)), dtype=torch.uint8, device=dev)
               for Ms, _ in shapes]
        sep = [(lambda i=i: [api.splitk_run(1, sets[j][0][i], x, shapes[j][0], Hs, n_split=1, ws=wss[j], out=ys[j],
                                            stream=stream) for j in range(3)]) for i in range(reps)]
        r = line(rb, _graph_us(torch, stream, fused))
        r["separate_us_per_call"] = round(_graph_us(torch, stream, sep), 3)
        res[str(n)] = r
    out["siblings_q4_k_qkv_5120"] = {"format": "Q4_K", "rows": [m for m, _ in shapes], "K": Hs,
                                     "bytes_per_call": rb, "replicas": reps, "n_tok": res}
    del sets

    # matvec + residual add in place (y += W x) on the Q4_K 17408 x 5120 matrix
    Ws, rb = _replicas(torch, api, 1, 17408, 5120, l2x2, dev, 2800)
    res = {}
    for n in (1, 16):
        x = torch.from_numpy(synth.activations(2810 + n, n, 5120)).to(dev)
        y = torch.zeros((n, 17408), device=dev)
        ws = torch.empty(max(16, api.splitk_workspace_fast_bytes(17408, 5120, n, 1)), dtype=torch.uint8, device=dev)
        calls = [(lambda W=W: api.run_residual(1, W, x, y, 17408, 5120, out=y, n_split=1, ws=ws, stream=stream))
                 for W in Ws]
        res[str(n)] = line(rb, _graph_us(torch, stream, calls))
    out["residual_q4_k_17408x5120"] = {"format": "Q4_K", "bytes_per_call": rb, "replicas": len(Ws), "n_tok": res}
    del Ws
    return out


def run_profile_moe(args):
    """Two eager MoE decode calls at --profile-moe tokens (for ncu captures)."""
    import torch
    from moe_matvec_gb300 import api, synth
    api.load()
    n = args.profile_moe
    c = synth.MOE_CASE
    g = torch.Generator(device="cuda")
    g.manual_seed(2200)
    H, F, E = c.hidden, c.ffn, c.n_experts
    wg = torch.empty((E, 2 * F, api.row_bytes(c.fmt_gate_up, H)), dtype=torch.uint8, device="cuda")
    wd = torch.empty((E, H, api.row_bytes(c.fmt_down, F)), dtype=torch.uint8, device="cuda")
    for e in range(E):
        wg[e] = api.quantize_weights(c.fmt_gate_up, torch.randn((2 * F, H), generator=g, device="cuda") * 0.02)
        wd[e] = api.quantize_weights(c.fmt_down, torch.randn((H, F), generator=g, device="cuda") * 0.02)
    ex = api.moe_experts(E, H, F, c.fmt_gate_up, c.fmt_down, wg, wd)
    x = torch.from_numpy(synth.activations(2400 + n, n, H)).cuda()
    y = torch.empty((n, H), device="cuda")
    ws = torch.empty(api.moe_workspace_bytes(ex, n, c.top_k), dtype=torch.uint8, device="cuda")
    for k in range(2):
        a, b = synth.routing(2300 + 17 * n + k, n, E, c.top_k)
        if args.skew:
            # every token picks the same top_k experts (each in its own order):
            # n slots per expert, so the expert groups split into n / slots groups
            a = np.stack([np.random.default_rng(2500 + 31 * k + t).permutation(c.top_k) for t in range(n)])
            a = a.astype(np.int32)
        api.moe_run(ex, torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), x, ws=ws, out=y)
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": "moe_128x_top8_h4096_f1536", "n_tok": n, "calls": 2,
                      "routing": "all tokens on experts 0-7" if args.skew else "random"}))
    return 0


def run_profile_float(args):
    """Two eager F16 17408 x 5120 calls at --profile-float tokens, in the bench's
    launch configuration (split chosen from the shape, workspace given), for
    ncu captures."""
    import torch
    from moe_matvec_gb300 import api, synth
    api.load()
    fmt, Mf, Kf, n = 7, 17408, 5120, args.profile_float
    g = torch.Generator(device="cuda")
    g.manual_seed(2007)
    W = api.quantize_weights(fmt, torch.randn((Mf, Kf), generator=g, device="cuda") * 0.02)
    x = torch.from_numpy(synth.activations(3000 + n, n, Kf)).cuda()
    S = api.splitk_choose(fmt, Mf, Kf, n)
    ws = torch.empty(max(16, api.splitk_workspace_fast_bytes(Mf, Kf, n, S)), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        api.splitk_run(fmt, W, x, Mf, Kf, n_split=S, ws=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": "f16_17408x5120", "n_tok": n, "n_split": S, "calls": 2}))
    return 0


def run_profile_prefill(args):
    """Two eager calls of the tensor-core MoE layer at --profile-prefill tokens
    (full-size pool), for ncu captures."""
    import torch
    from moe_matvec_gb300 import api, synth
    api.load()
    n = args.profile_prefill
    c = synth.MOE_CASE
    g = torch.Generator(device="cuda")
    g.manual_seed(2200)
    H, F, E = c.hidden, c.ffn, c.n_experts
    wg = torch.empty((E, 2 * F, api.row_bytes(c.fmt_gate_up, H)), dtype=torch.uint8, device="cuda")
    wd = torch.empty((E, H, api.row_bytes(c.fmt_down, F)), dtype=torch.uint8, device="cuda")
    for e in range(E):
        wg[e] = api.quantize_weights(c.fmt_gate_up, torch.randn((2 * F, H), generator=g, device="cuda") * 0.02)
        wd[e] = api.quantize_weights(c.fmt_down, torch.randn((H, F), generator=g, device="cuda") * 0.02)
    ex = api.moe_experts(E, H, F, c.fmt_gate_up, c.fmt_down, wg, wd)
    x = torch.from_numpy(synth.activations(2450 + n, n, H)).cuda()
    ws = torch.empty(api.moe_prefill_workspace_bytes(ex, n, c.top_k), dtype=torch.uint8, device="cuda")
    for k in range(2):
        a, b = synth.routing(2350 + 17 * n + k, n, E, c.top_k)
        api.moe_prefill_run(ex, torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), x, ws=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": "moe_prefill_128x_top8_h4096_f1536", "n_tok": n, "calls": 2}))
    return 0


def run_profile_dense(args):
    """Eager calls of one dense configuration fmt:M:K:n_tok in the bench's
    launch configuration (split from the shape, workspace with room for the
    once-quantized activations), rotating over replicas larger than L2 in all,
    for ncu captures: --profile-dense 2:6144:2048:1."""
    import torch
    from moe_matvec_gb300 import api, synth
    api.load()
    fmt, Md, Kd, n = (int(v) for v in args.profile_dense.split(":"))
    g = torch.Generator(device="cuda")
    g.manual_seed(2000 + fmt)
    W0 = api.quantize_weights(fmt, torch.randn((Md, Kd), generator=g, device="cuda") * 0.02)
    rb = Md * api.row_bytes(fmt, Kd)
    Ws = [W0] + [W0.clone() for _ in range(max(1, -(-2 * 135 * 2 ** 20 // rb)) - 1)]
    x = torch.from_numpy(synth.activations(3000 + n, n, Kd)).cuda()
    y = torch.empty((n, Md), device="cuda")
    S = api.splitk_choose(fmt, Md, Kd, n)
    ws = torch.empty(max(16, api.splitk_workspace_fast_bytes(Md, Kd, n, S)), dtype=torch.uint8, device="cuda")
    calls = max(4, len(Ws))
    for i in range(calls):
        api.splitk_run(fmt, Ws[i % len(Ws)], x, Md, Kd, n_split=S, ws=ws, out=y)
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": f"fmt{fmt}_{Md}x{Kd}", "n_tok": n, "n_split": S, "calls": calls,
                      "replicas": len(Ws)}))
    return 0


def run_profile(args):
    """A few eager calls of the timed workload (for ncu captures)."""
    import torch
    from moe_matvec_gb300 import api, synth
    api.load()
    g = torch.Generator(device="cuda")
    g.manual_seed(1001)
    w = torch.randn((M, K), generator=g, device="cuda", dtype=torch.float32) * 0.02
    Ws = [api.quantize_weights(FMT, w) for _ in range(3)]
    del w
    for rnd in range(2):
        for n in NTOKS:
            x = torch.from_numpy(synth.activations(1010 + n, n, K)).cuda()
            S = api.splitk_choose(FMT, M, K, n)
            ws = torch.empty(max(16, api.splitk_workspace_fast_bytes(M, K, n, S)), dtype=torch.uint8, device="cuda")
            api.splitk_run(FMT, Ws[(rnd * len(NTOKS) + n) % 3], x, M, K, n_split=S, ws=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": WORKLOAD, "calls": 2 * len(NTOKS)}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=12000)
    ap.add_argument("--warmup", type=int, default=24)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--profile", action="store_true", help="a few eager calls only (for ncu)")
    ap.add_argument("--profile-moe", type=int, default=0, help="two eager MoE calls at this many tokens (for ncu)")
    ap.add_argument("--skew", action="store_true", help="with --profile-moe: every token on the same top_k experts")
    ap.add_argument("--profile-float", type=int, default=0,
                    help="two eager F16 17408 x 5120 calls at this many tokens (for ncu)")
    ap.add_argument("--profile-prefill", type=int, default=0,
                    help="two eager tensor-core MoE calls at this many tokens (for ncu)")
    ap.add_argument("--profile-dense", default="",
                    help="eager calls of one dense configuration fmt:M:K:n_tok (for ncu)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_moe:
        return run_profile_moe(args)
    if args.profile_float:
        return run_profile_float(args)
    if args.profile_dense:
        return run_profile_dense(args)
    if args.profile_prefill:
        return run_profile_prefill(args)
    if args.profile:
        return run_profile(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
