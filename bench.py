#!/usr/bin/env python3
"""Benchmark of the GB300 q4_K x q8_0 decode matvec.

Default workload: the 7B-class whole decode step of matvecs -- 28 layers, per
layer q|k|v [4608 x 3584], o [3584 x 3584], ffn_gu [37888 x 3584] with fused
SiLU*mul and q8_0 of h, down [3584 x 18944]; batch 1; 3,670,474,752 bytes of
q4_K weights per step -- captured once as a CUDA graph and replayed.  One step
= one replay (every kernel of all 28 layers).  Weights are synthetic (seeded
generator), inputs are fp32 N(0,1) with 0.1% x20 outliers.

Prints ONE JSON line (rank 0): value = weight GB/s of the step (whole job,
all ranks), ms_per_step, the dominant kernel's roofline, the oracle's CPU
baseline, an end-to-end number through host buffers, clocks seen during the
timed region.  ``--impl reference`` times the CPU oracle instead (the
reference arm: there is no other implementation to run).

Multi-GPU: the step does not shard here (one GPU per box); N ranks run N
independent replicas (weak scaling), value = all ranks' bytes / max time.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "q4_K×q8_0 decode matvec weight GB/s vs HBM peak; 7B-class step µs (1 GPU)"
UNIT = "GB/s"
# per-config timings: timed graph replays (each of one or more calls) and untimed ones before them
CONFIG_REPS = 50
CONFIG_WARMUP = 10
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


# ---------------------------------------------------------------------------------------------------------
# multi-rank plumbing (torchrun): barrier, max of times, sum of work
# ---------------------------------------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_over_ranks(ms_local: float, units_local: float, device=None):
    """(max over ranks of ms, sum over ranks of units); identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms_local, units_local
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    u = torch.tensor([units_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="mq_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def mark(self):
        """Host time of the timed region's start (first call) and end (second call)."""
        self.window = getattr(self, "window", []) + [time.time()]

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = (self.window[0], self.window[-1]) if len(getattr(self, "window", [])) >= 2 else (None, None)
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if lo is not None:  # keep the samples taken inside the timed region
                    try:
                        import datetime
                        ts = datetime.datetime.strptime(parts[9], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        if ts < lo - 0.05 or ts > hi + 0.05:
                            continue
                    except ValueError:
                        pass
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------------------------------------

def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak():
    """Dense bf16 tensor TFLOP/s measured on this machine (burst); f16 runs at the same rate."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def kernel_source_sha(files=None) -> str:
    """Hash of the named kernel source files (default: every file of csrc/)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_decode_matvec_gb300", "csrc")
    for name in sorted(files if files else os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(profile_name: str):
    """DRAM bytes per launch from an ncu capture summarized in profiles/, if the source files the
    summary lists (its `source_files` line) still hash to its `kernel_source_sha`; else None."""
    path = os.path.join(ROOT, "profiles", profile_name)
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line and line.strip().startswith("- "):
                    k, v = line.strip()[2:].split(":", 1)
                    fields[k.strip()] = v.strip().strip("`")
        files = [x.strip() for x in fields.get("source_files", "").split(",") if x.strip()] or None
        if fields.get("kernel_source_sha") == kernel_source_sha(files):
            return float(fields["dram_bytes_per_launch"]), fields.get("traffic_note")
    except Exception:
        pass
    return None, None


def build_step(case, device, mq, host=None):
    """Upload the step's weights (q|k|v concatenated on the device with mq_concat_rows).
    With a list `host`, also keep each layer's host bytes there (for the oracle's baseline)."""
    import torch
    from quantized_decode_matvec_gb300 import synth
    stream = torch.cuda.current_stream().cuda_stream
    layers = []
    for l in range(case.n_layers):
        w = synth.step_layer_weights(case, l)
        if host is not None:
            host.append({"q": w["q"], "k": w["k"], "v": w["v"], "o": w["o"], "gu": w["gu"], "down": w["down"]})
        q, k, v = (torch.from_numpy(w[n]).to(device) for n in ("q", "k", "v"))
        qkv = torch.empty((case.qkv_rows, q.shape[1]), dtype=torch.uint8, device=device)
        st = mq.mq_concat_rows(qkv.data_ptr(), [q.data_ptr(), k.data_ptr(), v.data_ptr()],
                               [case.q_rows, case.kv_rows, case.kv_rows], mq.MQ_TYPE_Q4_K, case.H, stream)
        mq._check(st, "mq_concat_rows")
        layers.append({"qkv": qkv, "o": torch.from_numpy(w["o"]).to(device),
                       "gu": torch.from_numpy(w["gu"]).to(device), "down": torch.from_numpy(w["down"]).to(device)})
        del q, k, v
    torch.cuda.synchronize()
    return layers


def fill_inputs(bufs, case, replay):
    import torch
    from quantized_decode_matvec_gb300 import synth
    for l in range(case.n_layers):
        inp = synth.step_layer_inputs(case, l, replay)
        bufs.a[l].copy_(torch.from_numpy(inp["a"]))
        bufs.b[l].copy_(torch.from_numpy(inp["b"]))
        bufs.c[l].copy_(torch.from_numpy(inp["c"]))


def time_replays(run, stream, steps):
    """Per-step device times (ms) of `steps` runs, CUDA events on the launching stream."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record(stream)
    for i in range(steps):
        run()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    return [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]


def sem(v):
    return statistics.stdev(v) / len(v) ** 0.5 if len(v) > 1 else 0.0


# ---------------------------------------------------------------------------------------------------------
# CPU oracle baseline (test infrastructure, timed as it stands)
# ---------------------------------------------------------------------------------------------------------

def host_cores() -> int:
    """Host threads this process may run on (its CPU affinity)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleArm:
    """The CPU oracle as it stands, on `threads` host threads.

    One thread calls the oracle's own functions (``oracle.ffn`` is its whole
    FFN chain in C).  More threads split every matvec into a static partition
    of its rows, one contiguous slice per thread (ctypes releases the GIL for
    the duration of each C call), and keep the FFN chain's stage order: all of
    g|u, then SiLU*mul and the q8_0 of h, then down.  Each output row is the
    oracle's own per-row computation, so both give the same bytes.
    """

    def __init__(self, threads: int = 1):
        self.threads = max(1, int(threads))
        self.pool = None
        if self.threads > 1:
            from concurrent.futures import ThreadPoolExecutor
            self.pool = ThreadPoolExecutor(self.threads)

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()
            self.pool = None

    def _rows(self, fn, rows):
        bounds = np.linspace(0, rows, self.threads + 1).astype(np.int64)
        parts = [np.arange(bounds[i], bounds[i + 1], dtype=np.int64) for i in range(self.threads)
                 if bounds[i + 1] > bounds[i]]
        return np.concatenate(list(self.pool.map(fn, parts)), axis=1)

    def matvec(self, W, xq, rows, K):
        import oracle
        if self.pool is None:
            return oracle.matvec(W, xq, rows, K)[0]
        return self._rows(lambda ids: oracle.matvec(W, xq, rows, K, row_ids=ids)[0], rows)

    def matvec_w(self, wtype, W, xq, rows, K):
        import oracle
        if self.pool is None:
            return oracle.matvec_w(wtype, W, xq, rows, K)[0]
        return self._rows(lambda ids: oracle.matvec_w(wtype, W, xq, rows, K, row_ids=ids)[0], rows)

    def ffn(self, W_gu, W_down, x, H, I):
        import oracle
        if self.pool is None:
            return oracle.ffn(W_gu, W_down, x, H, I)[0]
        xq = oracle.quantize_q8_0(np.asarray(x, np.float32).reshape(-1, H))
        gu = self.matvec(W_gu, xq, 2 * I, H)
        h = oracle.silu_mul(gu[:, :I], gu[:, I:])
        hq = oracle.quantize_q8_0(h.astype(np.float32))
        return self.matvec(W_down, hq, H, I)

    def step_layer(self, case, w, inp):
        """One layer of the decode step: q|k|v, o, then the FFN, in order."""
        import oracle
        qkv = w["qkv"] if "qkv" in w else np.concatenate([w["q"], w["k"], w["v"]])
        self.matvec(qkv, oracle.quantize_q8_0(inp["a"]), case.qkv_rows, case.H)
        self.matvec(w["o"], oracle.quantize_q8_0(inp["b"]), case.H, case.q_rows)
        self.ffn(w["gu"], w["down"], inp["c"], case.H, case.I)

    def step(self, case, weights, inputs):
        """One whole step (every layer); returns seconds."""
        t0 = time.perf_counter()
        for l in range(case.n_layers):
            self.step_layer(case, weights[l], inputs[l])
        return time.perf_counter() - t0


def oracle_time(fn, reps=3):
    """Median seconds of `reps` calls of fn()."""
    t = []
    for _ in range(reps):
        t0 = time.perf_counter()
        fn()
        t.append(time.perf_counter() - t0)
    return statistics.median(t)


def host_step_weights(case):
    """Host copies of every layer's weights (q|k|v concatenated), as the GPU arm uploads them."""
    from quantized_decode_matvec_gb300 import synth
    out = []
    for l in range(case.n_layers):
        w = synth.step_layer_weights(case, l)
        out.append({"qkv": np.concatenate([w["q"], w["k"], w["v"]]), "o": w["o"], "gu": w["gu"],
                    "down": w["down"]})
    return out


def cpu_baseline(case, weights):
    """The oracle on the host cores over one whole step of the workload: one thread, and all the
    threads of this process's CPU affinity (static row partition).  The all-threads arm is the
    headline (value, cores); the one-thread arm rides along."""
    from quantized_decode_matvec_gb300 import synth
    inputs = [synth.step_layer_inputs(case, l, 0) for l in range(case.n_layers)]
    wbytes = synth.weight_bytes_step(case)
    n = host_cores()
    arm1 = OracleArm(1)
    s1 = arm1.step(case, weights, inputs)
    armn = OracleArm(n)
    sn = armn.step(case, weights, inputs)
    armn.close()
    return {"value": wbytes / sn / 1e9, "unit": UNIT, "cores": n, "kind": "oracle",
            "seconds": sn,
            "sample": f"one whole step ({case.n_layers} of {case.n_layers} layers: q|k|v, o, ffn_gu+SiLU*mul+q8_0, "
                      f"down), C oracle with fp64 accumulation, rows split statically over {n} threads "
                      f"(the process's CPU affinity), {sn:.2f} s",
            "single_thread": {"value": wbytes / s1 / 1e9, "unit": UNIT, "cores": 1, "seconds": s1,
                              "sample": "the same whole step on one thread"}}


def run_reference(args):
    """The reference arm: the CPU oracle as it stands on the host cores (all threads of the
    process's affinity, static row partition), each step one whole step of the workload."""
    from quantized_decode_matvec_gb300 import synth
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    case = synth.STEP_7B
    weights = host_step_weights(case)
    n = host_cores()
    arm = OracleArm(n)
    for i in range(args.warmup):
        arm.step(case, weights, [synth.step_layer_inputs(case, l, i) for l in range(case.n_layers)])
    times = []
    for i in range(args.steps):
        inputs = [synth.step_layer_inputs(case, l, args.warmup + i) for l in range(case.n_layers)]
        times.append(arm.step(case, weights, inputs))
    arm.close()
    wbytes = synth.weight_bytes_step(case)
    total = sum(times)
    value = wbytes * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{case.name}: {case.n_layers} layers x (q|k|v 4608x3584, o 3584x3584, ffn_gu "
                               f"37888x3584 + SiLU*mul + q8_0(h), down 3584x18944), batch 1",
                   "sample_per_step": "one whole step (every layer)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle", "cores": n,
                         "sample": f"one whole step per timed step, C oracle, rows split over {n} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------------------------------------

def config_suite(mq, device, oracle_arms=True):
    """The other workloads of the matvec, each timed on its own (context for the step's number).

    Every call is captured in a CUDA graph and replayed; times are CUDA events around whole
    replays (per-call = replay / calls).  Workloads smaller than twice the L2 are timed on
    rotated device copies of the same weights, so each call streams its weights from HBM;
    the single matvec is also reported warm (its 295 KB stay in L2).

    With oracle_arms, each entry also carries the CPU oracle's time for the same call on the
    same host bytes (median of up to 3 runs): on one thread and on all the threads of the
    process's affinity (static row partition); the 0.5B FFN as all 24 layers in order.
    """
    import torch
    import oracle
    from quantized_decode_matvec_gb300 import synth
    l2 = 2 * 129 * 1024 * 1024
    out = {}
    stream = torch.cuda.Stream(device)
    arms = [OracleArm(1), OracleArm(host_cores())] if oracle_arms else []

    def ora(name, fn, reps=3, per=1):
        """oracle seconds of fn(arm) on each arm, as µs per call (`per` calls per fn)"""
        if not arms:
            return
        t1 = oracle_time(lambda: fn(arms[0]), reps)
        tn = oracle_time(lambda: fn(arms[1]), reps)
        out[name].update(oracle_us_1_thread=round(t1 * 1e6 / per, 1),
                         oracle_us_all_threads=round(tn * 1e6 / per, 1), oracle_threads=arms[1].threads,
                         gpu_over_oracle_all_threads=round(tn * 1e6 / per / out[name]["us_per_call"], 1))

    last = {}

    def timed(calls, reps=CONFIG_REPS):
        """median per-call ms of a graph holding `calls` (a list of zero-arg launches), over at
        least CONFIG_REPS timed replays after CONFIG_WARMUP untimed ones; the mean and its
        standard error go to `last` for rec()."""
        reps = max(reps, CONFIG_REPS)
        with torch.cuda.stream(stream):
            for c in calls:  # warm (lazy state, caches)
                c()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in calls:
                c()
        for _ in range(CONFIG_WARMUP):
            g.replay()
        torch.cuda.synchronize()
        t = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            t.append(e0.elapsed_time(e1))
        per = [v / len(calls) for v in t]
        last.update(median=statistics.median(per), mean=statistics.mean(per), sem=sem(per), n=len(per))
        return last["median"]

    def stats_us(ms):
        """mean and standard error (µs) of the last timing, on the scale of `ms`"""
        k = ms / last["median"] if last.get("median") else 0.0
        return dict(us_mean=round(last["mean"] * k * 1e3, 3), us_sem=round(last["sem"] * k * 1e3, 3),
                    timed_replays=last["n"])

    def mv_calls(Ws, rows, K, x, y):
        descs = [mq.upload_struct(mq.mv_desc(W, rows, K, y, x=x, ncols=x.shape[0]), device) for W in Ws]

        def mk(d):
            return lambda: mq._check(mq.mq_matvec_q4K_q8_0(d.data_ptr(), rows, K, x.shape[0],
                                                           torch.cuda.current_stream().cuda_stream), "matvec")
        return [mk(d) for d in descs], descs

    def ffn_calls(pairs, H, I, x):
        nc = x.shape[0]
        y = torch.empty((nc, H), dtype=torch.float32, device=device)
        h = torch.empty((nc, I // 32 * 34), dtype=torch.uint8, device=device)
        descs = [mq.upload_struct(mq.ffn_desc(gu, dn, H, I, h, y, x=x, ncols=nc), device) for gu, dn in pairs]

        def mk(d):
            return lambda: mq._check(mq.mq_ffn_gu_silu_down(d.data_ptr(), H, I, nc,
                                                            torch.cuda.current_stream().cuda_stream), "ffn")
        return [mk(d) for d in descs], descs

    peak, _ = measured_hbm_peak()

    def rec(name, ms, wbytes, **extra):
        gbs = wbytes / (ms / 1e3) / 1e9
        out[name] = dict(us_per_call=round(ms * 1e3, 3), **stats_us(ms), weight_bytes=wbytes,
                         weight_gbs=round(gbs, 1), frac_of_measured_hbm=round(gbs / peak, 3), **extra)

    # single matvec 512 x 1024 (seed 0): warm, and rotated copies (HBM)
    c = synth.MATVEC_512x1024
    W_np, x_np = synth.matvec_case_inputs(c)
    W = torch.from_numpy(W_np).to(device)
    x = torch.from_numpy(x_np).to(device)
    y = torch.empty((1, c.rows), dtype=torch.float32, device=device)
    calls, keep = mv_calls([W] * 64, c.rows, c.K, x, y)
    rec("matvec_512x1024_warm_L2", timed(calls), W.numel(), note="weights L2-resident")
    ncopy = l2 // W.numel() + 1
    copies = [W.clone() for _ in range(ncopy)]
    calls, keep = mv_calls(copies, c.rows, c.K, x, y)
    rec("matvec_512x1024_hbm", timed(calls, 5), W.numel(), copies=ncopy)
    del copies, keep
    ora("matvec_512x1024_hbm", lambda a: a.matvec(W_np, oracle.quantize_q8_0(x_np), c.rows, c.K))

    # 0.5B-class FFN, 24 layers (202 MB: larger than L2 as it is)
    f = synth.FFN_05B
    host = [synth.ffn_layer_weights(f, l) for l in range(f.n_layers)]
    pairs = [tuple(torch.from_numpy(w).to(device) for w in hw) for hw in host]
    x_np = synth.ffn_layer_input(f, 0)
    x = torch.from_numpy(x_np).to(device)
    calls, keep = ffn_calls(pairs, f.H, f.I, x)
    ms = timed(calls)
    wb = sum(a.numel() + b.numel() for a, b in pairs)
    rec("ffn_0.5B_x24_per_layer", ms, wb // f.n_layers, total_us_24_layers=round(ms * 1e3 * f.n_layers, 2),
        launch="two kernels per layer (gate/up, down), 48 graph nodes")
    # the same 24 layers as one persistent launch (mq_step on an FFN-only stack: the down
    # phase reads h as tagged records, each layer's gate/up waits for every CTA's previous down)
    sb = mq.StepBuffers([{"gu": gu, "down": dn} for gu, dn in pairs], f.H, f.I, 0, 0, 0, 1)
    for l in range(f.n_layers):
        sb.c[l].copy_(torch.from_numpy(synth.ffn_layer_input(f, l)))
    ms_p = timed([lambda: sb.step(torch.cuda.current_stream(), mq.MQ_STEP_PERSISTENT)]) / f.n_layers
    rec("ffn_0.5B_x24_persistent_per_layer", ms_p, wb // f.n_layers,
        total_us_24_layers=round(ms_p * 1e3 * f.n_layers, 2),
        launch="one persistent kernel for the 24 layers (mq_step, FFN-only stack)")
    assert mq.mq_read_device_status(0) == 0
    del pairs, keep, sb
    ora("ffn_0.5B_x24_per_layer", lambda a: [a.ffn(gu, dn, x_np, f.H, f.I) for gu, dn in host], reps=1,
        per=f.n_layers)
    del host

    # 7B FFN (115 MB: rotated over 5 copies), batch 1 and 2/4/8 columns
    f = synth.FFN_7B
    gu_np, dn_np = synth.ffn_layer_weights(f, 0)
    gu, dn = torch.from_numpy(gu_np).to(device), torch.from_numpy(dn_np).to(device)
    pairs = [(gu, dn)] + [(gu.clone(), dn.clone()) for _ in range(4)]
    wb = gu.numel() + dn.numel()
    for nc in (1,) + tuple(synth.FFN_7B_NCOLS):
        x_np = synth.ffn_layer_input(f, 0, nc)
        x = torch.from_numpy(x_np).to(device)
        calls, keep = ffn_calls(pairs, f.H, f.I, x)
        rec(f"ffn_7B_ncols{nc}", timed(calls), wb, copies=len(pairs))
        ora(f"ffn_7B_ncols{nc}", lambda a: a.ffn(gu_np, dn_np, x_np, f.H, f.I), reps=1)
    del pairs, gu, dn, keep, gu_np, dn_np

    # K sweep, 4096 rows (rotated copies to exceed twice the L2)
    for K in synth.KSWEEP_KS:
        W_np, x_np = synth.ksweep_inputs(K)
        W = torch.from_numpy(W_np).to(device)
        x = torch.from_numpy(x_np).to(device)
        y = torch.empty((1, synth.KSWEEP_ROWS), dtype=torch.float32, device=device)
        ncopy = l2 // W.numel() + 1
        copies = [W] + [W.clone() for _ in range(ncopy - 1)]
        calls, keep = mv_calls(copies, synth.KSWEEP_ROWS, K, x, y)
        rec(f"ksweep_4096x{K}", timed(calls, 5), W.numel(), copies=ncopy)
        del copies, keep
        ora(f"ksweep_4096x{K}", lambda a: a.matvec(W_np, oracle.quantize_q8_0(x_np), synth.KSWEEP_ROWS, K))
    # the other weight types (q4_0: the pages' 0.5B model; q8_0), 4096 x 14336, rotated copies
    K = 14336
    x_np = synth.activation(K, 1, seed=synth.KSWEEP_SEED)
    x = torch.from_numpy(x_np).to(device)
    y = torch.empty((1, synth.KSWEEP_ROWS), dtype=torch.float32, device=device)
    for wt in ("q4_0", "q8_0"):
        W_np = synth.wq_matrix(wt, synth.KSWEEP_ROWS, K, seed=synth.KSWEEP_SEED)
        W = torch.from_numpy(W_np).to(device)
        ncopy = l2 // W.numel() + 1
        copies = [W] + [W.clone() for _ in range(ncopy - 1)]
        fn = mq.mq_matvec_q4_0_q8_0 if wt == "q4_0" else mq.mq_matvec_q8_0_q8_0
        descs = [mq.upload_struct(mq.mv_desc(c_, synth.KSWEEP_ROWS, K, y, x=x), device) for c_ in copies]

        def mk(d, fn=fn):
            return lambda: mq._check(fn(d.data_ptr(), synth.KSWEEP_ROWS, K, 1,
                                        torch.cuda.current_stream().cuda_stream), "matvec")
        rec(f"{wt}_weights_4096x{K}", timed([mk(d) for d in descs], 5), W.numel(), copies=ncopy)
        del copies, descs
        ora(f"{wt}_weights_4096x{K}",
            lambda a: a.matvec_w(wt, W_np, oracle.quantize_q8_0(x_np), synth.KSWEEP_ROWS, K))
    # more columns: the MMQ matmul on the tensor cores at the 7B FFN shapes (rotated weight copies),
    # beside the decode kernel (MMVQ, dp4a) where both apply
    f = synth.FFN_7B
    for name, (R, K, tag) in {"gu": (2 * f.I, f.H, synth.TAG_GU), "down": (f.H, f.I, synth.TAG_DOWN)}.items():
        W0 = torch.from_numpy(synth.q4K_matrix(R, K, seed=f.seed, tag=tag)).to(device)
        copies = [W0] + [W0.clone() for _ in range(l2 // W0.numel() + 1)]
        for nc in (8, 16, 32, 64):
            x = torch.from_numpy(synth.activation(K, nc, seed=92)).to(device)
            y = torch.empty((nc, R), dtype=torch.float32, device=device)
            ws = torch.empty(max(mq.mq_mmq_workspace_bytes(R, K, nc), 128), dtype=torch.uint8, device=device)
            descs = [mq.upload_struct(mq.mv_desc(Wc, R, K, y, x=x, ncols=nc), device) for Wc in copies]

            def mk(d, nc=nc, ws=ws):
                return lambda: mq._check(mq.mq_mmq_q4K_q8_0(d.data_ptr(), R, K, nc, ws.data_ptr(), ws.numel(),
                                                            torch.cuda.current_stream().cuda_stream), "mmq")
            ms = timed([mk(d) for d in descs], 5)
            rec(f"mmq_{name}_{R}x{K}_ncols{nc}", ms, W0.numel(), copies=len(copies),
                int_tops=round(2.0 * R * K * nc / (ms / 1e3) / 1e12, 1),
                kernel="mmq_kernel (tcgen05.mma kind::f16 on exact nibble and q8_0 codes)")
            if nc == 8:  # the decode kernel on the same call
                calls, keep = mv_calls(copies, R, K, x, y)
                rec(f"mmvq_{name}_{R}x{K}_ncols8", timed(calls, 5), W0.numel(), copies=len(copies),
                    kernel="ring_kernel (dp4a)")
                del calls, keep
            del descs, ws
        del copies, W0
    assert mq.mq_read_device_status(0) == 0

    # prefill on the tensor cores: one 7B-class layer's GEMMs at 2048 tokens over the resident
    # f16 weight cache (built by mq_dequant_q4K_f16), activations converted once to f16
    tflops_peak = measured_bf16_peak()
    T = 2048
    st = synth.STEP_7B
    shapes = {"qkv": (st.qkv_rows, st.H), "o": (st.H, st.q_rows), "ffn_gu": (2 * st.I, st.H), "down": (st.H, st.I)}
    layer_us = 0.0
    for name, (R, K) in shapes.items():
        W16 = mq.dequant_q4K_f16(torch.from_numpy(synth.q4K_matrix(R, K, seed=90, tag=synth.TAG_W)).to(device), R, K)
        X16 = mq.convert_f32_f16(torch.from_numpy(synth.activation(K, T, seed=91)).to(device))
        Y = torch.empty((T, R), dtype=torch.float32, device=device)
        ms = timed([lambda: mq.gemm_f16(W16, X16, out=Y, stream=torch.cuda.current_stream())], reps=5)
        tf = 2.0 * T * R * K / (ms / 1e3) / 1e12
        out[f"prefill_gemm_{name}_{R}x{K}_T{T}"] = dict(
            us_per_call=round(ms * 1e3, 2), **stats_us(ms), tflops=round(tf, 1), bound="tensor",
            frac_of_measured_f16_peak=round(tf / tflops_peak, 3) if tflops_peak else None,
            kernel="gemm_f16_kernel (tcgen05.mma kind::f16, 128x256 tiles, TMA 128-byte swizzle)")
        layer_us += ms * 1e3
        del W16, X16, Y
    out["prefill_7B_layer_T2048"] = dict(us_per_layer=round(layer_us, 1),
                                         tokens_per_s_28_layers=round(T / (28 * layer_us / 1e6), 0),
                                         note="the four projection GEMMs of one layer; no attention, SiLU*mul or norms")
    assert mq.mq_read_device_status(0) == 0
    torch.cuda.synchronize()
    for a in arms:
        a.close()
    return out


def scaled_weight_copy(W, shift):
    """A device copy of a q4_K matrix with every super-block's d and dmin times 2^-shift (benchmark
    data only: the same quants and scales, smaller block scales)."""
    import torch
    Wc = W.clone()
    blk = Wc.view(-1, 144)
    dd = blk[:, 0:4].contiguous().view(torch.float16)
    dd = (dd.float() * 2.0 ** -shift).to(torch.float16)
    blk[:, 0:4] = dd.contiguous().view(torch.uint8).view(-1, 4)
    return Wc


def chained_arm(mq, case, layers, stream, g_default, shift=11, rounds=3, reps=5):
    """The step as a real decode chain (MQ_STEP_CHAINED): o reads q|k|v's output, the FFN reads o's,
    layer l+1 reads layer l's FFN output, passed between CTAs as tagged records.  Timed interleaved
    with the default persistent step.  A chain with no normalization between layers does not keep its
    scale (each SwiGLU layer squares it, and the weights' positive mean adds a component common to all
    rows that grows about K*mean per projection), so its weights are copies with d and dmin times
    2^-shift: the values stay finite and shrink to zero within a few layers instead of overflowing to
    inf (the kernels' work is the same for any finite values)."""
    import torch
    from quantized_decode_matvec_gb300.graph import StepGraph
    from quantized_decode_matvec_gb300 import synth
    wc = [{k: scaled_weight_copy(v, shift) for k, v in w.items()} for w in layers]
    cb = mq.StepBuffers(wc, case.H, case.I, case.qkv_rows, case.H, case.q_rows, case.ncols, chained=True)
    cb.a[0].copy_(torch.from_numpy(synth.step_layer_inputs(case, 0, 0)["a"]))
    gc = StepGraph(cb, flags=mq.MQ_STEP_PERSISTENT, stream=stream)
    t_chain, t_def = [], []
    for _ in range(rounds):
        t_chain += time_replays(gc.run, stream, reps)
        t_def += time_replays(g_default.run, stream, reps)
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    mags = cb.y_ffn.abs().amax(dim=(1, 2)).cpu().tolist()
    nonzero = sum(1 for m in mags if m > 0)
    out = {"median_ms": statistics.median(t_chain), "mean_ms": statistics.mean(t_chain), "sem_ms": sem(t_chain),
           "default_persistent_interleaved_median_ms": statistics.median(t_def),
           "weights": f"the step's weights with d, dmin x 2^-{shift}",
           "max_abs_ffn_out_first_last_layer": [mags[0], mags[-1]],
           "layers_with_nonzero_ffn_out": nonzero,
           "finite": bool(torch.isfinite(cb.outputs).all().item())}
    del gc, cb, wc
    torch.cuda.empty_cache()
    return out


def run_kernel_case(args):
    """One kernel on one small, fixed case, a few launches: a target for ncu captures (one kernel,
    few launches, a few hundred MB on the device).  Prints one JSON line with the mean launch time."""
    import torch
    from quantized_decode_matvec_gb300 import build as mqbuild
    mqbuild.build()
    from quantized_decode_matvec_gb300 import mq, synth
    device = torch.device("cuda", torch.cuda.current_device())
    mq.init(device.index)
    f = synth.FFN_7B
    R, K = 2 * f.I, f.H  # the 7B ffn_gu projection
    if args.kernel_case.startswith("gemm_o"):
        R = K = f.H  # the 7B o projection: 224 tiles on 152 CTAs, the last wave split
    W = torch.from_numpy(synth.q4K_matrix(R, K, seed=f.seed, tag=synth.TAG_GU)).to(device)
    if args.kernel_case.startswith("ffn"):
        # the whole 7B FFN (gate/up + SiLU·mul + q8_0(h), then down) for ncols columns
        nc = int(args.kernel_case.split("ncols")[1])
        Wd = torch.from_numpy(synth.q4K_matrix(f.H, f.I, seed=f.seed + 1)).to(device)
        x = torch.from_numpy(synth.activation(f.H, nc, seed=93)).to(device)
        y = torch.empty((nc, f.H), dtype=torch.float32, device=device)
        h = torch.empty((nc, mq.mq_q8_0_bytes(f.I)), dtype=torch.uint8, device=device)
        d = mq.upload_struct(mq.ffn_desc(W, Wd, f.H, f.I, h, y, x=x, ncols=nc), device)
        run = lambda: mq._check(mq.mq_ffn_gu_silu_down(d.data_ptr(), f.H, f.I, nc,
                                                        torch.cuda.current_stream().cuda_stream), "ffn")
        work = {"weight_bytes_per_launch": W.numel() + Wd.numel()}
    elif args.kernel_case.startswith("gemm"):
        T = 2048
        W16 = mq.dequant_q4K_f16(W, R, K)
        X16 = mq.convert_f32_f16(torch.from_numpy(synth.activation(K, T, seed=91)).to(device))
        Y = torch.empty((T, R), dtype=torch.float32, device=device)
        run = lambda: mq.gemm_f16(W16, X16, out=Y)
        work = {"tflops_per_launch": 2.0 * T * R * K / 1e12}
    else:
        nc = int(args.kernel_case.split("ncols")[1])
        x = torch.from_numpy(synth.activation(K, nc, seed=92)).to(device)
        y = torch.empty((nc, R), dtype=torch.float32, device=device)
        ws = torch.empty(max(mq.mq_mmq_workspace_bytes(R, K, nc), 128), dtype=torch.uint8, device=device)
        d = mq.upload_struct(mq.mv_desc(W, R, K, y, x=x, ncols=nc), device)
        run = lambda: mq._check(mq.mq_mmq_q4K_q8_0(d.data_ptr(), R, K, nc, ws.data_ptr(), ws.numel(),
                                                    torch.cuda.current_stream().cuda_stream), "mmq")
        work = {"weight_bytes_per_launch": W.numel()}
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    t = time_replays(run, torch.cuda.current_stream(), args.steps)
    assert mq.mq_read_device_status(0) == 0
    print(json.dumps({"kernel_case": args.kernel_case, "launches": args.steps, "mean_us": 1e3 * sum(t) / len(t),
                      **work}), flush=True)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist
    from quantized_decode_matvec_gb300 import build as mqbuild
    mqbuild.build()
    from quantized_decode_matvec_gb300 import mq, synth
    from quantized_decode_matvec_gb300.graph import PinnedFeeder, StepGraph

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    mq.init(device.index)
    case = synth.STEP_7B
    if args.layers != case.n_layers:  # profiling aid: the same layers, fewer of them (not the bench workload)
        import dataclasses
        case = dataclasses.replace(case, name=f"{case.name}_slice{args.layers}L", n_layers=args.layers)
    wbytes = synth.weight_bytes_step(case)
    per_layer = wbytes // case.n_layers

    want_cpu = rank == 0 and ws == 1 and not args.no_cpu_baseline
    host_weights = [] if want_cpu else None
    layers = build_step(case, device, mq, host=host_weights)
    bufs = mq.StepBuffers(layers, case.H, case.I, case.qkv_rows, case.H, case.q_rows, case.ncols)
    fill_inputs(bufs, case, 0)
    mode_flags = {"persistent": mq.MQ_STEP_PERSISTENT, "graph": 0, "pdl": mq.MQ_STEP_PDL}
    flags = mode_flags[args.mode]
    g = StepGraph(bufs, flags=flags)
    stream = g.stream
    alt = {m: StepGraph(bufs, flags=f, stream=stream) for m, f in mode_flags.items() if m != args.mode}

    # warm-up (untimed)
    for _ in range(args.warmup):
        g.run()
        for a in alt.values():
            a.run()
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0

    # ---- the timed region: K graph replays, inputs resident in HBM (3.67 GB >> L2: no flush needed)
    clocks = ClockSampler(device.index)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    clocks.mark()
    per_step = time_replays(g.run, stream, args.steps)
    torch.cuda.synchronize()
    clocks.mark()
    barrier()
    clk = clocks.stop()
    ms_local = sum(per_step) / len(per_step)
    ms, total_bytes = reduce_over_ranks(ms_local, float(wbytes), device if ws > 1 else None)
    value = total_bytes / (ms / 1e3) / 1e9

    # ---- interleaved arms (context): the other launch modes, and eager launches
    arms = {args.mode: []}
    arms.update({m: [] for m in alt})
    arms["eager"] = []
    eager_run = lambda: bufs.step(stream, 0)
    for _ in range(3):
        arms[args.mode] += time_replays(g.run, stream, 5)
        for m, a in alt.items():
            arms[m] += time_replays(a.run, stream, 5)
        with torch.cuda.stream(stream):
            arms["eager"] += time_replays(eager_run, stream, 5)
    arm_stats = {k: {"median_ms": statistics.median(v), "mean_ms": statistics.mean(v), "sem_ms": sem(v)}
                 for k, v in arms.items()}
    if not args.no_chained_arm:
        arm_stats["persistent_chained"] = chained_arm(mq, case, layers, stream, g)


    peak, peak_kind = measured_hbm_peak()
    act_bytes = case.n_layers * (3 * case.H * 4 + case.I // 32 * 34 * 2) * case.ncols
    out_bytes = case.n_layers * (case.qkv_rows + case.H + case.H) * 4 * case.ncols
    traffic_step, traffic_note_step = recorded_traffic("step_kernel_7B.md")
    if args.mode == "persistent":
        step_bytes = wbytes + act_bytes + out_bytes
        gbs = step_bytes / (ms_local / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                    "traffic": traffic_step,
                    "traffic_source": traffic_note_step,
                    "kernel": "step_kernel<1> (persistent: all 28 layers, one launch per step)",
                    "peak_kind": f"{peak_kind} (copy bandwidth)", "avg_launch_us": ms_local * 1e3,
                    "algorithmic_bytes_per_launch": step_bytes}
    else:
        # dominant kernel alone: ffn_gu + SiLU*mul + q8_0(h), over the 28 layers' weights
        ffn_descs = [bufs.table[l * 192 + 112:l * 192 + 192] for l in range(case.n_layers)]
        reps = 3

        def gu_all():
            for l in range(case.n_layers):
                mq._check(mq.mq_ffn_gate_up(ffn_descs[l].data_ptr(), case.H, case.I, case.ncols,
                                            stream.cuda_stream), "mq_ffn_gate_up")

        with torch.cuda.stream(stream):
            gu_all()
            t = time_replays(gu_all, stream, reps)
        gu_ms = sum(t) / (reps * case.n_layers)
        gu_bytes = (2 * case.I * (case.H // 256) * 144 + case.H * 4 * case.ncols
                    + case.I // 32 * 34 * case.ncols)
        gu_gbs = gu_bytes / (gu_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": gu_gbs, "peak": peak, "unit": "GB/s", "frac": gu_gbs / peak,
                    "traffic": recorded_traffic("ffn_gate_up_7B.md")[0],
                    "kernel": "ring_kernel<1,GU> (ffn_gu matvec + SiLU*mul + q8_0 of h), 37888x3584",
                    "peak_kind": f"{peak_kind} (copy bandwidth)", "avg_launch_us": gu_ms * 1e3,
                    "algorithmic_bytes_per_launch": gu_bytes}

    # ---- end to end through host buffers: pinned H2D of the inputs, replay, D2H of the outputs
    feeder = PinnedFeeder(bufs)
    outs = [bufs.outputs]  # y_qkv, y_o and y_ffn of every layer, one device-to-host copy
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    d2h = sum(o.numel() * o.element_size() for o in outs)
    inp = [synth.step_layer_inputs(case, l, 1) for l in range(case.n_layers)]
    feeder.load(np.stack([i["a"] for i in inp]), np.stack([i["b"] for i in inp]), np.stack([i["c"] for i in inp]))

    # inputs in, the step and the outputs out, captured as one graph with the step
    g_io = StepGraph(bufs, flags=flags, stream=stream, io=(feeder.inputs, host_out[0]))

    def e2e_step():
        g_io.run()
        stream.synchronize()

    for _ in range(2):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    e2e_ms_local = (time.perf_counter() - t0) * 1e3 / args.steps
    barrier()
    e2e_ms, _ = reduce_over_ranks(e2e_ms_local, 0.0, device if ws > 1 else None)
    e2e = {"value": total_bytes / (e2e_ms / 1e3) / 1e9, "unit": UNIT, "ms_per_step": e2e_ms,
           "h2d_bytes_per_step": feeder.h2d_bytes, "d2h_bytes_per_step": d2h,
           "api": "mq_step, the input copy and the output copy captured as one CUDA graph (graph.StepGraph io); pinned host inputs and outputs"}
    assert mq.mq_read_device_status(0) == 0
    launches_per_step = 1 if args.mode == "persistent" else 4 * case.n_layers

    cpu = cpu_baseline(case, host_weights) if want_cpu else None
    host_weights = None
    suite = (config_suite(mq, device, oracle_arms=not args.no_cpu_baseline)
             if (rank == 0 and not args.no_configs and args.layers == 28) else None)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "step_us": ms * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {
                "workload": f"{case.name}: {case.n_layers} layers x (q|k|v 4608x3584, o 3584x3584, ffn_gu 37888x3584 + "
                            f"SiLU*mul + q8_0(h), down 3584x18944), batch 1, one CUDA graph replay per step",
                "weight_bytes_per_step": wbytes, "weight_bytes_per_layer": per_layer,
                "l2": "inputs larger than L2 (3.67 GB of weights per step vs 129 MB L2); no flush",
                "parallelism": "replicas" if ws > 1 else "single GPU",
                "launch_mode": args.mode,
            },
            "frac_of_measured_hbm": value / ws / peak, "frac_of_nominal_8TBs": value / ws / NOMINAL_HBM_GBS,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "configs": suite,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "arms": arm_stats,
            "graph_kernel_nodes": g.node_count(),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["persistent", "graph", "pdl"], default="persistent",
                    help="step launch mode: one persistent kernel, or four kernels per layer (plain or PDL)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config timings (context only)")
    ap.add_argument("--no-chained-arm", action="store_true", help="skip the chained-step arm (context only)")
    ap.add_argument("--kernel-case", choices=["gemm_gu_T2048", "gemm_o_T2048", "mmq_gu_ncols16", "mmq_gu_ncols64",
                                              "ffn_ncols4", "ffn_ncols8"],
                    default=None,
                    help="run one kernel on a fixed small case a few times (a target for ncu), not the benchmark")
    ap.add_argument("--layers", type=int, default=28,
                    help="layers of the 7B stack (28 = the bench workload; fewer only for small profiling runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel_case:
        return run_kernel_case(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
