"""Benchmark: one step = layout -> FP8 dispatch -> combine over the 4096-token
workload (H=7168, top-8 of 256 experts, 8 virtual ranks, cap = largest expert
count), on one GB300 per process.

Prints ONE JSON line.  `value` is the step's algorithmic HBM traffic (bytes
read + written by layout, dispatch and combine) divided by the device-timed
step, in GB/s, summed over ranks.  Per-kernel microseconds and GB/s, the
roofline of the dominant kernel, an end-to-end number through the public API
with host buffers, clocks, and the CPU oracle's speed on the same workload
ride along.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: the
path has no exchange step on one GPU, so ranks share no data.
"""
from __future__ import annotations

import argparse
import hashlib
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

WORKLOAD = "throughput"
HBM_NOMINAL_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
PROFILES = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------- bytes


def algorithmic_bytes(T, H, K, E, R, cap, N, fp8):
    """Bytes each kernel must move: every token row is read once (not K
    times), unfilled capacity rows are not counted."""
    G = H // 128
    b = 1 if fp8 else 2
    layout = 4 * T * K + 4 * T * K + T * R + 4 * E + 4 * R
    dispatch = 2 * H * T + N * (H * b + (4 * G if fp8 else 0)) + 8 * T * K + 4 * E * cap
    combine = N * 2 * H + 12 * T * K + 2 * T * H
    return dict(layout=layout, dispatch=dispatch, combine=combine)


def workload_config(c, n_gpus: int = 1):
    """The workload both arms run (identical keys and values in both lines)."""
    return {"workload": f"{c.name}: T={c.T} H={c.H} K={c.K} E={c.E} R={c.R} cap={c.cap} "
                        "fp8 e4m3 dispatch (per-128 fp32 scales), bf16 combine, uniform routing",
            "T": c.T, "H": c.H, "K": c.K, "E": c.E, "R": c.R, "cap": c.cap,
            "dispatch_dtype": "e4m3", "combine_dtype": "bf16", "seed": c.seed,
            "parallelism": f"replicas x{n_gpus}",
            "l2": "inputs larger than L2: ~0.9 GB of HBM touched per step vs 129 MB L2, no flush "
                  "between steps; the isolated per-kernel times read 1 GiB before each call"}


# ---------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        rows = []
        for ts, line in self.lines:
            p = [x.strip() for x in line.split(",")]
            if len(p) < 10:
                continue
            try:
                rows.append((ts, float(p[2]), float(p[3]), p[5], p[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[4]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": sorted(reasons),
                "samples": len(inside)}


# ------------------------------------------------------------------ peaks


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        v = float(json.load(open(p))["hbm_gbs"])
        return v, "measured (STREAM-style copy on this pool's GB300)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


def ncu_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the kernel source as it is now (matching source hash)."""
    p = os.path.join(PROFILES, "ncu_traffic.json")
    try:
        d = json.load(open(p))
    except Exception:
        return None
    ent = d.get(kernel)
    if not ent:
        return None
    if ent.get("source_sha256") != source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_full_launch")


# the sources each measured kernel is compiled from (its own file, the shared
# device helpers and the public header); traffic counters stay valid while
# these are unchanged
KERNEL_SOURCES = {
    "dispatch_kernel": ["csrc/dispatch.cu", "csrc/dispatch_item.cuh", "csrc/common.cuh"],
    "combine_kernel": ["csrc/combine.cu", "csrc/common.cuh"],
}


def source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "combine_moedc_layout_gb300")
    files = [os.path.join(pkg, f) for f in KERNEL_SOURCES[kernel]]
    files.append(os.path.join(ROOT, "include", "moedc.h"))
    for f in files:
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()


# ------------------------------------------------------------ CPU oracle


def _token_chunks(T_s: int, n: int) -> list[tuple[int, int]]:
    n = max(1, min(n, T_s))
    return [(T_s * j // n, T_s * (j + 1) // n) for j in range(n)]


def oracle_step(c, T_s: int, threads: int = 1, pool=None, keep: bool = False):
    """One oracle pass (layout, fp8 dispatch, combine) over the first T_s
    tokens of the workload; returns (seconds, algorithmic bytes, outputs or
    None).

    threads > 1 splits the tokens of dispatch and combine into contiguous
    runs, one oracle call per run on a thread of `pool` (the oracle's ctypes
    calls release the GIL).  The layout stays one call: its slots are a scan
    in token order.  The oracle functions are the same ones either way."""
    import oracle
    from combine_moedc_layout_gb300 import synth

    fp8 = c.dtype == synth.FP8_E4M3
    idx = np.ascontiguousarray(c.topk_idx[:T_s])
    x = np.ascontiguousarray(c.x[:T_s])
    w = np.ascontiguousarray(c.topk_weights[:T_s])
    eo = c.extra["eo_host"]
    t0 = time.perf_counter()
    lay = oracle.layout(idx, c.E, c.R, c.cap)
    sl = lay["slot"]
    if threads <= 1:
        d = oracle.dispatch(x, idx, sl, c.E, c.cap, fp8=fp8)
        y = oracle.combine(eo, idx, sl, w)["y"]
        parts = None
    else:
        recv = np.zeros((c.E, c.cap, c.H), np.uint8 if fp8 else np.uint16)

        def run(ab):
            lo, hi = ab
            dd = oracle.dispatch(x[lo:hi], idx[lo:hi], sl[lo:hi], c.E, c.cap, fp8=fp8,
                                 recv=recv)
            yy = oracle.combine(eo, idx[lo:hi], sl[lo:hi], w[lo:hi])["y"]
            return lo, dd, yy

        parts = list(pool.map(run, _token_chunks(T_s, threads)))
    dt = time.perf_counter() - t0
    N = int(((idx >= 0) & (idx < c.E)).sum())
    b = algorithmic_bytes(T_s, c.H, c.K, c.E, c.R, c.cap, N, fp8)
    out = None
    if keep:
        if parts is None:
            out = dict(layout=lay, recv=d["recv"], scales=d["scales"], src_idx=d["src_idx"], y=y)
        else:
            G = c.H // 128
            scales = np.zeros((c.E, c.cap, G), np.float32) if fp8 else None
            src_idx = np.full((c.E, c.cap), -1, np.int32)
            for lo, dd, _ in parts:
                filled = dd["src_idx"] >= 0
                src_idx[filled] = dd["src_idx"][filled] + lo
                if fp8:
                    scales[filled] = dd["scales"][filled]
            out = dict(layout=lay, recv=recv, scales=scales, src_idx=src_idx,
                       y=np.concatenate([yy for _, _, yy in parts], axis=0))
    return dt, sum(b.values()), out


def same_oracle_outputs(a: dict, b: dict) -> bool:
    """Bit equality of two oracle_step outputs (single- vs multi-threaded)."""
    for k in ("recv", "src_idx", "y"):
        if not np.array_equal(a[k], b[k]):
            return False
    if (a["scales"] is None) != (b["scales"] is None):
        return False
    if a["scales"] is not None and not np.array_equal(a["scales"].view(np.uint32),
                                                      b["scales"].view(np.uint32)):
        return False
    return True


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name as lscpu prints it ("Model name"); x86
    /proc/cpuinfo carries it as "model name"; Arm kernels give only the
    implementer / part codes, reported as such when lscpu is missing."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10,
                           env=dict(os.environ, LC_ALL="C"))
        for line in r.stdout.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    fields = {}
    try:
        for line in open("/proc/cpuinfo"):
            if ":" in line:
                k, v = line.split(":", 1)
                fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "cpu part" in fields:
        return f"Arm CPU implementer {fields.get('cpu implementer', '?')} part {fields['cpu part']}"
    import platform
    return platform.machine()


def cpu_baseline_full(c) -> dict:
    """The oracle timed on one full step of the workload: once on one core,
    once with the tokens split over every host core; the two runs' outputs
    must be bit-identical."""
    from concurrent.futures import ThreadPoolExecutor

    n = host_cores()
    dt1, b, out1 = oracle_step(c, c.T, keep=True)
    with ThreadPoolExecutor(max_workers=n) as pool:
        oracle_step(c, min(c.T, 4 * n), threads=n, pool=pool)     # warm the pool
        dtn, _, outn = oracle_step(c, c.T, threads=n, pool=pool, keep=True)
    if not same_oracle_outputs(out1, outn):
        raise RuntimeError("the multi-threaded oracle step differs from the single-threaded one")
    model = cpu_model()
    return {"value": b / dtn / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "seconds": dtn, "nproc": n, "cpu_model": model,
            "single_core": {"value": b / dt1 / 1e9, "seconds": dt1, "cores": 1},
            "sample": f"one full step of the workload (all {c.T} tokens): layout, fp8 dispatch, "
                      f"combine; plain-C oracle, dispatch and combine split by token runs over "
                      f"{n} threads (outputs bit-identical to the single-core run); {model}"}


def run_reference(args, rank: int) -> None:
    """The oracle as the reference arm: the same workload, on every host core
    of rank 0 (tokens split over threads for dispatch and combine), each step
    a token sample sized so that the run stays within about two minutes."""
    if rank != 0:
        return
    from concurrent.futures import ThreadPoolExecutor

    from combine_moedc_layout_gb300 import synth
    import oracle
    oracle.build()
    c = synth.make_case(WORKLOAD)
    c.extra["eo_host"] = synth.make_expert_out(c, 0)
    n = host_cores()
    budget_s = 120.0
    with ThreadPoolExecutor(max_workers=n) as pool:
        T_cal = min(c.T, 32 * n)
        dt, _, _ = oracle_step(c, T_cal, threads=n, pool=pool)     # calibration, not timed
        per_tok = dt / T_cal
        T_s = int(max(1, min(c.T, budget_s / (args.steps + args.warmup) / per_tok)))
        for _ in range(args.warmup):
            oracle_step(c, T_s, threads=n, pool=pool)
        tot_t = 0.0
        tot_b = 0
        for _ in range(args.steps):
            dt, b, _ = oracle_step(c, T_s, threads=n, pool=pool)
            tot_t += dt
            tot_b += b
    value = tot_b / tot_t / 1e9
    model = cpu_model()
    sample = (f"first {T_s} of {c.T} tokens of the workload per step (same H, K, E, R, cap); "
              f"plain-C oracle, dispatch and combine split by token runs over {n} threads; "
              f"{model}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 dispatch / bf16 combine (fp32 arithmetic)",
            "data": "synthetic (seeded numpy: x~N(0,1) bf16, uniform distinct top-8)",
            "config": workload_config(c, args.gpus),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": n, "kind": "oracle",
                             "nproc": n, "cpu_model": model, "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


METRIC = "dispatch & combine HBM GB/s (fraction of 8 TB/s) and us/call on 1 GB300"


# ------------------------------------------------------------- GPU arm


def max_over_ranks(v: float, world: int, device=None) -> float:
    """The slowest rank's time (every rank calls this)."""
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(step_bytes: int, world: int, ms_per_step: float) -> float:
    """Replicas each move step_bytes per step; the job's rate is bounded by
    the slowest rank's step time."""
    return step_bytes * world / (ms_per_step * 1e-3) / 1e9


def side_workloads(dev) -> dict:
    """Latency of the small workloads and per-kernel numbers of the skewed one.

    T = 4, 8, 16, 32, 64 (hidden 6144, top-8 of 128, 16 ranks) and the
    128-token / 288-expert workload: one MoE round = moedc_layout_dispatch (a
    single launch up to 1024 (token, k) entries, e4m3) -> moedc_dequant_e4m3
    (the identity expert) -> moedc_combine, reported as device us per round
    (events, eager, one round at a time), device us per CUDA-graph replay of
    the round, and host us to enqueue one round through the Python binding
    (ctypes included) or to launch the graph.  These footprints stay in L2:
    they are latencies, not HBM rates.  imbalanced: layout, bf16 dispatch and
    combine back to back, us and algorithmic GB/s per kernel.  rank_major: the
    same 4096-token e4m3 workload through rank layout, rank dispatch and rank
    combine (one row per token and destination rank).  combine_e4m3: combine
    from e4m3 rows.  dispatch_token_scale: e4m3 dispatch with one scale per
    token row.  large_t_layout_dispatch: moedc_layout_dispatch at 40000 tokens
    as one cooperative launch and as layout then dispatch.
    """
    import torch

    from combine_moedc_layout_gb300 import moedc, synth

    out = {}
    stream = torch.cuda.current_stream(dev)
    small = [("low4", 4), ("low8", 8), ("low16", 16), ("low32", 32), ("low64", 64),
             ("default_ll", None)]
    for name, t_over in small:
        c = synth.make_case("low16" if name.startswith("low") else name, T=t_over)
        T, H, K, E, R, cap = c.T, c.H, c.K, c.E, c.R, c.cap
        x = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).to(dev)
        idx = torch.from_numpy(c.topk_idx).to(dev)
        w = torch.from_numpy(c.topk_weights).to(dev)
        eo = torch.zeros((E, cap, H), dtype=torch.bfloat16, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        cnt = torch.empty(E, dtype=torch.int32, device=dev)
        rk = torch.empty(R, dtype=torch.int32, device=dev)
        inr = torch.empty((T, R), dtype=torch.uint8, device=dev)
        sl = torch.empty((T, K), dtype=torch.int32, device=dev)
        recv, scales, src = moedc.alloc_recv(E, cap, H, c.dtype, dev)
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

        def rnd(s_):
            r = moedc.moedc_layout_dispatch(x, idx, T, H, K, E, R, cap, c.dtype, cnt, rk, inr, sl,
                                            recv, scales, src, None, 0, st, s_)
            r |= moedc.moedc_dequant_e4m3(recv, scales, 0, cnt, E, cap, H, eo, s_)
            r |= moedc.moedc_combine(eo, E, cap, H, idx, sl, w, T, K, y, st, s_)
            if r != 0:
                raise RuntimeError(f"libmoedc returned {r}")

        for _ in range(20):
            rnd(stream)
        torch.cuda.synchronize(dev)
        reps = 200
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        host = []
        for a, b in evs:
            a.record(stream)
            h0 = time.perf_counter()
            rnd(stream)
            host.append(time.perf_counter() - h0)
            b.record(stream)
            torch.cuda.synchronize(dev)     # one round at a time: latency, not throughput
        dev_us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
        # the same round captured once in a CUDA graph and replayed
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            rnd(side)
            with torch.cuda.graph(graph, stream=side):
                rnd(side)
        torch.cuda.synchronize(dev)
        gevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(reps)]
        ghost = []
        for a, b in gevs:
            a.record(stream)
            h0 = time.perf_counter()
            graph.replay()
            ghost.append(time.perf_counter() - h0)
            b.record(stream)
            torch.cuda.synchronize(dev)
        g_us = sorted(a.elapsed_time(b) * 1e3 for a, b in gevs)
        if int(st.item()) != 0:
            raise RuntimeError(f"{name}: device status {int(st.item())}")
        med = lambda v: v[len(v) // 2]
        out[name] = {"T": T, "H": H, "K": K, "E": E, "R": R, "cap": cap,
                     "round": "moedc_layout_dispatch (e4m3, one launch) -> moedc_dequant_e4m3 "
                              "(identity expert) -> moedc_combine: 3 launches",
                     "device_us_per_round_median": med(dev_us),
                     "device_us_p10": dev_us[reps // 10], "device_us_p90": dev_us[9 * reps // 10],
                     "graph_replay_device_us_median": med(g_us),
                     "host_enqueue_us_median": med(sorted(host)) * 1e6,
                     "graph_replay_host_us_median": med(sorted(ghost)) * 1e6}
        del recv, scales, eo, graph

    # skewed routing, bf16 dispatch
    c = synth.make_case("imbalanced")
    T, H, K, E, R, cap = c.T, c.H, c.K, c.E, c.R, c.cap
    N = int(((c.topk_idx >= 0) & (c.topk_idx < E)).sum())
    nb = algorithmic_bytes(T, H, K, E, R, cap, N, False)
    x = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.from_numpy(c.topk_idx).to(dev)
    w = torch.from_numpy(c.topk_weights).to(dev)
    g_ = torch.Generator(device=dev).manual_seed(1)
    eo = torch.randn((E, cap, H), device=dev, generator=g_).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cnt = torch.empty(E, dtype=torch.int32, device=dev)
    rk = torch.empty(R, dtype=torch.int32, device=dev)
    inr = torch.empty((T, R), dtype=torch.uint8, device=dev)
    sl = torch.empty((T, K), dtype=torch.int32, device=dev)
    recv, scales, src = moedc.alloc_recv(E, cap, H, c.dtype, dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    wsb = moedc.moedc_layout_workspace_bytes(T, K, E, R)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    reps = 200
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
    for i in range(reps + 10):
        ev = evs[i - 10] if i >= 10 else None
        if ev:
            ev[0].record(stream)
        r = moedc.moedc_layout(idx, T, K, E, R, cap, cnt, rk, inr, sl, ws, wsb, st, stream)
        if ev:
            ev[1].record(stream)
        r |= moedc.moedc_dispatch(x, T, H, idx, sl, cnt, K, E, cap, c.dtype, recv, scales, src,
                                  st, stream)
        if ev:
            ev[2].record(stream)
        r |= moedc.moedc_combine(eo, E, cap, H, idx, sl, w, T, K, y, st, stream)
        if ev:
            ev[3].record(stream)
        if r != 0:
            raise RuntimeError(f"libmoedc returned {r}")
    torch.cuda.synchronize(dev)
    if int(st.item()) != 0:
        raise RuntimeError(f"imbalanced: device status {int(st.item())}")
    res = {"T": T, "H": H, "K": K, "E": E, "R": R, "cap": cap, "N": N,
           "rank0_load_ratio": c.extra["rank0_load_ratio"], "dispatch_dtype": "bf16"}
    for j, k in enumerate(("layout", "dispatch", "combine")):
        us = sorted(e[j].elapsed_time(e[j + 1]) * 1e3 for e in evs)
        m = sum(us) / len(us)
        res[k] = {"us_mean": m, "us_median": us[len(us) // 2], "algorithmic_bytes": nb[k],
                  "gbs": nb[k] / (m * 1e-6) / 1e9, "frac_of_8tbs": nb[k] / (m * 1e-6) / 1e9 / 8000}
    out["imbalanced"] = res
    del recv, scales, eo, src

    # rank-major packed receive on the 4096-token e4m3 workload: one row per
    # (token, destination rank) instead of one per (token, expert)
    c = synth.make_case(WORKLOAD)
    T, H, K, E, R, cap = c.T, c.H, c.K, c.E, c.R, c.cap
    G = H // 128
    x = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.from_numpy(c.topk_idx).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cnt = torch.empty(E, dtype=torch.int32, device=dev)
    rk = torch.empty(R, dtype=torch.int32, device=dev)
    inr = torch.empty((T, R), dtype=torch.uint8, device=dev)
    sl = torch.empty((T, K), dtype=torch.int32, device=dev)
    wsb = moedc.moedc_layout_workspace_bytes(T, K, E, R)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    assert moedc.moedc_layout(idx, T, K, E, R, cap, cnt, rk, inr, sl, ws, wsb, st, stream) == 0
    torch.cuda.synchronize(dev)
    rows = int(rk.sum().item())
    cap_rank = int(rk.max().item())
    rslot = torch.empty((T, R), dtype=torch.int32, device=dev)
    rrecv, rscales, rsrc = moedc.alloc_recv(R, cap_rank, H, c.dtype, dev)
    g_ = torch.Generator(device=dev).manual_seed(2)
    rout = torch.randn((R, cap_rank, H), device=dev, generator=g_).to(torch.bfloat16)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    rb = {"rank_layout": T * R + 4 * T * R,
          "rank_dispatch": 2 * H * T + rows * (H + 4 * G) + 4 * T * R + 4 * R * cap_rank,
          "rank_combine": rows * 2 * H + 4 * T * R + 2 * T * H}
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
    for i in range(reps + 10):
        ev = evs[i - 10] if i >= 10 else None
        if ev:
            ev[0].record(stream)
        r = moedc.moedc_rank_layout(inr, T, R, cap_rank, rslot, st, stream)
        if ev:
            ev[1].record(stream)
        r |= moedc.moedc_rank_dispatch(x, T, H, rslot, rk, R, cap_rank, c.dtype, rrecv, rscales,
                                       rsrc, stream)
        if ev:
            ev[2].record(stream)
        r |= moedc.moedc_rank_combine(rout, R, cap_rank, H, rslot, T, y, stream)
        if ev:
            ev[3].record(stream)
        if r != 0:
            raise RuntimeError(f"libmoedc returned {r}")
    torch.cuda.synchronize(dev)
    if int(st.item()) != 0:
        raise RuntimeError(f"rank-major: device status {int(st.item())}")
    res = {"T": T, "H": H, "R": R, "cap_rank": cap_rank, "rows": rows,
           "rows_expert_major": int(cnt.sum().item()), "dispatch_dtype": "e4m3"}
    for j, k in enumerate(("rank_layout", "rank_dispatch", "rank_combine")):
        us = sorted(e[j].elapsed_time(e[j + 1]) * 1e3 for e in evs)
        m = sum(us) / len(us)
        res[k] = {"us_mean": m, "us_median": us[len(us) // 2], "algorithmic_bytes": rb[k],
                  "gbs": rb[k] / (m * 1e-6) / 1e9, "frac_of_8tbs": rb[k] / (m * 1e-6) / 1e9 / 8000}
    out["rank_major"] = res
    del rrecv, rscales, rout

    # combine from e4m3 expert outputs (identity experts: the dispatched rows),
    # 4096-token workload, after the layout and e4m3 dispatch above
    recv, scales, src = moedc.alloc_recv(E, cap, H, c.dtype, dev)
    w = torch.from_numpy(c.topk_weights).to(dev)
    assert moedc.moedc_dispatch(x, T, H, idx, sl, cnt, K, E, cap, c.dtype, recv, scales, src, st,
                                stream) == 0
    N = int(((c.topk_idx >= 0) & (c.topk_idx < E)).sum())
    cb = N * (H + 4 * G) + 12 * T * K + 2 * T * H
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for i in range(reps + 10):
        ev = evs[i - 10] if i >= 10 else None
        if ev:
            ev[0].record(stream)
        r = moedc.moedc_combine_e4m3(recv, scales, 0, E, cap, H, idx, sl, w, T, K, y, st, stream)
        if ev:
            ev[1].record(stream)
        if r != 0:
            raise RuntimeError(f"libmoedc returned {r}")
    torch.cuda.synchronize(dev)
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    m = sum(us) / len(us)
    out["combine_e4m3"] = {"T": T, "H": H, "K": K, "E": E, "algorithmic_bytes": cb, "us_mean": m,
                           "us_median": us[len(us) // 2], "gbs": cb / (m * 1e-6) / 1e9,
                           "note": "back-to-back launches: the e4m3 rows (235 MB) partly stay in L2"}
    del recv, scales

    flush = torch.empty(256 << 20, dtype=torch.float32, device=dev)

    def flushed_us(fn):
        """median device us of fn, each call after a 1 GiB write that evicts L2"""
        for _ in range(5):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        v = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
        return v[len(v) // 2]

    # e4m3 dispatch with one scale per token row, same layout as above
    tok = moedc.FP8_E4M3 | moedc.SCALES_PER_TOKEN
    recv, scales, src = moedc.alloc_recv(E, cap, H, tok, dev)

    def tok_call():
        if moedc.moedc_dispatch(x, T, H, idx, sl, cnt, K, E, cap, tok, recv, scales, src, st,
                                stream) != 0:
            raise RuntimeError("moedc_dispatch (per-token scales) failed")

    tb = 2 * H * T + N * (H + 4) + 8 * T * K + 4 * E * cap
    us_tok = flushed_us(tok_call)
    out["dispatch_token_scale"] = {"T": T, "H": H, "K": K, "E": E, "algorithmic_bytes": tb,
                                   "us_median": us_tok, "gbs": tb / (us_tok * 1e-6) / 1e9,
                                   "timing": "L2 evicted before each call"}
    del recv, scales, src

    # one-call layout+dispatch beyond the single-launch layout (320000 entries):
    # the cooperative single launch against layout then dispatch
    c = synth.make_random_case(91, T=40000, H=128, K=8, E=128, R=8, cap=None, dtype=synth.BF16,
                               mask_p=0.01)
    T, H, K, E, R, cap = c.T, c.H, c.K, c.E, c.R, c.cap
    x = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.from_numpy(c.topk_idx).to(dev)
    cnt = torch.empty(E, dtype=torch.int32, device=dev)
    rk = torch.empty(R, dtype=torch.int32, device=dev)
    inr = torch.empty((T, R), dtype=torch.uint8, device=dev)
    sl = torch.empty((T, K), dtype=torch.int32, device=dev)
    recv, scales, src = moedc.alloc_recv(E, cap, H, c.dtype, dev)
    res = {"T": T, "H": H, "K": K, "E": E, "R": R, "cap": cap, "dtype": "bf16",
           "timing": "L2 evicted before each call"}
    for name, nbytes in (("single_cooperative_launch_us",
                          moedc.moedc_layout_dispatch_workspace_bytes(T, K, E, R)),
                         ("layout_then_dispatch_us", moedc.moedc_layout_workspace_bytes(T, K, E, R))):
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)

        def ld_call():
            if moedc.moedc_layout_dispatch(x, idx, T, H, K, E, R, cap, c.dtype, cnt, rk, inr, sl,
                                           recv, scales, src, ws, nbytes, st, stream) != 0:
                raise RuntimeError("moedc_layout_dispatch failed")

        res[name] = flushed_us(ld_call)
    if int(st.item()) != 0:
        raise RuntimeError(f"large-T layout+dispatch: device status {int(st.item())}")
    out["large_t_layout_dispatch"] = res
    return out


def isolated_kernels(dev, stream, calls: dict, nbytes: dict, reps: int = 400,
                     warm: int = 20) -> dict:
    """Each kernel timed alone: before every timed call a 1 GiB read evicts
    L2 (and writes back whatever the previous call left dirty, outside the
    timed region), then CUDA events on the launching stream bracket the one
    call.  `reps` timed calls after `warm` untimed ones, whatever --steps is;
    median, p10 and p90."""
    import torch

    flush = torch.ones(256 << 20, dtype=torch.float32, device=dev)
    peak, _ = hbm_peak()
    out = {}
    for name, fn in calls.items():
        for _ in range(warm):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        sink = []
        for a, b in ev:
            sink.append(flush.sum())
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        us = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
        med = us[len(us) // 2]
        gbs = nbytes[name] / (med * 1e-6) / 1e9
        out[name] = {"us_median": med, "us_p10": us[len(us) // 10],
                     "us_p90": us[(9 * len(us)) // 10], "reps": reps,
                     "algorithmic_bytes": nbytes[name], "gbs": gbs,
                     "frac_of_measured_peak": gbs / peak, "frac_of_8tbs": gbs / HBM_NOMINAL_GBS}
    del flush
    return out


def run_gpu(args, rank: int, world: int, local_rank: int) -> None:
    import torch

    from combine_moedc_layout_gb300 import build as mbuild
    from combine_moedc_layout_gb300 import moedc, synth

    if rank == 0 or world == 1:
        mbuild.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    lib = moedc.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    c = synth.make_case(WORKLOAD)
    fp8 = c.dtype == synth.FP8_E4M3
    T, H, K, E, R, cap = c.T, c.H, c.K, c.E, c.R, c.cap
    N = int(((c.topk_idx >= 0) & (c.topk_idx < E)).sum())
    nbytes = algorithmic_bytes(T, H, K, E, R, cap, N, fp8)
    step_bytes = sum(nbytes.values())

    # inputs resident in HBM
    x = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.from_numpy(c.topk_idx).to(dev)
    w = torch.from_numpy(c.topk_weights).to(dev)
    eo_host = synth.make_expert_out(c, 0)
    eo = torch.from_numpy(eo_host.view(np.int16)).view(torch.bfloat16).to(dev)
    # outputs and scratch, caller-owned and reused every step
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cnt = torch.empty(E, dtype=torch.int32, device=dev)
    rk = torch.empty(R, dtype=torch.int32, device=dev)
    inr = torch.empty((T, R), dtype=torch.uint8, device=dev)
    sl = torch.empty((T, K), dtype=torch.int32, device=dev)
    recv, scales, src = moedc.alloc_recv(E, cap, H, c.dtype, dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    wsb = moedc.moedc_layout_workspace_bytes(T, K, E, R)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    layout_kernels = 2 if T * K > 65536 else 1     # two launches only beyond 65536 entries
    launches_per_step = layout_kernels + 2

    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        r = moedc.moedc_layout(idx, T, K, E, R, cap, cnt, rk, inr, sl, ws, wsb, st, stream)
        if ev is not None:
            ev[1].record(stream)
        r |= moedc.moedc_dispatch(x, T, H, idx, sl, cnt, K, E, cap, c.dtype, recv, scales, src,
                                  st, stream)
        if ev is not None:
            ev[2].record(stream)
        r |= moedc.moedc_combine(eo, E, cap, H, idx, sl, w, T, K, y, st, stream)
        if ev is not None:
            ev[3].record(stream)
        if r != 0:
            raise RuntimeError(f"libmoedc returned {r}")

    if args.profile_steps:
        # a short run for profiler captures: the step's three kernels, then the
        # e4m3 combine over the dispatched rows, profile_steps times
        for _ in range(args.profile_steps):
            step()
            if moedc.moedc_combine_e4m3(recv, scales, 0, E, cap, H, idx, sl, w, T, K, y, st,
                                        stream) != 0:
                raise RuntimeError("moedc_combine_e4m3 failed")
        torch.cuda.synchronize(dev)
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        if rank == 0:
            print(json.dumps({"profile_steps": args.profile_steps, "workload": workload_config(c)}))
        return

    K_steps, W = args.steps, max(3, args.warmup)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.6)
    for _ in range(W):
        step()
    torch.cuda.synchronize(dev)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}: {moedc.strerror(int(st.item()))}")

    # the timed region: K steps back to back, events only at its two ends (events
    # recorded between kernels put a bubble between them on the device)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    start.record(stream)
    for _ in range(K_steps):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    # per-kernel durations: a second pass of the same steps with an event
    # between every two kernels (these include the bubbles the events add)
    K_inst = max(200, min(K_steps, 2000))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K_inst)]
    for i in range(K_inst):
        step(evs[i])
    torch.cuda.synchronize(dev)

    # every kernel alone, L2 evicted before each call (the per-call bar)
    def iso_layout():
        if moedc.moedc_layout(idx, T, K, E, R, cap, cnt, rk, inr, sl, ws, wsb, st, stream) != 0:
            raise RuntimeError("moedc_layout failed")

    def iso_dispatch():
        if moedc.moedc_dispatch(x, T, H, idx, sl, cnt, K, E, cap, c.dtype, recv, scales, src, st,
                                stream) != 0:
            raise RuntimeError("moedc_dispatch failed")

    def iso_combine():
        if moedc.moedc_combine(eo, E, cap, H, idx, sl, w, T, K, y, st, stream) != 0:
            raise RuntimeError("moedc_combine failed")

    def iso_combine_e4m3():
        if moedc.moedc_combine_e4m3(recv, scales, 0, E, cap, H, idx, sl, w, T, K, y, st,
                                    stream) != 0:
            raise RuntimeError("moedc_combine_e4m3 failed")

    iso_bytes = dict(nbytes, combine_e4m3=N * (H + 4 * (H // 128)) + 12 * T * K + 2 * T * H)
    t_iso0 = time.time()
    iso = isolated_kernels(dev, stream, {"layout": iso_layout, "dispatch": iso_dispatch,
                                         "combine": iso_combine,
                                         "combine_e4m3": iso_combine_e4m3}, iso_bytes)
    torch.cuda.synchronize(dev)
    t_iso1 = time.time()
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}: {moedc.strerror(int(st.item()))}")
    for k in ("dispatch", "combine"):
        iso[k]["meets_70pct_of_8tbs"] = iso[k]["gbs"] >= 0.7 * HBM_NOMINAL_GBS
    time.sleep(0.3)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    clocks_iso = sampler.summary(t_iso0, t_iso1)

    total_ms = start.elapsed_time(end)
    lay_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dis_ms = [e[1].elapsed_time(e[2]) for e in evs]
    com_ms = [e[2].elapsed_time(e[3]) for e in evs]
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / K_steps
    value = whole_job_gbs(step_bytes, world, ms_per_step)

    def kstats(ms_list, b):
        avg = sum(ms_list) / len(ms_list)
        srt = sorted(ms_list)
        return {"us_mean": avg * 1e3, "us_median": srt[len(srt) // 2] * 1e3,
                "us_p10": srt[len(srt) // 10] * 1e3, "us_p90": srt[(9 * len(srt)) // 10] * 1e3,
                "algorithmic_bytes": b, "gbs": b / (avg * 1e-3) / 1e9,
                "frac_of_8tbs": b / (avg * 1e-3) / 1e9 / HBM_NOMINAL_GBS}

    kern = {"layout": kstats(lay_ms, nbytes["layout"]),
            "dispatch": kstats(dis_ms, nbytes["dispatch"]),
            "combine": kstats(com_ms, nbytes["combine"])}
    peak, peak_src = hbm_peak()
    dom = max(("dispatch", "combine"), key=lambda k: kern[k]["us_mean"])
    kname = {"dispatch": "dispatch_kernel", "combine": "combine_kernel"}[dom]
    ach = kern[dom]["gbs"]
    for k in ("dispatch", "combine"):
        kern[k]["frac_of_measured_peak"] = kern[k]["gbs"] / peak
    roofline = {"bound": "hbm", "kernel": kname, "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak, "peak_source": peak_src + " (of measured)" if "measured" in
                peak_src else peak_src, "traffic": ncu_traffic(kname),
                "algorithmic_bytes_per_launch": kern[dom]["algorithmic_bytes"],
                "achieved_from": f"mean in-step duration over {K_inst} instrumented steps",
                "frac_isolated": {k: iso[k]["frac_of_measured_peak"]
                                  for k in ("dispatch", "combine", "combine_e4m3")},
                # each kernel alone (L2 evicted before every call): median us and
                # the fraction of the nominal 8 TB/s, the bar dispatch and combine
                # are held to at 4096 tokens
                "isolated_us": {k: iso[k]["us_median"]
                                for k in ("layout", "dispatch", "combine", "combine_e4m3")},
                "isolated_frac_of_8tbs": {k: iso[k]["frac_of_8tbs"]
                                          for k in ("dispatch", "combine", "combine_e4m3")}}

    # ---- end to end through the public API with host buffers.  A caller that
    # streams batches overlaps the next batch's host->device copies with this
    # batch's kernels: two device input sets, the copies split over several
    # copy streams, y and the counts copied back on their own stream.  Every
    # step still copies all of its inputs in and its result out.
    e2e_steps = max(4, min(20, K_steps))
    n_copy = 4
    h_x = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_idx = torch.from_numpy(c.topk_idx).pin_memory()
    h_w = torch.from_numpy(c.topk_weights).pin_memory()
    h_eo = torch.from_numpy(eo_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_ins = (h_x, h_idx, h_w, h_eo)
    h_outs = [(torch.empty((T, H), dtype=torch.bfloat16).pin_memory(),
               torch.empty(E, dtype=torch.int32).pin_memory()) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_ins)
    d2h = h_outs[0][0].numel() * 2 + h_outs[0][1].numel() * 4
    d_ins = [(x, idx, w, eo), tuple(torch.empty_like(t) for t in (x, idx, w, eo))]
    d_outs = [(y, cnt), (torch.empty_like(y), torch.empty_like(cnt))]
    copy_streams = [torch.cuda.Stream(dev) for _ in range(n_copy)]
    back_stream = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready = [[ev() for _ in range(n_copy)] for _ in range(2)]
    comp_done = [ev() for _ in range(2)]
    out_done = [ev() for _ in range(2)]
    for e_ in comp_done + out_done:
        e_.record(stream)

    def issue_h2d(b):
        for j, cs in enumerate(copy_streams):
            cs.wait_event(comp_done[b])           # the kernels two steps back are done with set b
            with torch.cuda.stream(cs):
                for src, dst in zip(h_ins, d_ins[b]):
                    fs, fd = src.view(-1), dst.view(-1)
                    n = fs.numel()
                    lo, hi = n * j // n_copy, n * (j + 1) // n_copy
                    if hi > lo:
                        fd[lo:hi].copy_(fs[lo:hi], non_blocking=True)
            in_ready[b][j].record(cs)

    def issue_compute(b):
        for e_ in in_ready[b]:
            stream.wait_event(e_)
        stream.wait_event(out_done[b])            # y / counts of set b were copied out
        bx, bidx, bw, beo = d_ins[b]
        by, bcnt = d_outs[b]
        r = moedc.moedc_layout(bidx, T, K, E, R, cap, bcnt, rk, inr, sl, ws, wsb, st, stream)
        r |= moedc.moedc_dispatch(bx, T, H, bidx, sl, bcnt, K, E, cap, c.dtype, recv, scales, src,
                                  st, stream)
        r |= moedc.moedc_combine(beo, E, cap, H, bidx, sl, bw, T, K, by, st, stream)
        if r != 0:
            raise RuntimeError(f"libmoedc returned {r}")
        comp_done[b].record(stream)

    def issue_d2h(b):
        back_stream.wait_event(comp_done[b])
        with torch.cuda.stream(back_stream):
            h_outs[b][0].copy_(d_outs[b][0], non_blocking=True)
            h_outs[b][1].copy_(d_outs[b][1], non_blocking=True)
        out_done[b].record(back_stream)

    def run_e2e(n):
        issue_h2d(0)
        for i in range(n):
            if i + 1 < n:
                issue_h2d((i + 1) % 2)
            issue_compute(i % 2)
            issue_d2h(i % 2)

    run_e2e(3)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for cs in copy_streams + [back_stream]:
        cs.wait_event(e0)
    run_e2e(e2e_steps)
    stream.wait_event(out_done[(e2e_steps - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    e2e_value = whole_job_gbs(step_bytes, world, e2e_ms)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    # the pipelined path still returns this workload's y
    if not torch.equal(h_outs[(e2e_steps - 1) % 2][0].view(torch.int16),
                       d_outs[(e2e_steps - 1) % 2][0].cpu().view(torch.int16)):
        raise RuntimeError("end-to-end result differs from the device result")

    side = None if args.no_side else side_workloads(dev)
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        c.extra["eo_host"] = eo_host
        cpu = cpu_baseline_full(c)

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": K_steps, "warmup": W, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 dispatch / bf16 combine (fp32 arithmetic)",
            "data": "synthetic (seeded numpy: x~N(0,1) bf16, uniform distinct top-8)",
            "config": workload_config(c, world),
            "frac_of_8tbs": value / world / HBM_NOMINAL_GBS,
            "kernels": kern, "kernels_isolated": iso, "roofline": roofline,
            "e2e": {"value": e2e_value, "unit": "GB/s", "ms_per_step": e2e_ms,
                    "steps": e2e_steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "path": "pinned host -> device copies of x, topk_idx, topk_weights, "
                            "expert_out (4 copy streams, two device input sets, the next "
                            "step's copies overlapping this step's kernels); moedc_layout, "
                            "moedc_dispatch, moedc_combine; y and counts back to pinned host "
                            "on a third stream"},
            "gpu_launches": launches_per_step * K_steps,
            "kernel_timing": f"kernels: in-step durations from a second pass of {K_inst} steps "
                             "with events between kernels (the step time comes from the clean "
                             "pass); kernels_isolated: each kernel alone, 1 GiB read before every "
                             "call to evict L2, 20 warm-ups then "
                             f"{iso['dispatch']['reps']} timed calls",
            "workloads": side,
            "clocks": clocks, "clocks_isolated": clocks_iso, "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the low-token / 128-token / imbalanced side measurements")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="only run this many steps (layout, e4m3 dispatch, combine, then the "
                         "e4m3 combine) and exit: a short command for profiler captures")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_gpu(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
