"""Benchmark of the QEvict decode step on GB300: decode steps/s and achieved HBM GB/s at 32K context.

One step = for every layer: append + split-K attention over sink / Full / Quantized / recent
windows + window-score update (one qevict_decode_step launch per layer), plus a routing event
(route + quantise + promote/copy launches) after every Omega-th step, for all sequences.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama8b_32k] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is whole-job decode steps/s with the inputs resident in HBM
(CUDA-graph replay of exactly K steps, CUDA events on the launching stream); `e2e` is the same
metric with every step's inputs copied from pinned host memory and its outputs copied back inside
the timed region; `roofline` is the decode kernel's algorithmic bytes per launch over its average
launch duration (CUDA events around each launch of an event-bracketed pass over the same
workload), against the measured HBM copy bandwidth.  `--impl reference` times the CPU oracle.
"""
from __future__ import annotations

import argparse
import ctypes
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
sys.path.insert(0, ROOT)

METRIC = "decode steps/sec and achieved HBM GB/s (% of GB300 peak) at 32K ctx, 1 GPU"
FALLBACK_HBM_GBS = 6800.0
D = 128


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--workload", default="llama8b_32k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--diag", type=int, default=0,
                    help="also run N routing events with the routing diagnostics against a FullKV cache")
    ap.add_argument("--int4", action="store_true", help="the INT4 / 64-token-window format of the workload")
    ap.add_argument("--ranker", type=int, default=0,
                    help="window ranking: 0 cumulative, 1 decayed, 2 p-norm, 3 key norm (GPU arm only)")
    ap.add_argument("--no-promotion", action="store_true", help="quantized windows never return to Full")
    ap.add_argument("--rope-base", type=float, default=0.0,
                    help="keys carry RoPE with this base and Quantized keys are kept before it (GPU arm only)")
    ap.add_argument("--budget", default=None, help="B_total as NUM/DEN of the full cache (overrides the workload)")
    ap.add_argument("--q", default=None, help="quantised fraction q as NUM/DEN (overrides the workload)")
    ap.add_argument("--sweep", action="store_true",
                    help="the long-context sweep: B_total in {10, 20, 40}%% x q in {0.5, 0.7, 0.9} of the workload "
                         "(INT2/W=32, or INT4/W=64 with --int4), one reduced measurement each; one JSON line")
    ap.add_argument("--layers", type=int, default=None,
                    help="run the workload with fewer layers (a smaller case for profiler captures; "
                         "the JSON line then reports that layer count)")
    ap.add_argument("--oracle-child", default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s: the measured cuBLAS burst figure, else the recipe's fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if d.get("bf16_tflops"):
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# --------------------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (the driver's library, read only)
    every ~2 ms while active; falls back to nvidia-smi polling when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting", 0x1: "gpu_idle"}

    def __init__(self, bus_id: str):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self._stop = threading.Event()
        self._on = threading.Event()
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            assert nv.nvmlInit_v2() == 0
            h = ctypes.c_void_p()
            assert nv.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(h)) == 0
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml, self._h = nv, h
            self._getr = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception:
            self._nvml = None
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def _run(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self._on.is_set() and self._nvml is not None:
                if self._nvml.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk)) == 0:
                    self.samples.append(clk.value)
                if self._getr(self._h, ctypes.byref(rs)) == 0:
                    for bit, name in self.REASONS.items():
                        if rs.value & bit and name != "gpu_idle":
                            self.reasons.add(name)
            time.sleep(0.002)

    def start(self):
        self._on.set()

    def pause(self):
        self._on.clear()

    def close(self):
        self._stop.set()
        self._t.join(timeout=2)

    def smi_snapshot(self):
        try:
            out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm", "--format=csv,noheader,nounits",
                                  "-i", "0"], capture_output=True, text=True, timeout=20).stdout.strip().splitlines()
            a, b = out[0].split(",")
            return int(a), int(b)
        except Exception:
            return None, None

    def summary(self):
        med = statistics.median(self.samples) if self.samples else None
        if med is None:
            med, mx = self.smi_snapshot()
            self.max_mhz = self.max_mhz or mx
        return {"sm_mhz": med, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "source": "nvml" if self._nvml is not None else "nvidia-smi"}


# --------------------------------------------------------------------------------------- CPU oracle

ORACLE_THREADS_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                      "CUDA_VISIBLE_DEVICES": ""}


def _oracle_worker(conn, wl_name, units, n_steps, seed):
    """One oracle process: owns the (layer, sequence) units given, prefill-routes them on seeded random
    prompt scores (the routing cost does not depend on their values; 32K-prompt attention on host
    cores is out of reach), then runs one decode step of every unit per request, with the routing
    event every Omega steps, and answers with its busy time."""
    import numpy as np
    from oracle import qevict_oracle as O
    from recoverable_quantized_kv_gb300 import synth
    wl = synth.workload(wl_name)
    cfg = O.Config.from_obj(wl, max_len=wl.prompt_len + n_steps + wl.omega)
    rng = np.random.default_rng(seed)
    state = []
    for layer, b in units:
        u = O.Unit(cfg)
        p = synth.prompt_inputs(wl, b, layer, with_queries=False)
        u.prefill_route(p["k"].float().numpy(), p["v"].float().numpy(), rng.random(O.prompt_windows(cfg)))
        d = synth.decode_inputs(wl, b, layer, steps=n_steps)
        state.append((u, d["q"].float().numpy(), d["k"].float().numpy(), d["v"].float().numpy()))
    conn.send("ready")
    while True:
        s = conn.recv()
        if s is None:
            break
        t0 = time.perf_counter()
        for u, q, k, v in state:
            u.decode_step(q[s], k[s], v[s])
            if (s + 1) % wl.omega == 0:
                u.route()
        conn.send(time.perf_counter() - t0)
    conn.close()


class OraclePool:
    """Oracle processes (spawned, one BLAS thread each) that decode the units of a workload in
    lockstep: a step is one decode step of every unit, the routing event included every Omega
    steps.  Units are dealt round-robin to the processes."""

    def __init__(self, wl_name, units, n_proc, n_steps, seed=12345):
        import multiprocessing as mp
        saved = {k: os.environ.get(k) for k in ORACLE_THREADS_ENV}
        os.environ.update(ORACLE_THREADS_ENV)
        try:
            ctx = mp.get_context("spawn")
            self.conns, self.procs = [], []
            for i in range(n_proc):
                a, b = ctx.Pipe()
                pr = ctx.Process(target=_oracle_worker, args=(b, wl_name, units[i::n_proc], n_steps, seed + i),
                                 daemon=True)
                pr.start()
                self.conns.append(a)
                self.procs.append(pr)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        for c in self.conns:
            assert c.recv() == "ready"

    def step(self, s):
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(s)
        busy = [c.recv() for c in self.conns]
        return time.perf_counter() - t0, busy

    def close(self):
        for c in self.conns:
            c.send(None)
        for pr in self.procs:
            pr.join(timeout=30)


def oracle_config1_full():
    """The tiny workload in full on one core: fp64 prompt attention for the scores, prefill routing,
    64 decode steps with 8 routing events (the oracle as it stands, one BLAS thread)."""
    import numpy as np
    from oracle import qevict_oracle as O
    from recoverable_quantized_kv_gb300 import synth
    wl = synth.workload("tiny_4k")
    cfg = O.Config.from_obj(wl)
    u = O.Unit(cfg)
    p = synth.prompt_inputs(wl, 0, 0)
    dec = synth.decode_inputs(wl, 0, 0)
    t0 = time.perf_counter()
    s0 = O.prefill_scores(p["q"].float().numpy(), p["k"].float().numpy(), cfg)
    u.prefill_route(p["k"].float().numpy(), p["v"].float().numpy(), s0)
    t1 = time.perf_counter()
    for s in range(wl.steps):
        u.decode_step(dec["q"][s].float().numpy(), dec["k"][s].float().numpy(), dec["v"][s].float().numpy())
        if (s + 1) % wl.omega == 0:
            u.route()
    t2 = time.perf_counter()
    return {"workload": "tiny_4k", "steps": wl.steps, "routing_events": wl.steps // wl.omega,
            "value": wl.steps / (t2 - t1), "unit": "steps/s", "prefill_s": round(t1 - t0, 3), "cores": 1}


def run_oracle_child(args):
    """Runs in a subprocess with one BLAS/OpenMP thread so `cores` is exact."""
    if args.oracle_child == "config1":
        print(json.dumps(oracle_config1_full()))


def oracle_steps(wl_name, n_units, n_proc, n_steps, warmup=0):
    """Steps/s of the oracle over the first n_units (layer, sequence) units of the workload, on n_proc
    processes: `warmup` untimed steps, then n_steps timed steps (wall clock of each lockstep step)."""
    from recoverable_quantized_kv_gb300 import synth
    wl = synth.workload(wl_name)
    units = [(l, b) for l in range(wl.n_layers) for b in range(wl.batch)][:n_units]
    pool = OraclePool(wl_name, units, n_proc, warmup + n_steps)
    try:
        walls = []
        for s in range(warmup + n_steps):
            wall, _ = pool.step(s)
            if s >= warmup:
                walls.append(wall)
    finally:
        pool.close()
    return sum(walls), wl


def cpu_baseline(args):
    """The oracle, as it stands, on the host cores of this machine (QEvict config-2 workload and the tiny
    workload): config 1 in full on one core; config 2 over every one of its 32 (layer, sequence)
    units on all cores (one process per core, one BLAS thread each), and on one core over a 2-unit
    sample scaled to the 32 units.  16 decode steps each, 2 routing events."""
    cores = len(os.sched_getaffinity(0))
    t0 = time.time()
    out = {"kind": "oracle", "unit": "steps/s", "cpu": _cpu_model(), "host_cores": cores}
    try:
        env = dict(os.environ, **ORACLE_THREADS_ENV)
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-child", "config1"],
                           capture_output=True, text=True, env=env, timeout=600)
        out["config1_full_1core"] = json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else \
            {"error": r.stderr[-300:]}
        from recoverable_quantized_kv_gb300 import synth
        wl = synth.workload(args.workload)
        U, steps = wl.n_layers * wl.batch, 16
        t_all, _ = oracle_steps(args.workload, U, min(cores, U), steps)
        t_one, _ = oracle_steps(args.workload, 2, 1, steps)
        out.update({
            "value": steps / t_all, "cores": min(cores, U),
            "sample": f"oracle on all {U} (layer, sequence) units of {wl.name}, {steps} decode steps with "
                      f"{steps // wl.omega} routing events, {min(cores, U)} processes x 1 BLAS thread; prompt "
                      f"scores seeded random (prefill excluded)",
            "config2_all_units_allcores": {"value": steps / t_all, "cores": min(cores, U), "units": U,
                                           "steps": steps, "measured": True},
            "config2_1core": {"value": steps / (t_one * U / 2), "cores": 1, "units_timed": 2, "steps": steps,
                              "measured": False, "note": f"2 units timed on one core, scaled to {U} units"},
        })
    except Exception as e:   # the GPU figures stand on their own; report why the baseline is missing
        out.update({"value": None, "cores": cores, "error": repr(e)[-300:]})
    out["wall_s"] = round(time.time() - t0, 1)
    return out


def _cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part", "hardware")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return os.uname().machine


# --------------------------------------------------------------------------------------- GPU bench

def algorithmic_bytes(wl, f_count, q_count, local_tokens, payload):
    """Bytes a decode launch must move for one (sequence, layer): Full windows bf16 K+V, Quantized
    windows' codes + parameters, sink + recent tokens, table entries, one score read+write per
    accessible window, and the step's q / out / k_new / v_new / ring write."""
    c_tok = 4 * wl.h_kv * D
    W = wl.window
    n_local_windows = math.ceil(local_tokens / W)
    return (f_count * W * c_tok + q_count * payload + (wl.n_sink + local_tokens) * c_tok
            + (f_count + q_count) * 8 + 8 * (f_count + q_count + n_local_windows)
            + 2 * wl.h_q * D * 2 + 2 * wl.h_kv * D * 2 + c_tok)


def route_bytes(wl, n_cand, firstq, promo, aged, payload):
    c_tok = 4 * wl.h_kv * D
    W = wl.window
    return 8 * n_cand + firstq * (W * c_tok + payload) + promo * (payload + W * c_tok) + aged * (W * c_tok + W * c_tok)


def traffic_from_profile(kernel_sha):
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    return d.get("dram_bytes_per_launch") if d.get("kernel_source_sha") == kernel_sha else None


def _strip_comments(src: str) -> str:
    """C++ source without comments, trailing blanks or blank lines (string literals kept)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            while i < n and src[i] != "\n":
                i += 1
        elif src.startswith("/*", i):
            k = src.find("*/", i + 2)
            i = n if k < 0 else k + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(ln.rstrip() for ln in "".join(out).split("\n") if ln.strip())


def kernel_sha():
    """Hash of the decode kernel's code (decode.cu, common.cuh, cache_dev.cuh), comments and blank lines
    left out, so that a DRAM capture stays tied to the code it measured."""
    h = hashlib.sha256()
    for f in ("decode.cu", "common.cuh", "cache_dev.cuh"):
        with open(os.path.join(ROOT, "recoverable_quantized_kv_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's time.  Ranks are independent replicas (each decodes its own cache: the
    path has no exchange step), so the whole job ends when the slowest replica does."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, steps: int, ms: float) -> float:
    """Steps per second of the whole job: every replica takes `steps` steps in `ms` (max over ranks)."""
    return world * steps / (ms / 1e3)


def run_gpu(args, rank, world):
    import numpy as np
    import torch
    from recoverable_quantized_kv_gb300 import binding, build, synth
    build.build()
    binding.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = synth.workload(args.workload) if args.layers is None else synth.workload(args.workload, n_layers=args.layers)
    if args.rope_base > 0:
        wl = wl.replace(rope_base=args.rope_base)
    if args.int4:
        wl = wl.replace(window=64, bits=4)
    if args.ranker or args.no_promotion:
        wl = wl.replace(ranker=args.ranker, no_promotion=1 if args.no_promotion else 0)
    if args.budget:
        num, den = (int(x) for x in args.budget.split("/"))
        wl = wl.replace(budget_num=num, budget_den=den)
    if args.q:
        num, den = (int(x) for x in args.q.split("/"))
        wl = wl.replace(q_num=num, q_den=den)
    K, Wm = args.steps, args.warmup
    Om = wl.omega
    K_kern = 2 * Om
    R_roof = 7                                       # replays of the steady-state graph
    K_e2e = 0 if args.no_e2e else K
    # (Om - 1) per phase: steps that realign the phase to a routing event
    total = Wm + 4 * (Om - 1) + K_kern + R_roof * Om + K + 2 * K_e2e
    steps_cap = max(wl.steps, int(math.ceil(total / Om) * Om) + Om)
    cfg = binding.make_config(wl, max_len=wl.prompt_len + steps_cap)
    cache = binding.Cache(cfg, device=dev)
    if wl.rope_base > 0:
        cache.set_rope_table(torch.from_numpy(synth.rope_table(cfg.max_len, wl.rope_base)).to(dev))
    bud = cache.bud
    L, B = wl.n_layers, wl.batch
    stream = torch.cuda.Stream(device=dev)      # graphs cannot be captured on the legacy default stream
    torch.cuda.set_stream(stream)

    # ---- prefill every layer (inputs generated on the device; scores from prompt attention)
    t_pre = time.time()
    for layer in range(L):
        ins = [synth.prompt_inputs(wl, b, layer, device=dev) for b in range(B)]
        q = torch.stack([x["q"] for x in ins])
        k = torch.stack([x["k"] for x in ins])
        v = torch.stack([x["v"] for x in ins])
        cache.prefill_route(layer, k, v, s0=None, q_prompt=q)
        del ins, q, k, v
    torch.cuda.synchronize()
    t_pre = time.time() - t_pre

    # ---- prefill scoring throughput: the two causal passes over one layer's prompt (tensor cores)
    pin = [synth.prompt_inputs(wl, b, 0, device=dev) for b in range(B)]
    pq = torch.stack([x["q"] for x in pin])
    pk = torch.stack([x["k"] for x in pin])
    del pin
    npw = (wl.prompt_len - wl.n_sink + wl.window - 1) // wl.window
    ps0 = torch.empty(B, npw, dtype=torch.float32, device=dev)
    cache.prefill_scores(pq, pk, ps0, stream)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(3):
        cache.prefill_scores(pq, pk, ps0, stream)
    p1.record(stream)
    torch.cuda.synchronize()
    pre_ms = p0.elapsed_time(p1) / 3
    pre_flops = 2.0 * wl.prompt_len * (wl.prompt_len + 1) * D * wl.h_q * B   # two passes of causal q.k
    pre_tf = pre_flops / (pre_ms / 1e3) / 1e12
    tpeak, tpeak_kind = measured_tensor_peak()
    prefill_scores = {"ms_per_layer": pre_ms, "tflops": pre_tf, "peak_tflops": tpeak, "frac": pre_tf / tpeak,
                      "flops_per_layer": pre_flops,
                      "tflops_single_product": pre_tf / 2, "frac_single_product": pre_tf / 2 / tpeak,
                      "note": "tflops/frac count the causal q.k products of both passes (row log-sum-exp, then "
                              "column sums, which recomputes q.k); *_single_product count the one causal product "
                              "the scores need.  tcgen05.mma M=N=128 bf16 with TMA tensor-map loads; "
                              f"peak = {tpeak_kind} dense bf16 burst"}
    del pq, pk, ps0

    # ---- decode inputs for every step resident in HBM: [step][layer][B][...]
    qs = torch.empty(total, L, B, wl.h_q, D, dtype=torch.bfloat16, device=dev)
    ks = torch.empty(total, L, B, wl.h_kv, D, dtype=torch.bfloat16, device=dev)
    vs = torch.empty_like(ks)
    for layer in range(L):
        for b in range(B):
            d = synth.decode_inputs(wl, b, layer, steps=total, device=dev)
            qs[:, layer, b] = d["q"]
            ks[:, layer, b] = d["k"]
            vs[:, layer, b] = d["v"]
    outs = torch.empty(L, B, wl.h_q, D, dtype=torch.bfloat16, device=dev)
    state = {"step": 0, "launches": 0}

    def one_step(i, q_src=None, k_src=None, v_src=None, out_dst=None, events=None):
        for layer in range(L):
            if events is not None:
                events[layer][0].record(stream)
            cache.decode_step(layer, (q_src if q_src is not None else qs[i])[layer],
                              (k_src if k_src is not None else ks[i])[layer],
                              (v_src if v_src is not None else vs[i])[layer],
                              (out_dst if out_dst is not None else outs)[layer], stream)
            if events is not None:
                events[layer][1].record(stream)
            state["launches"] += 1
        state["step"] += 1
        if state["step"] % Om == 0:
            cache.route(stream)
            state["launches"] += 4     # score flush, route, quantise, migrate

    def read_meta():
        lay = cache.layout
        ms = []
        for u in range(L * B):
            off = lay.off_meta + u * lay.stride_meta
            ms.append(cache.arena[off:off + 64].view(torch.int32).cpu().numpy().copy())
        return ms

    # ---- warm-up (untimed), then up to the next routing event so that every later phase starts on one
    for _ in range(Wm):
        one_step(state["step"])
    while state["step"] % Om:
        one_step(state["step"])
    torch.cuda.synchronize()

    # ---- event-bracketed pass: decode kernel duration and the algorithmic bytes of each launch
    kern_ms, kern_bytes, step_bytes = [], [], []
    c0 = cache.counters()
    per_event = []          # tier transitions of each routing event (counter deltas, all units)
    last_ctr = [c0]

    def record_event():
        cur = cache.counters()
        per_event.append({k: cur[k] - last_ctr[0][k] for k in cur})
        last_ctr[0] = cur

    for _ in range(K_kern):
        metas = read_meta()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
        i = state["step"]
        one_step(i, events=ev)
        torch.cuda.synchronize()
        if state["step"] % Om == 0:
            record_event()
        sb = 0
        for layer in range(L):
            by = 0
            for b in range(B):
                m = metas[layer * B + b]
                T, n_route, nf, nq = int(m[0]), int(m[1]), int(m[2]), int(m[3])
                local = T - wl.n_sink - n_route * wl.window + 1
                by += algorithmic_bytes(wl, nf, nq, local, bud.payload)
            kern_ms.append(ev[layer][0].elapsed_time(ev[layer][1]))
            kern_bytes.append(by)
            sb += by
        step_bytes.append(sb)
    c1 = cache.counters()
    n_events = K_kern // Om
    rb = route_bytes(wl, (bud.k_f + bud.k_q) * L * B * n_events, c1["first_quant"] - c0["first_quant"],
                     c1["promotions"] - c0["promotions"], (c1["aged_full"] - c0["aged_full"]), bud.payload)
    bytes_per_step = statistics.mean(step_bytes) + rb / K_kern

    # ---- steady-state decode launches: the Omega decode steps up to the next routing event (all
    # layers, no routing between them) captured in one CUDA graph and replayed between two events,
    # so consecutive launches overlap as they do inside a step; after each replay the host mirror of
    # the cache is resynchronised and the routing event runs untimed.  R_roof replays: median, spread
    assert state["step"] % Om == 0
    gd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gd, stream=stream):
        for j in range(Om):
            i = state["step"] + j
            for layer in range(L):
                cache.decode_step(layer, qs[i][layer], ks[i][layer], vs[i][layer], outs[layer], stream)
    torch.cuda.synchronize()
    replay_us = []
    for _ in range(R_roof):
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        gd.replay()
        d1.record(stream)
        torch.cuda.synchronize()
        replay_us.append(d0.elapsed_time(d1) * 1e3 / (Om * L))
        cache.check(stream)          # the host mirror learns the Omega steps the replay took
        cache.route(stream)
        state["step"] += Om
        torch.cuda.synchronize()
        record_event()
    steady_ms = statistics.median(replay_us) / 1e3

    def align_end(n):
        """Untimed steps until a run of n more steps ends on a routing event, so a timed run holds
        ceil(n / Omega) events (never fewer than its share)."""
        while (state["step"] + n) % Om:
            one_step(state["step"])
        torch.cuda.synchronize()

    # ---- timed region: exactly K steps, captured once in a CUDA graph and replayed once
    align_end(K)
    launches_before = state["launches"]
    g = torch.cuda.CUDAGraph()
    first = state["step"]
    with torch.cuda.graph(g, stream=stream):
        for i in range(K):
            one_step(first + i)
    timed_launches = state["launches"] - launches_before
    timed_events = sum(1 for i in range(first, first + K) if (i + 1) % Om == 0)
    torch.cuda.synchronize()
    ctr_before_timed = cache.counters()
    sampler = ClockSampler(_bus_id(torch, dev))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.start()
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.pause()
    if world > 1:
        torch.distributed.barrier()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, dev)
    cache.check(stream)
    ctr_after_timed = cache.counters()

    # ---- e2e: inputs from pinned host memory, outputs back to pinned host memory, every step
    e2e = None
    if K_e2e:
        align_end(K_e2e)
        hq = torch.empty(K_e2e, L, B, wl.h_q, D, dtype=torch.bfloat16, pin_memory=True)
        hk = torch.empty(K_e2e, L, B, wl.h_kv, D, dtype=torch.bfloat16, pin_memory=True)
        hv = torch.empty_like(hk, pin_memory=True)
        s_e = state["step"]
        hq.copy_(qs[s_e:s_e + K_e2e].cpu())
        hk.copy_(ks[s_e:s_e + K_e2e].cpu())
        hv.copy_(vs[s_e:s_e + K_e2e].cpu())
        ho = torch.empty(K_e2e, L, B, wl.h_q, D, dtype=torch.bfloat16, pin_memory=True)
        dq = torch.empty(L, B, wl.h_q, D, dtype=torch.bfloat16, device=dev)
        dk = torch.empty(L, B, wl.h_kv, D, dtype=torch.bfloat16, device=dev)
        dv = torch.empty_like(dk)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            for i in range(K_e2e):
                dq.copy_(hq[i], non_blocking=True)
                dk.copy_(hk[i], non_blocking=True)
                dv.copy_(hv[i], non_blocking=True)
                one_step(s_e + i, dq, dk, dv, outs)
                ho[i].copy_(outs, non_blocking=True)
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        g2.replay()
        f1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = max_over_ranks(f0.elapsed_time(f1), world, dev)
        in_bytes = (hq[0].numel() + hk[0].numel() + hv[0].numel()) * 2
        state["step"] = s_e + K_e2e
        cache.check(stream)
        # the same K steps as eager calls: every C-ABI call made from Python as the step runs, so the
        # host cost of the calls (ctypes, argument checks, launches) is inside the timed region too
        align_end(K_e2e)
        s_e = state["step"]
        hq.copy_(qs[s_e:s_e + K_e2e].cpu())
        hk.copy_(ks[s_e:s_e + K_e2e].cpu())
        hv.copy_(vs[s_e:s_e + K_e2e].cpu())
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for i in range(K_e2e):
            dq.copy_(hq[i], non_blocking=True)
            dk.copy_(hk[i], non_blocking=True)
            dv.copy_(hv[i], non_blocking=True)
            one_step(s_e + i, dq, dk, dv, outs)
            ho[i].copy_(outs, non_blocking=True)
        f1.record(stream)
        torch.cuda.synchronize()
        ms_eager = max_over_ranks(f0.elapsed_time(f1), world, dev)
        e2e = {"value": whole_job_rate(world, K_e2e, ms_eager), "unit": "steps/s", "h2d_bytes_per_step": in_bytes,
               "d2h_bytes_per_step": ho[0].numel() * 2, "ms_per_step": ms_eager / K_e2e,
               "routing_events": sum(1 for i in range(K_e2e) if (i + 1) % Om == 0),
               "timing": "eager: every step's C-ABI calls made from Python as the GPU runs them, each step's "
                         "inputs copied from pinned host memory and its outputs copied back, between CUDA "
                         "events on the launching stream (the host cost of the calls is inside)",
               "graph": {"value": whole_job_rate(world, K_e2e, ms_e2e), "ms_per_step": ms_e2e / K_e2e,
                         "timing": "the same calls and copies captured in one CUDA graph and replayed between "
                                   "CUDA events (the host cost of the calls is outside)"}}
        cache.check(stream)
    clocks = sampler.summary()
    sampler.close()

    peak, peak_kind = measured_peaks()
    isolated_ms = statistics.mean(kern_ms)
    bytes_per_launch = statistics.mean(kern_bytes)
    achieved = bytes_per_launch / (steady_ms / 1e3) / 1e9
    sha = kernel_sha()
    ms_step = ms_total / K
    result = {
        "metric": METRIC, "value": whole_job_rate(world, K, ms_total), "unit": "steps/s", "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "batch": B, "layers": L, "h_q": wl.h_q, "h_kv": wl.h_kv, "d_head": D,
                   "prompt_len": wl.prompt_len, "decode_steps_cached": steps_cap, "window": wl.window,
                   "bits": wl.bits, "omega": Om, "budget": f"{wl.budget_num}/{wl.budget_den}",
                   "q": f"{wl.q_num}/{wl.q_den}", "k_f": bud.k_f, "k_q": bud.k_q,
                   "parallelism": f"replicas x{world}", "rope_base": wl.rope_base,
                   "ranker": wl.ranker, "no_promotion": wl.no_promotion,
                   "l2": "inputs larger than L2: each step streams every layer's cache (%.0f MB)" %
                         (bytes_per_step / 1e6)},
        "hbm_gbs_step": bytes_per_step / (ms_step / 1e3) / 1e9,
        "hbm_frac_step": bytes_per_step / (ms_step / 1e3) / 1e9 / peak,
        "bytes_per_step": bytes_per_step,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic_from_profile(sha), "peak_kind": f"{peak_kind} copy bandwidth",
                     "kernel": "decode_kernel", "bytes_per_launch": bytes_per_launch, "avg_launch_us": steady_ms * 1e3,
                     "launches_timed": Om * L * R_roof,
                     "avg_launch_us_replays": [round(x, 3) for x in replay_us],
                     "avg_launch_us_spread": [round(min(replay_us), 3), round(max(replay_us), 3)],
                     "timing": f"median over {R_roof} replays of a CUDA graph of Omega decode-only steps (all "
                               "layers) between two CUDA events on the launching stream; consecutive launches "
                               "overlap as inside a step",
                     "isolated_launch_us": isolated_ms * 1e3,
                     "isolated_timing": f"{len(kern_ms)} launches, each alone between two events",
                     "kernel_source_sha": sha,
                     "vs_8tbs": achieved / 8000.0},
        "gpu_launches": timed_launches,
        "routing_events_timed": timed_events,
        "transitions_per_event": {
            "events": len(per_event), "units": L * B,
            "mean": {k: statistics.mean(e[k] for e in per_event) for k in per_event[0]},
            "max": {k: max(e[k] for e in per_event) for k in per_event[0]},
            "timed_events": timed_events,
            "timed_mean": {k: (ctr_after_timed[k] - ctr_before_timed[k]) / max(1, timed_events)
                           for k in ctr_after_timed},
            "note": "tier transitions per routing event over all (layer, sequence) units: mean/max from counter "
                    "deltas of each untimed event, timed_mean over the events of the timed region (QEvict "
                    "App. K Table 18's promotion counts)"},
        "clocks": clocks,
        "prefill_s": round(t_pre, 2), "prefill_scores": prefill_scores,
    }
    if e2e:
        result["e2e"] = e2e
    if args.diag:
        del cache
        torch.cuda.empty_cache()
        result["diagnostics"] = run_diag(wl, dev, stream, args.diag)
    return result


def run_diag(wl, dev, stream, n_events):
    """Routing diagnostics (QEvict App. I) of the policy against a FullKV cache fed the same inputs:
    n_events routing events, each timed through qevict_diag_route, then one more event of plain
    qevict_route calls on both caches for the cost without diagnostics."""
    import torch
    from recoverable_quantized_kv_gb300 import binding, synth
    Om, L, B = wl.omega, wl.n_layers, wl.batch
    steps = (n_events + 1) * Om
    max_len = wl.prompt_len + steps
    pol = binding.Cache(binding.make_config(wl, max_len=max_len), device=dev)
    fwl = wl.replace(budget_num=1000, q_num=0)
    full = binding.Cache(binding.make_config(fwl, max_len=max_len), device=dev)
    for c in (pol, full):
        if wl.rope_base > 0:
            c.set_rope_table(torch.from_numpy(synth.rope_table(max_len, wl.rope_base)).to(dev))
    for layer in range(L):
        ins = [synth.prompt_inputs(wl, b, layer, device=dev) for b in range(B)]
        q = torch.stack([x["q"] for x in ins])
        k = torch.stack([x["k"] for x in ins])
        v = torch.stack([x["v"] for x in ins])
        pol.prefill_route(layer, k, v, s0=None, q_prompt=q, stream=stream)
        full.prefill_route(layer, k, v, s0=None, q_prompt=q, stream=stream)
        del ins, q, k, v
    diag = binding.Diagnostics(pol, full, stream=stream)
    dec = [[synth.decode_inputs(wl, b, layer, steps=steps, device=dev) for b in range(B)] for layer in range(L)]
    out = torch.empty(B, wl.h_q, D, dtype=torch.bfloat16, device=dev)
    diag_ms, plain_ms = [], []
    for s in range(steps):
        for layer in range(L):
            q = torch.stack([d["q"][s] for d in dec[layer]])
            k = torch.stack([d["k"][s] for d in dec[layer]])
            v = torch.stack([d["v"][s] for d in dec[layer]])
            pol.decode_step(layer, q, k, v, out, stream)
            full.decode_step(layer, q, k, v, out, stream)
        if (s + 1) % Om == 0:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            if s + 1 < steps:
                diag.route(stream)
            else:
                pol.route(stream)
                full.route(stream)
            e1.record(stream)
            torch.cuda.synchronize()
            (diag_ms if s + 1 < steps else plain_ms).append(e0.elapsed_time(e1))
    rep = diag.report(stream)
    lag = rep["lag"]

    def p(a, b, d):
        n = lag[d - 1, a].sum()
        return float(lag[d - 1, a, b] / n) if n else None
    return {"events": rep["events"], "fmm_h32": rep["fmm"], "fmm_terms": rep["fmm_terms"], "churn": rep["churn"],
            "qsa": rep["qsa"], "r_q": rep["r_q"], "tier_mass_full_quant_evict_local": rep["tier_mass"].tolist(),
            "lir3_policy": [rep["lir_eligible"], rep["lir_rescued"]],
            "lir3_fullkv_topk": [rep["lir_fullkv_eligible"], rep["lir_fullkv_rescued"]],
            "p01": [p(0, 1, 1), p(0, 1, 8)], "p10": [p(1, 0, 1), p(1, 0, 8)],
            "route_ms_per_event_with_diag": statistics.mean(diag_ms), "route_ms_plain_pair": plain_ms[0],
            "note": "policy and FullKV caches decode the same synthetic inputs; route_ms covers both caches' "
                    "routing events (all layers); p01/p10 at Delta = 1 and 8"}


def _bus_id(torch, dev):
    p = torch.cuda.get_device_properties(dev)
    return "%08x:%02x:%02x.0" % (getattr(p, "pci_domain_id", 0), p.pci_bus_id, p.pci_device_id)


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: every (layer, sequence) unit of the workload decoded in
    lockstep on the host cores (one process per core, one BLAS thread each), W warm-up steps then K
    timed steps, each timed step one decode step of every unit with the routing event every Omega
    steps.  Rank 0 only."""
    if rank != 0:
        return None
    from recoverable_quantized_kv_gb300 import synth
    wl = synth.workload(args.workload)
    cores = len(os.sched_getaffinity(0))
    U = wl.n_layers * wl.batch
    n_proc = min(cores, U)
    t_start = time.time()
    t, _ = oracle_steps(args.workload, U, n_proc, args.steps, warmup=args.warmup)
    value = args.steps / t
    sample = (f"oracle on all {U} (layer, sequence) units of {wl.name} per step, {n_proc} processes x 1 BLAS "
              f"thread, routing every {wl.omega} steps; prompt scores seeded random (prefill excluded)")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.batch, "layers": wl.n_layers, "prompt_len": wl.prompt_len},
            "cpu_baseline": {"value": value, "unit": "steps/s", "kind": "oracle", "cores": n_proc, "cpu": _cpu_model(),
                             "sample": sample},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.time() - t_start, 1)}


def run_sweep(args, rank, world):
    """Config 4's grid (QEvict §5 "Ablations", App. G.2-G.3: budget and quantised fraction) on the
    given workload: each point a full run_gpu measurement with a short timed region."""
    import copy
    import torch
    pts = []
    for b in (10, 20, 40):
        for q in (50, 70, 90):
            a = copy.copy(args)
            a.budget, a.q, a.no_e2e = f"{b}/100", f"{q}/100", True
            r = run_gpu(a, rank, world)
            rf = r["roofline"]
            pts.append({"budget": b / 100, "q": q / 100, "k_f": r["config"]["k_f"], "k_q": r["config"]["k_q"],
                        "steps_per_s": r["value"], "ms_per_step": r["ms_per_step"],
                        "avg_launch_us": rf["avg_launch_us"], "bytes_per_launch": rf["bytes_per_launch"],
                        "achieved_gbs": rf["achieved"], "frac": rf["frac"], "hbm_frac_step": r["hbm_frac_step"],
                        "clocks": r["clocks"]})
            torch.cuda.empty_cache()
    return {"metric": METRIC, "sweep": pts, "workload": args.workload, "layers": args.layers,
            "format": "INT4/W=64" if args.int4 else "INT2/W=32", "steps": args.steps, "warmup": args.warmup,
            "note": "each point: decode steps/s over the timed steps (routing included) and the decode "
                    "kernel's roofline, as in the main bench line"}


def main():
    args = parse_args()
    if args.oracle_child:
        run_oracle_child(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        r = run_reference(args, rank, world)
        if r is not None:
            print(json.dumps(r))
        return
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl")
    if args.sweep:
        res = run_sweep(args, rank, world)
        if rank == 0:
            print(json.dumps(res))
        return
    res = run_gpu(args, rank, world)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
