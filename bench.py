#!/usr/bin/env python
"""Benchmark: compressed-KV decode attention on one GB300 (and N replicas).

One step = the whole hot path once on the Llama-2-7B-shaped decode workload
(batch 16, 32 heads, head_dim 128, context 8192, bf16, KQV at a 4-bit
budget): append-quantise one new K/V token per sequence into slot 8191, then
decode attention of one query per head over the 8192 compressed tokens
(query prep, decode, combine). `value` is the step's algorithmic bytes
(packed records + norms + signs read, new records written, q, output) per
second of device time; `append_quantize` reports the bulk append-quantise
throughput of refilling the whole cache; `paged` the same step on a paged
cache; `configs` (N = 1) the decode kernel, the decode call and the bulk
append on every other workload (single head; the scheme x budget sweep; GQA
over 131072 tokens; the four KIVI layouts); `cpu_baseline` the CPU oracle's
decode and quantise on one thread and on one single-threaded process per
core. Inputs are synthetic, drawn on the device from a seeded generator; the
587 MB cache is larger than the 129 MB L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica (the path has no
exchange step); rank 0 prints one JSON line. `--impl reference` times the CPU
oracle as the reference arm on the host's cores.
"""

import argparse
import json
import math
import os
import signal
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "compressed-KV decode attention GB/s and % of HBM peak; append-quantise tokens/s"
CAP = 8192
# kernels of one decode step (tq_decode_step): the persistent decode kernel, which also
# appends the step's keys and values and prepares the queries, and the combine
LAUNCHES_PER_STEP = 2
# DRAM bytes (read + written) of one launch of the decode-step kernel on this workload: the
# median over three launches (after three warm-up steps) of one ncu capture of this bench
# restricted to that kernel (dram__bytes_read.sum + dram__bytes_write.sum, context 8192;
# profiles/step_launches_kqv4_b16_h32_n8192.md); None whenever the kernel has changed since
# that capture, until it is captured again
DECODE_TRAFFIC_BYTES = 588_597_504


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class NvmlClocks:
    """SM clock, power and clock-event reasons of one GPU read through NVML (the driver's
    libnvidia-ml, read-only queries) every 10 ms on a host thread, each sample with its host
    time, so that the samples taken inside the timed loop can be picked out."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, uuid, index):
        import ctypes
        self.ct = ctypes
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.L, self.h = L, ctypes.c_void_p()
        found = uuid is not None and L.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(self.h)) == 0
        if not found and L.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")
        self.reasons_fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(L, "nvmlDeviceGetCurrentClocksThrottleReasons")
        v = ctypes.c_uint()
        self.max_mhz = float(v.value) if L.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(v)) == 0 else None
        self.samples, self.stop_flag, self.thread = [], False, None

    def _one(self):
        ct, L = self.ct, self.L
        clk, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if L.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) != 0:
            return None
        power = mw.value / 1e3 if L.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw)) == 0 else float("nan")
        reasons = rs.value if self.reasons_fn(self.h, ct.byref(rs)) == 0 else 0
        return (time.perf_counter(), float(clk.value), power, reasons)

    def start(self):
        import threading

        def loop():
            while not self.stop_flag:
                smp = self._one()
                if smp is not None:
                    self.samples.append(smp)
                time.sleep(0.01)
        self.thread = threading.Thread(target=loop, daemon=True)
        self.thread.start()

    def stop(self, window=None):
        self.stop_flag = True
        self.thread.join(timeout=5)
        rows = self.samples
        inside = [r for r in rows if window is None or window[0] <= r[0] <= window[1]]
        scope = "timed loop" if inside and window is not None else "whole run"
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": "nvml"}
        sm = sorted(r[1] for r in use)
        reasons = sorted({name for r in use for bit, name in self.REASONS.items() if r[3] & bit})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(use), "scope": scope, "power_w_max": max(r[2] for r in use), "source": "nvml"}


def clock_sampler(device_index):
    """NVML where the driver's library loads, else nvidia-smi."""
    try:
        import torch
        props = torch.cuda.get_device_properties(device_index)
        uuid = str(getattr(props, "uuid", "")) or None
        return NvmlClocks(uuid, device_index)
    except Exception:
        return Clocks(device_index)


class Clocks:
    """nvidia-smi sampled every 100 ms from the warm-up through the timed loops."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, window=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        busy = [r for r in rows if num(r[4]) > 0] or rows
        sm = sorted(num(r[1]) for r in busy)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i in range(4) if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": num(rows[0][2]), "reasons": reasons,
                "samples": len(busy), "power_w_max": max(num(r[3]) for r in busy)}


class OracleDecode:
    """The CPU oracle's decode attention on one (batch, head) unit of the workload.

    Setup (untimed): the oracle encodes one head's K/V (8192 tokens) into the
    stored-record format. Timed: unpack the records, reconstruct K and V in
    fp64, dense softmax attention of one query."""

    def __init__(self, N, bits, seed, data_seed=None):
        import numpy as np
        from oracle import turboquant as otq
        self.otq = otq
        self.params = otq.make_params(128, bits, "KQV", seed)
        self.rk, self.rv = self.params.roles()
        g = np.random.default_rng(seed if data_seed is None else data_seed)
        K = g.standard_normal((N, 128)) * np.exp(g.standard_normal(128))[None, :]
        V = g.standard_normal((N, 128))
        self.ek = otq.encode(K, self.rk, self.params)
        self.ev = otq.encode(V, self.rv, self.params)
        self.kc = otq.pack_codes(self.ek.idx, self.rk.bits)
        self.vc, self.vs = otq.pack_codes(self.ev.idx, self.rv.bits), otq.pack_signs(self.ev.signs)
        self.q = g.standard_normal(128)

    def one_head(self):
        from oracle import attention as oatt
        otq = self.otq
        ekk = otq.encoded_from_storage(self.rk, self.ek.norm, self.kc, 128)
        evv = otq.encoded_from_storage(self.rv, self.ev.norm, self.vc, 128, self.vs, self.ev.rnorm)
        return oatt.attend(self.q, otq.decode(ekk, self.params), otq.decode(evv, self.params))

    def run(self, target_s):
        """Decode heads until target_s seconds have passed (at least one). Returns (heads, seconds)."""
        heads, t0 = 0, time.perf_counter()
        while True:
            self.one_head()
            heads += 1
            el = time.perf_counter() - t0
            if el >= target_s:
                return heads, el


def cpu_model() -> str:
    """The host CPU's model string (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine() or "unknown"


_ONE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def _oracle_worker(job):
    """One single-threaded oracle process (spawned; BLAS limited to one thread by the
    environment it inherits): set up one unit of the workload untimed, then repeat the
    timed operation for `seconds`. Returns (units done, seconds)."""
    kind, seconds, seed = job
    import numpy as np
    if kind == "decode":
        od = OracleDecode(CAP, 4, 42, data_seed=seed)
        units, t0 = 0, time.perf_counter()
        while True:
            od.one_head()
            units += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return units, el
    from oracle import turboquant as otq
    params = otq.make_params(128, 4, "KQV", 42)
    rk, rv = params.roles()
    K, V = config2_like_vectors(QUANTISE_BATCH, seed)
    units, t0 = 0, time.perf_counter()
    while True:
        otq.encode(K, rk, params)
        otq.encode(V, rv, params)
        units += QUANTISE_BATCH
        el = time.perf_counter() - t0
        if el >= seconds:
            return units, el


QUANTISE_BATCH = 2048  # token-heads (one K and one V vector each) per timed oracle encode


def config2_like_vectors(n, seed):
    """n keys shaped like the decode workload's (N(0, 1) times per-channel log-normal(0, 1)
    scales with four x10 outlier channels) and n N(0, 1) values, rounded to bf16 values, as
    float64 for the oracle."""
    import numpy as np
    g = np.random.default_rng(seed)
    scale = np.exp(g.standard_normal(128))
    scale[g.choice(128, 4, replace=False)] *= 10.0
    K = g.standard_normal((n, 128)) * scale[None, :]
    V = g.standard_normal((n, 128))

    def bf16(x):
        u = x.astype(np.float32).view(np.uint32)
        u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
        return u.view(np.float32).astype(np.float64)
    return bf16(K), bf16(V)


def oracle_rates(kind: str, procs: int, seconds: float):
    """Units per second of the oracle's `kind` ("decode": (batch, head) units of 8192 tokens;
    "quantise": token-heads) over `procs` single-threaded spawned processes, each working
    on its own unit of the workload for `seconds`."""
    import multiprocessing as mp
    saved = {k: os.environ.get(k) for k in _ONE_THREAD_ENV}
    for k in _ONE_THREAD_ENV:
        os.environ[k] = "1"
    try:
        with mp.get_context("spawn").Pool(procs) as pool:
            res = pool.map(_oracle_worker, [(kind, seconds, 4242 + i) for i in range(procs)])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    units = sum(u for u, _ in res)
    rate = sum(u / el for u, el in res)
    return rate, units, max(el for _, el in res)


def cpu_baseline(seconds_each: float = 3.0):
    """The oracle timed on this host: decode attention and quantise, on one thread and on
    every core (one single-threaded process per core, each on its own unit)."""
    cores = os.cpu_count() or 1
    rec = 140
    out = {"kind": "oracle", "cores": cores, "cpu_model": cpu_model(), "unit": "GB/s"}
    for kind in ("decode", "quantise"):
        out[kind] = {}
        for label, procs in (("1_thread", 1), ("all_cores", cores)):
            rate, units, el = oracle_rates(kind, procs, seconds_each)
            if kind == "decode":
                row = {"heads_per_s": rate, "token_heads_per_s": rate * CAP,
                       "GB_per_s": rate * CAP * rec / 1e9, "units": units}
            else:
                row = {"token_heads_per_s": rate,
                       "GB_per_s": rate * (2 * 128 * 2 + rec) / 1e9, "units": units}
            row.update({"threads": procs, "seconds": el})
            out[kind][label] = row
    out["value"] = out["decode"]["all_cores"]["GB_per_s"]
    out["threads"] = cores
    out["sample"] = (f"decode: (batch, head) units of the decode workload (8192 tokens, KQV n=4) decoded "
                     f"from their records for {seconds_each:.0f} s per process; quantise: batches of "
                     f"{QUANTISE_BATCH} K and V vectors shaped like the workload's; each on 1 process and "
                     f"on {cores} single-threaded processes (one per core)")
    return out


_WORKER_OD = None


def _ref_init(seed):
    global _WORKER_OD
    _WORKER_OD = OracleDecode(CAP, 4, 42, data_seed=seed)


def _ref_decode_one(_):
    _WORKER_OD.one_head()
    return 1


def run_reference(args, rank):
    """The oracle as the reference arm, on this host's cores (rank 0 only): one
    single-threaded process per core, each holding one (batch, head) unit of the decode
    workload in the stored-record format (set up untimed). A step decodes one unit in
    every process at once; K steps are timed after W warm-up steps."""
    if rank != 0:
        return
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    rec = 140  # bytes per token-head, KQV n=4
    saved = {k: os.environ.get(k) for k in _ONE_THREAD_ENV}
    for k in _ONE_THREAD_ENV:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(cores, initializer=_ref_init, initargs=(0,)) as pool:
            for _ in range(args.warmup):
                pool.map(_ref_decode_one, range(cores), chunksize=1)
            t0 = time.perf_counter()
            heads = 0
            for _ in range(args.steps):
                heads += sum(pool.map(_ref_decode_one, range(cores), chunksize=1))
            total_s = time.perf_counter() - t0
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    gbs = heads * CAP * rec / total_s / 1e9
    sample = (f"{heads} (batch, head) decode units of the workload ({CAP} tokens each, from their stored "
              f"records), {cores} per step, one per single-threaded process")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "threads": cores,
                             "cpu_model": cpu_model(), "kind": "oracle", "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x (the job's time is its slowest replica's)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job throughput of `world` replicas: all ranks' units over the slowest rank's time."""
    return units_per_rank * world / seconds_max


def workload_config():
    return {"workload": "Llama-2-7B-shaped decode step: append 1 token/sequence + decode attention, "
                        "B16 H32 d128 context 8192 bf16, KQV n=4",
            "batch": 16, "heads_q": 32, "heads_kv": 32, "head_dim": 128, "context": CAP, "scheme": "KQV",
            "bits": 4, "input_dtype": "bf16", "l2": "inputs larger than L2 (587 MB compressed cache > 129 MB)",
            "parallelism": "replicas"}


def run_workload_decode(args, dev):
    """Decode calls on one of the other workloads, for profiler captures: the GQA long context
    (32 query heads on 8 KV heads, context 131072, KQV n=3; 113 MB of records) or the KIVI
    layout study (B8 H40 context 4096, per-channel keys and per-token values; 143 MB)."""
    import torch
    from quantised_kv_cache_gb300 import tq
    from quantised_kv_cache_gb300 import workloads as wl
    wid = 4 if args.case == "gqa-decode" else 5
    w = wl.WORKLOADS[wid]
    B, Hq, H, N = w.batch, w.heads_q, w.heads_kv, w.seq
    if wid == 5:
        ctx = tq.Context(128, 2, "KIVI", 42, k_per_channel=True, v_per_token=True)
    else:
        ctx = tq.Context(128, w.bits, w.scheme, 42)
    q, k, v = wl.generate(w, dev)
    cache = tq.Cache(ctx, B, H, N, device=dev)
    tq.tq_append_quantize(ctx.handle, cache, k, v, torch.zeros((B,), dtype=torch.int32, device=dev))
    del k, v
    lens = torch.full((B,), N, dtype=torch.int32, device=dev)
    ws = torch.empty(tq.tq_workspace_size(ctx.handle, B, Hq, H, N, w.splits), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    for _ in range(args.warmup + args.steps):
        tq.tq_decode_attention(ctx.handle, cache, q, lens, N, w.splits, ws, out)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    print(json.dumps({"case": args.case, "ok": True}), flush=True)


def run_workload_append(args, dev):
    """Bulk appends on one of the other workloads, for profiler captures: the KIVI layout study
    (B8 H40 context 4096, bf16, per-channel keys and per-token values) or the scheme sweep's
    unrotated KV scheme at 4 bits (B4 H8 context 16384, fp32). Each step re-appends the whole
    context from sequence length 0."""
    import torch
    from quantised_kv_cache_gb300 import tq
    from quantised_kv_cache_gb300 import workloads as wl
    wid = 5 if args.case == "kivi-append" else 3
    w = wl.WORKLOADS[wid]
    if wid == 5:
        ctx = tq.Context(128, 2, "KIVI", 42, k_per_channel=True, v_per_token=True)
    else:
        ctx = tq.Context(128, 4, "KV", 42)
    _, k, v = wl.generate(w, dev)
    cache = tq.Cache(ctx, w.batch, w.heads_kv, w.seq, device=dev)
    zeros = torch.zeros((w.batch,), dtype=torch.int32, device=dev)
    for _ in range(args.warmup + args.steps):
        tq.tq_append_quantize(ctx.handle, cache, k, v, zeros)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    print(json.dumps({"case": args.case, "ok": True}), flush=True)


def run_small_case(args, dev):
    """A smaller instance of the Llama-2-7B-shaped workload for profiler captures:
    B16 H32 context 4096 (294 MB of compressed records, 537 MB of bf16 K/V)."""
    import torch
    from quantised_kv_cache_gb300 import tq
    from quantised_kv_cache_gb300 import workloads as wl
    if args.case in ("gqa-decode", "kivi-decode"):
        run_workload_decode(args, dev)
        return
    if args.case in ("kivi-append", "kv-append"):
        run_workload_append(args, dev)
        return
    w = wl.WORKLOADS[2]
    N = 4096
    B, H = w.batch, w.heads_kv
    ctx = tq.Context(128, w.bits, "KQV", 42)
    cache = tq.Cache(ctx, B, H, N, device=dev)
    q, k, v = wl.generate(w, dev, seq=N)
    zeros = torch.zeros((B,), dtype=torch.int32, device=dev)
    tq.tq_append_quantize(ctx.handle, cache, k, v, zeros)
    lens = torch.full((B,), N - 1, dtype=torch.int32, device=dev)
    kn, vn = k[:, :, -1:].contiguous(), v[:, :, -1:].contiguous()
    for _ in range(args.warmup + args.steps):
        if args.case == "append-small":
            tq.tq_append_quantize(ctx.handle, cache, k, v, zeros)
        else:  # decode steps re-appending the last token
            tq.tq_decode_step(ctx.handle, cache, q, kn, vn, lens, N)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    print(json.dumps({"case": args.case, "ok": True}), flush=True)


CONFIG_CASES = ([(1, "KQV", 4, None)]
                + [(3, sch, n, None) for sch in ("KV", "KQV", "QKQV") for n in (2, 3, 4)]
                + [(4, "KQV", 3, None)]
                + [(5, "KIVI", 2, lay) for lay in ((True, True), (False, False), (False, True), (True, False))])


def measure_configs(dev, cases=CONFIG_CASES):
    """Decode and bulk append-quantise throughput on every workload (one row per case):
    config 1 (single head), config 3 (three schemes x three budgets), config 4 (GQA 32q/8kv,
    N=131072, KQV n=3, 64 chunks), config 5 (KIVI, four layouts). Caches smaller than 3x L2
    are replicated and rotated so that every decode call reads HBM. Decode times are CUDA
    events around the library's decode kernel (its profile events, on the call's stream),
    around the whole call (query prep + decode + combine, issued call by call from Python),
    and around a CUDA-graph replay of the same calls (the device time of the whole call);
    append times are events around a bulk append of the whole context into one cache."""
    import torch
    from quantised_kv_cache_gb300 import tq
    from quantised_kv_cache_gb300 import workloads as wl
    hbm_peak, peak_kind = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    rows = []
    for wid, scheme, n, kivi in cases:
        w = wl.WORKLOADS[wid]
        B, Hq, H, N = w.batch, w.heads_q, w.heads_kv, w.seq
        if kivi is not None:
            ctx = tq.Context(128, n, scheme, 42, k_per_channel=kivi[0], v_per_token=kivi[1])
        else:
            ctx = tq.Context(128, n, scheme, 42)
        q, k, v = wl.generate(w, dev)
        one = tq.Cache(ctx, B, H, N, device=dev)
        rec = one.record_bytes if scheme != "KIVI" else 96
        bytes_call = B * H * N * rec if scheme != "KIVI" else B * H * ((N - 128) * 96 + 128 * 512)
        reps = max(1, min(16, int(math.ceil(3 * l2 / max(bytes_call, 1)))))
        caches = [one] + [tq.Cache(ctx, B, H, N, device=dev) for _ in range(reps - 1)]
        zeros = torch.zeros((B,), dtype=torch.int32, device=dev)
        for c in caches:
            tq.tq_append_quantize(ctx.handle, c, k, v, zeros)
        # bulk append of the whole context (the first fill above was its warm-up)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        arep = 3
        torch.cuda.synchronize()
        a0.record()
        for _ in range(arep):
            tq.tq_append_quantize(ctx.handle, one, k, v, zeros)
        a1.record()
        torch.cuda.synchronize()
        append_ms = a0.elapsed_time(a1) / arep
        in_bytes = B * H * N * 128 * k.element_size() * 2
        append_bytes = in_bytes + (B * H * N * rec if scheme != "KIVI" else bytes_call)
        lens = torch.full((B,), N, dtype=torch.int32, device=dev)
        splits = w.splits
        ws = torch.empty(tq.tq_workspace_size(ctx.handle, B, Hq, H, N, splits), dtype=torch.uint8, device=dev)
        out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
        iters = max(20, 8 * reps)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for i in range(3 * reps):
            tq.tq_decode_attention(ctx.handle, caches[i % reps], q, lens, N, splits, ws, out)
        torch.cuda.synchronize()
        for a_, b_ in evs:
            a_.record()
            b_.record()
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        for i in range(iters):
            tq.tq_set_profile_events(ctx.handle, evs[i][0], evs[i][1])
            tq.tq_decode_attention(ctx.handle, caches[i % reps], q, lens, N, splits, ws, out)
        c1.record()
        torch.cuda.synchronize()
        tq.tq_set_profile_events(ctx.handle)
        assert tq.tq_get_device_error(ctx.handle) == 0
        # the same calls captured once as a CUDA graph and replayed: the device time of the
        # whole call without the host's launch gaps between calls
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for i in range(iters):
                    tq.tq_decode_attention(ctx.handle, caches[i % reps], q, lens, N, splits, ws, out,
                                           stream=torch.cuda.current_stream())
        graph.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record()
        graph.replay()
        g1.record()
        torch.cuda.synchronize()
        assert tq.tq_get_device_error(ctx.handle) == 0
        del graph
        ms_kernel = sum(a_.elapsed_time(b_) for a_, b_ in evs) / iters
        ms_call = c0.elapsed_time(c1) / iters
        ms_graph = g0.elapsed_time(g1) / iters
        gbs_k, gbs_c, gbs_g = bytes_call / ms_kernel / 1e6, bytes_call / ms_call / 1e6, bytes_call / ms_graph / 1e6
        append_gbs = append_bytes / append_ms / 1e6
        rows.append({"config": wid, "scheme": scheme, "bits": n,
                     "kivi_layout": None if kivi is None else {"k_per_channel": kivi[0], "v_per_token": kivi[1]},
                     "shape": {"batch": B, "heads_q": Hq, "heads_kv": H, "context": N,
                               "input_dtype": str(k.dtype).replace("torch.", "")},
                     "decode": {"bytes_per_call": bytes_call, "replicas": reps, "ms_kernel": ms_kernel,
                                "GB_per_s_kernel": gbs_k, "frac_kernel": gbs_k / hbm_peak, "ms_call": ms_call,
                                "GB_per_s_call": gbs_c, "frac_call": gbs_c / hbm_peak, "ms_graph": ms_graph,
                                "GB_per_s_graph": gbs_g, "frac_graph": gbs_g / hbm_peak},
                     "append": {"ms": append_ms, "tokens_per_s": B * N / (append_ms / 1e3),
                                "token_heads_per_s": B * H * N / (append_ms / 1e3), "bytes": append_bytes,
                                "GB_per_s": append_gbs, "frac": append_gbs / hbm_peak},
                     "peak": hbm_peak, "peak_kind": peak_kind})
        del caches, one, q, k, v, ws, out
        ctx.close()
        torch.cuda.empty_cache()
    return rows


def run_configs(args, dev):
    for row in measure_configs(dev):
        print(json.dumps(dict(case="configs", **row)), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload table of the N=1 line")
    ap.add_argument("--case", choices=["step", "decode-small", "append-small", "gqa-decode", "kivi-decode",
                                       "kivi-append", "kv-append", "configs"],
                    default="step",
                    help="step: the benchmark; *-small: one kernel family on B16 H32 N4096 (294 MB of records, "
                         "above L2) for profiler captures; gqa-decode / kivi-decode: decode calls of the GQA "
                         "and KIVI workloads, kivi-append / kv-append: bulk appends of the KIVI workload and "
                         "of the scheme sweep's KV scheme at 4 bits, for profiler captures")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import numpy as np
    import torch
    from quantised_kv_cache_gb300 import build
    from quantised_kv_cache_gb300 import tq
    from quantised_kv_cache_gb300 import workloads as wl

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or not os.path.exists(tq.LIB_PATH):
        build.build()
    if dist is not None:
        dist.barrier()

    if args.case == "configs":
        run_configs(args, dev)
        return
    if args.case != "step":
        run_small_case(args, dev)
        return

    w = wl.WORKLOADS[2]
    B, H, d = w.batch, w.heads_kv, w.d
    ctx = tq.Context(d, w.bits, "KQV", 42)
    cache = tq.Cache(ctx, B, H, CAP, device=dev)
    rec = cache.record_bytes  # 140 B per token-head
    q0, k_all, v_all = wl.generate(w, dev, seed=1002 + rank)
    zeros = torch.zeros((B,), dtype=torch.int32, device=dev)

    # ---------------- bulk append-quantise: refill the whole cache
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tq.tq_append_quantize(ctx.handle, cache, k_all, v_all, zeros)
    torch.cuda.synchronize()
    reps = 5
    e0.record()
    for _ in range(reps):
        tq.tq_append_quantize(ctx.handle, cache, k_all, v_all, zeros)
    e1.record()
    torch.cuda.synchronize()
    append_ms = e0.elapsed_time(e1) / reps
    assert tq.tq_get_device_error(ctx.handle) == 0
    token_heads = B * H * CAP
    append_bytes = token_heads * (2 * d * 2 + rec)
    hbm_peak, peak_kind = peaks()

    # ---------------- decode step
    pool = [wl.step_token(w, s, dev, data_seed=1002 + rank) for s in range(8)]
    lens_append = torch.full((B,), CAP - 1, dtype=torch.int32, device=dev)
    lens_decode = torch.full((B,), CAP, dtype=torch.int32, device=dev)
    ws = torch.empty(tq.tq_workspace_size(ctx.handle, B, w.heads_q, H, CAP, 0), dtype=torch.uint8, device=dev)
    out = torch.empty((B, w.heads_q, d), dtype=torch.float32, device=dev)

    def step(i):
        q, kn, vn = pool[i % len(pool)]
        tq.tq_decode_step(ctx.handle, cache, q, kn, vn, lens_append, CAP, ws, out)

    def step_two_calls(i):  # the same step as an append call and a decode call (context only)
        q, kn, vn = pool[i % len(pool)]
        tq.tq_append_quantize(ctx.handle, cache, kn, vn, lens_append)
        tq.tq_decode_attention(ctx.handle, cache, q, lens_decode, CAP, 0, ws, out)

    step_bytes = (B * H * CAP * rec            # compressed cache read by the decode kernel
                  + B * H * (2 * d * 2 + rec)  # new K/V token read, new records written
                  + B * w.heads_q * d * 2      # q (bf16)
                  + B * w.heads_q * d * 4)     # output (fp32)
    # the decode-step kernel: the cache, the queries, the new tokens read and their records
    # written, the output (written by the combine, counted here as in the step)
    decode_kernel_bytes = B * H * CAP * rec + B * w.heads_q * d * (2 + 4) + B * H * (2 * d * 2 + rec)

    clocks = clock_sampler(local)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    K = args.steps
    # the steps as a user runs them: the library's kernels follow one another with
    # programmatic overlap, so no event sits between them here
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    host0 = time.perf_counter()
    t_start.record()
    for i in range(K):
        step(i)
    t_stop.record()
    torch.cuda.synchronize()
    timed_window = (host0, time.perf_counter())
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_stop), dist, dev)
    ms_step = elapsed_ms / K
    value = job_throughput(step_bytes * K, world, elapsed_ms / 1e3) / 1e9
    # the same K steps again with events around every decode kernel launch (on the
    # library's stream) for the kernel's own duration
    dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in dec_ev:  # torch creates the CUDA event on first record; the library needs the handle
        a.record()
        b.record()
    torch.cuda.synchronize()
    for i in range(K):
        tq.tq_set_profile_events(ctx.handle, dec_ev[i][0], dec_ev[i][1])
        step(i)
    torch.cuda.synchronize()
    tq.tq_set_profile_events(ctx.handle)
    dec_ms = float(np.mean([a.elapsed_time(b) for a, b in dec_ev]))
    assert tq.tq_get_device_error(ctx.handle) == 0
    for i in range(args.warmup):
        step_two_calls(i)
    t_start.record()
    for i in range(K):
        step_two_calls(i)
    t_stop.record()
    torch.cuda.synchronize()
    two_calls_ms = t_start.elapsed_time(t_stop) / K
    assert tq.tq_get_device_error(ctx.handle) == 0

    # ---------------- the same step on a paged cache: every sequence-head's blocks scattered
    # over a pool by a shuffled block table (the records copied there untimed)
    nblk = cache.blocks_per_seq
    perm = torch.randperm(B * H * nblk, generator=torch.Generator().manual_seed(77)).to(torch.int32)
    paged = tq.PagedCache(ctx, B, H, CAP, B * H * nblk, perm.view(B, H, nblk).contiguous(), device=dev)
    paged.tensors["records"].view(B * H * nblk, -1)[perm.long().to(dev)] = cache.blocks().view(B * H * nblk, -1)

    def step_paged(i):
        q, kn, vn = pool[i % len(pool)]
        tq.tq_decode_step(ctx.handle, paged, q, kn, vn, lens_append, CAP, ws, out)

    for i in range(args.warmup):
        step_paged(i)
    torch.cuda.synchronize()
    t_start.record()
    for i in range(K):
        step_paged(i)
    t_stop.record()
    torch.cuda.synchronize()
    paged_ms = t_start.elapsed_time(t_stop) / K
    assert tq.tq_get_device_error(ctx.handle) == 0
    del paged

    # ---------------- end to end through the ABI with host buffers
    pin = [(q.cpu().pin_memory(), kn.cpu().pin_memory(), vn.cpu().pin_memory()) for q, kn, vn in pool]
    # two sets of device inputs / outputs: step i + 1's inputs are copied in on a copy stream
    # while step i computes, and step i's output is copied out while step i + 1 computes
    # (every step still moves its own inputs in and its own output out)
    dev_in = [tuple(torch.empty_like(x) for x in pool[0]) for _ in range(2)]
    dev_out = [torch.empty_like(out) for _ in range(2)]
    host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in dev_in[0])
    d2h = host_out[0].numel() * host_out[0].element_size()
    compute = torch.cuda.current_stream()
    copy_s = torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    for e in in_free + out_free:
        e.record(compute)

    def stage_in(i):
        j = i % 2
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(in_free[j])
            for dst, src in zip(dev_in[j], pin[i % len(pin)]):
                dst.copy_(src, non_blocking=True)
            in_ready[j].record(copy_s)

    def e2e_step(i):
        j = i % 2
        dq, dk, dv = dev_in[j]
        compute.wait_event(in_ready[j])
        compute.wait_event(out_free[j])
        tq.tq_decode_step(ctx.handle, cache, dq, dk, dv, lens_append, CAP, ws, dev_out[j])
        in_free[j].record(compute)
        out_ready[j].record(compute)
        stage_in(i + 1)
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(out_ready[j])
            host_out[j].copy_(dev_out[j], non_blocking=True)
            out_free[j].record(copy_s)

    stage_in(0)
    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    stage_in(0)  # the first step's inputs, inside the timed region
    for i in range(K):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist, dev)
    clk = clocks.stop(timed_window)
    e2e_value = job_throughput(step_bytes * K, world, e2e_s) / 1e9

    line = None
    if rank == 0:
        achieved = decode_kernel_bytes / (dec_ms / 1e3) / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": workload_config(),
            "pct_of_hbm_peak": 100.0 * (value / world) / hbm_peak,
            "roofline": {"bound": "hbm",
                         "kernel": "decode_persist_kernel<4,3,0,1,1> (persistent decode attention with the "
                                   "step's append and query preparation fused in)",
                         "achieved": achieved, "peak": hbm_peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": DECODE_TRAFFIC_BYTES, "ms_per_launch": dec_ms,
                         "bytes_per_launch": decode_kernel_bytes},
            "append_quantize": {"tokens_per_s": B * CAP / (append_ms / 1e3),
                                "token_heads_per_s": token_heads / (append_ms / 1e3),
                                "GB_per_s": append_bytes / (append_ms / 1e3) / 1e9,
                                "frac": append_bytes / (append_ms / 1e3) / 1e9 / hbm_peak,
                                "ms": append_ms, "bytes": append_bytes,
                                "what": "bulk re-quantise of all 8192 tokens x 512 heads from bf16 K/V"},
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": 1e3 * e2e_s / K},
            "two_calls": {"ms_per_step": two_calls_ms,
                          "what": "the same step as tq_append_quantize + tq_decode_attention (4 launches)"},
            "paged": {"ms_per_step": paged_ms, "GB_per_s": step_bytes / (paged_ms / 1e3) / 1e9,
                      "frac": step_bytes / (paged_ms / 1e3) / 1e9 / hbm_peak,
                      "what": "the same step on a paged cache: each sequence-head's 16-token blocks at "
                              "shuffled pool positions through a block table"},
            "gpu_launches": LAUNCHES_PER_STEP * K,
            "clocks": clk,
        }
        if world == 1 and not args.no_configs:
            line["configs"] = measure_configs(dev)
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
