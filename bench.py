#!/usr/bin/env python
"""Benchmark of the fused DeMo shard step on GB300: prints ONE JSON line.

Default workload: the largest single-GPU shard of the flat sweep, 2^30 =
1,073,741,824 float32 parameters, R = 2 resident replicas, DeMo scheme with
k = 4 of 32 (compression 1/8), ternary sign on, beta = 0.999, lr = 1e-3,
gradients N(0, 1e-3).  A step is one call of demo_step (every replica's
encode, the scatter-mean and the parameter update) on one batch of synthetic
gradients.  The model-shaped shards (T5-base, ViT-B/16, OLMo2-1B half) are
selected with --workload and measured by --sweep.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 is launched by torchrun, one rank per GPU; every rank runs its own
shard (weak scaling, no data-path collective); value = N * n / max-over-ranks
step time.  ``--impl reference`` times the float64 CPU oracle instead (rank 0
only) on a bounded sample of the same workload.
"""

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DeMo step params/s and achieved HBM GB/s (% of GB300 peak) per shard size"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=f"flat{1 << 30}")
    p.add_argument("--mode", default=None, help="demo | random | stride | diloco (default: the workload's first run)")
    p.add_argument("--k", type=int, default=None)
    p.add_argument("--sign", type=int, default=None)
    p.add_argument("--R", type=int, default=None)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--sustained-s", type=float, default=0.5,
                   help="also time a window of at least this many seconds of back-to-back steps on shards larger "
                        "than L2, with its own clock record (0: skip)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--sweep", default=None, help="measure every configuration of the results table into this JSONL file")
    p.add_argument("--sweep-match", default=None,
                   help="with --sweep: only the configurations whose 'workload mode k R' label matches this regex")
    p.add_argument("--only", choices=["split", "adamw"], default=None,
                   help="time only this path on the workload (R encodes + one decode, or the Decoupled AdamW step) "
                        "and print its time; for profiling those kernels")
    p.add_argument("--wire", default="f32", help="payload wire format of --only split and --exchange")
    p.add_argument("--exchange", action="store_true",
                   help="one replica per GPU: every rank steps its own replica of the workload's shard and the "
                        "payloads are exchanged by the process group (NCCL; R = the number of ranks); prints the "
                        "rank-0 line with the max-over-ranks step time")
    p.add_argument("--diloco-period", type=int, default=1,
                   help="DiLoCo sync period of the timed steps: 1 (default) makes every step a sync step, a "
                        "period longer than warm-up + steps times only the steps between syncs (momentum only)")
    a = p.parse_args()
    if a.diloco_period < 1 or 1 < a.diloco_period <= a.warmup + a.steps:
        p.error("--diloco-period must be 1 or longer than --warmup + --steps (one kind of step per run)")
    return a


def diloco_syncs(args):
    """Whether the run's DiLoCo steps are sync steps (all of them) or not (none)."""
    return args.diloco_period == 1


# ----------------------------------------------------------------------------
# Clock sampling (NVML read-only queries; nvidia-smi fallback)
# ----------------------------------------------------------------------------

_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
            0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting", 0x1: "gpu_idle"}


class ClockSampler:
    """Samples the SM clock and the active clock-event reasons of one GPU in a thread."""

    def __init__(self, cuda_index):
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._nvml = None
        self._dev = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            import torch

            bus = torch.cuda.get_device_properties(cuda_index)
            bus_id = "%04x:%02x:%02x.0" % (bus.pci_domain_id, bus.pci_bus_id, bus.pci_device_id)
            dev = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(dev)) != 0:
                raise OSError("no NVML handle for " + bus_id)
            mx = ctypes.c_uint(0)
            nv.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self._nvml, self._dev = nv, dev
            fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self._reasons_fn = fn
        except Exception:
            self._nvml = None

    def _loop(self):
        nv, dev = self._nvml, self._dev
        clk = ctypes.c_uint(0)
        rs = ctypes.c_ulonglong(0)
        while not self._stop.is_set():
            nv.nvmlDeviceGetClockInfo(dev, 1, ctypes.byref(clk))
            self._reasons_fn(dev, ctypes.byref(rs))
            self.samples.append((clk.value, rs.value))
            time.sleep(0.002)

    def __enter__(self):
        if self._nvml is not None:
            self._t = threading.Thread(target=self._loop, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self._nvml is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return None
        reasons = set()
        for _, r in self.samples:
            for bit, name in _REASONS.items():
                if r & bit and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples)}


# ----------------------------------------------------------------------------
# Shared helpers
# ----------------------------------------------------------------------------

def workload_settings(args):
    from decoupled_momentum_optimizer_gb300 import workloads as W

    wl = W.workload(args.workload)
    mode, k, sign = wl.runs[0]
    if args.mode is not None:
        mode = args.mode
    if args.k is not None:
        k = args.k
    if args.sign is not None:
        sign = bool(args.sign)
    R = args.R if args.R is not None else wl.R
    return wl, mode, k, sign, R


def algorithmic_bytes(n, R, grad_bytes, mode, sync=True):
    """Bytes one fused step must move: per replica g (read) and m (read + write), theta (read + write)."""
    theta = 8 * n if (mode != "diloco" or sync) else 0
    return n * R * (grad_bytes + 8) + theta


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


STEP_KERNEL_SOURCES = ("demo_step.cu", "demo_common.cuh", "demo_params.h", "dct32_factors.cuh")


def src_hash():
    """Hash of the fused step kernel's sources and compile options (the kernel the roofline
    and traffic describe); include paths are left out, so the hash is the same on every machine."""
    import hashlib

    from decoupled_momentum_optimizer_gb300 import build

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decoupled_momentum_optimizer_gb300", "csrc")
    for f in STEP_KERNEL_SOURCES:
        h.update(strip_comments(open(os.path.join(csrc, f)).read()).encode())
    h.update(" ".join(f for f in build.NVCC_FLAGS if not os.path.isabs(f)).encode())
    return h.hexdigest()[:16]


def strip_comments(src):
    """C/C++ source without its comments and trailing blanks (string and character literals kept),
    so that editing a comment does not change the source hash."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def ncu_traffic(workload, mode, k, R):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    cur = src_hash()
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if len(f) >= 6 and f[0] == workload and f[1] == mode and int(f[2]) == k and int(f[3]) == R and f[4] == cur:
            return float(f[5])
    return None


_ORACLE_TIMER = r"""
import json, sys, time
sys.path.insert(0, %r)
import numpy as np
import oracle.demo_ref as ref
mode, k, sign, R, nc, budget, max_steps = %r, %d, %r, %d, %d, %f, %d
n = nc * 32
rng = np.random.default_rng(0)
th = rng.standard_normal(n) * 2e-2
ms = [np.zeros(n) for _ in range(R)]
steps, el = 0, 0.0
for t in range(max_steps + 1):  # step 0 is an untimed warm-up
    gs = [rng.standard_normal(n).astype(np.float32).astype(np.float64) * 1e-3 for _ in range(R)]
    ts = time.perf_counter()
    th, ms, _ = ref.step(th, ms, gs, beta=0.999, lr=1e-3, k=k, mode=ref.__dict__["MODE_" + mode.upper()],
                         sign=sign, step_idx=t, period=1 if mode == "diloco" else 8)
    if t > 0:
        el += time.perf_counter() - ts
        steps += 1
        if el >= budget:
            break
print(json.dumps({"params_per_s": n * steps / el, "steps": steps, "seconds": el, "sample_params": n}))
"""


def oracle_time(mode, k, sign, R, nc, seconds, threads, max_steps=1000):
    """Time the float64 oracle in a fresh process (BLAS/OpenMP threads = `threads`) on nc
    chunks of synthetic input: one warm-up step, then steps until `seconds` or max_steps."""
    code = _ORACLE_TIMER % (ROOT, mode, k, sign, R, nc, seconds, max_steps)
    t = str(threads)
    env = dict(os.environ, OPENBLAS_NUM_THREADS=t, OMP_NUM_THREADS=t, MKL_NUM_THREADS=t)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return None, r.stderr[-300:]
    return json.loads(r.stdout.strip().splitlines()[-1]), None


def cpu_baseline(wl_name, mode, k, sign, R, seconds=10.0):
    """Time the float64 oracle in a fresh process on a sample of the workload: one thread
    (the reported value) and, beside it, with every host core available to BLAS."""
    nc = 16384
    d, err = oracle_time(mode, k, sign, R, nc, seconds, 1)
    if d is None:
        return {"value": None, "unit": "params/s", "cores": 1, "kind": "oracle", "error": err}
    out = {"value": d["params_per_s"], "unit": "params/s", "cores": 1, "kind": "oracle",
           "sample": f"{d['sample_params']} params ({nc} chunks) of the {wl_name} workload, {mode} k={k} "
                     f"sign={int(sign)} R={R}, {d['steps']} timed steps in {d['seconds']:.1f} s after one "
                     f"warm-up step, float64 numpy, one thread (BLAS threads = 1)",
           "host": host_cpu()}
    ncpu = os.cpu_count() or 1
    if ncpu > 1:
        # the same sample with every host core available to BLAS (the oracle's elementwise
        # numpy work stays on one thread, so this is its best case on this host)
        d2, _ = oracle_time(mode, k, sign, R, nc, seconds, ncpu)
        if d2 is not None:
            out["all_cores"] = {"value": d2["params_per_s"], "cores": ncpu, "steps": d2["steps"],
                                "seconds": round(d2["seconds"], 2)}
    return out


def host_cpu():
    """CPU description of this host (model name, or the ARM implementer/part codes) and its core count."""
    import platform

    desc = None
    try:
        fields = {}
        for line in open("/proc/cpuinfo"):
            if ":" in line:
                key, val = (x.strip() for x in line.split(":", 1))
                fields.setdefault(key, val)
        if "model name" in fields:
            desc = fields["model name"]
        elif "CPU implementer" in fields:
            desc = f"ARM implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    except OSError:
        pass
    return {"cpu": desc or platform.processor() or "unknown", "machine": platform.machine(), "cores": os.cpu_count()}


# ----------------------------------------------------------------------------
# Reference arm: the CPU oracle, rank 0 only
# ----------------------------------------------------------------------------

def run_config(wl, R, mode, k, sign, world, sync=True):
    """The JSON line's `config`: the workload one GPU's step covers (both arms print the same)."""
    step_bytes = algorithmic_bytes(wl.n, R, 2 if wl.g_dtype == "bf16" else 4, mode, sync=sync)
    flush = step_bytes < 2 * L2_BYTES
    return {"workload": f"{wl.name}: {wl.n} params, R={R} resident replicas, {mode} k={k}/32, "
                        f"sign={'on' if sign else 'off'}, grads {wl.g_dtype}"
                        + ((", every step a sync step" if sync else ", steps between syncs (momentum only)")
                           if mode == "diloco" else ""),
            "n": wl.n, "R": R, "mode": mode, "k": k, "sign": bool(sign), "grad_dtype": wl.g_dtype,
            "parallelism": f"one shard per GPU x {world}",
            "l2": "L2 flushed (256 MB write) between steps" if flush else
            f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB per step)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np

    import oracle.demo_ref as ref

    wl, mode, k, sign, R = workload_settings(args)
    nc = 4096
    n = nc * 32
    rng = np.random.default_rng(0)
    th = rng.standard_normal(n) * wl.theta_std
    ms = [np.zeros(n) for _ in range(R)]
    times = []
    for t in range(args.warmup + args.steps):
        gs = [rng.standard_normal(n).astype(np.float32).astype(np.float64) * wl.g_std for _ in range(R)]
        t0 = time.perf_counter()
        th, ms, _ = ref.step(th, ms, gs, beta=wl.beta, lr=wl.lr, k=k, mode=ref.__dict__["MODE_" + mode.upper()],
                             sign=sign, step_idx=t, period=args.diloco_period)
        if t >= args.warmup:
            times.append(time.perf_counter() - t0)
    per = sum(times) / len(times)
    value = n / per
    sample = (f"{n} params (4096 chunks) of the {wl.name} workload per step, {mode} k={k} sign={int(sign)} R={R}, "
              f"float64 numpy oracle, {os.cpu_count()} host cores available")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": run_config(wl, R, mode, k, sign, args.gpus, mode != "diloco" or diloco_syncs(args)),
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------

class Case:
    """Device state for one (workload, R) measurement: theta, m_r and gradient sets."""

    def __init__(self, wl, R, dev, n_sets):
        import torch

        from decoupled_momentum_optimizer_gb300 import workloads as W

        self.wl, self.R, self.n = wl, R, wl.n
        self.theta = W.make_theta0(wl, dev)
        self.ms = [torch.zeros(wl.n, device=dev) for _ in range(R)]
        streams = [W.GradStream(wl, r, dev) for r in range(R)]
        self.ring = [[s.next() for s in streams] for _ in range(n_sets)]
        self.grad_bytes = self.ring[0][0].element_size()


def time_fused(dm, case, mode, k, sign, seed, steps, warmup, stream, per_launch=True, sampler=None,
               step0=0, diloco_period=8):
    """Mean step and mean launch time (ms) of demo_step over ``steps`` timed steps, and the
    per-launch statistics (median, min, max) with whether L2 was flushed between steps."""
    import torch

    wl = case.wl
    flush = algorithmic_bytes(case.n, case.R, case.grad_bytes, mode) < 2 * L2_BYTES
    scratch = torch.empty(256 * 1024 * 1024 // 4, device=case.theta.device) if flush else None

    def one(t):
        dm.step(case.theta, case.ring[t % len(case.ring)], case.ms, k=k, beta=wl.beta, lr=wl.lr, mode=mode,
                sign=sign, seed=seed, step=t, diloco_period=diloco_period, stream=stream)

    for t in range(warmup):
        one(step0 + t)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        a.record(stream)
        for i in range(steps):
            if flush:
                scratch.fill_(float(i))
            ev[i][0].record(stream)
            one(step0 + warmup + i)
            ev[i][1].record(stream)
        b.record(stream)
        torch.cuda.synchronize()
    times = [x.elapsed_time(y) for x, y in ev]
    launch = sum(times) / steps
    step = launch if flush else a.elapsed_time(b) / steps
    return step, launch, {"l2_flush": flush, "median": statistics.median(times), "min": min(times),
                          "max": max(times)}


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def time_split(dm, case, mode, k, sign, seed, steps, warmup, stream, diloco_period=8, step0=0, wire="f32"):
    """Mean time (ms) of the split path, every replica's encode (one demo_encode_replicas call) + one
    demo_decode_update, in the wire format; each step timed alone after an L2 flush when it is smaller
    than twice the L2."""
    import torch

    wl, n, R = case.wl, case.n, case.R
    dev = case.theta.device
    bufs = [dm.payload_buffers(mode, n, k, step=diloco_period - 1, diloco_period=diloco_period, wire=wire,
                               device=dev) for _ in range(R)]
    vals = [b[0] for b in bufs]
    idx = [b[1] for b in bufs] if mode == "demo" else None

    sends = mode != "diloco" or diloco_period == 1

    def one(t):
        g = case.ring[t % len(case.ring)]
        dm.encode_replicas(g, case.ms, vals if sends else None, idx, k=k, beta=wl.beta, mode=mode, sign=sign,
                           diloco_period=diloco_period, seed=seed, step=t, wire=wire, stream=stream)
        dm.decode_update(case.theta, vals, idx, k=k, lr=wl.lr, mode=mode, diloco_period=diloco_period, seed=seed,
                         step=t, wire=wire, stream=stream)

    for t in range(warmup):
        one(step0 + t)
    torch.cuda.synchronize()
    nbytes = split_bytes(n, R, case.grad_bytes, mode, k, sync=mode != "diloco" or diloco_period == 1, wire=wire)
    return _timed_steps(lambda i: one(step0 + warmup + i), steps, stream, nbytes < 2 * L2_BYTES, dev)


def _timed_steps(fn, steps, stream, flush, dev):
    """Mean time (ms) of ``steps`` calls of fn(i) on ``stream``.  With ``flush`` (a step smaller than
    twice the L2) every call is timed alone by its own CUDA events after a 256 MB write flushes L2;
    otherwise the calls run back to back between two events (their inputs exceed L2)."""
    import torch

    if not flush:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps
    scratch = torch.empty(256 * 1024 * 1024 // 4, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        scratch.fill_(float(i))
        ev[i][0].record(stream)
        fn(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(x.elapsed_time(y) for x, y in ev) / steps


def time_split_graph(dm, case, mode, k, sign, seed, steps, warmup, stream, wire="f32"):
    """Mean time (ms) of the split path (demo_encode_replicas + demo_decode_update) captured once into a
    CUDA graph and replayed (each replay timed alone after an L2 flush when the step is smaller than
    twice the L2); the graph keeps its captured step index."""
    import torch

    wl, n, R = case.wl, case.n, case.R
    dev = case.theta.device
    bufs = [dm.payload_buffers(mode, n, k, wire=wire, device=dev) for _ in range(R)]
    vals = [b[0] for b in bufs]
    idx = [b[1] for b in bufs] if mode == "demo" else None
    g = case.ring[0]

    def one():
        dm.encode_replicas(g, case.ms, vals, idx, k=k, beta=wl.beta, mode=mode, sign=sign, seed=seed, step=1,
                           wire=wire)
        dm.decode_update(case.theta, vals, idx, k=k, lr=wl.lr, mode=mode, seed=seed, step=1, wire=wire)

    one()  # the first call of each kernel shape happens outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        one()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize()
        nbytes = split_bytes(n, R, case.grad_bytes, mode, k, wire=wire)
        return _timed_steps(lambda i: graph.replay(), steps, stream, nbytes < 2 * L2_BYTES, dev)


def time_adamw(dm, case, steps, warmup, stream):
    """Mean time (ms) of one Decoupled AdamW step (demo_adamw_step) over the case's replicas."""
    import torch

    vs = [torch.zeros_like(m) for m in case.ms]

    def one(t):
        dm.adamw_step(case.theta, case.ring[t % len(case.ring)], case.ms, vs, lr=1e-3, weight_decay=0.01, step=t,
                      stream=stream)

    for t in range(warmup):
        one(t)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        one(warmup + i)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def time_pipelined(dm, case, mode, k, sign, steps, warmup, stream, wire="f32", blocks=8):
    """Mean time (ms) of demo_step_pipelined (split path, exchange overlapped on a second stream)."""
    import torch

    wl, n, R = case.wl, case.n, case.R
    dev = case.theta.device
    send = [dm.payload_buffers(mode, n, k, wire=wire, device=dev) for _ in range(R)]
    recv = [dm.payload_buffers(mode, n, k, wire=wire, device=dev) for _ in range(R)]
    comm = torch.cuda.Stream(device=dev)

    def one(t):
        dm.step_pipelined(case.theta, case.ring[t % len(case.ring)], case.ms, send, recv, k=k, beta=wl.beta,
                          lr=wl.lr, mode=mode, sign=sign, step=t, wire=wire, blocks=blocks, stream=stream,
                          comm_stream=comm)

    for t in range(warmup):
        one(t)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        one(warmup + i)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def split_bytes(n, R, grad_bytes, mode, k, sync=True, wire="f32"):
    """Algorithmic bytes of the split path: R encodes (g, m, payload out) + decode (R payloads in, theta)."""
    import decoupled_momentum_optimizer_gb300 as dm

    vb, ib = dm.payload_bytes(mode, n, k, step=7 if sync else 0, diloco_period=8, wire=wire)
    P = vb + ib
    theta = 8 * n if (mode != "diloco" or sync) else 0
    return R * (n * (grad_bytes + 8) + P) + (R * P + theta if theta else 0)


def time_e2e(dm, case, mode, k, sign, seed, steps, dev, diloco_period=8, depth=3):
    """End to end through the public API: every step copies its R gradients from pinned host memory
    and reads theta back to pinned host memory, on three streams: uploads, steps, read-backs.

    The host link carries about 211 GB/s host-to-device and 193 GB/s device-to-host alone and
    about 340 GB/s in both directions together, so a step's copies (R gradients up, theta down)
    take longer than its kernel on large shards; the pipeline keeps the upload stream busy: the
    gradients of step t + depth are uploaded into a ring of ``depth`` device buffers as soon as
    step t has read its buffer, and theta is read back from a device snapshot (two, alternating)
    while later steps run."""
    import torch

    wl, n, R = case.wl, case.n, case.R
    host_g = [[g.cpu().pin_memory() for g in case.ring[i % len(case.ring)]] for i in range(2)]
    host_theta = torch.empty(n, dtype=torch.float32).pin_memory()
    dev_g = [[torch.empty_like(g) for g in case.ring[0]] for _ in range(depth)]
    snaps = [torch.empty_like(case.theta) for _ in range(2)]
    main = torch.cuda.current_stream()
    h2d = torch.cuda.Stream(device=dev)
    d2h = torch.cuda.Stream(device=dev)

    def run(K, t0):
        e_in = [torch.cuda.Event() for _ in range(K)]
        e_step = [torch.cuda.Event() for _ in range(K)]
        e_out = [torch.cuda.Event() for _ in range(K)]

        def load(t):
            with torch.cuda.stream(h2d):
                if t >= depth:
                    h2d.wait_event(e_step[t - depth])  # step t - depth has finished reading this buffer
                for r in range(R):
                    dev_g[t % depth][r].copy_(host_g[t % 2][r], non_blocking=True)
                e_in[t].record(h2d)

        for t in range(min(depth, K)):
            load(t)
        for t in range(K):
            main.wait_event(e_in[t])
            dm.step(case.theta, dev_g[t % depth], case.ms, k=k, beta=wl.beta, lr=wl.lr, mode=mode, sign=sign,
                    seed=seed, step=t0 + t, diloco_period=diloco_period, stream=main)
            if t >= 2:
                main.wait_event(e_out[t - 2])  # the snapshot buffer has been read back
            snaps[t % 2].copy_(case.theta)
            e_step[t].record(main)
            with torch.cuda.stream(d2h):
                d2h.wait_event(e_step[t])
                host_theta.copy_(snaps[t % 2], non_blocking=True)
                e_out[t].record(d2h)
            if t + depth < K:
                load(t + depth)
        return e_out[K - 1]

    run(2, 1000)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(main)
    last = run(steps, 2000)
    main.wait_event(last)
    b.record(main)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return ms, sum(g.numel() * g.element_size() for g in host_g[0]), n * 4


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.only:
        return run_only(args)
    if args.exchange:
        return run_exchange(args)

    import torch
    import torch.distributed as dist

    import decoupled_momentum_optimizer_gb300 as dm
    from decoupled_momentum_optimizer_gb300.sharding import shard_seed

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    wl, mode, k, sign, R = workload_settings(args)
    n = wl.n
    dm.init(local)
    dev = torch.device("cuda", local)
    case = Case(wl, R, dev, n_sets=3)  # three pre-drawn gradient sets per replica, cycled
    sync = mode != "diloco" or diloco_syncs(args)
    step_bytes = algorithmic_bytes(n, R, case.grad_bytes, mode, sync=sync)
    stream = torch.cuda.current_stream()
    seed = shard_seed(0, rank)  # each GPU steps its own shard with its own index seed

    period = args.diloco_period if mode == "diloco" else 8
    sampler = ClockSampler(local)
    barrier()
    step_ms, kernel_ms, lstats = time_fused(dm, case, mode, k, sign, seed, args.steps, args.warmup, stream,
                                            sampler=sampler, diloco_period=period)
    barrier()
    if world > 1:
        tt = torch.tensor([step_ms, kernel_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        step_ms, kernel_ms = tt.tolist()

    sustained = None
    if args.sustained_s > 0 and step_bytes >= 2 * L2_BYTES:
        # a window of at least --sustained-s seconds of back-to-back steps beside the K-step mean, with
        # its own clock record: K steps of a large shard may hold the GPU for only ~0.1 s
        S = max(args.steps, min(20000, int(args.sustained_s / (step_ms * 1e-3)) + 1))
        sampler2 = ClockSampler(local)
        barrier()
        s_ms, s_kernel, _ = time_fused(dm, case, mode, k, sign, seed, S, 0, stream, sampler=sampler2,
                                       step0=args.warmup + args.steps, diloco_period=period)
        barrier()
        if world > 1:
            tt = torch.tensor([s_ms, s_kernel], device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            s_ms, s_kernel = tt.tolist()
        sustained = {"steps": S, "seconds": S * s_ms * 1e-3, "ms_per_step": s_ms, "launch_ms_mean": s_kernel,
                     "value": world * n / (s_ms * 1e-3), "achieved_gbs": step_bytes / (s_kernel * 1e-3) / 1e9,
                     "clocks": sampler2.summary(),
                     "note": "timed after the K-step window, same stream and inputs; reported beside the headline"}

    e2e = None
    if not args.no_e2e:
        Ke = max(3, min(args.steps, 20))
        barrier()
        e_ms, hb, db = time_e2e(dm, case, mode, k, sign, seed, Ke, dev, diloco_period=period)
        if world > 1:
            tt = torch.tensor([e_ms], device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            e_ms = tt.item()
        e2e = {"value": world * n / (e_ms * 1e-3), "unit": "params/s", "h2d_bytes_per_step": hb,
               "d2h_bytes_per_step": db, "ms_per_step": e_ms, "steps": Ke,
               "note": "gradients copied from pinned host memory and theta read back every step; "
                       "uploads run up to three steps ahead into a ring of device buffers and theta "
                       "is read back from a device snapshot while later steps run (host link: about "
                       "211 GB/s host-to-device, 193 GB/s device-to-host, 340 GB/s both at once)"}

    fault = dm.device_fault()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = measured_peaks()
    achieved = step_bytes / (kernel_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": ncu_traffic(args.workload, mode, k, R),
            "kernel": "demo::step_kernel" if sync else "demo::momentum_kernel",
            "algorithmic_bytes_per_launch": step_bytes,
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s"}
    line = {
        "metric": METRIC,
        "value": world * n / (step_ms * 1e-3),
        "unit": "params/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": run_config(wl, R, mode, k, sign, world, sync),
        "achieved_gbs": achieved,
        "hbm_frac_of_peak": achieved / peak,
        "launch_ms": {"mean": kernel_ms, "median": lstats["median"], "min": lstats["min"], "max": lstats["max"],
                      "note": "CUDA events around each timed launch; mean is the max over ranks, the rest rank 0's"},
        "roofline": roof,
        "gpu_launches": args.steps,
        "clocks": sampler.summary(),
        "sustained": sustained,
        "e2e": e2e,
        "device_fault": fault,
    }
    if not args.no_cpu_baseline and world == 1:  # the CPU baseline is taken at N = 1 only
        line["cpu_baseline"] = cpu_baseline(wl.name, mode, k, sign, R)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------
# One replica per GPU: the payloads exchanged by the process group
# ----------------------------------------------------------------------------

def run_exchange(args):
    """Every rank holds one replica of the workload's shard (R = world size) and steps it through
    ReplicaExchange: the library's encode, an NCCL all_gather (DeMo) or all-reduce (the other
    schemes with float32 values) of the wire-format payloads, the library's decode.  Without
    torchrun it runs as a one-rank group.  Prints rank 0's JSON line (max-over-ranks step time)."""
    import torch
    import torch.distributed as dist

    import decoupled_momentum_optimizer_gb300 as dm
    from decoupled_momentum_optimizer_gb300 import workloads as W
    from decoupled_momentum_optimizer_gb300.exchange import ReplicaExchange

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    else:
        dist.init_process_group("nccl", rank=0, world_size=1, store=dist.HashStore(), device_id=dev)
    dm.init(local)
    wl, mode, k, sign, _ = workload_settings(args)
    n = wl.n
    period = args.diloco_period if mode == "diloco" else 8
    ex = ReplicaExchange(n, k, mode, wire=args.wire, diloco_period=period)
    theta = W.make_theta0(wl, dev)
    m = torch.zeros(n, device=dev)
    stream = W.GradStream(wl, rank, dev)  # this rank's replica draws its own gradients
    ring = [stream.next() for _ in range(3)]
    main = torch.cuda.current_stream()

    def one(t):
        ex.step(theta, ring[t % len(ring)], m, beta=wl.beta, lr=wl.lr, sign=sign, seed=0, step=t)

    for t in range(args.warmup):
        one(t)
    torch.cuda.synchronize()
    dist.barrier()
    grad_bytes = ring[0].element_size()
    step_bytes = n * (grad_bytes + 8) + (8 * n if (mode != "diloco" or diloco_syncs(args)) else 0)
    ms = _timed_steps(lambda i: one(args.warmup + i), args.steps, main, step_bytes < 2 * L2_BYTES, dev)
    dist.barrier()
    tt = torch.tensor([ms], device=dev)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    ms = tt.item()
    tx, rx = ex.bytes_per_step(period - 1 if mode == "diloco" else 0)
    fault = dm.device_fault()
    if rank == 0:
        line = {
            "metric": METRIC, "value": world * n / (ms * 1e-3), "unit": "params/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{wl.name}: {n} params, one replica per GPU (R = {world}), {mode} k={k}/32, "
                                   f"sign={'on' if sign else 'off'}, grads {wl.g_dtype}, payloads exchanged by "
                                   f"{ex.collective} ({args.wire})",
                       "n": n, "R": world, "mode": mode, "k": k, "sign": bool(sign), "wire": args.wire,
                       "collective": ex.collective, "payload_bytes_sent": tx, "payload_bytes_received": rx,
                       "parallelism": f"one replica per GPU x {world}",
                       "note": "value counts every rank's replica: world x n params per step"},
            "device_fault": fault,
        }
        print(json.dumps(line), flush=True)
    dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------
# Sweep: every configuration of the results table, one JSON line each
# ----------------------------------------------------------------------------

def sweep_cases():
    """(workload, mode, k, sign, R, paths) for the results table."""
    out = []
    for name in ("t5_base", "vit_b16", "olmo2_1b_half"):
        from decoupled_momentum_optimizer_gb300 import workloads as W

        wl = W.workload(name)
        for mode, k, sign in wl.runs:
            out.append((name, mode, k, sign, wl.R, ("fused", "split")))
    # compact wire formats of the split path (T5-base shard)
    out.append(("t5_base", "demo", 4, True, 2, ("split:ternary", "split:bf16")))
    out.append(("t5_base", "random", 8, True, 2, ("split:ternary",)))
    out.append(("t5_base", "demo", 4, False, 2, ("split:bf16", "split:f16")))
    # split path with the exchange (payload copies) overlapped on a second stream
    out.append(("t5_base", "demo", 4, True, 2, ("pipe:f32:4", "pipe:f32:16", "pipe:ternary:16")))
    # Decoupled AdamW (moments local, directions averaged densely)
    for name in ("t5_base", "olmo2_1b_half", f"flat{1 << 28}"):
        out.append((name, "adamw", 0, False, 2, ("adamw",)))
    # the 65,536-parameter shard (DeMo k=4, sign, R=2): fused and split
    out.append(("flat64k", "demo", 4, True, 2, ("fused", "split")))
    # the flat size sweep: 2^20..2^30 parameters x k in {1, 2, 4, 8} x R in {1, 2, 8, 64} (R = 64 up
    # to 2^26) x every scheme, sign on; DiLoCo (k does not apply) as steps between syncs and as
    # sync steps; the split path beside the fused step at 2^26
    for e in range(20, 31):
        for R in (1, 2, 8, 64):
            if R == 64 and e > 26:
                continue
            paths = ("fused", "split") if e == 26 else ("fused",)
            for mode in ("demo", "random", "stride"):
                for k in (1, 2, 4, 8):
                    out.append((f"flat{1 << e}", mode, k, True, R, paths))
            for kind in ("diloco", "diloco-sync"):
                out.append((f"flat{1 << e}", kind, 1, True, R, paths))
    # the split path on small shards, eager against a CUDA graph replay
    for e in (16, 20, 22, 24):
        out.append((f"flat{1 << e}" if e != 16 else "flat64k", "demo", 4, True, 2, ("graph",)))
        out.append((f"flat{1 << e}" if e != 16 else "flat64k", "random", 8, True, 2, ("graph",)))
    return out


def run_only(args):
    """Time one path (split or AdamW) on the workload; prints a line of its own, not the bench line."""
    import torch

    import decoupled_momentum_optimizer_gb300 as dm

    dm.init(0)
    wl, mode, k, sign, R = workload_settings(args)
    case = Case(wl, R, torch.device("cuda", 0), n_sets=2)
    stream = torch.cuda.current_stream()
    if args.only == "split":
        # DiLoCo: one kind of step per run (--diloco-period)
        ms = time_split(dm, case, mode, k, sign, 0, args.steps, args.warmup, stream, wire=args.wire,
                        diloco_period=args.diloco_period if mode == "diloco" else 8)
        nbytes = split_bytes(case.n, R, case.grad_bytes, mode, k, wire=args.wire,
                             sync=mode != "diloco" or diloco_syncs(args))
    else:
        ms = time_adamw(dm, case, args.steps, args.warmup, stream)
        nbytes = case.n * (R * (case.grad_bytes + 16) + 8)
    print(json.dumps({"only": args.only, "workload": wl.name, "n": case.n, "mode": mode, "k": k, "R": R,
                      "wire": args.wire if args.only == "split" else None, "ms": ms,
                      "gbs": nbytes / (ms * 1e-3) / 1e9, "device_fault": dm.device_fault()}))
    return 0


def run_sweep(args):
    import torch

    import decoupled_momentum_optimizer_gb300 as dm
    from decoupled_momentum_optimizer_gb300 import workloads as W

    dm.init(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peak, _ = measured_peaks()
    cache = {}
    f = open(args.sweep, "w")
    import re

    match = re.compile(args.sweep_match) if args.sweep_match else None
    for name, mode, k, sign, R, paths in sweep_cases():
        if match is not None and not match.search(f"{name} {mode} {k} {R}"):
            continue
        key = (name, R)
        if key not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            wl = W.workload(name)
            cache[key] = Case(wl, R, dev, n_sets=1 if wl.n >= (1 << 24) else 3)
        case = cache[key]
        n = case.n
        # DiLoCo: "diloco" times the steps between syncs, "diloco-sync" the sync steps; the
        # period makes every warm-up and timed step of the row of that one kind (1: every step
        # syncs; longer than the run: none does)
        real_mode = "diloco" if mode.startswith("diloco") else mode
        sync = mode == "diloco-sync"
        period = 1 if sync else 1 << 30
        rec = {"workload": name, "n": n, "mode": mode, "k": k, "sign": sign, "R": R, "grad_dtype": case.wl.g_dtype}
        steps, warmup = args.steps, args.warmup
        if "graph" in paths:
            # the split path on a small shard: R + 1 calls eagerly (host-bound) and as one replayed graph
            em = time_split(dm, case, real_mode, k, sign, 0, 10 * steps, warmup, stream)
            gm = time_split_graph(dm, case, real_mode, k, sign, 0, 10 * steps, warmup, stream)
            sb = split_bytes(n, R, case.grad_bytes, real_mode, k)
            r2 = dict(rec, mode=f"{mode}/graph", split_ms=em, split_graph_ms=gm, split_bytes=sb,
                      split_graph_gbs=sb / (gm * 1e-3) / 1e9, split_graph_frac=sb / (gm * 1e-3) / 1e9 / peak)
            f.write(json.dumps(r2) + "\n")
            f.flush()
            print(f"{name:16s} {mode + '/graph':16s} k={k:2d} sign={int(sign)} R={R:2d}  split eager {em * 1e3:7.1f} us"
                  f"  graph {gm * 1e3:7.1f} us {r2['split_graph_gbs']:7.0f} GB/s", flush=True)
            continue
        if mode == "adamw":
            am = time_adamw(dm, case, args.steps, args.warmup, stream)
            ab = n * (R * (case.grad_bytes + 16) + 8)
            r2 = dict(rec, fused_ms=am, fused_params_per_s=n / (am * 1e-3), fused_bytes=ab,
                      fused_gbs=ab / (am * 1e-3) / 1e9, fused_frac=ab / (am * 1e-3) / 1e9 / peak)
            f.write(json.dumps(r2) + "\n")
            f.flush()
            print(f"{name:16s} {'adamw':16s} R={R:2d}  step {am:8.3f} ms {r2['fused_gbs']:7.0f} GB/s "
                  f"{100 * r2['fused_frac']:5.1f}%", flush=True)
            continue
        pipes = [x.split(":")[1:] for x in paths if x.startswith("pipe:")]
        if pipes:
            for wire, blocks in pipes:
                pm = time_pipelined(dm, case, real_mode, k, sign, steps, warmup, stream, wire=wire, blocks=int(blocks))
                # bytes: the split path's plus the exchange copies (read + write of every payload)
                pb = split_bytes(n, R, case.grad_bytes, real_mode, k, wire=wire) + 2 * R * sum(
                    dm.payload_bytes(real_mode, n, k, wire=wire))
                r2 = dict(rec, mode=f"{mode}/{wire}/pipelined{blocks}", split_ms=pm, split_params_per_s=n / (pm * 1e-3),
                          split_bytes=pb, split_gbs=pb / (pm * 1e-3) / 1e9, split_frac=pb / (pm * 1e-3) / 1e9 / peak)
                f.write(json.dumps(r2) + "\n")
                f.flush()
                print(f"{name:16s} {mode + '/' + wire + '/pipe' + blocks:22s} R={R:2d}  {pm:8.3f} ms "
                      f"{r2['split_gbs']:7.0f} GB/s", flush=True)
            continue
        wires = [x.split(":")[1] for x in paths if x.startswith("split:")]
        if wires:
            # wire-format runs of the split path only
            for wire in wires:
                sm = time_split(dm, case, real_mode, k, sign, 0, steps, warmup, stream, wire=wire)
                sb = split_bytes(n, R, case.grad_bytes, real_mode, k, wire=wire)
                r2 = dict(rec, mode=f"{mode}/{wire}", split_ms=sm, split_params_per_s=n / (sm * 1e-3), split_bytes=sb,
                          split_gbs=sb / (sm * 1e-3) / 1e9, split_frac=sb / (sm * 1e-3) / 1e9 / peak,
                          payload_bytes_per_replica=sum(dm.payload_bytes(real_mode, n, k, wire=wire)))
                f.write(json.dumps(r2) + "\n")
                f.flush()
                print(f"{name:16s} {mode + '/' + wire:16s} k={k:2d} sign={int(sign)} R={R:2d}  split {sm:8.3f} ms "
                      f"{r2['split_gbs']:7.0f} GB/s  payload {r2['payload_bytes_per_replica'] / 1e6:8.2f} MB/replica",
                      flush=True)
            continue
        step_ms, launch_ms, lst = time_fused(dm, case, real_mode, k, sign, 0, steps, warmup, stream,
                                             diloco_period=period)
        fb = algorithmic_bytes(n, R, case.grad_bytes, real_mode, sync=sync or real_mode != "diloco")
        rec.update(fused_launch_ms_median=lst["median"], fused_launch_ms_min=lst["min"])
        rec.update(fused_ms=step_ms, fused_params_per_s=n / (step_ms * 1e-3), fused_bytes=fb,
                   fused_gbs=fb / (launch_ms * 1e-3) / 1e9, fused_frac=fb / (launch_ms * 1e-3) / 1e9 / peak)
        if "split" in paths:
            sm = time_split(dm, case, real_mode, k, sign, 0, steps, warmup, stream, diloco_period=period)
            sb = split_bytes(n, R, case.grad_bytes, real_mode, k, sync=sync or real_mode != "diloco")
            rec.update(split_ms=sm, split_params_per_s=n / (sm * 1e-3), split_bytes=sb,
                       split_gbs=sb / (sm * 1e-3) / 1e9, split_frac=sb / (sm * 1e-3) / 1e9 / peak)
        f.write(json.dumps(rec) + "\n")
        f.flush()
        print(f"{name:16s} {mode:11s} k={k:2d} sign={int(sign)} R={R:2d}  fused {step_ms:8.3f} ms "
              f"{rec['fused_gbs']:7.0f} GB/s {100 * rec['fused_frac']:5.1f}%"
              + (f"  split {rec['split_ms']:8.3f} ms {rec['split_gbs']:7.0f} GB/s" if "split_ms" in rec else ""),
              flush=True)
    # the float64 oracle on the host cores, on whole shards: the 65,536-parameter shard for its
    # five steps and a 2^20 shard for three, with one BLAS thread and with every core
    ncpu = os.cpu_count() or 1
    for name, nc, steps in (() if match is not None else (("flat64k", 2048, 5), ("flat1048576", 32768, 3))):
        for threads in sorted({1, ncpu}):
            d, err = oracle_time("demo", 4, True, 2, nc, 1e9, threads, max_steps=steps)
            rec = {"oracle": True, "workload": name, "n": nc * 32, "mode": "demo", "k": 4, "sign": True, "R": 2,
                   "threads": threads, "host": host_cpu()}
            rec.update(d if d is not None else {"error": err})
            f.write(json.dumps(rec) + "\n")
            f.flush()
            if d is not None:
                print(f"{name:16s} oracle {threads:3d} threads  {d['params_per_s']:10.3g} params/s "
                      f"({d['steps']} steps, {d['seconds']:.2f} s)", flush=True)
    f.close()
    print(json.dumps({"sweep": args.sweep, "device_fault": dm.device_fault()}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
