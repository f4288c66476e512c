#!/usr/bin/env python
"""Benchmark of the fused DeMo shard step on GB300: prints ONE JSON line.

Default workload: the T5-base-shaped shard (222,903,552 float32 parameters,
257 tensors each padded to 32), R = 2 resident replicas, DeMo scheme with
k = 4 of 32 (compression 1/8), ternary sign on, beta = 0.999, lr = 1e-3.
A step is one call of demo_step (every replica's encode, the scatter-mean and
the parameter update) on one batch of synthetic gradients.

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
    p.add_argument("--workload", default="t5_base")
    p.add_argument("--mode", default=None, help="demo | random | stride | diloco (default: the workload's first run)")
    p.add_argument("--k", type=int, default=None)
    p.add_argument("--sign", type=int, default=None)
    p.add_argument("--R", type=int, default=None)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


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


def src_hash():
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decoupled_momentum_optimizer_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


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


def cpu_baseline(wl_name, mode, k, sign, R, seconds=10.0):
    """Time the float64 oracle single-threaded in a fresh process on a sample of the workload."""
    code = r"""
import json, os, sys, time
sys.path.insert(0, %r)
import numpy as np
import oracle.demo_ref as ref
mode, k, sign, R, budget = %r, %d, %r, %d, %f
nc = 16384
n = nc * 32
rng = np.random.default_rng(0)
th = rng.standard_normal(n) * 2e-2
ms = [np.zeros(n) for _ in range(R)]
steps, t0 = 0, time.perf_counter()
while True:
    gs = [rng.standard_normal(n).astype(np.float32).astype(np.float64) * 1e-3 for _ in range(R)]
    ts = time.perf_counter()
    th, ms, _ = ref.step(th, ms, gs, beta=0.999, lr=1e-3, k=k, mode=ref.__dict__["MODE_" + mode.upper()],
                         sign=sign, step_idx=steps)
    steps += 1
    if steps == 1:
        el = 0.0
    el += time.perf_counter() - ts
    if el >= budget or steps >= 1000:
        break
print(json.dumps({"params_per_s": n * steps / el, "steps": steps, "seconds": el, "sample_params": n}))
""" % (ROOT, mode, k, sign, R, seconds)
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"value": None, "unit": "params/s", "cores": 1, "kind": "oracle", "error": r.stderr[-300:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["params_per_s"], "unit": "params/s", "cores": 1, "kind": "oracle",
            "sample": f"{d['sample_params']} params (16384 chunks) of the {wl_name} workload, {mode} k={k} "
                      f"sign={int(sign)} R={R}, {d['steps']} steps in {d['seconds']:.1f} s, "
                      f"float64 numpy, one thread (BLAS threads = 1)"}


# ----------------------------------------------------------------------------
# Reference arm: the CPU oracle, rank 0 only
# ----------------------------------------------------------------------------

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
                             sign=sign, step_idx=t)
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
        "config": {"workload": wl.name, "n": wl.n, "R": R, "mode": mode, "k": k, "sign": bool(sign)},
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------

def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    import decoupled_momentum_optimizer_gb300 as dm
    from decoupled_momentum_optimizer_gb300 import workloads as W
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

    # state and a ring of three pre-drawn gradient sets per replica (inputs >> L2)
    theta = W.make_theta0(wl, dev)
    ms = [torch.zeros(n, device=dev) for _ in range(R)]
    streams = [W.GradStream(wl, r, dev) for r in range(R)]
    ring = [[s.next() for s in streams] for _ in range(3)]
    grad_bytes = ring[0][0].element_size()
    step_bytes = algorithmic_bytes(n, R, grad_bytes, mode)
    flush = step_bytes < 2 * L2_BYTES
    scratch = torch.empty(256 * 1024 * 1024 // 4, device=dev) if flush else None
    stream = torch.cuda.current_stream()

    seed = shard_seed(0, rank)  # each GPU steps its own shard with its own index seed

    def one_step(t):
        dm.step(theta, ring[t % 3], ms, k=k, beta=wl.beta, lr=wl.lr, mode=mode, sign=sign, seed=seed, step=t,
                stream=stream)

    for t in range(args.warmup):
        one_step(t)
    torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    with sampler:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(K):
            if flush:
                scratch.fill_(float(i))
            ev[i][0].record(stream)
            one_step(args.warmup + i)
            ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    step_ms = sum(launch_ms) / K if flush else t_start.elapsed_time(t_end) / K
    kernel_ms = sum(launch_ms) / K
    if world > 1:
        tt = torch.tensor([step_ms, kernel_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        step_ms, kernel_ms = tt.tolist()

    # end to end through the public API from pinned host memory
    e2e = None
    if not args.no_e2e:
        host_g = [g.cpu().pin_memory() for g in ring[0]]
        host_theta = torch.empty(n, dtype=torch.float32).pin_memory()
        dev_g = [torch.empty_like(g) for g in ring[0]]
        Ke = max(3, min(K, 10))
        for t in range(2):
            for r in range(R):
                dev_g[r].copy_(host_g[r], non_blocking=True)
            dm.step(theta, dev_g, ms, k=k, beta=wl.beta, lr=wl.lr, mode=mode, sign=sign, step=1000 + t)
            host_theta.copy_(theta, non_blocking=True)
        barrier()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for t in range(Ke):
            for r in range(R):
                dev_g[r].copy_(host_g[r], non_blocking=True)
            dm.step(theta, dev_g, ms, k=k, beta=wl.beta, lr=wl.lr, mode=mode, sign=sign, step=2000 + t)
            host_theta.copy_(theta, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        e_ms = a.elapsed_time(b) / Ke
        if world > 1:
            tt = torch.tensor([e_ms], device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            e_ms = tt.item()
        e2e = {"value": world * n / (e_ms * 1e-3), "unit": "params/s",
               "h2d_bytes_per_step": sum(g.numel() * g.element_size() for g in host_g),
               "d2h_bytes_per_step": n * 4, "ms_per_step": e_ms, "steps": Ke}

    fault = dm.device_fault()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = measured_peaks()
    achieved = step_bytes / (kernel_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": ncu_traffic(args.workload, mode, k, R), "kernel": "demo::step_kernel",
            "algorithmic_bytes_per_launch": step_bytes, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s"}
    line = {
        "metric": METRIC,
        "value": world * n / (step_ms * 1e-3),
        "unit": "params/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{wl.name}: {n} params, R={R} resident replicas, {mode} k={k}/32, "
                               f"sign={'on' if sign else 'off'}, grads {wl.g_dtype}",
                   "n": n, "R": R, "mode": mode, "k": k, "sign": bool(sign), "grad_dtype": wl.g_dtype,
                   "parallelism": f"one shard per GPU x {world}",
                   "l2": "L2 flushed (256 MB write) between steps" if flush else
                   f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB per step)"},
        "achieved_gbs": achieved,
        "hbm_frac_of_peak": achieved / peak,
        "roofline": roof,
        "gpu_launches": K,
        "clocks": sampler.summary(),
        "e2e": e2e,
        "device_fault": fault,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl.name, mode, k, sign, R)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
