"""bench.py's host logic without a GPU: the reference arm's JSON line, the
algorithmic byte counts the roofline divides by, the comment-insensitive source
hash that keys the committed ncu traffic, the clock-reason decoding, and a loud
failure of the GPU arm on a machine without a GPU.
"""

import importlib.util
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def run_bench(*args, env=None, timeout=600):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          cwd=ROOT, env=e, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = run_bench("--impl", "reference", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["unit"] == "params/s" and d["higher_is_better"] is True and d["value"] > 0
    # value = params per step / seconds per step
    assert abs(d["value"] * d["ms_per_step"] / 1e3 - 4096 * 32) <= 1e-6 * 4096 * 32
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    cfg = d["config"]
    assert cfg["n"] == 1 << 30 and cfg["R"] == 2 and cfg["mode"] == "demo" and cfg["k"] == 4 and cfg["sign"]


def test_reference_arm_other_ranks_do_no_work():
    r = run_bench("--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
                  env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_diloco_runs_time_one_kind_of_step():
    r = run_bench("--impl", "reference", "--mode", "diloco", "--k", "1", "--diloco-period", "4", "--steps", "2",
                  "--warmup", "3")
    assert r.returncode != 0 and "--diloco-period" in r.stderr  # a period that mixes sync and non-sync steps
    for period, words, gain in (("1", "every step a sync step", 32), ("100", "steps between syncs", 24)):
        r = run_bench("--impl", "reference", "--mode", "diloco", "--k", "1", "--diloco-period", period, "--steps", "2",
                      "--warmup", "3")
        assert r.returncode == 0, r.stderr[-2000:]
        d = json.loads(r.stdout)
        assert words in d["config"]["workload"]
        # the config's L2 note counts the step's bytes: R (4 + 8) per parameter, plus 8 for theta on a sync step
        assert f"{gain * (1 << 30) / 1e9:.2f} GB per step" in d["config"]["l2"]


def test_gpu_arm_fails_loudly_without_a_gpu():
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = run_bench("--steps", "3", "--warmup", "3", "--no-e2e", "--no-cpu-baseline", timeout=300)
    assert r.returncode != 0
    assert r.stdout.strip() == ""  # no JSON line from a CPU path


def test_algorithmic_bytes_by_hand(bench):
    # T5-base shard, R = 2, float32 gradients: per element each replica reads g (4) and reads and
    # writes m (8); theta is read and written once (8): 2 * 12 + 8 = 32 bytes per parameter
    assert bench.algorithmic_bytes(222903552, 2, 4, "demo") == 32 * 222903552
    # bf16 gradients, R = 3: 3 * (2 + 8) + 8 = 38
    assert bench.algorithmic_bytes(1024, 3, 2, "random") == 38 * 1024
    # a DiLoCo step that does not synchronise leaves theta untouched
    assert bench.algorithmic_bytes(1024, 2, 4, "diloco", sync=False) == 24 * 1024
    assert bench.algorithmic_bytes(1024, 2, 4, "diloco", sync=True) == 32 * 1024


def test_split_bytes_by_hand(bench):
    n, R = 32 * 1000, 2
    # DeMo k = 4, float32 wire: per chunk 4 values (16 B) + 4 uint8 indices (4 B) = 20 B per replica;
    # each encode writes its payload, the decode reads all R payloads and theta (read + write)
    P = 1000 * 20
    assert bench.split_bytes(n, R, 4, "demo", 4) == R * (n * 12 + P) + R * P + 8 * n
    # ternary wire: 32-chunk tiles, 2 words per value and 5 per index slot, 4 B each
    Pt = 32 * 4 * 2 * 4 + 32 * 4 * 5 * 4  # T = 1000 / 32 rounded up = 32 tiles
    assert bench.split_bytes(n, R, 4, "demo", 4, wire="ternary") == R * (n * 12 + Pt) + R * Pt + 8 * n
    # DiLoCo off a sync step sends nothing and leaves theta alone
    assert bench.split_bytes(n, R, 4, "diloco", 1, sync=False) == R * n * 12


def test_strip_comments_keeps_code_and_literals(bench):
    a = 'int x = 1; // note\n/* block\n comment */ const char* s = "a // b /* c */";\n'
    b = 'int x = 1;   // another note\n\n/* changed */ const char* s = "a // b /* c */";\n'
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert '"a // b /* c */"' in bench.strip_comments(a)
    assert bench.strip_comments(a) != bench.strip_comments(a.replace("x = 1", "x = 2"))
    assert bench.strip_comments("char c = '\\'';  // q\n") == "char c = '\\'';"


def test_ncu_traffic_only_for_the_current_kernel(bench):
    got = bench.ncu_traffic("t5_base", "demo", 4, 2)
    entries = {}
    for line in open(os.path.join(ROOT, "profiles", "ncu_traffic.txt")):
        f = line.split()
        if line.startswith("#") or len(f) < 6:
            continue
        entries[(f[0], f[1], int(f[2]), int(f[3]), f[4])] = float(f[5])
    cur = bench.src_hash()
    assert got == entries.get(("t5_base", "demo", 4, 2, cur))
    assert bench.ncu_traffic("t5_base", "demo", 3, 2) is None  # no entry for k = 3


def test_clock_reasons_decoded(bench):
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.max_mhz = 2070
    cs.samples = [(2070, 0x1), (2062, 0x4), (2070, 0x4 | 0x1), (1980, 0x0)]
    s = cs.summary()
    assert s["reasons"] == ["sw_power_cap"] and s["sm_mhz"] == 2066 and s["samples"] == 4
    cs.samples = [(1500, 0x8 | 0x40)]
    assert cs.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_profile_commands_still_parse(bench, monkeypatch):
    """Every bench command a committed profile summary gives still parses with the current bench.py,
    names a known workload, and runs committed files only."""
    import glob
    import shlex

    from decoupled_momentum_optimizer_gb300 import workloads as W

    found = 0
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read().replace("\\\n", " ")
        for line in text.splitlines():
            if "python bench.py" not in line:
                continue
            words = shlex.split(line.split("python bench.py", 1)[1])
            monkeypatch.setattr(sys, "argv", ["bench.py"] + words)
            args = bench.parse_args()
            W.workload(args.workload)
            assert "_work" not in line, path
            found += 1
    assert found >= 8


def test_sweep_cases_are_valid(bench):
    """Every configuration the sweep measures names a known workload and a valid scheme, k and
    path, so a sweep on the GPU never stops at a malformed case."""
    from decoupled_momentum_optimizer_gb300 import workloads as W

    cases = bench.sweep_cases()
    assert len(cases) > 50
    for name, mode, k, sign, R, paths in cases:
        wl = W.workload(name)
        assert 1 <= R <= 64 and wl.n % 32 == 0
        base = "diloco" if mode.startswith("diloco") else mode
        assert base in ("demo", "random", "stride", "diloco", "adamw")
        if base in ("demo", "random", "stride"):
            assert 1 <= k <= 32
        if base == "stride":
            assert 32 % k == 0
        for p in paths:
            kind = p.split(":")[0]
            assert kind in ("fused", "split", "pipe", "adamw", "graph"), p
            if kind in ("split", "pipe") and ":" in p:
                assert p.split(":")[1] in ("f32", "ternary", "bf16", "f16"), p
                if p.split(":")[1] == "ternary":
                    assert sign, p  # the ternary format carries signed values only
