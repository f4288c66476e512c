"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle.

Sizes span several 32-chunk warp tiles and a ragged last tile; the full-size
model-shaped shards are checked on a sample of chunks (chunks are independent,
so a sample is exact for the chunks it covers).
"""

import os

import numpy as np
import pytest
import torch

import decoupled_momentum_optimizer_gb300 as dm
import oracle.demo_ref as ref
from decoupled_momentum_optimizer_gb300 import workloads as W

from parity import C, check_step, f64, gpu_fused

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _init():
    dm.init(0)
    yield
    assert dm.device_fault() == 0


def cuda_normal(n, std, seed, dtype=torch.float32):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(n, generator=g, device="cuda") * std).to(dtype)


def run_steps(n, R, k, mode, sign, steps, *, beta=0.999, lr=1e-3, g_std=1e-2, seed=0, period=8, bf16=False,
              rows=None, zero_chunks=(), stats=None, wire="f32"):
    theta = cuda_normal(n, 2e-2, 12345)
    ms = [torch.zeros(n, device="cuda") for _ in range(R)]
    for c in zero_chunks:
        theta[c * C:(c + 1) * C] = 0
    for t in range(steps):
        gs = [cuda_normal(n, g_std, 1000 * r + t, torch.bfloat16 if bf16 else torch.float32) for r in range(R)]
        for c in zero_chunks:
            for g in gs:
                g[c * C:(c + 1) * C] = 0
        theta, ms = check_step(theta, ms, gs, k=k, beta=beta, lr=lr, mode=mode, sign=sign, seed=seed, step=t,
                               period=period, rows=rows, stats=stats, wire=wire)
    return theta, ms


# ----------------------------------------------------------------------------
# The 65,536-parameter flat shard: DeMo k=4, sign, R=2, 5 steps, every chunk
# ----------------------------------------------------------------------------

def test_flat64k_demo_teacher_forced():
    stats = {}
    run_steps(65536, 2, 4, "demo", True, 5, g_std=1e-2, stats=stats)
    assert stats["near_tie"] <= stats["chunks"] // 100


def test_flat64k_demo_free_running():
    """Five GPU steps against five oracle steps from the same start (no teacher forcing)."""
    wl = W.workload("flat64k")
    n, R = wl.n, wl.R
    theta0 = W.make_theta0(wl, "cpu")
    streams = [W.GradStream(wl, r, "cpu") for r in range(R)]
    theta = theta0.cuda()
    ms = [torch.zeros(n, device="cuda") for _ in range(R)]
    th_o, ms_o = f64(theta0), [np.zeros(n) for _ in range(R)]
    excl = np.zeros(n // C, dtype=bool)
    for t in range(wl.steps):
        gs = [s.next() for s in streams]
        theta, ms = gpu_fused(theta, ms, [g.cuda() for g in gs], k=4, beta=wl.beta, lr=wl.lr, mode="demo", sign=True,
                              seed=0, step=t, period=8)
        th_o, ms_o, info = ref.step(th_o, ms_o, [f64(g) for g in gs], beta=wl.beta, lr=wl.lr, k=4,
                                    mode=ref.MODE_DEMO, sign=True, step_idx=t)
        excl |= info["near_tie"]
    torch.cuda.synchronize()
    from parity import chunk_close

    d_g = f64(theta) - f64(theta0)
    d_o = th_o - f64(theta0)
    # theta is stored in float32 after every step: allow 5 roundings of |theta| on top of the relative bound
    a, b = d_g.reshape(-1, C), d_o.reshape(-1, C)
    slack = 5 * np.spacing(np.abs(f64(theta)).astype(np.float32)).reshape(-1, C)
    bad = ((np.abs(a - b) > 1e-5 * np.abs(b).max(1, keepdims=True) + slack).any(1)) & ~excl
    assert not bad.any(), f"delta theta differs in {bad.sum()} chunks"
    for r in range(R):
        bad, worst = chunk_close(f64(ms[r]), ms_o[r], 1e-5, excl)
        assert not bad.any(), f"m[{r}] worst {worst}"
    assert excl.sum() <= len(excl) // 100


@pytest.mark.parametrize("mode,k,sign,period", [("demo", 4, False, 8), ("random", 8, True, 8),
                                                ("random", 1, False, 8), ("stride", 4, True, 8),
                                                ("diloco", 1, True, 2)])
def test_flat64k_free_running_other_schemes(mode, k, sign, period):
    """Five free-running GPU steps against five oracle steps for the other schemes and for
    unsigned DeMo: theta's update and every m within 1e-5 per chunk."""
    from parity import chunk_close

    wl = W.workload("flat64k")
    n, R = wl.n, wl.R
    theta0 = W.make_theta0(wl, "cpu")
    streams = [W.GradStream(wl, r, "cpu") for r in range(R)]
    theta = theta0.cuda()
    ms = [torch.zeros(n, device="cuda") for _ in range(R)]
    th_o, ms_o = f64(theta0), [np.zeros(n) for _ in range(R)]
    excl = np.zeros(n // C, dtype=bool)
    for t in range(wl.steps):
        gs = [s.next() for s in streams]
        theta, ms = gpu_fused(theta, ms, [g.cuda() for g in gs], k=k, beta=wl.beta, lr=wl.lr, mode=mode,
                              sign=sign, seed=4, step=t, period=period)
        th_o, ms_o, info = ref.step(th_o, ms_o, [f64(g) for g in gs], beta=wl.beta, lr=wl.lr, k=k,
                                    mode=ref.__dict__["MODE_" + mode.upper()], sign=sign, seed=4, step_idx=t,
                                    period=period)
        excl |= info["near_tie"]
    torch.cuda.synchronize()
    d_g = (f64(theta) - f64(theta0)).reshape(-1, C)
    d_o = (th_o - f64(theta0)).reshape(-1, C)
    slack = 5 * np.spacing(np.abs(f64(theta)).astype(np.float32)).reshape(-1, C)
    bad = ((np.abs(d_g - d_o) > 1e-5 * np.abs(d_o).max(1, keepdims=True) + slack).any(1)) & ~excl
    assert not bad.any(), f"delta theta differs in {bad.sum()} chunks"
    for r in range(R):
        bad, worst = chunk_close(f64(ms[r]), ms_o[r], 1e-5, excl)
        assert not bad.any(), f"m[{r}] worst {worst}"
    if mode != "demo":
        assert not excl.any()  # positions do not depend on values: no near-ties to exclude


# ----------------------------------------------------------------------------
# Every mode, k, sign, R and gradient dtype on a ragged shard (31 tiles + 8 rows)
# ----------------------------------------------------------------------------

RAGGED = 32 * (31 * 32 + 8)

CASES = [
    ("demo", 1, True, 2, False), ("demo", 2, False, 2, False), ("demo", 4, True, 1, False),
    ("demo", 8, False, 3, False), ("demo", 4, True, 2, True), ("demo", 5, True, 2, False),
    ("demo", 16, False, 2, False), ("demo", 32, False, 1, False),
    ("demo", 8, True, 2, False), ("demo", 4, True, 4, False),  # decode stages every replica in 3 KB
    # the DeMo step compiled for k with bfloat16 gradients (R = 5: the many-replica kernels)
    ("demo", 1, False, 2, True), ("demo", 2, True, 3, True), ("demo", 8, True, 5, True), ("demo", 8, False, 2, True),
    ("random", 1, True, 2, False), ("random", 8, False, 2, False), ("random", 8, True, 3, True),
    ("random", 3, False, 1, False), ("random", 32, True, 2, False),
    ("stride", 1, True, 2, False), ("stride", 4, False, 2, False), ("stride", 8, True, 5, True),
    ("stride", 32, False, 1, False),
    ("diloco", 1, True, 2, False), ("diloco", 1, False, 3, True),
]


@pytest.mark.parametrize("mode,k,sign,R,bf16", CASES, ids=lambda v: str(v))
def test_modes_ragged(mode, k, sign, R, bf16):
    steps = 4 if mode == "diloco" else 3
    run_steps(RAGGED, R, k, mode, sign, steps, g_std=1e-3, period=2 if mode == "diloco" else 8, bf16=bf16, seed=7)


def test_many_replicas():
    run_steps(32 * 300, 64, 4, "demo", True, 2, seed=3)
    run_steps(32 * 300, 17, 8, "random", False, 2, seed=3)


# ----------------------------------------------------------------------------
# Edge cases
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n", [32, 64, 96, 32 * 33])
def test_tiny_shards(n):
    for mode, k in (("demo", 4), ("random", 8), ("stride", 4), ("diloco", 1)):
        run_steps(n, 2, k, mode, True, 2, period=2)


def test_zero_chunks_select_lowest_indices():
    n = 32 * 70
    zero = (0, 5, 33, 69)
    theta, ms = run_steps(n, 2, 4, "demo", True, 2, zero_chunks=zero)
    for c in zero:
        assert torch.count_nonzero(theta[c * C:(c + 1) * C]).item() == 0
        for m in ms:
            assert torch.count_nonzero(m[c * C:(c + 1) * C]).item() == 0
    # the payload of an all-zero chunk: indices 0..k-1 (lowest index wins the tie), values 0
    g = torch.zeros(n, device="cuda")
    m = torch.zeros(n, device="cuda")
    vals = torch.full((n // C * 4,), 7.0, device="cuda")
    idx = torch.full((n // C * 4,), 99, dtype=torch.uint8, device="cuda")
    dm.encode(g, m, vals, idx, k=4, beta=0.9, mode="demo", sign=True)
    torch.cuda.synchronize()
    assert (idx.view(-1, 4).cpu() == torch.arange(4, dtype=torch.uint8)).all()
    assert (vals == 0).all()


def test_constant_chunks_keep_dc_first():
    n = 32 * 64
    g = torch.repeat_interleave(torch.linspace(-1, 1, n // C, device="cuda"), C).contiguous()
    m = torch.zeros(n, device="cuda")
    vals = torch.empty(n // C, device="cuda")
    idx = torch.empty(n // C, dtype=torch.uint8, device="cuda")
    dm.encode(g, m, vals, idx, k=1, beta=0.0, mode="demo", sign=False)
    torch.cuda.synchronize()
    nz = g.view(-1, C)[:, 0] != 0
    assert (idx[nz] == 0).all()
    want = g.view(-1, C)[:, 0].double() * np.sqrt(32)
    assert torch.allclose(vals.double(), want, rtol=1e-6, atol=1e-7)
    # the residual keeps only float32 rounding noise
    assert m.abs().max().item() < 1e-6


def test_k32_drains_momentum():
    n = 32 * 100
    g = cuda_normal(n, 1.0, 5)
    m = cuda_normal(n, 1.0, 6)
    vals = torch.empty(n, device="cuda")
    idx = torch.empty(n, dtype=torch.uint8, device="cuda")
    dm.encode(g, m, vals, idx, k=32, beta=0.5, mode="demo", sign=False)
    torch.cuda.synchronize()
    assert m.abs().max().item() < 5e-6  # fp32 round trip of the orthonormal transform
    assert (idx.view(-1, 32).cpu() == torch.arange(32, dtype=torch.uint8)).all()


def test_golden_tiny_step():
    import importlib.util

    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(GOLDEN, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    theta, gs = mg.tiny_inputs()
    th = torch.tensor(theta, dtype=torch.float32, device="cuda")
    g = [torch.tensor(x, dtype=torch.float32, device="cuda") for x in gs]
    ms = [torch.zeros_like(th) for _ in g]
    idx = {}
    th1 = []
    for line in open(os.path.join(GOLDEN, "demo_step_tiny.txt")):
        if line.startswith("idx"):
            head, v = line.split(":")
            _, r, c = head.split()
            idx[(int(r), int(c))] = [int(x) for x in v.split()]
        elif line.startswith("theta1"):
            th1.append(float(line.split()[1]))
    for r in range(2):
        m2 = ms[r].clone()
        vals = torch.empty(4 * 4, device="cuda")
        ix = torch.empty(4 * 4, dtype=torch.uint8, device="cuda")
        dm.encode(g[r], m2, vals, ix, k=4, beta=0.999, mode="demo", sign=True)
        torch.cuda.synchronize()
        for c in range(4):
            assert ix.view(4, 4)[c].tolist() == idx[(r, c)]
    dm.step(th, g, ms, k=4, beta=0.999, lr=1e-3, mode="demo", sign=True)
    torch.cuda.synchronize()
    d_g = f64(th) - theta
    d_o = np.array(th1) - theta
    assert np.abs(d_g - d_o).max() <= 1e-5 * np.abs(d_o).max() + 2 * np.spacing(np.float32(0.05))


# ----------------------------------------------------------------------------
# Determinism, resume, argument errors, guard bands
# ----------------------------------------------------------------------------

def test_deterministic_and_resumable():
    n = 32 * 2000
    R = 2

    def run(split_at=None):
        theta = cuda_normal(n, 2e-2, 1)
        ms = [torch.zeros(n, device="cuda") for _ in range(R)]
        for t in range(5):
            if split_at is not None and t == split_at:
                # save / restore the complete state (theta, m_r; the step counter is explicit)
                saved = (theta.cpu(), [m.cpu() for m in ms])
                theta, ms = saved[0].cuda(), [m.cuda() for m in saved[1]]
            gs = [cuda_normal(n, 1e-2, 100 * r + t) for r in range(R)]
            dm.step(theta, gs, ms, k=4, beta=0.999, lr=1e-3, mode="random", sign=True, seed=9, step=t)
            dm.step(theta, gs, ms, k=2, beta=0.999, lr=1e-3, mode="demo", sign=False, seed=9, step=t)
        torch.cuda.synchronize()
        return theta, ms

    a = run()
    b = run()
    c = run(split_at=2)
    for x in (b, c):
        assert torch.equal(a[0], x[0])
        for r in range(R):
            assert torch.equal(a[1][r], x[1][r])


def test_invalid_arguments_launch_nothing():
    n = 32 * 64
    theta = torch.ones(n, device="cuda")
    g = torch.ones(n, device="cuda")
    m = torch.ones(n, device="cuda")
    snap = theta.clone(), m.clone()
    bad = [
        dict(k=0), dict(k=33), dict(mode="stride", k=3), dict(beta=float("nan")), dict(lr=float("inf")),
    ]
    for kw in bad:
        args = dict(k=4, beta=0.9, lr=0.1, mode="demo", sign=True)
        args.update(kw)
        with pytest.raises(dm.DemoError) as e:
            dm.step(theta, [g], [m], **args)
        assert e.value.status == -1
    with pytest.raises(dm.DemoError) as e:  # misaligned view
        dm.step(theta[1:33], [g[1:33]], [m[1:33]], k=4, beta=0.9, lr=0.1)
    assert e.value.status == -2
    with pytest.raises(dm.DemoError):  # m aliases theta
        dm.step(theta, [g], [theta], k=4, beta=0.9, lr=0.1)
    torch.cuda.synchronize()
    assert torch.equal(theta, snap[0]) and torch.equal(m, snap[1])


def test_decode_repeated_indices_count_every_entry():
    """A malformed DeMo payload whose every index is 0 gives slot 0 of each chunk
    R*k = 160 entries, more than the replica count the kernels tabulate
    reciprocals for.  The decode still takes the mean over every entry, as the
    oracle's scatter-mean counts them, both for the replicas staged through
    shared memory and for the ones read directly, and stays inside its buffers."""
    R, k, n = 40, 4, 32 * 32 * 3 + 32 * 5  # three full tiles and a ragged one
    nc = n // C
    gen = torch.Generator().manual_seed(11)
    vals = [torch.randn(nc, k, generator=gen) * 1e-3 for _ in range(R)]
    idx = torch.zeros(nc * k, dtype=torch.uint8, device="cuda")
    Q = torch.zeros(n, device="cuda")
    dm.decode_update(Q, [v.reshape(-1).cuda() for v in vals], [idx] * R, k=k, lr=-1.0, mode="demo", seed=0, step=0)
    torch.cuda.synchronize()
    _, Qref, Yref, cnt = ref.decode_update(np.zeros(n), [v.double().numpy() for v in vals],
                                           [np.zeros((nc, k), dtype=np.int64)] * R, -1.0, ref.MODE_DEMO)
    assert (cnt[:, 0] == R * k).all()
    scale = np.abs(np.stack([v.double().numpy() for v in vals])).sum((0, 2)) / (R * k)  # mean |entry| per chunk
    err = np.abs(f64(Q).reshape(nc, C) - Qref) / scale[:, None]
    assert err.max() < 1e-5, err.max()


def test_binding_refuses_mixed_devices():
    """A call whose tensors are not all on one CUDA device is refused before any launch."""
    n = 32 * 64
    theta = cuda_normal(n, 2e-2, 1)
    g = cuda_normal(n, 1e-3, 2)
    with pytest.raises(ValueError):
        dm.step(theta, [g], [torch.zeros(n)], k=4, beta=0.9, lr=0.1)
    with pytest.raises(ValueError):
        dm.step(theta.cpu(), [g], [torch.zeros(n, device="cuda")], k=4, beta=0.9, lr=0.1)


def test_binding_refuses_other_gradient_dtypes():
    """Gradients are float32 or bfloat16; float16 ones are refused by every entry point, not read as float32."""
    n = 32 * 64
    theta = cuda_normal(n, 2e-2, 1)
    g = cuda_normal(n, 1e-3, 2).half()
    m = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    vals, idx = dm.payload_buffers("demo", n, 4)
    with pytest.raises(TypeError):
        dm.step(theta, [g], [m], k=4, beta=0.9, lr=0.1)
    with pytest.raises(TypeError):
        dm.encode(g, m, vals, idx, k=4, beta=0.9)
    with pytest.raises(TypeError):
        dm.adamw_step(theta, [g], [m], [v], lr=1e-3)
    with pytest.raises(TypeError):
        dm.step_pipelined(theta, [g], [m], [(vals, idx)], [(vals, idx)], k=4, beta=0.9, lr=0.1)
    with pytest.raises(TypeError):
        dm.step_pipelined_static(theta, [g], [m], k=4, beta=0.9, lr=0.1)
    torch.cuda.synchronize()
    assert (m == 0).all() and (v == 0).all()


def test_guard_bands_untouched():
    n = 32 * (64 + 5)
    pad = 4096 // 4
    big_t = torch.full((n + 2 * pad,), 12345.0, device="cuda")
    big_m = torch.full((n + 2 * pad,), -777.0, device="cuda")
    theta = big_t[pad:pad + n]
    m = big_m[pad:pad + n]
    theta.copy_(cuda_normal(n, 2e-2, 2))
    m.zero_()
    g = cuda_normal(n, 1e-2, 3)
    for mode, k in (("demo", 4), ("random", 8), ("stride", 8), ("diloco", 1)):
        for t in range(2):
            dm.step(theta, [g], [m], k=k, beta=0.9, lr=0.1, mode=mode, sign=True, step=t, diloco_period=2)
    torch.cuda.synchronize()
    assert (big_t[:pad] == 12345.0).all() and (big_t[pad + n:] == 12345.0).all()
    assert (big_m[:pad] == -777.0).all() and (big_m[pad + n:] == -777.0).all()


# ----------------------------------------------------------------------------
# Full-size model-shaped shards, sampled chunks, in the bench's launch setup
# ----------------------------------------------------------------------------

def sample_rows(nc, extra=(), count=4096):
    rows = {ref.index_hash(0xC0FFEE, 0, i, 0) % nc for i in range(count)}
    rows |= {0, nc - 1} | set(extra)
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("name", ["t5_base", "vit_b16", "olmo2_1b_half"])
def test_model_shards_sampled(name):
    """Every run of the workload for its configured number of steps (T5-base 20, the others 10)."""
    wl = W.workload(name)
    n, R = wl.n, wl.R
    rows = sample_rows(n // C, wl.layout.pad_chunks())
    theta0 = W.make_theta0(wl, "cuda")
    stats = {}
    for mode, k, sign in wl.runs:
        theta = theta0.clone()
        ms = [torch.zeros(n, device="cuda") for _ in range(R)]
        streams = [W.GradStream(wl, r, "cuda") for r in range(R)]
        for t in range(wl.steps):
            gs = [s.next() for s in streams]
            theta, ms = check_step(theta, ms, gs, k=k, beta=wl.beta, lr=wl.lr, mode=mode, sign=sign, step=t,
                                   rows=rows, stats=stats)
        del ms
        torch.cuda.empty_cache()
    assert stats["near_tie"] <= stats["chunks"] // 100


@pytest.mark.parametrize("n,R,mode,k", [(1 << 30, 2, "demo", 4), (1 << 28, 8, "random", 8)])
def test_largest_shards_sampled(n, R, mode, k):
    """The largest shards of the size sweep, one step, on sampled chunks."""
    rows = sample_rows(n // C)
    theta = cuda_normal(n, 2e-2, 5)
    ms = [cuda_normal(n, 1e-3, 6 + r) for r in range(R)]
    gs = [cuda_normal(n, 1e-3, 20 + r) for r in range(R)]
    check_step(theta, ms, gs, k=k, beta=0.999, lr=1e-3, mode=mode, sign=True, step=3, rows=rows)
    del theta, ms, gs
    torch.cuda.empty_cache()
