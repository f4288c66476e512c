"""The split path with its exchange overlapped on a second stream
(demo_step_pipelined): teacher-forced against the float64 oracle for every
scheme and wire format with 1, 3 and 64 blocks (ragged last blocks included),
and bit-identical to the fused step."""

import pytest
import torch

import decoupled_momentum_optimizer_gb300 as dm

from parity import check_pipelined_step, same_bits

pytestmark = pytest.mark.gpu

RAGGED = 32 * (31 * 32 + 8)
N64 = 32 * (63 * 32 + 5)  # 63 full tiles and a 64th of 5 chunks: 64 blocks are one tile each


@pytest.fixture(scope="module", autouse=True)
def _init():
    dm.init(0)
    yield
    assert dm.device_fault() == 0


def cuda_normal(n, std, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(n, generator=g, device="cuda") * std


CASES = [
    ("demo", 4, True, 2, "f32", 1), ("demo", 4, True, 2, "f32", 3), ("demo", 4, True, 2, "ternary", 8),
    ("demo", 1, False, 3, "bf16", 5), ("demo", 8, False, 2, "f16", 64),
    ("random", 8, True, 2, "f32", 4), ("random", 1, True, 3, "ternary", 7), ("stride", 4, False, 2, "bf16", 2),
    ("diloco", 1, True, 2, "ternary", 3), ("diloco", 1, False, 2, "f32", 4),
    ("demo", 4, True, 4, "f32", 5),  # decode stages all four replicas (10 warps, 3 KB) in every block
    ("demo", 3, True, 2, "ternary", 4),  # ternary spans of k = 3 are not 16-byte multiples: read directly
]


@pytest.mark.parametrize("mode,k,sign,R,wire,blocks", CASES, ids=lambda v: str(v))
def test_pipelined_equals_fused(mode, k, sign, R, wire, blocks):
    n = RAGGED
    comm = torch.cuda.Stream()
    theta0 = cuda_normal(n, 2e-2, 1)
    m0 = [cuda_normal(n, 1e-2, 10 + r) for r in range(R)]
    for step in (0, 1, 7):  # DiLoCo (period 8) syncs on step 7 only
        gs = [cuda_normal(n, 1e-3, 20 + 3 * r + step) for r in range(R)]
        th_f, ms_f = theta0.clone(), [m.clone() for m in m0]
        dm.step(th_f, gs, ms_f, k=k, beta=0.99, lr=1e-2, mode=mode, sign=sign, seed=3, step=step, wire=wire)
        th_p, ms_p = theta0.clone(), [m.clone() for m in m0]
        send = [dm.payload_buffers(mode, n, k, step=step, wire=wire) for _ in range(R)]
        recv = [dm.payload_buffers(mode, n, k, step=step, wire=wire) for _ in range(R)]
        dm.step_pipelined(th_p, gs, ms_p, send if send[0][0] is not None else None,
                          recv if recv[0][0] is not None else None, k=k, beta=0.99, lr=1e-2, mode=mode, sign=sign,
                          seed=3, step=step, wire=wire, blocks=blocks, comm_stream=comm)
        torch.cuda.synchronize()
        assert same_bits(th_f, th_p)
        for a, b in zip(ms_f, ms_p):
            assert same_bits(a, b)


# mode, k, sign, R, wire, blocks, n, steps (two in a row; DiLoCo with period 8: off-sync, then sync)
ORACLE_CASES = [
    ("demo", 4, True, 2, "f32", 1, RAGGED, (0, 1)),
    ("demo", 4, True, 3, "ternary", 64, N64, (0, 1)),
    ("demo", 2, False, 2, "bf16", 3, RAGGED, (0, 1)),
    ("demo", 8, False, 2, "f16", 64, N64, (0, 1)),
    ("demo", 1, True, 5, "f32", 3, RAGGED, (0, 1)),  # R = 5: the kernels' large parameter block
    ("random", 8, True, 2, "ternary", 3, RAGGED, (0, 1)),
    ("random", 1, False, 3, "f32", 64, N64, (0, 1)),
    ("stride", 4, True, 2, "bf16", 1, RAGGED, (2, 3)),
    ("diloco", 1, False, 2, "f32", 3, RAGGED, (6, 7)),
    ("diloco", 1, True, 3, "ternary", 64, N64, (6, 7)),
]


@pytest.mark.parametrize("mode,k,sign,R,wire,blocks,n,steps", ORACLE_CASES, ids=lambda v: str(v))
def test_pipelined_matches_oracle(mode, k, sign, R, wire, blocks, n, steps):
    comm = torch.cuda.Stream()
    theta = cuda_normal(n, 2e-2, 1)
    ms = [cuda_normal(n, 1e-2, 10 + r) for r in range(R)]
    ties = 0
    for step in steps:
        gs = [cuda_normal(n, 1e-3, 20 + 3 * r + step) for r in range(R)]
        ties += check_pipelined_step(theta, ms, gs, k=k, beta=0.99, lr=1e-2, mode=mode, sign=sign, seed=3,
                                     step=step, period=8, wire=wire, blocks=blocks, comm=comm)
    assert ties <= 0.01 * (n // 32) * len(steps)


def test_pipelined_argument_errors():
    n = 32 * 64
    th = torch.zeros(n, device="cuda")
    g = torch.zeros(n, device="cuda")
    m = torch.zeros(n, device="cuda")
    send = [dm.payload_buffers("demo", n, 4)]
    with pytest.raises(dm.DemoError):
        dm.step_pipelined(th, [g], [m], send, send, k=4, beta=0.9, lr=0.1, blocks=0)
    with pytest.raises(dm.DemoError):
        dm.step_pipelined(th, [g], [m], send, send, k=4, beta=0.9, lr=0.1, blocks=65)
    with pytest.raises(dm.DemoError):
        dm.step_pipelined(th, [g], [m], None, None, k=4, beta=0.9, lr=0.1, blocks=2)


def test_pipelined_from_two_host_threads():
    """Two host threads step their own shards through demo_step_pipelined at the same time, each
    on its own pair of streams (the binding releases the interpreter lock during the call, so the
    two enqueue sequences overlap on the host).  The library serialises each call's use of its
    event pool; every shard must end bit-identical to the same steps taken by the fused path."""
    import threading

    n, R, k, steps = RAGGED, 2, 4, 12
    kw = dict(k=k, beta=0.99, lr=1e-2, mode="demo", sign=True, seed=0, wire="f32")
    results, errors = {}, []

    def state(tid):
        theta = cuda_normal(n, 2e-2, 100 + tid)
        ms = [cuda_normal(n, 1e-2, 200 + 10 * tid + r) for r in range(R)]
        gsets = [[cuda_normal(n, 1e-3, 300 + 100 * tid + 10 * t + r) for r in range(R)] for t in range(steps)]
        return theta, ms, gsets

    states = [state(tid) for tid in range(2)]
    torch.cuda.synchronize()

    def worker(tid):
        try:
            theta, ms, gsets = states[tid]
            theta, ms = theta.clone(), [m.clone() for m in ms]
            cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
            send = [dm.payload_buffers("demo", n, k) for _ in range(R)]
            recv = [dm.payload_buffers("demo", n, k) for _ in range(R)]
            torch.cuda.synchronize()
            for t in range(steps):
                dm.step_pipelined(theta, gsets[t], ms, send, recv, step=t, blocks=7, stream=cs, comm_stream=xs, **kw)
            cs.synchronize()
            results[tid] = (theta, ms)
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(tid,)) for tid in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for tid in range(2):
        theta, ms, gsets = states[tid]
        theta, ms = theta.clone(), [m.clone() for m in ms]
        for t in range(steps):
            dm.step(theta, gsets[t], ms, step=t, **kw)
        torch.cuda.synchronize()
        assert same_bits(results[tid][0], theta)
        for a, b in zip(results[tid][1], ms):
            assert same_bits(a, b)
