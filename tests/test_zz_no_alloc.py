"""The pipelined step for callers that cannot allocate device memory.

Some callers cannot allocate device memory at the moment they step: a training
framework whose caching allocator already holds the whole device, or a runtime
that forbids allocation after start-up.  demo_step_pipelined_static serves them:
it takes the same inputs and outputs as demo_step_pipelined but keeps the send
and receive payload buffers in a fixed array inside the library.  These tests
call it through the C ABI twice in a row and require exactly the result of
demo_step_pipelined with caller-provided buffers, and check that a request too
large for the fixed array is refused before anything runs.
"""

import pytest
import torch

import decoupled_momentum_optimizer_gb300 as dm

from parity import check_pipelined_step

pytestmark = pytest.mark.gpu

ENOSPACE = -6


def cuda_normal(n, std, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(n, generator=g, device="cuda") * std


@pytest.mark.parametrize("mode,k,sign,wire", [("demo", 4, True, "f32"), ("demo", 4, True, "ternary"),
                                              ("random", 8, False, "bf16")])
def test_static_scratch_matches_pipelined_on_two_calls(mode, k, sign, wire):
    dm.init(0)
    n, R = 32 * (31 * 32 + 8), 2
    comm = torch.cuda.Stream()
    theta_a = cuda_normal(n, 2e-2, 1)
    ms_a = [cuda_normal(n, 1e-2, 2 + r) for r in range(R)]
    theta_b, ms_b = theta_a.clone(), [m.clone() for m in ms_a]
    for step in (0, 1):  # two calls in a row, each from the state the previous one left
        gs = [cuda_normal(n, 1e-3, 10 + 2 * step + r) for r in range(R)]
        kw = dict(k=k, beta=0.99, lr=1e-2, mode=mode, sign=sign, seed=7, step=step, wire=wire)
        dm.step_pipelined_static(theta_a, gs, ms_a, blocks=4, comm_stream=comm, **kw)
        send = [dm.payload_buffers(mode, n, k, step=step, wire=wire) for _ in range(R)]
        recv = [dm.payload_buffers(mode, n, k, step=step, wire=wire) for _ in range(R)]
        dm.step_pipelined(theta_b, gs, ms_b, send, recv, blocks=4, comm_stream=comm, **kw)
        torch.cuda.synchronize()
        assert torch.equal(theta_a, theta_b)
        for a, b in zip(ms_a, ms_b):
            assert torch.equal(a, b)
    assert dm.device_fault() == 0


# mode, k, sign, R, wire, steps (two in a row; DiLoCo with period 8: no payload, then a full one)
ORACLE_CASES = [
    ("demo", 4, True, 3, "f32", (0, 1)),
    ("demo", 2, False, 4, "bf16", (0, 1)),
    ("random", 8, True, 3, "ternary", (0, 1)),
    ("stride", 2, True, 5, "f16", (1, 2)),
    ("diloco", 1, False, 3, "f32", (6, 7)),
    ("diloco", 1, True, 2, "ternary", (6, 7)),
]


@pytest.mark.parametrize("mode,k,sign,R,wire,steps", ORACLE_CASES, ids=lambda v: str(v))
def test_static_scratch_matches_oracle(mode, k, sign, R, wire, steps):
    dm.init(0)
    n = 32 * (45 * 32 + 17)  # a ragged last tile
    comm = torch.cuda.Stream()
    theta = cuda_normal(n, 2e-2, 5)
    ms = [cuda_normal(n, 1e-2, 30 + r) for r in range(R)]
    for step in steps:
        gs = [cuda_normal(n, 1e-3, 40 + 7 * r + step) for r in range(R)]
        check_pipelined_step(theta, ms, gs, k=k, beta=0.99, lr=1e-2, mode=mode, sign=sign, seed=11, step=step,
                             period=8, wire=wire, blocks=5, comm=comm, static=True)
    assert dm.device_fault() == 0


def test_static_scratch_refuses_oversize_request():
    dm.init(0)
    n, R = 1 << 25, 2  # DeMo k=4 float32 payloads: 2 x 21 MB > the 32 MiB send half
    theta = torch.ones(n, device="cuda")
    gs = [torch.ones(n, device="cuda") for _ in range(R)]
    ms = [torch.zeros(n, device="cuda") for _ in range(R)]
    with pytest.raises(dm.DemoError) as e:
        dm.step_pipelined_static(theta, gs, ms, k=4, beta=0.9, lr=0.1, mode="demo", sign=True, wire="f32")
    assert e.value.status == ENOSPACE
    torch.cuda.synchronize()
    assert bool((theta == 1).all()) and all(bool((m == 0).all()) for m in ms)
    # the same shard fits once the payload is compact enough (ternary: 2 x 3.7 MB)
    dm.step_pipelined_static(theta, gs, ms, k=4, beta=0.9, lr=0.1, mode="demo", sign=True, wire="ternary")
    torch.cuda.synchronize()
    assert dm.device_fault() == 0
