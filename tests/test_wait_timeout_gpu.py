"""Failure detection on the device, without a GPU fault.

Every wait of the tile kernels on a load's barrier gives up after a time limit,
sets the library's fault word, waits (bounded) for the copies the warp still has
in flight and returns, so that a copy that never lands cannot hang the GPU.
demo_test_stall_next_launch makes that happen on purpose: the next tile-kernel
launch has its first warp announce 16 bytes more than one of its loads delivers,
so that load's barrier never completes (every copy still lands).  Each test
checks that the fault word reports the give-up exactly once, that the context
stays usable, and that the next normal step still matches the float64 oracle.
"""

import time

import pytest
import torch

import decoupled_momentum_optimizer_gb300 as dm

from parity import check_step

pytestmark = pytest.mark.gpu

FAULT_LOAD_TIMEOUT = 1
N = 32 * (3 * 32 * 32 + 7)  # 97 tiles, the last one ragged


def cuda_normal(n, std, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(n, generator=g, device="cuda") * std


def state(R, seed):
    theta = cuda_normal(N, 2e-2, seed)
    ms = [cuda_normal(N, 1e-2, seed + 1 + r) for r in range(R)]
    gs = [cuda_normal(N, 1e-3, seed + 10 + r) for r in range(R)]
    return theta, ms, gs


def expect_one_timeout():
    t0 = time.perf_counter()
    code = dm.device_fault()  # synchronises: includes the give-up time
    waited = time.perf_counter() - t0
    assert code == FAULT_LOAD_TIMEOUT, code
    assert waited >= 1.0, waited  # the wait ran to its limit (2 s) before giving up
    assert dm.device_fault() == 0  # read and cleared


@pytest.mark.parametrize("path", ["step", "encode", "decode"])
@pytest.mark.parametrize("mode,k,wire", [("demo", 4, "f32"), ("random", 8, "ternary")])
def test_a_load_that_never_lands_is_reported(path, mode, k, wire):
    dm.init(0)
    assert dm.device_fault() == 0
    R = 2
    theta, ms, gs = state(R, 100)
    kw = dict(k=k, mode=mode, sign=True, seed=1, step=0, wire=wire)
    bufs = [dm.payload_buffers(mode, N, k, wire=wire) for _ in range(R)]
    vals = [b[0] for b in bufs]
    idx = [b[1] for b in bufs] if mode == "demo" else None
    if path == "decode":
        for r in range(R):
            dm.encode(gs[r], ms[r], vals[r], idx[r] if idx else None, beta=0.9, **kw)
        torch.cuda.synchronize()
    dm.test_stall_next_launch(0)
    if path == "step":
        dm.step(theta, gs, ms, beta=0.9, lr=1e-2, **kw)
    elif path == "encode":
        dm.encode(gs[0], ms[0], vals[0], idx[0] if idx else None, beta=0.9, **kw)
    else:
        dm.decode_update(theta, vals, idx, lr=1e-2, **{a: b for a, b in kw.items() if a != "sign"})
    expect_one_timeout()
    # the context is still usable and the next step is right
    theta, ms, gs = state(R, 200)
    check_step(theta, ms, gs, k=k, beta=0.9, lr=1e-2, mode=mode, sign=True, seed=1, step=1, wire=wire)
    assert dm.device_fault() == 0


def test_a_cancelled_request_stalls_nothing():
    dm.init(0)
    theta, ms, gs = state(2, 300)
    dm.test_stall_next_launch(0)
    dm.test_stall_next_launch(-1)
    dm.step(theta, gs, ms, k=4, beta=0.9, lr=1e-2, mode="demo", sign=True)
    assert dm.device_fault() == 0


@pytest.mark.parametrize("mode,k,wire,R,item", [
    ("demo", 1, "ternary", 2, 0),   # lane copies of 4-byte units (R <= 4)
    ("demo", 1, "f32", 8, 0),       # lane copies of 16-byte units
    ("demo", 3, "f32", 64, 1),      # groups of 12 replicas by bulk copies: the tile's second of six items
    ("demo", 1, "f32", 64, 0),      # groups of 38 replicas by lane copies: the first of two items (no theta)
    ("random", 4, "f32", 64, 0),    # every replica read directly
])
def test_every_decode_staging_flavour_gives_up_cleanly(mode, k, wire, R, item):
    """The decode's staging flavours each give up the same way: the stalled barrier times out,
    the warp waits for its own copies (bulk or lane copies) and returns, the fault word reads
    1 once, and the next step is right."""
    dm.init(0)
    assert dm.device_fault() == 0
    theta, ms, gs = state(R, 400)
    kw = dict(k=k, mode=mode, seed=1, step=0, wire=wire)
    bufs = [dm.payload_buffers(mode, N, k, wire=wire) for _ in range(R)]
    vals = [b[0] for b in bufs]
    idx = [b[1] for b in bufs] if mode == "demo" else None
    for r in range(R):
        dm.encode(gs[r], ms[r], vals[r], idx[r] if idx else None, beta=0.9, sign=True, **kw)
    torch.cuda.synchronize()
    dm.test_stall_next_launch(item)
    dm.decode_update(theta, vals, idx, lr=1e-2, **kw)
    expect_one_timeout()
    theta, ms, gs = state(R, 500)
    check_step(theta, ms, gs, k=k, beta=0.9, lr=1e-2, mode=mode, sign=True, seed=1, step=1, wire=wire)
    assert dm.device_fault() == 0
    torch.cuda.empty_cache()
