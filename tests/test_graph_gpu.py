"""The entry points under CUDA stream capture.

Every step call makes only kernel launches, event records / waits and
asynchronous copies on the caller's streams, so it can be captured into a CUDA
graph once and replayed (for small shards this removes the host's per-call cost).
The arguments, the step index and the seed included, are fixed at capture
time: a replayed graph repeats the captured step on whatever its buffers hold
when it runs.  Each test captures one step into a graph, then per iteration
refills the gradient buffers and replays it, beside eager calls with the same
arguments on copies of the same state: every result must be bit-identical.
"""

import pytest
import torch

import decoupled_momentum_optimizer_gb300 as dm

from parity import same_bits

pytestmark = pytest.mark.gpu

N = 32 * (32 * 45 + 13)  # 46 tiles, the last ragged
ITERS = 3


@pytest.fixture(scope="module", autouse=True)
def _init():
    dm.init(0)
    yield
    assert dm.device_fault() == 0


def cuda_normal(n, std, seed, dtype=torch.float32):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(n, generator=g, device="cuda") * std).to(dtype)


def grads(R, i, dtype=torch.float32):
    return [cuda_normal(N, 1e-3, 100 * i + r, dtype) for r in range(R)]


def capture(fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def assert_same(a_list, b_list):
    for a, b in zip(a_list, b_list):
        assert same_bits(a, b)


@pytest.mark.parametrize("mode,k,sign,R,wire,bf16", [
    ("demo", 4, True, 2, "f32", False), ("demo", 1, False, 3, "bf16", True), ("random", 8, True, 2, "ternary", False),
    ("stride", 4, False, 2, "f16", False), ("diloco", 1, True, 2, "f32", False),
], ids=lambda v: str(v))
def test_fused_step_replay(mode, k, sign, R, wire, bf16):
    dt = torch.bfloat16 if bf16 else torch.float32
    kw = dict(k=k, beta=0.99, lr=1e-2, mode=mode, sign=sign, seed=11, step=5, diloco_period=2, wire=wire)
    theta = cuda_normal(N, 2e-2, 1)
    ms = [cuda_normal(N, 1e-2, 2 + r) for r in range(R)]
    gbuf = [torch.zeros(N, device="cuda", dtype=dt) for _ in range(R)]
    th_e, ms_e = theta.clone(), [m.clone() for m in ms]
    graph = capture(lambda: dm.step(theta, gbuf, ms, **kw))
    for i in range(ITERS):
        gs = grads(R, i, dt)
        for b, g in zip(gbuf, gs):
            b.copy_(g)
        graph.replay()
        dm.step(th_e, gs, ms_e, **kw)
        torch.cuda.synchronize()
        assert same_bits(theta, th_e)
        assert_same(ms, ms_e)


@pytest.mark.parametrize("mode,k,wire,together", [("demo", 4, "f32", False), ("demo", 2, "ternary", False),
                                                   ("random", 4, "bf16", False), ("demo", 4, "f32", True),
                                                   ("stride", 8, "ternary", True)],
                         ids=lambda v: str(v))
def test_split_path_replay(mode, k, wire, together):
    """R encodes (R calls, or one demo_encode_replicas call, whose later encodes wait for their
    predecessor only at their end) and the decode captured together, against the same calls made
    eagerly."""
    R = 3
    kw = dict(k=k, mode=mode, seed=4, step=2, wire=wire)
    theta = cuda_normal(N, 2e-2, 1)
    ms = [cuda_normal(N, 1e-2, 2 + r) for r in range(R)]
    gbuf = [torch.zeros(N, device="cuda") for _ in range(R)]
    pay = [dm.payload_buffers(mode, N, k, step=2, wire=wire) for _ in range(R)]
    th_e, ms_e = theta.clone(), [m.clone() for m in ms]
    pay_e = [dm.payload_buffers(mode, N, k, step=2, wire=wire) for _ in range(R)]

    def split(th, mm, gg, pp):
        if together:
            dm.encode_replicas(gg, mm, [p[0] for p in pp], [p[1] for p in pp] if mode == "demo" else None,
                               beta=0.99, sign=True, **kw)
        else:
            for r in range(R):
                dm.encode(gg[r], mm[r], pp[r][0], pp[r][1], beta=0.99, sign=True, **kw)
        dm.decode_update(th, [p[0] for p in pp], [p[1] for p in pp] if mode == "demo" else None, lr=1e-2, **kw)

    graph = capture(lambda: split(theta, ms, gbuf, pay))
    for i in range(ITERS):
        gs = grads(R, i)
        for b, g in zip(gbuf, gs):
            b.copy_(g)
        graph.replay()
        split(th_e, ms_e, gs, pay_e)
        torch.cuda.synchronize()
        assert same_bits(theta, th_e)
        assert_same(ms, ms_e)
        for (v, ix), (ve, ixe) in zip(pay, pay_e):
            assert torch.equal(v.view(torch.uint8), ve.view(torch.uint8))
            if ix is not None:
                assert torch.equal(ix.view(torch.uint8), ixe.view(torch.uint8))


@pytest.mark.parametrize("wire,blocks", [("f32", 4), ("ternary", 3)], ids=lambda v: str(v))
def test_pipelined_step_replay(wire, blocks):
    """The pipelined step forks its exchange onto a second stream and joins it back, so the
    whole block schedule lands in one graph; its replay equals the fused step."""
    R, k = 2, 4
    kw = dict(k=k, beta=0.99, lr=1e-2, mode="demo", sign=True, seed=0, step=1, wire=wire)
    comm = torch.cuda.Stream()
    theta = cuda_normal(N, 2e-2, 1)
    ms = [cuda_normal(N, 1e-2, 2 + r) for r in range(R)]
    gbuf = [torch.zeros(N, device="cuda") for _ in range(R)]
    send = [dm.payload_buffers("demo", N, k, wire=wire) for _ in range(R)]
    recv = [dm.payload_buffers("demo", N, k, wire=wire) for _ in range(R)]
    th_e, ms_e = theta.clone(), [m.clone() for m in ms]
    graph = capture(lambda: dm.step_pipelined(theta, gbuf, ms, send, recv, blocks=blocks, comm_stream=comm, **kw))
    for i in range(ITERS):
        gs = grads(R, i)
        for b, g in zip(gbuf, gs):
            b.copy_(g)
        graph.replay()
        dm.step(th_e, gs, ms_e, **kw)
        torch.cuda.synchronize()
        assert same_bits(theta, th_e)
        assert_same(ms, ms_e)


def test_adamw_replay():
    R = 2
    kw = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.05, step=3)
    theta = cuda_normal(N, 2e-2, 1)
    ms = [cuda_normal(N, 1e-3, 2 + r) for r in range(R)]
    vs = [cuda_normal(N, 1e-3, 5 + r).square() for r in range(R)]
    gbuf = [torch.zeros(N, device="cuda") for _ in range(R)]
    th_e, ms_e, vs_e = theta.clone(), [m.clone() for m in ms], [v.clone() for v in vs]
    graph = capture(lambda: dm.adamw_step(theta, gbuf, ms, vs, **kw))
    for i in range(ITERS):
        gs = grads(R, i)
        for b, g in zip(gbuf, gs):
            b.copy_(g)
        graph.replay()
        dm.adamw_step(th_e, gs, ms_e, vs_e, **kw)
        torch.cuda.synchronize()
        assert same_bits(theta, th_e)
        assert_same(ms, ms_e)
        assert_same(vs, vs_e)
