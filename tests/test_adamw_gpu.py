"""GPU parity of the Decoupled AdamW step against the float64 oracle (and, for
one replica, against torch.optim.AdamW running on the same GPU)."""

import numpy as np
import pytest
import torch

import decoupled_momentum_optimizer_gb300 as dm
import oracle.demo_ref as ref

from parity import chunk_close, f64

pytestmark = pytest.mark.gpu

TOL = 1e-5
KW = dict(beta1=0.9, beta2=0.999, eps=1e-8, lr=1e-3, weight_decay=0.05)


@pytest.fixture(scope="module", autouse=True)
def _init():
    dm.init(0)
    yield
    assert dm.device_fault() == 0


def cuda_normal(n, std, seed, dtype=torch.float32):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(n, generator=g, device="cuda") * std).to(dtype)


def gpu_direction(theta, gs, ms, vs, step):
    """U from the library itself: theta = 0, lr = -1, weight decay 0 gives theta' = U."""
    z = torch.zeros_like(theta)
    dm.adamw_step(z, gs, [m.clone() for m in ms], [v.clone() for v in vs], lr=-1.0, beta1=KW["beta1"],
                  beta2=KW["beta2"], eps=KW["eps"], weight_decay=0.0, step=step)
    return z


@pytest.mark.parametrize("R,bf16,n", [(1, False, 32 * 1000), (2, False, 32 * 1003), (3, True, 32 * 777),
                                      (2, False, 32), (4, False, 32 * 513),
                                      (7, True, 32 * 611)])  # R > 4: replicas in batches of four
def test_adamw_teacher_forced(R, bf16, n):
    theta = cuda_normal(n, 2e-2, 1)
    ms = [torch.zeros(n, device="cuda") for _ in range(R)]
    vs = [torch.zeros(n, device="cuda") for _ in range(R)]
    for t in range(4):
        gs = [cuda_normal(n, 1e-2, 10 * r + t, torch.bfloat16 if bf16 else torch.float32) for r in range(R)]
        U = gpu_direction(theta, gs, ms, vs, t)
        th0, m0, v0, g0 = f64(theta), [f64(m) for m in ms], [f64(v) for v in vs], [f64(g) for g in gs]
        dm.adamw_step(theta, gs, ms, vs, step=t, **KW)
        torch.cuda.synchronize()
        th1, m1, v1, Uo = ref.adamw_step(th0, m0, v0, g0, beta1=KW["beta1"], beta2=KW["beta2"], eps=KW["eps"],
                                         lr=KW["lr"], wd=KW["weight_decay"], step_idx=t)
        for r in range(R):
            assert not chunk_close(f64(ms[r]), m1[r], TOL)[0].any()
            assert not chunk_close(f64(vs[r]), v1[r], TOL)[0].any()
        # the direction: element-wise relative (no cancellation inside one replica's u)
        assert np.abs(f64(U) - Uo).max() <= TOL * np.abs(Uo).max()
        # theta' = theta - lr (U + wd theta) as two fused multiply-adds: the inner one rounds
        # U + wd theta (error <= 2^-24 of it, scaled by lr), the outer one rounds theta'
        inner = f64(U) + ref.f32(KW["weight_decay"]) * th0
        want = th0 - ref.f32(KW["lr"]) * inner
        got = f64(theta)
        bound = np.spacing(np.abs(want).astype(np.float32)) + 2.0 ** -23 * ref.f32(KW["lr"]) * np.abs(inner)
        assert (np.abs(got - want) <= bound).all()


def test_adamw_single_replica_matches_torch_on_gpu():
    n = 32 * 512
    theta = cuda_normal(n, 2e-2, 3)
    p = torch.nn.Parameter(theta.clone())
    opt = torch.optim.AdamW([p], lr=KW["lr"], betas=(KW["beta1"], KW["beta2"]), eps=KW["eps"],
                            weight_decay=KW["weight_decay"], foreach=False)
    m = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    for t in range(5):
        g = cuda_normal(n, 1e-2, 100 + t)
        p.grad = g.clone()
        opt.step()
        dm.adamw_step(theta, [g], [m], [v], step=t, **KW)
    torch.cuda.synchronize()
    assert np.abs(f64(theta) - f64(p.detach())).max() <= 1e-5 * np.abs(f64(p.detach())).max()


def test_adamw_argument_errors():
    n = 64
    t = torch.zeros(n, device="cuda")
    g = torch.zeros(n, device="cuda")
    m = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    with pytest.raises(dm.DemoError):
        dm.adamw_step(t, [g], [m], [v], lr=1e-3, beta1=1.0)
    with pytest.raises(dm.DemoError):
        dm.adamw_step(t, [g], [m], [m], lr=1e-3)  # m and v alias
    with pytest.raises(dm.DemoError):
        dm.adamw_step(t, [g], [m], [v], lr=float("nan"))
