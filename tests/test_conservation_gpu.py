"""A property that holds at any size, checked on EVERY element of full-size shards.

With the sign off and beta = 1 a step splits m + g exactly into the new momentum
and the sent component q (the chunk transform is orthonormal, so for DeMo the
parameter-domain q is the inverse transform of the kept coefficients), and the
replicas of Random, Striding and DiLoCo send the same slots, so Q is the plain
mean of the replicas' q (DeMo is taken with one replica).  Over T steps the
momenta telescope ("DeToNATION" notes, FlexDeMo Algorithm 1, from the momentum
accumulation to the parameter update):

    theta_T = theta_0 - lr / R * sum_r (m_r,0 + sum_t g_r,t - m_r,T).

The float32 step rounds theta once per step (half an ulp), and the transform
round trip adds about 2^-24 of the chunk's norm to each step's Q and new m; the
tolerance is T ulps of theta plus 1e-5 of lr times T times the chunk's norm bound
sqrt(32) * max_chunk(|m_0| + sum_t |g_t|).  A wrong update (a missing 1/R, a
dropped gradient, lr applied twice, a momentum not carried) is off by lr |g|,
orders above it.  The oracle cannot run these sizes; its own pins check the same
identity on small shards.
"""

import math

import numpy as np
import pytest
import torch

import decoupled_momentum_optimizer_gb300 as dm
from decoupled_momentum_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

C = 32
T = 3


@pytest.fixture(scope="module", autouse=True)
def _init():
    dm.init(0)
    yield
    assert dm.device_fault() == 0


def ulp32(x):
    x = x.abs().float()
    return (torch.nextafter(x, torch.full_like(x, math.inf)) - x).double()


@pytest.mark.parametrize("name,mode,k,R", [
    ("t5_base", "demo", 4, 1),  # the bench's shard, the step kernel the bench times (sign is a runtime flag)
    ("t5_base", "random", 8, 2),
    ("olmo2_1b_half", "demo", 1, 1),  # bfloat16 gradients
    ("vit_b16", "stride", 4, 2),
    ("vit_b16", "diloco", 1, 2),  # period 2: a sync step and an off-sync step
], ids=lambda v: str(v))
def test_conservation_full_shard(name, mode, k, R):
    wl = W.workload(name)
    n = wl.n
    theta = W.make_theta0(wl, "cuda")
    theta0 = theta.clone()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    ms = [torch.randn(n, generator=gen, device="cuda") * (3 * wl.g_std) for _ in range(R)]
    m0 = [m.clone() for m in ms]
    streams = [W.GradStream(wl, r, "cuda") for r in range(R)]
    gsum = [torch.zeros(n, device="cuda", dtype=torch.float64) for _ in range(R)]
    gabs = torch.zeros(n, device="cuda", dtype=torch.float64)
    for t in range(T):
        gs = [s.next() for s in streams]
        dm.step(theta, gs, ms, k=k, beta=1.0, lr=wl.lr, mode=mode, sign=False, seed=9, step=t, diloco_period=2)
        for r in range(R):
            gd = gs[r].double()
            gsum[r] += gd
            gabs += gd.abs()
        del gs
    torch.cuda.synchronize()
    lr32 = float(np.float32(wl.lr))
    S = torch.zeros(n, device="cuda", dtype=torch.float64)
    for r in range(R):
        S += m0[r].double() + gsum[r] - ms[r].double()
    want = theta0.double() - (lr32 / R) * S
    err = (theta.double() - want).abs()
    bound = sum(m.double().abs() for m in m0) + gabs
    chunk_bound = bound.view(-1, C).amax(1, keepdim=True).expand(-1, C).reshape(-1) * math.sqrt(C)
    tol = T * torch.maximum(ulp32(theta), ulp32(theta0)) + 1e-5 * lr32 * T * chunk_bound
    bad = err > tol
    assert not bad.any(), f"{int(bad.sum())} of {n} elements off (worst {float((err / tol).max()):.3g} x tol)"
    # the check is not vacuous: lr applied twice would fail it on nearly every element that was
    # sent at least once (elsewhere theta stays bit-identical, and m must then hold m_0 + sum g)
    moved = theta != theta0
    assert float(moved.double().mean()) > 0.3
    wrong = (theta.double() - (theta0.double() - (2 * lr32 / R) * S)).abs()
    assert float((wrong > tol)[moved].double().mean()) > 0.9
