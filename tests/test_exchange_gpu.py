"""The replica exchange through NCCL on the GPU, with a process group of one rank.

One GPU can hold only one rank of an NCCL group, so the exchange runs with R = 1:
the rank encodes its replica with the library, the payload goes through a real NCCL
all_gather (DeMo, and formats that do not add) or all-reduce (Random, Striding,
DiLoCo with float32 values), and the library decodes what came back.  The result
must be bit-identical to the fused step with one resident replica.  (Two or more
ranks are covered on the CPU by tests/test_exchange_gloo.py.)
"""

import pytest
import torch
import torch.distributed as dist

import decoupled_momentum_optimizer_gb300 as dm
from decoupled_momentum_optimizer_gb300.exchange import ReplicaExchange

from parity import same_bits

pytestmark = pytest.mark.gpu

N = 32 * (5 * 32 + 11)


@pytest.fixture(scope="module")
def nccl_group():
    dm.init(0)
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, store=dist.HashStore(), device_id=torch.device("cuda", 0))
    yield
    dist.destroy_process_group()


def cuda_normal(n, std, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(n, generator=g, device="cuda") * std


@pytest.mark.parametrize("mode,k,sign,wire,steps", [
    ("demo", 4, True, "f32", (0, 1)), ("demo", 2, False, "bf16", (0, 1)), ("demo", 4, True, "ternary", (0, 1)),
    ("random", 8, True, "f32", (0, 1)), ("stride", 4, False, "f32", (2, 3)), ("stride", 2, True, "f16", (0, 1)),
    ("diloco", 1, False, "f32", (6, 7)), ("diloco", 1, True, "ternary", (6, 7)),
])
def test_one_rank_exchange_equals_fused_step(nccl_group, mode, k, sign, wire, steps):
    ex = ReplicaExchange(N, k, mode, wire=wire, diloco_period=8)
    assert ex.R == 1 and ex.collective == ("all_reduce" if mode != "demo" and wire == "f32" else "all_gather")
    theta, m = cuda_normal(N, 2e-2, 1), cuda_normal(N, 1e-2, 2)
    theta2, m2 = theta.clone(), m.clone()
    for step in steps:
        g = cuda_normal(N, 1e-3, 10 + step)
        ex.step(theta, g, m, beta=0.99, lr=1e-2, sign=sign, seed=4, step=step)
        dm.step(theta2, [g], [m2], k=k, beta=0.99, lr=1e-2, mode=mode, sign=sign, diloco_period=8, seed=4, step=step,
                wire=wire)
        torch.cuda.synchronize()
        assert same_bits(theta, theta2) and same_bits(m, m2)
    assert dm.device_fault() == 0
