"""Forty configurations drawn with a fixed seed, each for two steps through the
parity harness (split == fused bit for bit; payloads, momentum and Q against the
oracle).  They mix every scheme with valid k, R from 1 to 17, every wire format,
both gradient dtypes and shards from 1 to 1,000 chunks (whole and ragged tiles),
so that combinations the hand-picked cases miss are exercised too."""

import numpy as np
import pytest

import decoupled_momentum_optimizer_gb300 as dm

from test_parity_gpu import run_steps

pytestmark = pytest.mark.gpu


def draw_configs(count=40, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        mode = str(rng.choice(["demo", "random", "stride", "diloco"]))
        if mode == "stride":
            k = int(rng.choice([1, 2, 4, 8, 16, 32]))
        elif mode == "diloco":
            k = 1
        else:
            k = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16, 32]))
        R = int(rng.choice([1, 2, 2, 3, 5, 9, 17]))
        wire = str(rng.choice(["f32", "f32", "bf16", "f16", "ternary"]))
        sign = True if wire == "ternary" else bool(rng.integers(0, 2))
        bf16 = bool(rng.integers(0, 2))
        nc = int(rng.choice([1, 7, 31, 32, 33, 63, 64, 65, 100, 1000]))
        out.append((mode, k, R, wire, sign, bf16, nc))
    return out


@pytest.fixture(scope="module", autouse=True)
def _init():
    dm.init(0)
    yield
    assert dm.device_fault() == 0


@pytest.mark.parametrize("mode,k,R,wire,sign,bf16,nc", draw_configs(), ids=lambda v: str(v))
def test_random_config(mode, k, R, wire, sign, bf16, nc):
    run_steps(32 * nc, R, k, mode, sign, 2, g_std=1e-3, period=2 if mode == "diloco" else 8, bf16=bf16, seed=9,
              wire=wire)
