"""Parity over the whole size-sweep grid: every scheme, k in {1, 2, 4, 8} and R in
{1, 2, 8, 64}, sign on, gradients N(0, 1e-3), two teacher-forced steps through the
parity harness (split == fused bit for bit; indices, payloads, momentum, Q and theta
against the float64 oracle).

Each combination runs in both launch regimes the library picks between: a small shard
(about 1,300 chunks, a ragged last tile), where every SM gets a CTA and each warp at most
three tiles, and a 2^24-parameter shard, where one CTA per SM streams HBM with the
per-mode warp count; the large one is checked on a hash-sampled set of chunks (fewer for
many replicas, whose oracle is slower).  DiLoCo uses a sync period of 2, so its two steps
are one step between syncs and one sync step.
"""

import numpy as np
import pytest
import torch

import decoupled_momentum_optimizer_gb300 as dm

from test_parity_gpu import run_steps, sample_rows

pytestmark = pytest.mark.gpu

GRID = [(mode, k, R) for mode in ("demo", "random", "stride") for k in (1, 2, 4, 8) for R in (1, 2, 8, 64)]
GRID += [("diloco", 1, R) for R in (1, 2, 8, 64)]


@pytest.fixture(scope="module", autouse=True)
def _init():
    dm.init(0)
    yield
    assert dm.device_fault() == 0


@pytest.mark.parametrize("regime", ["small", "large"])
@pytest.mark.parametrize("mode,k,R", GRID, ids=lambda v: str(v))
def test_grid_combination(mode, k, R, regime):
    if regime == "small":
        n, rows = 32 * (40 * 32 + 9), None
    else:
        n = 1 << 24
        rows = sample_rows(n // 32, count=4096 if R <= 8 else 384)
    stats = {}
    run_steps(n, R, k, mode, True, 2, g_std=1e-3, seed=17, period=2 if mode == "diloco" else 8, rows=rows,
              stats=stats)
    assert stats["near_tie"] <= max(1, stats["chunks"] // 50)
    torch.cuda.empty_cache()


# Receivers of at most four replicas on shards of at least 16 tiles per warp of the widest
# decode shape run with eight warps where the per-tile work is light (Striding, Random with
# float32 payloads and k <= 4 or k = 1 on two replicas, DeMo k = 4 with float32 payloads on
# two): 2^25- and 2^27-parameter shards, checked on sampled chunks, in every wire format the
# rule covers and in cases it leaves at eleven warps.
LIGHT_DECODES = [("random", 1, 2, "f32", 25), ("random", 4, 4, "f32", 25), ("random", 1, 2, "ternary", 25),
                 ("stride", 4, 2, "bf16", 25), ("stride", 8, 2, "ternary", 25), ("stride", 1, 3, "f16", 25),
                 ("demo", 4, 2, "f32", 25), ("demo", 4, 2, "f32", 27), ("random", 8, 2, "f32", 25), ("stride", 4, 4, "ternary", 25)]


@pytest.mark.parametrize("mode,k,R,wire,log_n", LIGHT_DECODES, ids=lambda v: str(v))
def test_decode_shapes_on_a_large_shard(mode, k, R, wire, log_n):
    n = 1 << log_n
    rows = sample_rows(n // 32, count=2048)
    stats = {}
    run_steps(n, R, k, mode, True, 2, g_std=1e-3, seed=19, rows=rows, stats=stats, wire=wire)
    assert stats["near_tie"] <= max(1, stats["chunks"] // 50)
    torch.cuda.empty_cache()
