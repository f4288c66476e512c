"""Every launch shape the library picks, checked once on a small ragged shard.

The fused step is compiled for 6, 8 and 11 warps per SM (each with a small and a
large parameter block), the encode for 6, 8 and 11 (DeMo also for k = 1, 2, 4, 8
at compile time), and the decode for four (warps, staging) shapes (DeMo also for
k = 1, 2, 4, 8); the host picks among them by mode, k, R, gradient dtype
and wire format (DeMo payloads too large for every shape are staged a group
of replicas per item).  DiLoCo steps between syncs go to an elementwise momentum
kernel and sync steps' decode to an elementwise dense decode.  Each case below lands on a different branch of that choice
(noted beside it) and runs the teacher-forced harness of tests/parity.py for
two steps: split and fused bit-identical, payloads, momentum and Q against the
oracle.  The shard has three full 32-chunk tiles and a ragged one of five chunks,
so staged and directly read tiles both occur.
"""

import pytest

import decoupled_momentum_optimizer_gb300 as dm

from test_parity_gpu import run_steps

pytestmark = pytest.mark.gpu

N = 32 * (32 * 3 + 5)


@pytest.fixture(scope="module", autouse=True)
def _init():
    dm.init(0)
    yield
    assert dm.device_fault() == 0


# (mode, k, R, bf16, wire, note): the note names the fused / encode / decode shapes the case takes
CASES = [
    ("stride", 4, 2, False, "f32", "fused 6 warps; encode 11; decode 11 warps"),
    ("stride", 2, 6, True, "f32", "fused 6 warps, large block; encode bf16 6; decode 11"),
    ("diloco", 1, 2, False, "f32", "fused 6 (sync); off-sync steps: momentum kernel; encode 8; dense decode"),
    ("diloco", 1, 5, True, "f32", "momentum kernel, bf16 gradients, replicas in batches of four (4 + 1)"),
    ("diloco", 1, 17, False, "f32", "momentum kernel and fused step with the large parameter block"),
    ("diloco", 1, 2, True, "bf16", "encode bf16 6; 16-bit DiLoCo payload"),
    ("random", 2, 2, False, "f32", "fused 6 (k <= R + 1); encode 6 (k <= 2)"),
    ("random", 3, 2, False, "f32", "encode 8 (k > 2)"),
    ("random", 8, 2, False, "f32", "fused 8; decode 11, every replica staged"),
    ("random", 8, 2, True, "f32", "encode bf16 11"),
    ("random", 8, 5, False, "f32", "fused 8, large block; decode 8 warps / 6 KB"),
    ("random", 3, 3, False, "ternary", "decode ternary bit-planes, k not a power of two"),
    ("demo", 1, 2, False, "f32", "fused 6 (f32 k = 1); encode k-compiled, 6 warps"),
    ("demo", 1, 2, True, "f32", "fused 8 (bf16 k = 1); encode runtime k, 8 warps"),
    ("demo", 2, 2, True, "f32", "encode bf16 gradients, k-compiled, 8 warps"),
    ("demo", 2, 2, False, "f32", "encode f32 gradients, k-compiled, 6 warps"),
    ("demo", 8, 2, True, "bf16", "encode k-compiled, 8 warps; 16-bit payload"),
    ("demo", 5, 2, False, "f32", "fused 8; encode 8; decode scalar entries"),
    ("demo", 6, 2, False, "bf16", "fused 8 (k = 6); 16-bit payload"),
    ("demo", 7, 2, False, "f32", "fused 11 (k = 7); encode 11; decode 10 warps / 3 KB"),
    ("demo", 16, 2, False, "f32", "fused 11; span over 2 KB: decode reads directly"),
    ("demo", 4, 4, False, "f32", "decode 10 warps / 3 KB (R x span = 2560)"),
    ("demo", 4, 6, False, "f32", "fused 8, large block; decode 9 warps / 4.5 KB"),
    ("demo", 4, 9, False, "f32", "decode 8 warps / 6 KB (5760)"),
    ("demo", 4, 10, False, "f32", "decode in groups of three replicas per item (four items per tile)"),
    ("demo", 8, 5, False, "f32", "fused 11, large block; decode one replica per item"),
    ("random", 8, 7, False, "f32", "decode 11 warps, two replicas staged, five direct"),
    ("demo", 4, 2, False, "ternary", "encode ternary 11; decode bit-planes staged"),
]


@pytest.mark.parametrize("mode,k,R,bf16,wire,note", CASES, ids=lambda v: str(v))
def test_launch_shape(mode, k, R, bf16, wire, note):
    sign = wire == "ternary" or mode in ("random", "stride")
    run_steps(N, R, k, mode, sign, 2, g_std=1e-3, period=2 if mode == "diloco" else 8, bf16=bf16, seed=5, wire=wire)


# A shard of 1,501 tiles (the last one ragged) lies between one wave of six-warp CTAs
# (152 x 6 = 912 tiles) and two waves of eight-warp CTAs (2,432): the fused step and the
# encode that would take six warps take eight.  Every 97th chunk is checked against the oracle.
N_SMALL = 32 * (32 * 1500 + 7)
SMALL_CASES = [
    ("demo", 1, 2, False, "f32", "fused and encode (k-compiled k = 1) 6 -> 8 warps"),
    ("stride", 4, 2, False, "f32", "fused 6 -> 8 warps"),
    ("random", 2, 2, False, "f32", "fused 6 -> 8 warps (k <= R + 1)"),
    ("diloco", 1, 2, True, "f32", "fused 6 -> 8 warps (sync step); encode bf16 6 -> 8"),
]


@pytest.mark.parametrize("mode,k,R,bf16,wire,note", SMALL_CASES, ids=lambda v: str(v))
def test_small_shard_shape(mode, k, R, bf16, wire, note):
    import numpy as np

    sign = mode in ("random", "stride") or k == 1
    rows = np.arange(0, N_SMALL // 32, 97)
    run_steps(N_SMALL, R, k, mode, sign, 2, g_std=1e-3, period=2 if mode == "diloco" else 8, bf16=bf16, seed=7,
              wire=wire, rows=rows)
