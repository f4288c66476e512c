"""CPU checks of the CUDA side's generated DCT-IV blocks (not the oracle).

The generator records each block as a straight-line float32 program; here the
program runs in numpy float32 and is compared with the DCT-IV matrix written
out from its definition, and the committed header must equal the generator's
output (so the kernels compile exactly the checked arithmetic).
"""

import importlib.util
import math
import os

import numpy as np
import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "decoupled_momentum_optimizer_gb300", "csrc")


def gen():
    spec = importlib.util.spec_from_file_location("gen_dct_factors", os.path.join(CSRC, "gen_dct_factors.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


@pytest.mark.parametrize("M", [16, 8, 4, 2])
def test_block_matches_dct4_definition(M):
    P = gen().blocks()[M]
    x = np.random.default_rng(M).standard_normal((2000, M)).astype(np.float32)
    S = np.array([[0.25 * math.cos(math.pi * (2 * n + 1) * (2 * j + 1) / (4 * M)) for n in range(M)]
                  for j in range(M)])
    want = x.astype(np.float64) @ S.T
    got = P.evaluate(x)
    err = np.abs(got - want).max(1) / np.abs(want).max(1)
    assert err.max() < 1e-6
    # an impulse reproduces one column of the matrix
    for n in range(M):
        e = np.zeros((1, M), dtype=np.float32)
        e[0, n] = 1.0
        assert np.abs(P.evaluate(e)[0] - S[:, n]).max() < 1e-7


def test_flop_counts():
    b = gen().blocks()
    assert [b[M].flops() for M in (16, 8, 4, 2)] == [116, 44, 16, 4]


def test_committed_header_is_generated():
    import io

    g = gen()
    buf = io.StringIO()
    g.emit(buf)
    assert open(os.path.join(CSRC, "dct32_factors.cuh")).read() == buf.getvalue()
