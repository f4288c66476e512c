"""The effect of 16-bit payload values on the step, measured with the float64 oracle.

The pages report that sending float32 rather than fp16 values matters for DeMo
and Random ("3. Sign function and hyperparameter analysis", communication
precision).  With the sign function on, every sent value is -1, 0 or +1, which
bf16 and fp16 hold exactly, so the format changes nothing (checked below).
With the sign off, the receiver decodes values rounded to nearest even; the
senders' momentum and error feedback use the unrounded values, so only Q (and
through it theta) moves.  This test measures by how much, over a ten-step
trajectory, and pins the measurement between bounds that follow from the
formats' unit roundoff u (bf16: 2^-8, fp16: 2^-11; relative rounding error
uniform in [-u, u] for values in the normal range, so its RMS is u / sqrt(3)):
a lower bound (the rounding is really there) and an upper bound (it is the
only difference).  The CUDA path reproduces the oracle's rounded decode value
for value (tests/test_wire_gpu.py), so these figures hold for it too.
"""

import numpy as np
import pytest

import oracle.demo_ref as ref

N = 32 * 512
R = 2
STEPS = 10
U = {ref.WIRE_BF16: 2.0 ** -8, ref.WIRE_F16: 2.0 ** -11}


def trajectory(mode, k, sign, wire, seed=3):
    rng = np.random.default_rng(seed)
    theta = rng.standard_normal(N) * 2e-2
    theta0 = theta.copy()
    ms = [np.zeros(N) for _ in range(R)]
    Qs = []
    for t in range(STEPS):
        gs = [rng.standard_normal(N).astype(np.float32).astype(np.float64) * 1e-3 for _ in range(R)]
        theta, ms, info = ref.step(theta, ms, gs, beta=0.999, lr=1e-3, k=k, mode=mode, sign=sign, seed=11,
                                   step_idx=t, wire=wire)
        Qs.append(info["Q"].reshape(-1))
    return theta0, theta, ms, Qs


def rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("mode,k", [(ref.MODE_DEMO, 4), (ref.MODE_RANDOM, 8)])
def test_sixteen_bit_payload_effect(mode, k):
    th0, th32, ms32, Q32 = trajectory(mode, k, False, ref.WIRE_F32)
    report = []
    for wire, u in U.items():
        _, thw, msw, Qw = trajectory(mode, k, False, wire)
        for a, b in zip(msw, ms32):
            assert np.array_equal(a, b)  # the senders' state never sees the rounding
        q = [rel(a, b) for a, b in zip(Qw, Q32)]
        th = rel(thw - th0, th32 - th0)
        report.append((wire, max(q), th))
        # per-step Q: RMS relative rounding error of the decoded values, between u/20 and u
        assert u / 20 < min(q) and max(q) < u, (wire, q)
        # the update over the trajectory: consecutive Q are strongly correlated (momentum),
        # and so are their rounding errors, so it deviates by about as much as one step's Q
        assert u / 50 < th < u, (wire, th)
    print(f"\n{ref.MODE_NAMES[mode]} k={k}, sign off, {STEPS} steps: "
          + "; ".join(f"{'bf16' if w == ref.WIRE_BF16 else 'fp16'}: max per-step |dQ|/|Q| = {a:.2e}, "
                      f"|d(theta - theta0)|/|theta - theta0| = {b:.2e}" for w, a, b in report))


@pytest.mark.parametrize("mode,k", [(ref.MODE_DEMO, 4), (ref.MODE_RANDOM, 8)])
def test_signed_payload_is_exact_in_sixteen_bits(mode, k):
    th0, th32, _, Q32 = trajectory(mode, k, True, ref.WIRE_F32)
    for wire in U:
        _, thw, _, Qw = trajectory(mode, k, True, wire)
        assert np.array_equal(thw, th32)
        assert all(np.array_equal(a, b) for a, b in zip(Qw, Q32))
