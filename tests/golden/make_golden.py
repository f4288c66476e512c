"""Write the oracle-derived regression fixtures in this folder.

Calls only ``oracle/``.  The inputs are closed-form (no random generator), so
the fixtures are reproducible on any machine:

* ``random_positions_seed0.txt``: Random-scheme positions for seed 0, steps
  0..2, chunks 0..3 and 2^20 - 1, k = 8, in draw order.
* ``demo_step_tiny.txt``: one DeMo step (k = 4, sign on, R = 2) on a 4-chunk
  shard with m_0 = 0, g_r[i] = sin(0.37 i + r) / 100, theta_0[i] = cos(0.11 i) / 50,
  beta = 0.999, lr = 1e-3: the kept indices of each replica and theta_1.

Run ``python tests/golden/make_golden.py`` from the repository root.
"""

import math
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle.demo_ref as ref  # noqa: E402


def tiny_inputs(R=2, nchunks=4):
    n = nchunks * ref.CHUNK
    i = np.arange(n)
    gs = [np.array([float(np.float32(math.sin(0.37 * k + r) / 100.0)) for k in i]) for r in range(R)]
    theta = np.array([float(np.float32(math.cos(0.11 * k) / 50.0)) for k in i])
    return theta, gs


def main():
    with open(os.path.join(HERE, "random_positions_seed0.txt"), "w") as f:
        f.write("# written by tests/golden/make_golden.py from oracle.random_positions\n")
        f.write("# seed step chunk : positions (k = 8, draw order)\n")
        for step in range(3):
            for chunk in (0, 1, 2, 3, (1 << 20) - 1):
                pos = ref.random_positions(0, step, chunk, 8)
                f.write(f"0 {step} {chunk} : {' '.join(map(str, pos))}\n")

    theta, gs = tiny_inputs()
    ms = [np.zeros_like(theta) for _ in gs]
    th1, _, info = ref.step(theta, ms, gs, beta=0.999, lr=1e-3, k=4, mode=ref.MODE_DEMO, sign=True)
    with open(os.path.join(HERE, "demo_step_tiny.txt"), "w") as f:
        f.write("# written by tests/golden/make_golden.py from oracle.step (DeMo, k=4, sign, R=2)\n")
        for r, e in enumerate(info["encodes"]):
            for c in range(e["idx"].shape[0]):
                f.write(f"idx {r} {c} : {' '.join(map(str, e['idx'][c]))}\n")
        for v in th1:
            f.write(f"theta1 {float(v)!r}\n")


if __name__ == "__main__":
    main()
