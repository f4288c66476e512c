"""GPU parity of the payload wire formats (ternary bit-planes, bf16, fp16).

Every case runs the teacher-forced harness of tests/parity.py with the wire
format (split path with the compact payload == fused path, bit for bit; the
decoded payload against the oracle), plus exact checks of the ternary words
against the oracle's own packing and of the ternary decode against the float32
decode of the same signed payload.
"""

import numpy as np
import pytest
import torch

import decoupled_momentum_optimizer_gb300 as dm
import oracle.demo_ref as ref

from parity import C, f64
from test_parity_gpu import RAGGED, cuda_normal, run_steps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _init():
    dm.init(0)
    yield
    assert dm.device_fault() == 0


CASES = [
    ("demo", 4, True, 2, "ternary"), ("demo", 1, True, 3, "ternary"), ("demo", 8, True, 2, "ternary"),
    ("demo", 5, True, 2, "ternary"),
    ("random", 8, True, 2, "ternary"), ("stride", 4, True, 2, "ternary"), ("diloco", 1, True, 2, "ternary"),
    ("demo", 4, False, 2, "bf16"), ("demo", 2, True, 2, "bf16"), ("demo", 8, False, 2, "f16"),
    ("demo", 3, False, 2, "f16"),
    ("random", 8, False, 2, "bf16"), ("random", 1, False, 3, "f16"), ("stride", 8, False, 2, "bf16"),
    ("diloco", 1, False, 2, "bf16"), ("diloco", 1, False, 2, "f16"),
]


@pytest.mark.parametrize("mode,k,sign,R,wire", CASES, ids=lambda v: str(v))
def test_wire_ragged(mode, k, sign, R, wire):
    steps = 4 if mode == "diloco" else 3
    run_steps(RAGGED, R, k, mode, sign, steps, g_std=1e-3, period=2 if mode == "diloco" else 8, seed=11, wire=wire)


# Receivers of many replicas in the compact formats: each staging method of the decode
# (spans staged whole or a group of replicas per item, moved by bulk or lane copies; DeMo
# payloads read directly, several replicas at a time) with a ragged last tile.
MANY_CASES = [
    ("demo", 4, True, 64, "ternary"), ("demo", 8, True, 33, "ternary"), ("demo", 1, True, 40, "ternary"),
    ("demo", 1, False, 64, "bf16"), ("demo", 2, False, 64, "bf16"), ("demo", 4, False, 64, "bf16"),
    ("demo", 8, False, 17, "f16"), ("demo", 3, False, 40, "f16"), ("demo", 4, False, 5, "bf16"),
    ("random", 4, False, 64, "bf16"), ("random", 8, False, 20, "f16"), ("stride", 4, True, 64, "ternary"),
    ("stride", 4, False, 8, "bf16"), ("random", 2, True, 37, "ternary"), ("demo", 5, True, 30, "f32"),
    # ternary spans that are not 16-byte multiples, staged by 4-byte lane copies: R <= 4, R > 4
    # whole, and in groups (k = 7, R = 50)
    ("demo", 2, True, 4, "ternary"), ("random", 3, True, 2, "ternary"), ("stride", 1, True, 3, "ternary"),
    ("demo", 3, True, 6, "ternary"), ("demo", 7, True, 50, "ternary"),
]


@pytest.mark.parametrize("mode,k,sign,R,wire", MANY_CASES, ids=lambda v: str(v))
def test_wire_many_replicas(mode, k, sign, R, wire):
    run_steps(RAGGED, R, k, mode, sign, 2, g_std=1e-3, seed=23, wire=wire)
    torch.cuda.empty_cache()


# DiLoCo with many replicas in every format, on a shard whose chunk count leaves a ragged last
# tile (1001 chunks) and whose groups of four parameters leave a ragged last row of every
# elementwise unit: the sync step's dense decode (the ternary format's per-chunk byte counters
# up to R = 64) and the momentum pass of the step between syncs (period 2: one of each).
N_ODD = 32 * 1001
DILOCO_MANY = [(True, 64, "ternary"), (True, 5, "ternary"), (True, 1, "ternary"), (False, 17, "bf16"),
               (False, 64, "f16"), (False, 1, "bf16"), (False, 9, "f32"), (False, 1, "f32")]


@pytest.mark.parametrize("sign,R,wire", DILOCO_MANY, ids=lambda v: str(v))
def test_diloco_many_replicas(sign, R, wire):
    run_steps(N_ODD, R, 1, "diloco", sign, 3, g_std=1e-3, period=2, seed=31, wire=wire)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_ternary_with_bf16_gradients(k):
    """The ternary DeMo encode compiled for k, fed bfloat16 gradients."""
    run_steps(RAGGED, 2, k, "demo", True, 2, g_std=1e-3, seed=29, bf16=True, wire="ternary")


def _encode(n, mode, k, wire, g, m, step=0):
    v, i = dm.payload_buffers(mode, n, k, step=step, diloco_period=8, wire=wire)
    dm.encode(g, m, v, i, k=k, beta=0.9, mode=mode, sign=True, seed=5, step=step, diloco_period=8, wire=wire)
    return v, i


@pytest.mark.parametrize("mode,k", [("demo", 4), ("demo", 1), ("random", 8), ("stride", 2)])
def test_ternary_words_match_oracle_packing(mode, k):
    n = RAGGED
    nc = n // C
    g = cuda_normal(n, 1e-2, 31)
    m = cuda_normal(n, 1e-2, 32)
    m_np = f64(m)
    v, i = _encode(n, mode, k, "ternary", g, m.clone())
    torch.cuda.synchronize()
    enc = ref.encode(m_np, f64(g), 0.9, k, ref.__dict__["MODE_" + mode.upper()], True, seed=5, step=0)
    want_v, want_i = ref.ternary_pack(enc["vals"], enc["idx"] if mode == "demo" else None)
    got_v = v.cpu().numpy().view(np.uint32).reshape(want_v.shape)
    # lanes (chunks) the oracle flags as near-ties are left out of the comparison
    keep = np.zeros(want_v.shape[0] * 32, dtype=np.uint64)
    keep[:nc] = ~enc["near_tie"]
    lane_mask = np.array([sum(int(keep[t * 32 + l]) << l for l in range(32)) for t in range(want_v.shape[0])],
                         dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(got_v & lane_mask[:, None, None], want_v & lane_mask[:, None, None])
    if mode == "demo":
        got_i = i.cpu().numpy().view(np.uint32).reshape(want_i.shape)
        assert np.array_equal(got_i & lane_mask[:, None, None], want_i & lane_mask[:, None, None])
    # bits of chunks past the end of the shard are zero
    tail = ~lane_mask[-1]
    assert (got_v[-1] & tail == 0).all()


@pytest.mark.parametrize("mode,k", [("demo", 4), ("random", 8), ("diloco", 1)])
def test_ternary_decode_equals_f32_decode(mode, k):
    n = 32 * 700
    step = 7  # a DiLoCo sync step for period 8
    R = 3
    gs = [cuda_normal(n, 1e-2, 40 + r) for r in range(R)]
    m0 = [cuda_normal(n, 1e-2, 50 + r) for r in range(R)]
    theta0 = cuda_normal(n, 2e-2, 60)
    out = {}
    for wire in ("f32", "ternary"):
        payloads = [_encode(n, mode, k, wire, gs[r], m0[r].clone(), step=step) for r in range(R)]
        th = theta0.clone()
        dm.decode_update(th, [p[0] for p in payloads], [p[1] for p in payloads] if mode == "demo" else None,
                         k=k, lr=1e-2, mode=mode, seed=5, step=step, diloco_period=8, wire=wire)
        out[wire] = th
    torch.cuda.synchronize()
    assert torch.equal(out["f32"], out["ternary"])


def test_wire_payload_sizes_and_validation():
    n = 32 * 1000 + 32 * 7
    g = cuda_normal(n, 1e-2, 70)
    for wire in ("f32", "bf16", "ternary"):
        v, i = _encode(n, "demo", 4, wire, g, torch.zeros(n, device="cuda"))
        vb, ib = dm.payload_bytes("demo", n, 4, wire=wire)
        assert v.numel() * v.element_size() == vb and i.numel() * i.element_size() == ib
        assert (vb, ib) == ref.payload_bytes_wire(ref.MODE_DEMO, n, 4, wire=dm.WIRES[wire])
        host = i.cpu()
        ok, bad = dm.validate_payload(host, n, 4, wire)
        assert ok and bad == -1
        # corrupt chunk 123: repeat an index
        if wire == "ternary":
            w = host.numpy().view(np.uint32).reshape(-1, 4, 5)
            t, lane = divmod(123, 32)
            u0 = sum(((int(w[t, 0, b]) >> lane) & 1) << b for b in range(5))
            for b in range(5):  # make index 1 equal to index 0
                bit = (u0 >> b) & 1
                w[t, 1, b] = (int(w[t, 1, b]) & ~(1 << lane)) | (bit << lane)
        else:
            host.view(-1, 4)[123, 1] = host.view(-1, 4)[123, 0]
        ok, bad = dm.validate_payload(host, n, 4, wire)
        assert not ok and bad == 123
    # an index beyond the chunk
    v, i = _encode(n, "demo", 4, "f32", g, torch.zeros(n, device="cuda"))
    host = i.cpu()
    host.view(-1, 4)[5, 3] = 40
    assert dm.validate_payload(host, n, 4, "f32") == (False, 5)


@pytest.mark.parametrize("mode,k,sign,wire", [("demo", 4, True, "f32"), ("demo", 4, False, "f32"),
                                              ("demo", 4, True, "ternary"), ("demo", 2, False, "bf16"),
                                              ("random", 8, True, "f32"), ("random", 8, False, "f16"),
                                              ("stride", 4, True, "ternary"), ("diloco", 1, False, "f32")])
def test_non_finite_inputs_stay_in_their_chunks(mode, k, sign, wire):
    """NaN, +-Inf and overflowing gradients in a few chunks: the call succeeds without a
    device fault, fused and split agree bit for bit, and every other chunk matches the
    oracle (the values of the poisoned chunks are unspecified)."""
    from parity import check_step

    n = 32 * (32 * 2 + 9)
    R = 2
    theta = cuda_normal(n, 2e-2, 7)
    ms = [cuda_normal(n, 1e-3, 8 + r) for r in range(R)]
    gs = [cuda_normal(n, 1e-3, 10 + r) for r in range(R)]
    bad = {3: float("nan"), 17: float("inf"), 40: -float("inf"), 70: 3e38}
    for c, v in bad.items():
        gs[c % R][c * C + 5] = v
        gs[c % R][c * C + 9] = -v if v == v else v
    good = [c for c in range(n // C) if c not in bad]
    check_step(theta, ms, gs, k=k, beta=0.999, lr=1e-3, mode=mode, sign=sign, step=7, period=8, rows=good,
               wire=wire)
    assert dm.device_fault() == 0
