"""Property tests of the oracle on arbitrary inputs (CPU; needs hypothesis).

The pins in test_oracle_pins.py fix the oracle on chosen inputs; these check
invariants that follow from the definitions on inputs hypothesis draws,
including exact ties, zeros, signed zeros and extreme magnitudes:

* top-k ("DeMo: Decoupled Momentum Optimization", abstract): k distinct slots in
  ascending order, and every kept slot beats every dropped one under the key
  (|X_u| larger, or equal with the lower index), checked pairwise;
* error feedback (FlexDeMo Algorithm 1, extraction and removal): the transform of the new
  momentum is the old coefficients with the kept slots cleared;
* Random positions ("2. Replication Schemes"): k distinct slots in [0, 32),
  the same for the same (seed, step, chunk), a prefix for a smaller k;
* scatter-mean: every slot's mean times its count gives back the sum of what
  was sent to it, and slots nobody sent stay zero;
* the ternary bit-plane format round-trips;
* conservation over several steps (sign off, beta = 1; DeMo with one replica,
  the other schemes with several): theta_T = theta_0 - lr / R * sum_r
  (m_r,0 + sum_t g_r,t - m_r,T).
"""

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402
from hypothesis.extra import numpy as hnp  # noqa: E402

import oracle.demo_ref as ref  # noqa: E402

C = ref.CHUNK
finite = st.floats(min_value=-2.0 ** 127, max_value=2.0 ** 127, width=32)
# values drawn from a small set make exact ties and zeros common
tied = st.sampled_from([0.0, -0.0, 1.0, -1.0, 0.5, -0.5, 2.0, 3.0e-38, -3.0e-38, 1e30])
row = hnp.arrays(np.float64, (C,), elements=st.one_of(finite, tied))


@settings(max_examples=300, deadline=None)
@given(X=row, k=st.integers(1, C))
def test_topk_beats_every_dropped_slot(X, k):
    kept, _ = ref.topk_select(X[None, :], k)
    kept = kept[0]
    assert len(kept) == k and len(set(kept.tolist())) == k
    assert (np.diff(kept) > 0).all()  # ascending slot order
    dropped = [u for u in range(C) if u not in set(kept.tolist())]
    for u in kept:
        for v in dropped:
            a, b = abs(X[u]), abs(X[v])
            assert a > b or (a == b and u < v), (u, v, X[u], X[v])


@settings(max_examples=150, deadline=None)
@given(x=hnp.arrays(np.float64, (3 * C,), elements=st.floats(-1e3, 1e3)),
       k=st.integers(1, C))
def test_feedback_clears_the_kept_coefficients(x, k):
    out = ref.encode(np.zeros_like(x), x, 0.9, k, ref.MODE_DEMO, False)
    X = out["X"]
    Xm = out["m"].reshape(-1, C) @ ref.dct_matrix().T  # the new momentum, transformed
    expect = X.copy()
    rows = np.arange(X.shape[0])[:, None]
    expect[rows, out["idx"]] = 0.0
    scale = np.abs(X).max() + 1e-300
    assert np.abs(Xm - expect).max() <= 1e-12 * scale


@settings(max_examples=200, deadline=None)
@given(seed=st.integers(0, 2**64 - 1), step=st.integers(0, 2**40), chunk=st.integers(0, 2**40),
       k=st.integers(1, C))
def test_random_positions_are_a_draw_without_replacement(seed, step, chunk, k):
    p = ref.random_positions(seed, step, chunk, k)
    assert len(p) == k and len(set(int(v) for v in p)) == k
    assert all(0 <= int(v) < C for v in p)
    assert list(ref.random_positions(seed, step, chunk, k)) == list(p)
    if k > 1:  # the draws are sequential: fewer draws give a prefix
        assert list(ref.random_positions(seed, step, chunk, k - 1)) == list(p[:k - 1])


@settings(max_examples=150, deadline=None)
@given(data=st.data(), R=st.integers(1, 5), k=st.integers(1, 6), nc=st.integers(1, 4))
def test_scatter_mean_preserves_each_slot_sum(data, R, k, nc):
    vals, poss = [], []
    for _ in range(R):
        vals.append(data.draw(hnp.arrays(np.float64, (nc, k), elements=st.floats(-1e6, 1e6))))
        poss.append(np.stack([np.asarray(data.draw(st.permutations(range(C))))[:k] for _ in range(nc)]))
    Y, cnt = ref.scatter_mean(vals, poss, nc)
    total = np.zeros((nc, C))
    sent = np.zeros((nc, C), dtype=int)
    for v, p in zip(vals, poss):
        for c in range(nc):
            for j in range(k):
                total[c, p[c, j]] += v[c, j]
                sent[c, p[c, j]] += 1
    assert np.array_equal(cnt, sent)
    assert (Y[sent == 0] == 0).all()
    assert np.allclose(Y * np.maximum(sent, 1), total, rtol=1e-12, atol=1e-6)


@settings(max_examples=100, deadline=None)
@given(data=st.data(), nc=st.integers(1, 70), k=st.integers(1, 8), demo=st.booleans())
def test_ternary_format_round_trips(data, nc, k, demo):
    vals = data.draw(hnp.arrays(np.float64, (nc, k), elements=st.sampled_from([-1.0, 0.0, 1.0])))
    idx = None
    if demo:
        idx = np.stack([np.sort(np.asarray(data.draw(st.permutations(range(C))))[:k]) for _ in range(nc)])
    vw, iw = ref.ternary_pack(vals, idx)
    assert vw.shape == ((nc + 31) // 32, k, 2)
    v2, i2 = ref.ternary_unpack(vw, iw, nc)
    assert np.array_equal(v2, vals)
    if demo:
        assert np.array_equal(i2, idx)


@settings(max_examples=60, deadline=None)
@given(mode=st.sampled_from([ref.MODE_DEMO, ref.MODE_RANDOM, ref.MODE_STRIDE, ref.MODE_DILOCO]),
       R=st.integers(1, 4), kexp=st.integers(0, 5), T=st.integers(1, 6), nc=st.integers(1, 5),
       period=st.integers(1, 4), seed=st.integers(0, 2 ** 64 - 1), data_seed=st.integers(0, 2 ** 32 - 1))
def test_conservation_over_steps(mode, R, kexp, T, nc, period, seed, data_seed):
    if mode == ref.MODE_DEMO:
        R = 1  # DeMo replicas may keep different slots: the mean is then per slot, not of the whole q
    k = 1 << kexp  # a divisor of 32, valid for every scheme
    r = np.random.default_rng(data_seed)
    n = nc * C
    lr = 0.125
    theta0 = r.standard_normal(n)
    m0 = [r.standard_normal(n) for _ in range(R)]
    theta, ms = theta0.copy(), [m.copy() for m in m0]
    gsum = [np.zeros(n) for _ in range(R)]
    for t in range(T):
        gs = [r.standard_normal(n) for _ in range(R)]
        theta, ms, _ = ref.step(theta, ms, gs, beta=1.0, lr=lr, k=k, mode=mode, sign=False, seed=seed, step_idx=t,
                                period=period)
        for q in range(R):
            gsum[q] += gs[q]
    want = theta0 - lr / R * sum(m0[q] + gsum[q] - ms[q] for q in range(R))
    assert np.abs(theta - want).max() <= 1e-12 * (1.0 + np.abs(want).max())
