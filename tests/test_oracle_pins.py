"""Pins of the float64 oracle against facts that do not come from the oracle itself.

Each pin checks the oracle against mathematics the pages fix (orthonormality,
closed forms, a library DCT computed by an FFT route, brute force over all
subsets, hand-computed scatter-means, the published splitmix64 stream, exact
reductions to momentum-free SGD).  The planted-mistake tests at the end swap a
plausible bug into the oracle and check that some pin fails.
"""

import itertools
import math
import os

import numpy as np
import pytest

import oracle.demo_ref as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
C = ref.CHUNK


def rng(seed=0):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------------
# Pin functions (return None, raise AssertionError on failure); each is run on
# the real oracle and, below, on planted mutants.
# ----------------------------------------------------------------------------

def pin_dct_orthonormal():
    D = ref._D
    assert np.abs(D @ D.T - np.eye(C)).max() < 1e-12
    assert np.abs(D.T @ D - np.eye(C)).max() < 1e-12


def pin_dct_vs_fft_library():
    sp = pytest.importorskip("scipy.fft")
    x = rng(1).standard_normal((64, C))
    enc = ref.encode(np.zeros(64 * C), x.reshape(-1), 0.0, C, ref.MODE_DEMO, False)
    assert np.abs(enc["X"] - sp.dct(x, type=2, norm="ortho", axis=1)).max() < 1e-12


def pin_dc_coefficient():
    a = 0.7
    enc = ref.encode(np.zeros(C), np.full(C, a), 0.0, 1, ref.MODE_DEMO, False)
    X = enc["X"][0]
    assert abs(X[0] - a * math.sqrt(C)) < 1e-12
    assert np.abs(X[1:]).max() < 1e-12 * a
    assert list(enc["idx"][0]) == [0]


def pin_single_cosine():
    # x_i = cos(pi (2i+1) u0 / 64): sum_i cos^2 = 16, so X_{u0} = (1/4) * 16 = 4 and all
    # other coefficients vanish (textbook orthogonality of the DCT-II basis).
    for u0 in (1, 5, 17, 31):
        x = np.array([math.cos(math.pi * (2 * i + 1) * u0 / 64) for i in range(C)])
        enc = ref.encode(np.zeros(C), x, 0.0, 1, ref.MODE_DEMO, False)
        X = enc["X"][0]
        assert abs(X[u0] - 4.0) < 1e-12
        X[u0] = 0.0
        assert np.abs(X).max() < 1e-12


def brute_topk(X, k):
    """All C(n, k) subsets: maximise sum |X_u|, then the lexicographically smallest."""
    best, best_key = None, None
    for S in itertools.combinations(range(len(X)), k):
        key = (-sum(abs(X[u]) for u in S), S)
        if best_key is None or key < best_key:
            best, best_key = S, key
    return list(best)


def pin_topk_bruteforce():
    r = rng(2)
    for trial in range(60):
        L = 8 if trial % 2 else 10
        X = r.integers(-3, 4, size=L).astype(np.float64)  # many exact ties
        for k in range(1, 5):
            kept, _ = ref.topk_select(X, k)
            assert list(kept[0]) == brute_topk(X, k), (X, k)


def pin_k32_zero_residual():
    r = rng(3)
    m = r.standard_normal(4 * C)
    g = r.standard_normal(4 * C)
    enc = ref.encode(m, g, 0.9, C, ref.MODE_DEMO, False)
    assert np.abs(enc["m"]).max() < 1e-12
    assert np.abs(enc["vals"] - enc["X"]).max() == 0.0


def pin_parseval_and_projection():
    sp = pytest.importorskip("scipy.fft")
    r = rng(4)
    m = r.standard_normal(16 * C)
    g = r.standard_normal(16 * C)
    for sign in (False, True):
        enc = ref.encode(m, g, 0.5, 4, ref.MODE_DEMO, sign)
        x = (float(np.float32(0.5)) * m + g).reshape(-1, C)
        q = enc["q"]
        res = enc["m"].reshape(-1, C)
        # ||x||^2 = ||q||^2 + ||x - q||^2 (q is an orthogonal projection of x)
        lhs = (x * x).sum(1)
        rhs = (q * q).sum(1) + (res * res).sum(1)
        assert np.abs(lhs - rhs).max() < 1e-10 * lhs.max()
        # the residual's spectrum (FFT route) is zero on the kept slots and X elsewhere
        Rspec = sp.dct(res, type=2, norm="ortho", axis=1)
        Xspec = sp.dct(x, type=2, norm="ortho", axis=1)
        rows = np.arange(x.shape[0])[:, None]
        assert np.abs(Rspec[rows, enc["idx"]]).max() < 1e-12
        Xspec[rows, enc["idx"]] = 0.0
        assert np.abs(Rspec - Xspec).max() < 1e-12


def pin_sgd_reduction():
    # R = 1, k = 32, sign off: every step drains m, so theta_{t+1} = theta_t - lr g_t.
    r = rng(5)
    n = 8 * C
    for mode in (ref.MODE_DEMO, ref.MODE_RANDOM, ref.MODE_STRIDE):
        theta = r.standard_normal(n)
        m = np.zeros(n)
        for t in range(3):
            g = r.standard_normal(n)
            th2, (m2,), _ = ref.step(theta, [m], [g], beta=0.9, lr=0.1, k=C, mode=mode, sign=False,
                                     seed=7, step_idx=t)
            assert np.abs(th2 - (theta - float(np.float32(0.1)) * g)).max() < 1e-12
            assert np.abs(m2).max() < 1e-12
            theta, m = th2, m2


def pin_replica_mean_identical():
    r = rng(6)
    n = 6 * C
    m = r.standard_normal(n)
    g = r.standard_normal(n)
    theta = r.standard_normal(n)
    for mode, k in ((ref.MODE_DEMO, 4), (ref.MODE_RANDOM, 8), (ref.MODE_STRIDE, 4)):
        th1, _, info1 = ref.step(theta, [m], [g], beta=0.9, lr=0.1, k=k, mode=mode, sign=False, seed=3)
        th3, _, info3 = ref.step(theta, [m] * 3, [g] * 3, beta=0.9, lr=0.1, k=k, mode=mode, sign=False,
                                 seed=3)
        # the mean of R identical payloads is the payload itself, so Q equals q
        assert np.abs(info3["Q"] - info1["encodes"][0]["q"]).max() < 1e-12
        assert np.abs(th3 - th1).max() < 1e-12


def pin_scatter_mean_hand_example():
    # chunk 0: replica 0 sends (u=1, 2.0), (u=5, -1.0); replica 1 sends (u=1, 4.0), (u=7, 3.0)
    # chunk 1: replica 0 sends (u=0, 1.0), (u=31, 1.0); replica 1 sends (u=2, -2.0), (u=31, 0.0)
    vals = [np.array([[2.0, -1.0], [1.0, 1.0]]), np.array([[4.0, 3.0], [-2.0, 0.0]])]
    pos = [np.array([[1, 5], [0, 31]]), np.array([[1, 7], [2, 31]])]
    Y, cnt = ref.scatter_mean(vals, pos, 2)
    want = np.zeros((2, C))
    want[0, 1], want[0, 5], want[0, 7] = 3.0, -1.0, 3.0
    want[1, 0], want[1, 2], want[1, 31] = 1.0, -2.0, 0.5
    assert np.array_equal(Y, want)
    assert cnt[0, 1] == 2 and cnt[0, 5] == 1 and cnt[1, 31] == 2 and cnt.sum() == 8


def pin_sign_values():
    r = rng(7)
    n = 32 * C
    ms = [r.standard_normal(n), r.standard_normal(n)]
    gs = [r.standard_normal(n), r.standard_normal(n)]
    _, _, info = ref.step(r.standard_normal(n), ms, gs, beta=0.9, lr=0.1, k=4, mode=ref.MODE_DEMO, sign=True)
    assert set(np.unique(info["Y"])) <= {-1.0, -0.5, 0.0, 0.5, 1.0}
    for e in info["encodes"]:
        assert set(np.unique(e["vals"])) <= {-1.0, 0.0, 1.0}


def pin_splitmix64_published():
    lines = [l for l in open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt")) if not l.startswith("#")]
    seed = int(lines[0].split()[1])
    want = [int(l) for l in lines[1:] if l.strip()]
    assert ref.splitmix64_stream(seed, len(want)) == want


def pin_random_positions():
    for c in range(200):
        for k in (1, 4, 8, 32):
            p = ref.random_positions(11, 3, c, k)
            assert len(p) == k and len(set(p)) == k and all(0 <= x < C for x in p)
            # draw j does not depend on k: a shorter draw is a prefix
            assert p == ref.random_positions(11, 3, c, C)[:k]
    # Lemire's reduction stays in range at the hash extremes: floor((2^32-1)(32-j)/2^32) = 31-j
    for j in range(C):
        assert (((1 << 32) - 1) * (C - j)) >> 32 == C - 1 - j
    # first-draw and ordered-pair frequencies are uniform (chi-square, fixed seed)
    N = 20000
    counts1 = np.zeros(C)
    pairs = np.zeros((C, C))
    for c in range(N):
        p = ref.random_positions(0, 1, c, 2)
        counts1[p[0]] += 1
        pairs[p[0], p[1]] += 1
    e1 = N / C
    chi1 = ((counts1 - e1) ** 2 / e1).sum()
    assert chi1 < 70.0  # 31 dof: p ~ 1e-4 at 70
    off = ~np.eye(C, dtype=bool)
    assert (pairs[~off] == 0).all()
    e2 = N / (C * (C - 1))
    chi2 = ((pairs[off] - e2) ** 2 / e2).sum()
    assert chi2 < 1160.0  # 991 dof: mean 991, sd ~44.5


def pin_stride_coverage():
    for k in (1, 2, 4, 8, 16, 32):
        ns = C // k
        for t0 in (0, 5, 13):
            seen = []
            for t in range(t0, t0 + ns):
                seen += ref.stride_positions(t, k)
            assert sorted(seen) == list(range(C))


def pin_diloco_closed_form():
    r = rng(8)
    n = 4 * C
    H = 8
    beta = 0.9
    b = float(np.float32(beta))  # computed here, not through the oracle
    theta0 = r.standard_normal(n)
    theta, m = theta0.copy(), np.zeros(n)
    gs = [r.standard_normal(n) for _ in range(2 * H)]
    for t in range(2 * H):
        th2, (m2,), info = ref.step(theta, [m], [gs[t]], beta=beta, lr=0.25, k=1, mode=ref.MODE_DILOCO,
                                    sign=False, step_idx=t, period=H)
        if (t + 1) % H:
            assert np.array_equal(th2, theta)  # theta moves only on sync steps
            assert info["encodes"][0]["vals"] is None
        else:
            acc = sum(b ** (H - 1 - j) * gs[t - H + 1 + j] for j in range(H))
            assert np.abs(info["encodes"][0]["vals"].reshape(-1) - acc).max() < 1e-12
            assert np.abs(th2 - (theta - float(np.float32(0.25)) * acc)).max() < 1e-12
            assert np.abs(m2).max() == 0.0
        theta, m = th2, m2


def pin_conservation_multistep():
    # Sign off, beta = 1: every step splits beta m + g exactly into the new momentum and the
    # component q that is sent (the chunk transform is orthonormal, so DeMo's q in the
    # parameter domain is the inverse transform of the kept coefficients).  Random, Striding
    # and DiLoCo replicas all send the same slots, so Q is the plain mean of the replicas' q
    # (DeMo is taken with one replica).  Summed over T steps the momenta telescope:
    #     theta_T = theta_0 - lr / R * sum_r (m_r,0 + sum_t g_r,t - m_r,T).
    r = rng(11)
    n = 6 * C
    lr, T = 0.25, 7
    for mode, k, R in ((ref.MODE_DEMO, 4, 1), (ref.MODE_DEMO, 1, 1), (ref.MODE_RANDOM, 3, 3),
                       (ref.MODE_STRIDE, 4, 2), (ref.MODE_DILOCO, 1, 2)):
        theta0 = r.standard_normal(n)
        m0 = [r.standard_normal(n) for _ in range(R)]
        theta, ms = theta0.copy(), [m.copy() for m in m0]
        gsum = [np.zeros(n) for _ in range(R)]
        for t in range(T):
            gs = [r.standard_normal(n) for _ in range(R)]
            theta, ms, _ = ref.step(theta, ms, gs, beta=1.0, lr=lr, k=k, mode=mode, sign=False, seed=3,
                                    step_idx=t, period=3)
            for q in range(R):
                gsum[q] += gs[q]
        want = theta0 - lr / R * sum(m0[q] + gsum[q] - ms[q] for q in range(R))
        assert np.abs(theta - want).max() < 1e-12 * (1.0 + np.abs(want).max()), mode


def pin_stride_constant_gradient():
    # Striding with a constant gradient g: position p of a chunk is sent on the steps t with
    # t = p (mod s), s = 32 / k, carrying everything accumulated since its last send: the
    # first send (t = p mod s) carries g (1 - b^(t+1)) / (1 - b), each later one
    # g (1 - b^s) / (1 - b); after T steps m holds what accumulated since the last send.
    beta, lr, T = 0.75, 0.5, 11
    b = float(np.float32(beta))
    for k in (1, 4, 8):
        s = C // k
        g = np.tile(np.linspace(-1.0, 2.0, C), 3)
        theta, m = np.zeros(g.size), np.zeros(g.size)
        for t in range(T):
            theta, (m,), _ = ref.step(theta, [m], [g], beta=beta, lr=lr, k=k, mode=ref.MODE_STRIDE, sign=False,
                                      step_idx=t)
        geo = lambda L: (1.0 - b ** L) / (1.0 - b)  # 1 + b + ... + b^(L-1)
        p = np.tile(np.arange(C), 3)
        first = p % s
        sends = np.where(first < T, (T - 1 - first) // s + 1, 0)
        sent = np.where(sends > 0, geo(first + 1) + (sends - 1) * geo(s), 0.0)
        last = first + (sends - 1) * s
        left = np.where(sends > 0, T - 1 - last, T)
        assert np.abs(theta - (-float(np.float32(lr)) * g * sent)).max() < 1e-12
        assert np.abs(m - g * geo(left)).max() < 1e-12


def _basis_row(u):
    """Row u of the orthonormal DCT-II basis, written out from its definition."""
    a = math.sqrt((1.0 if u == 0 else 2.0) / C)
    return np.array([a * math.cos(math.pi * (2 * i + 1) * u / (2 * C)) for i in range(C)])


def pin_signed_demo_basis_chunks():
    # Sign on, k = 1, every gradient chunk a multiple of ONE basis cosine u0 (its own per chunk):
    # the chunk's only nonzero coefficient is u0, so top-1 keeps u0 and the removal leaves m = 0
    # (for any beta); the replica sends sign(a) at u0, the mean over replicas is the mean of the
    # signs, and Q is that mean times basis row u0.  Over T steps, per chunk c:
    #     theta_T = theta_0 - lr * sum_t mean_r sign(a_{r,t,c}) * row(u0_c),   m_r = 0 throughout.
    # Three replicas with independent amplitudes make the mean of signs take the values
    # {+-1, +-1/3}, which a sign taken after the mean (or no sign) would not give.
    r = rng(31)
    u0 = [0, 1, 5, 17, 31, 0, 8]
    nc, R, T = len(u0), 3, 6
    n = nc * C
    rows = [_basis_row(u) for u in u0]
    cosv = [np.array([math.cos(math.pi * (2 * i + 1) * u / (2 * C)) for i in range(C)]) for u in u0]
    for beta in (0.5, 0.999):
        theta0 = r.standard_normal(n)
        theta, ms = theta0.copy(), [np.zeros(n) for _ in range(R)]
        want = theta0.copy()
        lr = 0.25
        for t in range(T):
            a = r.standard_normal((R, nc))
            gs = [np.concatenate([a[q, c] * cosv[c] for c in range(nc)]) for q in range(R)]
            theta, ms, info = ref.step(theta, ms, gs, beta=beta, lr=lr, k=1, mode=ref.MODE_DEMO, sign=True,
                                       step_idx=t)
            for c in range(nc):
                want[c * C:(c + 1) * C] -= float(np.float32(lr)) * np.sign(a[:, c]).mean() * rows[c]
                for q in range(R):
                    assert list(info["encodes"][q]["idx"][c]) == [u0[c]]
            for q in range(R):
                assert np.abs(ms[q]).max() < 1e-12 * np.abs(a).max()
        assert np.abs(theta - want).max() < 1e-12


def pin_signed_constant_gradient():
    # Sign on, a constant gradient w_r * g per replica (w = 1, 0.5, -2): a send at position p
    # carries w_r g_p times 1 + b + ... + b^(L-1) (L steps accumulated since its last send), whose
    # sign is sign(w_r g_p); every replica sends the same positions, so each send moves theta by
    # lr * mean_r sign(w_r) * sign(g_p) = lr * sign(g_p) / 3, and m_r holds w_r g_p times the
    # geometric sum of the steps since the last send.  Positions per step: Striding o + s j with
    # o = t mod s, s = 32 / k; Random the shared-seed draws; DiLoCo all 32 on sync steps.
    beta, lr, T = 0.75, 0.5, 13
    b = float(np.float32(beta))
    w = [1.0, 0.5, -2.0]
    geo = lambda L: (1.0 - b ** L) / (1.0 - b)
    g = np.concatenate([np.linspace(-1.0, 2.0, C), np.linspace(3.0, -0.5, C), -np.linspace(0.1, 1.0, C)])
    nc = g.size // C
    for mode, k in ((ref.MODE_STRIDE, 1), (ref.MODE_STRIDE, 4), (ref.MODE_STRIDE, 8), (ref.MODE_RANDOM, 3),
                    (ref.MODE_DILOCO, 1)):
        theta, ms = np.zeros(g.size), [np.zeros(g.size) for _ in w]
        sends = np.zeros(g.size)
        last = np.full(g.size, -1)
        for t in range(T):
            theta, ms, _ = ref.step(theta, ms, [wq * g for wq in w], beta=beta, lr=lr, k=k, mode=mode, sign=True,
                                    seed=5, step_idx=t, period=4)
            for c in range(nc):
                if mode == ref.MODE_STRIDE:
                    pos = [(t % (C // k)) + (C // k) * j for j in range(k)]
                elif mode == ref.MODE_RANDOM:
                    pos = ref.random_positions(5, t, c, k)
                else:
                    pos = list(range(C)) if (t + 1) % 4 == 0 else []
                for p in pos:
                    sends[c * C + p] += 1
                    last[c * C + p] = t
        assert np.abs(theta - (-float(np.float32(lr)) * sends * np.sign(g) / 3.0)).max() < 1e-12, mode
        left = T - 1 - last  # steps accumulated since the last send (all T when never sent)
        for wq, m in zip(w, ms):
            assert np.abs(m - wq * g * geo(left)).max() < 1e-12, mode


def pin_payload_bytes():
    n = 1 << 20
    for k in (1, 2, 4, 8):
        dv, di = ref.payload_bytes(ref.MODE_DEMO, n, k, idx_bytes_per_entry=4)
        rv, ri = ref.payload_bytes(ref.MODE_RANDOM, n, k)
        assert (dv + di) / (rv + ri) == 2.0  # Random needs half of DeMo's bytes (4-byte indices)
        dv, di = ref.payload_bytes(ref.MODE_DEMO, n, k, idx_bytes_per_entry=1)
        assert (dv + di) / (rv + ri) == 1.25
    assert ref.payload_bytes(ref.MODE_DILOCO, n, 1, step=7, period=8) == (4 * n, 0)
    assert ref.payload_bytes(ref.MODE_DILOCO, n, 1, step=6, period=8) == (0, 0)


ALL_PINS = [
    pin_dct_orthonormal, pin_dct_vs_fft_library, pin_dc_coefficient, pin_single_cosine,
    pin_topk_bruteforce, pin_k32_zero_residual, pin_parseval_and_projection, pin_sgd_reduction,
    pin_replica_mean_identical, pin_scatter_mean_hand_example, pin_sign_values, pin_splitmix64_published,
    pin_random_positions, pin_stride_coverage, pin_diloco_closed_form, pin_payload_bytes,
    pin_conservation_multistep, pin_stride_constant_gradient, pin_signed_demo_basis_chunks,
    pin_signed_constant_gradient,
]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_near_tie_flags_constant_chunk():
    # A constant chunk has one nonzero coefficient; with k = 4 the 4th and 5th
    # magnitudes are both 0, so the oracle flags the chunk as a near-tie.
    enc = ref.encode(np.zeros(C), np.full(C, 1.5), 0.0, 4, ref.MODE_DEMO, True)
    assert enc["near_tie"][0]
    enc = ref.encode(np.zeros(C), rng(9).standard_normal(C), 0.0, 4, ref.MODE_DEMO, False)
    assert not enc["near_tie"][0]


# ----------------------------------------------------------------------------
# Planted mistakes: each mutant must make at least one pin fail.
# ----------------------------------------------------------------------------

def _fails(pins):
    for p in pins:
        try:
            p()
        except AssertionError:
            return True
    return False


def test_mutant_transposed_basis(monkeypatch):
    monkeypatch.setattr(ref, "_D", ref._D.T.copy())
    assert _fails([pin_dc_coefficient, pin_single_cosine, pin_dct_vs_fft_library])


def test_mutant_unnormalised_dc(monkeypatch):
    D = ref._D.copy()
    D[0] *= math.sqrt(2.0)  # a_0 = sqrt(2/C) instead of sqrt(1/C)
    monkeypatch.setattr(ref, "_D", D)
    assert _fails([pin_dct_orthonormal])
    assert _fails([pin_dc_coefficient])


def test_mutant_unstable_topk(monkeypatch):
    def bad(X, k):
        # ties broken toward the HIGHEST index
        X = np.atleast_2d(np.asarray(X, dtype=np.float64))
        cols = np.broadcast_to(-np.arange(X.shape[1]), X.shape)
        order = np.lexsort((cols, -np.abs(X)), axis=1)
        return np.sort(order[:, :k], axis=1), order

    monkeypatch.setattr(ref, "topk_select", bad)
    assert _fails([pin_topk_bruteforce])


def test_mutant_mean_over_R(monkeypatch):
    orig = ref.scatter_mean

    def bad(vals_list, pos_list, nc):
        Y, cnt = orig(vals_list, pos_list, nc)
        S = Y * cnt
        return S / len(vals_list), cnt

    monkeypatch.setattr(ref, "scatter_mean", bad)
    assert _fails([pin_scatter_mean_hand_example])


def test_mutant_signed_feedback(monkeypatch):
    # error feedback subtracting the signed values instead of q
    orig = ref.encode

    def bad(m, g, beta, k, mode, sign, **kw):
        out = orig(m, g, beta, k, mode, sign, **kw)
        if sign and mode == ref.MODE_DEMO:
            x = (ref.f32(beta) * np.asarray(m) + np.asarray(g)).reshape(-1, C)
            Xs = np.zeros_like(out["X"])
            rows = np.arange(x.shape[0])[:, None]
            Xs[rows, out["idx"]] = out["vals"]
            out["q"] = Xs @ ref._D
            out["m"] = (x - out["q"]).reshape(-1)
        return out

    monkeypatch.setattr(ref, "encode", bad)
    assert _fails([pin_parseval_and_projection])
    assert _fails([pin_signed_demo_basis_chunks])


def test_mutant_signed_feedback_in_positional_schemes(monkeypatch):
    # Striding / Random / DiLoCo: the removal leaves x - sign(x) at the sent positions instead of 0
    orig = ref.encode

    def bad(m, g, beta, k, mode, sign, **kw):
        out = orig(m, g, beta, k, mode, sign, **kw)
        if sign and mode != ref.MODE_DEMO and out["pos"] is not None:
            x = (ref.f32(beta) * np.asarray(m) + np.asarray(g)).reshape(-1, C)
            mm = out["m"].reshape(-1, C).copy()
            rows = np.arange(x.shape[0])[:, None]
            mm[rows, out["pos"]] = x[rows, out["pos"]] - np.sign(x[rows, out["pos"]])
            out["m"] = mm.reshape(-1)
        return out

    monkeypatch.setattr(ref, "encode", bad)
    assert _fails([pin_signed_constant_gradient])


def test_mutant_sign_after_the_mean(monkeypatch):
    # the replicas send unsigned values and the receiver takes the sign of their mean
    orig = ref.step

    def bad(theta, ms, gs, *, sign, lr, mode, **kw):
        th, m2, info = orig(theta, ms, gs, sign=False, lr=lr, mode=mode, **kw)
        if sign:
            Y = np.sign(info["Y"])
            Q = Y @ ref._D if mode == ref.MODE_DEMO else Y
            th = np.asarray(theta, dtype=np.float64) - ref.f32(lr) * Q.reshape(-1)
        return th, m2, info

    monkeypatch.setattr(ref, "step", bad)
    assert _fails([pin_signed_demo_basis_chunks])
    assert _fails([pin_signed_constant_gradient])
    assert not _fails([pin_conservation_multistep, pin_stride_constant_gradient])  # unsigned pins cannot see it


def test_mutant_no_removal_in_fisher_yates(monkeypatch):
    def bad(seed, step, chunk, k, C=C):
        free = list(range(C))
        out = []
        for j in range(k):
            h = ref.index_hash(seed, step, chunk, j)
            out.append(free[((h >> 32) * (C - j)) >> 32])
        return out

    monkeypatch.setattr(ref, "random_positions", bad)
    assert _fails([pin_random_positions])


def test_mutant_stride_without_offset(monkeypatch):
    monkeypatch.setattr(ref, "stride_positions", lambda step, k, C=C: [(C // k) * j for j in range(k)])
    assert _fails([pin_stride_coverage])


def test_mutant_dropped_beta(monkeypatch):
    monkeypatch.setattr(ref, "f32", lambda x: 1.0 if x == 0.9 else float(np.float32(x)))
    assert _fails([pin_diloco_closed_form])


def test_mutant_forward_transform_in_decode(monkeypatch):
    orig = ref.decode_update

    def bad(theta, vals_list, pos_list, lr, mode, wire=0):
        new_theta, Q, Y, cnt = orig(theta, vals_list, pos_list, lr, mode, wire)
        if mode == ref.MODE_DEMO:  # DCT-II where the inverse (DCT-III) belongs
            Q = Y @ ref._D.T
            new_theta = np.asarray(theta) - ref.f32(lr) * Q.reshape(-1)
        return new_theta, Q, Y, cnt

    monkeypatch.setattr(ref, "decode_update", bad)
    assert _fails([pin_conservation_multistep])
    assert _fails([pin_signed_demo_basis_chunks])


def test_mutant_momentum_not_carried(monkeypatch):
    orig = ref.step

    def bad(theta, ms, gs, **kw):
        th, _, info = orig(theta, ms, gs, **kw)
        return th, [np.asarray(m, dtype=np.float64).copy() for m in ms], info  # the old m returned

    monkeypatch.setattr(ref, "step", bad)
    assert _fails([pin_conservation_multistep])
    assert _fails([pin_stride_constant_gradient])
    assert _fails([pin_signed_constant_gradient])


def test_mutant_wrong_hash_constant(monkeypatch):
    monkeypatch.setattr(ref, "_GAMMA", 0x9E3779B97F4A7C13)
    assert _fails([pin_splitmix64_published])


# ----------------------------------------------------------------------------
# Regression fixtures written by tests/golden/make_golden.py (oracle only)
# ----------------------------------------------------------------------------

def test_golden_random_positions_unchanged():
    for line in open(os.path.join(GOLDEN, "random_positions_seed0.txt")):
        if line.startswith("#"):
            continue
        head, pos = line.split(":")
        seed, step, chunk = map(int, head.split())
        assert ref.random_positions(seed, step, chunk, 8) == [int(p) for p in pos.split()]


def test_golden_demo_step_unchanged():
    import importlib.util

    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(GOLDEN, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    theta, gs = mg.tiny_inputs()
    th1, _, info = ref.step(theta, [np.zeros_like(theta)] * 2, gs, beta=0.999, lr=1e-3, k=4,
                            mode=ref.MODE_DEMO, sign=True)
    idx, th = {}, []
    for line in open(os.path.join(GOLDEN, "demo_step_tiny.txt")):
        if line.startswith("idx"):
            head, vals = line.split(":")
            _, r, c = head.split()
            idx[(int(r), int(c))] = [int(v) for v in vals.split()]
        elif line.startswith("theta1"):
            th.append(float(line.split()[1]))
    for (r, c), want in idx.items():
        assert list(info["encodes"][r]["idx"][c]) == want
    assert np.array_equal(np.array(th), th1)


# ----------------------------------------------------------------------------
# Wire formats
# ----------------------------------------------------------------------------

def test_ternary_pack_hand_example():
    # three chunks (one partial tile), k = 4
    vals = np.array([[1, 0, -1, 1], [0, 0, 0, 0], [-1, -1, 1, 0]], dtype=float)
    idx = np.array([[0, 3, 17, 31], [1, 2, 3, 4], [5, 6, 7, 8]])
    vw, iw = ref.ternary_pack(vals, idx)
    assert vw.shape == (1, 4, 2) and iw.shape == (1, 4, 5)
    # value 0: nonzero in chunks 0 and 2, negative in chunk 2
    assert vw[0, 0].tolist() == [0b101, 0b100]
    # value 1: nonzero only in chunk 2, negative there
    assert vw[0, 1].tolist() == [0b100, 0b100]
    # value 2: chunk 0 negative, chunk 2 positive
    assert vw[0, 2].tolist() == [0b101, 0b001]
    # index 3 of the chunks is 31, 4, 8: bit planes b0..b4
    assert iw[0, 3].tolist() == [0b001, 0b001, 0b011, 0b101, 0b001]


def test_ternary_round_trip_and_sizes():
    r = rng(20)
    for nc in (1, 31, 32, 33, 70):
        vals = r.integers(-1, 2, size=(nc, 8)).astype(float)
        idx = np.sort(np.stack([r.choice(32, 8, replace=False) for _ in range(nc)]), axis=1)
        vw, iw = ref.ternary_pack(vals, idx)
        v2, i2 = ref.ternary_unpack(vw, iw, nc)
        assert np.array_equal(v2, vals) and np.array_equal(i2, idx)
    n = 32 * 32 * 100  # 100 full tiles
    for k in (1, 2, 4, 8):
        vb, ib = ref.payload_bytes_wire(ref.MODE_DEMO, n, k, wire=ref.WIRE_TERNARY)
        assert (vb + ib) * 8 == (n // 32) * k * 7  # 2 bits per value + 5 per index
        vb, ib = ref.payload_bytes_wire(ref.MODE_RANDOM, n, k, wire=ref.WIRE_TERNARY)
        assert vb * 8 == (n // 32) * k * 2 and ib == 0
        assert ref.payload_bytes_wire(ref.MODE_DEMO, n, k, wire=ref.WIRE_F32) == ref.payload_bytes(ref.MODE_DEMO, n, k)
        assert ref.payload_bytes_wire(ref.MODE_DEMO, n, k, wire=ref.WIRE_BF16) == ((n // 32) * k * 2, (n // 32) * k)


def test_16bit_rounding_matches_torch():
    import torch

    x = np.concatenate([rng(21).standard_normal(20000) * s for s in (1e-3, 1.0, 1e3)]).astype(np.float32)
    x = np.concatenate([x, np.float32([1.00390625, 1.005859375, -0.0, 0.0, 65504.0])]).astype(np.float64)
    tb = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    th = torch.tensor(x, dtype=torch.float32).to(torch.float16).to(torch.float64).numpy()
    assert np.array_equal(ref.round_bf16(x), tb)
    assert np.array_equal(ref.round_f16(x), th)


def _nearest_in_table(x, table_bits, as_float):
    """Brute force: the nearest finite value of a 16-bit format to each float64 x, ties to the
    pattern with an even last bit; values beyond the largest finite one by half a step or more
    become infinities.  ``table_bits`` holds every bit pattern of the format."""
    vals = as_float(table_bits)
    fin = np.isfinite(vals)
    bits, vals = table_bits[fin], vals[fin]
    order = np.lexsort((bits, vals))  # -0 and +0 share a value: the sort keeps both
    bits, vals = bits[order], vals[order]
    top = vals.max()
    step_top = top - vals[vals < top].max()
    out = np.empty_like(x)
    for i, v in enumerate(x):
        if abs(v) >= top + step_top / 2:
            out[i] = math.copysign(math.inf, v)
            continue
        d = np.abs(vals - v)
        best = d.min()
        cand = np.flatnonzero(d == best)
        even = [c for c in cand if bits[c] % 2 == 0]
        pick = even[0] if even else cand[0]
        out[i] = vals[pick]
        if out[i] == 0.0:
            out[i] = math.copysign(0.0, v)
    return out


def test_16bit_rounding_from_float64_by_brute_force():
    # The oracle rounds a float64 payload value to bf16 / fp16 in ONE rounding.  Rounding it to
    # float32 first would differ wherever the float32 value lands on a 16-bit midpoint: x =
    # 1 + 2^-8 + 2^-30 is above the bf16 midpoint between 1 and 1 + 2^-7 (so it rounds up), but
    # float32 drops the 2^-30 and the midpoint then rounds to the even 1.0.
    import torch

    pats = np.arange(1 << 16, dtype=np.uint32)
    bf = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    hf = lambda b: b.astype(np.uint16).view(np.float16).astype(np.float64)
    r = rng(23)
    x = np.concatenate([r.standard_normal(300) * s for s in (1e-40, 1e-3, 1.0, 1e4)])
    mids = [1 + 2 ** -8, 1 + 2 ** -8 + 2 ** -30, 1 + 2 ** -8 - 2 ** -30, 1 + 3 * 2 ** -8, -(1 + 2 ** -8 + 2 ** -30),
            1 + 2 ** -11, 1 + 2 ** -11 + 2 ** -40, 1 + 2 ** -11 - 2 ** -40, 2.0 ** -134, 2.0 ** -134 * 1.0000001,
            2.0 ** -25, 2.0 ** -25 * 1.0000001, 65504.0, 65519.99, 65520.0, 3.3895313892515355e38, 3.4e38, 0.0, -0.0]
    x = np.concatenate([x, mids])
    with np.errstate(invalid="ignore"):  # the tables hold NaN patterns, dropped by _nearest_in_table
        assert np.array_equal(ref.round_bf16(x), _nearest_in_table(x, pats, bf))
        assert np.array_equal(ref.round_f16(x), _nearest_in_table(x, pats, hf))
    assert ref.round_bf16(np.array([1 + 2 ** -8 + 2 ** -30]))[0] == 1 + 2 ** -7
    # the double-rounding route (float32 first, then bf16, as torch converts) gives 1.0 there
    assert torch.tensor([1 + 2 ** -8 + 2 ** -30], dtype=torch.float64).float().to(torch.bfloat16).item() == 1.0
    assert np.isnan(ref.round_bf16(np.array([np.nan]))[0])


def test_ternary_wire_step_equals_signed_f32_step():
    r = rng(22)
    n = 40 * C
    th, ms, gs = r.standard_normal(n), [r.standard_normal(n)] * 2, [r.standard_normal(n), r.standard_normal(n)]
    for mode, k in ((ref.MODE_DEMO, 4), (ref.MODE_RANDOM, 8), (ref.MODE_DILOCO, 1)):
        a, _, _ = ref.step(th, ms, gs, beta=0.9, lr=0.1, k=k, mode=mode, sign=True, step_idx=7)
        b, _, _ = ref.step(th, ms, gs, beta=0.9, lr=0.1, k=k, mode=mode, sign=True, step_idx=7, wire=ref.WIRE_TERNARY)
        assert np.array_equal(a, b)
    with pytest.raises(ValueError):
        ref.step(th, ms, gs, beta=0.9, lr=0.1, k=4, mode=ref.MODE_DEMO, sign=False, wire=ref.WIRE_TERNARY)


# ----------------------------------------------------------------------------
# Decoupled AdamW
# ----------------------------------------------------------------------------

def test_adamw_single_replica_matches_torch():
    import torch

    r = rng(30)
    n = 5 * C
    theta0 = r.standard_normal(n)
    gs = [r.standard_normal(n) * 1e-2 for _ in range(4)]
    kw = dict(beta1=0.9, beta2=0.999, eps=1e-8, lr=1e-3, wd=0.1)
    p = torch.nn.Parameter(torch.tensor(theta0, dtype=torch.float64))
    opt = torch.optim.AdamW([p], lr=ref.f32(1e-3), betas=(ref.f32(0.9), ref.f32(0.999)), eps=ref.f32(1e-8),
                            weight_decay=ref.f32(0.1))
    th, m, v = theta0, [np.zeros(n)], [np.zeros(n)]
    for t, g in enumerate(gs):
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        th, m, v, _ = ref.adamw_step(th, m, v, [g], step_idx=t, **kw)
        assert np.abs(th - p.detach().numpy()).max() < 1e-14


def test_adamw_first_step_closed_form_and_replica_mean():
    r = rng(31)
    n = 3 * C
    theta0 = r.standard_normal(n)
    g = r.standard_normal(n)
    # t = 1: m_hat = g, v_hat = g^2, so u = g / (|g| + eps)
    th, _, _, U = ref.adamw_step(theta0, [np.zeros(n)], [np.zeros(n)], [g], beta1=0.9, beta2=0.99, eps=1e-3,
                                 lr=0.5, wd=0.0, step_idx=0)
    e = float(np.float32(1e-3))
    assert np.abs(U - g / (np.abs(g) + e)).max() < 1e-14
    assert np.abs(th - (theta0 - 0.5 * U)).max() < 1e-14
    # R identical replicas average to the single-replica direction; two opposite ones cancel
    _, _, _, U3 = ref.adamw_step(theta0, [np.zeros(n)] * 3, [np.zeros(n)] * 3, [g] * 3, beta1=0.9, beta2=0.99,
                                 eps=1e-3, lr=0.5, wd=0.0, step_idx=0)
    assert np.abs(U3 - U).max() < 1e-15
    _, _, _, U2 = ref.adamw_step(theta0, [np.zeros(n)] * 2, [np.zeros(n)] * 2, [g, -g], beta1=0.9, beta2=0.99,
                                 eps=1e-3, lr=0.5, wd=0.0, step_idx=0)
    assert np.abs(U2).max() == 0.0
