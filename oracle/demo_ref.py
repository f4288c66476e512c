"""Plain float64 CPU oracle for the decoupled-momentum (DeMo / FlexDeMo) step.

TEST INFRASTRUCTURE ONLY.  This module is the slow, obviously-correct
statement of what the GPU library computes.  Only the test-suite, the
smoke check and the CPU-baseline / reference legs of the benchmark may import
it.  It shares no code, tables, constants or helpers with the CUDA path, and it
never imports the product package.

Sources (cited by page title and section):

* "DeToNATION: Decoupled Torch Network-Aware Training on Interlinked Online
  Nodes" (Paper-Notes, AAAI 2026), section "方法详解", subsection "1. FlexDeMo
  优化器", Algorithm 1 -- the per-shard step: momentum accumulation,
  extraction of the fast components, their removal from the momentum,
  synchronisation of q in the replication group R, and the parameter update
  with the synchronised Q.
* Same page, subsection "2. 复制方案 (Replication Schemes)", scheme table --
  DeMo (DCT-II, indices sent), Random (shared seed, no indices), Striding
  (equally spaced, no indices), DiLoCo (full sync every n steps).
* Same page, subsection "3. Sign 函数与超参数分析" -- ternary sign before
  sync, chunk size 32, TopK 4.
* "DeMo: Decoupled Momentum Optimization" (arXiv 2411.19870), abstract --
  orthonormal transform (DCT) + top-k, momentum subtraction as error feedback.

Readings where the pages leave a step open (each one is listed in the design
notes of the repository):

* DCT: the orthonormal 1-D DCT-II of every length-32 chunk (Ahmed, Natarajan
  & Rao 1974), inverse = transpose (DCT-III).
* top-k key |X_u|; exact ties go to the lowest u.  The payload lists the kept
  coefficients in ASCENDING u order (a canonical wire order).
* error feedback subtracts the UNSIGNED q; the sign (ternary, sign(0) = 0) is
  applied only to the transmitted values, in every mode when the flag is set.
* scatter-mean divides each slot by the number of replicas that sent it.
* Random: k draws per chunk by partial Fisher-Yates over the 32 positions; draw
  j uses H(seed, step, chunk, j) built from splitmix64 and Lemire's
  multiply-shift range reduction.  Payload in draw order.
* Striding: stride n_s = 32 / k, offset = step mod n_s.
* DiLoCo: the whole momentum is sent on steps with (step + 1) mod H == 0 and
  nothing otherwise; theta moves only on those steps.
* beta and lr are rounded to float32 first (the GPU computes in float32).

Parity status: every function here is pinned by the CPU tests
(``tests/test_oracle_pins.py``) against closed forms, a library DCT, brute
force and published splitmix64 outputs.  The composed multi-step trajectory is
pinned where mathematics fixes it.  Sign off: with beta = 1 every scheme
conserves beta m + g = m' + q, so theta after T steps follows from the end
momenta alone, and Striding under a constant gradient has a closed form for any
beta.  Sign on: a DeMo chunk that is one cosine of the basis keeps exactly that
coefficient with k = 1, drains to zero momentum every step and moves theta by
the mean of the replicas' signs times that basis vector; under a constant
gradient every Striding, Random or DiLoCo send carries the sign of the gradient
(an accumulation of it), so theta moves by the mean sign once per send and the
momentum holds the geometric sum since the last send.
"""

import math

import numpy as np

CHUNK = 32

MODE_DEMO = 0
MODE_RANDOM = 1
MODE_STRIDE = 2
MODE_DILOCO = 3
MODE_NAMES = {MODE_DEMO: "demo", MODE_RANDOM: "random", MODE_STRIDE: "stride", MODE_DILOCO: "diloco"}

NEAR_TIE_REL = 1e-6

_M64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15  # splitmix64 increment (golden-ratio constant)


# ----------------------------------------------------------------------------
# float32 rounding of the step constants
# ----------------------------------------------------------------------------

def f32(x):
    """The float64 value of ``x`` rounded to float32 (the GPU's beta / lr)."""
    return float(np.float32(x))


# ----------------------------------------------------------------------------
# The orthonormal DCT-II of one chunk
# ----------------------------------------------------------------------------

def dct_matrix(C=CHUNK):
    """Orthonormal DCT-II matrix D[u][i] = a_u cos(pi (2i+1) u / (2C)).

    a_0 = sqrt(1/C), a_u = sqrt(2/C) for u >= 1.  X = D x is the transform of a
    chunk x and x = D^T X its inverse (DeMo abstract: an orthonormal
    transform such as the DCT; DeToNATION notes, replication table, DeMo row:
    DCT-II).
    """
    D = np.empty((C, C), dtype=np.float64)
    for u in range(C):
        a = math.sqrt((1.0 if u == 0 else 2.0) / C)
        for i in range(C):
            D[u, i] = a * math.cos(math.pi * (2 * i + 1) * u / (2 * C))
    return D


_D = dct_matrix()


# ----------------------------------------------------------------------------
# splitmix64 and the shared-seed index generator
# ----------------------------------------------------------------------------

def splitmix64_mix(z):
    """The splitmix64 output function applied to the state ``z`` + gamma.

    splitmix64 (Steele, Lea & Flood, OOPSLA 2014; Vigna's public-domain C
    version): state += 0x9e3779b97f4a7c15, then two xor-shift-multiply rounds
    and a final xor-shift.  Calling this on s, s+gamma, s+2 gamma, ... yields
    the generator's output stream for seed s.
    """
    z = (z + _GAMMA) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def splitmix64_stream(seed, count):
    """First ``count`` outputs of a splitmix64 generator seeded with ``seed``."""
    out = []
    state = seed & _M64
    for _ in range(count):
        out.append(splitmix64_mix(state))
        state = (state + _GAMMA) & _M64
    return out


def index_hash(seed, step, chunk, j):
    """H(s, t, c, j) = sm(sm(sm(sm(s) ^ t) ^ c) ^ j) on 64-bit words.

    The shared seed makes every replica draw the same positions, so no index
    is transmitted (DeToNATION notes, replication table, Random row: indices
    are not sent because the seed is shared).
    """
    h = splitmix64_mix(seed & _M64)
    h = splitmix64_mix(h ^ (step & _M64))
    h = splitmix64_mix(h ^ (chunk & _M64))
    return splitmix64_mix(h ^ (j & _M64))


def random_positions(seed, step, chunk, k, C=CHUNK):
    """k distinct positions of one chunk, in draw order (partial Fisher-Yates).

    Draw j takes r_j = floor(hi32(H) * (C - j) / 2^32) (Lemire's multiply-shift
    reduction to [0, C - j)) and picks the r_j-th still-free position counting
    upward from 0.
    """
    free = list(range(C))
    pos = []
    for j in range(k):
        h = index_hash(seed, step, chunk, j)
        r = ((h >> 32) * (C - j)) >> 32
        pos.append(free.pop(r))
    return pos


def stride_positions(step, k, C=CHUNK):
    """Equally spaced positions o + n_s j, n_s = C / k, o = step mod n_s."""
    if C % k != 0:
        raise ValueError("striding needs k to divide the chunk size")
    ns = C // k
    o = step % ns
    return [o + ns * j for j in range(k)]


def diloco_is_sync(step, period):
    """DiLoCo sends the full momentum once every ``period`` steps."""
    return (step + 1) % period == 0


# ----------------------------------------------------------------------------
# Top-k by magnitude
# ----------------------------------------------------------------------------

def topk_select(X, k):
    """Per row of X, the k slots of largest |X_u|; exact ties go to the lowest u.

    Returns (kept [rows, k] in ascending u, order [rows, C]) where ``order`` is
    the full ranking by the key (-|X_u|, u) (a stable sort keeps equal keys in
    index order).  DeMo abstract: the transform is followed by a top-k
    sparsification.
    """
    X = np.atleast_2d(np.asarray(X, dtype=np.float64))
    order = np.argsort(-np.abs(X), axis=1, kind="stable")
    kept = np.sort(order[:, :k], axis=1)
    return kept, order


# ----------------------------------------------------------------------------
# One replica's encode: momentum, extraction, error feedback, payload
# ----------------------------------------------------------------------------

def _ternary_sign(v):
    return np.sign(v)  # -1, 0 or +1; sign(0) = 0


def encode(m, g, beta, k, mode, sign, seed=0, step=0, period=8, chunk_ids=None):
    """Algorithm 1's accumulation, extraction and removal for one replica, plus its payload.

    m, g: float64 arrays of length n (n a multiple of 32); g holds the exact
    float32 / bfloat16 gradient values.  Returns a dict with

    * ``m``: the new momentum (after the subtraction of q),
    * ``q``: the extracted component, [nc, 32],
    * ``vals``: payload values ([nc, k]; DiLoCo: [nc, 32] on sync steps, None
      otherwise), signed when ``sign`` is set,
    * ``idx``: payload indices [nc, k] (DeMo only, ascending u), else None,
    * ``pos``: the positions selected in each chunk ([nc, k]; DiLoCo: all 32),
    * ``X``: the DCT coefficients (DeMo only),
    * ``near_tie``: bool [nc], chunks whose selection or sign is decided by a
      gap below 1e-6 of the chunk's largest coefficient (DeMo only).
    """
    m = np.asarray(m, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    n = m.shape[0]
    assert n % CHUNK == 0
    nc = n // CHUNK
    if chunk_ids is None:
        chunk_ids = np.arange(nc, dtype=np.int64)

    # Momentum accumulation: m <- beta m + Delta.
    x = (f32(beta) * m + g).reshape(nc, CHUNK)

    q = np.zeros_like(x)
    out = {"X": None, "idx": None, "near_tie": np.zeros(nc, dtype=bool)}

    if mode == MODE_DEMO:
        # Extraction: DCT-II of every chunk, keep the top-k by magnitude.
        X = x @ _D.T  # X[c, u] = sum_i D[u, i] x[c, i]
        kept, order = topk_select(X, k)
        mag = np.abs(X)
        rows = np.arange(nc)[:, None]
        Xs = np.zeros_like(X)
        Xs[rows, kept] = X[rows, kept]
        q = Xs @ _D  # inverse transform of the kept coefficients
        vals = X[rows, kept]
        # Near-tie diagnostics (for parity checks against a float32 kernel).
        srt = np.take_along_axis(mag, order, axis=1)
        top = srt[:, 0]
        tie = np.zeros(nc, dtype=bool)
        if k < CHUNK:
            tie |= (srt[:, k - 1] - srt[:, k]) <= NEAR_TIE_REL * top
        if sign:
            tie |= (np.abs(vals) <= NEAR_TIE_REL * top[:, None]).any(axis=1)
        out.update(X=X, idx=kept.astype(np.int64), pos=kept.astype(np.int64), near_tie=tie)
    elif mode in (MODE_RANDOM, MODE_STRIDE):
        pos = np.empty((nc, k), dtype=np.int64)
        for row in range(nc):
            if mode == MODE_RANDOM:
                pos[row] = random_positions(seed, step, int(chunk_ids[row]), k)
            else:
                pos[row] = stride_positions(step, k)
        rows = np.arange(nc)[:, None]
        q[rows, pos] = x[rows, pos]
        vals = x[rows, pos]
        out.update(pos=pos)
    elif mode == MODE_DILOCO:
        if diloco_is_sync(step, period):
            q = x.copy()
            vals = x.copy()
            out.update(pos=np.tile(np.arange(CHUNK), (nc, 1)))
        else:
            vals = None
            out.update(pos=None)
    else:
        raise ValueError("unknown mode")

    if vals is not None and sign:
        vals = _ternary_sign(vals)

    # Removal from the momentum: m <- m - q (the unsigned extracted component).
    out["m"] = (x - q).reshape(n)
    out["q"] = q
    out["vals"] = vals
    return out


# ----------------------------------------------------------------------------
# Combine the replicas' payloads and update the parameters
# ----------------------------------------------------------------------------

def scatter_mean(vals_list, pos_list, nc):
    """Per chunk and slot: sum of the replicas' values / number of senders.

    Replicas are summed in order r = 0..R-1; empty slots stay 0.
    """
    S = np.zeros((nc, CHUNK), dtype=np.float64)
    cnt = np.zeros((nc, CHUNK), dtype=np.int64)
    rows = np.arange(nc)
    for vals, pos in zip(vals_list, pos_list):
        if vals is None:
            continue
        for j in range(pos.shape[1]):
            S[rows, pos[:, j]] += vals[:, j]
            cnt[rows, pos[:, j]] += 1
    Y = np.zeros_like(S)
    nz = cnt > 0
    Y[nz] = S[nz] / cnt[nz]
    return Y, cnt


def decode_update(theta, vals_list, pos_list, lr, mode, wire=0):
    """Algorithm 1's synchronisation (combine) and parameter update (theta <- theta - lr Q).

    DeMo: Q = D^T Y (inverse DCT of the scatter-mean); the other schemes send
    values in the parameter domain, so Q = Y.  ``wire`` rounds the received
    values as the wire format does (see the wire-format section below).
    """
    theta = np.asarray(theta, dtype=np.float64)
    n = theta.shape[0]
    nc = n // CHUNK
    vals_list = [wire_round(v, wire) for v in vals_list]
    Y, cnt = scatter_mean(vals_list, pos_list, nc)
    Q = Y @ _D if mode == MODE_DEMO else Y
    new_theta = theta - f32(lr) * Q.reshape(n)
    return new_theta, Q, Y, cnt


def step(theta, ms, gs, *, beta, lr, k, mode, sign, seed=0, step_idx=0, period=8, chunk_ids=None, wire=0):
    """One full step over R replicas: encode every replica, combine, update.

    Returns (theta_new, [m_r new], info) where info holds the payloads, Q and
    the per-replica near-tie flags.  ``wire`` is the payload encoding (the
    ternary format needs the sign flag).
    """
    if wire == WIRE_TERNARY and not sign:
        raise ValueError("the ternary wire format carries signed values only")
    encs = [
        encode(m, g, beta, k, mode, sign, seed=seed, step=step_idx, period=period, chunk_ids=chunk_ids)
        for m, g in zip(ms, gs)
    ]
    vals_list = [e["vals"] for e in encs]
    pos_list = [e["pos"] for e in encs]
    new_theta, Q, Y, cnt = decode_update(theta, vals_list, pos_list, lr, mode, wire=wire)
    info = {
        "encodes": encs,
        "Q": Q,
        "Y": Y,
        "cnt": cnt,
        "near_tie": np.any([e["near_tie"] for e in encs], axis=0),
    }
    return new_theta, [e["m"] for e in encs], info


# ----------------------------------------------------------------------------
# Wire-format size (bytes per replica) of one step's payload
# ----------------------------------------------------------------------------

def payload_bytes(mode, n, k, step=0, period=8, idx_bytes_per_entry=1):
    """(value bytes, index bytes) one replica sends for a step.

    DeMo sends k float32 values and k indices per chunk; Random and Striding
    send only the k values (indices come from the shared seed / the step);
    DiLoCo sends the n float32 momentum values on sync steps and nothing
    otherwise (DeToNATION notes, replication table, the column on whether a
    scheme must send its indices).
    """
    nc = n // CHUNK
    if mode == MODE_DEMO:
        return nc * k * 4, nc * k * idx_bytes_per_entry
    if mode in (MODE_RANDOM, MODE_STRIDE):
        return nc * k * 4, 0
    if mode == MODE_DILOCO:
        return (n * 4 if diloco_is_sync(step, period) else 0), 0
    raise ValueError("unknown mode")


# ----------------------------------------------------------------------------
# Wire formats of the payload (the compact encodings of the sent values)
# ----------------------------------------------------------------------------
#
# WIRE_F32:     values float32 [nc][kv], DeMo indices uint8 [nc][k].
# WIRE_TERNARY: sign must be on.  Chunks are grouped in tiles of 32 (chunk c is
#               bit c mod 32 of tile c // 32).  Values: uint32 [T][kv][2], word 0
#               has bit l set when value j of chunk 32t+l is nonzero, word 1 when it
#               is negative.  DeMo indices: uint32 [T][k][5], word b holds bit b of
#               index j of each chunk of the tile.  T = ceil(nc / 32); bits of
#               chunks past nc are 0.
# WIRE_BF16 / WIRE_F16: values rounded to nearest-even bfloat16 / float16,
#               [nc][kv] 16-bit words; indices as WIRE_F32.
# kv = k for DeMo, Random and Striding, 32 for DiLoCo.  The sign subsection of
# the DeToNATION notes gives the three values; the fp32-versus-fp16 comparison
# of the same subsection is what the 16-bit formats measure.

WIRE_F32 = 0
WIRE_TERNARY = 1
WIRE_BF16 = 2
WIRE_F16 = 3


def round_bf16(x):
    """float64 -> nearest bfloat16 (ties to even), returned as float64.

    bfloat16 keeps 8 significant bits and float32's exponent range: a normal
    value in [2^(e-1), 2^e) is a multiple of 2^(e-8), and below 2^-126 the
    spacing is the subnormal step 2^-133.  The value is rounded once, from its
    full float64 value, to the nearest multiple of that spacing (half to even);
    results of 2^128 or more overflow to infinity.  Scaling by a power of two is
    exact in float64, so np.round sees the exact quotient.
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x) & (x != 0.0)
    _, e = np.frexp(x[fin])  # |x| in [2^(e-1), 2^e)
    q = np.ldexp(1.0, np.maximum(e - 8, -133))
    r = np.round(x[fin] / q) * q
    r[np.abs(r) >= 2.0 ** 128] = np.inf * np.sign(r[np.abs(r) >= 2.0 ** 128])
    out[fin] = r
    return out


def round_f16(x):
    """float64 -> nearest float16 (ties to even), returned as float64.

    numpy converts float64 to float16 in one rounding, from the full value.
    """
    with np.errstate(over="ignore"):  # beyond the largest float16 the result is an infinity
        return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def wire_round(vals, wire):
    """The value a receiver decodes from ``vals`` sent in ``wire``."""
    if vals is None or wire in (WIRE_F32, WIRE_TERNARY):
        return vals
    if wire == WIRE_BF16:
        return round_bf16(vals)
    if wire == WIRE_F16:
        return round_f16(vals)
    raise ValueError("unknown wire format")


def ternary_pack(vals, idx=None):
    """Pack ternary values [nc][kv] (and DeMo indices [nc][k]) into tile bit-planes."""
    vals = np.asarray(vals)
    nc, kv = vals.shape
    T = (nc + 31) // 32
    vw = np.zeros((T, kv, 2), dtype=np.uint64)
    iw = None if idx is None else np.zeros((T, idx.shape[1], 5), dtype=np.uint64)
    for c in range(nc):
        t, lane = divmod(c, 32)
        for j in range(kv):
            v = vals[c, j]
            if v not in (-1.0, 0.0, 1.0):
                raise ValueError("ternary wire format needs values in {-1, 0, 1}")
            if v != 0:
                vw[t, j, 0] |= 1 << lane
            if v < 0:
                vw[t, j, 1] |= 1 << lane
        if idx is not None:
            for j in range(idx.shape[1]):
                for b in range(5):
                    if (int(idx[c, j]) >> b) & 1:
                        iw[t, j, b] |= 1 << lane
    return vw.astype(np.uint32), (None if iw is None else iw.astype(np.uint32))


def ternary_unpack(vw, iw, nc):
    """Inverse of ternary_pack: values [nc][kv] as float64 and indices [nc][k] (or None)."""
    T, kv, _ = vw.shape
    vals = np.zeros((nc, kv))
    idx = None if iw is None else np.zeros((nc, iw.shape[1]), dtype=np.int64)
    for c in range(nc):
        t, lane = divmod(c, 32)
        for j in range(kv):
            nz = (int(vw[t, j, 0]) >> lane) & 1
            neg = (int(vw[t, j, 1]) >> lane) & 1
            vals[c, j] = 0.0 if not nz else (-1.0 if neg else 1.0)
        if iw is not None:
            for j in range(iw.shape[1]):
                idx[c, j] = sum(((int(iw[t, j, b]) >> lane) & 1) << b for b in range(5))
    return vals, idx


def payload_bytes_wire(mode, n, k, step=0, period=8, wire=WIRE_F32):
    """(value bytes, index bytes) one replica sends in ``wire`` for one step."""
    nc = n // CHUNK
    T = (nc + 31) // 32
    if mode == MODE_DILOCO:
        if not diloco_is_sync(step, period):
            return 0, 0
        kv = CHUNK
    else:
        kv = k
    if wire == WIRE_TERNARY:
        vb = T * kv * 8
        ib = T * k * 20 if mode == MODE_DEMO else 0
    else:
        vb = nc * kv * (4 if wire == WIRE_F32 else 2)
        ib = nc * k if mode == MODE_DEMO else 0
    return vb, ib


# ----------------------------------------------------------------------------
# Decoupled AdamW (moments local to each replica, update directions synced)
# ----------------------------------------------------------------------------
#
# DeToNATION notes, method section, "4. Decoupled AdamW": an AdamW variant whose
# first and second moments (the EMA of the gradient and of its square) are not
# synchronised; the ViT-B bandwidth table runs it with full synchronisation.
# Reading taken: every replica updates its own moments and forms its AdamW
# direction u_r = m_hat_r / (sqrt(v_hat_r) + eps) (Loshchilov & Hutter's AdamW,
# bias-corrected with the 1-based step t); the replicas' directions are averaged
# densely (full sync) and theta <- theta - lr (mean_r u_r + wd theta).

def adamw_step(theta, ms, vs, gs, *, beta1, beta2, eps, lr, wd, step_idx):
    """One Decoupled-AdamW step over R replicas; step_idx is 0-based (t = step_idx + 1).

    Returns (theta_new, [m_r], [v_r], U) with U the mean direction.
    """
    b1, b2, e, lr32, wd32 = f32(beta1), f32(beta2), f32(eps), f32(lr), f32(wd)
    t = step_idx + 1
    bc1 = 1.0 - b1 ** t
    bc2 = 1.0 - b2 ** t
    theta = np.asarray(theta, dtype=np.float64)
    new_m, new_v, us = [], [], []
    for m, v, g in zip(ms, vs, gs):
        g = np.asarray(g, dtype=np.float64)
        m = b1 * np.asarray(m, dtype=np.float64) + (1.0 - b1) * g
        v = b2 * np.asarray(v, dtype=np.float64) + (1.0 - b2) * g * g
        us.append((m / bc1) / (np.sqrt(v / bc2) + e))
        new_m.append(m)
        new_v.append(v)
    U = sum(us) / len(us)
    return theta - lr32 * (U + wd32 * theta), new_m, new_v, U
