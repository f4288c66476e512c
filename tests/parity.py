"""Parity harness: the CUDA library against the float64 oracle, step by step.

Every check is teacher-forced: the oracle takes one step from the GPU's own
float32 state (promoted exactly to float64), so each step is checked on its own.
For each step the harness

* runs the split path (demo_encode per replica, demo_decode_update) and the
  fused path (demo_step) on copies of the same state and requires them to be
  bit-identical;
* reads the GPU's Q exactly by decoding the payloads onto a zero theta with
  lr = -1 (theta' = 0 + 1 * Q);
* compares against the oracle on the chunks in ``rows`` (all chunks by default):
  DeMo indices exactly (except chunks the oracle flags as near-ties), Random /
  Striding positions exactly (the new momentum is exactly 0 there), payload
  values to TOL relative to the chunk's largest magnitude; Q against the
  oracle's decode of the GPU's own payloads to TOL, and against the oracle's
  own Q to TOL relative to the mean of the summands' magnitudes (a mean of
  nearly opposite values cancels float32 rounding up); m to TOL
  relative to the larger of that and the chunk's momentum before the
  subtraction (k = 32 cancels it to rounding noise), and the theta update to
  within one float32 rounding of theta - lr Q.

Paths whose payloads stay inside the library (the pipelined step and its
no-allocation variant) are checked with ``oracle_step`` + ``check_outcome``:
the same m, Q and theta checks, with Q read by running the path once more on a
zero theta with lr = -1.
"""

import numpy as np
import torch

import decoupled_momentum_optimizer_gb300 as dm
import oracle.demo_ref as ref

C = 32
TOL = 1e-5  # max |gpu - oracle| / max |oracle| per chunk (float32 vs float64)


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def chunk_close(gpu, orc, tol, excl=None, scale=None):
    """Per-chunk infinity-norm relative check; returns (bad chunk mask, worst ratio).

    The denominator is the chunk's largest oracle magnitude, or the largest
    magnitude of ``scale`` when that is bigger (for results that cancel, such as
    the momentum left after the subtraction, the error scale is the input's).
    """
    a = gpu if gpu.ndim == 2 else gpu.reshape(-1, C)
    b = orc if orc.ndim == 2 else orc.reshape(-1, C)
    num = np.abs(a - b).max(1)
    den = np.abs(b).max(1)
    if scale is not None:
        sc = scale if scale.ndim == 2 else scale.reshape(-1, C)
        den = np.maximum(den, np.abs(sc).max(1))
    zero = den == 0
    bad = np.where(zero, num > 0, num > tol * den)
    if excl is not None:
        bad &= ~excl
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(zero, np.where(num > 0, np.inf, 0.0), num / np.where(zero, 1, den))
    if excl is not None:
        ratio = np.where(excl, 0.0, ratio)
    return bad, float(ratio.max()) if ratio.size else 0.0


WIRE_REL = {"f32": 0.0, "ternary": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}  # one unit of the format's mantissa
WIRE_ABS = {"f32": 0.0, "ternary": 0.0, "bf16": 0.0, "f16": 2.0 ** -24}  # fp16 subnormal spacing below 2^-14


def gpu_split(theta, ms, gs, *, k, beta, lr, mode, sign, seed, step, period, wire="f32"):
    n = theta.numel()
    ms2 = [m.clone() for m in ms]
    vals, idxs = [], []
    for r in range(len(ms)):
        v, i = dm.payload_buffers(mode, n, k, step=step, diloco_period=period, wire=wire)
        if v is not None:
            v.fill_(0)
        if i is not None:
            i.fill_(0)
        dm.encode(gs[r], ms2[r], v, i, k=k, beta=beta, mode=mode, sign=sign, diloco_period=period, seed=seed,
                  step=step, wire=wire)
        vals.append(v)
        idxs.append(i)
    # the same encodes as one demo_encode_replicas call: bit-identical momenta and payloads
    ms3 = [m.clone() for m in ms]
    bufs3 = [dm.payload_buffers(mode, n, k, step=step, diloco_period=period, wire=wire) for _ in ms]
    for b in bufs3:
        for t in b:
            if t is not None:
                t.fill_(0)
    vals3 = [b[0] for b in bufs3] if vals[0] is not None else None
    idx3 = [b[1] for b in bufs3] if mode == "demo" else None
    dm.encode_replicas(gs, ms3, vals3, idx3, k=k, beta=beta, mode=mode, sign=sign, diloco_period=period, seed=seed,
                       step=step, wire=wire)
    same = lambda a, b: torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))
    for r in range(len(ms)):
        assert same(ms3[r], ms2[r]), f"encode_replicas: m of replica {r} differs from demo_encode's"
        if vals3 is not None:
            assert same(vals3[r], vals[r]), f"encode_replicas: payload of replica {r} differs"
        if idx3 is not None:
            assert same(idx3[r], idxs[r]), f"encode_replicas: indices of replica {r} differ"
    th2 = theta.clone()
    dvals = vals if vals[0] is not None else [torch.zeros(4, device=theta.device)] * len(ms)
    if vals[0] is None and wire != "f32":
        dvals = [dm.payload_buffers("random", 32 * 32, 1, wire=wire)[0] for _ in ms]
    didx = idxs if mode == "demo" else None
    dm.decode_update(th2, dvals, didx, k=k, lr=lr, mode=mode, diloco_period=period, seed=seed, step=step, wire=wire)
    Q = torch.zeros_like(theta)
    dm.decode_update(Q, dvals, didx, k=k, lr=-1.0, mode=mode, diloco_period=period, seed=seed, step=step, wire=wire)
    return th2, ms2, vals, idxs, Q


def gpu_fused(theta, ms, gs, *, k, beta, lr, mode, sign, seed, step, period, wire="f32"):
    th2 = theta.clone()
    ms2 = [m.clone() for m in ms]
    dm.step(th2, gs, ms2, k=k, beta=beta, lr=lr, mode=mode, sign=sign, diloco_period=period, seed=seed, step=step,
            wire=wire)
    return th2, ms2


def gpu_pipelined(theta, gs, ms, *, k, beta, lr, mode, sign, seed, step, period, wire, blocks, comm, static=False):
    """One demo_step_pipelined call (payload buffers made here) or, with ``static``, one call of its
    no-allocation variant, updating theta and ms in place."""
    kw = dict(k=k, beta=beta, lr=lr, mode=mode, sign=sign, seed=seed, step=step, diloco_period=period, wire=wire,
              blocks=blocks, comm_stream=comm)
    if static:
        dm.step_pipelined_static(theta, gs, ms, **kw)
        return
    n = theta.numel()
    send = [dm.payload_buffers(mode, n, k, step=step, diloco_period=period, wire=wire) for _ in ms]
    recv = [dm.payload_buffers(mode, n, k, step=step, diloco_period=period, wire=wire) for _ in ms]
    dm.step_pipelined(theta, gs, ms, send if send[0][0] is not None else None,
                      recv if recv[0][0] is not None else None, **kw)


def check_pipelined_step(theta, ms, gs, *, k, beta, lr, mode, sign, seed, step, period, wire, blocks, comm,
                         static=False):
    """One teacher-forced pipelined step against the oracle: the step runs on a copy of the state
    with a zero theta and lr = -1 (which leaves theta = Q exactly) and on the state itself, which
    it updates in place; then m, Q and theta are compared with the oracle's step from the same
    start (check_outcome)."""
    rows, el_t, th0, m0, g0, info = oracle_step(theta, ms, gs, k=k, beta=beta, lr=lr, mode=mode, sign=sign,
                                                seed=seed, step=step, period=period, wire=wire)
    kw = dict(k=k, beta=beta, mode=mode, sign=sign, seed=seed, step=step, period=period, wire=wire, blocks=blocks,
              comm=comm, static=static)
    Q = torch.zeros_like(theta)
    gpu_pipelined(Q, gs, [m.clone() for m in ms], lr=-1.0, **kw)
    gpu_pipelined(theta, gs, ms, lr=lr, **kw)
    torch.cuda.synchronize()
    pick = lambda t: f64(t.index_select(0, el_t))
    check_outcome(info, m0, g0, th0, [pick(m) for m in ms], pick(Q), pick(theta), beta=beta, lr=lr, sign=sign,
                  wire=wire)
    return int(info["near_tie"].sum())


def host_payload(vals, idx, *, wire, mode, nc, k, rows):
    """The GPU's payload decoded on the host: (values [rows][kv] float64, indices [rows][k] or None)."""
    kv = C if mode == "diloco" else k
    if vals is None:
        return None, None
    if wire == "ternary":
        vw = vals.view(torch.int32).cpu().numpy().view(np.uint32).reshape(-1, kv, 2)
        iw = None if idx is None else idx.cpu().numpy().view(np.uint32).reshape(-1, k, 5)
        v, i = ref.ternary_unpack(vw, iw, nc)
        return v[rows], (None if i is None else i[rows])
    v = vals.view(nc, kv)
    v = f64(v.index_select(0, torch.from_numpy(rows).to(vals.device)))
    i = None
    if idx is not None:
        i = idx.view(nc, k).index_select(0, torch.from_numpy(rows).to(idx.device)).cpu().numpy().astype(np.int64)
    return v, i


def same_bits(a, b):
    """Bit-for-bit equality of two float32 tensors (NaN equals the same NaN; -0 differs from +0)."""
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def check_outcome(info, m0, g0, th0, m_gpu, Q_gpu, th_gpu, *, beta, lr, sign, wire="f32", excl=None, tol=TOL):
    """The GPU's new momenta, Q and theta of one step against the oracle's step ``info`` from the
    same start (all float64 arrays over the same chunks; chunks flagged in ``excl`` are skipped).

    m to TOL relative to the larger of the new m and the momentum before the subtraction;
    Q to TOL (plus one rounding unit of a 16-bit wire format when unsigned) relative to the
    mean of the summands' magnitudes; theta within one float32 rounding of theta - lr Q_gpu.
    """
    R = len(m0)
    nrows = th0.size // C
    if excl is None:
        excl = info["near_tie"].copy()
    wrel, wabs = WIRE_REL[wire], WIRE_ABS[wire]
    for r in range(R):
        x = ref.f32(beta) * m0[r] + g0[r]  # the momentum before the subtraction of q
        mg = m_gpu[r].reshape(nrows, C)
        bad, worst = chunk_close(mg, info["encodes"][r]["m"], tol, excl, scale=x)
        assert not bad.any(), f"m[{r}] differs in {bad.sum()} chunks (worst {worst:.3g})"
    # the mean of R replicas can cancel, so the error scale is the mean of |values|
    Yabs, _ = ref.scatter_mean([None if e["vals"] is None else np.abs(e["vals"]) for e in info["encodes"]],
                               [e["pos"] for e in info["encodes"]], nrows)
    if wabs and not sign:  # the fp16 floor is absolute: compare it against the summand scale
        Yabs = np.maximum(Yabs, wabs / max(tol + wrel, 1e-30))
    bad, worst = chunk_close(Q_gpu, info["Q"], tol + (0.0 if sign else wrel), excl, scale=Yabs)
    assert not bad.any(), f"Q differs in {bad.sum()} chunks (worst {worst:.3g})"
    # theta' = theta - lr Q with one float32 rounding (checked to one ulp)
    want = (th0 - ref.f32(lr) * Q_gpu).astype(np.float32)
    got = th_gpu.astype(np.float32)
    ulp = np.spacing(np.maximum(np.abs(want), np.abs(got)).astype(np.float32))
    assert (np.abs(got.astype(np.float64) - want.astype(np.float64)) <= ulp).all(), "theta update is not theta - lr Q"


def oracle_step(theta, ms, gs, *, k, beta, lr, mode, sign, seed=0, step=0, period=8, rows=None, wire="f32"):
    """The oracle's step on ``rows`` (default all chunks) of the GPU tensors' current values.

    Returns (rows, element index tensor, th0, m0, g0, info) with the inputs as float64 arrays."""
    nc = theta.numel() // C
    rows = np.arange(nc) if rows is None else np.asarray(rows, dtype=np.int64)
    el = (rows[:, None] * C + np.arange(C)[None, :]).reshape(-1)
    el_t = torch.from_numpy(el).to(theta.device)
    pick = lambda t: f64(t.index_select(0, el_t))
    th0, m0, g0 = pick(theta), [pick(m) for m in ms], [pick(g) for g in gs]
    _, _, info = ref.step(th0, m0, g0, beta=beta, lr=lr, k=k, mode=ref.__dict__["MODE_" + mode.upper()], sign=sign,
                          seed=seed, step_idx=step, period=period, chunk_ids=rows, wire=dm.WIRES[wire])
    return rows, el_t, th0, m0, g0, info


def check_step(theta, ms, gs, *, k, beta, lr, mode, sign, seed=0, step=0, period=8, rows=None, tol=TOL,
               stats=None, wire="f32"):
    """One teacher-forced step (see module docstring); returns the fused path's new (theta, ms)."""
    n = theta.numel()
    nc = n // C
    R = len(ms)
    th_s, ms_s, vals, idxs, Q = gpu_split(theta, ms, gs, k=k, beta=beta, lr=lr, mode=mode, sign=sign, seed=seed,
                                          step=step, period=period, wire=wire)
    th_f, ms_f = gpu_fused(theta, ms, gs, k=k, beta=beta, lr=lr, mode=mode, sign=sign, seed=seed, step=step,
                           period=period, wire=wire)
    torch.cuda.synchronize()
    assert same_bits(th_f, th_s), "fused and split theta differ"
    for r in range(R):
        assert same_bits(ms_f[r], ms_s[r]), f"fused and split m[{r}] differ"

    rows, el_t, th0, m0, g0, info = oracle_step(theta, ms, gs, k=k, beta=beta, lr=lr, mode=mode, sign=sign,
                                                seed=seed, step=step, period=period, rows=rows, wire=wire)

    def pick(t):
        return f64(t.index_select(0, el_t))

    wrel, wabs = WIRE_REL[wire], WIRE_ABS[wire]
    excl = info["near_tie"].copy()
    nrows = len(rows)

    payloads = [host_payload(vals[r], idxs[r], wire=wire, mode=mode, nc=nc, k=k, rows=rows) for r in range(R)]
    for r in range(R):
        enc = info["encodes"][r]
        mg = pick(ms_f[r]).reshape(nrows, C)
        gv, gi = payloads[r]
        if mode == "demo":
            oi = enc["idx"]
            same = (gi == oi).all(1)
            assert (same | excl).all(), f"DeMo indices differ in {(~same & ~excl).sum()} non-tied chunks"
            X = enc["X"]
            ov = np.take_along_axis(X, oi, axis=1)
            if sign:
                ov = np.sign(ov)
                okv = (gv == ov).all(1)
                assert (okv | excl).all(), "signed DeMo payload values differ"
            else:
                scale = np.abs(X).max(1, keepdims=True)
                errv = np.abs(gv - ov) <= wrel * np.abs(ov) + wabs + tol * np.where(scale == 0, 1, scale)
                assert (errv.all(1) | excl).all(), "DeMo payload values differ"
        elif mode in ("random", "stride"):
            pos = enc["pos"]
            at = np.take_along_axis(mg, pos, axis=1)
            assert (at == 0.0).all(), "new momentum is not exactly 0 at the oracle's positions"
            ov = enc["vals"]
            if sign:
                assert np.array_equal(gv, ov), "signed payload values differ"
            else:
                err = np.abs(gv - ov) <= wrel * np.abs(ov) + wabs + tol * np.abs(ov).max(1, keepdims=True)
                assert err.all(), "payload values differ"
        elif mode == "diloco" and enc["vals"] is not None:
            if sign:
                assert np.array_equal(gv, enc["vals"]), "signed DiLoCo payload differs"
            else:
                ov = enc["vals"]
                err = np.abs(gv - ov) <= wrel * np.abs(ov) + wabs + tol * np.abs(ov).max(1, keepdims=True)
                assert err.all(), "DiLoCo payload differs"
    Qg = pick(Q)
    # decode alone: the oracle's scatter-mean and inverse transform of the GPU's own payloads
    gpu_vals, gpu_pos = [], []
    for r in range(R):
        enc = info["encodes"][r]
        if enc["vals"] is None:
            continue
        gpu_vals.append(payloads[r][0])
        gpu_pos.append(payloads[r][1] if mode == "demo" else enc["pos"])
    _, Qd, _, _ = ref.decode_update(np.zeros(nrows * C), gpu_vals, gpu_pos, 0.0,
                                    ref.__dict__["MODE_" + mode.upper()])
    bad, worst = chunk_close(Qg, Qd, tol)
    assert not bad.any(), f"decode of the GPU payloads: Q differs in {bad.sum()} chunks (worst {worst:.3g})"
    check_outcome(info, m0, g0, th0, [pick(m) for m in ms_f], Qg, pick(th_f), beta=beta, lr=lr, sign=sign,
                  wire=wire, excl=excl, tol=tol)

    if stats is not None:
        stats.setdefault("near_tie", 0)
        stats["near_tie"] += int(excl.sum())
        stats.setdefault("chunks", 0)
        stats["chunks"] += nrows
    return th_f, ms_f
