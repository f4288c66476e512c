"""The C ABI without a GPU: the library builds, loads, exports every declared
entry point, and its host-only logic (argument checks, payload sizes, status
strings) behaves as include/demo.h states.  No call here reaches a kernel:
argument checks run before any CUDA call, and valid arguments stop at
DEMO_ENOTINIT / DEMO_ENODEV on a machine without a GPU.
"""

import ctypes
import os
import re

import pytest

import oracle.demo_ref as ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "demo.h")

OK, EINVAL, EALIGN, ENODEV, ECUDA, ENOTINIT = 0, -1, -2, -3, -4, -5


@pytest.fixture(scope="module")
def L():
    from decoupled_momentum_optimizer_gb300 import build

    build.build()
    import decoupled_momentum_optimizer_gb300 as dm

    return dm.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(demo_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "demo_step" in names and "demo_encode" in names and "demo_decode_update" in names
    for name in names:
        assert hasattr(L, name), f"{name} declared in demo.h but not exported"


def test_status_strings(L):
    for code in (OK, EINVAL, EALIGN, ENODEV, ECUDA, ENOTINIT):
        assert L.demo_status_string(code).decode().startswith("DEMO_")
    assert b"UNKNOWN" in L.demo_status_string(12345)


def test_payload_bytes_match_oracle(L):
    import decoupled_momentum_optimizer_gb300 as dm

    for mode in ("demo", "random", "stride", "diloco"):
        for n in (32, 65536, 222903552):
            for k in (1, 2, 4, 8, 32):
                for step in (0, 6, 7):
                    got = dm.payload_bytes(mode, n, k, step=step, diloco_period=8)
                    want = ref.payload_bytes(dm.MODES[mode], n, k, step=step, period=8)
                    assert got == want, (mode, n, k, step)
    for wire in ("f32", "ternary", "bf16", "f16"):
        for mode in ("demo", "random", "diloco"):
            for n in (32, 32 * 33, 222903552):
                for step in (6, 7):
                    got = dm.payload_bytes(mode, n, 4, step=step, diloco_period=8, wire=wire)
                    want = ref.payload_bytes_wire(dm.MODES[mode], n, 4, step=step, period=8, wire=dm.WIRES[wire])
                    assert got == want, (wire, mode, n, step)
    assert dm.payload_bytes("stride", 64, 3) == (0, 0)  # invalid: 3 does not divide 32
    assert dm.payload_bytes("demo", 33, 4) == (0, 0)


F = ctypes.c_void_p


def p(a):
    return ctypes.c_void_p(a)


def encode_call(L, **kw):
    a = dict(g=p(0x10000), gd=0, m=p(0x20000), n=64, chunk=32, k=4, beta=0.9, mode=0, sign=1, period=8, seed=0,
             step=0, vals=p(0x30000), idx=p(0x40000), stream=None)
    a.update(kw)
    return L.demo_encode(a["g"], a["gd"], a["m"], a["n"], a["chunk"], a["k"], a["beta"], a["mode"], a["sign"],
                         a["period"], a["seed"], a["step"], a["vals"], a["idx"], a["stream"])


def step_call(L, R=2, **kw):
    gs = kw.pop("gs", [0x100000 * (r + 1) for r in range(R)])
    ms = kw.pop("ms", [0x1000000 * (r + 1) for r in range(R)])
    a = dict(theta=p(0x500000000), n=64, chunk=32, k=4, beta=0.9, lr=0.1, mode=0, sign=1, R=R, gd=0, period=8,
             seed=0, step=0, stream=None)
    a.update(kw)
    garr = (ctypes.c_void_p * max(1, len(gs)))(*gs)
    marr = (ctypes.c_void_p * max(1, len(ms)))(*ms)
    return L.demo_step(a["theta"], a["n"], a["chunk"], a["k"], a["beta"], a["lr"], a["mode"], a["sign"], a["R"],
                       garr, a["gd"], marr, a["period"], a["seed"], a["step"], a["stream"])


def test_encode_argument_checks(L):
    assert encode_call(L, chunk=16) == EINVAL
    assert encode_call(L, n=0) == EINVAL
    assert encode_call(L, n=48) == EINVAL
    assert encode_call(L, k=0) == EINVAL
    assert encode_call(L, k=33) == EINVAL
    assert encode_call(L, mode=2, k=3) == EINVAL
    assert encode_call(L, mode=7) == EINVAL
    assert encode_call(L, sign=2) == EINVAL
    assert encode_call(L, gd=5) == EINVAL
    assert encode_call(L, beta=float("nan")) == EINVAL
    assert encode_call(L, g=None) == EINVAL
    assert encode_call(L, idx=None) == EINVAL  # DeMo needs indices
    assert encode_call(L, mode=3, period=0) == EINVAL
    assert encode_call(L, g=p(0x10004)) == EALIGN
    assert encode_call(L, vals=p(0x30008)) == EALIGN
    assert encode_call(L, m=p(0x10000)) == EINVAL  # m overlaps g
    # the payload is written: n = 64, k = 4 gives 32 value bytes and 8 index bytes
    assert encode_call(L, vals=p(0x20010)) == EINVAL  # values inside m
    assert encode_call(L, vals=p(0x10000 + 240)) == EINVAL  # values overlap the end of g
    assert encode_call(L, idx=p(0x30010)) == EINVAL  # indices inside the values
    assert encode_call(L, idx=p(0x30020)) in (ENOTINIT, ENODEV)  # indices right after the values
    # valid arguments reach the device check
    assert encode_call(L) in (ENOTINIT, ENODEV)
    assert encode_call(L, mode=1, idx=None) in (ENOTINIT, ENODEV)
    assert encode_call(L, mode=3, vals=None, step=0, period=8) in (ENOTINIT, ENODEV)  # no payload off-sync
    assert encode_call(L, mode=3, vals=None, step=7, period=8) == EINVAL  # sync step needs a payload buffer


def test_step_argument_checks(L):
    assert step_call(L, R=0, gs=[], ms=[]) == EINVAL
    assert step_call(L, R=65, gs=[0x100000 * (r + 1) for r in range(65)],
                     ms=[0x100000000 + 0x1000000 * r for r in range(65)]) == EINVAL
    assert step_call(L, lr=float("inf")) == EINVAL
    assert step_call(L, theta=None) == EINVAL
    assert step_call(L, theta=p(0x500000004)) == EALIGN
    assert step_call(L, ms=[0x1000000, 0x1000000]) == EINVAL  # two replicas share one momentum buffer
    assert step_call(L, ms=[0x1000000, 0x500000000]) == EINVAL  # a momentum buffer is theta
    assert step_call(L, gs=[0x100000, 0x100000]) in (ENOTINIT, ENODEV)  # shared read-only gradient is fine
    assert step_call(L) in (ENOTINIT, ENODEV)


def test_decode_argument_checks(L):
    vals = (ctypes.c_void_p * 2)(0x30000, 0x40000)
    idx = (ctypes.c_void_p * 2)(0x50000, 0x60000)
    th = p(0x70000)
    assert L.demo_decode_update(th, 64, 32, 4, 0.1, 0, 2, vals, None, 8, 0, 0, None) == EINVAL
    assert L.demo_decode_update(th, 64, 32, 4, 0.1, 0, 0, vals, idx, 8, 0, 0, None) == EINVAL
    bad = (ctypes.c_void_p * 2)(0x30000, 0x40001)
    assert L.demo_decode_update(th, 64, 32, 4, 0.1, 1, 2, bad, None, 8, 0, 0, None) == EALIGN
    assert L.demo_decode_update(th, 64, 32, 4, 0.1, 0, 2, vals, idx, 8, 0, 0, None) in (ENOTINIT, ENODEV)
    # theta (256 bytes at 0x70000) is written while the payloads are read
    inside = (ctypes.c_void_p * 2)(0x30000, 0x70040)
    assert L.demo_decode_update(th, 64, 32, 4, 0.1, 0, 2, inside, idx, 8, 0, 0, None) == EINVAL
    idx_in = (ctypes.c_void_p * 2)(0x50000, 0x700f0)
    assert L.demo_decode_update(th, 64, 32, 4, 0.1, 0, 2, vals, idx_in, 8, 0, 0, None) == EINVAL
    shared = (ctypes.c_void_p * 2)(0x30000, 0x30000)  # read-only payloads may be shared
    assert L.demo_decode_update(th, 64, 32, 4, 0.1, 0, 2, shared, idx, 8, 0, 0, None) in (ENOTINIT, ENODEV)


def pipelined_call(L, sv, si, rv, ri, R=2):
    g = (ctypes.c_void_p * R)(*[0x100000 * (r + 1) for r in range(R)])
    m = (ctypes.c_void_p * R)(*[0x1000000 * (r + 1) for r in range(R)])
    arr = lambda xs: (ctypes.c_void_p * R)(*xs)
    return L.demo_step_pipelined(p(0x500000000), 64, 32, 4, 0.9, 0.1, 0, 1, R, g, 0, m, 8, 0, 0, 0, arr(sv), arr(si),
                                 arr(rv), arr(ri), 2, None, None)


def test_pipelined_buffer_checks(L):
    sv, si = [0x30000, 0x31000], [0x32000, 0x33000]
    rv, ri = [0x34000, 0x35000], [0x36000, 0x37000]
    assert pipelined_call(L, sv, si, rv, ri) in (ENOTINIT, ENODEV)
    assert pipelined_call(L, sv, si, sv, ri) == EINVAL  # receive values are the send values
    assert pipelined_call(L, sv, si, [0x34000, 0x34010], ri) == EINVAL  # two replicas' receive values overlap
    assert pipelined_call(L, sv, [0x32000, 0x31010], rv, ri) == EINVAL  # indices inside another replica's values
    assert pipelined_call(L, sv, si, [0x500000040, 0x35000], ri) == EINVAL  # receive values inside theta
    assert pipelined_call(L, sv, si, rv, [0x36000, 0x1000000]) == EINVAL  # receive indices inside m[0]
    assert pipelined_call(L, [0x100000, 0x31000], si, rv, ri) == EINVAL  # send values inside g[0]


def replicas_call(L, gs=None, ms=None, vals=None, idx=None, R=2, mode=0, step=0):
    arr = lambda xs: (ctypes.c_void_p * R)(*xs) if xs is not None else None
    gs = gs if gs is not None else [0x100000 * (r + 1) for r in range(R)]
    ms = ms if ms is not None else [0x1000000 * (r + 1) for r in range(R)]
    return L.demo_encode_replicas(arr(gs), 0, arr(ms), 64, 32, 4, 0.9, mode, 1, R, 8, 0, step, 0, arr(vals), arr(idx),
                                  None)


def test_encode_replicas_buffer_checks(L):
    # n = 64, DeMo k = 4: 32 bytes of values and 8 of indices per replica
    sv, si = [0x30000, 0x31000], [0x32000, 0x33000]
    assert replicas_call(L, vals=sv, idx=si) in (ENOTINIT, ENODEV)
    assert replicas_call(L, gs=[0x100000, 0x100000], vals=sv, idx=si) in (ENOTINIT, ENODEV)  # shared gradients
    assert replicas_call(L, R=0, gs=[], ms=[], vals=[], idx=[]) == EINVAL
    assert replicas_call(L, ms=[0x1000000, 0x1000000], vals=sv, idx=si) == EINVAL  # one momentum for two replicas
    assert replicas_call(L, ms=[0x1000000, 0x100000], vals=sv, idx=si) == EINVAL  # m[1] is g[0]
    assert replicas_call(L, vals=[0x30000, 0x30010], idx=si) == EINVAL  # two replicas' values overlap
    assert replicas_call(L, vals=sv, idx=[0x31010, 0x33000]) == EINVAL  # indices inside another replica's values
    assert replicas_call(L, vals=[0x1000000 + 64, 0x31000], idx=si) == EINVAL  # values inside m[0]
    assert replicas_call(L, vals=[0x30000, 0x2000000], idx=si) == EINVAL  # values inside m[1]: a replica's own
    assert replicas_call(L, vals=sv, idx=None) == EINVAL  # DeMo needs indices
    assert replicas_call(L, vals=[0x30008, 0x31000], idx=si) == EALIGN
    # DiLoCo between syncs sends nothing: no payload buffers
    assert replicas_call(L, mode=3, vals=None, idx=None) in (ENOTINIT, ENODEV)
    assert replicas_call(L, mode=3, step=7, vals=None, idx=None) == EINVAL  # a sync step needs them


def test_validate_payload_host(L):
    import torch

    import decoupled_momentum_optimizer_gb300 as dm

    good = torch.tensor([[0, 3, 7, 31], [1, 2, 3, 4], [5, 9, 10, 11]], dtype=torch.uint8).reshape(-1)
    assert dm.validate_payload(good, 96, 4) == (True, -1)
    bad = good.clone()
    bad[4 * 2 + 2] = 9  # duplicate in chunk 2
    assert dm.validate_payload(bad, 96, 4) == (False, 2)
    bad = good.clone()
    bad[3] = 32  # out of range in chunk 0
    assert dm.validate_payload(bad, 96, 4) == (False, 0)
    assert L.demo_validate_payload(96, 32, 4, 0, None, None) == EINVAL


def test_wire_argument_checks(L):
    # ternary needs the sign flag
    a = dict(g=p(0x10000), gd=0, m=p(0x20000), n=64, chunk=32, k=4, beta=0.9, mode=0, sign=0, period=8, seed=0,
             step=0, vals=p(0x30000), idx=p(0x40000), stream=None)
    assert L.demo_encode_wire(a["g"], 0, a["m"], 64, 32, 4, 0.9, 0, 0, 8, 0, 0, 1, a["vals"], a["idx"], None) == EINVAL
    assert L.demo_encode_wire(a["g"], 0, a["m"], 64, 32, 4, 0.9, 0, 1, 8, 0, 0, 7, a["vals"], a["idx"], None) == EINVAL
    assert L.demo_encode_wire(a["g"], 0, a["m"], 64, 32, 4, 0.9, 0, 1, 8, 0, 0, 1, a["vals"], a["idx"],
                              None) in (ENOTINIT, ENODEV)


def test_init_without_device(L):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert L.demo_init(0) == ENODEV
    code = ctypes.c_uint(0)
    assert L.demo_device_fault(ctypes.byref(code)) == ENOTINIT


def test_adamw_argument_checks(L):
    g = (ctypes.c_void_p * 1)(0x100000)
    m = (ctypes.c_void_p * 1)(0x200000)
    v = (ctypes.c_void_p * 1)(0x300000)
    th = p(0x400000)
    assert L.demo_adamw_step(th, 64, 0.9, 0.999, 1e-8, 1e-3, 0.0, 1, g, 0, m, v, 0, None) in (ENOTINIT, ENODEV)
    assert L.demo_adamw_step(th, 48, 0.9, 0.999, 1e-8, 1e-3, 0.0, 1, g, 0, m, v, 0, None) == EINVAL
    assert L.demo_adamw_step(th, 64, 1.0, 0.999, 1e-8, 1e-3, 0.0, 1, g, 0, m, v, 0, None) == EINVAL
    assert L.demo_adamw_step(th, 64, 0.9, 0.999, 0.0, 1e-3, 0.0, 1, g, 0, m, v, 0, None) == EINVAL
    assert L.demo_adamw_step(th, 64, 0.9, 0.999, 1e-8, 1e-3, 0.0, 0, g, 0, m, v, 0, None) == EINVAL
    assert L.demo_adamw_step(p(0x400004), 64, 0.9, 0.999, 1e-8, 1e-3, 0.0, 1, g, 0, m, v, 0, None) == EALIGN
    same = (ctypes.c_void_p * 1)(0x200000)
    assert L.demo_adamw_step(th, 64, 0.9, 0.999, 1e-8, 1e-3, 0.0, 1, g, 0, m, same, 0, None) == EINVAL


def test_binding_refuses_cpu_tensors():
    """The Python entry points fail loudly on CPU tensors: there is no CPU path."""
    import torch

    import decoupled_momentum_optimizer_gb300 as dm

    n = 64
    th, m, g, v = (torch.zeros(n) for _ in range(4))
    calls = [
        lambda: dm.step(th, [g], [m], k=4, beta=0.9, lr=0.1),
        lambda: dm.encode(g, m, torch.zeros(8), torch.zeros(8, dtype=torch.uint8), k=4, beta=0.9),
        lambda: dm.decode_update(th, [torch.zeros(8)], [torch.zeros(8, dtype=torch.uint8)], k=4, lr=0.1),
        lambda: dm.adamw_step(th, [g], [m], [v], lr=1e-3),
        lambda: dm.step_pipelined_static(th, [g], [m], k=4, beta=0.9, lr=0.1),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="no CPU path"):
            call()


def test_missing_library_fails_loudly(monkeypatch):
    """Without the built library every entry point raises: there is no fallback."""
    import torch

    import decoupled_momentum_optimizer_gb300 as dm

    monkeypatch.setattr(dm, "_lib", None)
    monkeypatch.setattr(dm, "LIB_PATH", os.path.join(ROOT, "_build", "no_such_library.so"))
    with pytest.raises(RuntimeError, match="missing"):
        dm.lib()
    with pytest.raises(RuntimeError, match="missing"):
        dm.payload_bytes("demo", 64, 4)
    with pytest.raises(RuntimeError, match="missing"):
        dm.validate_payload(torch.zeros(8, dtype=torch.uint8), 64, 4)
