"""GB300-native decoupled-momentum (DeMo / FlexDeMo) shard step.

A thin ctypes binding over the C ABI of ``libdemo_gb300.so`` (declared in
``include/demo.h``): it checks tensors, passes their device pointers and the
current CUDA stream, and raises :class:`DemoError` on a negative status.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU
path.  The library is loaded on first use and must have been built
(``python -m decoupled_momentum_optimizer_gb300.build``).
"""

import ctypes
import os

MODES = {"demo": 0, "random": 1, "stride": 2, "diloco": 3}
WIRES = {"f32": 0, "ternary": 1, "bf16": 2, "f16": 3}
GRAD_F32, GRAD_BF16 = 0, 1
CHUNK = 32
MAX_REPLICAS = 64

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdemo_gb300.so")

_c_i64, _c_u64, _c_vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
_SIGS = {
    "demo_init": (ctypes.c_int, [ctypes.c_int]),
    "demo_payload_bytes": (ctypes.c_size_t, [ctypes.c_int, _c_i64, ctypes.c_int, ctypes.c_int, _c_u64, ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_size_t)]),
    "demo_encode": (ctypes.c_int, [_c_vp, ctypes.c_int, _c_vp, _c_i64, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_u64, _c_u64, _c_vp, _c_vp, _c_vp]),
    "demo_decode_update": (ctypes.c_int, [_c_vp, _c_i64, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                          ctypes.c_int, _c_vp, _c_vp, ctypes.c_int, _c_u64, _c_u64, _c_vp]),
    "demo_step": (ctypes.c_int, [_c_vp, _c_i64, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_vp, ctypes.c_int, _c_vp, ctypes.c_int,
                                 _c_u64, _c_u64, _c_vp]),
    "demo_payload_bytes_wire": (ctypes.c_size_t, [ctypes.c_int, _c_i64, ctypes.c_int, ctypes.c_int, _c_u64,
                                                  ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "demo_encode_wire": (ctypes.c_int, [_c_vp, ctypes.c_int, _c_vp, _c_i64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_u64, _c_u64,
                                        ctypes.c_int, _c_vp, _c_vp, _c_vp]),
    "demo_encode_replicas": (ctypes.c_int, [_c_vp, ctypes.c_int, _c_vp, _c_i64, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            _c_u64, _c_u64, ctypes.c_int, _c_vp, _c_vp, _c_vp]),
    "demo_decode_update_wire": (ctypes.c_int, [_c_vp, _c_i64, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                               ctypes.c_int, ctypes.c_int, _c_vp, _c_vp, ctypes.c_int, _c_u64, _c_u64,
                                               ctypes.c_int, _c_vp]),
    "demo_step_wire": (ctypes.c_int, [_c_vp, _c_i64, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_vp, ctypes.c_int, _c_vp,
                                      ctypes.c_int, _c_u64, _c_u64, ctypes.c_int, _c_vp]),
    "demo_validate_payload": (ctypes.c_int, [_c_i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_vp,
                                             ctypes.POINTER(_c_i64)]),
    "demo_adamw_step": (ctypes.c_int, [_c_vp, _c_i64, ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                       ctypes.c_float, ctypes.c_int, _c_vp, ctypes.c_int, _c_vp, _c_vp, _c_u64,
                                       _c_vp]),
    "demo_step_pipelined": (ctypes.c_int, [_c_vp, _c_i64, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                           ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_vp,
                                           ctypes.c_int, _c_vp, ctypes.c_int, _c_u64, _c_u64, ctypes.c_int, _c_vp,
                                           _c_vp, _c_vp, _c_vp, ctypes.c_int, _c_vp, _c_vp]),
    "demo_step_pipelined_static": (ctypes.c_int, [_c_vp, _c_i64, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                                  ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_vp,
                                                  ctypes.c_int, _c_vp, ctypes.c_int, _c_u64, _c_u64, ctypes.c_int,
                                                  ctypes.c_int, _c_vp, _c_vp]),
    "demo_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "demo_device_fault": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint)]),
    "demo_test_stall_next_launch": (ctypes.c_int, [ctypes.c_longlong]),
}

_lib = None
_inited = set()


class DemoError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        name = lib().demo_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{what}: {name}" if what else name)


def lib():
    """The loaded C library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "python -m decoupled_momentum_optimizer_gb300.build")
        try:  # load the CUDA runtime the way torch does, so both share one runtime
            import torch  # noqa: F401
        except ImportError:  # pragma: no cover
            pass
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status, what):
    if status != 0:
        raise DemoError(status, what)


def init(device=None):
    """demo_init for ``device`` (default: torch's current device)."""
    import torch

    if device is None:
        device = torch.cuda.current_device()
    elif not isinstance(device, int):
        device = torch.device(device)
        device = device.index if device.index is not None else torch.cuda.current_device()
    if device not in _inited:
        _check(lib().demo_init(device), "demo_init")
        _inited.add(device)


def _stream(stream, device_index):
    """The cudaStream_t to launch on: the given stream, else torch's current stream of the device."""
    import torch

    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)  # torch's own launch path reads it this way
        return raw(device_index) if raw is not None else torch.cuda.current_stream(device_index).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t, dtypes, name, n=None, device_index=None, r=None):
    """The device pointer of a checked tensor (``name``, with replica ``r`` if given, names it in errors)."""
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{_name(name, r)} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{_name(name, r)} must be on a CUDA device (there is no CPU path)")
    if device_index is not None and t.get_device() != device_index:
        raise ValueError(f"{_name(name, r)} is on {t.device}, the call's other tensors on cuda:{device_index}")
    if t.dtype not in dtypes:
        raise TypeError(f"{_name(name, r)} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{_name(name, r)} must be contiguous")
    if n is not None and t.numel() != n:
        raise ValueError(f"{_name(name, r)} has {t.numel()} elements, expected {n}")
    return t.data_ptr()


def _name(name, r):
    return name if r is None else f"{name}[{r}]"


def _ptrs(ts, dtypes, name, n, device_index):
    """A host array of the R tensors' device pointers (each checked as by _ptr)."""
    return (ctypes.c_void_p * len(ts))(*[_ptr(t, dtypes, name, n, device_index, r) for r, t in enumerate(ts)])


class _OnDevice:
    """Makes the tensors' device current for a library call (the library launches on the
    current device) and initialises the library there; ``index`` is that device."""

    __slots__ = ("index", "_ctx")

    def __init__(self, device):
        if device.type != "cuda":
            raise ValueError(f"tensors are on {device}: the library runs on CUDA devices only (there is no CPU path)")
        self.index = device.index
        self._ctx = None

    def __enter__(self):
        import torch

        if self.index is None:
            self.index = torch.cuda.current_device()
        elif torch.cuda.current_device() != self.index:
            self._ctx = torch.cuda.device(self.index)
            self._ctx.__enter__()
        if self.index not in _inited:
            init(self.index)
        return self

    def __exit__(self, *exc):
        if self._ctx is not None:
            return self._ctx.__exit__(*exc)
        return False


def _grad_dtype(g):
    """The library's code for a gradient tensor's dtype (float32 or bfloat16; anything else is refused)."""
    import torch

    if g.dtype == torch.float32:
        return GRAD_F32
    if g.dtype == torch.bfloat16:
        return GRAD_BF16
    raise TypeError(f"gradients must be float32 or bfloat16, got {g.dtype}")


def _mode(mode):
    return MODES[mode] if isinstance(mode, str) else int(mode)


def _wire(wire):
    return WIRES[wire] if isinstance(wire, str) else int(wire)


def payload_bytes(mode, n, k, step=0, diloco_period=8, wire="f32"):
    """(value bytes, index bytes) one replica sends for a step in the given wire format."""
    ib = ctypes.c_size_t(0)
    vb = lib().demo_payload_bytes_wire(_mode(mode), n, CHUNK, k, step, diloco_period, _wire(wire), ctypes.byref(ib))
    return vb, ib.value


def payload_buffers(mode, n, k, step=0, diloco_period=8, wire="f32", device="cuda"):
    """Empty device buffers (vals, idx) sized for one replica's payload; None where nothing is sent."""
    import torch

    vb, ib = payload_bytes(mode, n, k, step=step, diloco_period=diloco_period, wire=wire)
    w = _wire(wire)
    vdt = {0: torch.float32, 1: torch.int32, 2: torch.bfloat16, 3: torch.float16}[w]
    vals = torch.empty(vb // torch.empty(0, dtype=vdt).element_size(), dtype=vdt, device=device) if vb else None
    idx = None
    if ib:
        idx = torch.empty(ib // 4, dtype=torch.int32, device=device) if w == 1 else \
            torch.empty(ib, dtype=torch.uint8, device=device)
    return vals, idx


def _val_dtypes(wire):
    import torch

    return {0: (torch.float32,), 1: (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,),
            2: (torch.bfloat16, torch.int16), 3: (torch.float16, torch.int16)}[wire]


def _idx_dtypes(wire):
    import torch

    return (torch.int32,) if wire == 1 else (torch.uint8,)


def encode(g, m, vals, idx=None, *, k, beta, mode="demo", sign=True, diloco_period=8, seed=0, step=0, wire="f32",
           stream=None):
    """One replica's encode (demo_encode_wire): updates m in place, writes vals (and idx for DeMo)."""
    import torch

    with _OnDevice(m.device) as d:
        n = m.numel()
        w = _wire(wire)
        gd = _grad_dtype(g)
        gp = _ptr(g, (g.dtype,), "g", n, d.index)
        mp = _ptr(m, (torch.float32,), "m", n, d.index)
        vp = _ptr(vals, _val_dtypes(w), "vals", None, d.index) if vals is not None else None
        ip = _ptr(idx, _idx_dtypes(w), "idx", None, d.index) if idx is not None else None
        _check(lib().demo_encode_wire(gp, gd, mp, n, CHUNK, k, beta, _mode(mode), int(bool(sign)), diloco_period,
                                      seed, step, w, vp, ip, _stream(stream, d.index)), "demo_encode")


def encode_replicas(gs, ms, vals, idx=None, *, k, beta, mode="demo", sign=True, diloco_period=8, seed=0, step=0,
                    wire="f32", stream=None):
    """Every replica's encode in one call (demo_encode_replicas): updates each m_r in place, writes
    vals[r] (and idx[r] for DeMo).  ``vals`` / ``idx`` are lists of R tensors, or None where the
    step sends nothing (DiLoCo between syncs) / carries no indices."""
    import torch

    with _OnDevice(ms[0].device) as d:
        n = ms[0].numel()
        R = len(ms)
        if len(gs) != R or (vals is not None and len(vals) != R) or (idx is not None and len(idx) != R):
            raise ValueError("need one gradient, payload and index buffer per replica")
        w = _wire(wire)
        gd = _grad_dtype(gs[0])
        garr = _ptrs(gs, (gs[0].dtype,), "g", n, d.index)
        marr = _ptrs(ms, (torch.float32,), "m", n, d.index)
        varr = _ptrs(vals, _val_dtypes(w), "vals", None, d.index) if vals is not None else None
        iarr = _ptrs(idx, _idx_dtypes(w), "idx", None, d.index) if idx is not None else None
        _check(lib().demo_encode_replicas(garr, gd, marr, n, CHUNK, k, beta, _mode(mode), int(bool(sign)), R,
                                          diloco_period, seed, step, w, varr, iarr, _stream(stream, d.index)),
               "demo_encode_replicas")


def decode_update(theta, vals, idx=None, *, k, lr, mode="demo", diloco_period=8, seed=0, step=0, wire="f32",
                  stream=None):
    """Scatter-mean of the R payloads in ``vals`` (and ``idx``) and theta -= lr Q (demo_decode_update_wire)."""
    import torch

    with _OnDevice(theta.device) as d:
        n = theta.numel()
        w = _wire(wire)
        tp = _ptr(theta, (torch.float32,), "theta", n, d.index)
        varr = _ptrs(vals, _val_dtypes(w), "vals", None, d.index)
        iarr = _ptrs(idx, _idx_dtypes(w), "idx", None, d.index) if idx is not None else None
        _check(lib().demo_decode_update_wire(tp, n, CHUNK, k, lr, _mode(mode), len(vals), varr, iarr, diloco_period,
                                             seed, step, w, _stream(stream, d.index)), "demo_decode_update")


def _replica_arrays(theta, gs, ms, index):
    """Checked pointers of theta and of the R gradients and momenta (one gradient dtype for all)."""
    import torch

    n = theta.numel()
    if len(gs) != len(ms):
        raise ValueError("need one gradient per replica")
    if not gs:
        raise ValueError("need at least one replica")
    gd = _grad_dtype(gs[0])
    tp = _ptr(theta, (torch.float32,), "theta", n, index)
    garr = _ptrs(gs, (gs[0].dtype,), "g", n, index)
    marr = _ptrs(ms, (torch.float32,), "m", n, index)
    return n, tp, gd, garr, marr


def step(theta, gs, ms, *, k, beta, lr, mode="demo", sign=True, diloco_period=8, seed=0, step=0, wire="f32",
         stream=None):
    """The fused shard step over R replicas (demo_step_wire); theta and every m_r update in place."""
    with _OnDevice(theta.device) as d:
        n, tp, gd, garr, marr = _replica_arrays(theta, gs, ms, d.index)
        _check(lib().demo_step_wire(tp, n, CHUNK, k, beta, lr, _mode(mode), int(bool(sign)), len(ms), garr, gd, marr,
                                    diloco_period, seed, step, _wire(wire), _stream(stream, d.index)), "demo_step")


def step_pipelined(theta, gs, ms, send, recv, *, k, beta, lr, mode="demo", sign=True, diloco_period=8, seed=0,
                   step=0, wire="f32", blocks=8, stream=None, comm_stream=None):
    """demo_step_pipelined: the split path with the payload exchange (send -> recv copies) overlapped.

    ``send`` and ``recv`` are lists of R (vals, idx) pairs as made by payload_buffers.
    """
    with _OnDevice(theta.device) as d:
        n, tp, gd, garr, marr = _replica_arrays(theta, gs, ms, d.index)
        w = _wire(wire)

        def arr(pairs, j, dts):
            if pairs is None or pairs[0][j] is None:
                return None
            return _ptrs([pq[j] for pq in pairs], dts, "payload", None, d.index)

        sv, si = arr(send, 0, _val_dtypes(w)), arr(send, 1, _idx_dtypes(w))
        rv, ri = arr(recv, 0, _val_dtypes(w)), arr(recv, 1, _idx_dtypes(w))
        cs = _stream(stream, d.index)
        xs = _stream(comm_stream, d.index) if comm_stream is not None else cs
        _check(lib().demo_step_pipelined(tp, n, CHUNK, k, beta, lr, _mode(mode), int(bool(sign)), len(ms), garr, gd,
                                         marr, diloco_period, seed, step, w, sv, si, rv, ri, blocks, cs, xs),
               "demo_step_pipelined")


def step_pipelined_static(theta, gs, ms, *, k, beta, lr, mode="demo", sign=True, diloco_period=8, seed=0, step=0,
                          wire="f32", blocks=8, stream=None, comm_stream=None):
    """demo_step_pipelined_static: the pipelined step with its payload buffers inside the library.

    For callers that cannot allocate device memory when they step; the payloads
    of all replicas must fit the library's fixed 32 MiB send / 32 MiB receive
    scratch (DemoError with DEMO_ENOSPACE otherwise).
    """
    with _OnDevice(theta.device) as d:
        n, tp, gd, garr, marr = _replica_arrays(theta, gs, ms, d.index)
        cs = _stream(stream, d.index)
        xs = _stream(comm_stream, d.index) if comm_stream is not None else cs
        _check(lib().demo_step_pipelined_static(tp, n, CHUNK, k, beta, lr, _mode(mode), int(bool(sign)), len(ms),
                                                garr, gd, marr, diloco_period, seed, step, _wire(wire), blocks, cs,
                                                xs), "demo_step_pipelined_static")


def adamw_step(theta, gs, ms, vs, *, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step=0, stream=None):
    """One Decoupled AdamW step (demo_adamw_step): theta, every m_r and v_r update in place."""
    import torch

    with _OnDevice(theta.device) as d:
        if len(vs) != len(ms):
            raise ValueError("need one gradient, first and second moment per replica")
        n, tp, gd, garr, marr = _replica_arrays(theta, gs, ms, d.index)
        varr = _ptrs(vs, (torch.float32,), "v", n, d.index)
        _check(lib().demo_adamw_step(tp, n, beta1, beta2, eps, lr, weight_decay, len(ms), garr, gd, marr, varr, step,
                                     _stream(stream, d.index)), "demo_adamw_step")


def validate_payload(idx_host, n, k, wire="f32"):
    """Host check of a DeMo index payload (a CPU tensor): returns (ok, first bad chunk or -1)."""
    bad = ctypes.c_int64(-1)
    status = lib().demo_validate_payload(n, CHUNK, k, _wire(wire), ctypes.c_void_p(idx_host.data_ptr()),
                                         ctypes.byref(bad))
    return status == 0, bad.value


def device_fault():
    """Read and clear the current device's fault word (0 = no kernel gave up on a wait)."""
    code = ctypes.c_uint(0)
    _check(lib().demo_device_fault(ctypes.byref(code)), "demo_device_fault")
    return code.value


def test_stall_next_launch(item=0):
    """demo_test_stall_next_launch: the next tile-kernel launch on the current device makes the
    load of its first warp's item ``item`` never complete, so that warp's bounded wait gives up
    and sets the fault word (read by device_fault).  For tests of the failure path."""
    _check(lib().demo_test_stall_next_launch(item), "demo_test_stall_next_launch")
