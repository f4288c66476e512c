"""The replica exchange over a process group (one replica per rank), two gloo ranks on the CPU.

Each rank encodes its own replica with the float64 oracle, writes the payload into the
exchange's send buffer in the wire format, and runs the exchange.  The gathered payloads
must be the ranks' own bytes in rank order, and decoding them must give the
single-process two-replica step; the summed (all-reduce) payload decoded with lr / 2
must give the same update.  Byte counts follow the wire format.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.demo_ref as ref

C = 32
N = 32 * (2 * 32 + 9)  # two full tiles and a ragged third
LR = 0.125
# mode, k, sign, wire, collective, step (DiLoCo period 8: step 7 syncs, step 3 does not)
CASES = [
    ("demo", 4, True, "f32", "auto", 0),
    ("demo", 2, False, "bf16", "auto", 1),
    ("demo", 4, True, "ternary", "auto", 2),
    ("random", 8, True, "f32", "auto", 3),
    ("random", 3, False, "f32", "all_gather", 4),
    ("stride", 4, False, "f16", "auto", 5),
    ("diloco", 1, False, "f32", "auto", 7),
    ("diloco", 1, True, "ternary", "auto", 7),
    ("diloco", 1, False, "f32", "auto", 3),
]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _state(r):
    rng = np.random.default_rng(50 + r)
    m = rng.standard_normal(N) * 1e-2
    g = rng.standard_normal(N).astype(np.float32).astype(np.float64) * 1e-2
    return m, g


def _encode(case, r):
    mode, k, sign, wire, _, step = case
    m, g = _state(r)
    return ref.encode(m, g, 0.9, k, ref.__dict__["MODE_" + mode.upper()], sign, seed=9, step=step, period=8)


def _wire_values(vals, wire):
    """The payload values as the sender puts them on the wire (float32, or the 16-bit rounding)."""
    if wire in ("f32", "ternary"):
        return vals.astype(np.float32)
    return ref.wire_round(vals, ref.WIRE_BF16 if wire == "bf16" else ref.WIRE_F16).astype(np.float32)


def _fill(send_vals, send_idx, enc, case):
    mode, k, sign, wire, _, _ = case
    vals = enc["vals"]
    if wire == "ternary":
        vw, iw = ref.ternary_pack(vals, enc["idx"] if mode == "demo" else None)
        send_vals.copy_(torch.from_numpy(vw.reshape(-1).view(np.int32)))
        if iw is not None:
            send_idx.copy_(torch.from_numpy(iw.reshape(-1).view(np.int32)))
        return
    v32 = torch.from_numpy(_wire_values(vals, wire).reshape(-1))
    send_vals.copy_(v32.to(send_vals.dtype))
    if mode == "demo":
        send_idx.copy_(torch.from_numpy(enc["idx"].astype(np.uint8).reshape(-1)))


def _raw(t):
    """The bytes of a tensor (any dtype) as a numpy uint8 array."""
    return t.contiguous().view(torch.uint8).clone().numpy()


def _worker(rank, world, port, out_q):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        from decoupled_momentum_optimizer_gb300.exchange import ReplicaExchange

        results = []
        for case in CASES:
            mode, k, sign, wire, coll, step = case
            ex = ReplicaExchange(N, k, mode, wire=wire, diloco_period=8, collective=coll)
            buf, sv, si = ex.send_buffer(step, "cpu")
            L = ex.layout(step)
            if buf is None:
                results.append((case, None, ex.collective, ex.bytes_per_step(step), ex.exchange(None, step), L.ioff))
                continue
            _fill(sv, si, _encode(case, rank), case)
            sent = _raw(buf)
            got = ex.exchange(buf, step)
            host = [(_raw(v), None if i is None else _raw(i)) for v, i in got]
            results.append((case, sent, ex.collective, ex.bytes_per_step(step), host, L.ioff))
        if rank == 0:
            out_q.put(results)
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:  # reported to the test instead of leaving it waiting
        out_q.put(repr(e))
        raise


@pytest.fixture(scope="module")
def exchanged():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=180)
    assert not isinstance(res, str), res
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


def _host_payload(vals, idx, case, nc):
    """(values [nc][kv] float64, indices [nc][k] or None) from the raw bytes of a wire-format payload."""
    mode, k, sign, wire, _, _ = case
    kv = C if mode == "diloco" else k
    if wire == "ternary":
        return ref.ternary_unpack(vals.view(np.uint32).reshape(-1, kv, 2),
                                  None if idx is None else idx.view(np.uint32).reshape(-1, k, 5), nc)
    if wire == "f32":
        v = vals.view(np.float32)
    elif wire == "bf16":
        v = (vals.view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    else:
        v = vals.view(np.float16)
    return v.astype(np.float64).reshape(nc, kv), (None if idx is None else idx.astype(np.int64).reshape(nc, k))


@pytest.mark.parametrize("ci", range(len(CASES)), ids=lambda i: "-".join(map(str, CASES[i])))
def test_exchange_equals_two_replica_step(exchanged, ci):
    case, sent0, coll, (tx, rx), host, ioff = exchanged[ci]
    mode, k, sign, wire, _, step = case
    nc = N // C
    vb, ib = ref.payload_bytes_wire(ref.__dict__["MODE_" + mode.upper()], N, k, step=step, period=8,
                                    wire=ref.__dict__["WIRE_" + wire.upper()])
    if vb == 0:  # DiLoCo between syncs: nothing is sent
        assert sent0 is None and host == [] and (tx, rx) == (0, 0)
        return
    want_coll = "all_reduce" if (mode != "demo" and wire == "f32" and case[4] == "auto") else "all_gather"
    assert coll == want_coll
    assert tx == vb + ib and rx == (tx if coll == "all_reduce" else 2 * tx)
    encs = [_encode(case, r) for r in range(2)]
    theta = np.random.default_rng(7).standard_normal(N)
    mode_id = ref.__dict__["MODE_" + mode.upper()]
    # what the two ranks sent, as the receiver decodes it
    sent_vals = [_wire_values(e["vals"], wire).astype(np.float64) for e in encs]
    pos = [e["idx"] if mode == "demo" else e["pos"] for e in encs]
    want, _, _, _ = ref.decode_update(theta, sent_vals, pos, LR, mode_id)
    if coll == "all_gather":
        assert len(host) == 2
        # the first received payload is rank 0's own bytes
        assert np.array_equal(host[0][0], sent0[:vb])
        if ib:
            assert np.array_equal(host[0][1], sent0[ioff:ioff + ib])
        got_vals, got_pos = [], []
        for r in range(2):
            v, i = _host_payload(host[r][0], host[r][1], case, nc)
            got_vals.append(v)
            got_pos.append(i if mode == "demo" else encs[r]["pos"])
            if mode == "demo":
                assert np.array_equal(i, encs[r]["idx"])
        got, _, _, _ = ref.decode_update(theta, got_vals, got_pos, LR, mode_id)
        assert np.array_equal(got, want)
    else:
        assert len(host) == 1 and host[0][1] is None
        vsum, _ = _host_payload(host[0][0], None, case, nc)
        assert np.array_equal(vsum, (sent_vals[0].astype(np.float32) + sent_vals[1].astype(np.float32))
                              .astype(np.float64))
        got, _, _, _ = ref.decode_update(theta, [vsum], [pos[0]], LR / 2, mode_id)
        # the float32 sum of two float32 values is their exact sum rounded once
        assert np.abs(got - want).max() <= 1e-6 * np.abs(want - theta).max()
