"""The replication group's exchange when each replica of a shard runs on its own GPU.

FlexDeMo synchronises the extracted components q_t within the replication group R
("DeToNATION: Decoupled Torch Network-Aware Training on Interlinked Online Nodes",
Paper-Notes AAAI 2026, method section, "1. FlexDeMo" Algorithm 1, the
synchronisation of q_t in the replication group).  On one GPU the library keeps the R
replicas resident and combines their payloads directly; here every rank of a
``torch.distributed`` process group holds ONE replica of the same shard, encodes it
with the library, sends its wire-format payload to the others and decodes what it
receives with the library:

* DeMo sends values AND their indices, which differ between replicas, so the payloads
  are all-gathered: every rank receives the R payloads and decodes them in rank order,
  exactly as the single-GPU step combines its resident replicas r = 0..R-1 (the same
  bits for any R).  The DeToNATION notes list DeMo's all_gather, whose received bytes
  grow with the number of replicas, among the scheme's limitations, and their 64-node
  experiment finds it does not scale there.
* Random, Striding and DiLoCo send values at positions every replica knows (a shared
  seed, the step, or all positions), so a sum all-reduce of the float32 values is
  enough: every rank receives one summed payload and decodes it as a single payload
  with lr / R.  For R a power of two that is the mean to the last bit, and with R = 2
  the sum itself is exact in either order, so the result equals the single-GPU step's.
  Otherwise it differs by the collective's summation order and one rounding of lr / R.
  Formats whose values do not add (ternary bit-planes, 16-bit values) are all-gathered.

Every collective is a plain call of the process group (NCCL between GPUs, gloo on the
CPU in tests); no peer pointer reaches a kernel.  The payload of one replica lives in one
contiguous byte buffer (values, then indices at a 256-byte offset), so one collective
moves it.
"""

import torch
import torch.distributed as dist

from . import CHUNK, MODES, WIRES, payload_bytes

ALIGN = 256


def _round(b):
    return (b + ALIGN - 1) // ALIGN * ALIGN


class PayloadLayout:
    """One replica's payload for one step in one byte buffer: values at 0, indices at ``ioff``."""

    def __init__(self, mode, n, k, step, diloco_period, wire):
        self.mode, self.wire = mode, wire
        self.vb, self.ib = payload_bytes(mode, n, k, step=step, diloco_period=diloco_period, wire=wire)
        self.ioff = _round(self.vb)
        self.total = max(self.ioff + _round(self.ib), ALIGN)

    @property
    def sends(self):
        return self.vb > 0

    def views(self, buf):
        """(values, indices or None) views of a byte buffer laid out as this payload, typed as the
        library's wire format wants them."""
        w = WIRES[self.wire]
        vdt = {0: torch.float32, 1: torch.int32, 2: torch.bfloat16, 3: torch.float16}[w]
        vals = buf[:self.vb].view(vdt)
        idx = None
        if self.ib:
            idx = buf[self.ioff:self.ioff + self.ib]
            if w == 1:
                idx = idx.view(torch.int32)
        return vals, idx


class ReplicaExchange:
    """Exchange of the replicas' payloads over a process group (one replica per rank).

    ``collective`` is "all_gather", "all_reduce" or "auto" (all_gather for DeMo and for
    formats that do not add, all_reduce for Random, Striding and DiLoCo with float32
    values).
    """

    def __init__(self, n, k, mode="demo", *, wire="f32", diloco_period=8, group=None, collective="auto"):
        if mode not in MODES or wire not in WIRES:
            raise ValueError("unknown mode or wire format")
        if n <= 0 or n % CHUNK:
            raise ValueError("n must be a positive multiple of 32")
        self.n, self.k, self.mode, self.wire, self.period = n, k, mode, wire, diloco_period
        self.group = group
        self.R = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        adds = mode != "demo" and wire == "f32"
        if collective == "auto":
            collective = "all_reduce" if adds else "all_gather"
        if collective not in ("all_gather", "all_reduce"):
            raise ValueError("collective must be all_gather, all_reduce or auto")
        if collective == "all_reduce" and not adds:
            raise ValueError("all_reduce needs positions every replica knows and float32 values")
        self.collective = collective
        self._bufs = {}

    def layout(self, step):
        return PayloadLayout(self.mode, self.n, self.k, step, self.period, self.wire)

    def _buffer(self, key, nbytes, device):
        b = self._bufs.get(key)
        if b is None or b.numel() != nbytes or b.device != torch.device(device):
            b = torch.zeros(nbytes, dtype=torch.uint8, device=device)
            self._bufs[key] = b
        return b

    def send_buffer(self, step, device):
        """This rank's send buffer for ``step`` and its (values, indices) views; None when the
        step sends nothing (DiLoCo between syncs)."""
        L = self.layout(step)
        if not L.sends:
            return None, None, None
        buf = self._buffer("send", L.total, device)
        vals, idx = L.views(buf)
        return buf, vals, idx

    def exchange(self, send, step):
        """Run the collective on ``send`` (this rank's payload buffer).  Returns the list of
        (values, indices) payloads to decode, in rank order (all_gather: R entries; all_reduce:
        one entry holding the sum), or [] when the step sends nothing."""
        L = self.layout(step)
        if not L.sends:
            return []
        if self.collective == "all_reduce":
            vals, _ = L.views(send)
            dist.all_reduce(vals, op=dist.ReduceOp.SUM, group=self.group)
            return [(vals, None)]
        recv = self._buffer("recv", self.R * L.total, send.device)
        dist.all_gather_into_tensor(recv, send, group=self.group)
        return [L.views(recv[r * L.total:(r + 1) * L.total]) for r in range(self.R)]

    def decode_lr(self, lr):
        """The learning rate to decode the received payloads with (lr / R for a summed payload)."""
        return lr / self.R if self.collective == "all_reduce" else lr

    def bytes_per_step(self, step):
        """(bytes this rank contributes, bytes it receives into its decode buffer) for one step."""
        L = self.layout(step)
        if not L.sends:
            return 0, 0
        payload = L.vb + L.ib
        return payload, (payload if self.collective == "all_reduce" else self.R * payload)

    def step(self, theta, g, m, *, beta, lr, sign=True, seed=0, step=0, stream=None):
        """One FlexDeMo step of this rank's replica: encode (library), exchange (process group),
        decode and update theta (library).  theta and m update in place."""
        import contextlib

        from . import decode_update, encode

        # the process group's collectives order themselves after torch's current stream, so the
        # library's calls run on that stream too
        with torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext():
            buf, vals, idx = self.send_buffer(step, theta.device)
            encode(g, m, vals, idx, k=self.k, beta=beta, mode=self.mode, sign=sign, diloco_period=self.period,
                   seed=seed, step=step, wire=self.wire)
            got = self.exchange(buf, step) if buf is not None else []
            if not got:
                return
            decode_update(theta, [v for v, _ in got], [i for _, i in got] if self.mode == "demo" else None,
                          k=self.k, lr=self.decode_lr(lr), mode=self.mode, diloco_period=self.period, seed=seed,
                          step=step, wire=self.wire)
