"""Seeded synthetic workloads for the decoupled-momentum shard step.

This module only describes and draws inputs: parameter-shard layouts shaped
like the models the DeToNATION experiments train (T5-base, ViT-B/16, OLMo2-1B),
and seeded Gaussian parameters / gradients.  It holds none of the optimizer's
arithmetic, so both the CUDA path and the float64 checker can be fed from it.

Layouts: every tensor is flattened and padded with zeros to a multiple of the
32-element chunk, then the tensors are laid end to end.  Padding entries have
theta = 0 and g = 0 in every step.

Draws: theta_0 ~ N(0, 2e-2) from a generator seeded 12345; replica r draws its
gradients from a generator seeded r, one full-shard draw per step in step
order; the second parameter of N(.,.) is the standard deviation.  A heavy-tail
option multiplies a Bernoulli(0.01) subset of each draw by 100 (the mask comes
from the same replica generator, right after the Gaussian draw).  bf16
gradients are the float32 draw rounded to bfloat16.
"""

from dataclasses import dataclass, field

import torch

CHUNK = 32


# ----------------------------------------------------------------------------
# Parameter-shard layouts
# ----------------------------------------------------------------------------

@dataclass
class ShardLayout:
    name: str
    tensors: list  # [(tensor name, numel)]
    offsets: list = field(default_factory=list)  # start of each tensor in the flat shard
    padded: list = field(default_factory=list)  # padded numel of each tensor

    def __post_init__(self):
        off = 0
        self.offsets, self.padded = [], []
        for _, numel in self.tensors:
            p = (numel + CHUNK - 1) // CHUNK * CHUNK
            self.offsets.append(off)
            self.padded.append(p)
            off += p
        self.n = off

    @property
    def n_raw(self):
        return sum(numel for _, numel in self.tensors)

    def pad_ranges(self):
        """[(start, stop)] of the zero padding inside the flat shard."""
        out = []
        for (_, numel), off, p in zip(self.tensors, self.offsets, self.padded):
            if p > numel:
                out.append((off + numel, off + p))
        return out

    def pad_chunks(self):
        return sorted({s // CHUNK for s, _ in self.pad_ranges()})


def flat_layout(n):
    if n % CHUNK:
        raise ValueError("a flat shard must hold whole chunks")
    return ShardLayout(f"flat{n}", [("flat", n)])


def t5_base_layout():
    """T5-base: d_model 768, d_ff 3072, 12 encoder + 12 decoder layers, vocab 32128."""
    d, ff, V, H = 768, 3072, 32128, 12
    t = [("shared.embedding", V * d)]
    for side, nl in (("encoder", 12), ("decoder", 12)):
        for i in range(nl):
            p = f"{side}.{i}"
            t += [(f"{p}.self.{w}", d * d) for w in "qkvo"]
            if i == 0:
                t.append((f"{p}.self.relative_bias", 32 * H))
            t.append((f"{p}.ln_self", d))
            if side == "decoder":
                t += [(f"{p}.cross.{w}", d * d) for w in "qkvo"]
                t.append((f"{p}.ln_cross", d))
            t += [(f"{p}.ff.wi", d * ff), (f"{p}.ff.wo", ff * d), (f"{p}.ln_ff", d)]
        t.append((f"{side}.final_ln", d))
    return ShardLayout("t5_base", t)


def vit_b16_layout():
    """ViT-B/16 at 224x224: 12 layers, width 768, MLP 3072, 1000 classes."""
    d, ff, L, ncls, ntok = 768, 3072, 12, 1000, 197
    t = [("patch_embed.w", d * 3 * 16 * 16), ("patch_embed.b", d), ("cls_token", d), ("pos_embed", ntok * d)]
    for i in range(L):
        p = f"block{i}"
        t += [
            (f"{p}.ln1.w", d), (f"{p}.ln1.b", d),
            (f"{p}.qkv.w", d * 3 * d), (f"{p}.qkv.b", 3 * d),
            (f"{p}.proj.w", d * d), (f"{p}.proj.b", d),
            (f"{p}.ln2.w", d), (f"{p}.ln2.b", d),
            (f"{p}.fc1.w", d * ff), (f"{p}.fc1.b", ff),
            (f"{p}.fc2.w", ff * d), (f"{p}.fc2.b", d),
        ]
    t += [("norm.w", d), ("norm.b", d), ("head.w", d * ncls), ("head.b", ncls)]
    return ShardLayout("vit_b16", t)


def olmo2_1b_layout(tied=True):
    """OLMo2-1B-shaped: d 2048, 16 layers, SwiGLU d_ff 8192, vocab 100352, q/k norms."""
    d, ff, L, V = 2048, 8192, 16, 100352
    t = [("embed", V * d)]
    for i in range(L):
        p = f"layer{i}"
        t += [(f"{p}.attn.{w}", d * d) for w in "qkvo"]
        t += [(f"{p}.q_norm", d), (f"{p}.k_norm", d)]
        t += [(f"{p}.mlp.gate", d * ff), (f"{p}.mlp.up", d * ff), (f"{p}.mlp.down", ff * d)]
        t += [(f"{p}.post_attn_norm", d), (f"{p}.post_ff_norm", d)]
    t.append(("final_norm", d))
    if not tied:
        t.append(("lm_head", V * d))
    return ShardLayout("olmo2_1b", t)


def half_shard(layout, which=0):
    """One of two intra-node shards: the flat buffer split at its midpoint (rounded to a chunk)."""
    mid = (layout.n // 2) // CHUNK * CHUNK
    lo, hi = (0, mid) if which == 0 else (mid, layout.n)
    return lo, hi


# ----------------------------------------------------------------------------
# Named workloads (shapes, distributions and step settings)
# ----------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    n: int
    layout: object
    shard: tuple  # (lo, hi) slice of the layout's flat buffer
    R: int
    runs: list  # [(mode name, k, sign)]
    steps: int
    g_std: float
    g_dtype: str = "f32"
    heavy_tail: bool = False
    beta: float = 0.999
    lr: float = 1e-3
    theta_std: float = 2e-2

    def pad_mask(self, device="cpu"):
        """Bool tensor [n]: True on the shard's padding entries."""
        mask = torch.zeros(self.n, dtype=torch.bool, device=device)
        lo, hi = self.shard
        for s, e in self.layout.pad_ranges():
            s2, e2 = max(s, lo), min(e, hi)
            if s2 < e2:
                mask[s2 - lo:e2 - lo] = True
        return mask


def workload(name):
    if name == "flat64k":
        lay = flat_layout(65536)
        return Workload(name, lay.n, lay, (0, lay.n), R=2, runs=[("demo", 4, True)], steps=5, g_std=1e-2)
    if name == "t5_base":
        lay = t5_base_layout()
        return Workload(name, lay.n, lay, (0, lay.n), R=2, runs=[("demo", 4, True), ("random", 8, True)],
                        steps=20, g_std=1e-3)
    if name == "vit_b16":
        lay = vit_b16_layout()
        return Workload(name, lay.n, lay, (0, lay.n), R=2,
                        runs=[("demo", 1, True), ("demo", 1, False), ("random", 1, True), ("random", 1, False)],
                        steps=10, g_std=1e-3, heavy_tail=True)
    if name == "olmo2_1b_half":
        lay = olmo2_1b_layout(tied=True)
        lo, hi = half_shard(lay, 0)
        return Workload(name, hi - lo, lay, (lo, hi), R=2,
                        runs=[("demo", 1, True), ("demo", 2, True), ("random", 8, True)],
                        steps=10, g_std=1e-3, g_dtype="bf16")
    if name.startswith("flat"):
        n = int(name[4:])
        lay = flat_layout(n)
        return Workload(name, n, lay, (0, n), R=2, runs=[("demo", 4, True)], steps=3, g_std=1e-3)
    raise KeyError(name)


# ----------------------------------------------------------------------------
# Seeded draws
# ----------------------------------------------------------------------------

def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_theta0(wl, device="cpu", seed=12345):
    gen = _gen(seed, device)
    th = torch.randn(wl.n, generator=gen, device=device, dtype=torch.float32) * wl.theta_std
    th[wl.pad_mask(device)] = 0.0
    return th


class GradStream:
    """Replica r's gradients, one full-shard draw per step from a generator seeded r."""

    def __init__(self, wl, r, device="cpu"):
        self.wl = wl
        self.device = device
        self.gen = _gen(r, device)
        self.pad = wl.pad_mask(device)

    def next(self):
        wl = self.wl
        g = torch.randn(wl.n, generator=self.gen, device=self.device, dtype=torch.float32) * wl.g_std
        if wl.heavy_tail:
            big = torch.rand(wl.n, generator=self.gen, device=self.device) < 0.01
            g = torch.where(big, g * 100.0, g)
        g[self.pad] = 0.0
        if wl.g_dtype == "bf16":
            g = g.to(torch.bfloat16)
        return g
