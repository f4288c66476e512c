"""The synthetic workloads against the models whose shapes they stand in for (CPU).

The pages train T5-base, ViT-B/16 and OLMo2-1B; the workloads lay those models'
parameter tensors end to end, each padded to a multiple of 32.  Here the totals
are recomputed per component from the architectures' dimensions (not by walking
the module's tensor lists), and the padding, the half-shard split and the seeded
draws are checked.
"""

import torch

from decoupled_momentum_optimizer_gb300 import workloads as W

C = 32


def test_t5_base_parameter_count():
    d, ff, V, layers, heads = 768, 3072, 32128, 12, 12
    embed = V * d
    enc_layer = 4 * d * d + 2 * d * ff + 2 * d  # self-attention, feed-forward, two layer norms
    dec_layer = 8 * d * d + 2 * d * ff + 3 * d  # self- and cross-attention, feed-forward, three norms
    rel_bias = 2 * 32 * heads  # one relative-position bias per stack (first layer)
    final = 2 * d
    total = embed + layers * (enc_layer + dec_layer) + rel_bias + final
    assert total == 222_903_552
    lay = W.t5_base_layout()
    assert lay.n_raw == total and lay.n == total  # every tensor is already a multiple of 32
    assert len(lay.tensors) == 1 + 12 * 8 + 1 + 12 * 13 + 1 + 2 == 257
    wl = W.workload("t5_base")
    assert wl.n == total and wl.R == 2 and ("demo", 4, True) in wl.runs and ("random", 8, True) in wl.runs


def test_vit_b16_parameter_count_and_padding():
    d, ff, layers, ncls, tokens = 768, 3072, 12, 1000, 14 * 14 + 1
    stem = 16 * 16 * 3 * d + d + d + tokens * d  # patch projection and bias, class token, positions
    layer = 2 * (2 * d) + (3 * d * d + 3 * d) + (d * d + d) + (d * ff + ff) + (ff * d + d)
    head = 2 * d + d * ncls + ncls
    total = stem + layers * layer + head
    assert total == 86_567_656  # the published ViT-B/16 count
    lay = W.vit_b16_layout()
    assert lay.n_raw == total and len(lay.tensors) == 4 + 12 * 12 + 4 == 152
    assert lay.n == 86_567_680  # only the 1,000-entry head bias needs padding (24 entries)
    assert lay.pad_ranges() == [(lay.n - 24, lay.n)]
    wl = W.workload("vit_b16")
    assert wl.heavy_tail and wl.pad_mask().sum().item() == 24


def test_olmo2_half_shard():
    d, ff, layers, V = 2048, 8192, 16, 100352
    layer = 4 * d * d + 2 * d + 3 * d * ff + 2 * d  # attention, q/k norms, SwiGLU, two norms
    tied = V * d + layers * layer + d
    assert tied == 1_279_395_840
    assert W.olmo2_1b_layout(tied=True).n == tied
    assert W.olmo2_1b_layout(tied=False).n == tied + V * d
    wl = W.workload("olmo2_1b_half")
    assert wl.n == tied // 2 == 639_697_920 and wl.shard == (0, tied // 2) and wl.n % C == 0
    assert wl.g_dtype == "bf16"


def test_flat_workloads():
    assert W.workload("flat64k").n == 65536
    assert W.workload(f"flat{1 << 26}").n == 1 << 26
    assert W.workload(f"flat{1 << 26}").pad_mask().sum().item() == 0


def test_seeded_draws_are_reproducible_and_padding_stays_zero():
    lay = W.ShardLayout("tiny", [("a", 40), ("b", 64), ("c", 7)])
    assert lay.n == 64 + 64 + 32 and lay.pad_ranges() == [(40, 64), (135, 160)]
    wl = W.Workload("tiny", lay.n, lay, (0, lay.n), R=2, runs=[("demo", 4, True)], steps=1, g_std=1e-3,
                    heavy_tail=True)
    th = W.make_theta0(wl)
    assert torch.equal(th, W.make_theta0(wl))
    mask = wl.pad_mask()
    assert (th[mask] == 0).all() and (th[~mask] != 0).all()
    g0, g0b, g1 = W.GradStream(wl, 0).next(), W.GradStream(wl, 0).next(), W.GradStream(wl, 1).next()
    assert torch.equal(g0, g0b) and not torch.equal(g0, g1)  # one generator per replica, seeded r
    assert (g0[mask] == 0).all()
    s = W.GradStream(wl, 0)
    assert not torch.equal(s.next(), s.next())  # a new draw every step
    wl16 = W.Workload("tiny16", lay.n, lay, (0, lay.n), R=1, runs=[], steps=1, g_std=1e-3, g_dtype="bf16")
    assert W.GradStream(wl16, 0).next().dtype == torch.bfloat16
