"""The seeded input recipe: shapes, counts and value laws of the workloads.

The shapes of c2 and c3's skinny part are the pages' fused example
(«MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能跃升», 矩阵融合优化,
Fig. 6-7: [24, 10240] x 74 and [32, 24, 10240]).  The rest are this library's
benchmark configurations; their draws must be reproducible and follow the
stated laws, since the GPU path and the oracle both take their inputs here.
"""
import math

import numpy as np
import pytest
import torch

from newton_schulz_bucket_gb300 import workloads as W


def test_c5_counts_are_the_stated_draw():
    counts = W.c5_counts(5)
    assert counts == [387, 211, 180, 92, 83, 10, 9, 7, 9, 4, 2, 6]
    assert sum(counts) == 1000 and min(counts) >= 1
    # smaller matrices are drawn more often (weights 1 / (rows * cols))
    assert counts[0] > counts[1] > counts[2] > counts[3] > counts[4]


def test_config_shapes():
    assert W.get("c1_fp32_64x128").shapes == [[64, 128]]
    assert W.get("c2_skinny_74x24x10240").shapes == [[24, 10240]] * 74
    assert W.get("c3_moe_64x2048x7168_32x24x10240").shapes == [[64, 2048, 7168], [32, 24, 10240]]
    c4 = W.get("c4_dense_h4096")
    assert len(c4.shapes) == 128 and c4.shapes[:4] == [[4096, 12288], [4096, 4096],
                                                         [4096, 16384], [16384, 4096]]
    c5 = W.get("c5_mixed_1000")
    assert len(c5.shapes) == 1000
    assert [c5.shapes.count(s) for s in W.C5_SHAPES] == W.c5_counts(5)
    g = W.get("c5_group_64x7168")
    assert g.shapes == [[64, 7168]] * 211
    with pytest.raises(KeyError):
        W.get("c5_group_3x3")
    assert W.get("c2_skinny_74x24x10240", ns_steps=10).ns_steps == 10


def test_c3_expert_scales_are_log_uniform_in_range():
    s = W.get("c3_moe_64x2048x7168_32x24x10240").g_std[0]
    assert len(s) == 64
    assert all(1e-4 <= v <= 1e-2 for v in s)
    logs = np.log10(s)
    assert logs.min() < -3.5 and logs.max() > -2.5  # spread over the two decades


def test_draws_are_seeded_and_follow_the_laws():
    w = W.custom([[64, 4096], [2, 32, 1024]], seed=7, g_std=1e-3, p_std=0.02)
    P, G, M = W.make_tensors(w)
    P2, G2, M2 = W.make_tensors(w)
    for a, b in zip(P + G + M, P2 + G2 + M2):
        assert torch.equal(a, b)
    assert P[0].dtype == torch.bfloat16 and G[0].dtype == torch.bfloat16
    assert M[0].dtype == torch.float32
    n = P[0].numel()
    for t, std in [(P[0], 0.02), (G[0], 1e-3), (M[0], 1e-3)]:
        x = t.double()
        assert abs(float(x.mean())) < 5 * std / math.sqrt(n)
        assert abs(float(x.std()) / std - 1) < 0.02
    other = W.make_tensors(W.custom([[64, 4096], [2, 32, 1024]], seed=8))[1][0]
    assert not torch.equal(other, G[0])


def test_bf16_inputs_are_round_to_nearest_even_casts():
    """P and G are fp32 draws cast to bf16 by round-to-nearest-even: replaying
    the generator gives the fp32 values, whose RNE rounding must match."""
    w = W.custom([[24, 1000]], seed=11)
    P, G, _ = W.make_tensors(w)
    g = torch.Generator().manual_seed(11)
    p32 = torch.randn([24, 1000], generator=g) * 0.02
    g32 = torch.randn([24, 1000], generator=g) * 1e-3
    for got, src in [(P[0], p32), (G[0], g32)]:
        u = src.numpy().view(np.uint32).astype(np.uint64)
        rne = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32).view(np.float32)
        np.testing.assert_array_equal(got.float().numpy(), rne)


def test_per_expert_stds_scale_each_slice():
    w = W.custom([[4, 64, 2048]], seed=3)
    w.g_std = [[1e-4, 1e-3, 1e-2, 1e-1]]
    _, G, M = W.make_tensors(w)
    for e, std in enumerate(w.g_std[0]):
        for t in (G[0][e], M[0][e]):
            assert abs(float(t.double().std()) / std - 1) < 0.03


def test_zero_momentum_option():
    _, _, M = W.make_tensors(W.custom([[8, 64]], m_zero=True))
    assert not M[0].any()


def test_spread_spectrum_draws():
    """spectrum_decades: M0 and G are one draw U diag(s) V^T per member, s
    log-spaced over the stated decades, entries of the stated rms; G is that
    draw rounded to bf16 and P follows its usual law."""
    w = W.custom([[24, 512], [300, 40], [2, 16, 64]], seed=5, spectrum_decades=3)
    P, G, M = W.make_tensors(w)
    for i, shp in enumerate(w.shapes):
        ms = M[i].reshape(-1, *shp[-2:])
        gs = G[i].reshape(-1, *shp[-2:])
        assert ms.dtype == torch.float32 and gs.dtype == torch.bfloat16
        for m, g in zip(ms, gs):
            s = torch.linalg.svdvals(m.double())
            want = torch.logspace(0, -3, s.numel(), dtype=torch.float64)
            assert torch.allclose(s / s[0], want, rtol=1e-3)
            assert abs(float(m.double().pow(2).mean().sqrt()) / 1e-3 - 1) < 1e-5
            assert torch.equal(g, m.to(torch.bfloat16))
        assert abs(float(P[i].double().std()) / 0.02 - 1) < 0.2
    again = W.make_tensors(w)
    assert all(torch.equal(a, b) for a, b in zip(M + G + P, again[2] + again[1] + again[0]))
    _, _, Mz = W.make_tensors(W.custom([[8, 64]], spectrum_decades=2, m_zero=True))
    assert not Mz[0].any()


def test_reduced_batch_group_workloads():
    """'group_<rows>x<cols>_b<B>': B matrices of one shape with the dense
    model's value law, for profiling one group at a reduced batch."""
    w = W.get("group_16384x4096_b2")
    assert w.shapes == [[16384, 4096]] * 2 and w.mode == "bf16" and w.ns_steps == 5
    assert w.g_std == [1e-3, 1e-3] and w.p_std == [0.02, 0.02]
    for bad in ("group_16384x4096", "group_0x4_b2", "group_4x4_b0", "group_axb_b1"):
        with pytest.raises(KeyError):
            W.get(bad)
