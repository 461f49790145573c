"""The seeded input recipe: shapes, sizes and spectra of the synthetic workloads.

The generators draw every matrix from its own seed, so the checks here run on
the CPU generator with the same code the GPU tests and the benchmark use on the
device: the stated shapes and nominal FLOPs of each workload, the singular
values each spectrum kind promises (which fail if the orthonormal factors are
not orthonormal), the weight and momentum distributions, and that a subset of
a workload regenerates the same matrices as the whole.
"""
import pytest
import torch

from muon_newton_schulz_step_gb300 import workloads as wl


def _one(spec, seed_id=9, **kw):
    return wl.Workload("probe", seed_id, "step", [spec], g_dtype=torch.float32, w_dtype=torch.float32,
                       on_host=True, **kw)


def test_workload_shapes_counts_and_nominal_flops():
    expect = {  # name: (count, call, distinct shapes, nominal NS5 FLOPs)
        "tiny": (8, "step", {(64, 256)}, 1.887e8),
        "expert_gate": (96, "ns", {(2048, 6144)}, 5.773e13),
        "dense_attn": (6, "step", {(6144, 6144), (1024, 6144)}, 2.810e13),
        "moe_layer": (288, "step", {(2048, 6144), (6144, 2048)}, 1.732e14),
        "mixed_block": (295, "step", {(2048, 6144), (6144, 2048), (6144, 6144), (1024, 6144)}, 1.892e14),
    }
    assert set(wl.WORKLOADS) == set(expect)
    for name, (count, call, shapes, flops) in expect.items():
        w = wl.workload(name)
        assert w.count == count and w.call == call and set(w.shapes()) == shapes, name
        total = sum(wl.nominal_ns_flops(*s) for s in w.shapes())
        assert abs(total - flops) < 1e-3 * flops, (name, total)
    moe = wl.workload("moe_layer").shapes()
    assert moe.count((6144, 2048)) == 96 and moe.count((2048, 6144)) == 192
    with pytest.raises(KeyError):
        wl.workload("no_such_workload")


def test_nominal_flops_counts_the_three_products():
    # Gram 2 r^2 k + polynomial 2 r^3 + update 2 r^2 k per iteration, r = min side
    assert wl.nominal_ns_flops(3, 5, steps=1) == 2 * 9 * 5 + 2 * 27 + 2 * 9 * 5
    assert wl.nominal_ns_flops(5, 3, steps=2) == wl.nominal_ns_flops(3, 5, steps=2)


def test_mixed_block_order_is_a_fixed_shuffle():
    a, b = wl.workload("mixed_block"), wl.workload("mixed_block")
    assert [m.role for m in a.mats] == [m.role for m in b.mats]
    roles = [m.role for m in a.mats]
    assert roles[:3] != ["gate", "up", "down"]        # shuffled, not in construction order
    assert sorted(set(roles)) == ["down", "gate", "k", "o", "q", "shared", "up", "v"]


@pytest.mark.parametrize("shape", [(128, 512), (512, 128)])
def test_const_spectrum_gives_equal_singular_values(shape):
    g = wl.gradient(_one(wl.MatrixSpec(*shape, "const", 32, 0.1, 0.1, 0.0)), 0, "cpu")
    s = torch.linalg.svdvals(g.double())
    assert torch.allclose(s[:32], torch.full((32,), 0.1, dtype=torch.float64), rtol=0, atol=2e-6)
    assert float(s[32]) < 1e-6


def test_uniform_and_loguniform_spectra_stay_in_their_ranges():
    g = wl.gradient(_one(wl.MatrixSpec(64, 256, "uniform", 4, 0.1, 10.0, 0.0)), 0, "cpu")
    s = torch.linalg.svdvals(g.double())
    assert 0.1 - 1e-5 <= float(s[3]) and float(s[0]) <= 10.0 + 1e-5 and float(s[4]) < 1e-5
    g = wl.gradient(_one(wl.MatrixSpec(256, 768, "loguniform", 16, 1e-2, 1.0, 0.0)), 0, "cpu")
    s = torch.linalg.svdvals(g.double())
    assert 1e-2 - 1e-6 <= float(s[15]) and float(s[0]) <= 1.0 + 1e-6 and float(s[16]) < 1e-6
    # full rank (rank None): every singular value in the range
    g = wl.gradient(_one(wl.MatrixSpec(64, 192, "loguniform", None, 1e-3, 1.0, 0.0)), 0, "cpu")
    s = torch.linalg.svdvals(g.double())
    assert 1e-3 - 1e-6 <= float(s[-1]) and float(s[0]) <= 1.0 + 1e-6


def test_noise_only_gradient_has_the_stated_std():
    g = wl.gradient(_one(wl.MatrixSpec(256, 1024, "none", 0, 0.0, 0.0, 1e-3)), 0, "cpu")
    assert abs(float(g.std()) / 1e-3 - 1.0) < 0.01 and abs(float(g.mean())) < 1e-5


def test_tiny_gradients_are_rank_four_plus_noise():
    w = wl.workload("tiny")
    for i in range(w.count):
        s = torch.linalg.svdvals(wl.gradient(w, i, "cpu").double())
        # the noise (std 1e-3 on 64 x 256) has spectral norm about 1e-3 * (8 + 16)
        assert float(s[3]) > 0.1 - 0.03 and float(s[0]) < 10.0 + 0.03 and float(s[4]) < 0.03


def test_weights_and_momentum_distributions():
    w = wl.workload("moe_layer")
    W = wl.weights(w, 2, "cpu")
    M = wl.momentum(w, 2, "cpu")
    assert W.dtype == torch.bfloat16 and W.shape == (6144, 2048)
    assert M.dtype == torch.float32 and M.shape == (6144, 2048)
    assert abs(float(W.float().std()) / 0.02 - 1.0) < 0.01
    assert abs(float(M.std()) / 1e-3 - 1.0) < 0.01
    t = wl.workload("tiny")
    assert torch.count_nonzero(wl.momentum(t, 0, "cpu")) == 0
    assert wl.weights(t, 0, "cpu").dtype == torch.float32


def test_streams_are_independent_and_subsets_regenerate():
    w = wl.workload("tiny")
    full = wl.make_inputs(w, "cpu")
    sub = wl.make_inputs(w, "cpu", indices=[5, 2])
    for key in ("W", "G", "M"):
        assert torch.equal(sub[key][0], full[key][5]) and torch.equal(sub[key][1], full[key][2])
    assert not torch.equal(full["G"][0], full["G"][1])
    # weights, gradient and momentum of one matrix come from different seeds
    base = wl.SEED_STRIDE * w.seed_id
    assert len({base, base + wl.STREAM_W, base + wl.STREAM_M}) == 3
    assert wl.SEED_STRIDE > max(x.count for x in map(wl.workload, wl.WORKLOADS))
    ns = wl.make_inputs(wl.workload("expert_gate"), "cpu", indices=[0])
    assert set(ns) == {"G"} and ns["G"][0].dtype == torch.bfloat16
