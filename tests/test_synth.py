"""The seeded input recipe: deterministic, with the stated distributions and structure."""
import math

import torch

import synth


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def test_layer_and_step_draws_are_deterministic_per_seed():
    w = synth.small(B=2, Hq=4, Hkv=2, D=32, dp=8, N=300, seed=5, outliers=2, planted=3)
    a, b = synth.make_layer(w), synth.make_layer(w)
    for key in ("Wk", "K", "V", "q", "q_imp", "outlier_ch", "planted_pos"):
        assert torch.equal(_bits(a[key]), _bits(b[key])), key
    c = synth.make_layer(synth.small(B=2, Hq=4, Hkv=2, D=32, dp=8, N=300, seed=6, outliers=2, planted=3))
    assert not torch.equal(_bits(a["K"]), _bits(c["K"]))
    s1, s2 = synth.make_step(w, 0, 3, a["outlier_ch"]), synth.make_step(w, 0, 3, a["outlier_ch"])
    for key in s1:
        assert torch.equal(_bits(s1[key]), _bits(s2[key])), key
    assert not torch.equal(_bits(s1["q"]), _bits(synth.make_step(w, 0, 4, a["outlier_ch"])["q"]))
    assert not torch.equal(_bits(s1["q"]), _bits(synth.make_step(w, 1, 3, a["outlier_ch"])["q"]))


def test_distributions_and_outlier_channels():
    w = synth.small(B=1, Hq=8, Hkv=4, D=128, dp=32, N=4096, seed=7, outliers=4)
    L = synth.make_layer(w)
    ch = L["outlier_ch"].tolist()
    assert len(set(ch)) == 4
    K = L["K"].float()
    rest = [d for d in range(w.D) if d not in ch]
    assert abs(K[..., rest].std().item() - 1.0) < 0.02
    assert abs(K[..., ch].std().item() - w.outlier_scale) < 0.2
    assert abs(L["V"].float().std().item() - 1.0) < 0.02
    assert abs(L["Wk"].float().std().item() - 1.0 / math.sqrt(w.D)) < 0.005
    Kn = synth.make_step(w, 0, 0, L["outlier_ch"])["K_new"].float()
    assert Kn[..., ch].abs().mean() > 4 * Kn[..., rest].abs().mean()


def test_cache_rows_beyond_n_are_zero():
    w = synth.small(B=1, Hq=4, Hkv=2, D=16, dp=8, N=50, seed=8)
    L = synth.make_layer(w, cap=64, n=40)
    assert L["K"].shape == (1, 2, 64, 16) and L["V"].shape == (1, 2, 64, 16)
    assert not L["K"][:, :, 40:].float().any() and not L["V"][:, :, 40:].float().any()
    assert L["K"][:, :, :40].float().abs().sum() > 0


def test_workload_table_and_budgets():
    w1 = synth.WORKLOADS[1]
    assert (w1.B, w1.Hq, w1.Hkv, w1.D, w1.dp, w1.N, w1.k) == (1, 32, 8, 128, 32, 32768, 3277)
    assert synth.budget(0.10, 32768) == 3277
    w4 = synth.WORKLOADS[4]
    assert [synth.budget(p, w4.N) for p in w4.budgets] == [656, 3277, 6554, 16384, 65536]
    w2 = synth.WORKLOADS[2]
    assert (w2.layers, w2.B, w2.N, w2.k, w2.T, w2.r, w2.steps) == (32, 8, 16384, 1024, 16, 1, 64)
    w3 = synth.WORKLOADS[3]
    assert (w3.B, w3.N, w3.k, w3.planted) == (4, 131072, 2048, 64)
