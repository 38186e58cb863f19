"""The synthetic inputs follow the stated recipe (CPU): log-normal channel
scales with four x10 outlier channels per (layer, kv, head) row, the residual
mu - x drawn from 0.95 N(0, sc^2) + 0.03 N(0, (3 sc)^2) + 0.02 Laplace(0, 20 sc),
the e4m3 caches scaled by absmax/448 per (layer, head), and every draw a pure
function of (workload, seed)."""
import numpy as np
import torch

import synth

SPEC = synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(name="recipe", L=2, H=4, T=2048, D=128,
                                                 calib_draws=1, calib_tokens=64)


def test_channel_scales_lognormal_with_four_outliers_per_row():
    s = synth.channel_scale(SPEC, "cpu").numpy().reshape(-1, SPEC.D)
    plain = synth.channel_scale(SPEC.scaled(outliers=False), "cpu").numpy().reshape(-1, SPEC.D)
    ratio = s / plain
    assert np.all(np.isclose(ratio, 1.0) | np.isclose(ratio, 10.0))
    assert np.all((np.isclose(ratio, 10.0)).sum(axis=1) == 4)
    lg = np.log(plain.reshape(-1))
    assert abs(lg.mean()) < 0.15 and abs(lg.std() - 1.0) < 0.1   # 2048 draws of N(0, 1)


def test_residual_mixture_moments_and_tail():
    w = synth.make(SPEC)
    x = w.kv.float().numpy()
    mu = w.mu.float().numpy()
    sc = (SPEC.sigma_c * synth.channel_scale(SPEC, "cpu")).numpy()[:, :, :, None, :]
    z = ((mu - x) / sc).reshape(-1)
    # E z^2 = 0.95 + 0.03 * 9 + 0.02 * 2 * 20^2 = 17.22 (bf16 rounding of mu adds ~1e-3)
    assert abs(np.mean(z * z) / 17.22 - 1.0) < 0.05
    # P(|z| > 10): the Laplace part 0.02 exp(-1/2) = 0.01213, the 3-sigma part 2.6e-5
    tail = np.mean(np.abs(z) > 10.0)
    assert abs(tail / 0.01216 - 1.0) < 0.1
    # the core: 95% of mass in N(0, 1); |z| < 1 holds 0.95 * 0.6827 + 0.03 * 0.2611 + small
    core = np.mean(np.abs(z) < 1.0)
    assert abs(core - (0.95 * 0.6827 + 0.03 * 0.2611 + 0.02 * 0.0488)) < 0.01


def test_e4m3_absmax_scaling():
    spec = synth.WORKLOADS["qwen3-8b-e4m3"].scaled(name="recipe8", L=2, H=2, T=512)
    w = synth.make(spec)
    vals = w.kv.view(torch.float8_e4m3fn).float().numpy()        # [L, 2, H, T, D]
    amax = np.abs(vals).max(axis=(1, 3, 4))                        # per (layer, head)
    assert np.all(amax == 448.0)                                   # the absmax element maps to 448
    assert not np.isnan(vals).any()


def test_draws_are_pure_functions_of_workload_and_seed():
    a = synth.make(SPEC, seed=3)
    b = synth.make(SPEC, seed=3)
    c = synth.make(SPEC, seed=4)
    assert torch.equal(a.kv.view(torch.int16), b.kv.view(torch.int16))
    assert torch.equal(a.mu.view(torch.int16), b.mu.view(torch.int16))
    assert torch.equal(a.counts, b.counts) and torch.equal(a.sigma, b.sigma)
    assert not torch.equal(a.kv.view(torch.int16), c.kv.view(torch.int16))
