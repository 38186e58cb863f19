"""Statistical and closed-form pins from the pages, plus ideal bits vs mpmath.

P1 = "推测式 KV 编码无损压缩 KV 缓存最高可达约 4 倍" (Speculative KV coding).
* section "q 应是什么样的": for a Gaussian residual the rate is the Gaussian's
  entropy, 1/2 log2(2 pi e sigma^2 / Delta^2) bits for bin width Delta << sigma,
  and the best sigma^2 is E[(x - mu)^2];
* section "什么能预测 KV 缓存": a pure-noise predictor costs close to 16 bits;
* the oracle's float64 -log2 q(x) agrees with an 80-digit mpmath evaluation of
  the same mixture mass (tails, narrow bins, bins straddling mu, +-inf).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _val(u):
    with np.errstate(invalid="ignore"):
        return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _model(O, T, D, sigma, counts, weights, G=4, Tb=256, dtype=0):
    sig = np.full(2 * D, sigma, dtype=np.float32)
    return O.Model(dtype, 1, 1, T, D, Tb, G, sig, counts=counts, weights=weights)


def _gaussian_binade(rng, mu, sigma, n):
    """x = bf16(mu + N(0, sigma^2)) kept inside the binade [1, 2) (bin width 2^-7)."""
    x = mu + sigma * rng.standard_normal(int(n * 1.01) + 100)
    x = x[(x > 1.0 + 2 ** -7) & (x < 2.0 - 2 ** -7)][:n]
    assert x.size == n
    return _bf16(x)


@pytest.mark.parametrize("k", [4, 8, 16])
def test_gaussian_rate_closed_form(oracle_mod, k):
    O = oracle_mod
    gold = json.load(open(os.path.join(GOLD, "pages_constants.json")))
    assert "2*pi*e" in gold["gaussian_rate_bits"]["value"]
    rng = np.random.default_rng(k)
    delta = 2.0 ** -7
    sigma = k * delta
    D, T = 8, 1 << 16          # 2^20 samples
    n = 2 * T * D
    x = _gaussian_binade(rng, 1.5, sigma, n)
    mu = np.full(n, 0x3FC0, dtype=np.uint16)          # 1.5
    H = 0.5 * math.log2(2 * math.pi * math.e * sigma ** 2 / delta ** 2)
    counts = np.zeros(65536, dtype=np.uint64)
    # one chunk per K/V row, so flush and offset overhead is ~1e-4 bits/scalar
    pure = _model(O, T, D, sigma, counts, (100, 0, 0), Tb=T)
    rc, buf = O.encode(pure, x, mu)
    assert rc == 0
    coded = 8.0 * buf.size / n
    ideal = O.ideal_bits(pure, x, mu) / n
    assert abs(ideal - H) < 0.01
    assert abs(coded - H) < 0.01
    # the production mixture pays at most log2(1/0.95) on a Gaussian residual
    mix = _model(O, T, D, sigma, counts, (95, 3, 2), Tb=T)
    rc, buf = O.encode(mix, x, mu)
    coded_mix = 8.0 * buf.size / n
    assert H - 0.005 <= coded_mix <= H + math.log2(1 / 0.95) + 0.01


@pytest.mark.parametrize("weights", [(100, 0, 0), (95, 3, 2)])
def test_sigma_sweep_minimum_bf16(oracle_mod, weights):
    """The rate as a function of the model's sigma is convex with its minimum at E[(x-mu)^2]."""
    O = oracle_mod
    rng = np.random.default_rng(31)
    sigma = 6 * 2.0 ** -7
    D, T = 8, 1 << 14
    n = 2 * T * D
    x = _gaussian_binade(rng, 1.5, sigma, n)
    mu = np.full(n, 0x3FC0, dtype=np.uint16)
    rms = float(np.sqrt(np.mean((_val(x) - 1.5) ** 2)))
    counts = np.zeros(65536, dtype=np.uint64)
    cs = [0.5, 0.7, 0.85, 1.0, 1.2, 1.4, 2.0]
    rate = []
    for c in cs:
        m = _model(O, T, D, c * rms, counts, weights)
        rate.append(O.ideal_bits(m, x, mu) / n)
    assert int(np.argmin(rate)) == cs.index(1.0)
    slopes = np.diff(rate) / np.diff(cs)
    assert np.all(np.diff(slopes) > 0)


def test_sigma_sweep_minimum_e4m3(oracle_mod):
    """Bin-integrated Gaussian on e4m3: the true sigma minimises the coded size."""
    O = oracle_mod
    rng = np.random.default_rng(32)
    D, T = 8, 1 << 13
    n = 2 * T * D
    mu_v = rng.uniform(-60, 60, n)
    sigma = 20.0
    x = np.clip(mu_v + sigma * rng.standard_normal(n), -448, 448)
    x8 = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mu = _bf16(mu_v)
    cs = [0.5, 0.7, 0.85, 1.0, 1.2, 1.4, 2.0]
    rate = []
    for c in cs:
        m = _model(O, T, D, c * sigma, None, (95, 3, 2), dtype=O.E4M3, Tb=T)
        rc, buf = O.encode(m, x8, mu)
        assert rc == 0
        rate.append(8.0 * buf.size / n)
    assert int(np.argmin(rate)) == cs.index(1.0)
    slopes = np.diff(rate) / np.diff(cs)
    assert np.all(np.diff(slopes) > 0)


def test_pure_noise_predictor_costs_about_16_bits(oracle_mod):
    """mu independent of x and uninformative: the cost falls to the p-hat floor, ~16 bits."""
    O = oracle_mod
    gold = json.load(open(os.path.join(GOLD, "pages_constants.json")))
    target = gold["pure_noise_bits_per_bf16_scalar"]["value"]
    rng = np.random.default_rng(41)
    D, T = 8, 8192
    n = 2 * T * D
    x = _bf16(rng.standard_normal(n))
    calib = _bf16(rng.standard_normal(4 * n))
    counts = np.bincount(calib, minlength=65536).astype(np.uint64)
    pat = rng.integers(0, 65536, n).astype(np.uint16)
    v = _val(pat)
    mu = np.where(np.isfinite(v) & (np.abs(v) < 1e30), pat, 0x3F80).astype(np.uint16)
    d = _val(x) - _val(mu)
    m = _model(O, T, D, float(np.sqrt(np.mean(d * d))), counts, (95, 3, 2), Tb=T)
    rc, buf = O.encode(m, x, mu)
    assert rc == 0
    coded = 8.0 * buf.size / n
    assert target - 2 <= coded <= target + 2
    # the floor: -log2(0.02 p-hat(x)) on the calibrated empirical distribution
    cnt = counts.astype(np.float64) + 1.0
    stot = cnt.sum() - (65536 - 65282)  # NaN patterns carry no count
    floor = float(np.mean(-np.log2(0.02 * cnt[x] / stot)))
    assert abs(coded - floor) < 0.2


def _mp_bits(mp, lo, hi, mu, s, phat, w, dtype):
    lo, hi, mu, s = (mp.mpf(v) for v in (lo, hi, mu, s))

    def mass(sd):
        a = (lo - mu) / sd if lo != -mp.inf else -mp.inf
        b = (hi - mu) / sd if hi != mp.inf else mp.inf
        if a >= 0:
            return (mp.erfc(a / mp.sqrt(2)) - (mp.erfc(b / mp.sqrt(2)) if b != mp.inf else 0)) / 2
        if b <= 0:
            return ((mp.erfc(-b / mp.sqrt(2))) - (mp.erfc(-a / mp.sqrt(2)) if a != -mp.inf else 0)) / 2
        return mp.ncdf(b) - mp.ncdf(a)

    if dtype == 1:
        q = mass(s)
    else:
        q = w[0] * mass(s) + w[1] * mass(3 * s) + w[2] * mp.mpf(phat)
    return float(-mp.log(q, 2))


@pytest.mark.parametrize("dtype", [0, 1])
def test_ideal_bits_against_mpmath(oracle_mod, dtype):
    O = oracle_mod
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = 80
    rng = np.random.default_rng(50 + dtype)
    counts = rng.integers(0, 1000, 65536).astype(np.uint64)
    counts[0x3F80] = 10 ** 9
    m = O.Model(dtype, 1, 1, 8, 8, 8, 1, np.ones(16, np.float32),
                counts=counts if dtype == 0 else None)
    pat = np.array([O.bits(0, r) for r in range(65282)])
    stot = float((counts[pat].astype(np.float64) + 1).sum())
    cases = []
    if dtype == 0:
        syms = [0x3F80, 0x3F81, 0x0001, 0x8001, 0x0000, 0x8000, 0x7F80, 0xFF80, 0x7F7F, 0x4120,
                0xC2C8, 0x3A83, 0x2000]
        for u in syms:
            for mu_v, s in [(1.0, 0.01), (1.0, 1e-4), (0.0, 1.0), (10.0, 0.1), (-100.0, 0.5),
                            (1e-30, 1e-38), (3.0, 1e5)]:
                cases.append((u, mu_v, s))
    else:
        for u in [0x00, 0x80, 0x01, 0x38, 0x39, 0x7E, 0xFE, 0x50, 0xD0]:
            for mu_v, s in [(1.0, 0.05), (0.0, 1.0), (400.0, 3.0), (-1.0, 0.001), (448.0, 1.0),
                            (0.01, 10.0)]:
                cases.append((u, mu_v, s))
    for u, mu_v, s in cases:
        mub = int(_bf16([mu_v])[0])
        muv = float(_val(np.array([mub], np.uint16))[0])
        s32 = float(np.float32(s))
        r = O.rank(dtype, u)
        lo, hi = O.lo(dtype, r), O.lo(dtype, r + 1)
        phat = (float(counts[u]) + 1.0) / stot if dtype == 0 else 0.0
        want = _mp_bits(mp, lo, hi, muv, s32, phat, (0.95, 0.03, 0.02), dtype)
        got = O.ideal_bits_one(m, u, mub, s32)
        if math.isinf(want):
            assert math.isinf(got)
        else:
            assert abs(got - want) <= 1e-9 * max(1.0, abs(want)), (hex(u), mu_v, s, got, want)
