"""Pins of the oracle's fixed-point probability model.

* the Phi table and Phi_q against scipy.special.ndtr (an independent Phi);
* brute force over every rank: cum(0) = 0, cum(|S|) = 2^M, every freq >= 1;
* freq / 2^M against the continuous mixture mass computed with scipy, so a
  dropped component, a wrong weight, 3 sigma applied to the variance, or an
  off-by-one in the p-hat index fails;
* E_q against an empirical CDF built by numpy from raw samples.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import ndtr

GOLD = os.path.join(os.path.dirname(__file__), "golden")
ONE = 1 << 26


def _model(O, dtype, counts=None, weights=(95, 3, 2)):
    sigma = np.ones(2 * 8, dtype=np.float32)
    if dtype == O.BF16 and counts is None:
        counts = np.zeros(65536, dtype=np.uint64)
    return O.Model(dtype, 1, 1, 8, 8, 8, 1, sigma, counts=counts, weights=weights)


def test_phi_table_against_scipy(oracle_mod):
    T = oracle_mod.phi_table().astype(np.float64)
    z = -8.0 + np.arange(8193) / 512.0
    ref = ndtr(z) * ONE
    assert T[0] == 0 and T[8192] == ONE
    assert np.all(np.diff(T) >= 0)
    assert np.max(np.abs(T[1:-1] - ref[1:-1])) <= 0.5 + 1e-6
    assert abs(T[4096] - ONE / 2) == 0


def test_phi_q_against_scipy(oracle_mod):
    O = oracle_mod
    rng = np.random.default_rng(1)
    z = np.concatenate([rng.uniform(-8.5, 8.5, 20000).astype(np.float32),
                        np.float32([-8.0, 8.0, 0.0, -0.0, 1e-30, -1e-30, -1e-10, 7.9999995])])
    got = np.array([O.phi_q(v) for v in z], dtype=np.float64)
    ref = ndtr(z.astype(np.float64))
    # table rounding (0.5/2^26) + linear interpolation (h^2/8 max|phi'| ~ 1.2e-7)
    assert np.max(np.abs(got / ONE - ref)) <= 2e-7
    assert O.phi_q(-np.inf) == 0 and O.phi_q(np.inf) == ONE
    assert O.phi_q(-8.0) == 0 and O.phi_q(8.0) == ONE


def test_phi_q_monotone_and_exact_fraction(oracle_mod):
    O = oracle_mod
    z = np.sort(np.concatenate([
        np.linspace(-8.1, 8.1, 30001, dtype=np.float32),
        -np.logspace(-40, -1, 2000).astype(np.float32),
        np.logspace(-40, -1, 2000).astype(np.float32)]))
    got = np.array([O.phi_q(v) for v in z], dtype=np.int64)
    assert np.all(np.diff(got) >= 0)
    # a tiny negative z sits just below the centre knot: T[4095] + 65535/65536 of the step,
    # which only an exact fraction gives (fp32 t - floor(t) would round up to 1)
    T = O.phi_table().astype(np.int64)
    want = T[4095] + (((T[4096] - T[4095]) * 65535) >> 16)
    for z in (-1e-12, -3.2e-19, -1e-20, -1e-30, -1e-38, -1e-45):
        assert O.phi_q(np.float32(z)) == want, z
    assert O.phi_q(np.float32(-0.0)) == T[4096]
    assert O.phi_q(np.float32(1e-45)) == T[4096]
    # just below every knot: floor(65536 (t - floor t)) = 65535 with i one knot down
    for i in (1, 100, 4000, 4096, 8000, 8191):
        z = np.nextafter(np.float32((-4096 + i) / 512.0), np.float32(-np.inf))
        want_i = T[i - 1] + (((T[i] - T[i - 1]) * 65535) >> 16)
        assert O.phi_q(z) == want_i, i


EXTREME_SIGMA = [1.1754944e-38, 1e-30, 1e-8, 1.0, 1e30, 1e37]
EXTREME_MU = [0.0, -0.0, 9.2e-41, -9.2e-41, 1e-38, 3.3895314e38, -3.3895314e38, 1.0, -2.5]


@pytest.mark.parametrize("dtype", [0, 1])
def test_freq_invariants_brute_force(oracle_mod, dtype):
    O = oracle_mod
    rng = np.random.default_rng(7 + dtype)
    counts = rng.integers(0, 1000, 65536).astype(np.uint64) if dtype == O.BF16 else None
    m = _model(O, dtype, counts)
    M = O.PRECISION[dtype]
    cases = [(mu, s) for mu in EXTREME_MU for s in EXTREME_SIGMA]
    n_rand = 300 if dtype == O.BF16 else 2000
    for _ in range(n_rand):
        mu = float(np.float32(rng.standard_normal() * 10 ** rng.uniform(-6, 3)))
        s = float(np.float32(10 ** rng.uniform(-5, 3)))
        cases.append((mu, s))
    for mu, s in cases:
        c = O.cum_all(m, mu, s).astype(np.int64)
        assert c[0] == 0 and c[-1] == (1 << M), (mu, s)
        assert np.all(np.diff(c) >= 1), (mu, s)


def _bf16_values(O):
    return np.array([O.bf16_value(O.bits(O.BF16, r)) for r in range(65282)])


def test_bf16_freq_matches_mixture_mass(oracle_mod):
    """freq/2^M equals 0.95 m(sigma) + 0.03 m(3 sigma) + 0.02 p-hat to table accuracy."""
    O = oracle_mod
    gold = json.load(open(os.path.join(GOLD, "pages_constants.json")))
    w1, w3, we = gold["mixture_weights"]["value"]
    k3 = gold["wide_component_std_factor"]["value"]
    rng = np.random.default_rng(3)
    # heavy-tailed counts, so neighbouring ranks have very different p-hat and an
    # off-by-one in the p-hat index moves freq far outside the tolerance
    counts = (rng.pareto(0.7, 65536) * 1e4).astype(np.uint64)
    m = _model(O, O.BF16, counts)
    lo = np.array([O.lo(O.BF16, r) for r in range(65283)], dtype=np.float64)
    pat = np.array([O.bits(O.BF16, r) for r in range(65282)])
    cnt = counts[pat].astype(np.float64) + 1.0
    phat = cnt / cnt.sum()
    K = (1 << 28) - 65282
    for mu, s in [(0.37, 0.01), (-3.0, 0.2), (1e-3, 1e-4), (120.0, 2.0)]:
        mu = float(np.float32(mu)); s = float(np.float32(s))
        c = O.cum_all(m, mu, s).astype(np.float64)
        freq = np.diff(c)
        mass = (w1 * (ndtr((lo[1:] - mu) / s) - ndtr((lo[:-1] - mu) / s)) +
                w3 * (ndtr((lo[1:] - mu) / (k3 * s)) - ndtr((lo[:-1] - mu) / (k3 * s))) +
                we * phat)
        expect = K * mass + 1.0
        # Phi_q error (2e-7 of K per edge, weighted) + floor rounding
        tol = 2 * 2e-7 * K + 2.0 + we * 2 * 1.0
        assert np.max(np.abs(freq - expect)) <= tol, (mu, s)
        big = mass > 1e-3
        assert big.sum() > 3


def test_e4m3_freq_matches_gaussian_mass(oracle_mod):
    O = oracle_mod
    m = _model(O, O.E4M3)
    lo = np.array([O.lo(O.E4M3, r) for r in range(255)], dtype=np.float64)
    K = (1 << 16) - 254
    for mu, s in [(0.0, 1.0), (100.3, 3.0), (-7.7, 0.4), (447.0, 20.0), (0.01, 0.002)]:
        mu = float(np.float32(mu)); s = float(np.float32(s))
        c = O.cum_all(m, mu, s).astype(np.float64)
        mass = ndtr((lo[1:] - mu) / s) - ndtr((lo[:-1] - mu) / s)
        assert np.max(np.abs(np.diff(c) - (K * mass + 1.0))) <= 2 * 2e-7 * K + 1.0


def test_ecdf_against_empirical_cdf(oracle_mod):
    """E_q[r] / 2^26 is the smoothed fraction of calibration samples below value(r)."""
    O = oracle_mod
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200000) * 0.7).astype(np.float32)
    pat = (x.view(np.uint32) >> 16).astype(np.uint16)   # truncation: any bf16 sample set
    counts = np.bincount(pat, minlength=65536).astype(np.uint64)
    E = O.build_ecdf(counts).astype(np.float64)
    assert E[0] == 0 and E[65282] == ONE and np.all(np.diff(E) >= 0)
    vals = (pat.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    svals = np.sort(vals)
    for r in [1, 100, 20000, 32640, 32641, 32642, 40000, 65281]:
        v = O.bf16_value(O.bits(O.BF16, r))
        below = np.searchsorted(svals, v, side="left")
        if v == 0.0:   # -0 sorts before +0 in rank order, numpy ties them
            below = np.searchsorted(svals, 0.0, side="left") + (
                np.count_nonzero((pat == 0x8000)) if r == 32641 else 0)
        want = ONE * (below + r) / (len(x) + 65282)
        assert abs(E[r] - want) <= 1.0, r


def test_model_hash_sensitivity(oracle_mod):
    O = oracle_mod
    counts = np.zeros(65536, dtype=np.uint64)
    a = _model(O, O.BF16, counts)
    h = O.model_hash(a)
    sig = a.sigma.copy(); sig[3] = np.nextafter(sig[3], np.float32(2))
    b = O.Model(O.BF16, 1, 1, 8, 8, 8, 1, sig, counts=counts)
    assert O.model_hash(b) != h
    c2 = counts.copy(); c2[0x3F80] = 5
    c = O.Model(O.BF16, 1, 1, 8, 8, 8, 1, a.sigma, counts=c2)
    assert O.model_hash(c) != h
    assert O.model_hash(_model(O, O.BF16, counts)) == h
