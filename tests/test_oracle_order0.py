"""Pins for the oracle's order-0 baseline coder (page "推测式 KV 编码无损压缩 KV 缓存
最高可达约 4 倍", introduction: an entropy coder over the bf16 symbols alone,
with one static distribution and no prediction, gets to about 11 bits per
value).  The baseline is the same rANS coder with q = p-hat: weights
(0, 0, 100), no mu, no sigma.

Pinned against: the pages' ~11-bit figure on the Qwen3-shaped synthetic
cache; the rANS code-length bounds against frequencies recomputed here from
the raw counts with Python integers; independence of mu and sigma; the
container's feature bit and model separation.
"""
import math

import numpy as np
import pytest

import synth


def _setup(O, name="qwen3-0.6b-bf16", **kw):
    kw.setdefault("L", 1)
    kw.setdefault("H", 2)
    kw.setdefault("T", 520)
    kw.setdefault("calib_draws", 4)
    spec = synth.WORKLOADS[name].scaled(name="o0-" + name, **kw)
    w = synth.make(spec)
    kv, mu, sigma, counts = synth.to_numpy(w)
    m = O.Model(0, spec.L, spec.H, spec.T, spec.D, spec.Tb, spec.G, None, counts=counts,
                weights=(0, 0, 100))
    return spec, kv.reshape(-1), mu.reshape(-1), sigma, counts, m


def test_about_eleven_bits_on_the_qwen3_shaped_cache(oracle_mod):
    O = oracle_mod
    spec, kv, mu, sigma, counts, m = _setup(O, T=1024)
    rc, buf = O.encode(m, kv, None)
    assert rc == 0
    bits = 8.0 * buf.size / kv.size
    assert 10.5 <= bits <= 11.7, bits
    # the predictive coder on the same cache is far below it
    mm = O.Model(0, spec.L, spec.H, spec.T, spec.D, spec.Tb, spec.G, sigma, counts=counts)
    rc, buf2 = O.encode(mm, kv, mu)
    assert rc == 0 and 8.0 * buf2.size / kv.size < 0.6 * bits


def test_code_length_against_frequencies_from_the_raw_counts(oracle_mod):
    """Per chunk: 32 G - eps <= coded bits - sum(M - log2 freq) <= 64 G + eps, with
    freq(r) = cum(r+1) - cum(r), cum(r) = floor(K floor(2^26 S_r / S) / 2^26) + r
    computed here from the counts in exact integer arithmetic."""
    O = oracle_mod
    spec, kv, mu, sigma, counts, m = _setup(O, T=300, calib_draws=1)
    nsym, M = 65282, 28
    K = (1 << M) - nsym
    # ranks in value order: negative patterns from -inf up to -0, then +0 .. +inf
    pats = [0xFF80 - i for i in range(0x7F81)] + list(range(0x7F81))
    assert len(pats) == nsym
    cnt = [int(counts[p]) + 1 for p in pats]
    S = sum(cnt)
    cum, acc = [], 0
    for r in range(nsym + 1):
        E = (acc << 26) // S if r < nsym else 1 << 26
        cum.append(((K * E) >> 26) + r)
        if r < nsym:
            acc += cnt[r]
    assert cum[0] == 0 and cum[-1] == 1 << M
    rank = {p: r for r, p in enumerate(pats)}
    nc = m.num_chunks()
    words = O.encode_chunks(m, kv, None, range(nc))
    Tb, D, G = spec.Tb, spec.D, spec.G
    ntb = (spec.T + Tb - 1) // Tb
    for c in range(nc):
        row, tb = divmod(c, ntb)
        base = row * spec.T * D + tb * Tb * D
        n_c = min(Tb, spec.T - tb * Tb) * D
        ideal = sum(M - math.log2(cum[rank[int(u)] + 1] - cum[rank[int(u)]])
                    for u in kv[base: base + n_c])
        extra = 32 * len(words[c]) - ideal
        assert 32 * G - 1e-6 <= extra <= 64 * G + 1e-6, (c, extra)


def test_mu_and_sigma_are_not_read(oracle_mod):
    O = oracle_mod
    spec, kv, mu, sigma, counts, m = _setup(O, T=260, calib_draws=1)
    rc, a = O.encode(m, kv, None)
    rng = np.random.default_rng(3)
    m2 = O.Model(0, spec.L, spec.H, spec.T, spec.D, spec.Tb, spec.G,
                 rng.random(sigma.size).astype(np.float32), counts=counts, weights=(0, 0, 100))
    rc2, b = O.encode(m2, kv, rng.integers(0, 65535, kv.size).astype(np.uint16))
    assert rc == rc2 == 0 and np.array_equal(a, b)
    assert int(a[38]) | int(a[39]) << 8 == 2                # header feature bit 1
    rc, dec = O.decode(m, a, None)
    assert rc == 0 and np.array_equal(dec, kv)
    # the predictive model refuses the order-0 container and the reverse
    mm = O.Model(0, spec.L, spec.H, spec.T, spec.D, spec.Tb, spec.G, sigma, counts=counts)
    assert O.decode(mm, a, mu)[0] == O.ERR_CORRUPT
    rc, c = O.encode(mm, kv, mu)
    assert rc == 0 and O.decode(m, c, None)[0] == O.ERR_CORRUPT


@pytest.mark.parametrize("G,Tb,T", [(1, 16, 37), (4, 64, 130), (32, 256, 300)])
def test_round_trip_ragged(oracle_mod, G, Tb, T):
    O = oracle_mod
    spec, kv, mu, sigma, counts, m = _setup(O, name="tiny-bf16", L=1, H=1, T=T, Tb=Tb, G=G)
    rc, buf = O.encode(m, kv, None)
    assert rc == 0
    rc, dec = O.decode(m, buf, None)
    assert rc == 0 and np.array_equal(dec, kv)
    tot = O.ideal_bits(m, kv, None)
    stot = float((counts.astype(np.float64) + 1).sum() - 254)   # NaN patterns excluded
    assert abs(tot - sum(-math.log2((float(counts[u]) + 1) / stot) for u in kv)) < 1e-6 * tot


def test_invalid_combinations(oracle_mod):
    O = oracle_mod
    sigma = np.ones(2 * 64, dtype=np.float32)
    kv8 = np.zeros(2 * 16 * 64, dtype=np.uint8)
    m8 = O.Model(1, 1, 1, 16, 64, 16, 4, sigma, weights=(0, 0, 100))
    assert O.encode(m8, kv8, np.zeros(kv8.size, dtype=np.uint16))[0] == O.ERR_ARG
    mb = O.Model(0, 1, 1, 16, 64, 16, 4, sigma, counts=np.ones(65536, dtype=np.uint64),
                 weights=(0, 0, 100), block_scale=True)
    kv = np.zeros(2 * 16 * 64, dtype=np.uint16)
    assert O.encode(mb, kv, np.zeros(kv.size, dtype=np.uint16))[0] == O.ERR_ARG
