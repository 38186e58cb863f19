"""Pins for the oracle's per-block sigma scales (page "推测式 KV 编码无损压缩 KV 缓存
最高可达约 4 倍", section "下一步计划": the error scale moves with prompt and
position, so a static per-channel sigma costs bits).

The rule: s = clamp(b_med + C, 0, 255) per (chunk, 8-channel group), b the
1/32-octave bin of |x - mu| / sigma read from the fp32 bits, C = 18 (bf16) or
21 (e4m3); sigma_eff = fp32(sigma * fp32(2^((s - 128) / 32))).  Pinned here
against things other than the oracle: mpmath for m(s); hand-built residuals
whose bins follow from frexp; the already-pinned static coder and ideal bits
run with sigma_eff written into the sigma table.
"""
import math

import numpy as np
import pytest

import synth

mp = pytest.importorskip("mpmath")


def _bin_frexp(a: float) -> int:
    """32 (e + f) for a = 2^e (1 + f), by frexp (not by reading float bits)."""
    if not a > 0:
        return 0
    if math.isinf(a):
        return 255
    m, e = math.frexp(a)          # a = m 2^e, m in [0.5, 1)
    e, f = e - 1, 2.0 * m - 1.0   # a = 2^e (1 + f)
    return min(max(int(math.floor(32 * (e + f))) + 128, 0), 255)


def _model(O, dtype, T, D, Tb, G, sigma, counts=None, bs=True):
    return O.Model(dtype, 1, 1, T, D, Tb, G, sigma, counts=counts, block_scale=bs)


def _flat_counts():
    return np.ones(65536, dtype=np.uint64)


def test_scale_multipliers_are_rounded_powers_of_two(oracle_mod):
    mp.mp.prec = 80
    for s in range(256):
        want = np.float32(float(mp.power(2, mp.mpf(s - 128) / 32)))  # exact -> RN to binary32
        assert np.float32(oracle_mod.scale_mult(s)) == want, s
    assert oracle_mod.scale_mult(128) == 1.0
    assert oracle_mod.scale_mult(96) == 0.5 and oracle_mod.scale_mult(160) == 2.0


@pytest.mark.parametrize("v", [0.0078125, 0.3, 0.7, 1.0, 1.03, 2.5, 17.0, 300.0])
def test_constant_residual_gives_its_bin(oracle_mod, v):
    """bf16: mu = 0, sigma = 1, every x = +-v: the median bin is bin(v)."""
    O = oracle_mod
    T, D = 16, 16
    sigma = np.ones(2 * D, dtype=np.float32)
    xv = np.float32(v)
    xb = (np.array([xv], dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)[0]
    vb = float(np.array([xb], dtype=np.uint32).astype(np.uint32).__lshift__(16).view(np.float32)[0])
    kv = np.full((1, 2, 1, T, D), xb, dtype=np.uint16)
    kv[..., ::2, :] |= 0x8000                          # half of them negative
    mu = np.zeros_like(kv)
    m = _model(O, 0, T, D, T, 4, sigma, _flat_counts())
    sc = O.chunk_scales(m, kv, mu, 0)
    want = min(max(_bin_frexp(vb) + 18, 0), 255)
    assert sc.tolist() == [want, want]


def test_lower_median_and_group_independence(oracle_mod):
    """n = 8 T residuals per group: exactly half at bin b1 -> b1; one fewer -> b2;
    the two groups of a 16-channel chunk are chosen independently."""
    O = oracle_mod
    T, D = 8, 16
    sigma = np.ones(2 * D, dtype=np.float32)
    one, four = np.uint16(0x3F80), np.uint16(0x4080)    # 1.0 and 4.0
    kv = np.full((1, 2, 1, T, D), four, dtype=np.uint16)
    g0 = kv[0, 0, 0, :, :8].reshape(-1)
    g0[:32] = one                                       # 32 of 64 at bin(1)
    g1 = kv[0, 0, 0, :, 8:].reshape(-1)
    g1[:31] = one                                       # 31 of 64 at bin(1)
    kv[0, 0, 0, :, :8] = g0.reshape(T, 8)
    kv[0, 0, 0, :, 8:] = g1.reshape(T, 8)
    mu = np.zeros_like(kv)
    m = _model(O, 0, T, D, T, 2, sigma, _flat_counts())
    sc = O.chunk_scales(m, kv, mu, 0)
    assert sc.tolist() == [_bin_frexp(1.0) + 18, _bin_frexp(4.0) + 18]
    # the same with e4m3 codes (1.0 = 0x38, 4.0 = 0x48) and C = 21
    kv8 = np.where(kv == one, 0x38, 0x48).astype(np.uint8)
    m8 = _model(O, 1, T, D, T, 2, sigma)
    assert O.chunk_scales(m8, kv8, mu, 0).tolist() == [_bin_frexp(1.0) + 21,
                                                      _bin_frexp(4.0) + 21]


def test_zero_nan_inf_and_clamps(oracle_mod):
    O = oracle_mod
    T, D = 4, 8
    sigma = np.ones(2 * D, dtype=np.float32)
    mu = np.zeros((1, 2, 1, T, D), dtype=np.uint16)
    m = _model(O, 0, T, D, T, 1, sigma, _flat_counts())
    zero = np.zeros_like(mu)                            # |x - mu| = 0: bin 0, s = 18
    assert O.chunk_scales(m, zero, mu, 0).tolist() == [18]
    inf = np.full_like(mu, 0x7F80)                      # +inf: bin 255, s clamps to 255
    # sigma * 2^(127/32) stays valid, so 255 is kept
    assert O.chunk_scales(m, inf, mu, 0).tolist() == [255]
    # a group whose sigma_eff would overflow takes 128
    big = np.full(2 * D, 3e37, dtype=np.float32)
    mb = _model(O, 0, T, D, T, 1, big, _flat_counts())
    assert O.chunk_scales(mb, inf, mu, 0).tolist() == [128]


@pytest.mark.parametrize("rho", [0.25, 0.5, 1.0, 2.0, 5.0])
def test_recovers_a_known_sigma_multiplier(oracle_mod, rho):
    """Residuals drawn from the model's own core 0.95 N(0, (rho s)^2) + 0.03
    N(0, (3 rho s)^2): s lands within the bin rule's bias of 128 + 32 log2 rho."""
    O = oracle_mod
    rng = np.random.default_rng(7)
    T, D = 512, 8
    sig = 0.01
    sigma = np.full(2 * D, sig, dtype=np.float32)
    n = 2 * T * D
    wide = rng.random(n) < 0.03 / 0.98
    r = rng.standard_normal(n) * rho * sig * np.where(wide, 3.0, 1.0)
    mu_f = (rng.standard_normal(n) * 0.5).astype(np.float32)
    mu = (mu_f.view(np.uint32) >> 16).astype(np.uint16)
    mu_v = (mu.astype(np.uint32) << 16).view(np.float32)
    x = (mu_v + r).astype(np.float32)
    xb = ((x.view(np.uint32) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
    m = _model(O, 0, T, D, T, 4, sigma, _flat_counts())
    s = int(O.chunk_scales(m, xb.reshape(1, 2, 1, T, D), mu.reshape(1, 2, 1, T, D), 0)[0])
    assert abs(s - (128 + 32 * math.log2(rho))) <= 5, s


@pytest.mark.parametrize("dtype", [0, 1])
def test_block_scaled_coder_is_the_static_coder_with_sigma_eff(oracle_mod, dtype):
    """One chunk per row (Tb = T): the chunk's payload after its scale words is
    exactly the static coder's payload for the sigma table sigma_eff, and the
    ideal bits agree scalar by scalar."""
    O = oracle_mod
    spec = synth.WORKLOADS["qwen3-0.6b-bf16-drift" if dtype == 0 else "qwen3-8b-e4m3"].scaled(
        name="bs-eq-%d" % dtype, L=1, H=2, T=96, D=32, calib_draws=1, Tb=96, G=4)
    w = synth.make(spec)
    kv, mu, sigma, counts = synth.to_numpy(w)
    mb = O.Model(dtype, 1, 2, 96, 32, 96, 4, sigma, counts=counts, block_scale=True)
    rc, buf = O.encode(mb, kv, mu)
    assert rc == 0
    assert int(buf[38]) | int(buf[39]) << 8 == 1          # header feature bit
    nc = mb.num_chunks()
    head = 64 + 8 * (nc + 1)
    offs = buf[64:head].view(np.uint64)
    sig_eff = sigma.reshape(2, 2, 32).copy()              # [kv][h][d]; chunk c = row c
    for c in range(nc):
        words = buf[head + int(offs[c]): head + int(offs[c + 1])].view(np.uint32)
        sc = O.chunk_scales(mb, kv, mu, c)
        packed = np.zeros(4 * ((32 // 8 + 3) // 4), dtype=np.uint8)
        packed[: sc.size] = sc
        assert np.array_equal(words[:1].view(np.uint8), packed)
        kv_i, h = divmod(c, 2)
        mult = np.array([O.scale_mult(int(s)) for s in sc], dtype=np.float32)
        sig_eff[kv_i, h] = (sigma.reshape(2, 2, 32)[kv_i, h] * np.repeat(mult, 8)).astype(np.float32)
    ms = O.Model(dtype, 1, 2, 96, 32, 96, 4, sig_eff.reshape(-1), counts=counts)
    rc, ref = O.encode(ms, kv, mu)
    assert rc == 0
    roffs = ref[64:head].view(np.uint64)
    for c in range(nc):
        got = buf[head + int(offs[c]): head + int(offs[c + 1])].view(np.uint32)[1:]
        want = ref[head + int(roffs[c]): head + int(roffs[c + 1])].view(np.uint32)
        assert np.array_equal(got, want), c
    tb, pb = O.ideal_bits(mb, kv, mu, 0, kv.size, per_scalar=True)
    ts, ps = O.ideal_bits(ms, kv, mu, 0, kv.size, per_scalar=True)
    assert np.array_equal(pb, ps)
    rc, dec = O.decode(mb, buf, mu)
    assert rc == 0 and np.array_equal(dec.reshape(-1), kv.reshape(-1))


@pytest.mark.parametrize("name", ["qwen3-0.6b-bf16-drift", "qwen3-8b-e4m3"])
def test_round_trip_ragged_and_gain_on_drift(oracle_mod, name):
    O = oracle_mod
    spec = synth.WORKLOADS[name].scaled(name="bs-rt-" + name, L=1, H=2, T=700, calib_draws=2)
    w = synth.make(spec)
    kv, mu, sigma, counts = synth.to_numpy(w)
    out = {}
    for bs in (False, True):
        m = O.Model(spec.dtype, 1, 2, 700, 128, spec.Tb, spec.G, sigma, counts=counts,
                    block_scale=bs)
        rc, buf = O.encode(m, kv, mu)
        assert rc == 0
        rc, dec = O.decode(m, buf, mu)
        assert rc == 0 and np.array_equal(dec.reshape(-1), kv.reshape(-1))
        out[bs] = buf.size
        if bs:
            # a static-sigma model refuses the scaled container (feature bit)
            m0 = O.Model(spec.dtype, 1, 2, 700, 128, spec.Tb, spec.G, sigma, counts=counts)
            assert O.decode(m0, buf, mu)[0] == O.ERR_CORRUPT
    if spec.drift > 0:
        assert out[True] < 0.95 * out[False]


def test_scale_byte_tampering(oracle_mod):
    """A scale byte the encoder cannot have chosen is corrupt; any other change
    decodes to a different cache or fails, never to the same one silently."""
    O = oracle_mod
    spec = synth.WORKLOADS["qwen3-0.6b-bf16-drift"].scaled(name="bs-tamper", L=1, H=1, T=256,
                                                            calib_draws=1)
    w = synth.make(spec)
    kv, mu, sigma, counts = synth.to_numpy(w)
    # group 0 of row (kv=0, h=0): sigma just above FLT_MIN and x = mu, so the
    # median bin is 0, s would be 18 and sigma_eff = sigma 2^(-110/32) underflows
    small = sigma.reshape(-1).copy()
    small[:8] = 1.2e-38
    kv = kv.copy()
    kv[0, 0, 0, :, :8] = mu[0, 0, 0, :, :8]
    m = O.Model(0, 1, 1, 256, 128, 256, 16, small, counts=counts, block_scale=True)
    rc, buf = O.encode(m, kv, mu)
    assert rc == 0
    head = 64 + 8 * (m.num_chunks() + 1)
    assert buf[head] == 128                           # forced by the range check
    t = buf.copy()
    t[head] = 18
    assert O.decode(m, t, mu)[0] == O.ERR_CORRUPT
    t = buf.copy()
    t[head + 1] ^= 1
    rc, dec = O.decode(m, t, mu)
    assert rc == O.ERR_CORRUPT or not np.array_equal(dec.reshape(-1), kv.reshape(-1))
