"""Pins of the oracle's rANS coder and container.

* decode(encode(x)) == x: random bf16 and e4m3 caches, every lane count, ragged
  last token blocks, and every e4m3 symbol against several (mu, sigma);
* the rANS length invariant: per chunk, the coded bits exceed the model's own
  code length sum(-log2(freq / 2^M)) by the flush cost only, i.e. by between
  32 and 64 bits per lane (initial state 2^31, final state < 2^63);
* the container header and offsets reject tampering.
"""
import numpy as np
import pytest

import synth


def _tiny_model(O, dtype, L, H, T, D, Tb, G, rng, counts=None):
    sigma = (np.exp(rng.standard_normal(L * 2 * H * D)) * 0.05).astype(np.float32)
    if dtype == O.BF16 and counts is None:
        counts = rng.integers(0, 100, 65536).astype(np.uint64)
    return O.Model(dtype, L, H, T, D, Tb, G, sigma, counts=counts)


def _random_cache(O, m, rng, outlier_frac=0.02):
    L, _, H, T, D = m.shape
    n = m.n
    ch = np.arange(n) % D
    row = np.arange(n) // (T * D)
    s = m.sigma[row * D + ch].astype(np.float64)
    if m.dtype == O.BF16:
        x = rng.standard_normal(n) * 1.0
        xb = (x.astype(np.float32).view(np.uint32) + 0x8000 >> 16).astype(np.uint16)  # approx RNE
        xv = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        r = rng.standard_normal(n) * s
        out = rng.random(n) < outlier_frac
        r[out] *= 40
        mu = (xv + r).astype(np.float32)
        mub = (mu.view(np.uint32) + 0x8000 >> 16).astype(np.uint16)
        return xb, mub
    x = rng.standard_normal(n) * 60.0
    import torch
    x8 = torch.from_numpy(np.clip(x, -448, 448).astype(np.float32)).to(torch.float8_e4m3fn)
    xv = x8.float().numpy().astype(np.float64)
    r = rng.standard_normal(n) * s * 40
    mub = torch.from_numpy((xv + r).astype(np.float32)).to(torch.bfloat16)
    return x8.view(torch.uint8).numpy(), mub.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32])
def test_roundtrip_random_ragged(oracle_mod, dtype, G):
    O = oracle_mod
    rng = np.random.default_rng(100 + G + 7 * dtype)
    # T = 70 with Tb = 32: two full blocks and a ragged block of 6 tokens
    m = _tiny_model(O, dtype, 1, 2, 70, 16, 32, G, rng)
    kv, mu = _random_cache(O, m, rng)
    rc, buf = O.encode(m, kv, mu)
    assert rc == 0
    rc, dec = O.decode(m, buf, mu)
    assert rc == 0 and np.array_equal(dec, kv)


def test_roundtrip_every_e4m3_symbol(oracle_mod):
    O = oracle_mod
    rng = np.random.default_rng(5)
    codes = np.array([u for u in range(256) if u not in (0x7F, 0xFF)], dtype=np.uint8)
    for mu_v, s in [(0.0, 1.0), (300.0, 5.0), (-0.01, 1e-3), (40.0, 200.0), (-448.0, 0.5)]:
        D = 8
        T = 254 * 4 // D
        sigma = np.full(2 * D, s, dtype=np.float32)
        m = O.Model(O.E4M3, 1, 1, T, D, 32, 4, sigma)
        kv = np.concatenate([rng.permutation(codes), rng.permutation(codes),
                             rng.permutation(codes), rng.permutation(codes)]).astype(np.uint8)
        kv = np.concatenate([kv, kv])  # K and V
        import torch
        mub = torch.full((kv.size,), mu_v, dtype=torch.bfloat16).view(torch.int16).numpy()
        mub = mub.view(np.uint16)
        rc, buf = O.encode(m, kv, mub)
        assert rc == 0
        rc, dec = O.decode(m, buf, mub)
        assert rc == 0 and np.array_equal(dec, kv)


def test_roundtrip_bf16_specials(oracle_mod):
    """+-inf, +-0, +-max and subnormals round-trip."""
    O = oracle_mod
    rng = np.random.default_rng(9)
    special = np.array([0xFF80, 0x7F80, 0x0000, 0x8000, 0x7F7F, 0xFF7F, 0x0001, 0x8001, 0x3F80],
                       dtype=np.uint16)
    m = _tiny_model(O, O.BF16, 1, 1, 72, 8, 16, 4, rng)
    kv = rng.choice(special, m.n).astype(np.uint16)
    mu = rng.choice(np.array([0x3F80, 0x0000, 0xC2C8, 0x0001], dtype=np.uint16), m.n)
    rc, buf = O.encode(m, kv, mu)
    assert rc == 0
    rc, dec = O.decode(m, buf, mu)
    assert rc == 0 and np.array_equal(dec, kv)


@pytest.mark.parametrize("dtype", [0, 1])
def test_rans_length_invariant(oracle_mod, dtype):
    O = oracle_mod
    rng = np.random.default_rng(21 + dtype)
    G = 4
    m = _tiny_model(O, dtype, 1, 2, 512, 32, 128, G, rng)
    kv, mu = _random_cache(O, m, rng)
    for c in range(m.num_chunks()):
        words = O.encode_chunk(m, kv, mu, c)
        ideal = O.model_bits_chunk(m, kv, mu, c)
        over = 32.0 * words.size - ideal
        assert 32 * G - 1.0 <= over <= 64 * G + 1.0, (c, over)


def test_errors(oracle_mod):
    O = oracle_mod
    rng = np.random.default_rng(2)
    m = _tiny_model(O, O.BF16, 1, 1, 32, 8, 16, 2, rng)
    kv, mu = _random_cache(O, m, rng)
    bad = kv.copy(); bad[5] = 0x7FC0  # NaN symbol
    assert O.encode(m, bad, mu)[0] == O.ERR_SYMBOL
    badmu = mu.copy(); badmu[7] = 0x7F80  # mu = +inf
    assert O.encode(m, kv, badmu)[0] == O.ERR_PARAM
    sig = m.sigma.copy(); sig[0] = 0.0
    m0 = O.Model(O.BF16, 1, 1, 32, 8, 16, 2, sig, counts=m.counts)
    assert O.encode(m0, kv, mu)[0] == O.ERR_PARAM
    e = _tiny_model(O, O.E4M3, 1, 1, 32, 8, 16, 2, rng)
    kv8, mu8 = _random_cache(O, e, rng)
    kv8 = kv8.copy(); kv8[3] = 0x7F
    assert O.encode(e, kv8, mu8)[0] == O.ERR_SYMBOL


def test_container_tamper(oracle_mod):
    O = oracle_mod
    rng = np.random.default_rng(4)
    m = _tiny_model(O, O.BF16, 1, 2, 64, 16, 32, 4, rng)
    kv, mu = _random_cache(O, m, rng)
    rc, buf = O.encode(m, kv, mu)
    assert rc == 0 and O.check_header(m, buf) == 0
    assert buf[:4].tobytes() == b"SKV1"
    nc = m.num_chunks()
    assert int.from_bytes(buf[40:48].tobytes(), "little") == nc
    head = 64 + 8 * (nc + 1)
    assert int.from_bytes(buf[48:56].tobytes(), "little") == buf.size - head
    for off in (0, 4, 6, 7, 8, 20, 28, 32, 40, 56):
        t = buf.copy(); t[off] ^= 1
        assert O.decode(m, t, mu)[0] == O.ERR_CORRUPT, off
    # truncated payload, flipped payload bits, a wrong-mu decode
    assert O.decode(m, buf[:-4], mu)[0] == O.ERR_CORRUPT
    for k in range(20):
        t = buf.copy(); pos = head + int(rng.integers(0, buf.size - head)); t[pos] ^= 1 << int(rng.integers(0, 8))
        rc, dec = O.decode(m, t, mu)
        # a clean finish (every state back at L, every word used) on a changed
        # stream implies different symbols: the encoder is injective
        assert rc == O.ERR_CORRUPT or (rc == 0 and not np.array_equal(dec, kv))
    mu2 = mu.copy(); mu2[0] ^= 1
    rc, dec = O.decode(m, buf, mu2)
    assert rc in (0, O.ERR_CORRUPT)


def test_synthetic_tiny_workload_near_ideal(oracle_mod):
    """On the tiny synthetic cache the coded size is within 1% of the ideal cost."""
    O = oracle_mod
    w = synth.make("tiny-bf16")
    kv, mu, sigma, counts = synth.to_numpy(w)
    s = w.spec
    m = O.Model(O.BF16, s.L, s.H, s.T, s.D, s.Tb, s.G, sigma, counts=counts)
    rc, buf = O.encode(m, kv, mu)
    assert rc == 0
    rc, dec = O.decode(m, buf, mu)
    assert rc == 0 and np.array_equal(dec, kv.reshape(-1))
    ideal = O.ideal_bits(m, kv, mu)
    coded = 8.0 * buf.size
    assert ideal <= coded <= 1.01 * ideal


@pytest.mark.parametrize("dtype", [0, 1])
def test_compare_container_accepts_own_and_finds_every_change(oracle_mod, dtype):
    """The whole-container check (chunk slices on several threads) accepts the
    oracle's own container and names the chunk of any changed payload byte or
    offset; a changed header is refused before any chunk is coded."""
    O = oracle_mod
    rng = np.random.default_rng(300 + dtype)
    m = _tiny_model(O, dtype, 2, 2, 70, 16, 16, 4, rng)
    kv, mu = _random_cache(O, m, rng)
    rc, buf = O.encode(m, kv, mu)
    assert rc == 0
    assert O.compare_container(m, kv, mu, buf, threads=3)[:2] == (0, -1)
    nc = m.num_chunks()
    head = 64 + 8 * (nc + 1)
    offs = buf[64:head].view(np.uint64)
    for c in rng.choice(nc, 6, replace=False):
        t = buf.copy()
        pos = head + int(offs[c]) + int(rng.integers(0, int(offs[c + 1] - offs[c])))
        t[pos] ^= 1 << int(rng.integers(0, 8))
        rc, bad, _ = O.compare_container(m, kv, mu, t, threads=3)
        assert rc == O.ERR_CORRUPT and bad == c
    t = buf.copy()
    t[64 + 8 * 5] += 4                # chunk 4 one word longer, chunk 5 one shorter
    rc, bad, _ = O.compare_container(m, kv, mu, t, threads=2)
    assert rc == O.ERR_CORRUPT and bad == 4
    t = buf.copy()
    t[20] ^= 1                        # the token count in the header
    assert O.compare_container(m, kv, mu, t)[0] == O.ERR_CORRUPT
    # a range of chunks alone
    assert O.compare_container(m, kv, mu, buf, begin=3, end=9)[:2] == (0, -1)
