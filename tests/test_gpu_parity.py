"""GPU parity: the CUDA path through the C ABI against the oracle.

Bar: containers byte-identical to the oracle's, decoded caches identical to the
input, per-scalar ideal bits within |gpu - oracle| <= 1e-3 |oracle| + 1e-6 bits,
and coded size at most 1% over the summed ideal.  Sizes span several chunks
and lanes with a ragged last token block; the lane count G is swept.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import (check_encode_with_bits, check_model_bits, device_views, gpu_codec,
                         host_views, oracle_model)

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-3, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _roundtrip(O, w, Tb=None, G=None, ideal=True, max_overhead=None):
    """max_overhead: bound on coded/ideal - 1 (the configs' 1%); by default only the
    fixed container and flush costs are allowed on top of 0.5%."""
    codec = gpu_codec(w, Tb, G)
    kv_d, mu_d = device_views(w)
    buf, nb = codec.encode(kv_d, mu_d)
    torch.cuda.synchronize()
    got = buf[:nb].cpu().numpy()
    m = oracle_model(O, w, Tb, G)
    kv, mu = host_views(w)
    rc, want = O.encode(m, kv, mu)
    assert rc == 0
    assert got.size == want.size and np.array_equal(got, want)
    dec = codec.decode(buf, nb, mu_d)
    assert torch.equal(dec, kv_d)
    # the reference bisection search returns the same symbols
    ref = gpu_codec(w, Tb, G, flags=1).decode(buf, nb, mu_d)
    assert torch.equal(ref, kv_d)
    check_model_bits(O, codec, m, kv_d, mu_d, kv, mu, got)
    if ideal:
        tot, ps = codec.ideal_bits(kv_d, mu_d, per_scalar=True)
        ref_tot, ref = O.ideal_bits(m, kv, mu, per_scalar=True)
        ps = ps.double().cpu().numpy()
        assert np.all(np.abs(ps - ref) <= RTOL * np.abs(ref) + ATOL)
        assert abs(tot - ps.sum()) <= 1e-6 * abs(tot)  # fp32 sums of 8 inside fp64
        assert abs(tot - ref_tot) <= RTOL * ref_tot
        # encode and ideal bits in one pass: the same container, the same bits
        check_encode_with_bits(codec, kv_d, mu_d, got, ref, ref_tot)
        nc = m.num_chunks()
        if max_overhead is not None:
            assert 8.0 * nb <= (1.0 + max_overhead) * ref_tot
        else:
            fixed = 512 + 64 * (nc + 1) + 64 * m.s.G * nc
            assert 8.0 * nb <= 1.005 * ref_tot + fixed
    return nb


def test_tiny_bf16_workload(oracle_mod):
    _roundtrip(oracle_mod, synth.make("tiny-bf16"), max_overhead=0.01)


@pytest.mark.parametrize("name", ["qwen3-0.6b-bf16", "qwen3-8b-e4m3"])
def test_scaled_workload_ragged(oracle_mod, name):
    # the full-size recipe on 2 layers x 2 heads x 600 tokens: 3 token blocks of
    # 256, the last one ragged (88 tokens), 8 lanes
    spec = synth.WORKLOADS[name].scaled(L=2, H=2, T=600, calib_draws=4)
    _roundtrip(oracle_mod, synth.make(spec))


@pytest.mark.parametrize("dtype", [synth.BF16, synth.E4M3])
@pytest.mark.parametrize("G", [1, 2, 4, 16, 32])
def test_lane_sweep(oracle_mod, dtype, G):
    base = "qwen3-0.6b-bf16" if dtype == synth.BF16 else "qwen3-8b-e4m3"
    spec = synth.WORKLOADS[base].scaled(name="lanes%d" % G, L=1, H=2, T=200, D=64, Tb=64,
                                        calib_draws=2)
    _roundtrip(oracle_mod, synth.make(spec), G=G)


@pytest.mark.parametrize("T,Tb,D", [(1, 256, 8), (7, 4, 8), (33, 1000, 16), (5, 1, 128)])
def test_odd_geometries(oracle_mod, T, Tb, D):
    spec = synth.WORKLOADS["tiny-bf16"].scaled(name="odd", L=1, H=1, T=T, D=D, Tb=Tb, G=8)
    _roundtrip(oracle_mod, synth.make(spec))
    spec8 = synth.WORKLOADS["qwen3-8b-e4m3"].scaled(name="odd8", L=1, H=1, T=T, D=D, Tb=Tb, G=2)
    _roundtrip(oracle_mod, synth.make(spec8))


def _custom(dtype, kv_np, mu_np, sigma_np, counts=None, T=None, D=8, Tb=32, G=4):
    n = kv_np.size
    T = T or n // (2 * D)
    spec = synth.Spec("custom", dtype, 1, 1, T, D, 0.03, False, 0, 0, False, Tb, G)
    kv = torch.from_numpy(kv_np.view(np.int16) if dtype == synth.BF16 else kv_np).reshape(1, 2, 1, T, D)
    if dtype == synth.BF16:
        kv = kv.view(torch.bfloat16)
    mu = torch.from_numpy(mu_np.view(np.int16)).view(torch.bfloat16).reshape(1, 2, 1, T, D)
    sig = torch.from_numpy(sigma_np.astype(np.float32)).reshape(1, 2, 1, D)
    cnt = None if counts is None else torch.from_numpy(counts.astype(np.int64))
    return synth.Workload(spec, kv, mu, sig, cnt)


def test_bf16_special_symbols(oracle_mod):
    rng = np.random.default_rng(3)
    specials = np.array([0xFF80, 0x7F80, 0x0000, 0x8000, 0x7F7F, 0xFF7F, 0x0001, 0x8001, 0x3F80,
                         0x0080, 0x807F], dtype=np.uint16)
    n = 2 * 64 * 8
    kv = rng.choice(specials, n).astype(np.uint16)
    mu = rng.choice(np.array([0x3F80, 0x0000, 0xC2C8, 0x0001, 0x7F7F, 0xFF7F], np.uint16), n)
    sigma = np.array([1e-30, 1e-8, 1.0, 1e30, 1.17549435e-38, 3.0, 0.5, 1e37] * 2)
    counts = rng.integers(0, 50, 65536).astype(np.uint64)
    # coded size against ideal: a random mix of specials under absurd sigma is
    # far from the model, so only a loose bound applies
    _roundtrip(oracle_mod, _custom(synth.BF16, kv, mu, sigma, counts), max_overhead=1.0)


# every non-NaN bf16 pattern, in rank order: from -inf (0xFF80) down the
# negative patterns to -0, then +0 up to +inf (0x7F80)
_BF16_ALL = np.concatenate([np.arange(0xFF80, 0x7FFF, -1, dtype=np.int64),
                            np.arange(0x0000, 0x7F81, dtype=np.int64)]).astype(np.uint16)

# (sigma per channel, mu values): tiny to huge sigma, mu at zero, at the
# smallest subnormals and at the largest finite values of both signs
_ALPHABET_CASES = [
    ([1.17549435e-38, 1e-30, 1e-8], [0x0000, 0x0001, 0x8001]),
    ([1.0, 3.0, 0.01], [0x0000, 0x3F80, 0xC2C8, 0x4120]),
    ([1e30, 1e37, 1e20], [0x7F7F, 0xFF7F, 0x0000]),
    ([1e-8, 1.0, 1e37], [0x7F7F, 0x0001, 0xFF7F, 0x8001]),
]


@pytest.mark.parametrize("case", range(len(_ALPHABET_CASES)))
def test_every_bf16_symbol(oracle_mod, case):
    """All 65,282 non-NaN bf16 symbols, each twice in a seeded permutation, under
    extreme sigma and mu: the GPU's cum and ideal bits reach every rank,
    including the subnormal edges, +-max and +-inf."""
    assert _BF16_ALL.size == 65282 and len(set(_BF16_ALL.tolist())) == 65282
    sigmas, mus = _ALPHABET_CASES[case]
    rng = np.random.default_rng(100 + case)
    D = 64
    T = (2 * _BF16_ALL.size + 2 * D - 1) // (2 * D)
    n = 2 * T * D
    kv = np.concatenate([rng.permutation(_BF16_ALL), rng.permutation(_BF16_ALL)])
    kv = np.concatenate([kv, rng.choice(_BF16_ALL, n - kv.size)]).astype(np.uint16)
    mu = rng.choice(np.array(mus, dtype=np.uint16), n).astype(np.uint16)
    sigma = np.resize(np.array(sigmas, dtype=np.float64), 2 * D)
    counts = rng.integers(0, 200, 65536).astype(np.uint64)
    _roundtrip(oracle_mod, _custom(synth.BF16, kv, mu, sigma, counts, T=T, D=D, Tb=128, G=8),
               max_overhead=1.0)


def test_every_e4m3_symbol(oracle_mod):
    rng = np.random.default_rng(4)
    codes = np.array([u for u in range(256) if u not in (0x7F, 0xFF)], dtype=np.uint8)
    kv = np.concatenate([rng.permutation(codes) for _ in range(8)])
    for mu_v, s in [(0.0, 1.0), (300.0, 5.0), (-0.01, 1e-3), (40.0, 200.0), (-448.0, 0.5)]:
        mu = torch.full((kv.size,), mu_v, dtype=torch.bfloat16).view(torch.int16).numpy()
        sigma = np.full(16, s)
        _roundtrip(oracle_mod, _custom(synth.E4M3, kv, mu.view(np.uint16), sigma))


def test_repeat_calls_are_deterministic(oracle_mod):
    w = synth.make(synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(L=1, H=2, T=512, calib_draws=2))
    codec = gpu_codec(w)
    kv_d, mu_d = device_views(w)
    a, na = codec.encode(kv_d, mu_d)
    a = a[:na].clone()
    b, nb = codec.encode(kv_d, mu_d)
    assert na == nb and torch.equal(a, b[:nb])
    t1 = codec.ideal_bits(kv_d, mu_d)
    t2 = codec.ideal_bits(kv_d, mu_d)
    assert t1 == t2


def _bf16_near_case_edges(rng, T, D):
    """bf16 scalars whose bins sit on both sides of the ideal-bits kernel's case
    boundaries (bin width w < 1 and w |z_m| < 2, in sigma units): sigma is a
    power of two times (1 + delta), the symbol's binade sets w near 2^k_w, and mu
    is the symbol a few patterns away, so that w |z_m| lands near |steps| w^2."""
    deltas = np.array([-1e-2, -1e-3, -1e-5, 0.0, 1e-5, 1e-3, 1e-2])
    j = rng.integers(-8, 9, 2 * D)
    sig = np.ldexp(1.0 + rng.choice(deltas, 2 * D), j)
    n = 2 * T * D
    ch = (np.arange(n) // (T * D)) * D + np.arange(n) % D
    kw = rng.choice([-2, -1, 0, 0, 1], n)
    e = 7 + j[ch] + kw
    x = np.ldexp(1.0 + rng.integers(0, 128, n) / 128.0, e) * rng.choice([-1.0, 1.0], n)
    kv = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # exact in bf16
    steps = rng.choice([0, 1, 2, 3, 7, 8, 9, 31, 32, 33], n) * rng.choice([-1, 1], n)
    mu = (kv.astype(np.int64) + steps).astype(np.uint16)
    # keep mu finite and on x's side of zero (adjacent patterns are adjacent values there)
    bad = ((mu & 0x7F80) == 0x7F80) | ((mu ^ kv) & 0x8000 != 0)
    mu[bad] = kv[bad]
    return kv, mu, sig


def test_ideal_bits_case_edges(oracle_mod):
    """Per-scalar ideal bits on both sides of every case boundary of the kernel
    (bf16 series / erfc tails, e4m3 difference of tails / deep tail at 9 sigma)."""
    rng = np.random.default_rng(11)
    T, D = 128, 64
    kv, mu, sig = _bf16_near_case_edges(rng, T, D)
    counts = rng.integers(0, 50, 65536).astype(np.uint64)
    w = _custom(synth.BF16, kv, mu, sig, counts, T=T, D=D, Tb=32, G=4)
    _roundtrip(oracle_mod, w, max_overhead=0.05)
    # e4m3: mu placed 8.5 to 9.5 sigma beyond the bin edge on its side
    codes = np.array([u for u in range(256) if u not in (0x7F, 0xFF)], dtype=np.uint8)
    n = 2 * T * D
    kv8 = rng.choice(codes, n).astype(np.uint8)
    r = np.array([oracle_mod.rank(1, int(u)) for u in kv8])
    lo = np.array([oracle_mod.lo(1, int(q)) for q in r])
    hi = np.array([oracle_mod.lo(1, int(q) + 1) for q in r])
    val = np.where(np.isfinite(lo), lo, hi)
    sig8 = np.exp(rng.uniform(np.log(1e-2), np.log(10.0), 2 * D))
    ch = (np.arange(n) // (T * D)) * D + np.arange(n) % D
    a = rng.uniform(8.5, 9.5, n) * sig8[ch]
    above = rng.random(n) < 0.5  # mu above the bin: the far edge is hi
    mu_v = np.where(above, np.where(np.isfinite(hi), hi, val) + a, np.where(np.isfinite(lo), lo, val) - a)
    mu8 = (torch.from_numpy(mu_v.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
           .numpy().view(np.uint16))
    _roundtrip(oracle_mod, _custom(synth.E4M3, kv8, mu8, sig8, T=T, D=D, Tb=32, G=4),
               max_overhead=1.0)


def test_ideal_bits_e4m3_narrow_bins(oracle_mod):
    """e4m3 bins 0.0095 to 1 sigma wide (both sides of the kernel's 0.01 sigma
    cut-off between its tail table and the full evaluation), mu within two
    sigma of the bin's lower edge: one-sided and straddling bins near z = 0,
    where the table's error bound is tightest.  Per-scalar ideal bits against
    the oracle."""
    rng = np.random.default_rng(12)
    T, D = 64, 64
    n = 2 * T * D
    normal = np.array([u for u in range(0x08, 0x7F)] + [u | 0x80 for u in range(0x08, 0x7F)], dtype=np.uint8)
    codes = rng.choice(normal, 2 * D)
    r = np.array([oracle_mod.rank(1, int(u)) for u in codes])
    width = np.array([oracle_mod.lo(1, int(q) + 1) - oracle_mod.lo(1, int(q)) for q in r])
    lo = np.array([oracle_mod.lo(1, int(q)) for q in r])
    w_target = rng.choice([0.0095, 0.0099, 0.0101, 0.0105, 0.02, 0.05, 0.2, 1.0], 2 * D)
    sig = width / w_target
    ch = (np.arange(n) // (T * D)) * D + np.arange(n) % D
    kv8 = codes[ch].astype(np.uint8)
    mu_v = lo[ch] + rng.uniform(-2.0, 2.0, n) * sig[ch]
    mu8 = (torch.from_numpy(mu_v.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
           .numpy().view(np.uint16))
    _roundtrip(oracle_mod, _custom(synth.E4M3, kv8, mu8, sig, T=T, D=D, Tb=32, G=4),
               max_overhead=1.0)


@pytest.mark.parametrize("flags", [0, 2], ids=["static", "block-scale"])
def test_encode_with_bits_inside_the_encoder(oracle_mod, flags):
    """skv_encode_with_bits computes the ideal bits inside the encoder on bf16
    mixture caches of any size, with or without per-block scales (e4m3 and the
    order-0 coder run the ideal-bits pass behind it): here a cache with more
    chunk lanes than one round of the encoder's blocks holds, 2 layers x 8
    heads x 4090 tokens x 64 in 16-token blocks (8,192 chunks, the last token
    block ragged) x 16 lanes, with the model's sigma or per-block scales."""
    spec = synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(name="fused-bits", L=2, H=8, T=4090, D=64,
                                                     Tb=16, G=16, calib_draws=2)
    w = synth.make(spec)
    codec = gpu_codec(w, flags=flags)
    assert codec.encode_with_bits_fused()
    assert gpu_codec(synth.make("tiny-bf16")).encode_with_bits_fused()
    tiny8 = synth.WORKLOADS["qwen3-8b-e4m3"].scaled(name="tiny-e4m3", L=1, H=2, T=300, D=64,
                                                    Tb=128, G=4)
    assert not gpu_codec(synth.make(tiny8)).encode_with_bits_fused()
    kv_d, mu_d = device_views(w)
    buf, nb = codec.encode(kv_d, mu_d)
    got = buf[:nb].cpu().numpy()
    m = oracle_model(oracle_mod, w, block_scale=bool(flags))
    kv, mu = host_views(w)
    rc, want = oracle_mod.encode(m, kv, mu)
    assert rc == 0 and np.array_equal(got, want)
    ref_tot, ref = oracle_mod.ideal_bits(m, kv, mu, per_scalar=True)
    check_encode_with_bits(codec, kv_d, mu_d, got, ref, ref_tot)
    # the separate pass gives the same per-scalar values within the tolerance
    tot, ps = codec.ideal_bits(kv_d, mu_d, per_scalar=True)
    _, _, tot2, ps2 = codec.encode_with_bits(kv_d, mu_d, per_scalar=True)
    assert torch.allclose(ps2, ps, rtol=RTOL, atol=ATOL)
    assert abs(tot2 - tot) <= 1e-6 * tot


@pytest.mark.parametrize("shrink", [0.2, 0.05, 0.01], ids=["5x", "20x", "100x"])
def test_model_far_too_narrow(oracle_mod, shrink):
    """A sigma table 5-100 times narrower than the residuals: most symbols sit
    in the tails, where the first guess and Newton miss, so warp steps end with
    many lanes open at once (the warp search then serves 2-16 lanes side by
    side).  Containers byte-equal to the oracle, both searches decode exactly.
    2 layers x 2 heads x 600 tokens x 128, 256-token blocks (the last ragged),
    8 lanes."""
    w = synth.make(synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(name="narrow", L=2, H=2, T=600,
                                                             G=8, calib_draws=2))
    w.sigma.mul_(shrink)
    _roundtrip(oracle_mod, w, ideal=False)
