"""GPU parity of the order-0 baseline coder (SKV_FLAG_ORDER0; page "推测式 KV 编码
无损压缩 KV 缓存最高可达约 4 倍", introduction: an entropy coder over the bf16
symbols alone, about 11 bits per value).

Byte-identical containers against the oracle on ragged cases across lane
counts, decode with NULL mu and sigma, ideal bits per scalar within 1e-3
relative, model separation from the predictive coder, and the full-size
Qwen3-0.6B-shaped cache on sampled chunks in the configuration bench.py times.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import check_encode_with_bits, check_model_bits, container_chunk, skv

pytestmark = pytest.mark.gpu

O0 = 4  # SKV_FLAG_ORDER0


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _codec(w, flags=O0, Tb=None, G=None):
    P = skv()
    s = w.spec
    E, ph = P.skv_build_ecdf(w.counts.cpu().numpy().astype(np.uint64))
    ecdf = torch.from_numpy(E.view(np.int32)).cuda()
    phat = torch.from_numpy(ph).cuda()
    sigma = None if flags & O0 else w.sigma.cuda()
    return P.Codec(s.dtype, s.L, s.H, s.T, s.D, Tb or s.Tb, G or s.G, sigma, ecdf, phat,
                   flags=flags)


def _oracle(O, w, Tb=None, G=None):
    s = w.spec
    return O.Model(0, s.L, s.H, s.T, s.D, Tb or s.Tb, G or s.G, None,
                   counts=w.counts.cpu().numpy().astype(np.uint64), weights=(0, 0, 100))


CASES = [dict(L=1, H=2, T=600), dict(L=1, H=1, T=37, D=64, Tb=16, G=1),
         dict(L=1, H=1, T=130, D=40, Tb=64, G=4), dict(L=2, H=1, T=300, Tb=128, G=32)]


@pytest.mark.parametrize("kw", CASES, ids=[str(i) for i in range(len(CASES))])
def test_order0_parity(oracle_mod, kw):
    O = oracle_mod
    spec = synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(name="o0g-%d-%d" % (kw["T"], kw.get("D", 128)),
                                                     calib_draws=2, **kw)
    w = synth.make(spec)
    codec = _codec(w)
    kv_d = w.kv.view(torch.int16).reshape(-1).cuda()
    buf, nb = codec.encode(kv_d, None)
    got = buf[:nb].cpu().numpy()
    m = _oracle(O, w)
    kv_h = kv_d.cpu().numpy().view(np.uint16)
    rc, want = O.encode(m, kv_h, None)
    assert rc == 0 and got.size == want.size and np.array_equal(got, want)
    rc, dec = O.decode(m, got, None)
    assert rc == 0 and np.array_equal(dec, kv_h)
    assert torch.equal(codec.decode(buf, nb, None), kv_d)
    check_model_bits(O, codec, m, kv_d, None, kv_h, None, got)
    tot, ps = codec.ideal_bits(kv_d, None, per_scalar=True)
    ref_tot, ref = O.ideal_bits(m, kv_h, None, 0, kv_h.size, per_scalar=True)
    assert np.all(np.abs(ps.double().cpu().numpy() - ref) <= 1e-3 * np.abs(ref) + 1e-6)
    assert abs(tot - ref_tot) <= 1e-5 * ref_tot
    check_encode_with_bits(codec, kv_d, None, got, ref, ref_tot)
    # the predictive codec refuses the order-0 container (feature bit)
    P = skv()
    mu_d = w.mu.view(torch.int16).reshape(-1).cuda()
    with pytest.raises(P.SkvError) as e:
        _codec(w, flags=0).decode(buf, nb, mu_d)
    assert e.value.status == P.SKV_ERR_CORRUPT


def test_order0_tampering_and_nan():
    P = skv()
    spec = synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(name="o0g-t", L=1, H=1, T=256,
                                                     calib_draws=1)
    w = synth.make(spec)
    codec = _codec(w)
    kv_d = w.kv.view(torch.int16).reshape(-1).cuda()
    buf, nb = codec.encode(kv_d, None)
    rng = np.random.default_rng(1)
    head = 64 + 8 * 3
    for _ in range(20):
        t = buf[:nb].clone()
        pos = int(rng.integers(head, nb))
        t[pos] ^= 1 << int(rng.integers(0, 8))
        try:
            out = codec.decode(t, nb, None)
            assert not torch.equal(out, kv_d)
        except P.SkvError as err:
            assert err.status == P.SKV_ERR_CORRUPT
    bad = kv_d.clone()
    bad[5] = 0x7FC1
    with pytest.raises(P.SkvError) as e:
        codec.encode(bad, None)
    assert e.value.status == P.SKV_ERR_SYMBOL
    assert torch.equal(codec.decode(buf, nb, None), kv_d)


@pytest.mark.slow
def test_order0_fullsize_sampled(oracle_mod):
    O = oracle_mod
    w = synth.make("qwen3-0.6b-bf16", device="cuda")
    s = w.spec
    codec = _codec(w)
    kv_d = w.kv.view(torch.int16).reshape(-1)
    buf, nb = codec.encode(kv_d, None)
    assert torch.equal(codec.decode(buf, nb, None), kv_d)
    tot = codec.ideal_bits(kv_d, None)
    assert 10.5 <= 8.0 * nb / s.n <= 11.7                  # the pages' ~11 bits
    assert 8.0 * nb <= 1.01 * tot
    m = _oracle(O, w)
    nc = m.num_chunks()
    host = buf[:nb].cpu().numpy()
    assert O.check_header(m, host) == 0
    chunks = sorted(set(np.linspace(0, nc - 1, 24).astype(np.int64).tolist()))
    kv_h = kv_d.cpu().numpy().view(np.uint16)
    want = O.encode_chunks(m, kv_h, None, chunks)
    for c, ww in zip(chunks, want):
        assert np.array_equal(container_chunk(host, nc, c), ww), c
