"""GPU parity of the adaptive-counts coder (SKV_FLAG_ORDER0 | SKV_FLAG_ADAPTIVE;
page "KV 缓存压缩的熵估计与动态适应": decayed counts per (layer, kv, head), smoothed
updates every N_update tokens).

Containers byte-identical to the oracle's on ragged cases and lane counts,
decode back to the input, ideal bits per scalar within 1e-3 relative, model
separation from the static order-0 coder, and the full-size Qwen3-0.6B-shaped
cache (N_update = 128) on sampled chunks.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import container_chunk, skv

pytestmark = pytest.mark.gpu

O0, AD = 4, 8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _codec(w, flags=O0 | AD):
    P = skv()
    s = w.spec
    E, ph = P.skv_build_ecdf(w.counts.cpu().numpy().astype(np.uint64))
    return P.Codec(s.dtype, s.L, s.H, s.T, s.D, s.Tb, s.G, None,
                   torch.from_numpy(E.view(np.int32)).cuda(), torch.from_numpy(ph).cuda(),
                   flags=flags)


def _oracle(O, w, adaptive=True):
    s = w.spec
    return O.Model(0, s.L, s.H, s.T, s.D, s.Tb, s.G, None,
                   counts=w.counts.cpu().numpy().astype(np.uint64), weights=(0, 0, 100),
                   adaptive=adaptive)


CASES = [dict(L=1, H=2, T=600, Tb=128), dict(L=1, H=1, T=37, D=64, Tb=8, G=1),
         dict(L=2, H=1, T=130, D=40, Tb=32, G=4), dict(L=1, H=1, T=300, Tb=64, G=32)]


@pytest.mark.parametrize("kw", CASES, ids=[str(i) for i in range(len(CASES))])
def test_adaptive_parity(oracle_mod, kw):
    O = oracle_mod
    spec = synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(
        name="adg-%d-%d-%d" % (kw["T"], kw.get("D", 128), kw["Tb"]), calib_draws=2, **kw)
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
    tot, ps = codec.ideal_bits(kv_d, None, per_scalar=True)
    ref_tot, ref = O.ideal_bits(m, kv_h, None, 0, kv_h.size, per_scalar=True)
    assert np.all(np.abs(ps.double().cpu().numpy() - ref) <= 1e-3 * np.abs(ref) + 1e-6)
    assert abs(tot - ref_tot) <= 1e-5 * ref_tot
    P = skv()
    with pytest.raises(P.SkvError) as e:          # the static order-0 model refuses it
        _codec(w, flags=O0).decode(buf, nb, None)
    assert e.value.status == P.SKV_ERR_CORRUPT


@pytest.mark.slow
def test_adaptive_fullsize_sampled(oracle_mod):
    O = oracle_mod
    spec = synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(Tb=128)
    w = synth.make(spec, device="cuda")
    codec = _codec(w)
    kv_d = w.kv.view(torch.int16).reshape(-1)
    buf, nb = codec.encode(kv_d, None)
    assert torch.equal(codec.decode(buf, nb, None), kv_d)
    tot = codec.ideal_bits(kv_d, None)
    assert 8.0 * nb <= 1.01 * tot
    m = _oracle(O, w)
    nc = m.num_chunks()
    host = buf[:nb].cpu().numpy()
    assert O.check_header(m, host) == 0
    ntb = spec.T // spec.Tb
    chunks = sorted(set([0, 1, ntb - 1, ntb, nc - 1] +
                        np.linspace(0, nc - 1, 12).astype(np.int64).tolist()))
    kv_h = kv_d.cpu().numpy().view(np.uint16)
    want = O.encode_chunks(m, kv_h, None, chunks)
    for c, ww in zip(chunks, want):
        assert np.array_equal(container_chunk(host, nc, c), ww), c
