"""GPU parity of per-block sigma scales (SKV_FLAG_BLOCK_SCALE; page "推测式 KV 编码
无损压缩 KV 缓存最高可达约 4 倍", section "下一步计划": the error scale moves with
prompt and position).

The encoder's scale choice is an exact integer rule, so the CUDA containers
must equal the oracle's byte for byte; the oracle must decode them; ideal bits
must match per scalar within 1e-3 relative, and the coder's model bits per
chunk within 1e-5.  Small cases span several chunks
with a ragged last token block, every lane count class, and a head_dim whose
scale bytes do not fill their last word.  The full-size drift workload is
checked on an even sample of chunks in the configuration bench.py times.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import (check_encode_with_bits, check_model_bits, container_chunk, device_views,
                         gpu_codec, host_views, oracle_model)

pytestmark = pytest.mark.gpu

BS = 2  # SKV_FLAG_BLOCK_SCALE


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


CASES = [
    ("qwen3-0.6b-bf16-drift", dict(L=1, H=2, T=600, calib_draws=2)),
    ("qwen3-0.6b-bf16-drift", dict(L=1, H=1, T=300, D=40, calib_draws=1, Tb=64, G=4)),
    ("qwen3-0.6b-bf16-drift", dict(L=1, H=1, T=130, D=64, calib_draws=1, Tb=32, G=32)),
    ("qwen3-32b-bf16", dict(L=1, H=2, T=520, calib_draws=2)),
    ("qwen3-8b-e4m3", dict(L=1, H=2, T=600)),
    ("qwen3-8b-e4m3", dict(L=1, H=1, T=70, D=24, Tb=16, G=1)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[f"{c[0]}-{i}" for i, c in enumerate(CASES)])
def test_block_scale_parity(oracle_mod, name, kw):
    O = oracle_mod
    spec = synth.WORKLOADS[name].scaled(name="bsg-%s-%d-%d" % (name, kw["T"], kw.get("D", 128)),
                                        **kw)
    w = synth.make(spec)
    codec = gpu_codec(w, flags=BS)
    kv_d, mu_d = device_views(w)
    buf, nb = codec.encode(kv_d, mu_d)
    got = buf[:nb].cpu().numpy()
    m = oracle_model(O, w, block_scale=True)
    kv_h, mu_h = host_views(w)
    rc, want = O.encode(m, kv_h, mu_h)
    assert rc == 0
    assert got.size == want.size and np.array_equal(got, want)
    rc, dec = O.decode(m, got, mu_h)                      # the oracle reads the GPU container
    assert rc == 0 and np.array_equal(dec.reshape(-1), kv_h)
    assert torch.equal(codec.decode(buf, nb, mu_d), kv_d)
    assert torch.equal(gpu_codec(w, flags=BS | 1).decode(buf, nb, mu_d), kv_d)  # bisection
    # model bits under the scales the encoder chose, and the rANS length bound
    check_model_bits(O, codec, m, kv_d, mu_d, kv_h, mu_h, got)
    tot, ps = codec.ideal_bits(kv_d, mu_d, per_scalar=True)
    ref_tot, ref = O.ideal_bits(m, kv_h, mu_h, 0, kv_h.size, per_scalar=True)
    got_ps = ps.double().cpu().numpy()
    assert np.all(np.abs(got_ps - ref) <= 1e-3 * np.abs(ref) + 1e-6)
    assert abs(tot - ref_tot) <= 1e-4 * ref_tot
    check_encode_with_bits(codec, kv_d, mu_d, got, ref, ref_tot)
    # a static-sigma codec refuses the container (feature bit in the header)
    import lossless_kv_cache_fixed_gb300 as P
    with pytest.raises(P.SkvError) as e:
        gpu_codec(w).decode(buf, nb, mu_d)
    assert e.value.status == P.SKV_ERR_CORRUPT


def test_scale_byte_tampering():
    import lossless_kv_cache_fixed_gb300 as P
    spec = synth.WORKLOADS["qwen3-0.6b-bf16-drift"].scaled(name="bsg-tamper", L=1, H=1, T=256,
                                                            calib_draws=1)
    w = synth.make(spec)
    # channels 0..7 of row (kv=0, h=0): sigma near FLT_MIN and x = mu, so the
    # range check forces s = 128 and s = 18 would put sigma_eff below it
    sig = w.sigma.clone()
    sig.view(-1)[:8] = 1.2e-38
    kv = w.kv.clone()
    kv[0, 0, 0, :, :8] = w.mu[0, 0, 0, :, :8]
    w2 = synth.Workload(w.spec, kv, w.mu, sig, w.counts)
    codec = gpu_codec(w2, flags=BS)
    kv_d, mu_d = device_views(w2)
    buf, nb = codec.encode(kv_d, mu_d)
    head = 64 + 8 * (codec.n // (128 * 256) + 1)
    assert int(buf[head]) == 128
    t = buf[:nb].clone()
    t[head] = 18
    with pytest.raises(P.SkvError) as e:
        codec.decode(t, nb, mu_d)
    assert e.value.status == P.SKV_ERR_CORRUPT
    for j in range(1, 16):
        t = buf[:nb].clone()
        t[head + j] ^= 1
        try:
            out = codec.decode(t, nb, mu_d)
            assert not torch.equal(out, kv_d), j
        except P.SkvError as err:
            assert err.status == P.SKV_ERR_CORRUPT
    assert torch.equal(codec.decode(buf, nb, mu_d), kv_d)   # still usable


@pytest.mark.slow
def test_drift_fullsize_sampled(oracle_mod):
    O = oracle_mod
    w = synth.make("qwen3-0.6b-bf16-drift", device="cuda")
    s = w.spec
    codec = gpu_codec(w, flags=BS)
    kv_d = w.kv.view(torch.int16).reshape(-1)
    mu_d = w.mu.view(torch.int16).reshape(-1)
    buf, nb = codec.encode(kv_d, mu_d)
    assert torch.equal(codec.decode(buf, nb, mu_d), kv_d)
    tot, ps = codec.ideal_bits(kv_d, mu_d, per_scalar=True)
    static = gpu_codec(w)
    _, nb0 = static.encode(kv_d, mu_d)
    assert nb < 0.95 * nb0                     # the scales pay on a drifting error scale
    assert 8.0 * nb <= 1.01 * tot
    m = oracle_model(O, w, block_scale=True)
    nc = m.num_chunks()
    host = buf[:nb].cpu().numpy()
    assert O.check_header(m, host) == 0
    chunks = sorted(set(np.linspace(0, nc - 1, 24).astype(np.int64).tolist()))
    kv_h = kv_d.cpu().numpy().view(np.uint16)
    mu_h = mu_d.cpu().numpy().view(np.uint16)
    want = O.encode_chunks(m, kv_h, mu_h, chunks)
    ntb = (s.T + s.Tb - 1) // s.Tb
    for c, ww in zip(chunks, want):
        assert np.array_equal(container_chunk(host, nc, c), ww), c
        row, tb = divmod(c, ntb)
        base = row * s.T * s.D + tb * s.Tb * s.D
        n_c = min(s.Tb, s.T - tb * s.Tb) * s.D
        _, ref = O.ideal_bits(m, kv_h, mu_h, base, base + n_c, per_scalar=True)
        got = ps[base: base + n_c].double().cpu().numpy()
        assert np.all(np.abs(got - ref) <= 1e-3 * np.abs(ref) + 1e-6), c
