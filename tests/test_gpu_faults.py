"""Fault injection on the GPU path, made on the host (no GPU fault is ever
provoked): corrupted, truncated or mismatched containers and invalid inputs
must come back as an error status -- or, for a payload bit flip that still
decodes cleanly, as different data -- and the library must stay usable.

Every read of the decoder is bounded by its chunk's extent and every wait is
absent by construction, so none of these cases can fault or hang.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import device_views, gpu_codec, oracle_model

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture(scope="module")
def enc():
    import lossless_kv_cache_fixed_gb300 as P
    spec = synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(name="faults", L=1, H=2, T=512,
                                                     calib_draws=2)
    w = synth.make(spec)
    codec = gpu_codec(w)
    kv, mu = device_views(w)
    buf, nb = codec.encode(kv, mu)
    return P, w, codec, kv, mu, buf[:nb].clone(), nb


def _decode_rc(P, codec, buf, nb, mu, stream=None):
    out = torch.empty(codec.n, dtype=torch.int16, device="cuda")
    ws = codec.workspace(P.SKV_OP_DECODE)
    rc = P.skv_decode(codec.params, codec.shape, buf.data_ptr(), nb, mu.data_ptr(),
                      out.data_ptr(), ws.data_ptr(), ws.numel(), P._stream_handle(stream))
    return rc, out


def test_clean_roundtrip_then_library_still_usable(enc):
    P, w, codec, kv, mu, buf, nb = enc
    rc, out = _decode_rc(P, codec, buf, nb, mu)
    assert rc == P.SKV_OK and torch.equal(out, kv)


def test_payload_bit_flips(enc):
    P, w, codec, kv, mu, buf, nb = enc
    nc = codec.n // (codec.shape.head_dim * codec.params.token_block)
    head = 64 + 8 * (nc + 1)
    rng = np.random.default_rng(0)
    for _ in range(40):
        t = buf.clone()
        pos = int(rng.integers(head, nb))
        t[pos] ^= 1 << int(rng.integers(0, 8))
        rc, out = _decode_rc(P, codec, t, nb, mu)
        # a clean finish on a changed stream would be a different cache
        assert rc == P.SKV_ERR_CORRUPT or (rc == P.SKV_OK and not torch.equal(out, kv))
    test_clean_roundtrip_then_library_still_usable(enc)


def test_truncated_and_padded(enc):
    P, w, codec, kv, mu, buf, nb = enc
    for cut in (4, 64, 1000, nb // 2):
        rc, _ = _decode_rc(P, codec, buf, nb - cut, mu)
        assert rc == P.SKV_ERR_CORRUPT, cut
    longer = torch.cat([buf, torch.zeros(16, dtype=torch.uint8, device="cuda")])
    rc, _ = _decode_rc(P, codec, longer, nb + 16, mu)
    assert rc == P.SKV_ERR_CORRUPT
    rc, _ = _decode_rc(P, codec, buf, 10, mu)
    assert rc == P.SKV_ERR_CORRUPT


def test_header_and_offset_tampering(enc):
    P, w, codec, kv, mu, buf, nb = enc
    for off in (0, 4, 6, 7, 8, 16, 20, 24, 28, 32, 40, 48, 56, 63):
        t = buf.clone()
        t[off] ^= 0x10
        assert _decode_rc(P, codec, t, nb, mu)[0] == P.SKV_ERR_CORRUPT, off
    # offsets: point a chunk past the payload, make one decrease, misalign one
    for j, val in ((3, 1 << 40), (5, 4), (7, None)):
        t = buf.clone()
        o = t[64:64 + 8 * 16].view(torch.int64)
        o[j] = val if val is not None else o[j] + 2
        assert _decode_rc(P, codec, t, nb, mu)[0] == P.SKV_ERR_CORRUPT, j
    # every offset shifted by 2: all differences stay multiples of 4, but no
    # chunk starts on a word boundary (the decoder must not read misaligned)
    nc = codec.n // (codec.shape.head_dim * codec.params.token_block)
    t = buf.clone()
    o = t[64:64 + 8 * (nc + 1)].view(torch.int64)
    o[:nc] += 2
    assert _decode_rc(P, codec, t, nb, mu)[0] == P.SKV_ERR_CORRUPT


def test_model_mismatch(enc, oracle_mod):
    P, w, codec, kv, mu, buf, nb = enc
    # one sigma one ulp off: the fingerprint in the header no longer matches
    sig = w.sigma.clone()
    sig.view(-1)[3] = torch.nextafter(sig.view(-1)[3], torch.tensor(10.0))
    w2 = synth.Workload(w.spec, w.kv, w.mu, sig, w.counts)
    rc, _ = _decode_rc(P, gpu_codec(w2), buf, nb, mu)
    assert rc == P.SKV_ERR_CORRUPT
    # a different p-hat table
    cnt = w.counts.clone()
    cnt[0x3F80] += 1000
    w3 = synth.Workload(w.spec, w.kv, w.mu, w.sigma, cnt)
    rc, _ = _decode_rc(P, gpu_codec(w3), buf, nb, mu)
    assert rc == P.SKV_ERR_CORRUPT
    # mu off by one ulp somewhere: the decoder must do exactly what the oracle
    # does with the same wrong mu (an error, or the same different cache),
    # and never fault
    O = oracle_mod
    m = oracle_model(O, w)
    kv_h = kv.cpu().numpy().view(np.uint16)
    for pos in (1234, 77777):
        mu2 = mu.clone()
        mu2[pos] ^= 1
        rc, out = _decode_rc(P, codec, buf, nb, mu2)
        rc_o, out_o = O.decode(m, buf.cpu().numpy(), mu2.cpu().numpy().view(np.uint16))
        assert rc == rc_o and rc in (P.SKV_OK, P.SKV_ERR_CORRUPT)
        # the model at that scalar's true symbol changed, so a clean decode
        # cannot return the input
        sym = int(kv_h[pos])
        r = O.rank(0, sym)
        row = pos // (w.spec.T * w.spec.D) * w.spec.D + pos % w.spec.D
        sg = float(w.sigma.reshape(-1)[row])
        mu_a = O.bf16_value(int(mu[pos].item()) & 0xFFFF)
        mu_b = O.bf16_value(int(mu2[pos].item()) & 0xFFFF)
        changed = (O.cum(m, r, mu_a, sg), O.cum(m, r + 1, mu_a, sg)) != (
            O.cum(m, r, mu_b, sg), O.cum(m, r + 1, mu_b, sg))
        if rc == P.SKV_OK:
            out_h = out.cpu().numpy().view(np.uint16)
            assert np.array_equal(out_h, out_o)
            if changed:
                assert not np.array_equal(out_h, kv_h)
    test_clean_roundtrip_then_library_still_usable(enc)


def test_invalid_inputs(enc):
    P, w, codec, kv, mu, buf, nb = enc
    bad = kv.clone()
    bad[77] = 0x7FC1                          # a NaN pattern
    with pytest.raises(P.SkvError) as e:
        codec.encode(bad, mu)
    assert e.value.status == P.SKV_ERR_SYMBOL
    badmu = mu.clone()
    badmu[5] = 0x7F80                         # mu = +inf
    with pytest.raises(P.SkvError) as e:
        codec.encode(kv, badmu)
    assert e.value.status == P.SKV_ERR_PARAM
    for v in (0.0, float("nan"), float("inf"), -1.0, 1e-39):
        sig = w.sigma.clone()
        sig.view(-1)[0] = v
        c2 = gpu_codec(synth.Workload(w.spec, w.kv, w.mu, sig, w.counts))
        with pytest.raises(P.SkvError) as e:
            c2.encode(kv, mu)
        assert e.value.status == P.SKV_ERR_PARAM, v
    # too small an output buffer
    small = torch.empty(nb - 100, dtype=torch.uint8, device="cuda")
    with pytest.raises(P.SkvError) as e:
        codec.encode(kv, mu, out=small)
    assert e.value.status == P.SKV_ERR_CAPACITY
    # a p-hat prefix table that is not non-decreasing
    import lossless_kv_cache_fixed_gb300 as PP
    E, ph = PP.skv_build_ecdf(w.counts.cpu().numpy().astype(np.uint64))
    E[1000], E[1001] = E[1001] + 5, E[1000]
    c3 = PP.Codec(w.spec.dtype, w.spec.L, w.spec.H, w.spec.T, w.spec.D, w.spec.Tb, w.spec.G,
                  w.sigma.cuda(), torch.from_numpy(E.view(np.int32)).cuda(),
                  torch.from_numpy(ph).cuda())
    with pytest.raises(P.SkvError) as e:
        c3.encode(kv, mu)
    assert e.value.status == P.SKV_ERR_PARAM
    test_clean_roundtrip_then_library_still_usable(enc)


def test_encode_with_bits_reports_data_errors(enc):
    """skv_encode_with_bits inside the encoder (bf16: this small cache, one
    round of tasks, and one of several rounds) and on the two-pass path
    (e4m3) reports a NaN symbol, an infinite mu and a short output buffer
    like skv_encode, and the library stays usable."""
    P, w, codec, kv, mu, buf, nb = enc
    big_spec = synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(name="fused-faults", L=2, H=8, T=4096,
                                                         D=64, Tb=16, G=16, calib_draws=2)
    big = synth.make(big_spec)
    bcodec = gpu_codec(big)
    bkv = big.kv.view(torch.int16).reshape(-1).cuda()
    bmu = big.mu.view(torch.int16).reshape(-1).cuda()
    e8 = synth.make(synth.WORKLOADS["qwen3-8b-e4m3"].scaled(name="faults-e4m3", L=1, H=2, T=512))
    ecodec = gpu_codec(e8)
    ekv, emu = device_views(e8)
    assert codec.encode_with_bits_fused() and bcodec.encode_with_bits_fused()
    assert not ecodec.encode_with_bits_fused()
    for c, k, m, nan in ((codec, kv, mu, 0x7FC1), (bcodec, bkv, bmu, 0x7FC1),
                         (ecodec, ekv, emu, 0x7F)):
        bad = k.clone()
        bad[77] = nan                             # a NaN pattern
        with pytest.raises(P.SkvError) as e:
            c.encode_with_bits(bad, m)
        assert e.value.status == P.SKV_ERR_SYMBOL
        badmu = m.clone()
        badmu[5] = 0x7F80                         # mu = +inf
        with pytest.raises(P.SkvError) as e:
            c.encode_with_bits(k, badmu)
        assert e.value.status == P.SKV_ERR_PARAM
        _, n_ok = c.encode(k, m)
        small = torch.empty(n_ok - 100, dtype=torch.uint8, device="cuda")
        with pytest.raises(P.SkvError) as e:
            c.encode_with_bits(k, m, out=small)
        assert e.value.status == P.SKV_ERR_CAPACITY
        out, n2, tot = c.encode_with_bits(k, m)
        assert n2 == n_ok and tot > 0
    test_clean_roundtrip_then_library_still_usable(enc)
