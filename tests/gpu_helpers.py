"""Shared set-up for the GPU tests: one synthetic workload, fed identically to the
CUDA library (through the C ABI) and to the oracle."""
import numpy as np
import torch

import synth


def skv():
    import lossless_kv_cache_fixed_gb300 as P
    P.build()
    return P


def gpu_codec(w: synth.Workload, Tb=None, G=None, flags=0):
    P = skv()
    s = w.spec
    dev = torch.device("cuda")
    ecdf = phat = None
    if s.dtype == synth.BF16:
        E, ph = P.skv_build_ecdf(w.counts.cpu().numpy().astype(np.uint64))
        ecdf = torch.from_numpy(E.view(np.int32)).to(dev)
        phat = torch.from_numpy(ph).to(dev)
    return P.Codec(s.dtype, s.L, s.H, s.T, s.D, Tb or s.Tb, G or s.G, w.sigma.to(dev), ecdf, phat,
                   flags=flags)


def oracle_model(O, w: synth.Workload, Tb=None, G=None, block_scale=False):
    s = w.spec
    sigma = w.sigma.cpu().numpy().astype(np.float32)
    counts = None if w.counts is None else w.counts.cpu().numpy().astype(np.uint64)
    return O.Model(s.dtype, s.L, s.H, s.T, s.D, Tb or s.Tb, G or s.G, sigma, counts=counts,
                   block_scale=block_scale)


def host_views(w: synth.Workload):
    kv, mu, _, _ = synth.to_numpy(w)
    return kv.reshape(-1), mu.reshape(-1)


def device_views(w: synth.Workload):
    dev = torch.device("cuda")
    if w.spec.dtype == synth.BF16:
        kv = w.kv.view(torch.int16).to(dev).reshape(-1)
    else:
        kv = w.kv.to(dev).reshape(-1)
    mu = w.mu.view(torch.int16).to(dev).reshape(-1)
    return kv, mu


def container_chunk(buf_host: np.ndarray, nchunks: int, c: int) -> np.ndarray:
    head = 64 + 8 * (nchunks + 1)
    offs = buf_host[64:head].view(np.uint64)
    return buf_host[head + int(offs[c]): head + int(offs[c + 1])].view(np.uint32)


def check_model_bits(O, codec, m, kv_d, mu_d, kv, mu, container):
    """skv_model_bits against the oracle chunk by chunk, and the rANS length
    invariant on the GPU's own container: every chunk's payload exceeds its
    model bits by 32 to 64 bits per lane (initial state and flush)."""
    tot, ps = codec.model_bits(kv_d, mu_d, per_scalar=True)
    ps = ps.double().cpu().numpy()
    assert abs(tot - ps.sum()) <= 1e-6 * abs(tot) + 1e-3
    L, _, H, T, D = m.shape
    Tb, G = m.s.Tb, m.s.G
    ntb = (T + Tb - 1) // Tb
    nc = m.num_chunks()
    head = 64 + 8 * (nc + 1)
    offs = container[64:head].view(np.uint64)
    ref_tot = 0.0
    for c in range(nc):
        row, tb = divmod(c, ntb)
        base = row * T * D + tb * Tb * D
        n_c = min(Tb, T - tb * Tb) * D
        ref = O.model_bits_chunk(m, kv, mu, c)
        ref_tot += ref
        got = ps[base:base + n_c].sum()
        assert abs(got - ref) <= 1e-5 * ref + 1e-3, c
        payload_bits = 8.0 * (int(offs[c + 1]) - int(offs[c]))
        nsw = (D // 8 + 3) // 4 if m.s.block_scale else 0
        extra = payload_bits - 32 * nsw - ref
        assert 32 * G - 1e-3 * ref - 1 <= extra <= 64 * G + 1e-3 * ref + 1, c
    assert abs(tot - ref_tot) <= 1e-6 * ref_tot + 1e-3


def check_encode_with_bits(codec, kv_d, mu_d, container, ref, ref_tot, rtol=1e-3, atol=1e-6):
    """skv_encode_with_bits writes the container skv_encode writes, per-scalar
    ideal bits within the tolerance of the oracle's (ref), a total that agrees
    with them, and the same total on a second call (fixed summation order)."""
    import numpy as np
    buf, nb, tot, ps = codec.encode_with_bits(kv_d, mu_d, per_scalar=True)
    assert nb == container.size and np.array_equal(buf[:nb].cpu().numpy(), container)
    got = ps.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= rtol * np.abs(ref) + atol)
    assert abs(tot - got.sum()) <= 1e-6 * abs(tot) + 1e-6
    assert abs(tot - ref_tot) <= rtol * abs(ref_tot) + 1e-6
    _, nb2, tot2 = codec.encode_with_bits(kv_d, mu_d)
    assert nb2 == nb and tot2 == tot
