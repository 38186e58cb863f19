"""Decode fused with its consumer (skv_decode_range; page "推测式 KV 编码无损压缩 KV
缓存最高可达约 4 倍", section "该方法的用途": caches offloaded to host memory come
back over the slow link and are decoded where they are used).

Decoding a container range by range -- from device memory, from pinned host
memory, from a device buffer whose chunk ranges are copied in just before
they are decoded, or from a container still being committed range by range
as it is encoded -- and into a paged layout must give exactly the cache the
whole-container decode gives (which the parity tests tie to the oracle).
Page-index and corruption errors surface through skv_decode_status.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import device_views, gpu_codec, skv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _chunks(spec, Tb):
    """(base, length) of every chunk in container order."""
    ntb = (spec.T + Tb - 1) // Tb
    out = []
    for row in range(spec.L * 2 * spec.H):
        for tb in range(ntb):
            out.append((row * spec.T * spec.D + tb * Tb * spec.D,
                        min(Tb, spec.T - tb * Tb) * spec.D))
    return out


def _ranges(nc, rng):
    cuts = sorted(set([0, nc] + rng.integers(0, nc + 1, 5).tolist()))
    return list(zip(cuts[:-1], cuts[1:])) + [(nc // 2, nc // 2)]   # and one empty range


CASES = [("qwen3-0.6b-bf16", 0, dict(L=1, H=2, T=600, calib_draws=2)),
         ("qwen3-8b-e4m3", 0, dict(L=2, H=1, T=300, Tb=64, G=4)),
         ("qwen3-0.6b-bf16-drift", 2, dict(L=1, H=2, T=520, calib_draws=2)),
         ("qwen3-0.6b-bf16", 4, dict(L=1, H=2, T=330, Tb=128, G=8, calib_draws=2))]


@pytest.mark.parametrize("name,flags,kw", CASES, ids=[f"{c[0]}-{c[1]}" for c in CASES])
def test_ranges_paged_hostmem_and_staged(name, flags, kw):
    spec = synth.WORKLOADS[name].scaled(name="rng-%s-%d" % (name, flags), **kw)
    w = synth.make(spec)
    s = w.spec
    codec = gpu_codec(w, flags=flags) if not flags & 4 else None
    if flags & 4:   # order-0 baseline: no mu, no sigma
        import lossless_kv_cache_fixed_gb300 as P
        E, ph = P.skv_build_ecdf(w.counts.cpu().numpy().astype(np.uint64))
        codec = P.Codec(s.dtype, s.L, s.H, s.T, s.D, s.Tb, s.G, None,
                        torch.from_numpy(E.view(np.int32)).cuda(),
                        torch.from_numpy(ph).cuda(), flags=flags)
    kv, mu = device_views(w)
    if flags & 4:
        mu = None
    buf, nb = codec.encode(kv, mu)
    buf = buf[:nb].clone()
    chunks = _chunks(s, s.Tb)
    nc = len(chunks)
    rng = np.random.default_rng(nc)
    ranges = _ranges(nc, rng)

    # 1. contiguous layout, device container, ranges in a shuffled order
    out = torch.zeros_like(kv)
    codec.decode_range(buf, nb, 0, 0, mu, out, first=True)       # prepare only
    for c0, c1 in [ranges[i] for i in rng.permutation(len(ranges))]:
        codec.decode_range(buf, nb, c0, c1, mu, out)
    codec.decode_status()
    assert torch.equal(out, kv)

    # 2. paged layout: a shuffled page table with spare pages; mu in the same pages
    P_ = s.Tb * s.D
    npages = nc + 3
    perm = rng.permutation(npages)[:nc].astype(np.uint32)
    pages = torch.from_numpy(perm.view(np.int32)).cuda()
    mu_pool = None
    if mu is not None:
        mu_pool = torch.zeros(npages * P_, dtype=mu.dtype, device="cuda")
        for c, (b, n) in enumerate(chunks):
            mu_pool[int(perm[c]) * P_: int(perm[c]) * P_ + n] = mu[b: b + n]
    pool = torch.zeros(npages * P_, dtype=kv.dtype, device="cuda")
    for i, (c0, c1) in enumerate(ranges):
        codec.decode_range(buf, nb, c0, c1, mu_pool, pool, pages, npages, first=(i == 0))
    codec.decode_status()
    for c, (b, n) in enumerate(chunks):
        assert torch.equal(pool[int(perm[c]) * P_: int(perm[c]) * P_ + n], kv[b: b + n]), c

    # 3. container in pinned host memory: the kernels read it over the link
    host = buf.cpu().pin_memory()
    out = torch.zeros_like(kv)
    for i, (c0, c1) in enumerate(ranges):
        codec.decode_range(host, nb, c0, c1, mu, out, first=(i == 0))
    codec.decode_status()
    assert torch.equal(out, kv)

    # 4. staged: a device buffer holding only the header and offsets, each range's
    #    payload copied in on a side stream just before its decode
    head = 64 + 8 * (nc + 1)
    offs = host[64:head].view(torch.int64)
    dev = torch.zeros_like(buf)
    dev[:head].copy_(host[:head])
    out = torch.zeros_like(kv)
    copy = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    codec.decode_range(dev, nb, 0, 0, mu, out, first=True)
    for c0, c1 in ranges:
        a, b = head + int(offs[c0]), head + int(offs[c1])
        with torch.cuda.stream(copy):
            dev[a:b].copy_(host[a:b], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(copy)
        main.wait_event(ev)
        codec.decode_range(dev, nb, c0, c1, mu, out)
    codec.decode_status()
    assert torch.equal(out, kv)

    # 5. committed as it is encoded: each range placed in a container still
    #    being written (skv_encode_commit) and decoded from it into the page
    #    pool (SKV_RANGE_PARTIAL) before the next range is encoded
    cont = torch.zeros(codec.max_bytes, dtype=torch.uint8, device="cuda")
    pool = torch.zeros(npages * P_, dtype=kv.dtype, device="cuda")
    cover = ranges[:-1]
    for i, (c0, c1) in enumerate(cover):
        codec.encode_range(kv, mu, c0, c1, first=(i == 0))
        codec.encode_commit(c0, c1, cont)
        codec.decode_range(cont, cont.numel(), c0, c1, mu_pool, pool, pages, npages,
                           first=(i == 0), partial=True)
    codec.decode_status()
    for c, (b, n) in enumerate(chunks):
        assert torch.equal(pool[int(perm[c]) * P_: int(perm[c]) * P_ + n], kv[b: b + n]), c
    done, nb5 = codec.encode_finish(out=cont)
    assert nb5 == nb and torch.equal(done[:nb], buf)


def test_page_errors_and_corruption_reach_the_status():
    P = skv()
    # 1 layer x {K,V} x 1 head x 2 token blocks: 4 chunks of 256 x 128 in order
    spec = synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(name="rng-err", L=1, H=1, T=512,
                                                     calib_draws=1)
    w = synth.make(spec)
    codec = gpu_codec(w)
    kv, mu = device_views(w)
    buf, nb = codec.encode(kv, mu)
    nc = 4
    P_ = 256 * 128
    perm = np.array([2, 0, 7, 1], dtype=np.uint32)       # page 7 is out of range
    pages = torch.from_numpy(perm.view(np.int32)).cuda()
    mu_pool = torch.zeros(4 * P_, dtype=mu.dtype, device="cuda")
    for c in range(nc):
        if perm[c] < 4:
            mu_pool[int(perm[c]) * P_: (int(perm[c]) + 1) * P_] = mu[c * P_: (c + 1) * P_]
    pool = torch.zeros(4 * P_, dtype=kv.dtype, device="cuda")
    codec.decode_range(buf, nb, 0, nc, mu_pool, pool, pages, 4, first=True)
    with pytest.raises(P.SkvError) as e:
        codec.decode_status()
    assert e.value.status == P.SKV_ERR_ARG
    for c in (0, 1, 3):                                   # the other chunks were decoded
        assert torch.equal(pool[int(perm[c]) * P_: (int(perm[c]) + 1) * P_],
                           kv[c * P_: (c + 1) * P_])
    # a corrupted chunk in a later range; the status stays set until the next FIRST
    t = buf[:nb].clone()
    head = 64 + 8 * (nc + 1)
    off3 = int(t[64 + 8 * 3: 64 + 8 * 4].view(torch.int64)[0])
    t[head + off3 + 40] ^= 0x55
    out = torch.zeros_like(kv)
    codec.decode_range(t, nb, 0, 2, mu, out, first=True)
    codec.decode_status()
    codec.decode_range(t, nb, 2, 4, mu, out)
    try:
        codec.decode_status()
        assert not torch.equal(out, kv)
    except P.SkvError as err:
        assert err.status == P.SKV_ERR_CORRUPT
    codec.decode_range(buf, nb, 0, nc, mu, out, first=True)
    codec.decode_status()
    assert torch.equal(out, kv)


@pytest.mark.parametrize("name,kw", [("qwen3-0.6b-bf16", dict(L=1, H=2, T=600, calib_draws=2)),
                                     ("qwen3-8b-e4m3", dict(L=2, H=1, T=300, Tb=64, G=4))])
def test_pinned_host_buffers(name, kw):
    """Pinned host memory mapped into the device's address space works wherever a
    device pointer is taken: encode reading KV and mu from host memory gives the
    same container as from device memory, ideal bits the same total, and the
    decoder writing straight into a host buffer gives the input back."""
    spec = synth.WORKLOADS[name].scaled(name="pin-" + name, **kw)
    w = synth.make(spec)
    codec = gpu_codec(w)
    kv_d, mu_d = device_views(w)
    ref, nref = codec.encode(kv_d, mu_d)
    ref = ref[:nref].clone()
    kv_h = kv_d.cpu().pin_memory()
    mu_h = mu_d.cpu().pin_memory()
    box, nb = codec.encode(kv_h, mu_h)
    assert nb == nref and torch.equal(box[:nb], ref)
    assert codec.ideal_bits(kv_h, mu_h) == codec.ideal_bits(kv_d, mu_d)
    out_h = torch.empty(kv_d.numel(), dtype=kv_d.dtype).pin_memory()
    codec.decode(box, nb, mu_d, out=out_h)
    torch.cuda.synchronize()
    assert torch.equal(out_h, kv_d.cpu())
