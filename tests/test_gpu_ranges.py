"""Encoding by chunk ranges, and one container from per-range parts, on the GPU
through the C ABI.

* skv_encode_range over a shuffled cover of the chunks (one stream, or two
  streams after the first range) then skv_encode_finish writes exactly the
  container of skv_encode and of the oracle;
* a chunk left out or coded twice is refused by skv_encode_finish before any
  stack is read, and a bad symbol in one range is reported there;
* skv_model_fingerprint equals the oracle's model fingerprint;
* containers of consecutive layer ranges, each encoded on the GPU with its
  rows of sigma, merge (skv_merge_parts, host) into the whole container;
* ranges committed as they are encoded (skv_encode_commit) build the same
  container, and each committed range decodes before the rest is encoded;
  commits out of order, of chunks not yet encoded, of a prefix only, or past
  the buffer's capacity are reported by skv_encode_finish.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import device_views, gpu_codec, host_views, oracle_model

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


CASES = {
    "bf16": synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(name="ranges-bf16", L=3, H=2, T=600,
                                                       calib_draws=2),
    "e4m3": synth.WORKLOADS["qwen3-8b-e4m3"].scaled(name="ranges-e4m3", L=3, H=2, T=600),
}


def _cover(nc, rng, pieces):
    cuts = sorted(set([0, nc] + rng.choice(np.arange(1, nc), pieces - 1, replace=False).tolist()))
    ranges = list(zip(cuts[:-1], cuts[1:]))
    first = ranges[0]
    rest = ranges[1:]
    rng.shuffle(rest)
    return [first] + rest


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
@pytest.mark.parametrize("flags", [0, 2], ids=["static", "block-scale"])
def test_ranges_write_the_container(oracle_mod, kind, flags):
    import lossless_kv_cache_fixed_gb300 as P
    w = synth.make(CASES[kind])
    codec = gpu_codec(w, flags=flags)
    kv_d, mu_d = device_views(w)
    whole, nb = codec.encode(kv_d, mu_d)
    whole = whole[:nb].clone()
    m = oracle_model(oracle_mod, w, block_scale=bool(flags & P.SKV_FLAG_BLOCK_SCALE))
    kv_h, mu_h = host_views(w)
    rc, want = oracle_mod.encode(m, kv_h, mu_h)
    assert rc == 0 and np.array_equal(whole.cpu().numpy(), want)
    nc = codec.num_chunks()
    rng = np.random.default_rng(7 + flags)
    for pieces in (2, 5, nc):
        ranges = _cover(nc, rng, pieces)
        for i, (a, b) in enumerate(ranges):
            codec.encode_range(kv_d, mu_d, a, b, first=(i == 0))
        out, nb2 = codec.encode_finish()
        assert nb2 == nb and torch.equal(out[:nb2], whole)
    # two streams after the first range: the later ranges may run side by side
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ranges = _cover(nc, rng, 6)
    codec.encode_range(kv_d, mu_d, *ranges[0], first=True)
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(ranges[1:]):
        codec.encode_range(kv_d, mu_d, a, b, stream=s1 if i % 2 else s2)
    torch.cuda.synchronize()
    out, nb2 = codec.encode_finish()
    assert nb2 == nb and torch.equal(out[:nb2], whole)


def test_finish_refuses_a_wrong_cover():
    import lossless_kv_cache_fixed_gb300 as P
    w = synth.make(CASES["bf16"])
    codec = gpu_codec(w)
    kv_d, mu_d = device_views(w)
    nc = codec.num_chunks()
    out = torch.empty(codec.max_bytes, dtype=torch.uint8, device="cuda")
    ws = codec.workspace(P.SKV_OP_ENCODE)
    st = P._stream_handle()

    def finish():
        return P.skv_encode_finish(codec.params, codec.shape, out.data_ptr(), out.numel(),
                                   ws.data_ptr(), ws.numel(), st)[0]

    # one chunk missing
    codec.encode_range(kv_d, mu_d, 0, nc // 2, first=True)
    codec.encode_range(kv_d, mu_d, nc // 2 + 1, nc)
    assert finish() == P.SKV_ERR_ARG
    # one chunk twice
    codec.encode_range(kv_d, mu_d, 0, nc // 2 + 1, first=True)
    codec.encode_range(kv_d, mu_d, nc // 2, nc)
    assert finish() == P.SKV_ERR_ARG
    # arguments checked at once
    assert P.skv_encode_range(codec.params, codec.shape, kv_d.data_ptr(), mu_d.data_ptr(), 3, 2,
                              0, ws.data_ptr(), ws.numel(), st) == P.SKV_ERR_ARG
    assert P.skv_encode_range(codec.params, codec.shape, kv_d.data_ptr(), mu_d.data_ptr(), 0,
                              nc + 1, 0, ws.data_ptr(), ws.numel(), st) == P.SKV_ERR_ARG
    # a NaN symbol in the second range is reported by the finish
    bad = kv_d.clone()
    bad[-5] = 0x7FC1
    codec.encode_range(bad, mu_d, 0, nc // 2, first=True)
    codec.encode_range(bad, mu_d, nc // 2, nc)
    assert finish() == P.SKV_ERR_SYMBOL
    # and a clean cover still works afterwards
    codec.encode_range(kv_d, mu_d, 0, nc, first=True)
    o2, nb = codec.encode_finish()
    ref, nb_ref = codec.encode(kv_d, mu_d)
    assert nb == nb_ref and torch.equal(o2[:nb], ref[:nb_ref])


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_fingerprint_matches_oracle(oracle_mod, kind):
    w = synth.make(CASES[kind])
    codec = gpu_codec(w)
    assert codec.fingerprint() == oracle_mod.model_hash(oracle_model(oracle_mod, w))


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_gpu_parts_merge_into_the_whole_container(kind):
    import lossless_kv_cache_fixed_gb300 as P
    spec = CASES[kind]
    w = synth.make(spec)
    codec = gpu_codec(w)
    kv_d, mu_d = device_views(w)
    whole, nb = codec.encode(kv_d, mu_d)
    want = whole[:nb].cpu().numpy()
    parts = []
    for l0, l1 in ((0, 1), (1, 3)):
        part = synth.make(spec, layers=(l0, l1))
        pc = gpu_codec(part)
        pk, pm = device_views(part)
        buf, pnb = pc.encode(pk, pm)
        parts.append(buf[:pnb].cpu().numpy())
    out = np.zeros(nb, dtype=np.uint8)
    rc, nb2 = P.skv_merge_parts(codec.params, codec.shape, codec.fingerprint(), parts, out)
    assert rc == P.SKV_OK and nb2 == nb and np.array_equal(out, want)


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
@pytest.mark.parametrize("flags", [0, 2], ids=["static", "block-scale"])
def test_commits_build_the_container_and_decode_early(oracle_mod, kind, flags):
    """Chunk ranges encoded in order, each committed right after (or several at
    once), give the oracle's container (the one skv_encode writes); every
    committed range decodes (SKV_RANGE_PARTIAL) before the later ones are
    encoded."""
    import lossless_kv_cache_fixed_gb300 as P
    w = synth.make(CASES[kind])
    codec = gpu_codec(w, flags=flags)
    kv_d, mu_d = device_views(w)
    whole, nb = codec.encode(kv_d, mu_d)
    whole = whole[:nb].clone()
    m = oracle_model(oracle_mod, w, block_scale=bool(flags & P.SKV_FLAG_BLOCK_SCALE))
    kv_h, mu_h = host_views(w)
    rc, want = oracle_mod.encode(m, kv_h, mu_h)
    assert rc == 0 and np.array_equal(whole.cpu().numpy(), want)
    nc = codec.num_chunks()
    rng = np.random.default_rng(11 + flags)
    for pieces, batch in ((1, 1), (3, 1), (7, 2), (nc, 5)):
        cuts = sorted(set([0, nc] + rng.choice(np.arange(1, nc), pieces - 1, replace=False).tolist()))
        out = torch.zeros(codec.max_bytes, dtype=torch.uint8, device="cuda")
        dec = torch.zeros_like(kv_d)
        ends = torch.zeros(nc + 1, dtype=torch.int64).pin_memory()  # written by the device
        done, ncommit = 0, 0
        for i, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
            codec.encode_range(kv_d, mu_d, a, b, first=(i == 0))
            if (i + 1) % batch == 0 or b == nc:
                codec.encode_commit(done, b, out, end_bytes=ends[ncommit:ncommit + 1])
                codec.decode_range(out, out.numel(), done, b, mu_d, dec, first=(done == 0),
                                   partial=True)
                done, ncommit = b, ncommit + 1
        codec.decode_status()
        assert torch.equal(dec, kv_d)
        out2, nb2 = codec.encode_finish(out=out)
        assert nb2 == nb and torch.equal(out2[:nb2], whole)
        # the sizes so far: increasing, the last one the container's
        e = ends[:ncommit].tolist()
        assert e == sorted(e) and e[-1] == nb
        # the finished container passes the full header check
        assert torch.equal(codec.decode(out2, nb2, mu_d), kv_d)


def test_commit_errors_are_reported_by_finish():
    import lossless_kv_cache_fixed_gb300 as P
    w = synth.make(CASES["bf16"])
    codec = gpu_codec(w)
    kv_d, mu_d = device_views(w)
    nc = codec.num_chunks()
    h = nc // 2
    out = torch.zeros(codec.max_bytes, dtype=torch.uint8, device="cuda")

    def finish_rc(buf=out):
        ws = codec.workspace(P.SKV_OP_ENCODE)
        rc, _ = P.skv_encode_finish(codec.params, codec.shape, buf.data_ptr(), buf.numel(),
                                    ws.data_ptr(), ws.numel(), P._stream_handle())
        return rc

    # a range that does not start where the committed prefix ends
    codec.encode_range(kv_d, mu_d, 0, nc, first=True)
    codec.encode_commit(h, nc, out)
    assert finish_rc() == P.SKV_ERR_ARG
    # a chunk committed before it was encoded (its start is still the sentinel)
    codec.encode_range(kv_d, mu_d, 0, h, first=True)
    codec.encode_commit(0, h + 1, out)
    codec.encode_range(kv_d, mu_d, h, nc)
    assert finish_rc() == P.SKV_ERR_ARG
    # only a prefix committed
    codec.encode_range(kv_d, mu_d, 0, nc, first=True)
    codec.encode_commit(0, h, out)
    assert finish_rc() == P.SKV_ERR_ARG
    # a buffer with room for the offset table but not for the payload
    small = torch.zeros(64 + 8 * (nc + 1) + 4096, dtype=torch.uint8, device="cuda")
    codec.encode_range(kv_d, mu_d, 0, nc, first=True)
    codec.encode_commit(0, nc, small)
    assert finish_rc(small) == P.SKV_ERR_CAPACITY
    # and a clean run afterwards
    codec.encode_range(kv_d, mu_d, 0, nc, first=True)
    codec.encode_commit(0, h, out)
    codec.encode_commit(h, nc, out)
    o2, nb = codec.encode_finish(out=out)
    ref, nb_ref = codec.encode(kv_d, mu_d)
    assert nb == nb_ref and torch.equal(o2[:nb], ref[:nb_ref])


def _scalar_base(spec, c):
    """First scalar of chunk c in the [L][2][H][T][D] tensor (chunks of
    consecutive indices are consecutive in memory: the last chunk's end is n)."""
    ntb = (spec.T + spec.Tb - 1) // spec.Tb
    row, tb = divmod(c, ntb)
    return row * spec.T * spec.D + min(tb * spec.Tb, spec.T) * spec.D


@pytest.mark.parametrize("flags", [0, 2], ids=["static", "block-scale"])
@pytest.mark.parametrize("size", ["small", "multi-round"])
def test_ranges_with_their_ideal_bits(oracle_mod, size, flags):
    """SKV_RANGE_BITS: a cover of the cache in pieces, all but one encoded with
    their ideal bits inside the encoder, gives skv_encode's container, and the
    running total equals the oracle's ideal bits over the flagged pieces'
    scalars (the per-scalar tolerance of the ideal bits) and the GPU's own
    ideal-bits pass over them; the same sequence gives the same total again.
    'small': ranges of one round of tasks or less; 'multi-round': 8,192 chunks
    of 16 lanes (2 layers x 8 heads x 4090 tokens x 64, 16-token blocks, the
    last ragged), where the pieces run several rounds; with the model's sigma
    or per-block scales."""
    if size == "small":
        spec = CASES["bf16"]
    else:
        spec = synth.WORKLOADS["qwen3-0.6b-bf16"].scaled(name="range-bits", L=2, H=8, T=4090,
                                                         D=64, Tb=16, G=16, calib_draws=2)
    w = synth.make(spec)
    codec = gpu_codec(w, flags=flags)
    kv_d, mu_d = device_views(w)
    whole, nb = codec.encode(kv_d, mu_d)
    whole = whole[:nb].clone()
    m = oracle_model(oracle_mod, w, block_scale=bool(flags))
    kv_h, mu_h = host_views(w)
    _, ref = oracle_mod.ideal_bits(m, kv_h, mu_h, per_scalar=True)
    _, gps = codec.ideal_bits(kv_d, mu_d, per_scalar=True)
    gps = gps.double().cpu().numpy()
    nc = codec.num_chunks()
    rng = np.random.default_rng(17)
    ranges = _cover(nc, rng, 5)
    skip = 2                                   # this piece is encoded without its bits
    totals = []
    for _ in range(2):
        for i, (a, b) in enumerate(ranges):
            codec.encode_range(kv_d, mu_d, a, b, first=(i == 0), bits=(i != skip))
        totals.append(codec.encode_range_bits())
        out, nb2 = codec.encode_finish()
        assert nb2 == nb and torch.equal(out[:nb2], whole)
    assert totals[0] == totals[1]
    sel = np.zeros(spec.n, dtype=bool)
    for i, (a, b) in enumerate(ranges):
        if i != skip:
            sel[_scalar_base(spec, a):_scalar_base(spec, b)] = True
    want = ref[sel].sum()
    assert abs(totals[0] - want) <= 1e-3 * abs(want) + 1e-6
    assert abs(totals[0] - gps[sel].sum()) <= 1e-5 * abs(want) + 1e-6
    # a fresh FIRST range clears the total
    codec.encode_range(kv_d, mu_d, 0, nc, first=True)
    assert codec.encode_range_bits() == 0.0
