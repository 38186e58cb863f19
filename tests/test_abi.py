"""The C-ABI library without a GPU: it loads, exports every symbol declared in
include/skv.h, its host-side helpers agree bit for bit with the oracle, and
argument errors are reported before any device work."""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def skv():
    import lossless_kv_cache_fixed_gb300 as P
    P.build()
    return P


def _declared():
    src = open(os.path.join(ROOT, "include", "skv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(skv_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(skv):
    lib = skv.lib()
    names = _declared()
    assert set(names) == set(skv.EXPORTS)
    for name in names:
        assert hasattr(lib, name), name
    assert skv.skv_version() == 1
    assert skv.skv_strerror(skv.SKV_ERR_CORRUPT).startswith("corrupt")


def test_phi_table_matches_oracle_and_exact_rounding(skv, oracle_mod):
    mpmath = pytest.importorskip("mpmath")
    T = skv.skv_phi_table()
    assert np.array_equal(T, oracle_mod.phi_table())
    mp = mpmath.mp
    mp.dps = 40
    for i in list(range(1, 8192, 37)) + [1, 3382, 4095, 4096, 4097, 8191]:
        v = mp.ncdf(mp.mpf(-8) + mp.mpf(i) / 512) * 2 ** 26
        assert int(T[i]) == int(mp.nint(v)), i


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_build_ecdf_matches_oracle(skv, oracle_mod, seed):
    rng = np.random.default_rng(seed)
    if seed == 0:
        counts = np.zeros(65536, dtype=np.uint64)
    elif seed == 1:
        counts = rng.integers(0, 1 << 20, 65536).astype(np.uint64)
    else:
        counts = np.minimum(rng.pareto(0.5, 65536) * 1e3, 1e6).astype(np.uint64)
        counts[0x3F80] = 1 << 35
    E, ph = skv.skv_build_ecdf(counts)
    assert np.array_equal(E, oracle_mod.build_ecdf(counts))
    pat = np.array([oracle_mod.bits(0, r) for r in range(65282)])
    cnt = counts[pat].astype(np.float64) + 1
    np.testing.assert_allclose(ph, cnt / cnt.sum(), rtol=1e-6)


def test_build_ecdf_rejects_huge_totals(skv):
    counts = np.zeros(65536, dtype=np.uint64)
    counts[0] = 1 << 40
    with pytest.raises(skv.SkvError):
        skv.skv_build_ecdf(counts)


def test_argument_errors_without_gpu(skv):
    P = skv
    good = P.SkvParams(P.SKV_BF16, 256, 8, 0, 1 << 20, 1 << 21, None)
    shape = P.SkvShape(2, 2, 2, 256, 64)
    assert P.skv_max_encoded_bytes(good, shape) == 64 + 8 * 9 + 4 * (131072 + 2 * 8 * 8)
    assert P.skv_workspace_bytes(good, shape, P.SKV_OP_ENCODE) > 0
    assert P.skv_workspace_bytes(good, shape, 7) == 0
    for bad_shape in [P.SkvShape(2, 3, 2, 256, 64), P.SkvShape(2, 2, 2, 256, 60),
                      P.SkvShape(0, 2, 2, 256, 64), P.SkvShape(2, 2, 2, -1, 64)]:
        assert P.skv_max_encoded_bytes(good, bad_shape) == 0
    for bad in [P.SkvParams(P.SKV_BF16, 256, 3, 0, 1, 1, None),
                P.SkvParams(P.SKV_BF16, 256, 64, 0, 1, 1, None),
                P.SkvParams(P.SKV_BF16, 0, 8, 0, 1, 1, None),
                P.SkvParams(5, 256, 8, 0, 1, 1, None),
                P.SkvParams(P.SKV_BF16, 256, 8, 8, 1, 1, None)]:
        assert P.skv_max_encoded_bytes(bad, shape) == 0
        rc, _ = P.skv_encode(bad, shape, 1 << 20, 1 << 20, 1 << 20, 1 << 30, 1 << 20, 1 << 30, None)
        assert rc == P.SKV_ERR_ARG
    # per-block scales: ceil(head_dim / 32) more words per chunk, head_dim <= 2048,
    # and no fixed-scratch ideal bits
    scaled = P.SkvParams(P.SKV_BF16, 256, 8, P.SKV_FLAG_BLOCK_SCALE, 1 << 20, 1 << 21, 1 << 22)
    assert P.skv_max_encoded_bytes(scaled, shape) == 64 + 8 * 9 + 4 * (131072 + (2 * 8 + 2) * 8)
    assert (P.skv_workspace_bytes(scaled, shape, P.SKV_OP_ENCODE)
            > P.skv_workspace_bytes(good, shape, P.SKV_OP_ENCODE))
    assert P.skv_max_encoded_bytes(scaled, P.SkvShape(1, 2, 1, 4, 2048)) > 0
    assert P.skv_max_encoded_bytes(scaled, P.SkvShape(1, 2, 1, 4, 2056)) == 0
    rc, _ = P.skv_ideal_bits_noalloc(scaled, shape, 1 << 20, 1 << 20, None, None)
    assert rc == P.SKV_ERR_ARG
    # the order-0 baseline: bf16 only, not with block scales, no fixed-scratch ideal bits
    o0 = P.SkvParams(P.SKV_BF16, 256, 8, P.SKV_FLAG_ORDER0, None, 1 << 21, 1 << 22)
    assert P.skv_max_encoded_bytes(o0, shape) == P.skv_max_encoded_bytes(good, shape)
    for f, dt in ((P.SKV_FLAG_ORDER0, P.SKV_E4M3),
                  (P.SKV_FLAG_ORDER0 | P.SKV_FLAG_BLOCK_SCALE, P.SKV_BF16), (8, P.SKV_BF16)):
        assert P.skv_max_encoded_bytes(P.SkvParams(dt, 256, 8, f, 1, 1, 1), shape) == 0
    rc, _ = P.skv_ideal_bits_noalloc(o0, shape, 1 << 20, None, None, None)
    assert rc == P.SKV_ERR_ARG
    rc, _ = P.skv_encode(o0, shape, None, None, 1 << 20, 1 << 30, 1 << 20, 1 << 30, None)
    assert rc == P.SKV_ERR_ARG                       # kv is still required
    # adaptive counts: only with the order-0 coder, head_dim <= 512, whole containers
    ad = P.SkvParams(P.SKV_BF16, 256, 8, P.SKV_FLAG_ORDER0 | P.SKV_FLAG_ADAPTIVE, None, 1 << 21,
                     1 << 22)
    assert P.skv_max_encoded_bytes(ad, shape) > 0
    assert (P.skv_workspace_bytes(ad, shape, P.SKV_OP_DECODE)
            > P.skv_workspace_bytes(o0, shape, P.SKV_OP_DECODE))
    assert P.skv_max_encoded_bytes(P.SkvParams(P.SKV_BF16, 256, 8, P.SKV_FLAG_ADAPTIVE, 1, 1, 1),
                                   shape) == 0
    assert P.skv_max_encoded_bytes(ad, P.SkvShape(1, 2, 1, 4, 520)) == 0
    rc = P.skv_decode_range(ad, shape, 1 << 20, 1 << 20, 0, 8, None, 1 << 20, None, 0, 1,
                            1 << 20, 1 << 30, None)
    assert rc == P.SKV_ERR_ARG
    # range decode: range, flags and page-table arguments are checked on the host
    for c0, c1, fl, pages, npg in ((5, 4, 1, None, 0), (0, 9, 1, None, 0), (0, 8, 4, None, 0),
                                   (0, 8, 1, 1 << 20, 0), (0, 8, 1, (1 << 20) + 2, 8)):
        rc = P.skv_decode_range(good, shape, 1 << 20, 1 << 20, c0, c1, 1 << 20, 1 << 20, pages,
                                npg, fl, 1 << 20, 1 << 30, None)
        assert rc == P.SKV_ERR_ARG, (c0, c1, fl, pages, npg)
    assert P.skv_decode_status(None, None) == P.SKV_ERR_ARG
    # commits: range, buffer alignment and room for the offset table, on the host
    for c0, c1, out, cap in ((5, 4, 1 << 20, 1 << 30), (0, 9, 1 << 20, 1 << 30),
                             (0, 8, (1 << 20) + 4, 1 << 30)):
        assert P.skv_encode_commit(good, shape, c0, c1, out, cap, None, 1 << 20, 1 << 30,
                                   None) == P.SKV_ERR_ARG, (c0, c1, out, cap)
    assert P.skv_encode_commit(good, shape, 0, 8, 1 << 20, 64 + 8 * 8, None, 1 << 20, 1 << 30,
                               None) == P.SKV_ERR_CAPACITY
    assert P.skv_encode_commit(good, shape, 0, 8, 1 << 20, 1 << 30, (1 << 20) + 4, 1 << 20,
                               1 << 30, None) == P.SKV_ERR_ARG   # end_bytes misaligned
    assert P.skv_encode_commit(good, shape, 3, 3, 1 << 20, 1 << 30, None, 1 << 20, 1 << 30,
                               None) == P.SKV_OK           # an empty range places nothing
    assert P.skv_encode_commit(ad, shape, 0, 8, 1 << 20, 1 << 30, None, 1 << 20, 1 << 30,
                               None) == P.SKV_ERR_ARG      # adaptive counts: whole caches
    # ranges with their ideal bits: the bf16 mixture coder with p-hat only
    with_phat = P.SkvParams(P.SKV_BF16, 256, 8, 0, 1 << 20, 1 << 21, 1 << 22)
    for prm in (P.SkvParams(P.SKV_E4M3, 256, 8, 0, 1 << 20, None, None), good,
                P.SkvParams(P.SKV_BF16, 256, 8, P.SKV_FLAG_ORDER0, None, 1 << 21, 1 << 22)):
        assert P.skv_encode_range(prm, shape, 1 << 20, 1 << 20, 0, 8,
                                  P.SKV_RANGE_FIRST | P.SKV_RANGE_BITS, 1 << 20, 1 << 30,
                                  None) == P.SKV_ERR_ARG
    assert P.skv_encode_range(with_phat, shape, 1 << 20, 1 << 20, 0, 8, 8, 1 << 20, 1 << 30,
                              None) == P.SKV_ERR_ARG     # an unknown flag
    assert P.skv_encode_range(with_phat, shape, 1 << 20, 1 << 20, 0, 8, P.SKV_RANGE_BITS,
                              1 << 20, 16, None) == P.SKV_ERR_CAPACITY
    assert P.skv_encode_range_bits(with_phat, shape, 1 << 20, 16, None)[0] == P.SKV_ERR_CAPACITY
    assert P.skv_encode_range_bits(with_phat, shape, (1 << 20) + 8, 1 << 30,
                                   None)[0] == P.SKV_ERR_ARG   # workspace misaligned
    # NULL and misaligned pointers
    rc, _ = P.skv_encode(good, shape, None, 1 << 20, 1 << 20, 1 << 30, 1 << 20, 1 << 30, None)
    assert rc == P.SKV_ERR_ARG
    rc, _ = P.skv_encode(good, shape, (1 << 20) + 2, 1 << 20, 1 << 20, 1 << 30, 1 << 20, 1 << 30,
                         None)
    assert rc == P.SKV_ERR_ARG
    no_ecdf = P.SkvParams(P.SKV_BF16, 256, 8, 0, 1 << 20, None, None)
    rc, _ = P.skv_encode(no_ecdf, shape, 1 << 20, 1 << 20, 1 << 20, 1 << 30, 1 << 20, 1 << 30, None)
    assert rc == P.SKV_ERR_ARG
    # ideal bits on bf16 needs p-hat
    rc, _ = P.skv_ideal_bits(good, shape, 1 << 20, 1 << 20, None, 1 << 20, 1 << 30, None)
    assert rc == P.SKV_ERR_ARG
    # workspace too small
    rc, _ = P.skv_encode(good, shape, 1 << 20, 1 << 20, 1 << 20, 1 << 30, 1 << 20, 16, None)
    assert rc == P.SKV_ERR_CAPACITY
    # a container shorter than its own offset table
    rc = P.skv_decode(good, shape, 1 << 20, 100, 1 << 20, 1 << 20, 1 << 20, 1 << 30, None)
    assert rc == P.SKV_ERR_CORRUPT


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "lossless_kv_cache_fixed_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in txt and "skv_oracle" not in txt, f
