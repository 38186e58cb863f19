"""Pins of the oracle's alphabets, ranks and bins against independent decoders.

The oracle builds ranks by sorting its own value decoders; these tests compare
them with numpy's float ordering, torch's bf16 / e4m3 decoders and rounding,
and the OCP FP8 table in tests/golden/e4m3_values.json.
"""
import json
import os

import numpy as np
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_all_values():
    u = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        return (u << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def test_bf16_rank_is_value_order(oracle_mod):
    O = oracle_mod
    vals = _bf16_all_values()
    nan = np.isnan(vals)
    assert (~nan).sum() == O.NSYM[O.BF16] == 65282
    ranks = np.array([O.rank(O.BF16, u) for u in range(65536)])
    assert np.all(ranks[nan] == -1)
    # numpy's order, with -0 placed before +0 (IEEE totalOrder on non-NaN)
    finite_u = np.nonzero(~nan)[0]
    key = np.lexsort((-(finite_u >> 15), vals[finite_u]))
    expect = np.empty(65282, dtype=np.int64)
    expect[key] = np.arange(65282)
    assert np.array_equal(ranks[finite_u], expect)
    for r in (0, 1, 32640, 32641, 65280, 65281):
        assert O.rank(O.BF16, O.bits(O.BF16, r)) == r
    assert O.bits(O.BF16, 0) == 0xFF80 and O.bits(O.BF16, 65281) == 0x7F80
    assert O.bits(O.BF16, 32640) == 0x8000 and O.bits(O.BF16, 32641) == 0x0000


def test_bf16_bins_are_rounding_intervals(oracle_mod):
    """lo(r) is the tie point between value(r-1) and value(r) under torch's RNE."""
    O = oracle_mod
    n = 65282
    lo = np.array([O.lo(O.BF16, r) for r in range(n + 1)], dtype=np.float32)
    assert lo[0] == -np.inf and lo[1] == -np.inf
    assert lo[n - 1] == np.inf and lo[n] == np.inf
    assert lo[32641] == 0.0
    vals = np.array([O.bf16_value(O.bits(O.BF16, r)) for r in range(n)])
    inner = np.arange(2, n - 1)
    mid = (vals[inner - 1] + vals[inner]) / 2.0
    assert np.array_equal(lo[inner].astype(np.float64), mid)
    # every finite value lies in its own bin
    fin = np.setdiff1d(np.arange(1, n - 1), [32640])
    assert np.all(lo[fin] <= vals[fin]) and np.all(vals[fin] < lo[fin + 1])
    # -0 owns [-tiny, 0): numerically its value is the upper edge
    assert lo[32640] < 0.0 and lo[32641] == 0.0
    # fp32 points strictly inside (lo, hi) round to the symbol (torch RNE)
    lo_in = lo[inner]
    up = np.nextafter(lo_in, np.float32(np.inf))
    hi_in = lo[inner + 1]
    dn = np.nextafter(hi_in, np.float32(-np.inf))
    for pts in (up, dn):
        t = torch.from_numpy(pts.astype(np.float32)).to(torch.bfloat16)
        got = t.view(torch.int16).numpy().view(np.uint16)
        want = np.array([O.bits(O.BF16, r) for r in inner], dtype=np.uint16)
        ok = (got == want) | (np.abs(pts) >= 3.3895e38)  # beyond max: torch gives inf
        assert ok.all()


def test_e4m3_alphabet_matches_ocp_and_torch(oracle_mod):
    O = oracle_mod
    gold = json.load(open(os.path.join(GOLD, "e4m3_values.json")))
    for code, v in gold["values"].items():
        got = O.e4m3_value(int(code, 16))
        assert got == v and np.signbit(got) == np.signbit(v), code
    codes = torch.arange(256, dtype=torch.uint8)
    tv = codes.view(torch.float8_e4m3fn).double().numpy()
    for u in range(256):
        if u in (0x7F, 0xFF):
            assert np.isnan(tv[u]) and O.rank(O.E4M3, u) == -1
        else:
            assert O.e4m3_value(u) == tv[u]
    ranks = [O.rank(O.E4M3, u) for u in range(256) if u not in (0x7F, 0xFF)]
    assert sorted(ranks) == list(range(254))
    vals = [O.e4m3_value(O.bits(O.E4M3, r)) for r in range(254)]
    assert vals == sorted(vals)
    assert O.bits(O.E4M3, 126) == 0x80 and O.bits(O.E4M3, 127) == 0x00
    assert vals[0] == -448.0 and vals[253] == 448.0


def test_e4m3_bins_are_rounding_intervals(oracle_mod):
    O = oracle_mod
    lo = np.array([O.lo(O.E4M3, r) for r in range(255)], dtype=np.float32)
    assert lo[0] == -np.inf and lo[254] == np.inf and lo[127] == 0.0
    assert lo[1] == -432.0 and lo[253] == 432.0
    want = np.array([O.bits(O.E4M3, r) for r in range(1, 253)], dtype=np.uint8)
    for pts in (np.nextafter(lo[1:253], np.float32(np.inf)),
                np.nextafter(lo[2:254], np.float32(-np.inf))):
        t = torch.from_numpy(pts.astype(np.float32)).to(torch.float8_e4m3fn)
        got = t.view(torch.uint8).numpy()
        assert np.array_equal(got, want)
