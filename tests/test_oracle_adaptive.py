"""Pins for the oracle's adaptive-counts coder (page "KV 缓存压缩的熵估计与动态适应",
sections "虚拟滑动窗口的设计原理" (C_t = alpha C_{t-1} + delta), "平滑更新算法"
(P_new = beta P_old + (1 - beta) P_est), "参数配置建议" (alpha 0.97, beta 0.9,
N_update 128)): an order-0 model per (layer, kv, head) row, updated after every
chunk from the row's earlier blocks, the calibration histogram as its prior.

Pinned against: a float64 exponentially weighted histogram (the counts, within
the integer truncation bound); the static prefix table (the first block);
learning on a stationary 64-symbol source whose entropy is 6 bits; adaptation
after a switch of source; round trips and model separation.
"""

import numpy as np
import pytest

import synth

BF16 = 0


def _pats_of_values(vals):
    v = np.asarray(vals, dtype=np.float32).view(np.uint32)
    return ((v + 0x7FFF + ((v >> 16) & 1)) >> 16).astype(np.uint16)


def _model(O, L, H, T, D, Tb, G, counts, adaptive=True):
    return O.Model(BF16, L, H, T, D, Tb, G, None, counts=counts, weights=(0, 0, 100),
                   adaptive=adaptive)


def _broad_counts(seed=0):
    rng = np.random.default_rng(seed)
    pats = _pats_of_values(rng.standard_normal(200000))
    return np.bincount(pats, minlength=65536).astype(np.uint64)


def _chunk_bits(O, m, buf, nc):
    head = 64 + 8 * (nc + 1)
    offs = buf[64:head].view(np.uint64)
    return np.diff(offs.astype(np.int64)) * 8


def test_first_block_is_the_static_table(oracle_mod):
    O = oracle_mod
    counts = _broad_counts()
    kv = _pats_of_values(np.random.default_rng(1).standard_normal(2 * 64 * 8)).reshape(1, 2, 1, 64, 8)
    m = _model(O, 1, 1, 64, 8, 16, 4, counts)
    E0, P0 = O.adaptive_table(m, kv, 0)
    Eq = O.build_ecdf(counts).astype(np.int64)
    assert E0[0] == 0 and E0[-1] == 1 << 26 and np.all(np.diff(E0.astype(np.int64)) >= 0)
    # P_0 = 64 (E_q[r+1] - E_q[r]): the same distribution, moved only by the add-one
    # floor's 65282 units of 2^-32 (at most 2^26 * 65282 / 2^32 ~ 1020 table units)
    assert np.max(np.abs(E0.astype(np.int64) - Eq)) <= 2 ** 26 * 65282 // 2 ** 32 + 2
    assert int(P0.sum()) == 1 << 32


def test_counts_follow_the_exponentially_weighted_histogram(oracle_mod):
    """Rebuild P_est of block 3 from a float64 weighted histogram (weights alpha^age
    in tokens) and check P_b against beta-smoothing of those estimates."""
    O = oracle_mod
    rng = np.random.default_rng(2)
    T, D, Tb = 64, 8, 16
    vals = rng.integers(0, 40, size=(2, T, D))
    pats = _pats_of_values(1.0 + vals / 64.0).reshape(1, 2, 1, T, D)
    counts = _broad_counts()
    m = _model(O, 1, 1, T, D, Tb, 2, counts)
    alpha, beta = 0.97, 0.9
    Eq = O.build_ecdf(counts).astype(np.float64)
    P = np.diff(Eq) * 64.0
    rank = np.array([O.rank(BF16, int(u)) for u in range(65536)])
    for b in range(3):
        # float64 C after block b: sum over tokens t of blocks <= b of alpha^(t_end - t)
        C = np.zeros(65282)
        t_end = (b + 1) * Tb - 1
        for t in range((b + 1) * Tb):
            np.add.at(C, rank[pats[0, 0, 0, t]], alpha ** (t_end - t))
        P = beta * P + (1 - beta) * (C / C.sum()) * 2.0 ** 32
    _, Pb = O.adaptive_table(m, pats, 3)     # chunk 3 = row 0, block 3
    Pb = Pb.astype(np.float64)
    # integer truncations: relative 1e-3 on the weights (2^16 scale), a unit per floor
    assert np.max(np.abs(Pb - P) / (P + 2 ** 20)) < 2e-3


def test_learns_a_stationary_source(oracle_mod):
    """iid symbols from 64 values (entropy 6 bits), prior from a broad N(0,1)
    histogram: static order-0 codes them far above 6 bits, the adaptive model
    comes down to about 6 after a few dozen updates."""
    O = oracle_mod
    rng = np.random.default_rng(3)
    T, D, Tb, G = 64 * 16, 8, 16, 1
    vals = 1.0 + rng.integers(0, 64, size=(2, T, D)) / 64.0
    kv = _pats_of_values(vals).reshape(1, 2, 1, T, D)
    counts = _broad_counts()
    out = {}
    for ad in (False, True):
        m = _model(O, 1, 1, T, D, Tb, G, counts, adaptive=ad)
        rc, buf = O.encode(m, kv, None)
        assert rc == 0
        rc, dec = O.decode(m, buf, None)
        assert rc == 0 and np.array_equal(dec.reshape(-1), kv.reshape(-1))
        bits = _chunk_bits(O, m, buf, m.num_chunks()) / (Tb * D)
        out[ad] = bits
    assert out[False].mean() > 9.0
    tail = out[True][48:64]               # the last quarter of row 0's blocks
    assert tail.mean() < 6.0 + 0.6, tail.mean()
    assert out[True][:4].mean() > tail.mean() + 2.0


def test_adapts_after_a_switch(oracle_mod):
    O = oracle_mod
    rng = np.random.default_rng(4)
    T, D, Tb = 64 * 16, 8, 16
    a = 1.0 + rng.integers(0, 32, size=(2, T, D)) / 64.0
    b = -2.0 - rng.integers(0, 32, size=(2, T, D)) / 32.0
    vals = np.where(np.arange(T)[None, :, None] < T // 2, a, b)
    kv = _pats_of_values(vals).reshape(1, 2, 1, T, D)
    m = _model(O, 1, 1, T, D, Tb, 1, _broad_counts())
    rc, buf = O.encode(m, kv, None)
    assert rc == 0
    bits = _chunk_bits(O, m, buf, m.num_chunks())[:64] / (Tb * D)
    before, after_switch, settled = bits[24:32].mean(), bits[32:34].mean(), bits[56:64].mean()
    assert after_switch > before + 2.0        # the old model no longer fits
    assert settled < before + 0.5             # and the new source is learnt


@pytest.mark.parametrize("G,Tb,T", [(1, 16, 37), (4, 32, 130), (16, 128, 300)])
def test_round_trip_ragged_and_separation(oracle_mod, G, Tb, T):
    O = oracle_mod
    spec = synth.WORKLOADS["tiny-bf16"].scaled(name="ad-rt", L=1, H=1, T=T, Tb=Tb, G=G)
    w = synth.make(spec)
    kv, _, _, counts = synth.to_numpy(w)
    m = _model(O, 1, 1, T, spec.D, Tb, G, counts)
    rc, buf = O.encode(m, kv, None)
    assert rc == 0 and int(buf[38]) | int(buf[39]) << 8 == 2 | 4
    rc, dec = O.decode(m, buf, None)
    assert rc == 0 and np.array_equal(dec.reshape(-1), kv.reshape(-1))
    static = _model(O, 1, 1, T, spec.D, Tb, G, counts, adaptive=False)
    assert O.decode(static, buf, None)[0] == O.ERR_CORRUPT
    tot, ps = O.ideal_bits(m, kv, None, 0, kv.size, per_scalar=True)
    assert np.all(ps > 0) and abs(ps.sum() - tot) < 1e-6 * tot
    # e4m3 and the predictive mixture do not take the flag
    bad = O.Model(BF16, 1, 1, T, spec.D, Tb, G, np.ones(2 * spec.D, np.float32), counts=counts,
                  adaptive=True)
    assert O.encode(bad, kv, np.zeros(kv.size, np.uint16))[0] == O.ERR_ARG
