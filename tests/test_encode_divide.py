"""The bf16 encoder's exact division (skv_model.cuh, divmod_u64 for M = 28),
emulated on the host in IEEE fp32 with numpy: floor(x / f) and x mod f for
x < f 2^35, 1 <= f <= 2^28, from a first estimate fl(x) rf and one rounded
refinement.  The reciprocal is the hardware's approximate one, within 1 ulp of
1/fl(f); every case here runs with the correctly rounded reciprocal and with
its two neighbours, and must come out exact with at most one fix-up step (the
bound the kernel's comment derives).  The GPU parity tests then compare every
coded byte with the oracle, which divides exactly."""
import numpy as np

M = 28
QMAX = 1 << (63 - M)


def _emulate(x, f, rf):
    """The kernel's steps; x, f int64 arrays, rf float32 array."""
    two32 = np.float32(4294967296.0)
    xh = (x >> 32).astype(np.uint32).astype(np.float32)
    xl = (x & 0xFFFFFFFF).astype(np.uint32).astype(np.float32)
    xf = (xh * two32 + xl).astype(np.float32)      # xh 2^32 exact: one rounding, as fmaf
    qf = (xf * rf).astype(np.float32)
    v = np.floor((qf * np.float32(0.125)).astype(np.float64))
    q = np.minimum(v, 2.0 ** 32 - 1).astype(np.int64) << 3   # float -> u32, toward zero, saturating
    r = x - q * f
    rh = (r >> 24).astype(np.int32).astype(np.float32)
    rlo = (r & 0xFFFFFF).astype(np.uint32).astype(np.float32)
    rl = (rh * np.float32(16777216.0) + rlo).astype(np.float32)
    d = np.rint((rl * rf).astype(np.float32)).astype(np.int64)  # to nearest, ties to even
    q = q + d
    r = r - d * f
    return q, r


def _cases():
    rng = np.random.default_rng(11)
    f = np.concatenate([
        np.array([1, 2, 3, 5, 7, 255, 65535, 65537, (1 << 24) - 1, 1 << 24, (1 << 24) + 1,
                  (1 << 28) - 1, 1 << 28], dtype=np.int64),
        rng.integers(1, 1 << 28, 4000, dtype=np.int64),
        (2.0 ** rng.uniform(0, 28, 4000)).astype(np.int64).clip(1, 1 << 28),
    ])
    xs, fs = [], []
    for fv in f:
        hi = int(fv) * QMAX                      # x < f 2^35 <= 2^63
        cand = [0, 1, int(fv) - 1, int(fv), hi - 1, hi - int(fv), hi // 2, (1 << 31),
                (1 << 32) - 1, 1 << 32]
        cand += [int(v) for v in rng.integers(0, hi, 40, dtype=np.uint64)]
        # near multiples of f, where the floor steps
        for qv in rng.integers(0, QMAX, 8):
            for dv in (-1, 0, 1):
                cand.append(int(qv) * int(fv) + dv)
        cand = [c for c in cand if 0 <= c < hi]
        xs += cand
        fs += [int(fv)] * len(cand)
    return np.array(xs, dtype=np.int64), np.array(fs, dtype=np.int64)


def test_division_is_exact_with_one_fixup_at_most():
    x, f = _cases()
    ff = f.astype(np.float32)                          # (float)f, rounded to nearest
    r0 = (np.float32(1.0) / ff).astype(np.float32)     # the correctly rounded reciprocal
    want_q = x // f
    want_r = x % f
    for rf in (r0, np.nextafter(r0, np.float32(0)), np.nextafter(r0, np.float32(np.inf))):
        q, r = _emulate(x, f, rf.astype(np.float32))
        # the estimate lands within (-0.505 f, 0.505 f) of the remainder
        assert np.all(np.abs(r.astype(np.float64)) < 0.505 * f.astype(np.float64))
        neg = r < 0
        q = np.where(neg, q - 1, q)
        r = np.where(neg, r + f, r)
        assert np.array_equal(q, want_q)
        assert np.array_equal(r, want_r)
    assert len(x) > 300000
