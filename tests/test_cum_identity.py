"""The bf16 cum quotient in the kernels (skv_model.cuh, cum_bf16) is the high
word of F * M, M = ceil(K 2^38 / 100), in place of floor(K F / (100 2^26)).
Checked here on the host, exactly: the constant, the error bound against the
spacing of the quotient's fractional parts over the whole range of F, and the
two floors on random and extreme F (the GPU parity tests then compare every
coded byte with the oracle, which divides)."""
import math
import os
import random
import re
from fractions import Fraction

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
K = (1 << 28) - 65282           # 2^M - |S| for bf16
D = 100 << 26                   # the mixture weights' 100 times Phi_q's 2^26
F_MAX = 100 << 26               # 95 Phi_q + 3 Phi_q + 2 E_q, each at most 2^26


def _magic():
    src = open(os.path.join(ROOT, "lossless_kv_cache_fixed_gb300", "csrc", "skv_model.cuh")).read()
    return int(re.search(r"kCumMagicBf16\s*=\s*(\d+)ull", src).group(1))


def test_constant_is_the_rounded_up_ratio():
    M = _magic()
    assert M == -(-(K << 38) // 100)
    assert M < 1 << 64


def test_error_bound_below_the_fraction_spacing():
    M = _magic()
    delta = M - Fraction(K << 38, 100)          # M exceeds K 2^38 / 100 by delta in [0, 1)
    assert 0 <= delta < 1
    worst = F_MAX * delta / Fraction(1 << 64)   # F M / 2^64 - K F / D, at most
    spacing = Fraction(math.gcd(K, D), D)       # fractional parts of K F / D are multiples of it
    assert worst < spacing


def test_floors_agree_on_random_and_extreme_values():
    M = _magic()
    rng = random.Random(3)
    values = [0, 1, 2, 3, F_MAX, F_MAX - 1, F_MAX - 2] + [rng.randrange(F_MAX + 1)
                                                          for _ in range(200000)]
    # just below every multiple of D / gcd where the floor steps
    step = D // math.gcd(K, D)
    values += [q * step - 1 for q in range(1, F_MAX // step + 1, max(1, F_MAX // step // 5000))]
    for F in values:
        assert (F * M) >> 64 == (K * F) // D, F
