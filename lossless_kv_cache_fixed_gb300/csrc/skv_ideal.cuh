// skv_ideal.cuh -- ideal code length -log2 q(x) of one scalar in fp32, shared by
// the ideal-bits kernel and the encoder that reports the ideal code length as
// it codes.
//
// Page "推测式 KV 编码无损压缩 KV 缓存最高可达约 4 倍" (Speculative KV coding),
// section "KV 缓存并非真正随机": the cost of a scalar is -log2 q(x), q the model's
// mass on the symbol's bin; section "早期结果" gives q for bf16 (the 0.95 / 0.03
// / 0.02 mixture), section "原生 FP8 KV 缓存" the bin-integrated N(mu, sigma^2)
// for e4m3.  The evaluation cases and their error bounds are described where
// each function is defined.
#pragma once
#include <cstdint>

#include "skv_internal.h"
#include "skv_model.cuh"

namespace skv {
namespace ideal {

__device__ __forceinline__ float log_upper_tail(float z) {
  if (z == INFINITY) return -INFINITY;
  if (z == -INFINITY) return 0.0f;
  if (z < 0.0f) return log1pf(-0.5f * erfcf(-z * 0.70710678f));
  return logf(0.5f * erfcxf(z * 0.70710678f)) - 0.5f * z * z;
}

constexpr float kLog2e = 1.44269504f;
constexpr float kLog2Sqrt2Pi = 1.32574806f;  // log2 sqrt(2 pi)

// The mass on the far side of mu in the natural-log domain, for wide bins and
// outliers; kept out of line so that the common path stays small.
static __device__ __noinline__ float log2_gauss_tail(float lo, float hi, float mu, float inv_s) {
  const float za = (lo - mu) * inv_s, zb = (hi - mu) * inv_s;
  float ln;
  if (za >= 0.0f) {
    const float a = log_upper_tail(za), b = log_upper_tail(zb);
    ln = a + logf(-expm1f(b - a));
  } else if (zb <= 0.0f) {
    const float a = log_upper_tail(-zb), b = log_upper_tail(-za);
    ln = a + logf(-expm1f(b - a));
  } else {
    const float qa = isfinite(za) ? 0.5f * erfcf(-za * 0.70710678f) : 0.0f;
    const float qb = isfinite(zb) ? 0.5f * erfcf(zb * 0.70710678f) : 0.0f;
    ln = log1pf(-(qa + qb));
  }
  return ln * kLog2e;
}

// log2 of the N(mu, s^2) mass on [lo, hi) by the midpoint rule, for bins with
// w max(1, |zm|) < 0.5 (else ok = false and 0): w phi(zm) (1 + y),
// y = He2 w^2/24 + He4 w^4/1920 + He6 w^6/322560 (He_n the probabilists'
// Hermite polynomials), the logarithm of 1 + y by its series (|y| < 0.02).
__device__ __forceinline__ float log2_gauss_series(float lo, float hi, float mu, float inv_s,
                                                   float log2_s, bool &ok) {
  ok = true;
  if (!(hi > lo)) return -INFINITY;
  if (isfinite(lo) && isfinite(hi)) {
    const float width = hi - lo;
    const float w = width * inv_s;
    const float zm = (lo + 0.5f * width - mu) * inv_s;
    if (w * fmaxf(1.0f, fabsf(zm)) < 0.5f) {
      const float z2 = zm * zm, w2 = w * w;
      const float he2 = z2 - 1.0f, he4 = fmaf(z2, z2 - 6.0f, 3.0f);
      const float he6 = fmaf(z2, fmaf(z2, z2 - 15.0f, 45.0f), -15.0f);
      const float y = w2 * fmaf(w2, fmaf(w2, he6 * (1.0f / 322560.0f), he4 * (1.0f / 1920.0f)),
                                he2 * (1.0f / 24.0f));
      const float l1p = y * fmaf(y, fmaf(y, 1.0f / 3.0f, -0.5f), 1.0f);
      return fmaf(-0.5f * kLog2e, z2, -kLog2Sqrt2Pi) + (__log2f(width) - log2_s) + l1p * kLog2e;
    }
  }
  ok = false;
  return 0.0f;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Q(z) for z >= 0 from the table, 0 from z = 12 on (Q(12) < 1.8e-33).  log2 Q is
// linear between knots 1/256 apart; its second derivative, -h (h - z) / ln 2
// with h = phi / Q, is below 1 / ln 2 in magnitude, so the interpolation error
// is below 1.45 / (8 256^2) = 2.8e-6 in log2.  With the fp32 rounding of the
// knots (up to 4e-6 at z = 9, where log2 Q = -63) and of ex2.approx, Q carries
// at most 5e-6 relative error below z = 9 (2e-6 below z = 3).
__device__ __forceinline__ float q_tab(float z, const float2 *__restrict__ log2q) {
  if (!(z < 12.0f)) return 0.0f;
  const float t = z * (float)kTailPerUnit;
  const int k = (int)t;
  const float2 e = __ldg(log2q + k);
  return ex2_approx(fmaf(t - (float)k, e.y, e.x));
}

// N(mu, s^2) mass on [lo, hi) as Q(a) - Q(b), Q(z) = erfc(z / sqrt 2) / 2 the
// upper tail, with the bin mirrored when it lies below mu so that a < b and a
// is the edge on the far side of mu (both of a straddling bin's edges: Q(a)
// near 1 then carries absolute error only).  On the bf16 bins outside the
// series case (w >= 1 or w |zm| >= 2) Q(a) / Q(b) >= e^0.5, so the difference
// keeps the relative accuracy of erfcf.  `far` receives a (deep tails: a >= 9).
__device__ __forceinline__ float gauss_mass(float lo, float hi, float mu, float inv_s, float &far) {
  const float za = (lo - mu) * inv_s, zb = (hi - mu) * inv_s;
  const bool below = zb <= 0.0f;
  const float a = below ? -zb : za, b = below ? -za : zb;
  far = a;
  return 0.5f * (erfcf(a * 0.70710678f) - erfcf(b * 0.70710678f));
}

// bf16, the series case w < 1 and w |zm| < 2, |zm| < 64 (then w/3 and zm/3 qualify for
// the 3 sigma component too): the mixture in the linear domain, each component
// w phi(zm) (1 + y) with the Hermite correction y of log2_gauss_series, then
// one logarithm.  The first dropped term, He8 w^8 / 92897280, is at most
// 132 / 92897280 (|zm| <= 1, w < 1) or about 2^8 / 92897280 (w |zm| < 2), both
// below 3e-6 relative.  A Gaussian term too small for fp32 only drops below the
// p-hat term's 0.02 p-hat floor.  Returns false (and nothing) when the bin
// needs the tail evaluation.
__device__ __forceinline__ bool ideal_series_bf16(float lo, float hi, float mu, float inv_s,
                                                  float ph, float &bits) {
  if (!(hi > lo) || !isfinite(lo) || !isfinite(hi)) return false;
  const float width = hi - lo;
  const float w = width * inv_s;
  const float zm = (lo + 0.5f * width - mu) * inv_s;
  if (!(w < 1.0f)) return false;
  if (!(fabsf(zm) < 64.0f)) {
    // a narrow bin beyond 63.5 sigma (or whose centre's distance from mu
    // overflows fp32): the 3-sigma component's mass is below 1e-98 and the
    // narrow one's below that, under 1e-85 of p-hat's 0.02 floor (p-hat >=
    // 2^-37), so q is that floor; the series below would compute 0 * inf there
    bits = -__log2f(0.02f * ph);
    return true;
  }
  if (!(w * fabsf(zm) < 2.0f)) return false;
  auto comp =[](float w, float zm) {
    const float z2 = zm * zm, w2 = w * w;
    const float he2 = z2 - 1.0f, he4 = fmaf(z2, z2 - 6.0f, 3.0f);
    const float he6 = fmaf(z2, fmaf(z2, z2 - 15.0f, 45.0f), -15.0f);
    const float y = w2 * fmaf(w2, fmaf(w2, he6 * (1.0f / 322560.0f), he4 * (1.0f / 1920.0f)),
                              he2 * (1.0f / 24.0f));
    return w * 0.39894228f * __expf(-0.5f * z2) * (1.0f + y);  // w phi(zm) (1 + y)
  };
  // the 3 sigma component has w/3 < 1/3 and (w/3) |zm/3| < 2/9, where its He4
  // and He6 terms stay below 1.9e-5 and 6e-8 relative: He2 alone
  const float w3 = w * (1.0f / 3.0f), z3 = zm * (1.0f / 3.0f);
  const float z32 = z3 * z3, w32 = w3 * w3;
  const float c3 = w3 * 0.39894228f * __expf(-0.5f * z32) *
                   fmaf(w32 * (1.0f / 24.0f), z32 - 1.0f, 1.0f);
  const float q = fmaf(0.95f, comp(w, zm), fmaf(0.03f, c3, 0.02f * ph));
  bits = -__log2f(q);
  return true;
}

// -log2 q of one scalar.  FULL = false evaluates only the common cases (bf16:
// the series; e4m3: the tail table) and sets `deferred` when the scalar needs
// the rest.
// inv_s = 1 / sigma (any rounding within an ulp or two); log2q: the tail table
// (g_log2q of skv_bits.cu), read for e4m3 only.
// e4m3 common case, bins at least 0.01 sigma wide whose near edge lies within
// 9 sigma (all but about 1.3% of a cache): the mass from the tail table,
// Q(a) - Q(b) for a bin on one side of mu (mirrored below it) and
// 1 - Q(-a) - Q(b) for a bin around mu, so the error scales with the tails.
// With epsilon <= 5e-6 per tail, a one-sided bin's mass is off by at most
// epsilon (Q(a) + Q(b)) / (Q(a) - Q(b)) <= 250 epsilon relative (w = 0.01 at
// a = 0, where such a bin costs 8 bits: 2e-3 bits of a 8e-3 tolerance), a bin
// around mu's by epsilon (1 - m) absolute.  Returns false (and nothing) for
// the rest.
__device__ __forceinline__ bool ideal_table_e4m3(float lo, float hi, float mu, float inv_s,
                                                 const float2 *__restrict__ log2q, float &bits) {
  const float wz = (hi - lo) * inv_s;
  const float za = (lo - mu) * inv_s, zb = (hi - mu) * inv_s;
  const bool below = zb <= 0.0f;
  const float a = below ? -zb : za, b = below ? -za : zb;
  if (!(wz >= 0.01f && a < 9.0f)) return false;
  const float m = a >= 0.0f ? q_tab(a, log2q) - q_tab(b, log2q)
                            : 1.0f - q_tab(-a, log2q) - q_tab(b, log2q);
  bits = -__log2f(m);
  return true;
}

// The full evaluation of a bin [lo, hi) with p-hat mass ph (bf16; unused for
// e4m3).  bf16: the mixture in the linear domain, each component's mass a
// difference of erfc tails on the far side of mu (p-hat's 0.02 floor keeps q
// normal, so a Gaussian mass below fp32's range does not matter).  e4m3: one
// branch-free difference of erfc tails for every bin but the deep tails (log
// domain) and bins under 1e-3 sigma wide (the series, where the difference
// would cancel); the difference's relative error, about 6e-8 / (a w), is
// below 1e-4 of the mass from w = 1e-3 on.
template <int DT>
__device__ __forceinline__ float ideal_full(float lo, float hi, float mu, float inv_s, float ph) {
  if (DT == 0) {
    float far;
    const float m1 = hi > lo ? gauss_mass(lo, hi, mu, inv_s, far) : 0.0f;
    const float m3 = hi > lo ? gauss_mass(lo, hi, mu, inv_s * (1.0f / 3.0f), far) : 0.0f;
    return -log2f(fmaf(0.95f, fmaxf(m1, 0.0f), fmaf(0.03f, fmaxf(m3, 0.0f), 0.02f * ph)));
  }
  const float wz = (hi - lo) * inv_s;
  bool ok = false;
  float l1 = 0.0f;
  if (wz < 1e-3f) l1 = log2_gauss_series(lo, hi, mu, inv_s, -__log2f(inv_s), ok);
  if (!ok) {
    float far;
    const float m = hi > lo ? gauss_mass(lo, hi, mu, inv_s, far) : 0.0f;
    l1 = (far < 9.0f && m > 0.0f) ? log2f(m) : log2_gauss_tail(lo, hi, mu, inv_s);
  }
  return -l1;
}

// bf16 bins outside the series case, from the tail table: each component's
// mass Q(a) - Q(b) on one side of mu (mirrored below it), 1 - Q(-a) - Q(b)
// around it.  Such a bin has w >= 1 or w |zm| >= 2, so on one side Q(a) / Q(b)
// >= e^0.5 for the sigma component, and the 3-sigma one has w |zm| / 9 >=
// 2 / 9: with epsilon <= 5e-6 per tail below z = 9 the masses keep about
// 10 epsilon relative error; a bin around mu is at least 1 sigma wide, its
// mass at least 0.38.  Beyond z = 9 a Gaussian mass is below 1.2e-19, under
// 1e-6 of p-hat's 0.02 floor (p-hat >= 2^-37), so the table's coarser values
// there (0 from z = 12) do not matter.
__device__ __forceinline__ float mass_tab(float lo, float hi, float mu, float inv_s,
                                          const float2 *__restrict__ log2q) {
  const float za = (lo - mu) * inv_s, zb = (hi - mu) * inv_s;
  if (za >= 0.0f) return q_tab(za, log2q) - q_tab(zb, log2q);
  if (zb <= 0.0f) return q_tab(-zb, log2q) - q_tab(-za, log2q);
  return 1.0f - q_tab(-za, log2q) - q_tab(zb, log2q);
}

__device__ __forceinline__ float ideal_rare_bf16(float lo, float hi, float mu, float inv_s,
                                                 float ph, const float2 *__restrict__ log2q) {
  float m1 = 0.0f, m3 = 0.0f;
  if (hi > lo) {
    m1 = fmaxf(mass_tab(lo, hi, mu, inv_s, log2q), 0.0f);
    m3 = fmaxf(mass_tab(lo, hi, mu, inv_s * (1.0f / 3.0f), log2q), 0.0f);
  }
  return -__log2f(fmaf(0.95f, m1, fmaf(0.03f, m3, 0.02f * ph)));
}

// -log2 q of one scalar (its symbol and mu's bf16 bits), inv_s = 1 / sigma
// (any rounding within an ulp or two); log2q: the tail table (g_log2q of
// skv_bits.cu), read for e4m3 only.  FULL = false evaluates only the common
// cases (bf16: the series; e4m3: the tail table) and sets `deferred` when the
// scalar needs the full evaluation.
template <int DT, bool FULL>
__device__ __forceinline__ float ideal_one(uint32_t sym, uint32_t mu_bits, float inv_s,
                                           const float *phat, const float *lo8,
                                           const float2 *__restrict__ log2q, uint32_t &flags,
                                           bool &deferred) {
  const int32_t NS = DT == 0 ? kNsymBf16 : kNsymE4m3;
  int32_t r = DT == 0 ? rank_bf16(sym) : rank_e4m3(sym);
  if (r < 0 || r >= NS) {
    flags |= kFlagSymbol;
    return 0.0f;
  }
  if (!mu_valid(mu_bits)) {
    flags |= kFlagParam;
    return 0.0f;
  }
  const float mu = bf16_to_f32(mu_bits);
  const float lo = DT == 0 ? lo_bf16(r) : lo8[r];
  const float hi = DT == 0 ? lo_bf16(r + 1) : lo8[r + 1];
  const float ph = DT == 0 ? phat[r] : 0.0f;
  if (!FULL) {
    float bits;
    const bool ok = DT == 0 ? ideal_series_bf16(lo, hi, mu, inv_s, ph, bits)
                            : ideal_table_e4m3(lo, hi, mu, inv_s, log2q, bits);
    if (ok) return bits;
    deferred = true;
    return 0.0f;
  }
  return ideal_full<DT>(lo, hi, mu, inv_s, ph);
}

}  // namespace ideal
}  // namespace skv
