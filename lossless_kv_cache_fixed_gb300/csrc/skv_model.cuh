// skv_model.cuh -- the fixed-point probability model on the device.
//
// Page "推测式 KV 编码无损压缩 KV 缓存最高可达约 4 倍" (Speculative KV coding):
//   section "q 应是什么样的": Gaussian q(x) = N(x; mu, sigma^2) around the
//     per-scalar prediction;
//   section "早期结果": bf16 symbols use 0.95 N(mu, sigma^2) + 0.03 N(mu, (3 sigma)^2)
//     + 0.02 p-hat_bf16;
//   section "原生 FP8 KV 缓存": e4m3 symbols use the bin-integrated N(mu, sigma^2);
//   section "下一步计划": both ends must obtain bit-identical probabilities.
//
// Every function below is exact integer or IEEE round-to-nearest fp32
// arithmetic through explicit intrinsics (never contracted into FMAs), so the
// frequencies are the same on every GPU and on any IEEE CPU.
#pragma once
#include <cstdint>

namespace skv {

constexpr int kNsymBf16 = 65282;            // non-NaN bf16 patterns
constexpr int kNsymE4m3 = 254;              // non-NaN e4m3 codes
constexpr uint32_t kPhiOne = 1u << 26;      // Phi_q scale
constexpr int kPhiKnots = 8193;             // z = -8 + i/512, i = 0..8192
constexpr uint64_t kStateL = 1ull << 31;    // rANS lower bound
constexpr int kMBf16 = 28, kME4m3 = 16;     // frequency precision
constexpr uint32_t kKBf16 = (1u << 28) - kNsymBf16;  // 2^M - |S|
constexpr uint32_t kKE4m3 = (1u << 16) - kNsymE4m3;

// ---- symbol <-> rank (monotone value order, -0 before +0) ----

// bf16: the IEEE totalOrder key of a pattern is (u | 0x8000) for a clear sign
// bit and (~u & 0xFFFF) otherwise; the 127 NaNs below -inf are skipped.
// Valid iff 0 <= result < kNsymBf16.
__device__ __forceinline__ int32_t rank_bf16(uint32_t u) {
  uint32_t key = (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u);
  return (int32_t)key - 127;
}

__device__ __forceinline__ uint32_t bits_bf16(int32_t r) {
  uint32_t key = (uint32_t)(r + 127);
  return (key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu);
}

// e4m3: magnitude 0x7F is NaN; negatives are ranks 0..126 (-448 .. -0).
__device__ __forceinline__ int32_t rank_e4m3(uint32_t u) {
  uint32_t mag = u & 0x7Fu;
  int32_t r = (u & 0x80u) ? 126 - (int32_t)mag : 127 + (int32_t)mag;
  return mag == 0x7Fu ? -1 : r;
}

__device__ __forceinline__ uint32_t bits_e4m3(int32_t r) {
  return r >= 127 ? (uint32_t)(r - 127) : (0x80u | (uint32_t)(126 - r));
}

// Lower edge of bf16 symbol r's round-to-nearest bin, as fp32 bits.  The edge
// between two neighbours is their midpoint: the smaller magnitude's pattern
// followed by a half-ulp bit.  With k = r - rank(+0) and a = |k|, the edge's
// magnitude bits are (a << 16) - 0x8000 (0 for a = 0: -0 | +0 split at 0) and
// its sign is k's; a >= 32640 gives infinity, so ranks 0, 1 (-inf, -max) start
// at -inf and ranks 65281, 65282 (+inf, end) at +inf.
__device__ __forceinline__ float lo_bf16(int32_t r) {
  const int32_t k = r - 32641;
  const int32_t a = abs(k);
  const uint32_t mag = a >= 32640 ? 0x7F800000u : (uint32_t)max(a * 65536 - 0x8000, 0);
  return __uint_as_float(mag | ((uint32_t)k & 0x80000000u));
}

// ---- Phi_q: 2^26 Phi(z) by integer interpolation of the knot table ----
// With t = 512 z: Phi_q = 0 for t <= -4096, 2^26 for t >= 4096, else
// T[i] + ((T[i+1] - T[i]) fr >> 16) with i = floor(t) + 4096 and
// fr = floor(65536 (t - floor t)).  Both come out of one integer,
// q = floor(2^25 z) = 65536 floor(t) + fr: i = (q >> 16) + 4096, fr = q & 0xFFFF.
// 2^25 z is an exact scaling (or +-inf, which the clamps map to the ends).
// `phi` holds (T[i], (T[i+1] - T[i]) << 16) pairs (the step is below 2^16);
// the last pair is (2^26, 0).  ((T[i+1] - T[i]) fr) >> 16 is then the high
// word of ((T[i+1] - T[i]) << 16) * fr.
__device__ __forceinline__ uint32_t phi_q(float z, const uint2 *phi) {
  int32_t q = __float2int_rd(__fmul_rn(z, 33554432.0f));
  q = max(q, -(1 << 28));
  q = min(q, 1 << 28);
  const uint2 e = phi[(q >> 16) + 4096];
  return e.x + __umulhi(e.y, (uint32_t)q & 0xFFFFu);
}

// Per-channel reciprocals: IEEE round-to-nearest 1/sigma and 1/(3 sigma).
struct ChanInv {
  float s, s3;
};

__device__ __forceinline__ bool sigma_valid(float s) {
  // finite and >= FLT_MIN, with 3 sigma finite (NaN fails the first test)
  return s >= 1.17549435e-38f && __fmul_rn(3.0f, s) <= 3.40282347e38f;
}

__device__ __forceinline__ ChanInv chan_inv(float sigma) {
  ChanInv c;
  c.s = __frcp_rn(sigma);
  c.s3 = __frcp_rn(__fmul_rn(3.0f, sigma));
  return c;
}

// cum(r) for bf16: floor(K (95 Phi_q(z1) + 3 Phi_q(z3) + 2 E_q[r]) / (100 2^26)) + r,
// z1 = (lo - mu) / sigma, z3 = (lo - mu) / (3 sigma), each product rounded.
// The quotient is the high word of F M with M = ceil(K 2^38 / 100): F M / 2^64
// exceeds K F / (100 2^26) by F (M - K 2^38 / 100) / 2^64 <= 0.44 F / 2^64 <=
// 1.6e-10 (F <= 100 2^26), less than the 2 / (100 2^26) = 3.0e-10 spacing of
// that quotient's fractional parts (gcd(K, 100 2^26) = 2), so the floor is the
// same for every F: one 64-bit multiply-high in place of the multiply by K,
// the shift and the division by 100.
constexpr uint64_t kCumMagicBf16 = 737690317153170883ull;  // ceil(K 2^38 / 100)
__device__ __forceinline__ uint32_t cum_bf16(int32_t r, float mu, ChanInv inv, const uint2 *phi,
                                             const uint32_t *__restrict__ ecdf) {
  float d = __fsub_rn(lo_bf16(r), mu);
  uint32_t p1 = phi_q(__fmul_rn(d, inv.s), phi);
  uint32_t p3 = phi_q(__fmul_rn(d, inv.s3), phi);
  uint32_t e = __ldg(ecdf + r);
  uint64_t F = 95ull * p1 + 3ull * p3 + 2ull * e;
  return (uint32_t)__umul64hi(F, kCumMagicBf16) + (uint32_t)r;
}

// cum(r) for e4m3: floor(K Phi_q(z1) / 2^26) + r; K Phi_q / 2^26 =
// (Phi_q K 2^6) / 2^32 exactly, one multiply-high (Phi_q <= 2^26, K 2^6 < 2^23).
__device__ __forceinline__ uint32_t cum_e4m3(int32_t r, float mu, float inv_s, const uint2 *phi,
                                             const float *lo8) {
  float d = __fsub_rn(lo8[r], mu);
  uint32_t p = phi_q(__fmul_rn(d, inv_s), phi);
  return __umulhi(p, kKE4m3 << 6) + (uint32_t)r;
}

// floor(n / f), n mod f for n < 2^32 from m = floor((2^32 - 1) / f): the
// multiply-high estimate is at most one below the quotient.
__device__ __forceinline__ uint32_t div32_recip(uint32_t n, uint32_t f, uint32_t m, uint32_t &r) {
  uint32_t q = __umulhi(n, m);
  r = n - q * f;
  if (r >= f) {
    ++q;
    r -= f;
  }
  return q;
}

// floor(x / f) and x mod f for x < 2^63, 1 <= f <= 2^M and x / f < 2^(63 - M)
// (the encoder renormalises to x < f 2^(63 - M) first), without the FP64
// division routine or 64-bit integer <-> float conversions (both run on the
// slow FP64 unit of this part).  M <= 16 (e4m3): exact 32-bit steps.  M = 28
// (bf16), in fp32 with an approximate reciprocal rf of f (1 ulp, PTX
// rcp.approx), so rf carries at most 3 2^-24 relative error with the rounding
// of f itself:
//  1. q0 = 8 floor(fl(x) rf / 8), x converted as two 32-bit halves (2 2^-24
//     relative with their sum) and the product rounded: 6 2^-24 relative in
//     all, so |x / f - q0| < 6 2^-24 2^35 + 8 < 2^14 (the conversion to u32
//     saturates only within that bound);
//  2. r0 = x - q0 f (exact, |r0| < 2^14 f <= 2^42) splits into exact 24-bit
//     limbs, so fl(r0) rf is within 5 2^-24 2^14 < 0.005 of r0 / f and its
//     nearest integer d within 0.505;
//  3. q1 = q0 + d leaves r1 = x - q1 f in (-0.505 f, 0.505 f): the quotient
//     is q1 or q1 - 1.  The bounded fix-up loops below take that step.
template <int M>
__device__ __forceinline__ uint64_t divmod_u64(uint64_t x, uint32_t f, uint64_t &rem) {
  if (M <= 16) {
    // f < 2^16 and x < f 2^47: three exact 32-bit divisions by one reciprocal,
    // over the high word and then 16 bits at a time (each partial remainder is
    // below f, so every dividend stays below f 2^16 <= 2^32)
    const uint32_t m = 0xFFFFFFFFu / f;
    const uint32_t xh = (uint32_t)(x >> 32), xl = (uint32_t)x;
    uint32_t r1, r2, r3;
    const uint32_t q1 = div32_recip(xh, f, m, r1);
    const uint32_t q2 = div32_recip((r1 << 16) | (xl >> 16), f, m, r2);
    const uint32_t q3 = div32_recip((r2 << 16) | (xl & 0xFFFFu), f, m, r3);
    rem = r3;
    return ((uint64_t)q1 << 32) + ((uint64_t)q2 << 16) + q3;
  }
  static_assert(M <= 16 || M == 28, "the error bounds above are for M = 28");
  float rf;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rf) : "f"((float)f));
  const float xf = fmaf((float)(uint32_t)(x >> 32), 4294967296.0f, (float)(uint32_t)x);
  const float qf = xf * rf;
  int64_t q = (int64_t)__float2uint_rz(qf * 0.125f) << 3;
  int64_t r = (int64_t)x - q * (int64_t)f;
  const float rl = fmaf((float)(int32_t)(r >> 24), 16777216.0f, (float)(uint32_t)(r & 0xFFFFFF));
  const int32_t d = __float2int_rn(rl * rf);
  q += d;
  r -= (int64_t)d * (int64_t)f;
  for (int i = 0; i < 4 && r < 0; ++i) {
    q -= 1;
    r += f;
  }
  for (int i = 0; i < 4 && r >= (int64_t)f; ++i) {
    q += 1;
    r -= f;
  }
  rem = (uint64_t)r;
  return (uint64_t)q;
}

__device__ __forceinline__ float bf16_to_f32(uint32_t u) { return __uint_as_float(u << 16); }

__device__ __forceinline__ bool mu_valid(uint32_t mu_bits) { return (mu_bits & 0x7F80u) != 0x7F80u; }

// Error flag bits gathered in the workspace.
enum : uint32_t {
  kFlagSymbol = 1u,
  kFlagParam = 2u,
  kFlagCorrupt = 4u,
  kFlagOverflow = 8u,
  kFlagCapacity = 16u,
  kFlagArg = 32u,  // an argument only the device can check (a page index)
};

}  // namespace skv
