// skv_bits.cu -- ideal code length -log2 q(x) per scalar and its total.
//
// Page "推测式 KV 编码无损压缩 KV 缓存最高可达约 4 倍" (Speculative KV coding),
// section "KV 缓存并非真正随机": the true distribution of a given cache is a
// point mass, so every coded bit is cross-entropy and the ideal cost of a
// scalar is -log2 q(x), q the model's mass on the symbol's bin.  Section
// "早期结果" gives q for bf16 (0.95 / 0.03 / 0.02 mixture), section
// "原生 FP8 KV 缓存" the bin-integrated N(mu, sigma^2) for e4m3.
//
// Evaluated in fp32 (w = bin width and zm = bin centre, both in sigma units):
//   * bf16, w < 1 and w |zm| < 2 (about 99% of scalars): each Gaussian
//     component's bin mass by the midpoint rule with Hermite corrections up to
//     He6 (the first dropped term is below 3e-6 relative there), the mixture in
//     the linear domain, one logarithm; narrow bins beyond 64 sigma cost p-hat's
//     floor -log2(0.02 p-hat) (the Gaussian masses are negligible there);
//   * bf16 otherwise (queued per warp): each component's mass as a difference
//     of complementary error functions on the far side of mu, the mixture in
//     the linear domain (p-hat's 0.02 floor keeps it a normal float);
//   * e4m3: the difference of tails from a table of log2 Q for bins at least
//     0.01 sigma wide with the near edge within 9 sigma (about 98.7% of
//     scalars); for the rest (queued per warp) the difference of erfc tails,
//     the log-domain tail log Q(z) = log(erfcx(z/sqrt2)/2) - z^2/2 for deep
//     tails, the series (in log2) for bins under 1e-3 sigma wide.
// Per-thread sums, then a fixed-order block tree and a fixed-order final sum,
// all in fp64: the total does not depend on scheduling.
#include <cuda_runtime.h>

#include "skv_internal.h"
#include "skv_model.cuh"

namespace skv {

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
__device__ __noinline__ float log2_gauss_tail(float lo, float hi, float mu, float inv_s) {
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

__device__ __forceinline__ float lo_e4m3_value(int32_t r);

// (log2 Q(z_k), log2 Q(z_{k+1}) - log2 Q(z_k)) at z_k = k / kTailPerUnit.
__device__ float2 g_log2q[kTailN];

cudaError_t upload_tail_table(const float *l2q) {
  float2 pairs[kTailN];
  for (int k = 0; k < kTailN; ++k)
    pairs[k] = make_float2(l2q[k], k + 1 < kTailN ? l2q[k + 1] - l2q[k] : 0.0f);
  return cudaMemcpyToSymbol(g_log2q, pairs, sizeof(pairs));
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
__device__ __forceinline__ float q_tab(float z) {
  if (!(z < 12.0f)) return 0.0f;
  const float t = z * (float)kTailPerUnit;
  const int k = (int)t;
  const float2 e = __ldg(&g_log2q[k]);
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
template <int DT, bool FULL>
__device__ __forceinline__ float ideal_one(uint32_t sym, uint32_t mu_bits, float sigma,
                                           const float *phat, const float *lo8, uint32_t &flags,
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
  // fp32 to about 1e-7 relative is far inside the 1e-3 tolerance of the ideal
  const float inv_s = __fdividef(1.0f, sigma);
  if (DT == 0) {
    if (!FULL) {
      float bits;
      if (ideal_series_bf16(lo, hi, mu, inv_s, phat[r], bits)) return bits;
      deferred = true;
      return 0.0f;
    }
    // the mixture in the linear domain: p-hat's 0.02 floor keeps q normal, so a
    // Gaussian mass below fp32's range does not matter
    float far;
    const float m1 = hi > lo ? gauss_mass(lo, hi, mu, inv_s, far) : 0.0f;
    const float m3 = hi > lo ? gauss_mass(lo, hi, mu, inv_s * (1.0f / 3.0f), far) : 0.0f;
    return -log2f(fmaf(0.95f, fmaxf(m1, 0.0f), fmaf(0.03f, fmaxf(m3, 0.0f), 0.02f * phat[r])));
  }
  const float wz = (hi - lo) * inv_s;
  if (!FULL) {
    // e4m3 common case, bins at least 0.01 sigma wide whose near edge lies
    // within 9 sigma (all but about 1.3% of a cache): the mass from the tail
    // table, Q(a) - Q(b) for a bin on one side of mu (mirrored below it) and
    // 1 - Q(-a) - Q(b) for a bin around mu, so the error scales with the
    // tails.  With epsilon <= 5e-6 per tail, a one-sided bin's mass is off by
    // at most epsilon (Q(a) + Q(b)) / (Q(a) - Q(b)) <= 250 epsilon relative (w =
    // 0.01 at a = 0, where such a bin costs 8 bits: 2e-3 bits of a 8e-3
    // tolerance), a bin around mu's by epsilon (1 - m) absolute.  The rest
    // waits for the full evaluation below.
    const float za = (lo - mu) * inv_s, zb = (hi - mu) * inv_s;
    const bool below = zb <= 0.0f;
    const float a = below ? -zb : za, b = below ? -za : zb;
    if (!(wz >= 0.01f && a < 9.0f)) {
      deferred = true;
      return 0.0f;
    }
    const float m = a >= 0.0f ? q_tab(a) - q_tab(b) : 1.0f - q_tab(-a) - q_tab(b);
    return -__log2f(m);
  }
  // e4m3 full evaluation: one branch-free difference of erfc tails for every
  // bin but the deep tails (log domain) and bins under 1e-3 sigma wide (the
  // series, where the difference would cancel); the difference's relative
  // error, about 6e-8 / (a w), is below 1e-4 of the mass from w = 1e-3 on
  bool ok = false;
  float l1 = 0.0f;
  if (wz < 1e-3f) l1 = log2_gauss_series(lo, hi, mu, inv_s, __log2f(sigma), ok);
  if (!ok) {
    float far;
    const float m = hi > lo ? gauss_mass(lo, hi, mu, inv_s, far) : 0.0f;
    l1 = (far < 9.0f && m > 0.0f) ? log2f(m) : log2_gauss_tail(lo, hi, mu, inv_s);
  }
  return -l1;
}

template <int DT>
__device__ __forceinline__ uint32_t sym_at(uint4 kv4, int k) {
  if (DT == 0) {
    const uint32_t w = k < 2 ? kv4.x : (k < 4 ? kv4.y : (k < 6 ? kv4.z : kv4.w));
    return (w >> (16 * (k & 1))) & 0xFFFFu;
  }
  const uint32_t w = k < 4 ? kv4.x : kv4.y;
  return (w >> (8 * (k & 3))) & 0xFFu;
}

__device__ __forceinline__ uint32_t mu_at(uint4 mu4, int k) {
  const uint32_t w = k < 2 ? mu4.x : (k < 4 ? mu4.y : (k < 6 ? mu4.z : mu4.w));
  return (w >> (16 * (k & 1))) & 0xFFFFu;
}

// Index of scalar i's sigma: (row, channel) in the static table, or (chunk,
// channel) in the per-block table.
__device__ __forceinline__ uint64_t sigma_index(const IdealLaunch &a, uint64_t i, uint64_t TD) {
  const uint64_t D = (uint64_t)a.geo.D;
  // i / TD by multiply-high with the host's reciprocal (at most one below), then exact
  uint64_t row = __umul64hi(i, a.td_rcp);
  if ((row + 1) * TD <= i) ++row;
  const uint64_t in_row = i - row * TD;
  const uint64_t ch = (in_row >> 32) == 0 ? (uint32_t)in_row % (uint32_t)D : in_row % D;
  if (!a.sigma_chunk) return row * D + ch;
  const uint64_t cw = D * (uint64_t)a.geo.Tb;  // scalars of a full chunk
  const uint64_t tb = (TD >> 32) == 0 && (cw >> 32) == 0 ? (uint32_t)in_row / (uint32_t)cw
                                                         : in_row / cw;
  return (row * (uint64_t)a.geo.ntb + tb) * D + ch;
}

// Per-warp ring of deferred scalars (power of two).  At most 31 wait between
// loop iterations and one iteration adds at most 256, so 512 never overflows.
constexpr uint32_t kIdealRing = 512;

template <int DT, bool O0>
__global__ void __launch_bounds__(256) k_ideal(IdealLaunch a) {
  __shared__ float s_lo8[256];
  __shared__ double s_part[256];
  __shared__ uint32_t s_ring[8 * kIdealRing];
  if (DT == 1) {
    // e4m3 bin edges: midpoints of neighbouring values, +-inf at the ends
    for (int r = threadIdx.x; r < 255; r += blockDim.x) {
      float v;
      if (r == 0) v = -INFINITY;
      else if (r == 254) v = INFINITY;
      else v = 0.5f * (lo_e4m3_value(r - 1) + lo_e4m3_value(r));
      s_lo8[r] = v;
    }
    __syncthreads();
  }
  constexpr bool kDefer = !O0;  // the order-0 baseline has no rare case
  const uint64_t TD = (uint64_t)a.geo.T * (uint64_t)a.geo.D;
  const int64_t n8 = a.geo.n / 8;
  const float *sig = a.sigma_chunk ? a.sigma_chunk : a.sigma;
  uint32_t flags = 0;
  double acc = 0.0;
  const int lane = threadIdx.x & 31;
  const int64_t gw0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31);
  const int64_t gstride = (int64_t)gridDim.x * blockDim.x;
  // Scalars outside the common cases (about 1% of a bf16 cache outside the
  // series case, about 1.3% of an e4m3 cache in the deep tails or in bins
  // narrower than 0.01 sigma) wait in the warp's ring as (iteration << 8) | (k << 5) | lane until 32 have gathered;
  // then the whole warp evaluates them at once, so the long tail code runs once
  // per 32 of them, not once per loop iteration that holds one.  Iterations fit
  // in 24 bits: with fewer than 4096 blocks the loop runs once, and with 4096
  // blocks 2^24 iterations would be 2^47 scalars.
  uint32_t *ring = s_ring + (threadIdx.x >> 5) * kIdealRing;
  uint32_t head = 0, tail = 0;  // warp-uniform
  auto work_off = [&](uint32_t cnt) {  // the oldest cnt <= 32 entries, one per lane
    if ((uint32_t)lane < cnt) {
      const uint32_t e = ring[(head + lane) & (kIdealRing - 1)];
      const int k = (int)((e >> 5) & 7u), owner = (int)(e & 31u);
      const uint64_t j = (uint64_t)(gw0 + (int64_t)(e >> 8) * gstride + owner) * 8 + k;
      bool unused = false;
      const uint32_t sym = DT == 0 ? (uint32_t)static_cast<const uint16_t *>(a.kv)[j]
                                   : (uint32_t)static_cast<const uint8_t *>(a.kv)[j];
      const float b = ideal_one<DT, true>(sym, (uint32_t)a.mu[j], __ldg(sig + sigma_index(a, j, TD)),
                                          a.phat, s_lo8, flags, unused);
      acc += (double)b;
      if (a.per_scalar) a.per_scalar[j] = b;  // after the owner's store of 0 (a barrier apart)
    }
    head += cnt;
    __syncwarp();  // the slots just read may be written by the next iteration
  };
  // The loop runs the same number of times for every lane of a warp (lanes past
  // the end are switched off), because the ring is filled and worked off by the
  // whole warp.
  uint32_t it = 0;
  for (int64_t gw = gw0; gw < n8; gw += gstride, ++it) {
    const int64_t g = gw + lane;
    const bool act = g < n8;
    const uint64_t i0 = act ? (uint64_t)g * 8 : 0;
    const uint64_t srow = sigma_index(a, i0, TD);
    uint4 kv4 = make_uint4(0, 0, 0, 0), mu4 = make_uint4(0, 0, 0, 0);
    if (act) {
      if (DT == 0) {
        kv4 = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.kv) + i0));
      } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint8_t *>(a.kv) + i0));
        kv4.x = v.x;
        kv4.y = v.y;
      }
      if (!O0) mu4 = __ldg(reinterpret_cast<const uint4 *>(a.mu + i0));
    }
    // Unrolled: only the common cases are inlined here (the rare ones wait in
    // the ring, below), so eight copies stay small, and the symbols, mu and
    // the results are picked from registers with constant indices.
    float bits[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      bool deferred = false;
      float b = 0.0f;
      if (act && O0) {
        // order-0 baseline: q = p-hat
        const int32_t r = rank_bf16(sym_at<DT>(kv4, k));
        if (r < 0 || r >= kNsymBf16) flags |= kFlagSymbol;
        else b = -log2f(__ldg(a.phat + r));
      } else if (act) {
        b = ideal_one<DT, false>(sym_at<DT>(kv4, k), mu_at(mu4, k), __ldg(sig + srow + k),
                                 a.phat, s_lo8, flags, deferred);
      }
      bits[k] = b;
      if (kDefer) {
        const uint32_t dm = __ballot_sync(0xFFFFFFFFu, deferred);
        if (deferred)
          ring[(tail + __popc(dm & ((1u << lane) - 1u))) & (kIdealRing - 1)] =
              (it << 8) | ((uint32_t)k << 5) | (uint32_t)lane;
        tail += __popc(dm);
      }
    }
    if (act) {
      float part = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) part += bits[k];
      acc += (double)part;
      if (a.per_scalar) {
        float4 *o = reinterpret_cast<float4 *>(a.per_scalar + i0);
        o[0] = make_float4(bits[0], bits[1], bits[2], bits[3]);
        o[1] = make_float4(bits[4], bits[5], bits[6], bits[7]);
      }
    }
    if (kDefer) {
      __syncwarp();  // ring entries and the owners' stores before the work-off
      while (tail - head >= 32u) work_off(32u);
    }
  }
  if (kDefer) {
    __syncwarp();
    if (tail != head) work_off(tail - head);
  }
  if (flags) atomicOr(&a.head->flags, flags);
  s_part[threadIdx.x] = acc;
  __syncthreads();
  for (int off = 128; off; off >>= 1) {
    if (threadIdx.x < off) s_part[threadIdx.x] += s_part[threadIdx.x + off];
    __syncthreads();
  }
  if (threadIdx.x == 0) a.partials[blockIdx.x] = s_part[0];
}

// e4m3 value of rank r (r in [0, 254)): OCP E4M3, bias 7, no infinities
__device__ __forceinline__ float lo_e4m3_value(int32_t r) {
  const uint32_t u = bits_e4m3(r);
  const uint32_t e = (u >> 3) & 15u, m = u & 7u;
  float v = e ? ldexpf(1.0f + (float)m * 0.125f, (int)e - 7) : ldexpf((float)m * 0.125f, -6);
  return (u & 0x80u) ? -v : v;
}

// Sum of the block partials, in a fixed order: a strided pass per thread,
// then a tree.
__global__ void __launch_bounds__(1024) k_ideal_final(const double *partials, int nb, WsHead *head) {
  __shared__ double s_sum[1024];
  double v = 0.0;
  for (int i = threadIdx.x; i < nb; i += 1024) v += partials[i];
  s_sum[threadIdx.x] = v;
  __syncthreads();
  for (int off = 512; off; off >>= 1) {
    if (threadIdx.x < off) s_sum[threadIdx.x] += s_sum[threadIdx.x + off];
    __syncthreads();
  }
  if (threadIdx.x == 0) head->bits = s_sum[0];
}

cudaError_t launch_ideal_final(const double *partials, int n, WsHead *head, cudaStream_t s) {
  k_ideal_final<<<1, 1024, 0, s>>>(partials, n, head);
  return cudaGetLastError();
}

cudaError_t launch_ideal(const IdealLaunch &a, cudaStream_t s) {
  if (a.dtype == 0 && a.order0) k_ideal<0, true><<<a.nblocks, 256, 0, s>>>(a);
  else if (a.dtype == 0) k_ideal<0, false><<<a.nblocks, 256, 0, s>>>(a);
  else k_ideal<1, false><<<a.nblocks, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_ideal_final<<<1, 1024, 0, s>>>(a.partials, a.nblocks, a.head);
  return cudaGetLastError();
}

}  // namespace skv
