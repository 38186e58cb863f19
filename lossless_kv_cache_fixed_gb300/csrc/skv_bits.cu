// skv_bits.cu -- ideal code length -log2 q(x) per scalar and its total.
//
// Page "推测式 KV 编码无损压缩 KV 缓存最高可达约 4 倍" (Speculative KV coding),
// section "KV 缓存并非真正随机": the true distribution of a given cache is a
// point mass, so every coded bit is cross-entropy and the ideal cost of a
// scalar is -log2 q(x), q the model's mass on the symbol's bin.  Section
// "早期结果" gives q for bf16 (0.95 / 0.03 / 0.02 mixture), section
// "原生 FP8 KV 缓存" the bin-integrated N(mu, sigma^2) for e4m3.
//
// Evaluated in fp32 in the log domain so that nothing underflows:
//   * bins narrow against sigma (width w and centre zm in sigma units with
//     w max(1,|zm|) < 0.5): the midpoint rule with Hermite corrections;
//   * otherwise the tail mass on the far side of mu via the scaled
//     complementary error function, log Q(z) = log(erfcx(z/sqrt2)/2) - z^2/2;
//   * the mixture by log-sum-exp in base 2.
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

// The common case of log2_gauss_bin alone: sets ok = false (and returns 0)
// when the bin needs the tail evaluation.
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

// log2 of the N(mu, s^2) mass on [lo, hi); inv_s = 1/s, log2_s = log2 s.
//  * w max(1, |zm|) < 0.5 (w = width/s, zm = centre in sigma units): the
//    mass is w phi(zm) (1 + He2 w^2/24 + He4 w^4/1920 + He6 w^6/322560),
//    He_n the probabilists' Hermite polynomials; the next term is below
//    4e-6 relative there.
//  * otherwise the tail on the far side of mu, in the natural-log domain.
__device__ float log2_gauss_bin(float lo, float hi, float mu, float inv_s, float log2_s) {
  if (!(hi > lo)) return -INFINITY;
  if (isfinite(lo) && isfinite(hi)) {
    const float width = hi - lo;  // neighbouring midpoints: exact
    const float w = width * inv_s;
    const float zm = (lo + 0.5f * width - mu) * inv_s;
    if (w * fmaxf(1.0f, fabsf(zm)) < 0.5f) {
      const float z2 = zm * zm, w2 = w * w;
      const float he2 = z2 - 1.0f, he4 = fmaf(z2, z2 - 6.0f, 3.0f);
      const float he6 = fmaf(z2, fmaf(z2, z2 - 15.0f, 45.0f), -15.0f);
      const float y = w2 * fmaf(w2, fmaf(w2, he6 * (1.0f / 322560.0f), he4 * (1.0f / 1920.0f)),
                                he2 * (1.0f / 24.0f));
      const float l1p = y * fmaf(y, fmaf(y, 1.0f / 3.0f, -0.5f), 1.0f);  // log(1 + y), |y| < 0.02
      return fmaf(-0.5f * kLog2e, z2, -kLog2Sqrt2Pi) + (log2f(width) - log2_s) + l1p * kLog2e;
    }
  }
  return log2_gauss_tail(lo, hi, mu, inv_s);
}

__device__ __forceinline__ float lo_e4m3_value(int32_t r);

// -log2 q of one scalar.  FULL = false evaluates only the common (series)
// case and sets `deferred` when the scalar needs the tail evaluation.
// N(mu, s^2) mass on [lo, hi) as Q(a) - Q(b), Q(z) = erfc(z / sqrt 2) / 2 the
// upper tail, with the bin mirrored when it lies below mu so that a < b and a
// is the edge on the far side of mu (both of a straddling bin's edges: Q(a)
// near 1 then carries absolute error only).  Outside the series case
// w max(1, |z_m|) >= 0.5 gives Q(a) / Q(b) >= e^0.5, so the difference keeps
// the relative accuracy of erfcf.  `far` receives a (deep tails: a >= 9).
__device__ __forceinline__ float gauss_mass(float lo, float hi, float mu, float inv_s, float &far) {
  const float za = (lo - mu) * inv_s, zb = (hi - mu) * inv_s;
  const bool below = zb <= 0.0f;
  const float a = below ? -zb : za, b = below ? -za : zb;
  far = a;
  return 0.5f * (erfcf(a * 0.70710678f) - erfcf(b * 0.70710678f));
}

// bf16, both Gaussian bins narrow against their sigma (the series case): the
// mixture in the linear domain, each component w phi(z_m) (1 + y) with the
// Hermite correction y of log2_gauss_series, then one logarithm.  A Gaussian
// term too small for fp32 only drops below the p-hat term's 0.02 p-hat floor.
// Returns false (and nothing) when the bin needs the tail evaluation.
__device__ __forceinline__ bool ideal_series_bf16(float lo, float hi, float mu, float inv_s,
                                                  float ph, float &bits) {
  if (!(hi > lo) || !isfinite(lo) || !isfinite(hi)) return false;
  const float width = hi - lo;
  const float w = width * inv_s;
  const float zm = (lo + 0.5f * width - mu) * inv_s;
  if (!(w * fmaxf(1.0f, fabsf(zm)) < 0.5f)) return false;  // then also for 3 sigma
  auto comp = [](float w, float zm) {
    const float z2 = zm * zm, w2 = w * w;
    const float he2 = z2 - 1.0f, he4 = fmaf(z2, z2 - 6.0f, 3.0f);
    const float he6 = fmaf(z2, fmaf(z2, z2 - 15.0f, 45.0f), -15.0f);
    const float y = w2 * fmaf(w2, fmaf(w2, he6 * (1.0f / 322560.0f), he4 * (1.0f / 1920.0f)),
                              he2 * (1.0f / 24.0f));
    return w * 0.39894228f * __expf(-0.5f * z2) * (1.0f + y);  // w phi(zm) (1 + y)
  };
  const float q = fmaf(0.95f, comp(w, zm),
                       fmaf(0.03f, comp(w * (1.0f / 3.0f), zm * (1.0f / 3.0f)), 0.02f * ph));
  bits = -__log2f(q);
  return true;
}

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
  if (DT == 0 && !FULL) {
    float bits;
    if (ideal_series_bf16(lo, hi, mu, inv_s, phat[r], bits)) return bits;
    deferred = true;
    return 0.0f;
  }
  const float log2_s = __log2f(sigma);
  float l1, l3 = 0.0f;
  if (FULL && DT == 0) {
    // the mixture in the linear domain: p-hat's 0.02 floor keeps q normal, so a
    // Gaussian mass below fp32's range does not matter
    float far;
    const float m1 = hi > lo ? gauss_mass(lo, hi, mu, inv_s, far) : 0.0f;
    const float m3 = hi > lo ? gauss_mass(lo, hi, mu, inv_s * (1.0f / 3.0f), far) : 0.0f;
    return -log2f(fmaf(0.95f, fmaxf(m1, 0.0f), fmaf(0.03f, fmaxf(m3, 0.0f), 0.02f * phat[r])));
  }
  if (FULL) {
    // e4m3: one branch-free difference of tails for every bin but the deep
    // tails (log domain) and bins under 1e-3 sigma wide (the series, where the
    // difference would cancel); the difference's relative error, about
    // 6e-8 / (a w), is below 1e-4 of the mass from w = 1e-3 on
    const float wz = (hi - lo) * inv_s;
    bool ok = false;
    if (wz < 1e-3f) l1 = log2_gauss_series(lo, hi, mu, inv_s, log2_s, ok);
    if (!ok) {
      float far;
      const float m = hi > lo ? gauss_mass(lo, hi, mu, inv_s, far) : 0.0f;
      l1 = (far < 9.0f && m > 0.0f) ? log2f(m) : log2_gauss_tail(lo, hi, mu, inv_s);
    }
  } else {
    bool ok1 = true, ok3 = true;
    l1 = log2_gauss_series(lo, hi, mu, inv_s, log2_s, ok1);
    if (DT == 0) l3 = log2_gauss_series(lo, hi, mu, inv_s * (1.0f / 3.0f), log2_s + 1.5849625f, ok3);
    if (!ok1 || !ok3) {
      deferred = true;
      return 0.0f;
    }
  }
  if (DT == 1) return -l1;
  const float ph = phat[r];
  if (l1 > -100.0f && l3 > -100.0f) {
    // no component can underflow: sum the mixture directly
    return -__log2f(fmaf(0.95f, exp2f(l1), fmaf(0.03f, exp2f(l3), 0.02f * ph)));
  }
  const float a = -0.07400058f + l1;  // log2 0.95
  const float b = -5.0588937f + l3;   // log2 0.03 (the wide component: sigma * 3)
  const float c = -5.6438562f + __log2f(ph);  // log2 0.02
  const float m = fmaxf(a, fmaxf(b, c));
  if (m == -INFINITY) return INFINITY;
  return -(m + __log2f(exp2f(a - m) + exp2f(b - m) + exp2f(c - m)));
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

template <int DT, bool O0>
__global__ void __launch_bounds__(256) k_ideal(IdealLaunch a) {
  __shared__ float s_lo8[256];
  __shared__ double s_part[256];
  __shared__ float s_bits[8 * 256];
  __shared__ uint16_t s_queue[8 * 256];  // per warp: up to 8 deferred scalars per lane
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
  const uint64_t TD = (uint64_t)a.geo.T * (uint64_t)a.geo.D;
  const int64_t n8 = a.geo.n / 8;
  const float *sig = a.sigma_chunk ? a.sigma_chunk : a.sigma;
  uint32_t flags = 0;
  double acc = 0.0;
  // The loop runs the same number of times for every lane of a warp (lanes past
  // the end are switched off), because the deferred-scalar queue below is
  // filled and worked off by the whole warp.
  const int lane = threadIdx.x & 31;
  for (int64_t gw = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); gw < n8;
       gw += (int64_t)gridDim.x * blockDim.x) {
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
    // pass 1: the common case for all 8 scalars.  Scalars that need the tail
    // evaluation go to a per-warp queue, which the whole warp then works off
    // 32 at a time, so that no lane idles through the (long) tail code.
    uint16_t *q = s_queue + (threadIdx.x >> 5) * 256;
    int qn = 0;
#pragma unroll 1
    for (int k = 0; k < 8; ++k) {
      bool deferred = false;
      float b = 0.0f;
      // e4m3 bins are wide against sigma, so the tail case is the common one
      // there: evaluate it in place instead of queueing nearly every scalar
      if (act && O0) {
        // order-0 baseline: q = p-hat
        const int32_t r = rank_bf16(sym_at<DT>(kv4, k));
        if (r < 0 || r >= kNsymBf16) flags |= kFlagSymbol;
        else b = -log2f(__ldg(a.phat + r));
      } else if (act) {
        b = ideal_one<DT, DT == 1>(sym_at<DT>(kv4, k), mu_at(mu4, k), __ldg(sig + srow + k),
                                   a.phat, s_lo8, flags, deferred);
      }
      s_bits[k * 256 + threadIdx.x] = b;
      const uint32_t dm = __ballot_sync(0xFFFFFFFFu, deferred);
      if (deferred) q[qn + __popc(dm & ((1u << lane) - 1u))] = (uint16_t)((k << 5) | lane);
      qn += __popc(dm);
    }
    __syncwarp();
    for (int base = 0; base < qn; base += 32) {
      if (base + lane < qn) {
        const uint32_t e = q[base + lane];
        const int k = (int)(e >> 5), owner = (int)(e & 31u);
        const uint64_t j = (uint64_t)(gw + owner) * 8 + k;  // the owner's scalar
        const uint32_t sym = DT == 0 ? (uint32_t)static_cast<const uint16_t *>(a.kv)[j]
                                     : (uint32_t)static_cast<const uint8_t *>(a.kv)[j];
        const uint64_t srow_j = sigma_index(a, j, TD);
        bool unused = false;
        s_bits[k * 256 + (threadIdx.x & ~31) + owner] =
            ideal_one<DT, true>(sym, (uint32_t)a.mu[j], __ldg(sig + srow_j), a.phat, s_lo8,
                                flags, unused);
      }
    }
    __syncwarp();
    if (!act) continue;
    float bits[8], part = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      bits[k] = s_bits[k * 256 + threadIdx.x];
      part += bits[k];
    }
    acc += (double)part;
    if (a.per_scalar) {
      float4 *o = reinterpret_cast<float4 *>(a.per_scalar + i0);
      o[0] = make_float4(bits[0], bits[1], bits[2], bits[3]);
      o[1] = make_float4(bits[4], bits[5], bits[6], bits[7]);
    }
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
