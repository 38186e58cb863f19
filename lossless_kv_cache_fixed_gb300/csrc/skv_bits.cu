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
//   * narrow bins (width w and centre zm in sigma units with w max(1,|zm|) <
//     0.05): the midpoint rule with its second-order term;
//   * otherwise the tail mass on the far side of mu via the scaled
//     complementary error function, log Q(z) = log(erfcx(z/sqrt2)/2) - z^2/2;
//   * the mixture by log-sum-exp.
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

// log of the N(mu, s^2) mass on [lo, hi); inv_s = 1/s, log_s = log s.
__device__ float log_gauss_bin(float lo, float hi, float mu, float inv_s, float log_s) {
  if (!(hi > lo)) return -INFINITY;
  if (isfinite(lo) && isfinite(hi)) {
    const float width = hi - lo;  // neighbouring midpoints: exact
    const float w = width * inv_s;
    const float zm = (lo + 0.5f * width - mu) * inv_s;
    if (w * fmaxf(1.0f, fabsf(zm)) < 0.05f) {
      return -0.5f * zm * zm - 0.91893853f + (logf(width) - log_s) +
             log1pf((zm * zm - 1.0f) * w * w * (1.0f / 24.0f));
    }
  }
  const float za = (lo - mu) * inv_s, zb = (hi - mu) * inv_s;
  if (za >= 0.0f) {
    const float a = log_upper_tail(za), b = log_upper_tail(zb);
    return a + logf(-expm1f(b - a));
  }
  if (zb <= 0.0f) {
    const float a = log_upper_tail(-zb), b = log_upper_tail(-za);
    return a + logf(-expm1f(b - a));
  }
  const float qa = isfinite(za) ? 0.5f * erfcf(-za * 0.70710678f) : 0.0f;
  const float qb = isfinite(zb) ? 0.5f * erfcf(zb * 0.70710678f) : 0.0f;
  return log1pf(-(qa + qb));
}

__device__ __forceinline__ float lo_e4m3_value(int32_t r);

template <int DT>
__device__ __forceinline__ float ideal_one(uint32_t sym, uint32_t mu_bits, float sigma,
                                           const float *phat, const float *lo8,
                                           uint32_t &flags) {
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
  const float inv_s = 1.0f / sigma;
  const float log_s = logf(sigma);
  const float l1 = log_gauss_bin(lo, hi, mu, inv_s, log_s);
  if (DT == 1) return -l1 * 1.44269504f;
  const float a = -0.05129329f + l1;                                            // log 0.95
  const float b = -3.5065579f + log_gauss_bin(lo, hi, mu, inv_s * (1.0f / 3.0f),
                                              log_s + 1.0986123f);             // log 0.03
  const float c = -3.912023f + logf(phat[r]);                                   // log 0.02
  const float m = fmaxf(a, fmaxf(b, c));
  if (m == -INFINITY) return INFINITY;
  const float lse = m + logf(expf(a - m) + expf(b - m) + expf(c - m));
  return -lse * 1.44269504f;
}

template <int DT>
__global__ void __launch_bounds__(256) k_ideal(IdealLaunch a) {
  __shared__ float s_lo8[256];
  __shared__ double s_part[256];
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
  const uint32_t D = (uint32_t)a.geo.D;
  const int64_t n8 = a.geo.n / 8;
  uint32_t flags = 0;
  double acc = 0.0;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < n8;
       g += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t i0 = (uint64_t)g * 8;
    const uint64_t srow = (i0 / TD) * D + (uint32_t)(i0 % D);
    uint32_t sym[8], mub[8];
    if (DT == 0) {
      uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.kv) + i0));
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) sym[k] = (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
    } else {
      uint2 v = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint8_t *>(a.kv) + i0));
      uint32_t w[2] = {v.x, v.y};
#pragma unroll
      for (int k = 0; k < 8; ++k) sym[k] = (w[k >> 2] >> (8 * (k & 3))) & 0xFFu;
    }
    {
      uint4 v = __ldg(reinterpret_cast<const uint4 *>(a.mu + i0));
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) mub[k] = (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
    }
    float bits[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      bits[k] = ideal_one<DT>(sym[k], mub[k], __ldg(a.sigma + srow + k), a.phat, s_lo8, flags);
      acc += (double)bits[k];
    }
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

__global__ void k_ideal_final(const double *partials, int nb, WsHead *head) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  double s = 0.0;
  for (int i = 0; i < nb; ++i) s += partials[i];
  head->bits = s;
}

cudaError_t launch_ideal(const IdealLaunch &a, cudaStream_t s) {
  if (a.dtype == 0) k_ideal<0><<<a.nblocks, 256, 0, s>>>(a);
  else k_ideal<1><<<a.nblocks, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_ideal_final<<<1, 32, 0, s>>>(a.partials, a.nblocks, a.head);
  return cudaGetLastError();
}

}  // namespace skv
