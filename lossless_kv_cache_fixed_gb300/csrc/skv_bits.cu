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
#include "skv_ideal.cuh"
#include "skv_model.cuh"

namespace skv {

using namespace ideal;

__device__ __forceinline__ float lo_e4m3_value(int32_t r);

// (log2 Q(z_k), log2 Q(z_{k+1}) - log2 Q(z_k)) at z_k = k / kTailPerUnit.
__device__ float2 g_log2q[kTailN];

const float2 *tail_table() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_log2q) != cudaSuccess) return nullptr;
  return static_cast<const float2 *>(p);
}

cudaError_t upload_tail_table(const float *l2q) {
  float2 pairs[kTailN];
  for (int k = 0; k < kTailN; ++k)
    pairs[k] = make_float2(l2q[k], k + 1 < kTailN ? l2q[k + 1] - l2q[k] : 0.0f);
  return cudaMemcpyToSymbol(g_log2q, pairs, sizeof(pairs));
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
      const float b = ideal_one<DT, true>(sym, (uint32_t)a.mu[j],
                                          __fdividef(1.0f, __ldg(sig + sigma_index(a, j, TD))),
                                          a.phat, s_lo8, g_log2q, flags, unused);
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
        // fp32 1/sigma to about 1e-7 relative is far inside the 1e-3 tolerance
        b = ideal_one<DT, false>(sym_at<DT>(kv4, k), mu_at(mu4, k),
                                 __fdividef(1.0f, __ldg(sig + srow + k)), a.phat, s_lo8, g_log2q,
                                 flags, deferred);
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
// then a tree; added to the head's total (zeroed with the head, so that
// encoded chunk ranges add up their bits in call order).
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
  if (threadIdx.x == 0) head->bits += s_sum[0];
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
