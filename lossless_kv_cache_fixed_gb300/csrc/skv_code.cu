// skv_code.cu -- encode, size scan, compaction, header check and decode kernels.
//
// Page "推测式 KV 编码无损压缩 KV 缓存最高可达约 4 倍" (Speculative KV coding),
// section "什么能预测 KV 缓存": an arithmetic coder maps (KV_full, mu, sigma) to
// bits and (bits, mu, sigma) back to KV_full.  Here the coder is interleaved
// rANS (64-bit state x in [2^31, 2^63), 32-bit words) over the fixed-point
// model of skv_model.cuh.
//
// GPU mapping.  One thread is one rANS lane; the G lanes of a chunk sit in
// consecutive threads of one warp (32/G chunks per warp), so the order in which
// lanes emit or consume renormalisation words inside a round comes from one
// ballot plus a prefix popcount.  A lane's symbols are 8-scalar groups: the
// encoder reads KV and mu as 16-byte vectors (8-byte for e4m3 KV); the decoder
// reads mu a symbol at a time (fewer live registers) and writes each group's
// 8 decoded symbols as one vector.  Warps loop over 32-lane tasks (the decoder
// hands out tasks after the first round from an atomic counter); the grid has
// at most one block per SM (768 threads; smaller blocks spread a small launch
// over all SMs, larger ones carry decode launches with several rounds of tasks:
// task_shape).  The Phi knot table (64 KiB), the e4m3 bin edges and the
// decoder's guess tables sit in shared memory, once per SM.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "skv_ideal.cuh"
#include "skv_internal.h"
#include "skv_model.cuh"

namespace skv {

__device__ uint2 g_phi[kPhiKnots];
__device__ float g_lo8[256];
__device__ float2 g_hinv[2][kHinvN + 1];

// At most one resident block per SM (24 warps as a rule): a single copy of the
// tables per SM leaves the rest of the unified L1 / shared memory to the L1
// cache (the p-hat prefix table, mu, the streams).  See task_shape.
constexpr int kCodeThreads = 768;
constexpr size_t kCodeSmem = sizeof(uint2) * kPhiKnots + sizeof(float) * 256;
constexpr int kDecThreads = 768;
// Decode blocks of launches with several rounds of tasks: as many warps as the
// registers allow (65,536 per SM; bf16 64 a thread: 28 warps, e4m3 56: 32),
// which the decoder's latency uses (32B bf16 decode 129 -> 143 GB/s, 8B e4m3
// 106 -> 125).  bf16 at 32 warps would drop to 62 registers and lost 3%.
template <int DT>
constexpr int dec_threads_max() { return DT == 0 ? 896 : 1024; }
constexpr size_t kDecSmem = kCodeSmem + sizeof(float2) * (kHinvN + 1) + sizeof(int32_t) * (kHinvN + 1);

cudaError_t upload_tables(const uint32_t *T, const float *lo8, const float *hb, const float *he) {
  uint2 pairs[kPhiKnots];
  for (int i = 0; i < kPhiKnots; ++i) {
    const uint32_t step = i + 1 < kPhiKnots ? T[i + 1] - T[i] : 0u;
    if (step >= 65536u) return cudaErrorInvalidValue;  // 2^26 phi(0) / 512 < 52,300
    pairs[i].x = T[i];
    pairs[i].y = step << 16;
  }
  cudaError_t e = cudaMemcpyToSymbol(g_phi, pairs, sizeof(pairs));
  if (e != cudaSuccess) return e;
  if ((e = cudaMemcpyToSymbol(g_lo8, lo8, sizeof(float) * 256)) != cudaSuccess) return e;
  float2 h[2][kHinvN + 1];
  for (int t = 0; t < 2; ++t)
    for (int k = 0; k <= kHinvN; ++k) {
      const float *src = t == 0 ? hb : he;
      h[t][k] = make_float2(src[k], k < kHinvN ? src[k + 1] - src[k] : 0.0f);
    }
  return cudaMemcpyToSymbol(g_hinv, h, sizeof(h));
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

__device__ __forceinline__ void stage_tables(uint2 *s_phi, float *s_lo8) {
  for (int i = threadIdx.x; i < kPhiKnots; i += blockDim.x) s_phi[i] = g_phi[i];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) s_lo8[i] = g_lo8[i];
  __syncthreads();
}

// 8 consecutive symbols of a group (bf16 patterns or e4m3 codes)
template <int DT>
__device__ __forceinline__ void load_syms(const void *kv, uint64_t at, uint32_t (&s)[8]) {
  if (DT == 0) {
    uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(kv) + at));
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) s[k] = (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
  } else {
    uint2 v = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint8_t *>(kv) + at));
    uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int k = 0; k < 8; ++k) s[k] = (w[k >> 2] >> (8 * (k & 3))) & 0xFFu;
  }
}

// The first 4 of them (the encoder with the ideal bits inside codes a group in
// two halves: its unrolled body stays half as long)
template <int DT>
__device__ __forceinline__ void load_syms(const void *kv, uint64_t at, uint32_t (&s)[4]) {
  if (DT == 0) {
    uint2 v = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(kv) + at));
    uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int k = 0; k < 4; ++k) s[k] = (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
  } else {
    const uint32_t v = __ldg(reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(kv) + at));
#pragma unroll
    for (int k = 0; k < 4; ++k) s[k] = (v >> (8 * k)) & 0xFFu;
  }
}

__device__ __forceinline__ void load_mu(const uint16_t *mu, uint64_t at, uint32_t (&m)[4]) {
  uint2 v = __ldg(reinterpret_cast<const uint2 *>(mu + at));
  uint32_t w[2] = {v.x, v.y};
#pragma unroll
  for (int k = 0; k < 4; ++k) m[k] = (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
}

__device__ __forceinline__ void load_inv(const float2 *inv, uint64_t at, ChanInv (&c)[4]) {
  const float4 *p = reinterpret_cast<const float4 *>(inv + at);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    float4 v = __ldg(p + k);
    c[2 * k].s = v.x;
    c[2 * k].s3 = v.y;
    c[2 * k + 1].s = v.z;
    c[2 * k + 1].s3 = v.w;
  }
}

__device__ __forceinline__ void load_mu(const uint16_t *mu, uint64_t at, uint32_t (&m)[8]) {
  uint4 v = __ldg(reinterpret_cast<const uint4 *>(mu + at));
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
}

__device__ __forceinline__ void load_inv(const float2 *inv, uint64_t at, ChanInv (&c)[8]) {
  const float4 *p = reinterpret_cast<const float4 *>(inv + at);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float4 v = __ldg(p + k);
    c[2 * k].s = v.x;
    c[2 * k].s3 = v.y;
    c[2 * k + 1].s = v.z;
    c[2 * k + 1].s3 = v.w;
  }
}

// Order-0 baseline: cum(r) = floor(K E_q[r] / 2^26) + r (the mixture with
// weights (0, 0, 100): the factor 100 cancels exactly).
__device__ __forceinline__ uint32_t cum_order0(int32_t r, const uint32_t *__restrict__ ecdf) {
  return (uint32_t)(((uint64_t)kKBf16 * __ldg(ecdf + r)) >> 26) + (uint32_t)r;
}

template <int DT>
__device__ __forceinline__ uint32_t cum_of(int32_t r, float mu, ChanInv inv, const uint2 *phi,
                                           const float *lo8, const uint32_t *ecdf) {
  if (DT == 0) return cum_bf16(r, mu, inv, phi, ecdf);
  return cum_e4m3(r, mu, inv.s, phi, lo8);
}

// ------------------------------------------------------------------------
// Model preparation
// ------------------------------------------------------------------------

__global__ void k_prep(const float *__restrict__ sigma, int64_t nsig,
                       const uint32_t *__restrict__ ecdf, float2 *__restrict__ inv,
                       WsHead *head) {
  uint64_t h = 0;
  uint32_t bad = 0;
  const int64_t nE = ecdf ? (int64_t)kNsymBf16 + 1 : 0;
  for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < nsig + nE;
       k += (int64_t)gridDim.x * blockDim.x) {
    uint32_t w;
    if (k < nsig) {
      float s = sigma[k];
      if (!sigma_valid(s)) {
        bad = 1;
        s = 1.0f;
      }
      ChanInv c = chan_inv(s);
      inv[k] = make_float2(c.s, c.s3);
      w = __float_as_uint(sigma[k]);
    } else {
      int64_t r = k - nsig;
      w = ecdf[r];
      if (r == 0 && w != 0u) bad = 1;
      if (r == kNsymBf16 && w != kPhiOne) bad = 1;
      if (r > 0 && w < ecdf[r - 1]) bad = 1;
    }
    h += mix64(((uint64_t)k << 32) | w);
  }
  if (bad) atomicOr(&head->flags, kFlagParam);
  for (int o = 16; o; o >>= 1) h += __shfl_xor_sync(0xFFFFFFFFu, h, o);
  if ((threadIdx.x & 31) == 0) atomicAdd(&head->hash_acc, (unsigned long long)h);
}

cudaError_t launch_prep(const float *sigma, int64_t nsig, const uint32_t *ecdf, float2 *inv,
                        WsHead *head, cudaStream_t s) {
  int64_t n = nsig + (ecdf ? kNsymBf16 + 1 : 0);
  if (n == 0) return cudaSuccess;  // nothing to check or hash (order-0 ideal bits)
  int blocks = (int)((n + 255) / 256);
  if (blocks > 1024) blocks = 1024;
  k_prep<<<blocks, 256, 0, s>>>(sigma, nsig, ecdf, inv, head);
  return cudaGetLastError();
}

// The bound on the guess's p-hat slope term a (below): large enough that the
// guess sits at mu's symbol, small enough that 1 + a dz/du stays finite.
constexpr float kGuessSlopeMax = 1e30f * kHscaleBf16;

// Inverse of the p-hat prefix table for the decoder's guess in the tails that
// only the p-hat component reaches, and (gmu) the guess's p-hat terms for each
// rank r of mu, in knots of the guess table (u times kHscaleBf16): 0.02 E(mu),
// and the slope 0.02 rho, with rho the p-hat mass of mu's bin per unit
// width (the width from mu's exponent: the bin of a mantissa step), so that
// the decoder's slope term is one multiply by sigma.  A guess only: any error
// costs search steps, never a wrong symbol.
__global__ void k_einv(const uint32_t *__restrict__ ecdf, int32_t *__restrict__ einv, int n,
                       float2 *__restrict__ gmu) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k <= n) {
    const uint32_t target = (uint32_t)(((uint64_t)k << 26) / (uint64_t)n);
    int32_t lo = 0, hi = kNsymBf16;  // smallest r in [0, 65282] with ecdf[r] >= target
    while (lo < hi) {
      const int32_t mid = (lo + hi) >> 1;
      if (ecdf[mid] >= target) hi = mid;
      else lo = mid + 1;
    }
    einv[k] = lo;
  }
  if (gmu && k < kNsymBf16) {
    const uint32_t ea = ecdf[k], eb = ecdf[k + 1];
    const uint32_t mub = bits_bf16(k);
    const float w = __uint_as_float(max(mub & 0x7F80u, 0x0080u) << 16) * (1.0f / 128.0f);
    float slope = 0.02f * (1.0f / 67108864.0f) * (float)(eb - ea) / w * kHscaleBf16;
    slope = slope >= 0.0f ? fminf(slope, kGuessSlopeMax) : 0.0f;  // a NaN (0 inf) gives 0
    gmu[k] = make_float2(0.02f * ((float)ea * (1.0f / 67108864.0f)) * kHscaleBf16, slope);
  }
}

cudaError_t launch_einv(const uint32_t *ecdf, int32_t *einv, int n, float2 *gmu, cudaStream_t s) {
  const int m = gmu && kNsymBf16 > n + 1 ? kNsymBf16 : n + 1;
  k_einv<<<(m + 255) / 256, 256, 0, s>>>(ecdf, einv, n, gmu);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------
// Encode: one thread per lane, rounds descending, lanes descending.
// ------------------------------------------------------------------------

// NT: most threads per block (the register budget follows from it).  BITS
// (bf16, multi-round launches only, where it pays): also the ideal code
// length -log2 q of every scalar (the per-scalar values of skv_ideal_bits),
// from the symbol's bin edges, mu and reciprocal already in registers.  The
// rare scalars outside the series' range (about 1%) are evaluated where they
// are met, out of line; a per-warp ring of them, as in the ideal-bits kernel,
// cost more in bookkeeping than it saved here.
template <int DT, bool O0, int NT = kCodeThreads, bool BITS = false>
__global__ void __launch_bounds__(NT, 1) k_encode(EncodeLaunch a) {
  static_assert(!BITS || (DT == 0 && !O0), "ideal bits fuse into the bf16 mixture coder only");
  extern __shared__ uint2 s_phi[];
  float *s_lo8 = reinterpret_cast<float *>(s_phi + kPhiKnots);
  __shared__ double s_bpart[BITS ? NT / 32 : 1];
  stage_tables(s_phi, s_lo8);
  double bacc = 0.0;

  constexpr int M = DT == 0 ? kMBf16 : kME4m3;
  constexpr int32_t NS = DT == 0 ? kNsymBf16 : kNsymE4m3;
  const int G = a.geo.G;
  const int lane = threadIdx.x & 31;
  const int ell = lane & (G - 1);
  const uint32_t seg = G == 32 ? 0xFFFFFFFFu : (((1u << G) - 1u) << (lane & ~(G - 1)));
  const uint32_t lt = seg & ((1u << lane) - 1u);
  const int64_t ntasks = (a.c_count * G + 31) / 32;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const uint32_t D = (uint32_t)a.geo.D;

  for (int64_t task = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); task < ntasks;
       task += nwarps) {
    const int64_t ci = (task * 32 + lane) / G;
    const bool live = ci < a.c_count;
    const int64_t c = live ? a.c_first + a.c_step * ci : 0;
    ChunkGeo cg = chunk_geo(a.geo, c);
    const uint32_t *ecdf = a.ecdf + (a.ecdf_row_stride ? (uint64_t)(c / a.geo.ntb) * a.ecdf_row_stride : 0);
    const uint32_t my_groups =
        (live && (uint32_t)ell < cg.ngroup) ? (cg.ngroup - ell + G - 1) / G : 0u;
    const uint32_t max_groups = __reduce_max_sync(0xFFFFFFFFu, my_groups);
    uint32_t *region = a.scratch + c * a.stride;
    const float2 *invrow = a.inv_chunk ? a.inv_chunk + (uint64_t)c * D : a.inv + cg.srow;
    int32_t sp = (int32_t)a.stride;  // a chunk's stack holds below 2^31 words (make_plan)
    uint64_t x = kStateL;
    uint32_t flags = 0;
    // p0 % D (the group's first channel), stepped down by 8 G mod D a group
    const uint32_t dstep = (8u * (uint32_t)G) % D;
    uint32_t pmod = max_groups
                        ? (8u * ((uint32_t)ell + (uint32_t)G * (max_groups - 1u))) % D : 0u;
    // symbols per pass over a group: the encoder with the ideal bits inside
    // codes each group in two halves, so that its unrolled body, twice the
    // plain encoder's, stays in the instruction cache (193.9 against 177.7
    // GB/s on the Qwen3-32B shape); the multi-round bf16 encoder gains a
    // little from them too (260.6 against 258.4), the 768-thread ones lose
    // (Qwen3-0.6B 247.8 against 252.4, Qwen3-8B e4m3 155.5 against 161.4)
    constexpr int KH = BITS || NT > kCodeThreads ? 4 : 8;
    for (int64_t gi = (int64_t)max_groups - 1; gi >= 0;
         --gi, pmod = pmod >= dstep ? pmod - dstep : pmod + D - dstep) {
      const bool has = (uint32_t)gi < my_groups;
      const uint32_t p0g = 8u * ((uint32_t)ell + (uint32_t)G * (uint32_t)gi);
      const uint32_t ch0 = pmod;
#pragma unroll 1
      for (int hh = 8 / KH - 1; hh >= 0; --hh) {
        const uint32_t p0 = p0g + (uint32_t)(KH * hh);  // a group never crosses a row of D
        uint32_t sym[KH], mub[KH];
        ChanInv inv[KH];
        float bk[KH];
        if (has) {
          load_syms<DT>(a.kv, cg.base + p0, sym);
          if (!O0) {
            load_mu(a.mu, cg.base + p0, mub);
            load_inv(invrow, ch0 + (uint32_t)(KH * hh), inv);
          }
        }
#pragma unroll
        for (int k = KH - 1; k >= 0; --k) {
          uint32_t cst = 0, f = 1;
          bool emit = false;
          if (has) {
            int32_t r = DT == 0 ? rank_bf16(sym[k]) : rank_e4m3(sym[k]);
            if (r < 0 || r >= NS) {
              flags |= kFlagSymbol;
              r = 0;
            }
            if (O0) {
              cst = cum_order0(r, ecdf);
              f = cum_order0(r + 1, ecdf) - cst;
            } else {
              if (!mu_valid(mub[k])) {
                flags |= kFlagParam;
                mub[k] = 0;
              }
              const float muf = bf16_to_f32(mub[k]);
              cst = cum_of<DT>(r, muf, inv[k], s_phi, s_lo8, a.ecdf);
              f = cum_of<DT>(r + 1, muf, inv[k], s_phi, s_lo8, a.ecdf) - cst;
              if (BITS) {
                const float lo = lo_bf16(r), hi = lo_bf16(r + 1), ph = __ldg(a.phat + r);
                if (!ideal::ideal_series_bf16(lo, hi, muf, inv[k].s, ph, bk[k]))
                  bk[k] = ideal::ideal_rare_bf16(lo, hi, muf, inv[k].s, ph, a.log2q);
              }
            }
            // x >= f 2^(63 - M), a multiple of 2^32: a test of x's high word
            emit = (uint32_t)(x >> 32) >= (f << (31 - M));
          } else if (BITS) {
            bk[k] = 0.0f;
          }
          const uint32_t m = __ballot_sync(0xFFFFFFFFu, emit) & seg;
          const int n = __popc(m);
          if (emit) {
            const int32_t idx = sp - n + __popc(m & lt);
            if (idx >= 0) region[idx] = (uint32_t)x;
            else flags |= kFlagOverflow;
            x >>= 32;
          }
          sp -= n;
          if (has) {
            uint64_t rem;
            const uint64_t q = divmod_u64<M>(x, f, rem);
            x = (q << M) + rem + cst;
          }
        }
        if (BITS) {
          if (has) {
            float part = 0.0f;
#pragma unroll
            for (int k = 0; k < KH; ++k) part += bk[k];
            bacc += (double)part;
            if (a.bits_out) {
              float4 *o = reinterpret_cast<float4 *>(a.bits_out + cg.base + p0);
#pragma unroll
              for (int k = 0; k < KH; k += 4) o[k / 4] = make_float4(bk[k], bk[k + 1], bk[k + 2], bk[k + 3]);
            }
          }
        }
      }
    }
    if (live) {
      const int64_t at = sp - 2 * G + 2 * ell;
      if (at >= 0) {
        region[at] = (uint32_t)x;
        region[at + 1] = (uint32_t)(x >> 32);
      } else {
        flags |= kFlagOverflow;
      }
      // the scale words open the chunk, ahead of the lane states
      const int64_t s0 = sp - 2 * G - a.nsw;
      for (int j = ell; j < a.nsw; j += G) {
        if (s0 + j >= 0) region[s0 + j] = a.scale_words[(uint64_t)c * a.nsw + j];
        else flags |= kFlagOverflow;
      }
      if (ell == 0) {
        const int64_t start = s0 < 0 ? 0 : s0;
        a.starts[c] = (uint32_t)start;
        a.sizes[c] = 4ull * (uint64_t)(a.stride - start);
        atomicAdd(&a.head->chunks_done, 1ull);
      }
    }
    if (flags) atomicOr(&a.head->flags, flags);
  }
  if (BITS) {
    // fixed order: a shuffle tree per warp, then the warps in order
    for (int o = 16; o; o >>= 1) bacc += __shfl_xor_sync(0xFFFFFFFFu, bacc, o);
    if (lane == 0) s_bpart[threadIdx.x >> 5] = bacc;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += s_bpart[w];
      a.bits_partials[blockIdx.x] = t;
    }
  }
}

// ------------------------------------------------------------------------
// Model bits: the code length of the coder's own integer frequencies, the
// cost the rANS stream approaches (it adds at most 32 to 64 bits per lane for
// the initial state and the flush).
// ------------------------------------------------------------------------

// -log2(f / 2^M) of a frequency 1 <= f < 2^M in fp32: above half the range
// through log1p of the exact complement (a cost below one bit keeps its
// relative accuracy), else M - log2 f.
template <int M>
__device__ __forceinline__ float code_length(uint32_t f) {
  constexpr uint32_t one = 1u << M;
  if (f > one / 2) return -1.44269504f * log1pf(-(float)(one - f) * (1.0f / (float)one));
  return (float)M - log2f((float)f);
}

template <int DT, bool O0>
__global__ void __launch_bounds__(256) k_model_bits(ModelBitsLaunch a) {
  extern __shared__ uint2 s_phi[];
  float *s_lo8 = reinterpret_cast<float *>(s_phi + kPhiKnots);
  __shared__ double s_part[256];
  stage_tables(s_phi, s_lo8);
  constexpr int M = DT == 0 ? kMBf16 : kME4m3;
  constexpr int32_t NS = DT == 0 ? kNsymBf16 : kNsymE4m3;
  const uint64_t D = (uint64_t)a.geo.D, TD = (uint64_t)a.geo.T * D, cw = D * (uint64_t)a.geo.Tb;
  const int64_t n8 = a.geo.n / 8;
  double acc = 0.0;
  uint32_t flags = 0;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < n8;
       g += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t i0 = 8ull * (uint64_t)g;
    const uint64_t row = i0 / TD, in_row = i0 - row * TD;
    uint32_t sym[8], mub[8];
    ChanInv inv[8];
    load_syms<DT>(a.kv, i0, sym);
    if (!O0) {
      load_mu(a.mu, i0, mub);
      const float2 *ip = a.inv_chunk ? a.inv_chunk + (row * (uint64_t)a.geo.ntb + in_row / cw) * D
                                     : a.inv + row * D;
      load_inv(ip, in_row % D, inv);
    }
    float bits[8], part = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      int32_t r = DT == 0 ? rank_bf16(sym[k]) : rank_e4m3(sym[k]);
      if (r < 0 || r >= NS) {
        flags |= kFlagSymbol;
        r = 0;
      }
      uint32_t c0, c1;
      if (O0) {
        c0 = cum_order0(r, a.ecdf);
        c1 = cum_order0(r + 1, a.ecdf);
      } else {
        if (!mu_valid(mub[k])) {
          flags |= kFlagParam;
          mub[k] = 0;
        }
        const float muf = bf16_to_f32(mub[k]);
        c0 = cum_of<DT>(r, muf, inv[k], s_phi, s_lo8, a.ecdf);
        c1 = cum_of<DT>(r + 1, muf, inv[k], s_phi, s_lo8, a.ecdf);
      }
      bits[k] = code_length<M>(c1 - c0);
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

template <int DT, bool O0>
static cudaError_t run_model_bits(const ModelBitsLaunch &a, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k_model_bits<DT, O0>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kCodeSmem);
  if (e != cudaSuccess) return e;
  k_model_bits<DT, O0><<<a.nblocks, 256, kCodeSmem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_model_bits(const ModelBitsLaunch &a, cudaStream_t s) {
  cudaError_t e;
  if (a.dtype == 0 && a.order0) e = run_model_bits<0, true>(a, s);
  else if (a.dtype == 0) e = run_model_bits<0, false>(a, s);
  else e = run_model_bits<1, false>(a, s);
  if (e != cudaSuccess) return e;
  return launch_ideal_final(a.partials, a.nblocks, a.head, s);
}

// ------------------------------------------------------------------------
// Exclusive scan of chunk sizes: block-local scans, then the block totals.
// ------------------------------------------------------------------------

__global__ void __launch_bounds__(256) k_scan_local(uint64_t *sizes, int64_t n,
                                                    uint64_t *partials) {
  __shared__ uint64_t s[256];
  const int64_t b0 = (int64_t)blockIdx.x * kScanBlock + threadIdx.x * 8;
  uint64_t v[8], sum = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    v[k] = b0 + k < n ? sizes[b0 + k] : 0;
    sum += v[k];
  }
  s[threadIdx.x] = sum;
  __syncthreads();
  for (int off = 1; off < 256; off <<= 1) {
    uint64_t t = threadIdx.x >= off ? s[threadIdx.x - off] : 0;
    __syncthreads();
    s[threadIdx.x] += t;
    __syncthreads();
  }
  uint64_t excl = s[threadIdx.x] - sum;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (b0 + k < n) sizes[b0 + k] = excl;  // in place: block-local exclusive offset
    excl += v[k];
  }
  if (threadIdx.x == 255) partials[blockIdx.x] = s[255];
}

__global__ void __launch_bounds__(1024) k_scan_partials(uint64_t *partials, int64_t nb,
                                                        WsHead *head) {
  __shared__ uint64_t s[1024];
  uint64_t carry = 0;
  for (int64_t b0 = 0; b0 < nb; b0 += 1024) {
    const int64_t i = b0 + threadIdx.x;
    const uint64_t v = i < nb ? partials[i] : 0;
    s[threadIdx.x] = v;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      uint64_t t = threadIdx.x >= off ? s[threadIdx.x - off] : 0;
      __syncthreads();
      s[threadIdx.x] += t;
      __syncthreads();
    }
    if (i < nb) partials[i] = carry + s[threadIdx.x] - v;
    carry += s[1023];
    __syncthreads();
  }
  if (threadIdx.x == 0) head->total = carry;
}

// ------------------------------------------------------------------------
// Compaction into the container: header | offsets | payload.
// ------------------------------------------------------------------------

// Copies nw words from a chunk's stack to its place in the container with the
// lanes of a warp, four loads in flight per lane before their stores (a
// chunk's offsets are only word-aligned, so the copy moves words).
__device__ __forceinline__ void warp_copy_words(uint32_t *dst, const uint32_t *src, int64_t nw,
                                                int lane) {
  int64_t k = lane;
  for (; k + 96 < nw; k += 128) {
    const uint32_t v0 = src[k], v1 = src[k + 32], v2 = src[k + 64], v3 = src[k + 96];
    dst[k] = v0;
    dst[k + 32] = v1;
    dst[k + 64] = v2;
    dst[k + 96] = v3;
  }
  for (; k < nw; k += 32) dst[k] = src[k];
}

__global__ void __launch_bounds__(256) k_compact(EncodeLaunch a) {
  const uint64_t total = a.head->total;
  const int64_t nc = a.geo.nchunks;
  const uint64_t hbytes = 64 + 8 * (uint64_t)(nc + 1);
  if (hbytes + total > a.capacity) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&a.head->flags, kFlagCapacity);
    return;
  }
  uint64_t *offs = reinterpret_cast<uint64_t *>(a.out + 64);
  uint32_t *payload = reinterpret_cast<uint32_t *>(a.out + hbytes);
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t c = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); c < nc;
       c += nwarps) {
    const uint64_t off = a.sizes[c] + a.partials[c / kScanBlock];
    const int64_t start = a.starts[c];
    const int64_t nw = a.stride - start;
    const uint32_t *src = a.scratch + c * a.stride + start;
    warp_copy_words(payload + off / 4, src, nw, lane);
    if (lane == 0) offs[c] = off;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    offs[nc] = total;
    uint8_t h[64];
    make_header(h, a.geo, a.dtype, total, mix64(a.head->hash_acc ^ a.hash_words),
                (a.nsw > 0 ? 1u : 0u) | (a.order0 ? 2u : 0u) | (a.adaptive ? 4u : 0u));
    for (int i = 0; i < 64; ++i) a.out[i] = h[i];
  }
}

// Incremental compaction (skv_encode_commit).  The sizes of the range's chunks
// are scanned in place by k_scan_local (block-local offsets, block sums in
// partials[0 ..]); k_commit_partials turns the block sums into offsets after
// the payload committed before and records the new prefix; k_commit_compact
// copies the chunks' stacks.  A range that does not start where the committed
// prefix ends is an argument error and nothing is placed.  The chunk after the
// range gets its offset now (the range's end), so the range can be decoded
// before the next commit; that commit writes the same value again.
__global__ void __launch_bounds__(1024) k_commit_partials(EncodeLaunch a, int64_t nb,
                                                           uint64_t *end_bytes) {
  __shared__ uint64_t s[1024];
  const bool in_order = a.head->committed == (unsigned long long)a.c_first;
  uint64_t carry = a.head->commit_total;
  for (int64_t b0 = 0; b0 < nb; b0 += 1024) {
    const int64_t i = b0 + threadIdx.x;
    const uint64_t v = i < nb ? a.partials[i] : 0;
    s[threadIdx.x] = v;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      uint64_t t = threadIdx.x >= off ? s[threadIdx.x - off] : 0;
      __syncthreads();
      s[threadIdx.x] += t;
      __syncthreads();
    }
    if (i < nb) a.partials[i] = carry + s[threadIdx.x] - v;
    carry += s[1023];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int64_t c_end = a.c_first + a.c_count;
    const uint64_t hbytes = 64 + 8 * (uint64_t)(a.geo.nchunks + 1);
    if (!in_order) {
      atomicOr(&a.head->flags, kFlagArg);
    } else if (hbytes + carry > a.capacity) {
      atomicOr(&a.head->flags, kFlagCapacity);
    } else {
      reinterpret_cast<uint64_t *>(a.out + 64)[c_end] = carry;
      a.head->commit_total = carry;
      a.head->committed = (unsigned long long)c_end;
    }
    if (end_bytes) *end_bytes = hbytes + a.head->commit_total;
  }
}

__global__ void __launch_bounds__(256) k_commit_compact(EncodeLaunch a) {
  // an out-of-order range or a full container: k_commit_partials has flagged it
  if (a.head->committed != (unsigned long long)(a.c_first + a.c_count)) return;
  const uint64_t hbytes = 64 + 8 * (uint64_t)(a.geo.nchunks + 1);
  uint64_t *offs = reinterpret_cast<uint64_t *>(a.out + 64);
  uint32_t *payload = reinterpret_cast<uint32_t *>(a.out + hbytes);
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < a.c_count;
       i += nwarps) {
    const int64_t c = a.c_first + i;
    const uint64_t off = a.sizes[c] + a.partials[i / kScanBlock];
    const uint32_t start = a.starts[c];
    // a chunk not encoded since SKV_RANGE_FIRST still holds the sentinel start
    if (start > a.stride) {
      if (lane == 0) atomicOr(&a.head->flags, kFlagArg);
      continue;
    }
    const int64_t nw = a.stride - start;
    if (hbytes + off + 4 * (uint64_t)nw > a.capacity) {  // only if sizes and starts disagree
      if (lane == 0) atomicOr(&a.head->flags, kFlagArg);
      continue;
    }
    const uint32_t *src = a.scratch + c * a.stride + start;
    warp_copy_words(payload + off / 4, src, nw, lane);
    if (lane == 0) offs[c] = off;
  }
}

// The header of a container placed by commits, once every chunk is committed.
__global__ void k_commit_header(EncodeLaunch a) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const int64_t nc = a.geo.nchunks;
  if (a.head->committed != (unsigned long long)nc) {
    atomicOr(&a.head->flags, kFlagArg);
    return;
  }
  const uint64_t total = a.head->commit_total;
  a.head->total = total;
  uint8_t h[64];
  make_header(h, a.geo, a.dtype, total, mix64(a.head->hash_acc ^ a.hash_words),
              (a.nsw > 0 ? 1u : 0u) | (a.order0 ? 2u : 0u) | (a.adaptive ? 4u : 0u));
  for (int i = 0; i < 64; ++i) a.out[i] = h[i];
  reinterpret_cast<uint64_t *>(a.out + 64)[0] = 0;
}

// Grid for ntasks >= 1 warp tasks of a coder kernel (blocks of at most
// max_threads, at most one block per SM).  A lane's symbols are coded one after
// another, so a launch takes at least one lane's chain of steps, and a step is
// several times shorter on an SM running a few warps than on one whose 24
// warps contend for issue slots (one lane's 2048-symbol chunk: about 1.9 ms
// alone, 4 ms on a full SM).  A launch too small to fill an eighth of the SMs
// with full blocks (a chunk range of up to ~900 chunks of 16 lanes, one token
// block of the adaptive coder) therefore spreads over all SMs with fewer warps
// per block.  Larger launches keep full blocks on as few SMs as they need, so
// that launches on other streams (a cache coded as four layer groups side by
// side: a quarter each) get SMs of their own rather than sharing theirs: a
// block holds 65-79 KiB of tables, so few fit per SM.
static void task_shape(int64_t ntasks, int max_threads, int &blocks, int &threads,
                       int multi_round_threads = 0) {
  const int64_t sms = (int64_t)device_sm_count();
  const int64_t wmax = max_threads / 32;
  if (multi_round_threads > max_threads && ntasks > sms * wmax) {
    // more tasks than one round of full blocks: larger blocks where they fit
    blocks = (int)sms;
    threads = multi_round_threads;
    return;
  }
  if (8 * ntasks >= sms * wmax) {
    const int64_t want = (ntasks + wmax - 1) / wmax;
    blocks = (int)(want < sms ? want : sms);
    threads = max_threads;
    return;
  }
  const int64_t wpb = (ntasks + sms - 1) / sms;  // 1 .. wmax / 8
  threads = (int)(32 * wpb);
  blocks = (int)((ntasks + wpb - 1) / wpb);
}

cudaError_t launch_encode(const EncodeLaunch &a, cudaStream_t s) {
  cudaError_t e = launch_encode_chunks(a, s);
  if (e != cudaSuccess) return e;
  return launch_encode_finish(a, s);
}

template <int DT, bool O0, int NT, bool BITS = false>
static cudaError_t run_encode(const EncodeLaunch &a, int blocks, int threads, cudaStream_t s) {
  cudaError_t e;
  if (BITS) {
    if (blocks > kMaxBitsBlocks) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(k_encode<DT, O0, NT, BITS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kCodeSmem);
    if (e != cudaSuccess) return e;
    k_encode<DT, O0, NT, BITS><<<blocks, threads, kCodeSmem, s>>>(a);
    return cudaGetLastError();
  }
  e = cudaFuncSetAttribute(k_encode<DT, O0, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kCodeSmem);
  if (e != cudaSuccess) return e;
  k_encode<DT, O0, NT><<<blocks, threads, kCodeSmem, s>>>(a);
  return cudaGetLastError();
}

// bf16 encode launches with more tasks than one round of 768-thread blocks
// run 896-thread blocks (72 registers instead of 78): 32B shape encode 197 ->
// 208 GB/s.  Single-round launches (the 0.6B shape: 209 -> 200) lose with
// them and keep 768.  e4m3 multi-round launches run 1024-thread blocks with
// their groups coded in halves (58 registers; see launch_encode_chunks).
constexpr int kEncMultiRoundThreads = 896;
constexpr int kEncMultiRoundThreadsE4m3 = 1024;

// The ideal bits ride along with the bf16 mixture encoder, whatever the
// launch's size and with or without per-block scales: the series' extra work
// per scalar costs less than a separate pass re-reading kv and mu (Qwen3-32B
// shape: 10.9 ms fused against 8.1 + 4.8 ms; Qwen3-0.6B shape, one round of
// tasks, where it fills issue slots the lanes' serial chains leave idle: step
// +5.4%; with per-block scales +6.5% and +9.7%), now that the scalars
// outside the series take the tail table and each group is coded in halves.
// It costs caches whose model fits badly, where most warp steps hold such
// scalars (the drift workload: step -4.5% with the static sigma, -4.6% with
// per-block scales).  e4m3's rare scalars, several per warp step, stall whole
// warps (8B shape: 32 against 7.7 + 5.6 ms), and the order-0 coder has no
// series: those run the two kernels.
bool encode_fuses_bits(int dtype, bool order0, bool scaled, int64_t chunks, int G) {
  (void)scaled;
  return dtype == 0 && !order0 && chunks > 0 && G > 0;
}

cudaError_t launch_encode_chunks(const EncodeLaunch &a, cudaStream_t s) {
  const int64_t ntasks = (a.c_count * a.geo.G + 31) / 32;
  if (ntasks == 0) return cudaSuccess;
  int blocks, threads;
  if (a.dtype == 0 && a.order0) {
    task_shape(ntasks, kCodeThreads, blocks, threads);
    return run_encode<0, true, kCodeThreads>(a, blocks, threads, s);
  }
  if (a.dtype == 0) {
    task_shape(ntasks, kCodeThreads, blocks, threads, kEncMultiRoundThreads);
    if (a.bits_partials) {
      // skv_encode_with_bits and chunk ranges with their bits; launches of one
      // round of tasks run a 768-bound instantiation (77 registers against
      // 71: Qwen3-0.6B shape encode with bits 179.5 -> 181.0 GB/s)
      if (a.order0) return cudaErrorInvalidValue;
      if (threads <= kCodeThreads)
        return run_encode<0, false, kCodeThreads, true>(a, blocks, threads, s);
      return run_encode<0, false, kEncMultiRoundThreads, true>(a, blocks, threads, s);
    }
    if (threads > kCodeThreads)
      return run_encode<0, false, kEncMultiRoundThreads>(a, blocks, threads, s);
    return run_encode<0, false, kCodeThreads>(a, blocks, threads, s);
  }
  if (a.bits_partials) return cudaErrorInvalidValue;
  // e4m3 launches of several rounds: 1024-thread blocks, groups coded in
  // halves (58 registers): Qwen3-8B shape encode 162.3 -> 191.9 GB/s (whole
  // groups in 896-thread blocks had lost, 157 -> 140)
  task_shape(ntasks, kCodeThreads, blocks, threads, kEncMultiRoundThreadsE4m3);
  if (threads > kCodeThreads)
    return run_encode<1, false, kEncMultiRoundThreadsE4m3>(a, blocks, threads, s);
  return run_encode<1, false, kCodeThreads>(a, blocks, threads, s);
}

cudaError_t launch_encode_commit(const EncodeLaunch &a, uint64_t *end_bytes, cudaStream_t s) {
  cudaError_t e;
  const int64_t nb = (a.c_count + kScanBlock - 1) / kScanBlock;
  if (nb > 0) {
    k_scan_local<<<(unsigned)nb, 256, 0, s>>>(a.sizes + a.c_first, a.c_count, a.partials);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  k_commit_partials<<<1, 1024, 0, s>>>(a, nb, end_bytes);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.c_count <= 0) return cudaSuccess;
  int64_t cblocks = (a.c_count + 7) / 8;
  if (cblocks > (int64_t)device_sm_count() * 16) cblocks = (int64_t)device_sm_count() * 16;
  k_commit_compact<<<(unsigned)cblocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_commit_header(const EncodeLaunch &a, cudaStream_t s) {
  k_commit_header<<<1, 32, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_encode_finish(const EncodeLaunch &a, cudaStream_t s) {
  cudaError_t e;
  const int64_t nb = (a.geo.nchunks + kScanBlock - 1) / kScanBlock;
  k_scan_local<<<(unsigned)nb, 256, 0, s>>>(a.sizes, a.geo.nchunks, a.partials);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_scan_partials<<<1, 1024, 0, s>>>(a.partials, nb, a.head);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  int64_t cblocks = (a.geo.nchunks + 7) / 8;
  if (cblocks > (int64_t)device_sm_count() * 16) cblocks = (int64_t)device_sm_count() * 16;
  k_compact<<<(unsigned)cblocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------
// Decode
// ------------------------------------------------------------------------

__device__ __forceinline__ uint64_t get_u64(const uint8_t *p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}

// Header, fingerprint and offset-table ends; per-chunk offsets are checked by
// the decode kernel itself.
__global__ void k_check_header(DecodeLaunch a) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const int64_t nc = a.geo.nchunks;
  const uint64_t hbytes = 64 + 8 * (uint64_t)(nc + 1);
  const uint64_t payload = a.in_bytes - hbytes;
  uint8_t want[64];
  make_header(want, a.geo, a.dtype, payload, mix64(a.head->hash_acc ^ a.hash_words),
              (a.nsw > 0 ? 1u : 0u) | (a.order0 ? 2u : 0u) | (a.adaptive ? 4u : 0u));
  bool ok = true;
  for (int i = 0; i < 64; ++i) ok &= a.in[i] == want[i];
  ok &= get_u64(a.in + 64) == 0;
  ok &= get_u64(a.in + 64 + 8 * (uint64_t)nc) == payload;
  if (!ok) atomicOr(&a.head->flags, kFlagCorrupt);
}

// One symbol's search state: the answer r satisfies lo <= r < hi, with
// clo = cum(lo) <= slot < chi = cum(hi); done when hi = lo + 1.
struct Bracket {
  int32_t lo, hi;
  uint32_t clo, chi;
};

// Narrows the bracket with cum(r) = c (never widens it).
__device__ __forceinline__ void bracket_add(Bracket &b, int32_t r, uint32_t c, uint32_t slot) {
  if (c <= slot) {
    if (r > b.lo) {
      b.lo = r;
      b.clo = c;
    }
  } else if (r < b.hi) {
    b.hi = r;
    b.chi = c;
  }
}

__device__ __forceinline__ float lo_value(int DT, int32_t r, const float *lo8) {
  return DT == 0 ? lo_bf16(r) : lo8[r];
}

// Position of the n-th (from 0) set bit of m; m has more than n set bits.
__device__ __forceinline__ int nth_set_bit(uint32_t m, int n) {
  int pos = 0;
#pragma unroll
  for (int w = 16; w; w >>= 1) {
    const int c = __popc(m & ((1u << w) - 1u));
    if (n >= c) {
      n -= c;
      m >>= w;
      pos += w;
    }
  }
  return pos;
}

// The warp search's first-round distances from a bracket end, j = 0 .. 15:
// 1, 2, 3, 4, 6, 8, 12, 16, ..., 192, 256.
__device__ __forceinline__ int32_t ladder_step(int j) {
  return j < 4 ? j + 1 : (3 + ((j - 4) & 1)) << (((j - 4) >> 1) + 1);
}

// Rank of the symbol an fp32 value rounds to (the decoder's guesses only).
template <int DT>
__device__ __forceinline__ int32_t rank_of_value(float x) {
  if (DT == 0) {
    const uint32_t u = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
    // a NaN rounds to a NaN pattern, whose key lies outside [0, |S|): the
    // unsigned clamp sends both signs to the last rank (a guess, still in range)
    return (int32_t)min((uint32_t)rank_bf16(u), (uint32_t)(kNsymBf16 - 1));
  }
  const uint32_t u = (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
  const int32_t r = rank_e4m3(u);
  return r < 0 ? 0 : r;
}

// Decode.  Per symbol: slot = x mod 2^M; find r with cum(r) <= slot < cum(r+1);
// x = freq * (x >> M) + slot - cum(r); refill from the stream if x < 2^31.
// Reference search (bisect): 16 (bf16) or 8 (e4m3) cum evaluations.  Default
// search: (1) a guess from the inverted Gaussian part of the model CDF,
// verified with cum(r), cum(r+1); (2) if it missed, one Newton step in value
// space with that bin's exact density, verified the same way; (3) lanes still
// unresolved are finished one at a time by the whole warp, 32 candidates per
// step: first 16 stepping inwards from each end of the lane's bracket (its
// answer is usually close to one of them), then evenly spread.  Every answer
// is checked by the exact cum bracket, so both searches return the same symbol.
// First scalar of chunk c in mu and in the output: its place in the
// [L][2][H][T][D] tensor, or its page in a page pool (then an out-of-range
// page index is an argument error and the chunk is skipped).
__device__ __forceinline__ uint64_t chunk_out_base(const DecodeLaunch &a, int64_t c, bool &ok,
                                                   uint32_t &flags) {
  if (!a.page_of_chunk) return chunk_geo(a.geo, c < a.c_end ? c : 0).base;
  if (!ok) return 0;
  const uint32_t pg = a.page_of_chunk[c];
  if ((uint64_t)pg >= a.num_pages) {
    flags |= kFlagArg;
    ok = false;
    return 0;
  }
  return (uint64_t)pg * a.page_scalars;
}

// The warp's next task: after a first round in grid order, tasks go to whichever
// warp is free first, so a few slow chunks (their search work depends on how
// well the model fits) do not leave the rest of the GPU idle.  Called by all
// lanes of the warp.
__device__ __forceinline__ int64_t next_task(WsHead *h, int64_t nwarps) {
  unsigned long long t = 0;
  if ((threadIdx.x & 31) == 0) t = atomicAdd(&h->next_task, 1ull);
  return nwarps + (int64_t)__shfl_sync(0xFFFFFFFFu, t, 0);
}

// The decoder's warp search for open lane l (all 32 lanes call it): 32
// candidates per round.  On a wide bracket the first round steps inwards from
// both ends, 16 candidates each, 1, 2, 3, 4, 6, 8, 12, ..., 192, 256 ranks
// away: the answer lies next to one of them far more often than in the middle
// (after Newton within 256 ranks of an end for ~96% of lanes, within one rank
// for ~30%).  Later rounds spread the candidates evenly (33 subintervals: at
// most 4 more rounds).  Leaves lane l's bracket in blo .. bchi (all lanes),
// one rank wide unless cum were not monotone.
template <int DT>
__device__ __forceinline__ void search_lane(int l, uint32_t slot, float muf, ChanInv inv,
                                            const Bracket &br, const uint2 *s_phi,
                                            const float *s_lo8, const uint32_t *__restrict__ ecdf,
                                            int32_t &blo, int32_t &bhi, uint32_t &bclo,
                                            uint32_t &bchi) {
  const int lane = threadIdx.x & 31;
  const uint32_t s_slot = __shfl_sync(0xFFFFFFFFu, slot, l);
  const float s_mu = __shfl_sync(0xFFFFFFFFu, muf, l);
  ChanInv s_inv;
  s_inv.s = __shfl_sync(0xFFFFFFFFu, inv.s, l);
  s_inv.s3 = __shfl_sync(0xFFFFFFFFu, inv.s3, l);
  blo = __shfl_sync(0xFFFFFFFFu, br.lo, l);
  bhi = __shfl_sync(0xFFFFFFFFu, br.hi, l);
  bclo = __shfl_sync(0xFFFFFFFFu, br.clo, l);
  bchi = __shfl_sync(0xFFFFFFFFu, br.chi, l);
  for (int it = 0; it < 12 && bhi - blo > 1; ++it) {
    const int32_t wdt = bhi - blo;
    const int32_t nact = min(wdt - 1, 32);
    int32_t cand;
    if (wdt - 1 <= 32) {
      cand = blo + 1 + lane;
    } else if (it == 0 && wdt > 2 * 256 + 1) {
      cand = lane < 16 ? blo + ladder_step(lane) : bhi - ladder_step(31 - lane);
    } else {
      // (lane + 1) wdt < 32 * 65283: 32-bit
      cand = blo + (int32_t)(((uint32_t)(lane + 1) * (uint32_t)wdt) / 33u);
    }
    const bool act = lane < nact;
    const uint32_t cv = act ? cum_of<DT>(cand, s_mu, s_inv, s_phi, s_lo8, ecdf) : 0u;
    const int kle = __popc(__ballot_sync(0xFFFFFFFFu, act && cv <= s_slot));
    const int32_t c_lo = __shfl_sync(0xFFFFFFFFu, cand, kle > 0 ? kle - 1 : 0);
    const uint32_t v_lo = __shfl_sync(0xFFFFFFFFu, cv, kle > 0 ? kle - 1 : 0);
    const int32_t c_hi = __shfl_sync(0xFFFFFFFFu, cand, kle < nact ? kle : 0);
    const uint32_t v_hi = __shfl_sync(0xFFFFFFFFu, cv, kle < nact ? kle : 0);
    if (kle > 0) {
      blo = c_lo;
      bclo = v_lo;
    }
    if (kle < nact) {
      bhi = c_hi;
      bchi = v_hi;
    }
  }
}

// The same for two or more open lanes of a warp step (all 32 lanes call it),
// side by side: up to kp = 2, 4, 8 or 16 open lanes at a time, each in a
// segment of S = 32 / kp lanes that tries S candidates per round -- on a wide
// bracket first every (16 / (S / 2))-th step of the ladder above, then S
// candidates evenly spread (S + 1 subintervals a round: at most 11 rounds after
// the first for S = 2).  Each open lane gets back its bracket.  Out of line:
// it runs in few warp steps except where the model fits badly, and inlined
// its code slowed every step of the rest.
template <int DT>
static __device__ __noinline__ Bracket search_lanes(uint32_t pend, bool mine_open, uint32_t slot,
                                                    float muf, ChanInv inv, Bracket br,
                                                    const uint2 *s_phi, const float *s_lo8,
                                                    const uint32_t *__restrict__ ecdf) {
  const int lane = threadIdx.x & 31;
  const int npend = __popc(pend);
  const int lg_kp = npend <= 2 ? 1 : (npend <= 4 ? 2 : (npend <= 8 ? 3 : 4));
  const int lg_s = 5 - lg_kp;
  const int S = 1 << lg_s, half = S >> 1;
  const int sgi = lane >> lg_s, j = lane & (S - 1);
  const int sbase = sgi << lg_s;  // first lane of my segment
  const uint32_t smask = (1u << S) - 1u;
  const int myord = __popc(pend & ((1u << lane) - 1u));  // my place among the open lanes
  // floor(n / (S + 1)) = umulhi(n, ceil(2^32 / (S + 1))) for n < 2^27 (the
  // error n (m (S + 1) - 2^32) / 2^32 stays below 1 / (S + 1)); here n =
  // (j + 1) wdt < 16 * 65283
  const uint32_t inv_s1 = 0xFFFFFFFFu / (uint32_t)(S + 1) + 1u;
  for (int b0 = 0; b0 < npend; b0 += 1 << lg_kp) {
    const bool valid = b0 + sgi < npend;
    const int src = valid ? nth_set_bit(pend, b0 + sgi) : lane;
    const uint32_t s_slot = __shfl_sync(0xFFFFFFFFu, slot, src);
    const float s_mu = __shfl_sync(0xFFFFFFFFu, muf, src);
    ChanInv s_inv;
    s_inv.s = __shfl_sync(0xFFFFFFFFu, inv.s, src);
    s_inv.s3 = __shfl_sync(0xFFFFFFFFu, inv.s3, src);
    int32_t blo = __shfl_sync(0xFFFFFFFFu, br.lo, src);
    int32_t bhi = __shfl_sync(0xFFFFFFFFu, br.hi, src);
    uint32_t bclo = __shfl_sync(0xFFFFFFFFu, br.clo, src);
    uint32_t bchi = __shfl_sync(0xFFFFFFFFu, br.chi, src);
    for (int it = 0; it < 24; ++it) {
      const bool open = valid && bhi - blo > 1;
      if (!__any_sync(0xFFFFFFFFu, open)) break;
      const int32_t wdt = bhi - blo;
      const int32_t nact = open ? min(wdt - 1, S) : 0;
      int32_t cand;
      if (wdt - 1 <= S) {
        cand = blo + 1 + j;
      } else if (it == 0 && wdt > 2 * 256 + 1) {
        const int jj = j < half ? j : S - 1 - j;
        const int32_t g = ladder_step(((jj + 1) << (5 - lg_s)) - 1);
        cand = j < half ? blo + g : bhi - g;
      } else {
        cand = blo + (int32_t)__umulhi((uint32_t)(j + 1) * (uint32_t)wdt, inv_s1);
      }
      const bool act = j < nact;
      const uint32_t cv = act ? cum_of<DT>(cand, s_mu, s_inv, s_phi, s_lo8, ecdf) : 0u;
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, act && cv <= s_slot);
      const int kle = __popc((bal >> sbase) & smask);
      const int32_t c_lo = __shfl_sync(0xFFFFFFFFu, cand, sbase + (kle > 0 ? kle - 1 : 0));
      const uint32_t v_lo = __shfl_sync(0xFFFFFFFFu, cv, sbase + (kle > 0 ? kle - 1 : 0));
      const int32_t c_hi = __shfl_sync(0xFFFFFFFFu, cand, sbase + (kle < nact ? kle : 0));
      const uint32_t v_hi = __shfl_sync(0xFFFFFFFFu, cv, sbase + (kle < nact ? kle : 0));
      if (open && kle > 0) {
        blo = c_lo;
        bclo = v_lo;
      }
      if (open && kle < nact) {
        bhi = c_hi;
        bchi = v_hi;
      }
    }
    // each open lane of this batch takes its segment's bracket
    const bool mine = mine_open && myord >= b0 && myord < b0 + (1 << lg_kp);
    const int from = mine ? (myord - b0) << lg_s : lane;
    const int32_t r_lo = __shfl_sync(0xFFFFFFFFu, blo, from);
    const int32_t r_hi = __shfl_sync(0xFFFFFFFFu, bhi, from);
    const uint32_t r_clo = __shfl_sync(0xFFFFFFFFu, bclo, from);
    const uint32_t r_chi = __shfl_sync(0xFFFFFFFFu, bchi, from);
    if (mine) {
      br.lo = r_lo;
      br.hi = r_hi;
      br.clo = r_clo;
      br.chi = r_chi;
    }
  }
  return br;
}

template <int DT, bool BISECT, int NT = dec_threads_max<DT>()>
__global__ void __launch_bounds__(NT, 1) k_decode(DecodeLaunch a) {
  extern __shared__ uint2 s_phi[];
  float *s_lo8 = reinterpret_cast<float *>(s_phi + kPhiKnots);
  float2 *s_hinv = reinterpret_cast<float2 *>(s_lo8 + 256);
  int32_t *s_einv = reinterpret_cast<int32_t *>(s_hinv + kHinvN + 1);
  for (int i = threadIdx.x; i < kPhiKnots; i += blockDim.x) s_phi[i] = g_phi[i];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) s_lo8[i] = g_lo8[i];
  for (int i = threadIdx.x; i <= kHinvN; i += blockDim.x) {
    s_hinv[i] = g_hinv[DT][i];
    s_einv[i] = (DT == 0 && a.einv) ? a.einv[i] : 0;
  }
  __syncthreads();

  constexpr int M = DT == 0 ? kMBf16 : kME4m3;
  constexpr int32_t NS = DT == 0 ? kNsymBf16 : kNsymE4m3;
  constexpr uint32_t kMask = (1u << M) - 1u;
  constexpr float kInvK = 1.0f / (float)(DT == 0 ? kKBf16 : kKE4m3);
  constexpr float kHscale = (float)kHinvN / (DT == 0 ? kHinvUmaxBf16 : kHinvUmaxE4m3);
  const int G = a.geo.G;
  const int lane = threadIdx.x & 31;
  const int ell = lane & (G - 1);
  const uint32_t seg = G == 32 ? 0xFFFFFFFFu : (((1u << G) - 1u) << (lane & ~(G - 1)));
  const uint32_t lt = seg & ((1u << lane) - 1u);
  const int64_t ntasks = (((a.c_end - a.c_begin + a.c_step - 1) / a.c_step) * G + 31) / 32;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const uint32_t D = (uint32_t)a.geo.D;
  const int64_t nc = a.geo.nchunks;
  const uint64_t hbytes = 64 + 8 * (uint64_t)(nc + 1);
  const uint64_t payload_bytes = a.in_bytes - hbytes;
  const uint8_t *payload = a.in + hbytes;

  for (int64_t task = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); task < ntasks;
       task = next_task(a.head, nwarps)) {
    const int64_t c = a.c_begin + a.c_step * ((task * 32 + lane) / G);
    const bool live = c < a.c_end;
    uint32_t flags = 0;
    uint64_t off_a = 0, off_b = 0;
    if (live) {
      const uint64_t *offs = reinterpret_cast<const uint64_t *>(a.in + 64);
      off_a = offs[c];
      off_b = offs[c + 1];
    }
    // both ends word-aligned (a misaligned word read would fault), inside the
    // payload; a chunk's words fit 32 bits (a full chunk holds below 2^31)
    bool ok = live && off_a <= off_b && off_b <= payload_bytes && ((off_a | off_b) & 3) == 0 &&
              (off_b - off_a) / 4 >= 2ull * G + (uint64_t)a.nsw && (off_b - off_a) / 4 < (1ull << 32);
    if (live && !ok) flags |= kFlagCorrupt;
    const uint64_t obase = chunk_out_base(a, c, ok, flags);  // mu and output
    const uint32_t *w = reinterpret_cast<const uint32_t *>(payload + (ok ? off_a : 0));
    const uint32_t nw = ok ? (uint32_t)((off_b - off_a) / 4) : 0u;
    ChunkGeo cg = chunk_geo(a.geo, live ? c : 0);
    const uint32_t my_groups =
        (ok && (uint32_t)ell < cg.ngroup) ? (cg.ngroup - ell + G - 1) / G : 0u;
    const uint32_t max_groups = __reduce_max_sync(0xFFFFFFFFu, my_groups);
    const uint32_t *ws0 = w + a.nsw;  // the lane states follow the scale words
    uint64_t x = ok ? ((uint64_t)ws0[2 * ell] | ((uint64_t)ws0[2 * ell + 1] << 32)) : kStateL;
    uint32_t cur = 2u * (uint32_t)G + (uint32_t)a.nsw;
    const float2 *invrow = a.inv_chunk ? a.inv_chunk + (uint64_t)(live ? c : 0) * D
                                       : a.inv + cg.srow;

    // p0 % D (the group's first channel), stepped up by 8 G mod D a group
    const uint32_t dstep = (8u * (uint32_t)G) % D;
    uint32_t pmod = (8u * (uint32_t)ell) % D;
    for (uint32_t gi = 0; gi < max_groups;
         ++gi, pmod = pmod + dstep >= D ? pmod + dstep - D : pmod + dstep) {
      const bool has = gi < my_groups;
      const uint32_t p0 = 8u * ((uint32_t)ell + (uint32_t)G * gi);
      const uint16_t *mup = a.mu + obase + p0;
      const float2 *ivp2 = invrow + pmod;
      uint64_t out_lo = 0, out_hi = 0;  // the group's 8 symbols, shifted in from the top
#pragma unroll 1
      for (int k = 0; k < 8; ++k) {
        uint32_t mub = has ? (uint32_t)__ldg(mup + k) : 0u;
        ChanInv inv;
        if (has) {
          const float2 v = __ldg(ivp2 + k);
          inv.s = v.x;
          inv.s3 = v.y;
        } else {
          inv.s = 1.0f;
          inv.s3 = 1.0f;
        }
        if (has && !mu_valid(mub)) {
          flags |= kFlagParam;
          mub = 0;
        }
        const float muf = bf16_to_f32(mub);
        const uint32_t slot = (uint32_t)x & kMask;
        Bracket br;
        br.lo = 0;
        br.hi = NS;
        br.clo = 0;
        br.chi = 1u << M;
        if (BISECT) {
          if (has) {
            int32_t r = 0;
#pragma unroll
            for (int step = DT == 0 ? (1 << 15) : (1 << 7); step >= 1; step >>= 1) {
              const int32_t cand = r + step;
              if (cand < NS) {
                const uint32_t cv = cum_of<DT>(cand, muf, inv, s_phi, s_lo8, a.ecdf);
                if (cv <= slot) {
                  r = cand;
                  br.clo = cv;
                } else {
                  br.chi = cv;
                }
              }
            }
            br.lo = r;
            br.hi = r + 1;
          }
        } else {
          bool done = true;
          if (has) {
            // (1) guess: invert the CDF's Gaussian part around a reference
            // symbol: slot ~ K F(x) + rank(x) with F = 0.95 Phi(z) + 0.03 Phi(z/3)
            // + 0.02 E(x), with rank and E taken at mu.  For e4m3, whose rank
            // term is up to 0.4% of the CDF, one step along the table's slope
            // then takes it at the first guess (for bf16 a second look mainly
            // helps through E at the guess, whose dependent load costs as much
            // as the Newton steps it saves).
            const float sig = __fdividef(1.0f, inv.s);  // a guess: approximate is enough
            // bf16: near mu the p-hat term grows about linearly in value,
            // E(x) ~ E(mu) + rho (x - mu) with rho the p-hat mass of mu's bin
            // per unit width (the width from mu's exponent: a guess needs no
            // more), so the guess solves G0(z) + a z = u with a = 0.02 rho sigma.
            // Without it the p-hat term at mu alone misses where bins are narrow
            // against sigma (values near zero): about 2 in 3 of the misses.
            // Both terms come from one per-rank entry (k_einv), in the guess
            // table's knot units: 0.02 E(mu), and 0.02 rho, taken times sigma here.
            float e_mu2 = 0.0f, a_knot = 0.0f;
            const int32_t rmu = DT == 0 ? rank_bf16(mub) : rank_of_value<DT>(muf);
            if (DT == 0) {
              const float2 g = __ldg(a.gmu + rmu);
              e_mu2 = g.x;
              a_knot = fminf(g.y * sig, kGuessSlopeMax);  // NaN (sigma NaN) gives the bound
            }
            auto guess = [&](int32_t rref) -> int32_t {
              const int32_t dr = (int32_t)(slot - (uint32_t)rref);
              // u = dr / K (bf16: less 0.02 E(mu)) in the table's knot units
              const float tu = DT == 0 ? fmaf((float)dr, kInvK * kHscale, -e_mu2)
                                       : (float)dr * (kInvK * kHscale);
              if (DT == 1) {
                // beyond both ends of Phi_q's range cum(r) = r (below mu) or
                // K + r (above): the rank follows from the slot directly.  Exact
                // integer tests: in fp32, K (1/K) rounds below 1.
                if (dr <= 0) return min((int32_t)slot, NS - 1);
                if (dr >= (int32_t)kKE4m3) return max(min((int32_t)slot - (int32_t)kKE4m3, NS - 1), 0);
              }
              const float t = fminf(fmaxf(tu, 0.0f), (float)kHinvN - 0.001f);
              const int kk = (int)t;
              const float2 h = s_hinv[kk];
              float z0 = fmaf(t - (float)kk, h.y, h.x);
              // the linear p-hat term: z0 / (1 + a dz/du), dz/du = h.y kHscale from
              // the table; it only moves the guess towards mu, never past it
              if (DT == 0) z0 = __fdividef(z0, fmaf(a_knot, h.y, 1.0f));
              int32_t r = rank_of_value<DT>(fmaf(sig, z0, muf));
              if (DT == 1) {
                // the rank term at the guess: u falls by (r - rref) / K, one step
                // along the table's slope dz/du = h.y kHscale
                const float dz = (float)(r - rref) * (kInvK * kHscale);
                r = rank_of_value<DT>(fmaf(sig, fmaf(-dz, h.y, z0), muf));
              }
              if (DT == 0 && (tu < 0.0f || tu > (float)kHinvN)) {
                // beyond both Gaussian parts only p-hat moves the CDF: invert it
                const float uraw = (float)dr * kInvK;
                const float tgt = (tu < 0.0f ? uraw : uraw - kHinvUmaxBf16) * (50.0f * kHinvN);
                const float te = fminf(fmaxf(tgt, 0.0f), (float)kHinvN - 0.001f);
                const int ke = (int)te;
                const int32_t r0 = s_einv[ke], r1 = s_einv[ke + 1];
                r = min(r0 + (int32_t)((te - (float)ke) * (float)(r1 - r0)), NS - 1);
              }
              return r;
            };
            const int32_t rg = guess(rmu);
            const uint32_t ca = cum_of<DT>(rg, muf, inv, s_phi, s_lo8, a.ecdf);
            const uint32_t cb = cum_of<DT>(rg + 1, muf, inv, s_phi, s_lo8, a.ecdf);
            // the guess's bracket [rg, rg + 1); on a miss, the full one cut by
            // these two points (cum(0) = 0, cum(|S|) = 2^M): below rg or above
            // rg + 1
            const bool at_lo = ca <= slot;
            br.lo = rg;
            br.hi = rg + 1;
            br.clo = ca;
            br.chi = cb;
            done = at_lo && slot < cb;
            if (!done) {
              if (!at_lo) {
                br.lo = 0;
                br.clo = 0u;
                br.hi = rg;
                br.chi = ca;
              } else {
                br.lo = rg + 1;
                br.clo = cb;
                br.hi = NS;
                br.chi = 1u << M;
              }
              // (2) Newton in value space with the density of bin rg
              const float blo = lo_value(DT, rg, s_lo8), bhi = lo_value(DT, rg + 1, s_lo8);
              const float dens_inv = __fdividef(bhi - blo, (float)(cb - ca));
              const float xn = slot < ca ? blo - (float)(ca - slot) * dens_inv
                                         : bhi + (float)(slot - cb) * dens_inv;
              int32_t sN = isfinite(xn) ? rank_of_value<DT>(xn) : (br.lo + br.hi) >> 1;
              sN = max(sN, br.lo);
              sN = min(sN, br.hi - 1);
              bool upper = true;
              if (sN > br.lo) {
                const uint32_t cs = cum_of<DT>(sN, muf, inv, s_phi, s_lo8, a.ecdf);
                bracket_add(br, sN, cs, slot);
                upper = cs <= slot;
              }
              if (upper && sN + 1 < br.hi) {
                const uint32_t cs1 = cum_of<DT>(sN + 1, muf, inv, s_phi, s_lo8, a.ecdf);
                bracket_add(br, sN + 1, cs1, slot);
              }
              done = br.hi - br.lo == 1;
            }
          }
          // (3) the warp finishes its unresolved lanes: one lane at a time with
          // all 32 candidates per round (search_lane), or (bf16) two or more
          // side by side (search_lanes), so that a warp whose chunks fit the
          // model badly (many lanes open in one step) does not finish them one
          // after another
          uint32_t pend = __ballot_sync(0xFFFFFFFFu, !done);
          if constexpr (DT == 0) {
            if (__popc(pend) == 1) {
              const int l = __ffs(pend) - 1;
              int32_t blo, bhi;
              uint32_t bclo, bchi;
              search_lane<DT>(l, slot, muf, inv, br, s_phi, s_lo8, a.ecdf, blo, bhi, bclo, bchi);
              if (lane == l) {
                br.lo = blo;
                br.hi = bhi;
                br.clo = bclo;
                br.chi = bchi;
              }
            } else if (pend) {
              br = search_lanes<DT>(pend, !done, slot, muf, inv, br, s_phi, s_lo8, a.ecdf);
            }
            if (!done) {
              if (br.hi - br.lo != 1) flags |= kFlagCorrupt;  // only if cum were not monotone
              br.hi = br.lo + 1;
            }
          } else {
            // (e4m3 misses are rarer, and there the out-of-line search's
            // register cost lost more than it gained)
            while (pend) {
              const int l = __ffs(pend) - 1;
              pend &= pend - 1;
              int32_t blo, bhi;
              uint32_t bclo, bchi;
              search_lane<DT>(l, slot, muf, inv, br, s_phi, s_lo8, a.ecdf, blo, bhi, bclo, bchi);
              if (lane == l) {
                if (bhi - blo != 1) flags |= kFlagCorrupt;  // only if cum were not monotone
                br.lo = blo;
                br.hi = blo + 1;
                br.clo = bclo;
                br.chi = bchi;
              }
            }
          }
        }
        bool need = false;
        if (has) {
          x = (uint64_t)(br.chi - br.clo) * (x >> M) + (slot - br.clo);
          need = x < kStateL;
          const uint32_t sym = DT == 0 ? bits_bf16(br.lo) : bits_e4m3(br.lo);
          if (DT == 0) {
            out_lo = (out_lo >> 16) | (out_hi << 48);
            out_hi = (out_hi >> 16) | ((uint64_t)sym << 48);
          } else {
            out_lo = (out_lo >> 8) | ((uint64_t)sym << 56);
          }
        }
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, need) & seg;
        if (need) {
          const uint32_t pos = cur + __popc(m & lt);  // pos < nw keeps the read in the chunk
          if (pos < nw) {
            x = (x << 32) | w[pos];
          } else {
            flags |= kFlagCorrupt;
            x = kStateL;
          }
        }
        cur += __popc(m);
      }
      // one vector store per group (one lane per chunk would otherwise write
      // 32 scattered sectors per symbol)
      if (has) {
        if (DT == 0)
          *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.kv_out) + obase + p0) =
              make_uint4((uint32_t)out_lo, (uint32_t)(out_lo >> 32), (uint32_t)out_hi,
                         (uint32_t)(out_hi >> 32));
        else
          *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(a.kv_out) + obase + p0) =
              make_uint2((uint32_t)out_lo, (uint32_t)(out_lo >> 32));
      }
    }
    if (ok) {
      if (x != kStateL) flags |= kFlagCorrupt;
      if (ell == 0 && cur != nw) flags |= kFlagCorrupt;
    }
    if (flags) atomicOr(&a.head->flags, flags);
  }
}


// Order-0 baseline decode: cum(r) = floor(K E_q[r] / 2^26) + r needs no mu and
// no sigma.  einv[k] is the smallest r with E_q[r] >= k 2^26 / n (n = kO0InvN).
// Because K E_q[r] / 2^26 - 1 + r < cum(r) <= K E_q[r] / 2^26 + r and r < |S|,
// the answer r* (cum(r*) <= slot < cum(r* + 1)) satisfies
//   E_q[r*] < (slot + 1) 2^26 / K       ->  r* < einv[floor((slot + 1) n / K) + 1]
//   E_q[r* + 1] > (slot - |S|) 2^26 / K ->  r* >= einv[floor((slot - |S|) n / K)] - 1,
// a bracket of one or two table steps, which bisection finishes.
__global__ void __launch_bounds__(dec_threads_max<0>(), 1) k_decode_o0(DecodeLaunch a) {
  extern __shared__ int32_t s_einv0[];
  if (!a.einv_row_stride)  // one table for all chunks: stage it once per SM
    for (int i = threadIdx.x; i <= kO0InvN; i += blockDim.x) s_einv0[i] = a.einv[i];
  __syncthreads();
  constexpr int M = kMBf16;
  constexpr uint32_t kMask = (1u << M) - 1u;
  const int G = a.geo.G;
  const int lane = threadIdx.x & 31;
  const int ell = lane & (G - 1);
  const uint32_t seg = G == 32 ? 0xFFFFFFFFu : (((1u << G) - 1u) << (lane & ~(G - 1)));
  const uint32_t lt = seg & ((1u << lane) - 1u);
  const int64_t ntasks = (((a.c_end - a.c_begin + a.c_step - 1) / a.c_step) * G + 31) / 32;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t nc = a.geo.nchunks;
  const uint64_t hbytes = 64 + 8 * (uint64_t)(nc + 1);
  const uint64_t payload_bytes = a.in_bytes - hbytes;
  const uint8_t *payload = a.in + hbytes;
  uint16_t *out = static_cast<uint16_t *>(a.kv_out);

  for (int64_t task = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); task < ntasks;
       task = next_task(a.head, nwarps)) {
    const int64_t c = a.c_begin + a.c_step * ((task * 32 + lane) / G);
    const bool live = c < a.c_end;
    uint32_t flags = 0;
    uint64_t off_a = 0, off_b = 0;
    if (live) {
      const uint64_t *offs = reinterpret_cast<const uint64_t *>(a.in + 64);
      off_a = offs[c];
      off_b = offs[c + 1];
    }
    bool ok = live && off_a <= off_b && off_b <= payload_bytes && ((off_a | off_b) & 3) == 0 &&
              (off_b - off_a) / 4 >= 2ull * G;
    if (live && !ok) flags |= kFlagCorrupt;
    const uint64_t obase = chunk_out_base(a, c, ok, flags);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(payload + (ok ? off_a : 0));
    const uint64_t nw = ok ? (off_b - off_a) / 4 : 0;
    ChunkGeo cg = chunk_geo(a.geo, live ? c : 0);
    const uint32_t my_groups =
        (ok && (uint32_t)ell < cg.ngroup) ? (cg.ngroup - ell + G - 1) / G : 0u;
    const uint32_t max_groups = __reduce_max_sync(0xFFFFFFFFu, my_groups);
    uint64_t x = ok ? ((uint64_t)w[2 * ell] | ((uint64_t)w[2 * ell + 1] << 32)) : kStateL;
    uint64_t cur = 2ull * G;
    // adaptive counts: the chunk's row has its own tables
    const uint64_t arow = live && a.ecdf_row_stride ? (uint64_t)(c / a.geo.ntb) : 0;
    const uint32_t *ecdf = a.ecdf + arow * a.ecdf_row_stride;
    const int32_t *einv = a.einv_row_stride ? a.einv + arow * a.einv_row_stride : s_einv0;

    for (uint32_t gi = 0; gi < max_groups; ++gi) {
      const bool has = gi < my_groups;
      const uint32_t p0 = 8u * ((uint32_t)ell + (uint32_t)G * gi);
      uint64_t out_lo = 0, out_hi = 0;  // the group's 8 symbols, shifted in from the top
#pragma unroll 1
      for (int k = 0; k < 8; ++k) {
        bool need = false;
        if (has) {
          const uint32_t slot = (uint32_t)x & kMask;
          const uint32_t kh = (uint32_t)(((uint64_t)(slot + 1u) * kO0InvN) / kKBf16) + 1u;
          int32_t hi = kh <= (uint32_t)kO0InvN ? einv[kh] : kNsymBf16;
          int32_t lo = 0;
          if (slot >= (uint32_t)kNsymBf16) {
            const uint32_t kl = (uint32_t)(((uint64_t)(slot - kNsymBf16) * kO0InvN) / kKBf16);
            lo = max(einv[kl] - 1, 0);
          }
          hi = max(hi, lo + 1);
          while (hi - lo > 1) {  // cum(lo) <= slot < cum(hi)
            const int32_t mid = (lo + hi) >> 1;
            if (cum_order0(mid, ecdf) <= slot) lo = mid;
            else hi = mid;
          }
          const uint32_t clo = cum_order0(lo, ecdf), chi = cum_order0(lo + 1, ecdf);
          if (clo > slot || chi <= slot) flags |= kFlagCorrupt;  // only if E_q were not monotone
          x = (uint64_t)(chi - clo) * (x >> M) + (slot - clo);
          need = x < kStateL;
          out_lo = (out_lo >> 16) | (out_hi << 48);
          out_hi = (out_hi >> 16) | ((uint64_t)bits_bf16(lo) << 48);
        }
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, need) & seg;
        if (need) {
          const uint64_t pos = cur + __popc(m & lt);
          if (pos < nw) {
            x = (x << 32) | w[pos];
          } else {
            flags |= kFlagCorrupt;
            x = kStateL;
          }
        }
        cur += __popc(m);
      }
      if (has)
        *reinterpret_cast<uint4 *>(out + obase + p0) =
            make_uint4((uint32_t)out_lo, (uint32_t)(out_lo >> 32), (uint32_t)out_hi,
                       (uint32_t)(out_hi >> 32));
    }
    if (ok) {
      if (x != kStateL) flags |= kFlagCorrupt;
      if (ell == 0 && cur != nw) flags |= kFlagCorrupt;
    }
    if (flags) atomicOr(&a.head->flags, flags);
  }
}

template <int DT, bool BISECT>
static cudaError_t run_decode(const DecodeLaunch &a, int blocks, int threads, cudaStream_t s) {
  // bf16 launches of one round of tasks at most: blocks of up to 768 threads,
  // whose launch bound leaves 80 registers a thread instead of 72
  if constexpr (DT == 0 && !BISECT) {
    if (threads <= kDecThreads) {
      cudaError_t e = cudaFuncSetAttribute(k_decode<DT, BISECT, kDecThreads>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
      if (e != cudaSuccess) return e;
      k_decode<DT, BISECT, kDecThreads><<<blocks, threads, kDecSmem, s>>>(a);
      return cudaGetLastError();
    }
  }
  cudaError_t e = cudaFuncSetAttribute(k_decode<DT, BISECT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
  if (e != cudaSuccess) return e;
  k_decode<DT, BISECT><<<blocks, threads, kDecSmem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeLaunch &a, cudaStream_t s) {
  cudaError_t e;
  if (a.check_header) {
    k_check_header<<<1, 32, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.c_end <= a.c_begin) return cudaSuccess;
  // the task counter of this launch starts at zero
  e = cudaMemsetAsync(&a.head->next_task, 0, sizeof(unsigned long long), s);
  if (e != cudaSuccess) return e;
  const int64_t ntasks = (((a.c_end - a.c_begin + a.c_step - 1) / a.c_step) * a.geo.G + 31) / 32;
  int blocks, threads;
  task_shape(ntasks, kDecThreads, blocks, threads,
             a.dtype == 0 ? dec_threads_max<0>() : dec_threads_max<1>());
  if (a.order0) {
    constexpr size_t smem = sizeof(int32_t) * (kO0InvN + 1);
    e = cudaFuncSetAttribute(k_decode_o0, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k_decode_o0<<<blocks, threads, smem, s>>>(a);
    return cudaGetLastError();
  }
  if (a.dtype == 0)
    return a.bisect ? run_decode<0, true>(a, blocks, threads, s)
                    : run_decode<0, false>(a, blocks, threads, s);
  return a.bisect ? run_decode<1, true>(a, blocks, threads, s)
                  : run_decode<1, false>(a, blocks, threads, s);
}

}  // namespace skv
