// skv_adapt.cu -- adaptive order-0 counts per (layer, kv, head) row.
//
// Page "KV 缓存压缩的熵估计与动态适应" (entropy estimation and dynamic
// adaptation for KV-cache compression), sections "虚拟滑动窗口的设计原理"
// (decayed counts C_t = alpha C_{t-1} + delta), "平滑更新算法" (P_new = beta
// P_old + (1 - beta) P_est) and "参数配置建议" (alpha 0.97, beta 0.9, an update
// every N_update tokens): the order-0 coder with one model per row, updated
// after every chunk, so the token block is the update period.  Integers only,
// so that the decoder rebuilds the encoder's tables bit for bit:
//   A = round(0.97 2^16) = 63570, B = round(0.9 2^16) = 58982;
//   W[Tb-1] = 2^16, W[t-1] = floor(W[t] A / 2^16), Dk = floor(W[0] A / 2^16);
//   C_0 = 0, C_{b+1}[r] = floor(C_b[r] Dk / 2^16) + sum of W[token] over the
//   block's scalars of rank r;
//   P_0[r] = (E_q[r+1] - E_q[r]) 2^6 (the calibration prior);
//   P_{b+1}[r] = floor((B P_b[r] + (2^16 - B) floor(2^32 C[r] / sum C)) / 2^16);
//   block b codes with E[r] = floor(2^26 S[r] / S_tot), S the prefix of P_b + 1.
// Rows are independent; blocks of a row are sequential (the decoder needs block
// b to build block b + 1's table), so the coder runs one phase per token block:
// tables of all rows, that block's chunks, the update of all rows.
#include <cuda_runtime.h>

#include "skv_internal.h"
#include "skv_model.cuh"

namespace skv {

constexpr int kAdThreads = 1024;
constexpr uint64_t kAdA = 63570, kAdB = 58982;

// floor(x / d) for x < 2^63, d >= 1, from r = floor((2^64 - 1) / d): the
// estimate umulhi(x, r) is at most 2 below the quotient; fixed up exactly.
__device__ __forceinline__ uint64_t div_by_recip(uint64_t x, uint64_t d, uint64_t r) {
  uint64_t q = __umul64hi(x, r);
  for (int i = 0; i < 3 && (q + 1) * d <= x; ++i) ++q;
  return q;
}

__global__ void k_ad_init(const uint32_t *__restrict__ ecdf, uint64_t *P, uint64_t *C, int64_t nrows,
                          uint64_t *W, int Tb) {
  const int64_t n = nrows * (int64_t)kNsymBf16;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t r = (int32_t)(i % kNsymBf16);
    P[i] = (uint64_t)(__ldg(ecdf + r + 1) - __ldg(ecdf + r)) << 6;
    C[i] = 0;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // token weights alpha^(Tb-1-t) and the block decay alpha^Tb, at 2^16
    W[Tb - 1] = 65536;
    for (int t = Tb - 1; t > 0; --t) W[t - 1] = (W[t] * kAdA) >> 16;
    W[Tb] = (W[0] * kAdA) >> 16;
  }
}

// Sum of v over the block (all threads get it).
__device__ uint64_t block_sum(uint64_t v, uint64_t *s_part) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = v;
  __syncthreads();
  uint64_t t = threadIdx.x < (blockDim.x >> 5) ? s_part[threadIdx.x] : 0;
  if (threadIdx.x < 32)
    for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
  if (threadIdx.x == 0) s_part[32] = t;
  __syncthreads();
  const uint64_t total = s_part[32];
  __syncthreads();
  return total;
}

// One block per row: E[r] = floor(2^26 S[r] / S_tot) over P + 1, then (decode)
// einv[k] = the smallest r with E[r] >= k 2^26 / n.
__global__ void __launch_bounds__(kAdThreads) k_ad_table(const uint64_t *__restrict__ P, uint32_t *E,
                                                         int32_t *einv, int n_inv) {
  __shared__ uint64_t s_scan[kAdThreads];
  const int64_t row = blockIdx.x;
  const uint64_t *p = P + row * (int64_t)kNsymBf16;
  uint32_t *e = E + row * (int64_t)(kNsymBf16 + 1);
  const int per = (kNsymBf16 + kAdThreads - 1) / kAdThreads;  // 64 ranks per thread
  const int r0 = threadIdx.x * per, r1 = min(r0 + per, kNsymBf16);
  uint64_t mine = 0;
  for (int r = r0; r < r1; ++r) mine += p[r] + 1;
  // exclusive scan of the thread sums (Hillis-Steele in shared memory)
  s_scan[threadIdx.x] = mine;
  __syncthreads();
  for (int o = 1; o < kAdThreads; o <<= 1) {
    const uint64_t t = threadIdx.x >= o ? s_scan[threadIdx.x - o] : 0;
    __syncthreads();
    s_scan[threadIdx.x] += t;
    __syncthreads();
  }
  const uint64_t stot = s_scan[kAdThreads - 1];
  uint64_t acc = s_scan[threadIdx.x] - mine;
  const uint64_t rc = ~0ull / stot;
  for (int r = r0; r < r1; ++r) {
    e[r] = (uint32_t)div_by_recip(acc << 26, stot, rc);
    acc += p[r] + 1;
  }
  if (threadIdx.x == 0) e[kNsymBf16] = kPhiOne;
  if (!einv) return;
  __syncthreads();
  int32_t *ei = einv + row * (int64_t)(n_inv + 1);
  for (int k = threadIdx.x; k <= n_inv; k += blockDim.x) {
    const uint32_t target = (uint32_t)(((uint64_t)k << 26) / (uint64_t)n_inv);
    int32_t lo = 0, hi = kNsymBf16;
    while (lo < hi) {
      const int32_t mid = (lo + hi) >> 1;
      if (e[mid] >= target) hi = mid;
      else lo = mid + 1;
    }
    ei[k] = lo;
  }
}

// One block per row: fold token block b of `kv` (the input, or the blocks just
// decoded) into the row's counts and probabilities.
__global__ void __launch_bounds__(kAdThreads) k_ad_update(Geo g, const uint16_t *__restrict__ kv,
                                                          int64_t b, uint64_t *P, uint64_t *C,
                                                          const uint64_t *__restrict__ W,
                                                          WsHead *head) {
  __shared__ uint64_t s_part[33];
  const int64_t row = blockIdx.x;
  uint64_t *c = C + row * (int64_t)kNsymBf16;
  uint64_t *p = P + row * (int64_t)kNsymBf16;
  const uint64_t Dk = W[g.Tb];
  for (int r = threadIdx.x; r < kNsymBf16; r += blockDim.x) c[r] = (c[r] * Dk) >> 16;
  __syncthreads();
  const int64_t t0 = b * (int64_t)g.Tb;
  const int64_t tn = min((int64_t)g.Tb, (int64_t)g.T - t0);
  const uint16_t *src = kv + ((uint64_t)row * g.T + (uint64_t)t0) * (uint64_t)g.D;
  uint32_t flags = 0;
  for (int64_t i = threadIdx.x; i < tn * g.D; i += blockDim.x) {
    const int32_t r = rank_bf16(src[i]);
    if (r < 0 || r >= kNsymBf16) {
      flags |= kFlagSymbol;
      continue;
    }
    atomicAdd(reinterpret_cast<unsigned long long *>(c + r),
              (unsigned long long)W[i / g.D]);
  }
  if (flags) atomicOr(&head->flags, flags);
  __syncthreads();
  uint64_t mine = 0;
  for (int r = threadIdx.x; r < kNsymBf16; r += blockDim.x) mine += c[r];
  const uint64_t sum = block_sum(mine, s_part);
  if (sum == 0) return;
  const uint64_t rc = ~0ull / sum;
  for (int r = threadIdx.x; r < kNsymBf16; r += blockDim.x) {
    const uint64_t est = div_by_recip(c[r] << 32, sum, rc);
    p[r] = (kAdB * p[r] + (65536 - kAdB) * est) >> 16;
  }
}

// Ideal bits of token block b of every row: -log2((P_b[r] + 1) / S_tot), S_tot
// the sum of P_b + 1 over the row's ranks.
__global__ void __launch_bounds__(256) k_ad_ideal(Geo g, const uint16_t *__restrict__ kv, int64_t b,
                                                  const uint64_t *__restrict__ P,
                                                  float *per_scalar, double *partials,
                                                  WsHead *head) {
  __shared__ uint64_t s_part[33];
  __shared__ double s_acc[256];
  const int64_t row = blockIdx.y;
  const uint64_t *p = P + row * (int64_t)kNsymBf16;
  uint64_t mine = 0;
  for (int r = threadIdx.x; r < kNsymBf16; r += blockDim.x) mine += p[r] + 1;
  const uint64_t stot = block_sum(mine, s_part);
  const float log2_stot = log2f((float)stot);
  const int64_t t0 = b * (int64_t)g.Tb;
  const int64_t n = min((int64_t)g.Tb, (int64_t)g.T - t0) * g.D;
  const uint64_t base = ((uint64_t)row * g.T + (uint64_t)t0) * (uint64_t)g.D;
  double acc = 0.0;
  uint32_t flags = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t r = rank_bf16(kv[base + i]);
    float bits = 0.0f;
    if (r < 0 || r >= kNsymBf16) flags |= kFlagSymbol;
    else bits = log2_stot - log2f((float)(p[r] + 1));
    if (per_scalar) per_scalar[base + i] = bits;
    acc += (double)bits;
  }
  if (flags) atomicOr(&head->flags, flags);
  s_acc[threadIdx.x] = acc;
  __syncthreads();
  for (int o = 128; o; o >>= 1) {
    if (threadIdx.x < o) s_acc[threadIdx.x] += s_acc[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) partials[row * gridDim.x + blockIdx.x] = s_acc[0];
}

cudaError_t launch_ad_init(const uint32_t *ecdf, uint64_t *P, uint64_t *C, int64_t nrows, uint64_t *W,
                           int Tb, cudaStream_t s) {
  int64_t blocks = (nrows * kNsymBf16 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  k_ad_init<<<(unsigned)blocks, 256, 0, s>>>(ecdf, P, C, nrows, W, Tb);
  return cudaGetLastError();
}

cudaError_t launch_ad_table(const uint64_t *P, uint32_t *E, int32_t *einv, int n_inv, int64_t nrows,
                            cudaStream_t s) {
  k_ad_table<<<(unsigned)nrows, kAdThreads, 0, s>>>(P, E, einv, n_inv);
  return cudaGetLastError();
}

cudaError_t launch_ad_update(const Geo &g, const uint16_t *kv, int64_t b, uint64_t *P, uint64_t *C,
                             const uint64_t *W, WsHead *head, int64_t nrows, cudaStream_t s) {
  k_ad_update<<<(unsigned)nrows, kAdThreads, 0, s>>>(g, kv, b, P, C, W, head);
  return cudaGetLastError();
}

cudaError_t launch_ad_ideal(const Geo &g, const uint16_t *kv, int64_t b, const uint64_t *P,
                            float *per_scalar, double *partials, int bx, WsHead *head,
                            int64_t nrows, cudaStream_t s) {
  k_ad_ideal<<<dim3((unsigned)bx, (unsigned)nrows), 256, 0, s>>>(g, kv, b, P, per_scalar, partials,
                                                               head);
  return cudaGetLastError();
}

}  // namespace skv
