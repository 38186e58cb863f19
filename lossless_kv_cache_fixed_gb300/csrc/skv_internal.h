// skv_internal.h -- launcher interface between the C-ABI layer (skv_api.cu)
// and the kernel translation units.  Not installed; not part of the ABI.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

namespace skv {

// Tensor geometry shared by every kernel.  A chunk is one (layer, kv, head,
// token block); chunk c covers rows ((l*2 + kv)*H + h) = c / ntb, block c % ntb.
struct Geo {
  int32_t L, H, T, D, Tb, G;
  int64_t ntb, nchunks;
  int64_t n;  // scalars
};

// Workspace head, at offset 0 of every workspace (256 bytes reserved).
struct WsHead {
  uint32_t flags;                 // skv::kFlag* bits
  uint32_t pad0;
  unsigned long long hash_acc;    // sum of mix64 terms of the model tables
  unsigned long long total;       // encode: payload bytes
  double bits;                    // ideal bits total
};

constexpr int kScanBlock = 2048;  // chunks per scan block

struct EncodeLaunch {
  Geo geo;
  int dtype;
  const void *kv;
  const uint16_t *mu;
  const float2 *inv;        // per-channel (1/sigma, 1/(3 sigma)) table in the workspace
  const uint32_t *ecdf;
  uint32_t *scratch;        // nchunks * stride words
  int64_t stride;           // words per chunk stack
  uint64_t *sizes;          // bytes per chunk, later block-local offsets
  uint32_t *starts;         // first word of each chunk's stack
  uint64_t *partials;       // scan block totals
  WsHead *head;
  uint8_t *out;
  uint64_t capacity;
  uint64_t hash_words;      // number of 32-bit words hashed by the prep kernel
};

struct DecodeLaunch {
  Geo geo;
  int dtype;
  int bisect;               // 1: plain bisection search (reference path)
  const int32_t *einv;      // bf16: inverse of the p-hat prefix table (kHinvN + 1 ranks)
  const uint8_t *in;
  uint64_t in_bytes;
  const uint16_t *mu;
  const float2 *inv;
  const uint32_t *ecdf;
  void *kv_out;
  WsHead *head;
  uint64_t hash_words;
};

struct IdealLaunch {
  Geo geo;
  int dtype;
  const void *kv;
  const uint16_t *mu;
  const float *sigma;
  const float *phat;
  float *per_scalar;
  double *partials;
  int nblocks;
  WsHead *head;
};

// Inverse of the model CDF's Gaussian part, G0(z) = 0.95 Phi(z) + 0.03 Phi(z/3)
// (bf16) or Phi(z) (e4m3), tabulated at kHinvN + 1 equally spaced u in
// [0, kHinvUmax[dtype]] as (z_k, z_{k+1} - z_k): the decoder's first guess.
constexpr int kHinvN = 1024;
constexpr float kHinvUmaxBf16 = 0.98f, kHinvUmaxE4m3 = 1.0f;

// Device constants (Phi knot pairs, e4m3 bin edges, the two inverse tables)
// for the current device.
cudaError_t upload_tables(const uint32_t *phi_knots, const float *lo8, const float *hinv_bf16,
                          const float *hinv_e4m3);

// Model preparation: sigma validation, per-channel reciprocals, E_q checks and
// the model fingerprint accumulation.
cudaError_t launch_prep(const float *sigma, int64_t nsig, const uint32_t *ecdf, float2 *inv,
                        WsHead *head, cudaStream_t s);
cudaError_t launch_encode(const EncodeLaunch &a, cudaStream_t s);
// einv[k] = the smallest rank r with E_q[r] >= k 2^26 / kHinvN, k = 0..kHinvN.
cudaError_t launch_einv(const uint32_t *ecdf, int32_t *einv, cudaStream_t s);
cudaError_t launch_decode(const DecodeLaunch &a, cudaStream_t s);
cudaError_t launch_ideal(const IdealLaunch &a, cudaStream_t s);

int device_sm_count();

}  // namespace skv
