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

// One chunk's extent: its first scalar, the first sigma entry of its
// (l, kv, h) row and its number of 8-scalar groups.
struct ChunkGeo {
  uint64_t base;
  uint64_t srow;
  uint32_t ngroup;
};

__device__ __forceinline__ ChunkGeo chunk_geo(const Geo &g, int64_t c) {
  int64_t row = c / g.ntb, tb = c - row * g.ntb;
  int64_t t0 = tb * g.Tb;
  int64_t tn = (int64_t)g.T - t0;
  if (tn > g.Tb) tn = g.Tb;
  ChunkGeo r;
  r.base = (uint64_t)row * (uint64_t)g.T * (uint64_t)g.D + (uint64_t)t0 * (uint64_t)g.D;
  r.srow = (uint64_t)row * (uint64_t)g.D;
  r.ngroup = (uint32_t)(tn * g.D / 8);
  return r;
}

// Per-block sigma scales: one byte per (chunk, 8-channel group), packed four
// to a word, low byte first; the words open the chunk's payload.
__host__ __device__ constexpr int32_t scale_words(int32_t D) { return (D / 8 + 3) / 4; }
constexpr int kMaxScaledD = 2048;  // 256 groups

// Workspace head, at offset 0 of every workspace (256 bytes reserved).
struct WsHead {
  uint32_t flags;                 // skv::kFlag* bits
  uint32_t pad0;
  unsigned long long hash_acc;    // sum of mix64 terms of the model tables
  unsigned long long total;       // encode: payload bytes
  double bits;                    // ideal bits total
  unsigned long long next_task;   // decode: tasks handed out after the first round
  unsigned long long chunks_done; // encode: chunks coded since the head was cleared
  unsigned long long committed;   // encode: chunks placed by skv_encode_commit (a prefix)
  unsigned long long commit_total;  // encode: payload bytes of those chunks
};

// ---- container header (spec v1), built the same way on the host and the device ----

__host__ __device__ inline void put_u16(uint8_t *p, uint32_t v) {
  p[0] = (uint8_t)v;
  p[1] = (uint8_t)(v >> 8);
}
__host__ __device__ inline void put_u32(uint8_t *p, uint32_t v) {
  for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
__host__ __device__ inline void put_u64(uint8_t *p, uint64_t v) {
  for (int i = 0; i < 8; ++i) p[i] = (uint8_t)(v >> (8 * i));
}

// The 64-byte container header of a cache of geometry g (see skv.h).
// features: bit 0 per-block scales, bit 1 order-0, bit 2 adaptive counts.
__host__ __device__ inline void make_header(uint8_t *h, const Geo &g, int dtype, uint64_t payload,
                                            uint64_t fingerprint, uint32_t features) {
  for (int i = 0; i < 64; ++i) h[i] = 0;
  put_u32(h + 0, 0x31564B53u);  // "SKV1"
  put_u16(h + 4, 1);
  h[6] = (uint8_t)dtype;
  h[7] = (uint8_t)(dtype == 0 ? 28 : 16);
  put_u32(h + 8, (uint32_t)g.L);
  put_u32(h + 12, 2);
  put_u32(h + 16, (uint32_t)g.H);
  put_u32(h + 20, (uint32_t)g.T);
  put_u32(h + 24, (uint32_t)g.D);
  put_u32(h + 28, (uint32_t)g.Tb);
  put_u16(h + 32, (uint32_t)g.G);
  h[34] = 8;
  h[35] = 9;
  put_u16(h + 36, 8);
  put_u16(h + 38, features);
  put_u64(h + 40, (uint64_t)g.nchunks);
  put_u64(h + 48, payload);
  put_u64(h + 56, fingerprint);
}

// SplitMix64 output function (Steele, Lea, Flood, OOPSLA 2014): the model
// fingerprint is sum_k mix64(k << 32 | word_k) mod 2^64, then mix64(sum ^ nwords).
__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

constexpr int kScanBlock = 2048;  // chunks per scan block

struct EncodeLaunch {
  Geo geo;
  int dtype;
  const void *kv;
  const uint16_t *mu;
  const float2 *inv;        // per-channel (1/sigma, 1/(3 sigma)) table in the workspace
  const float2 *inv_chunk;  // per-block scales: the same per (chunk, channel), else null
  const uint32_t *scale_words;  // per-block scales: nsw words per chunk
  int32_t nsw;              // scale words per chunk (0 without per-block scales)
  int32_t order0;           // 1: order-0 baseline (p-hat alone; kv only)
  int32_t adaptive;         // 1: adaptive counts (header feature bit 2)
  int64_t c_first, c_step, c_count;  // chunks c_first + c_step * i, i < c_count
  uint64_t ecdf_row_stride; // adaptive counts: one E table per row, else 0
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
  // the ideal code length as the encoder codes (bits_partials set; bf16
  // launches that encode_fuses_bits accepts): the p-hat table, per-scalar
  // output (or null) and one fp64 partial sum per block
  const float *phat;
  float *bits_out;
  double *bits_partials;
  const float2 *log2q;      // the Gaussian tail table (tail_table()) for the rare scalars
};

struct DecodeLaunch {
  Geo geo;
  int dtype;
  int bisect;               // 1: plain bisection search (reference path)
  const int32_t *einv;      // bf16: inverse of the p-hat prefix table (kHinvN + 1 ranks)
  const float2 *gmu;        // bf16 mixture: per rank of mu, the guess's p-hat terms (k_einv)
  const uint8_t *in;
  uint64_t in_bytes;
  const uint16_t *mu;
  const float2 *inv;
  const float2 *inv_chunk;  // per-block scales: per (chunk, channel) reciprocals, else null
  int32_t nsw;
  int32_t order0;           // 1: order-0 baseline; einv then has kO0InvN + 1 entries
  int32_t adaptive;         // 1: adaptive counts (header feature bit 2)
  const uint32_t *ecdf;
  void *kv_out;
  WsHead *head;
  uint64_t hash_words;
  int64_t c_begin, c_end;   // chunks to decode: c_begin + c_step * i < c_end
  int64_t c_step;
  uint64_t ecdf_row_stride, einv_row_stride;  // adaptive counts: per-row tables, else 0
  int32_t check_header;     // 1: check the header and offset-table ends first
  const uint32_t *page_of_chunk;  // paged layout (mu and kv_out are page pools), else null
  uint64_t num_pages;
  uint64_t page_scalars;    // token_block * head_dim
};

struct IdealLaunch {
  Geo geo;
  int dtype;
  const void *kv;
  const uint16_t *mu;
  const float *sigma;
  const float *sigma_chunk;  // per-block scales: sigma_eff per (chunk, channel), else null
  int32_t order0;            // 1: order-0 baseline, -log2 p-hat (kv only)
  const float *phat;
  float *per_scalar;
  double *partials;
  int nblocks;
  WsHead *head;
  uint64_t td_rcp;           // floor((2^64 - 1) / (T * D)): row of a scalar by multiply-high
};

// Model bits: the code length -log2(freq / 2^M) of every scalar under the
// coder's own integer frequencies, summed like the ideal bits.
struct ModelBitsLaunch {
  Geo geo;
  int dtype;
  int32_t order0;           // 1: order-0 baseline (kv only)
  const void *kv;
  const uint16_t *mu;
  const float2 *inv;        // per-channel (1/sigma, 1/(3 sigma)) table in the workspace
  const float2 *inv_chunk;  // per-block scales: the same per (chunk, channel), else null
  const uint32_t *ecdf;
  float *per_scalar;
  double *partials;
  int nblocks;
  WsHead *head;
};

// Inverse of the model CDF's Gaussian part, G0(z) = 0.95 Phi(z) + 0.03 Phi(z/3)
// (bf16) or Phi(z) (e4m3), tabulated at kHinvN + 1 equally spaced u in
// [0, kHinvUmax[dtype]] as (z_k, z_{k+1} - z_k): the decoder's first guess.
constexpr int kHinvN = 1024;
// Order-0 decode: inverse of the p-hat prefix table at kO0InvN + 1 points.
constexpr int kO0InvN = 8192;
constexpr float kHinvUmaxBf16 = 0.98f, kHinvUmaxE4m3 = 1.0f;
// The guess table's knots per unit of u (bf16).
constexpr float kHscaleBf16 = (float)kHinvN / kHinvUmaxBf16;
// Ideal bits (e4m3): log2 Q(z), Q(z) = erfc(z / sqrt 2) / 2 the Gaussian upper
// tail, at z = k / kTailPerUnit for k = 0 .. kTailN - 1 (z from 0 to 12).
constexpr int kTailPerUnit = 256;
constexpr int kTailN = 12 * kTailPerUnit + 1;

// Per-block sigma scales.  Estimate mode (kv, mu set): choose each group's
// scale byte from the residuals; load mode (in set): read them from the
// container's chunks.  Either way, write sigma_eff = sigma m(s) per (chunk,
// channel) as reciprocal pairs (inv) and/or plain values (sig), and in
// estimate mode the packed scale words.
struct ScaleLaunch {
  Geo geo;
  int dtype;
  const void *kv;
  const uint16_t *mu;
  const uint8_t *in;
  uint64_t in_bytes;
  const float *sigma;
  uint32_t *words;
  float2 *inv;
  float *sig;
  WsHead *head;
  int64_t c_begin, c_end;   // chunks to estimate or to read
};

// Device constants (Phi knot pairs, e4m3 bin edges, the two inverse tables,
// the scale multipliers m(s)) for the current device.
cudaError_t upload_tables(const uint32_t *phi_knots, const float *lo8, const float *hinv_bf16,
                          const float *hinv_e4m3);
cudaError_t upload_scale_mult(const float *mult);
cudaError_t upload_tail_table(const float *log2_q);  // kTailN values
// Most blocks of an ideal-bits reduction (one fp64 partial sum each).
constexpr int kMaxBitsBlocks = 4096;
cudaError_t launch_scales(const ScaleLaunch &a, cudaStream_t s);

// Model preparation: sigma validation, per-channel reciprocals, E_q checks and
// the model fingerprint accumulation.
cudaError_t launch_prep(const float *sigma, int64_t nsig, const uint32_t *ecdf, float2 *inv,
                        WsHead *head, cudaStream_t s);
cudaError_t launch_encode(const EncodeLaunch &a, cudaStream_t s);
// The encode kernel alone over a.c_first + a.c_step * i, and the size scan and
// compaction that follow it (launch_encode = both).
cudaError_t launch_encode_chunks(const EncodeLaunch &a, cudaStream_t s);
// Whether a launch of `chunks` chunks computes the ideal bits inside the
// encoder (skv_encode_with_bits) rather than in a second kernel.
bool encode_fuses_bits(int dtype, bool order0, bool scaled, int64_t chunks, int G);
cudaError_t launch_encode_finish(const EncodeLaunch &a, cudaStream_t s);
// skv_encode_commit: chunks [a.c_first, a.c_first + a.c_count), the next after
// those committed before, placed in the container a.out (offsets and payload),
// and the container's size so far in *end_bytes (if not null);
// launch_commit_header then writes the header once every chunk is committed.
cudaError_t launch_encode_commit(const EncodeLaunch &a, uint64_t *end_bytes, cudaStream_t s);
cudaError_t launch_commit_header(const EncodeLaunch &a, cudaStream_t s);

// Adaptive counts (skv_adapt.cu): per-row probabilities P and counts C (u64,
// kNsymBf16 per row), per-row tables E (kNsymBf16 + 1) and, for decode, their
// inverses; W holds the Tb token weights and the block decay.
cudaError_t launch_ad_init(const uint32_t *ecdf, uint64_t *P, uint64_t *C, int64_t nrows, uint64_t *W,
                           int Tb, cudaStream_t s);
cudaError_t launch_ad_table(const uint64_t *P, uint32_t *E, int32_t *einv, int n_inv, int64_t nrows,
                            cudaStream_t s);
cudaError_t launch_ad_update(const Geo &g, const uint16_t *kv, int64_t b, uint64_t *P, uint64_t *C,
                             const uint64_t *W, WsHead *head, int64_t nrows, cudaStream_t s);
cudaError_t launch_ad_ideal(const Geo &g, const uint16_t *kv, int64_t b, const uint64_t *P,
                            float *per_scalar, double *partials, int bx, WsHead *head,
                            int64_t nrows, cudaStream_t s);
cudaError_t launch_ideal_final(const double *partials, int n, WsHead *head, cudaStream_t s);
// einv[k] = the smallest rank r with E_q[r] >= k 2^26 / n, k = 0..n (n divides 2^26);
// with gmu, also the decoder's per-rank guess terms (kNsymBf16 entries).
cudaError_t launch_einv(const uint32_t *ecdf, int32_t *einv, int n, float2 *gmu, cudaStream_t s);
// Device address of the Gaussian tail table (log2 Q at kTailN points), or null.
const float2 *tail_table();
cudaError_t launch_decode(const DecodeLaunch &a, cudaStream_t s);
cudaError_t launch_ideal(const IdealLaunch &a, cudaStream_t s);
cudaError_t launch_model_bits(const ModelBitsLaunch &a, cudaStream_t s);

int device_sm_count();

}  // namespace skv
