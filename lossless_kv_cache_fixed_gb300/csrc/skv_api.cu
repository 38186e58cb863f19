// skv_api.cu -- the C ABI declared in include/skv.h: argument checks, workspace
// layout, the host-built model constants, launches and status readback.
//
// Page "推测式 KV 编码无损压缩 KV 缓存最高可达约 4 倍" (Speculative KV coding):
// section "什么能预测 KV 缓存" defines the encode (KV, mu, sigma) -> bits and
// decode (bits, mu, sigma) -> KV operations; section "早期结果" the mixture with
// the empirical bf16 distribution that skv_build_ecdf tabulates.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/skv.h"
#include "skv_internal.h"
#include "skv_model.cuh"

using namespace skv;

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
// The workspace head takes the first kAlign-byte slot of every workspace.
static_assert(sizeof(WsHead) <= kAlign, "the workspace head must fit one aligned slot");

// ---- host-built model constants ----

uint32_t g_phi_host[kPhiKnots];
float g_lo8_host[256];
float g_hinv_host[2][kHinvN + 1];
float g_scale_mult_host[256];
float g_log2q_host[kTailN];
std::once_flag g_const_once;

double e4m3_value_host(uint32_t u) {
  uint32_t e = (u >> 3) & 15u, m = u & 7u;
  double v = e ? std::ldexp(1.0 + m / 8.0, (int)e - 7) : std::ldexp(m / 8.0, -6);
  return (u & 0x80u) ? -v : v;
}

uint32_t e4m3_bits_host(int r) { return r >= 127 ? (uint32_t)(r - 127) : (0x80u | (uint32_t)(126 - r)); }

void build_constants() {
  // T[i] = RNE(2^26 Phi(-8 + i/512)), Phi(z) = erfc(-z/sqrt 2)/2.  The nearest
  // tie of 2^26 Phi over these knots is 2.3e-4 units away, far beyond the
  // error of any binary64 erfc, so the table is the same on every host.
  for (int i = 0; i < kPhiKnots; ++i) {
    double z = -8.0 + (double)i / 512.0;
    g_phi_host[i] = (uint32_t)std::nearbyint(std::ldexp(0.5 * std::erfc(-z / std::sqrt(2.0)), 26));
  }
  g_phi_host[0] = 0;
  g_phi_host[kPhiKnots - 1] = kPhiOne;
  // e4m3 bin lower edges by rank: midpoints, with the +-448 bins open-ended
  g_lo8_host[0] = -INFINITY;
  for (int r = 1; r < kNsymE4m3; ++r)
    g_lo8_host[r] = (float)(0.5 * (e4m3_value_host(e4m3_bits_host(r - 1)) +
                                   e4m3_value_host(e4m3_bits_host(r))));
  g_lo8_host[kNsymE4m3] = INFINITY;
  g_lo8_host[255] = INFINITY;
  // Inverse of the Gaussian part of the model CDF (the decoder's first guess;
  // any error here costs search steps, never correctness).
  auto Phi = [](double z) { return 0.5 * std::erfc(-z / std::sqrt(2.0)); };
  for (int t = 0; t < 2; ++t) {
    const double umax = t == 0 ? kHinvUmaxBf16 : kHinvUmaxE4m3;
    for (int k = 0; k <= kHinvN; ++k) {
      const double u = umax * k / kHinvN;
      double a = -40.0, b = 40.0;
      for (int it = 0; it < 100; ++it) {
        const double m = 0.5 * (a + b);
        const double g = t == 0 ? 0.95 * Phi(m) + 0.03 * Phi(m / 3.0) : Phi(m);
        (g < u ? a : b) = m;
      }
      const double z = 0.5 * (a + b);
      g_hinv_host[t][k] = (float)(z < -14.0 ? -14.0 : (z > 14.0 ? 14.0 : z));
    }
  }
  // log2 Q(z) of the Gaussian upper tail at z = k / kTailPerUnit, in binary64
  for (int k = 0; k < kTailN; ++k) {
    const double z = (double)k / kTailPerUnit;
    g_log2q_host[k] = (float)std::log2(0.5 * std::erfc(z / std::sqrt(2.0)));
  }
  // per-block scale multipliers m(s) = fp32(2^((s - 128) / 32)); binary64 exp2
  // is within an ulp of 2^(k/32), whose fp32 rounding is never that close to a tie
  for (int k = 0; k < 256; ++k) g_scale_mult_host[k] = (float)std::exp2((k - 128) / 32.0);
}

std::mutex g_dev_mu;
bool g_dev_ready[1024];

int ensure_device_tables() {
  std::call_once(g_const_once, build_constants);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SKV_ERR_CUDA;
  if (dev < 0 || dev >= 1024) return SKV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev_ready[dev]) {
    if (upload_tables(g_phi_host, g_lo8_host, g_hinv_host[0], g_hinv_host[1]) != cudaSuccess)
      return SKV_ERR_CUDA;
    if (upload_scale_mult(g_scale_mult_host) != cudaSuccess) return SKV_ERR_CUDA;
    if (upload_tail_table(g_log2q_host) != cudaSuccess) return SKV_ERR_CUDA;
    g_dev_ready[dev] = true;
  }
  return SKV_OK;
}

struct Plan {
  Geo geo;
  int dtype;
  int64_t nsig;
  int32_t nsw;     // per-block scale words per chunk (0: static sigma)
  int order0;      // order-0 baseline: p-hat alone, no mu and no sigma
  int adaptive;    // adaptive counts per row (order 0), one phase per token block
  int64_t nrows;   // layers * 2 * heads
  size_t ad_P, ad_C, ad_E, ad_W, ad_inv, ad_part;  // adaptive regions, relative offsets
  size_t ad_bytes_enc, ad_bytes_dec, ad_bytes_bits;
  size_t ad_base_enc, ad_base_dec, ad_base_bits;  // where each operation's region starts
  int ad_bx;       // ideal-bits blocks per (row, token block)
  int64_t nsig_model;  // sigma entries the model reads (0 for the order-0 baseline)
  // workspace layout (byte offsets)
  size_t off_inv, off_sizes, off_starts, off_partials, off_scratch, off_bits, off_einv, total;
  size_t off_enc_cinv, off_enc_words, off_enc_bits, enc_total;  // encode: per-chunk tables after the stacks
  size_t off_dec_gmu, off_dec_cinv, dec_total;    // decode: after the inverse p-hat table
  size_t off_bits_csig, bits_total;               // ideal bits: after the partial sums
  size_t off_mb_cinv, mb_total;                   // model bits: reciprocals per (chunk, channel)
  int64_t stride;  // words per chunk stack
  int bits_blocks;
};

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

int make_plan(const skv_params *p, const skv_shape *s, Plan *out) {
  if (!p || !s || !out) return SKV_ERR_ARG;
  if (p->dtype != SKV_BF16 && p->dtype != SKV_E4M3) return SKV_ERR_ARG;
  if (p->flags & ~(SKV_FLAG_DECODE_BISECT | SKV_FLAG_BLOCK_SCALE | SKV_FLAG_ORDER0 |
                   SKV_FLAG_ADAPTIVE))
    return SKV_ERR_ARG;
  const bool order0 = (p->flags & SKV_FLAG_ORDER0) != 0;
  if (order0 && (p->dtype != SKV_BF16 || (p->flags & SKV_FLAG_BLOCK_SCALE))) return SKV_ERR_ARG;
  const bool adaptive = (p->flags & SKV_FLAG_ADAPTIVE) != 0;
  // the counts' fixed point (a row's decayed total below 2^31) needs head_dim <= 512
  if (adaptive && (!order0 || s->head_dim > 512 || p->token_block > 65536)) return SKV_ERR_ARG;
  if (s->kv != 2 || s->layers <= 0 || s->heads <= 0 || s->tokens <= 0 || s->head_dim <= 0)
    return SKV_ERR_ARG;
  if (s->head_dim % 8) return SKV_ERR_ARG;
  const bool scaled = (p->flags & SKV_FLAG_BLOCK_SCALE) != 0;
  if (scaled && s->head_dim > kMaxScaledD) return SKV_ERR_ARG;
  const int G = p->lanes;
  if (G < 1 || G > 32 || (G & (G - 1))) return SKV_ERR_ARG;
  if (p->token_block <= 0) return SKV_ERR_ARG;
  Plan pl;
  pl.dtype = p->dtype;
  pl.geo.L = s->layers;
  pl.geo.H = s->heads;
  pl.geo.T = s->tokens;
  pl.geo.D = s->head_dim;
  pl.geo.Tb = p->token_block;
  const int64_t tb_eff = p->token_block < s->tokens ? p->token_block : s->tokens;
  pl.geo.G = G;
  pl.geo.ntb = ((int64_t)s->tokens + pl.geo.Tb - 1) / pl.geo.Tb;
  const int64_t rows = (int64_t)s->layers * 2 * s->heads;
  pl.geo.nchunks = rows * pl.geo.ntb;
  pl.geo.n = rows * (int64_t)s->tokens * s->head_dim;
  // a chunk's scalar offsets are 32-bit inside the kernels
  if (tb_eff * s->head_dim >= (1ll << 31)) return SKV_ERR_ARG;
  pl.nsig = rows * s->head_dim;
  pl.order0 = order0 ? 1 : 0;
  pl.nsig_model = order0 ? 0 : pl.nsig;
  pl.adaptive = adaptive ? 1 : 0;
  pl.nrows = rows;
  // worst case words of one full chunk: every lane emits at most one word per
  // symbol and, since a symbol adds at most M + log2(1 + 2^(M-31)) < M + 1
  // bits of state, at most ceil(n (M + 1) / 32) words; plus 2 flush words.
  const int M = p->dtype == SKV_BF16 ? kMBf16 : kME4m3;
  const int64_t ngroup = tb_eff * s->head_dim / 8;
  const int64_t nlane = 8 * ((ngroup + G - 1) / G);
  int64_t wl = (nlane * (M + 1) + 31) / 32;
  if (wl > nlane) wl = nlane;
  pl.nsw = scaled ? scale_words(s->head_dim) : 0;
  pl.stride = ((G * (wl + 2)) + pl.nsw + 3) / 4 * 4;
  if (pl.stride >= (1ll << 31)) return SKV_ERR_ARG;  // the encoder's stack index is 32-bit
  size_t off = align_up(sizeof(WsHead));
  pl.off_inv = off;
  off = align_up(off + sizeof(float2) * (size_t)pl.nsig);
  pl.off_sizes = off;
  off = align_up(off + sizeof(uint64_t) * (size_t)(pl.geo.nchunks + 1));
  pl.off_starts = off;
  off = align_up(off + sizeof(uint32_t) * (size_t)pl.geo.nchunks);
  pl.off_partials = off;
  off = align_up(off + sizeof(uint64_t) * (size_t)((pl.geo.nchunks + kScanBlock - 1) / kScanBlock + 1));
  pl.off_scratch = off;
  off = align_up(off + sizeof(uint32_t) * (size_t)pl.stride * (size_t)pl.geo.nchunks);
  pl.total = off;
  int64_t n8 = pl.geo.n / 8;
  int64_t nb = (n8 + 255) / 256;
  pl.bits_blocks = (int)(nb < kMaxBitsBlocks ? (nb > 0 ? nb : 1) : kMaxBitsBlocks);
  pl.off_bits = align_up(pl.off_inv + sizeof(float2) * (size_t)pl.nsig);
  pl.off_einv = pl.off_bits;  // decode only: the inverse p-hat table follows the reciprocals
  // per-block scales: (chunk, channel) tables appended to each operation's layout
  const size_t ccells = scaled ? (size_t)pl.geo.nchunks * (size_t)s->head_dim : 0;
  pl.off_enc_cinv = pl.total;
  pl.off_enc_words = align_up(pl.off_enc_cinv + sizeof(float2) * ccells);
  pl.off_enc_bits = align_up(pl.off_enc_words + sizeof(uint32_t) * (size_t)pl.nsw * (size_t)pl.geo.nchunks);
  pl.off_bits_csig = align_up(pl.off_bits + sizeof(double) * (size_t)pl.bits_blocks);
  pl.bits_total = align_up(pl.off_bits_csig + sizeof(float) * ccells);
  // skv_encode_with_bits: one fp64 partial sum per encode block when the
  // encoder computes the bits, else an ideal-bits workspace of its own
  pl.enc_total = align_up(pl.off_enc_bits +
                          std::max(sizeof(double) * (size_t)kMaxBitsBlocks, pl.bits_total));
  // the decoder's inverse p-hat table: kHinvN + 1 entries, kO0InvN + 1 for order 0;
  // then (bf16 mixture) its per-rank guess terms for mu
  pl.off_dec_gmu = align_up(pl.off_einv + sizeof(int32_t) * ((order0 ? kO0InvN : kHinvN) + 1));
  const bool gmu = p->dtype == SKV_BF16 && !order0;
  pl.off_dec_cinv = align_up(pl.off_dec_gmu + (gmu ? sizeof(float2) * (size_t)kNsymBf16 : 0));
  pl.dec_total = align_up(pl.off_dec_cinv + sizeof(float2) * ccells);
  pl.off_mb_cinv = pl.off_bits_csig;
  pl.mb_total = align_up(pl.off_mb_cinv + sizeof(float2) * ccells);
  // adaptive counts: per-row P, C, E (and decode's inverse tables), the token
  // weights and the ideal-bits partial sums, appended to each operation's layout
  pl.ad_bx = (int)std::min<int64_t>(16, (tb_eff * s->head_dim + 2047) / 2048);
  if (adaptive) {
    const size_t nr = (size_t)rows;
    pl.ad_P = 0;
    pl.ad_C = align_up(pl.ad_P + sizeof(uint64_t) * nr * kNsymBf16);
    pl.ad_E = align_up(pl.ad_C + sizeof(uint64_t) * nr * kNsymBf16);
    pl.ad_W = align_up(pl.ad_E + sizeof(uint32_t) * nr * (kNsymBf16 + 1));
    pl.ad_inv = align_up(pl.ad_W + sizeof(uint64_t) * (size_t)(p->token_block + 1));
    pl.ad_part = pl.ad_inv;  // ideal bits use this region for its partial sums instead
    pl.ad_bytes_enc = pl.ad_inv;
    pl.ad_bytes_dec = align_up(pl.ad_inv + sizeof(int32_t) * nr * (kO0InvN + 1));
    pl.ad_bytes_bits = align_up(pl.ad_part + sizeof(double) * (size_t)pl.geo.ntb * nr * pl.ad_bx);
    pl.ad_base_enc = pl.enc_total;
    pl.ad_base_dec = pl.dec_total;
    pl.ad_base_bits = pl.bits_total;
    pl.enc_total += pl.ad_bytes_enc;
    pl.dec_total += pl.ad_bytes_dec;
    pl.bits_total += pl.ad_bytes_bits;
  }
  *out = pl;
  return SKV_OK;
}

size_t ws_bytes_for(const Plan &pl, int op) {
  if (op == SKV_OP_ENCODE) return pl.enc_total;
  if (op == SKV_OP_DECODE) return pl.dec_total;
  if (op == SKV_OP_MODEL_BITS) return pl.mb_total;
  return pl.bits_total;
}

uint64_t hash_words(const Plan &pl) {
  return (uint64_t)pl.nsig_model + (pl.dtype == SKV_BF16 ? (uint64_t)kNsymBf16 + 1 : 0);
}

int status_from_flags(uint32_t f) {
  if (f & kFlagArg) return SKV_ERR_ARG;
  if (f & kFlagSymbol) return SKV_ERR_SYMBOL;
  if (f & kFlagParam) return SKV_ERR_PARAM;
  if (f & kFlagCorrupt) return SKV_ERR_CORRUPT;
  if (f & kFlagCapacity) return SKV_ERR_CAPACITY;
  if (f & kFlagOverflow) return SKV_ERR_CUDA;  // an internal bound was broken
  return SKV_OK;
}

// Reads the workspace head back (a synchronising copy).
int read_head(WsHead *dev, WsHead *host, cudaStream_t st) {
  if (cudaMemcpyAsync(host, dev, sizeof(WsHead), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SKV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SKV_ERR_CUDA;
  return SKV_OK;
}

int common_inputs(const skv_params *p, const Plan &pl, const void *kv, const uint16_t *mu) {
  if (!kv || !aligned(kv, 16)) return SKV_ERR_ARG;
  // the order-0 baseline reads neither mu nor sigma (both may be NULL)
  if (!pl.order0) {
    if (!mu || !p->sigma || !aligned(mu, 16) || !aligned(p->sigma, 4)) return SKV_ERR_ARG;
  }
  if (pl.dtype == SKV_BF16 && (!p->ecdf || !aligned(p->ecdf, 4))) return SKV_ERR_ARG;
  return SKV_OK;
}

ScaleLaunch scale_launch(const Plan &pl, const skv_params *p, WsHead *head) {
  ScaleLaunch sl;
  std::memset(&sl, 0, sizeof(sl));
  sl.geo = pl.geo;
  sl.dtype = pl.dtype;
  sl.sigma = p->sigma;
  sl.head = head;
  sl.c_begin = 0;
  sl.c_end = pl.geo.nchunks;
  return sl;
}

// The encode launch for a plan and its workspace (no chunk range yet).
EncodeLaunch encode_launch(const skv_params *params, const Plan &pl, uint8_t *ws) {
  EncodeLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.geo = pl.geo;
  a.dtype = pl.dtype;
  a.inv = reinterpret_cast<float2 *>(ws + pl.off_inv);
  a.nsw = pl.nsw;
  a.order0 = pl.order0;
  a.adaptive = pl.adaptive;
  a.ecdf = pl.dtype == SKV_BF16 ? params->ecdf : nullptr;
  a.scratch = reinterpret_cast<uint32_t *>(ws + pl.off_scratch);
  a.stride = pl.stride;
  a.sizes = reinterpret_cast<uint64_t *>(ws + pl.off_sizes);
  a.starts = reinterpret_cast<uint32_t *>(ws + pl.off_starts);
  a.partials = reinterpret_cast<uint64_t *>(ws + pl.off_partials);
  a.head = reinterpret_cast<WsHead *>(ws);
  a.hash_words = hash_words(pl);
  a.c_step = 1;
  if (pl.nsw) {
    a.inv_chunk = reinterpret_cast<float2 *>(ws + pl.off_enc_cinv);
    a.scale_words = reinterpret_cast<uint32_t *>(ws + pl.off_enc_words);
  }
  return a;
}

// Encode of chunks [c0, c1) into the workspace's chunk stacks, enqueued on
// `stream` without a host synchronisation.  `first` clears the status and the
// chunk count and prepares the model tables (reciprocals, fingerprint).
int encode_enqueue(const skv_params *params, const Plan &pl, const void *kv, const uint16_t *mu,
                   uint64_t c0, uint64_t c1, bool first, void *workspace, cudaStream_t st,
                   bool bits = false, float *bits_out = nullptr) {
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  EncodeLaunch a = encode_launch(params, pl, ws);
  if (bits) {
    // the ideal code length as it codes: the partial sums start at zero
    a.bits_partials = reinterpret_cast<double *>(ws + pl.off_enc_bits);
    a.bits_out = bits_out;
    a.phat = params->phat;
    if (!(a.log2q = tail_table())) return SKV_ERR_CUDA;
    if (cudaMemsetAsync(a.bits_partials, 0, sizeof(double) * kMaxBitsBlocks, st) != cudaSuccess)
      return SKV_ERR_CUDA;
  }
  if (first) {
    if (cudaMemsetAsync(a.head, 0, sizeof(WsHead), st) != cudaSuccess) return SKV_ERR_CUDA;
    // no chunk coded yet: skv_encode_commit refuses a chunk whose start is the sentinel
    if (cudaMemsetAsync(a.starts, 0xFF, sizeof(uint32_t) * (size_t)pl.geo.nchunks, st) !=
        cudaSuccess)
      return SKV_ERR_CUDA;
    if (launch_prep(params->sigma, pl.nsig_model, a.ecdf, const_cast<float2 *>(a.inv), a.head,
                    st) != cudaSuccess)
      return SKV_ERR_CUDA;
  }
  if (c1 <= c0) return SKV_OK;
  a.kv = kv;
  a.mu = mu;
  if (pl.nsw) {
    // the scales of these chunks, from their residuals
    ScaleLaunch sl = scale_launch(pl, params, a.head);
    sl.kv = kv;
    sl.mu = mu;
    sl.inv = const_cast<float2 *>(a.inv_chunk);
    sl.words = const_cast<uint32_t *>(a.scale_words);
    sl.c_begin = (int64_t)c0;
    sl.c_end = (int64_t)c1;
    if (launch_scales(sl, st) != cudaSuccess) return SKV_ERR_CUDA;
  }
  a.c_first = (int64_t)c0;
  a.c_count = (int64_t)(c1 - c0);
  if (launch_encode_chunks(a, st) != cudaSuccess) return SKV_ERR_CUDA;
  if (bits && launch_ideal_final(a.bits_partials, kMaxBitsBlocks, a.head, st) != cudaSuccess)
    return SKV_ERR_CUDA;
  return SKV_OK;
}

// Size scan, compaction and header once every chunk is in its stack; reads the
// status back (synchronises).  The chunk count is checked first, so a stack
// that was never written is never copied.
int encode_finish(const skv_params *params, const Plan &pl, void *out, size_t out_capacity,
                  size_t *out_bytes, void *workspace, cudaStream_t st, double *bits = nullptr) {
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  EncodeLaunch a = encode_launch(params, pl, ws);
  WsHead h;
  int rc = read_head(a.head, &h, st);
  if (rc) return rc;
  if ((rc = status_from_flags(h.flags))) return rc;
  if (h.chunks_done != (unsigned long long)pl.geo.nchunks) return SKV_ERR_ARG;
  a.out = static_cast<uint8_t *>(out);
  a.capacity = out_capacity;
  if (h.committed) {
    // placed by skv_encode_commit: every chunk must be, then only the header is left
    if (h.committed != (unsigned long long)pl.geo.nchunks) return SKV_ERR_ARG;
    if (launch_commit_header(a, st) != cudaSuccess) return SKV_ERR_CUDA;
  } else if (launch_encode_finish(a, st) != cudaSuccess) {
    return SKV_ERR_CUDA;
  }
  if ((rc = read_head(a.head, &h, st))) return rc;
  if ((rc = status_from_flags(h.flags))) return rc;
  *out_bytes = 64 + 8 * (size_t)(pl.geo.nchunks + 1) + (size_t)h.total;
  if (bits) *bits = h.bits;
  return SKV_OK;
}

// Decode of chunks [c0, c1) of a container, enqueued on `stream` without a
// host synchronisation.  `first` zeroes the status, prepares the model tables
// (reciprocals, fingerprint, inverse p-hat table) and checks the header; later
// calls for the same container reuse them.  With a page table, mu and kv_out
// are page pools of num_pages pages of token_block * head_dim scalars.
int decode_enqueue(const skv_params *params, const Plan &pl, const void *in, size_t in_bytes,
                   uint64_t c0, uint64_t c1, const uint16_t *mu, void *kv_out,
                   const uint32_t *pages, uint64_t num_pages, bool first, void *workspace,
                   size_t workspace_bytes, skv_stream_t stream, bool check_header = true) {
  int rc = common_inputs(params, pl, kv_out, mu);
  if (rc) return rc;
  if (!in || !aligned(in, 8) || !workspace || !aligned(workspace, kAlign)) return SKV_ERR_ARG;
  if (workspace_bytes < ws_bytes_for(pl, SKV_OP_DECODE)) return SKV_ERR_CAPACITY;
  if (in_bytes < 64 + 8 * (size_t)(pl.geo.nchunks + 1)) return SKV_ERR_CORRUPT;
  if ((rc = ensure_device_tables())) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  WsHead *head = reinterpret_cast<WsHead *>(ws);
  float2 *inv = reinterpret_cast<float2 *>(ws + pl.off_inv);
  const uint32_t *ecdf = pl.dtype == SKV_BF16 ? params->ecdf : nullptr;
  int32_t *einv = pl.dtype == SKV_BF16 ? reinterpret_cast<int32_t *>(ws + pl.off_einv) : nullptr;
  float2 *gmu = pl.dtype == SKV_BF16 && !pl.order0 ? reinterpret_cast<float2 *>(ws + pl.off_dec_gmu)
                                                   : nullptr;
  if (first) {
    if (cudaMemsetAsync(head, 0, sizeof(WsHead), st) != cudaSuccess) return SKV_ERR_CUDA;
    if (launch_prep(params->sigma, pl.nsig_model, ecdf, inv, head, st) != cudaSuccess)
      return SKV_ERR_CUDA;
    if (einv && launch_einv(ecdf, einv, pl.order0 ? kO0InvN : kHinvN, gmu, st) != cudaSuccess)
      return SKV_ERR_CUDA;
  }
  DecodeLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.geo = pl.geo;
  a.dtype = pl.dtype;
  a.in = static_cast<const uint8_t *>(in);
  a.in_bytes = in_bytes;
  a.mu = mu;
  a.inv = inv;
  a.inv_chunk = nullptr;
  a.nsw = pl.nsw;
  a.order0 = pl.order0;
  a.c_begin = (int64_t)c0;
  a.c_end = (int64_t)c1;
  a.c_step = 1;
  a.ecdf_row_stride = 0;
  a.einv_row_stride = 0;
  a.adaptive = pl.adaptive;
  a.check_header = first && check_header ? 1 : 0;
  a.page_of_chunk = pages;
  a.num_pages = num_pages;
  a.page_scalars = (uint64_t)pl.geo.Tb * (uint64_t)pl.geo.D;
  if (pl.nsw) {
    ScaleLaunch sl = scale_launch(pl, params, head);
    sl.in = static_cast<const uint8_t *>(in);
    sl.in_bytes = in_bytes;
    sl.inv = reinterpret_cast<float2 *>(ws + pl.off_dec_cinv);
    sl.c_begin = (int64_t)c0;
    sl.c_end = (int64_t)c1;
    if (launch_scales(sl, st) != cudaSuccess) return SKV_ERR_CUDA;
    a.inv_chunk = sl.inv;
  }
  a.ecdf = ecdf;
  a.kv_out = kv_out;
  a.head = head;
  a.hash_words = hash_words(pl);
  a.bisect = (params->flags & SKV_FLAG_DECODE_BISECT) ? 1 : 0;
  a.einv = einv;
  a.gmu = gmu;
  if (pl.adaptive) {
    // the whole container, one phase per token block: each block's tables come
    // from the blocks decoded before it
    uint8_t *ad = ws + pl.ad_base_dec;
    uint64_t *P = reinterpret_cast<uint64_t *>(ad + pl.ad_P);
    uint64_t *Cn = reinterpret_cast<uint64_t *>(ad + pl.ad_C);
    uint32_t *Et = reinterpret_cast<uint32_t *>(ad + pl.ad_E);
    uint64_t *W = reinterpret_cast<uint64_t *>(ad + pl.ad_W);
    int32_t *Ei = reinterpret_cast<int32_t *>(ad + pl.ad_inv);
    if (launch_ad_init(ecdf, P, Cn, pl.nrows, W, pl.geo.Tb, st) != cudaSuccess) return SKV_ERR_CUDA;
    a.ecdf = Et;
    a.ecdf_row_stride = kNsymBf16 + 1;
    a.einv = Ei;
    a.einv_row_stride = kO0InvN + 1;
    a.c_step = pl.geo.ntb;
    a.c_end = pl.geo.nchunks;
    for (int64_t b = 0; b < pl.geo.ntb; ++b) {
      if (launch_ad_table(P, Et, Ei, kO0InvN, pl.nrows, st) != cudaSuccess) return SKV_ERR_CUDA;
      a.c_begin = b;
      a.check_header = b == 0 ? 1 : 0;
      if (launch_decode(a, st) != cudaSuccess) return SKV_ERR_CUDA;
      if (b + 1 < pl.geo.ntb &&
          launch_ad_update(pl.geo, static_cast<const uint16_t *>(kv_out), b, P, Cn, W, head,
                           pl.nrows, st) != cudaSuccess)
        return SKV_ERR_CUDA;
    }
    return SKV_OK;
  }
  if (launch_decode(a, st) != cudaSuccess) return SKV_ERR_CUDA;
  return SKV_OK;
}

// ---- scratch for skv_ideal_bits_noalloc ----
// A fixed device array instead of a caller workspace.  Every device that loads
// the library holds it until the process exits.  Layout: the 256-byte head,
// the per-channel reciprocal table, then the per-block fp64 partial sums.
constexpr size_t kNoallocBytes = 2u << 20;  // 2 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];
// sigma entries that fit beside the head and the largest partial-sum array,
// whatever the token count (bits_blocks never exceeds kMaxBitsBlocks)
constexpr size_t kNoallocMaxChannels =
    (kNoallocBytes - 2 * kAlign - sizeof(double) * kMaxBitsBlocks) / sizeof(float2);
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[1024];

// Device address of g_noalloc_scratch for the current device.  In host code the
// symbol's name is only a host-side stand-in, so it is looked up once per device.
int noalloc_scratch(uint8_t **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 1024) return SKV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return SKV_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = static_cast<uint8_t *>(g_noalloc_ptr[dev]);
  return SKV_OK;
}

// The ideal-bits pass enqueued on `st` over a workspace of pl.bits_total
// bytes (its head, reciprocals and partial sums); the total and the status
// land in that head.
int ideal_enqueue(const skv_params *params, const Plan &pl, const void *kv, const uint16_t *mu,
                  float *per_scalar, uint8_t *ws, cudaStream_t st) {
  WsHead *head = reinterpret_cast<WsHead *>(ws);
  if (cudaMemsetAsync(head, 0, sizeof(WsHead), st) != cudaSuccess) return SKV_ERR_CUDA;
  float2 *inv = reinterpret_cast<float2 *>(ws + pl.off_inv);
  // sigma validity only: the p-hat table enters through `phat`
  if (launch_prep(params->sigma, pl.nsig_model, nullptr, inv, head, st) != cudaSuccess) return SKV_ERR_CUDA;
  IdealLaunch a;
  a.geo = pl.geo;
  a.dtype = pl.dtype;
  a.kv = kv;
  a.mu = mu;
  a.sigma = params->sigma;
  a.sigma_chunk = nullptr;
  a.order0 = pl.order0;
  if (pl.nsw) {
    ScaleLaunch sl = scale_launch(pl, params, head);
    sl.kv = kv;
    sl.mu = mu;
    sl.sig = reinterpret_cast<float *>(ws + pl.off_bits_csig);
    if (launch_scales(sl, st) != cudaSuccess) return SKV_ERR_CUDA;
    a.sigma_chunk = sl.sig;
  }
  a.phat = params->phat;
  a.per_scalar = per_scalar;
  a.partials = reinterpret_cast<double *>(ws + pl.off_bits);
  a.nblocks = pl.bits_blocks;
  a.td_rcp = ~0ull / ((uint64_t)pl.geo.T * (uint64_t)pl.geo.D);
  a.head = head;
  if (pl.adaptive) {
    // per-row models, one phase per token block, partial sums in a fixed order
    uint8_t *ad = ws + pl.ad_base_bits;
    uint64_t *P = reinterpret_cast<uint64_t *>(ad + pl.ad_P);
    uint64_t *Cn = reinterpret_cast<uint64_t *>(ad + pl.ad_C);
    uint64_t *W = reinterpret_cast<uint64_t *>(ad + pl.ad_W);
    double *part = reinterpret_cast<double *>(ad + pl.ad_part);
    const uint32_t *ecdf = params->ecdf;
    const uint16_t *kv16 = static_cast<const uint16_t *>(kv);
    if (launch_ad_init(ecdf, P, Cn, pl.nrows, W, pl.geo.Tb, st) != cudaSuccess) return SKV_ERR_CUDA;
    for (int64_t b = 0; b < pl.geo.ntb; ++b) {
      if (launch_ad_ideal(pl.geo, kv16, b, P, per_scalar, part + b * pl.nrows * pl.ad_bx, pl.ad_bx,
                          head, pl.nrows, st) != cudaSuccess)
        return SKV_ERR_CUDA;
      if (b + 1 < pl.geo.ntb &&
          launch_ad_update(pl.geo, kv16, b, P, Cn, W, head, pl.nrows, st) != cudaSuccess)
        return SKV_ERR_CUDA;
    }
    if (launch_ideal_final(part, (int)(pl.geo.ntb * pl.nrows * pl.ad_bx), head, st) != cudaSuccess)
      return SKV_ERR_CUDA;
  } else if (launch_ideal(a, st) != cudaSuccess) {
    return SKV_ERR_CUDA;
  }
  return SKV_OK;
}

}  // namespace

extern "C" {

size_t skv_max_encoded_bytes(const skv_params *params, const skv_shape *shape) {
  Plan pl;
  if (make_plan(params, shape, &pl) != SKV_OK) return 0;
  return 64 + 8 * (size_t)(pl.geo.nchunks + 1) +
         4 * ((size_t)pl.geo.n + (2 * (size_t)pl.geo.G + (size_t)pl.nsw) * (size_t)pl.geo.nchunks);
}

size_t skv_workspace_bytes(const skv_params *params, const skv_shape *shape, int op) {
  Plan pl;
  if (make_plan(params, shape, &pl) != SKV_OK) return 0;
  if (op < SKV_OP_ENCODE || op > SKV_OP_MODEL_BITS) return 0;
  return ws_bytes_for(pl, op);
}

int skv_encode(const skv_params *params, const skv_shape *shape, const void *kv,
               const uint16_t *mu, void *out, size_t out_capacity, size_t *out_bytes,
               void *workspace, size_t workspace_bytes, skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if ((rc = common_inputs(params, pl, kv, mu))) return rc;
  if (!out || !out_bytes || !workspace || !aligned(out, 8) || !aligned(workspace, kAlign))
    return SKV_ERR_ARG;
  if (workspace_bytes < ws_bytes_for(pl, SKV_OP_ENCODE)) return SKV_ERR_CAPACITY;
  if ((rc = ensure_device_tables())) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!pl.adaptive) {
    if ((rc = encode_enqueue(params, pl, kv, mu, 0, (uint64_t)pl.geo.nchunks, true, workspace, st)))
      return rc;
    return encode_finish(params, pl, out, out_capacity, out_bytes, workspace, st);
  }
  // adaptive counts: one phase per token block -- the rows' tables, block b of
  // every row, then the update from that block
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  if ((rc = encode_enqueue(params, pl, kv, mu, 0, 0, true, workspace, st))) return rc;
  EncodeLaunch a = encode_launch(params, pl, ws);
  a.kv = kv;
  a.mu = mu;
  uint8_t *ad = ws + pl.ad_base_enc;
  uint64_t *P = reinterpret_cast<uint64_t *>(ad + pl.ad_P);
  uint64_t *Cn = reinterpret_cast<uint64_t *>(ad + pl.ad_C);
  uint32_t *Et = reinterpret_cast<uint32_t *>(ad + pl.ad_E);
  uint64_t *W = reinterpret_cast<uint64_t *>(ad + pl.ad_W);
  if (launch_ad_init(params->ecdf, P, Cn, pl.nrows, W, pl.geo.Tb, st) != cudaSuccess)
    return SKV_ERR_CUDA;
  a.ecdf = Et;
  a.ecdf_row_stride = kNsymBf16 + 1;
  a.c_step = pl.geo.ntb;
  a.c_count = pl.nrows;
  for (int64_t b = 0; b < pl.geo.ntb; ++b) {
    if (launch_ad_table(P, Et, nullptr, 0, pl.nrows, st) != cudaSuccess) return SKV_ERR_CUDA;
    a.c_first = b;
    if (launch_encode_chunks(a, st) != cudaSuccess) return SKV_ERR_CUDA;
    if (b + 1 < pl.geo.ntb &&
        launch_ad_update(pl.geo, static_cast<const uint16_t *>(kv), b, P, Cn, W, a.head, pl.nrows,
                         st) != cudaSuccess)
      return SKV_ERR_CUDA;
  }
  return encode_finish(params, pl, out, out_capacity, out_bytes, workspace, st);
}

int skv_encode_with_bits(const skv_params *params, const skv_shape *shape, const void *kv,
                         const uint16_t *mu, void *out, size_t out_capacity, size_t *out_bytes,
                         float *per_scalar, double *total, void *workspace,
                         size_t workspace_bytes, skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  // adaptive tables change between token blocks: the two passes apart
  if (pl.adaptive) return SKV_ERR_ARG;
  if ((rc = common_inputs(params, pl, kv, mu))) return rc;
  if (!out || !out_bytes || !total || !workspace || !aligned(out, 8) ||
      !aligned(workspace, kAlign))
    return SKV_ERR_ARG;
  if (per_scalar && !aligned(per_scalar, 16)) return SKV_ERR_ARG;
  if (pl.dtype == SKV_BF16 && (!params->phat || !aligned(params->phat, 4))) return SKV_ERR_ARG;
  if (workspace_bytes < ws_bytes_for(pl, SKV_OP_ENCODE)) return SKV_ERR_CAPACITY;
  if ((rc = ensure_device_tables())) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  if (encode_fuses_bits(pl.dtype == SKV_BF16 ? 0 : 1, pl.order0, pl.nsw > 0, pl.geo.nchunks,
                        pl.geo.G)) {
    if ((rc = encode_enqueue(params, pl, kv, mu, 0, (uint64_t)pl.geo.nchunks, true, workspace, st,
                             true, per_scalar)))
      return rc;
    return encode_finish(params, pl, out, out_capacity, out_bytes, workspace, st, total);
  }
  // the encoder, then the ideal-bits pass on a workspace of its own behind it
  uint8_t *bws = ws + pl.off_enc_bits;
  if ((rc = encode_enqueue(params, pl, kv, mu, 0, (uint64_t)pl.geo.nchunks, true, workspace, st)))
    return rc;
  if ((rc = ideal_enqueue(params, pl, kv, mu, per_scalar, bws, st))) return rc;
  if ((rc = encode_finish(params, pl, out, out_capacity, out_bytes, workspace, st))) return rc;
  WsHead h;
  if ((rc = read_head(reinterpret_cast<WsHead *>(bws), &h, st))) return rc;
  if ((rc = status_from_flags(h.flags))) return rc;
  *total = h.bits;
  return SKV_OK;
}

int skv_encode_with_bits_fused(const skv_params *params, const skv_shape *shape, int *fused) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if (!fused || pl.adaptive) return SKV_ERR_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SKV_ERR_CUDA;
  *fused = encode_fuses_bits(pl.dtype == SKV_BF16 ? 0 : 1, pl.order0, pl.nsw > 0,
                             pl.geo.nchunks, pl.geo.G)
               ? 1 : 0;
  return SKV_OK;
}

int skv_encode_range(const skv_params *params, const skv_shape *shape, const void *kv,
                     const uint16_t *mu, uint64_t chunk_begin, uint64_t chunk_end,
                     int range_flags, void *workspace, size_t workspace_bytes,
                     skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if (range_flags & ~(SKV_RANGE_FIRST | SKV_RANGE_BITS)) return SKV_ERR_ARG;
  // adaptive tables depend on every earlier block of a row: whole caches only
  if (pl.adaptive) return SKV_ERR_ARG;
  if (chunk_begin > chunk_end || chunk_end > (uint64_t)pl.geo.nchunks) return SKV_ERR_ARG;
  if ((rc = common_inputs(params, pl, kv, mu))) return rc;
  if (!workspace || !aligned(workspace, kAlign)) return SKV_ERR_ARG;
  const bool bits = (range_flags & SKV_RANGE_BITS) != 0;
  // the bits ride along with the bf16 mixture coder only (the fused encoder)
  if (bits && (pl.dtype != SKV_BF16 || pl.order0 || !params->phat || !aligned(params->phat, 4)))
    return SKV_ERR_ARG;
  if (workspace_bytes < ws_bytes_for(pl, SKV_OP_ENCODE)) return SKV_ERR_CAPACITY;
  if ((rc = ensure_device_tables())) return rc;
  return encode_enqueue(params, pl, kv, mu, chunk_begin, chunk_end,
                        (range_flags & SKV_RANGE_FIRST) != 0, workspace,
                        reinterpret_cast<cudaStream_t>(stream), bits && chunk_end > chunk_begin);
}

int skv_encode_range_bits(const skv_params *params, const skv_shape *shape, double *total,
                          void *workspace, size_t workspace_bytes, skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if (pl.adaptive || !total || !workspace || !aligned(workspace, kAlign)) return SKV_ERR_ARG;
  if (workspace_bytes < ws_bytes_for(pl, SKV_OP_ENCODE)) return SKV_ERR_CAPACITY;
  WsHead h;
  if ((rc = read_head(reinterpret_cast<WsHead *>(workspace), &h,
                      reinterpret_cast<cudaStream_t>(stream))))
    return rc;
  if ((rc = status_from_flags(h.flags))) return rc;
  *total = h.bits;
  return SKV_OK;
}

int skv_encode_finish(const skv_params *params, const skv_shape *shape, void *out,
                      size_t out_capacity, size_t *out_bytes, void *workspace,
                      size_t workspace_bytes, skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if (pl.adaptive) return SKV_ERR_ARG;
  if (!out || !out_bytes || !workspace || !aligned(out, 8) || !aligned(workspace, kAlign))
    return SKV_ERR_ARG;
  if (workspace_bytes < ws_bytes_for(pl, SKV_OP_ENCODE)) return SKV_ERR_CAPACITY;
  return encode_finish(params, pl, out, out_capacity, out_bytes, workspace,
                       reinterpret_cast<cudaStream_t>(stream));
}

int skv_encode_commit(const skv_params *params, const skv_shape *shape, uint64_t chunk_begin,
                      uint64_t chunk_end, void *out, size_t out_capacity, uint64_t *end_bytes,
                      void *workspace, size_t workspace_bytes, skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if (pl.adaptive) return SKV_ERR_ARG;
  if (chunk_begin > chunk_end || chunk_end > (uint64_t)pl.geo.nchunks) return SKV_ERR_ARG;
  if (!out || !workspace || !aligned(out, 8) || !aligned(workspace, kAlign)) return SKV_ERR_ARG;
  if (workspace_bytes < ws_bytes_for(pl, SKV_OP_ENCODE)) return SKV_ERR_CAPACITY;
  if (out_capacity < 64 + 8 * (size_t)(pl.geo.nchunks + 1)) return SKV_ERR_CAPACITY;
  if (end_bytes && !aligned(end_bytes, 8)) return SKV_ERR_ARG;
  if (chunk_begin == chunk_end && !end_bytes) return SKV_OK;
  EncodeLaunch a = encode_launch(params, pl, static_cast<uint8_t *>(workspace));
  a.out = static_cast<uint8_t *>(out);
  a.capacity = out_capacity;
  a.c_first = (int64_t)chunk_begin;
  a.c_count = (int64_t)(chunk_end - chunk_begin);
  if (launch_encode_commit(a, end_bytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SKV_ERR_CUDA;
  return SKV_OK;
}

int skv_model_fingerprint(const skv_params *params, const skv_shape *shape,
                          uint64_t *fingerprint, void *workspace, size_t workspace_bytes,
                          skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if (!fingerprint || !workspace || !aligned(workspace, kAlign)) return SKV_ERR_ARG;
  if (!pl.order0 && (!params->sigma || !aligned(params->sigma, 4))) return SKV_ERR_ARG;
  if (pl.dtype == SKV_BF16 && (!params->ecdf || !aligned(params->ecdf, 4))) return SKV_ERR_ARG;
  // the head and the reciprocal table, which every operation's workspace starts with
  if (workspace_bytes < pl.off_inv + sizeof(float2) * (size_t)pl.nsig) return SKV_ERR_CAPACITY;
  if ((rc = ensure_device_tables())) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  WsHead *head = reinterpret_cast<WsHead *>(ws);
  if (cudaMemsetAsync(head, 0, sizeof(WsHead), st) != cudaSuccess) return SKV_ERR_CUDA;
  if (launch_prep(params->sigma, pl.nsig_model, pl.dtype == SKV_BF16 ? params->ecdf : nullptr,
                  reinterpret_cast<float2 *>(ws + pl.off_inv), head, st) != cudaSuccess)
    return SKV_ERR_CUDA;
  WsHead h;
  if ((rc = read_head(head, &h, st))) return rc;
  if ((rc = status_from_flags(h.flags))) return rc;
  *fingerprint = mix64(h.hash_acc ^ hash_words(pl));
  return SKV_OK;
}

namespace {
uint64_t get_u64(const uint8_t *p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}
}  // namespace

int skv_merge_parts(const skv_params *params, const skv_shape *shape, uint64_t fingerprint,
                    const void *const *parts, const size_t *part_bytes, int nparts, void *out,
                    size_t out_capacity, size_t *out_bytes) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if (!parts || !part_bytes || nparts < 1 || !out || !out_bytes) return SKV_ERR_ARG;
  const uint32_t features = (pl.nsw ? 1u : 0u) | (pl.order0 ? 2u : 0u) | (pl.adaptive ? 4u : 0u);
  // every part is a container of a contiguous layer range of this cache, in
  // order: its header must be this cache's but for the layer count, the chunk
  // count, the payload size and the fingerprint (which covers its own slice)
  int64_t layers = 0, chunks = 0;
  uint64_t payload = 0;
  for (int i = 0; i < nparts; ++i) {
    const uint8_t *p = static_cast<const uint8_t *>(parts[i]);
    if (!p || part_bytes[i] < 64) return SKV_ERR_CORRUPT;
    const int32_t pl_layers = (int32_t)(p[8] | p[9] << 8 | p[10] << 16 | (uint32_t)p[11] << 24);
    if (pl_layers <= 0 || pl_layers > pl.geo.L - layers) return SKV_ERR_CORRUPT;
    Geo g = pl.geo;
    g.L = pl_layers;
    g.nchunks = (int64_t)pl_layers * 2 * g.H * g.ntb;
    const uint64_t hb = 64 + 8 * (uint64_t)(g.nchunks + 1);
    if (part_bytes[i] < hb) return SKV_ERR_CORRUPT;
    const uint64_t pp = part_bytes[i] - hb;
    uint8_t want[64];
    make_header(want, g, pl.dtype, pp, get_u64(p + 56), features);
    if (std::memcmp(want, p, 64) != 0) return SKV_ERR_CORRUPT;
    if (get_u64(p + 64) != 0 || get_u64(p + 64 + 8 * (uint64_t)g.nchunks) != pp)
      return SKV_ERR_CORRUPT;
    layers += pl_layers;
    chunks += g.nchunks;
    payload += pp;
  }
  if (layers != pl.geo.L || chunks != pl.geo.nchunks) return SKV_ERR_ARG;
  const uint64_t hbytes = 64 + 8 * (uint64_t)(pl.geo.nchunks + 1);
  if (out_capacity < hbytes + payload) return SKV_ERR_CAPACITY;
  uint8_t *o = static_cast<uint8_t *>(out);
  make_header(o, pl.geo, pl.dtype, payload, fingerprint, features);
  // the offsets: each part's own, shifted by the exclusive scan of the payload
  // sizes of the parts before it; then the payloads one after another
  uint64_t base = 0, c = 0;
  for (int i = 0; i < nparts; ++i) {
    const uint8_t *p = static_cast<const uint8_t *>(parts[i]);
    const int64_t nc = ((int64_t)(p[8] | p[9] << 8 | p[10] << 16 | (uint32_t)p[11] << 24)) * 2 *
                       pl.geo.H * pl.geo.ntb;
    const uint64_t hb = 64 + 8 * (uint64_t)(nc + 1);
    const uint64_t pp = part_bytes[i] - hb;
    uint64_t prev = 0;
    for (int64_t k = 0; k < nc; ++k) {
      const uint64_t off = get_u64(p + 64 + 8 * (uint64_t)k);
      if (off < prev || off > pp || (off & 3)) return SKV_ERR_CORRUPT;
      prev = off;
      put_u64(o + 64 + 8 * (c + (uint64_t)k), base + off);
    }
    std::memcpy(o + hbytes + base, p + hb, pp);
    base += pp;
    c += (uint64_t)nc;
  }
  put_u64(o + 64 + 8 * c, base);
  *out_bytes = hbytes + payload;
  return SKV_OK;
}

int skv_decode(const skv_params *params, const skv_shape *shape, const void *in, size_t in_bytes,
               const uint16_t *mu, void *kv_out, void *workspace, size_t workspace_bytes,
               skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if ((rc = decode_enqueue(params, pl, in, in_bytes, 0, (uint64_t)pl.geo.nchunks, mu, kv_out,
                           nullptr, 0, true, workspace, workspace_bytes, stream)))
    return rc;
  WsHead h;
  if ((rc = read_head(static_cast<WsHead *>(workspace), &h,
                      reinterpret_cast<cudaStream_t>(stream))))
    return rc;
  return status_from_flags(h.flags);
}

int skv_decode_range(const skv_params *params, const skv_shape *shape, const void *in,
                     size_t in_bytes, uint64_t chunk_begin, uint64_t chunk_end,
                     const uint16_t *mu, void *kv_out, const uint32_t *page_of_chunk,
                     uint64_t num_pages, int range_flags, void *workspace,
                     size_t workspace_bytes, skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if (range_flags & ~(SKV_RANGE_FIRST | SKV_RANGE_PARTIAL)) return SKV_ERR_ARG;
  // adaptive tables depend on every earlier block of a row: whole containers only
  if (pl.adaptive) return SKV_ERR_ARG;
  if (chunk_begin > chunk_end || chunk_end > (uint64_t)pl.geo.nchunks) return SKV_ERR_ARG;
  if (page_of_chunk && (!aligned(page_of_chunk, 4) || num_pages == 0)) return SKV_ERR_ARG;
  return decode_enqueue(params, pl, in, in_bytes, chunk_begin, chunk_end, mu, kv_out,
                        page_of_chunk, num_pages, (range_flags & SKV_RANGE_FIRST) != 0, workspace,
                        workspace_bytes, stream, (range_flags & SKV_RANGE_PARTIAL) == 0);
}

int skv_decode_status(const void *workspace, skv_stream_t stream) {
  if (!workspace || !aligned(workspace, kAlign)) return SKV_ERR_ARG;
  WsHead h;
  int rc = read_head(static_cast<WsHead *>(const_cast<void *>(workspace)), &h,
                     reinterpret_cast<cudaStream_t>(stream));
  if (rc) return rc;
  return status_from_flags(h.flags);
}

int skv_ideal_bits(const skv_params *params, const skv_shape *shape, const void *kv,
                   const uint16_t *mu, float *per_scalar, double *total, void *workspace,
                   size_t workspace_bytes, skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if ((rc = common_inputs(params, pl, kv, mu))) return rc;
  if (!total || !workspace || !aligned(workspace, kAlign)) return SKV_ERR_ARG;
  if (per_scalar && !aligned(per_scalar, 16)) return SKV_ERR_ARG;
  if (pl.dtype == SKV_BF16 && (!params->phat || !aligned(params->phat, 4))) return SKV_ERR_ARG;
  if (workspace_bytes < ws_bytes_for(pl, SKV_OP_IDEAL_BITS)) return SKV_ERR_CAPACITY;
  if ((rc = ensure_device_tables())) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  if ((rc = ideal_enqueue(params, pl, kv, mu, per_scalar, ws, st))) return rc;
  WsHead *head = reinterpret_cast<WsHead *>(ws);
  WsHead h;
  if ((rc = read_head(head, &h, st))) return rc;
  if ((rc = status_from_flags(h.flags))) return rc;
  *total = h.bits;
  return SKV_OK;
}

int skv_model_bits(const skv_params *params, const skv_shape *shape, const void *kv,
                   const uint16_t *mu, float *per_scalar, double *total, void *workspace,
                   size_t workspace_bytes, skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  // adaptive tables change from one token block to the next: no single pass
  if (pl.adaptive) return SKV_ERR_ARG;
  if ((rc = common_inputs(params, pl, kv, mu))) return rc;
  if (!total || !workspace || !aligned(workspace, kAlign)) return SKV_ERR_ARG;
  if (per_scalar && !aligned(per_scalar, 16)) return SKV_ERR_ARG;
  if (workspace_bytes < ws_bytes_for(pl, SKV_OP_MODEL_BITS)) return SKV_ERR_CAPACITY;
  if ((rc = ensure_device_tables())) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  WsHead *head = reinterpret_cast<WsHead *>(ws);
  if (cudaMemsetAsync(head, 0, sizeof(WsHead), st) != cudaSuccess) return SKV_ERR_CUDA;
  float2 *inv = reinterpret_cast<float2 *>(ws + pl.off_inv);
  const uint32_t *ecdf = pl.dtype == SKV_BF16 ? params->ecdf : nullptr;
  // the same sigma and E_q checks as encode
  if (launch_prep(params->sigma, pl.nsig_model, ecdf, inv, head, st) != cudaSuccess)
    return SKV_ERR_CUDA;
  ModelBitsLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.geo = pl.geo;
  a.dtype = pl.dtype;
  a.order0 = pl.order0;
  a.kv = kv;
  a.mu = mu;
  a.inv = inv;
  if (pl.nsw) {
    // the encoder's choice of scales, recomputed from the inputs
    ScaleLaunch sl = scale_launch(pl, params, head);
    sl.kv = kv;
    sl.mu = mu;
    sl.inv = reinterpret_cast<float2 *>(ws + pl.off_mb_cinv);
    if (launch_scales(sl, st) != cudaSuccess) return SKV_ERR_CUDA;
    a.inv_chunk = sl.inv;
  }
  a.ecdf = ecdf;
  a.per_scalar = per_scalar;
  a.partials = reinterpret_cast<double *>(ws + pl.off_bits);
  a.nblocks = pl.bits_blocks;
  a.head = head;
  if (launch_model_bits(a, st) != cudaSuccess) return SKV_ERR_CUDA;
  WsHead h;
  if ((rc = read_head(head, &h, st))) return rc;
  if ((rc = status_from_flags(h.flags))) return rc;
  *total = h.bits;
  return SKV_OK;
}

int skv_ideal_bits_noalloc(const skv_params *params, const skv_shape *shape, const void *kv,
                           const uint16_t *mu, float *per_scalar, double *total,
                           skv_stream_t stream) {
  Plan pl;
  int rc = make_plan(params, shape, &pl);
  if (rc) return rc;
  if ((rc = common_inputs(params, pl, kv, mu))) return rc;
  if (!total) return SKV_ERR_ARG;
  // the per-(chunk, channel) table of per-block scales grows with the cache;
  // the order-0 baseline has its own entry points' workspace only
  if (pl.nsw || pl.order0) return SKV_ERR_ARG;
  if (per_scalar && !aligned(per_scalar, 16)) return SKV_ERR_ARG;
  if (pl.dtype == SKV_BF16 && (!params->phat || !aligned(params->phat, 4))) return SKV_ERR_ARG;
  // the same layout as the workspace of skv_ideal_bits, inside the fixed array;
  // the sigma limit is the documented one, the byte check guards the layout
  if ((size_t)pl.nsig > kNoallocMaxChannels) return SKV_ERR_CAPACITY;
  if (ws_bytes_for(pl, SKV_OP_IDEAL_BITS) > kNoallocBytes) return SKV_ERR_CAPACITY;
  if ((rc = ensure_device_tables())) return rc;
  uint8_t *ws = nullptr;
  if ((rc = noalloc_scratch(&ws))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  WsHead *head = reinterpret_cast<WsHead *>(ws);
  // the array keeps the previous call's contents: the flags and sums start at zero
  if (cudaMemsetAsync(head, 0, sizeof(WsHead), st) != cudaSuccess) return SKV_ERR_CUDA;
  float2 *inv = reinterpret_cast<float2 *>(ws + pl.off_inv);
  if (launch_prep(params->sigma, pl.nsig_model, nullptr, inv, head, st) != cudaSuccess) return SKV_ERR_CUDA;
  IdealLaunch a;
  a.geo = pl.geo;
  a.dtype = pl.dtype;
  a.kv = kv;
  a.mu = mu;
  a.sigma = params->sigma;
  a.sigma_chunk = nullptr;
  a.order0 = 0;
  a.phat = params->phat;
  a.per_scalar = per_scalar;
  a.partials = reinterpret_cast<double *>(ws + pl.off_bits);
  a.nblocks = pl.bits_blocks;
  a.td_rcp = ~0ull / ((uint64_t)pl.geo.T * (uint64_t)pl.geo.D);
  a.head = head;
  if (launch_ideal(a, st) != cudaSuccess) return SKV_ERR_CUDA;
  WsHead h;
  if ((rc = read_head(head, &h, st))) return rc;
  if ((rc = status_from_flags(h.flags))) return rc;
  *total = h.bits;
  return SKV_OK;
}

size_t skv_ideal_bits_noalloc_max_channels(void) { return kNoallocMaxChannels; }

int skv_build_ecdf(const uint64_t *counts, uint32_t *ecdf, float *phat) {
  if (!counts || !ecdf) return SKV_ERR_ARG;
  // ranks in value order: negatives from -inf up to -0, then +0 up to +inf
  auto pattern = [](int r) -> uint32_t {
    uint32_t key = (uint32_t)(r + 127);
    return (key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu);
  };
  unsigned __int128 tot = 0;
  for (int r = 0; r < kNsymBf16; ++r) tot += (unsigned __int128)counts[pattern(r)] + 1;
  if (tot >= ((unsigned __int128)1 << 37)) return SKV_ERR_ARG;
  const uint64_t S_tot = (uint64_t)tot;
  uint64_t S = 0;
  for (int r = 0; r <= kNsymBf16; ++r) {
    ecdf[r] = (uint32_t)(((unsigned __int128)S << 26) / S_tot);
    if (r < kNsymBf16) {
      const uint64_t c = counts[pattern(r)] + 1;
      if (phat) phat[r] = (float)((double)c / (double)S_tot);
      S += c;
    }
  }
  return SKV_OK;
}

int skv_phi_table(uint32_t *table) {
  if (!table) return SKV_ERR_ARG;
  std::call_once(g_const_once, build_constants);
  std::memcpy(table, g_phi_host, sizeof(g_phi_host));
  return SKV_OK;
}

const char *skv_strerror(int status) {
  switch (status) {
    case SKV_OK: return "ok";
    case SKV_ERR_ARG: return "invalid argument";
    case SKV_ERR_CAPACITY: return "output buffer or workspace too small";
    case SKV_ERR_SYMBOL: return "NaN symbol in the KV input";
    case SKV_ERR_PARAM: return "invalid sigma, mu or p-hat table";
    case SKV_ERR_CORRUPT: return "corrupt or mismatched container";
    case SKV_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int skv_version(void) { return 1; }

}  // extern "C"
