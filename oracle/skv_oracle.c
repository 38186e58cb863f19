/*
 * skv_oracle.c -- the ORACLE for speculative KV coding.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, the smoke() check in
 * __graft_entry__.py and the cpu_baseline / reference leg of bench.py may load
 * or call this library.  It shares no code, header, table or constant
 * generator with the CUDA library in lossless_kv_cache_fixed_gb300/csrc/, and
 * neither side includes the other.  It is deliberately plain: one scalar at a
 * time, single-threaded, every step written in the order the method states it.
 *
 * Sources, cited by page title and section heading:
 *   [P1] "推测式 KV 编码无损压缩 KV 缓存最高可达约 4 倍" (Speculative KV coding:
 *        losslessly compressing the KV cache by up to ~4x), lpnh.cn/news/878951.
 *        Sections: "KV 缓存并非真正随机" (the cache is not random: cost is the
 *        cross-entropy), "q 应是什么样的" (what q should look like: Gaussian
 *        N(mu, sigma^2)), "什么能预测 KV 缓存" (what can predict the cache: the
 *        arithmetic coder maps (KV, mu, sigma) to bits and back), "早期结果"
 *        (early results: the 0.95/0.03/0.02 mixture with the empirical bf16
 *        distribution; sigma^2 per (kv, head, channel)), "原生 FP8 KV 缓存"
 *        (native FP8 cache: bin-integrated N(mu, sigma^2) over e4m3 symbols),
 *        "下一步计划" (next steps: (mu, sigma) must be bit-identical at both ends).
 *   [P3] "推测解码与KV缓存压缩的协同优化" (hotdry blog), section
 *        "工程实现的关键约束" (engineering constraints: bit-identical predictor).
 *
 * Where the pages are silent the oracle takes these readings (spec v1):
 *   R1  alphabet: bf16 = the 65,282 non-NaN patterns (+-0 and +-inf included);
 *       e4m3 (OCP "fn") = the 254 non-NaN codes.  A NaN symbol is an error.
 *   R2  rank = position in increasing value order, -0 before +0.
 *   R3  a symbol's bin is its round-to-nearest interval [lo, hi): edges at the
 *       midpoints of neighbouring values; the extreme finite values own the
 *       half-lines to -inf / +inf; +-inf have zero-width bins.
 *   R4  Phi is evaluated from a 8193-entry table T[i] = RNE(2^26 Phi(-8+i/512))
 *       by integer linear interpolation, with the fraction taken EXACTLY:
 *       i = floor(t), fr = floor(65536 (t - floor t)) in exact arithmetic,
 *       t = 512 z.
 *   R5  z is fp32: d = lo - mu, z1 = d * (1/sigma), z3 = d * (1/(3 sigma)),
 *       each op rounded to nearest, no fused multiply-add.
 *   R6  mixture in integers: F100 = 95 Phi_q(z1) + 3 Phi_q(z3) + 2 E_q[r],
 *       E_q[r] = floor(2^26 S[r] / S_tot), S[r] = sum_{j<r} (count_j + 1).
 *   R7  cum(r) = floor(K F / one) + r,  K = 2^M - |alphabet|; M = 28 (bf16,
 *       one = 100 * 2^26) or 16 (e4m3, F = Phi_q(z1), one = 2^26).
 *   R8  coder: interleaved rANS, 64-bit state, L = 2^31, 32-bit words,
 *       lane/round layout and container as documented at or_encode_chunk.
 *   R9  sigma is given per (layer, kv, head, channel); valid iff finite,
 *       >= FLT_MIN and 3 sigma finite.  mu must be finite.
 *   R10 ideal bits = -log2 q(x), q the exact bin mass of the continuous model.
 *   R11 optional per-block sigma scales (section "下一步计划": sigma varies
 *       with prompt and position, so a static per-channel sigma costs bits):
 *       one byte s per (chunk, 8-channel group), sigma_eff = fp32(sigma m(s)),
 *       m(s) = fp32(2^((s - 128) / 32)).  s = b + C, b the median of the
 *       group's bins of |x - mu| / sigma, a bin being 32 (exponent + mantissa
 *       fraction) read from the fp32 bits (floor of 32 log2 with the mantissa
 *       taken as linear: 2.33 bins low on average).  C puts s at 128 when the
 *       residuals follow the model with the static sigma: the median of |r|
 *       is 0.706 sigma under 0.95 N(0, s^2) + 0.03 N(0, 9 s^2) (bf16: C = 18)
 *       and 0.6745 sigma under N(0, s^2) (e4m3: C = 21).  A group whose
 *       sigma_eff would leave the valid range takes s = 128.  The bytes open
 *       the chunk's payload.
 *   R12 order-0 baseline (the pages' introduction: an entropy coder over the
 *       bf16 symbols alone reaches about 11 bits per value): the same coder
 *       with weights (0, 0, 100), i.e. q = p-hat, one static histogram with no
 *       mu and no sigma.  bf16 only; mu and sigma are never read (they may be
 *       NULL), sigma is left out of the fingerprint, header feature bit 1.
 *   R13 adaptive counts (the virtual-sliding-window estimator of the page
 *       "KV 缓存压缩的熵估计与动态适应", sections "虚拟滑动窗口的设计原理",
 *       "平滑更新算法", "参数配置建议"): the order-0 coder with one model per
 *       (layer, kv, head) row, updated after every chunk, so the token block
 *       is the update period N_update.  Integers only: A = round(0.97 2^16) =
 *       63570, B = round(0.9 2^16) = 58982; token weights W[Tb-1] = 2^16,
 *       W[t-1] = floor(W[t] A / 2^16) (alpha^(Tb-1-t)), block decay
 *       Dk = floor(W[0] A / 2^16); counts C_0 = 0,
 *       C_{b+1}[r] = floor(C_b[r] Dk / 2^16) + sum over the block's scalars of
 *       rank r of W[token in block]; P_0[r] = (E_q[r+1] - E_q[r]) 2^6 (the
 *       calibration prior, the page's cold-start remedy),
 *       P_{b+1}[r] = floor((B P_b[r] + (2^16 - B) floor(2^32 C[r] / sum C)) / 2^16);
 *       block b codes with E[r] = floor(2^26 S[r] / S_tot), S over P_b + 1.
 *       bf16 only, weights (0, 0, 100), no block scales; header feature bit 2.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "skv_oracle.h"

#define NSYM_BF16 65282
#define NSYM_E4M3 254
#define PHI_N 8193
#define PHI_ONE 67108864u /* 2^26 */
#define STATE_L 0x80000000ull /* rANS lower bound L = 2^31 */

/* ------------------------------------------------------------------ */
/* Alphabets (R1, R2, R3): built from the plain definitions by sorting. */
/* ------------------------------------------------------------------ */

static int g_ready = 0;
static int32_t g_rank_bf16[65536];
static uint16_t g_bits_bf16[NSYM_BF16];
static float g_lo_bf16[NSYM_BF16 + 1];
static int32_t g_rank_e4m3[256];
static uint8_t g_bits_e4m3[NSYM_E4M3];
static float g_lo_e4m3[NSYM_E4M3 + 1];
static uint32_t g_phi[PHI_N];

static int bf16_is_nan(uint16_t u) {
  return ((u & 0x7F80u) == 0x7F80u) && ((u & 0x007Fu) != 0);
}

double or_bf16_value(uint16_t u) {
  uint32_t w = (uint32_t)u << 16;
  float f;
  memcpy(&f, &w, 4);
  return (double)f;
}

static int e4m3_is_nan(uint8_t u) { return (u & 0x7Fu) == 0x7Fu; }

/* OCP FP8 E4M3 ("fn"): bias 7, no infinities, S.1111.111 is NaN. */
double or_e4m3_value(uint8_t u) {
  int s = u >> 7, e = (u >> 3) & 15, m = u & 7;
  double v = e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp(m / 8.0, -6);
  return s ? -v : v;
}

/* order by value; the only equal values are -0 and +0: negative sign first */
static int cmp_bf16(const void *a, const void *b) {
  uint16_t ua = *(const uint16_t *)a, ub = *(const uint16_t *)b;
  double va = or_bf16_value(ua), vb = or_bf16_value(ub);
  if (va < vb) return -1;
  if (va > vb) return 1;
  return (int)(ub >> 15) - (int)(ua >> 15);
}

static int cmp_e4m3(const void *a, const void *b) {
  uint8_t ua = *(const uint8_t *)a, ub = *(const uint8_t *)b;
  double va = or_e4m3_value(ua), vb = or_e4m3_value(ub);
  if (va < vb) return -1;
  if (va > vb) return 1;
  return (int)(ub >> 7) - (int)(ua >> 7);
}

/* lower edge of bin r from the values of ranks r-1 and r (R3) */
static float bin_lo(double below, double here) {
  if (below == -INFINITY) return -INFINITY; /* -inf is zero-width; -max owns (-inf, .) */
  if (here == INFINITY) return INFINITY;    /* +max owns (., +inf); +inf is zero-width */
  return (float)((below + here) / 2.0);     /* a midpoint: exact in binary32 */
}

void or_phi_table(uint32_t *T) {
  /* Phi(z) = erfc(-z / sqrt 2) / 2, scaled by 2^26, rounded to nearest even */
  for (int i = 0; i < PHI_N; ++i) {
    double z = -8.0 + (double)i / 512.0;
    double v = ldexp(0.5 * erfc(-z * M_SQRT1_2), 26);
    T[i] = (uint32_t)nearbyint(v);
  }
  T[0] = 0;
  T[PHI_N - 1] = PHI_ONE;
}

static void init_tables(void) {
  if (g_ready) return;
  int n = 0;
  uint16_t all[65536];
  for (uint32_t u = 0; u < 65536; ++u)
    if (!bf16_is_nan((uint16_t)u)) all[n++] = (uint16_t)u;
  qsort(all, (size_t)n, sizeof(uint16_t), cmp_bf16);
  for (uint32_t u = 0; u < 65536; ++u) g_rank_bf16[u] = -1;
  for (int r = 0; r < n; ++r) {
    g_bits_bf16[r] = all[r];
    g_rank_bf16[all[r]] = r;
  }
  g_lo_bf16[0] = -INFINITY;
  for (int r = 1; r < n; ++r)
    g_lo_bf16[r] = bin_lo(or_bf16_value(all[r - 1]), or_bf16_value(all[r]));
  g_lo_bf16[n] = INFINITY;

  uint8_t e[256];
  int m = 0;
  for (uint32_t u = 0; u < 256; ++u)
    if (!e4m3_is_nan((uint8_t)u)) e[m++] = (uint8_t)u;
  qsort(e, (size_t)m, 1, cmp_e4m3);
  for (uint32_t u = 0; u < 256; ++u) g_rank_e4m3[u] = -1;
  for (int r = 0; r < m; ++r) {
    g_bits_e4m3[r] = e[r];
    g_rank_e4m3[e[r]] = r;
  }
  g_lo_e4m3[0] = -INFINITY;
  for (int r = 1; r < m; ++r)
    g_lo_e4m3[r] = bin_lo(or_e4m3_value(e[r - 1]), or_e4m3_value(e[r]));
  g_lo_e4m3[m] = INFINITY;

  or_phi_table(g_phi);
  g_ready = 1;
}

int32_t or_nsym(int dtype) { return dtype == OR_BF16 ? NSYM_BF16 : NSYM_E4M3; }

int32_t or_rank(int dtype, uint32_t u) {
  init_tables();
  return dtype == OR_BF16 ? g_rank_bf16[u & 0xFFFF] : g_rank_e4m3[u & 0xFF];
}

uint32_t or_bits(int dtype, int32_t r) {
  init_tables();
  return dtype == OR_BF16 ? g_bits_bf16[r] : g_bits_e4m3[r];
}

float or_lo(int dtype, int32_t r) {
  init_tables();
  return dtype == OR_BF16 ? g_lo_bf16[r] : g_lo_e4m3[r];
}

/* ------------------------------------------------------------------ */
/* Deterministic Phi (R4) and the per-rank cumulative frequency (R5-R7) */
/* ------------------------------------------------------------------ */

uint32_t or_phi_q(float z) {
  init_tables();
  float t = z * 512.0f; /* a power-of-two scaling: exact */
  if (!(t > -4096.0f)) return 0;
  if (t >= 4096.0f) return PHI_ONE;
  float f = floorf(t);
  int i = (int)f + 4096;
  /* fr = floor(65536 (t - f)) exactly: 65536 f is an integer, so this is
   * floor(65536 t) - 65536 f, and 65536 t is an exact binary32 scaling.
   * (t - f evaluated in floating point rounds to 1 for tiny negative t.) */
  int64_t fr64 = (int64_t)floorf(t * 65536.0f) - 65536 * (int64_t)f;
  uint32_t fr = (uint32_t)fr64;
  uint32_t a = g_phi[i], b = g_phi[i + 1];
  return a + (uint32_t)(((uint64_t)(b - a) * fr) >> 16);
}

int or_sigma_valid(float s) {
  return isfinite(s) && s >= FLT_MIN && isfinite(3.0f * s);
}

static float mu_value(uint16_t mu_bits) { return (float)or_bf16_value(mu_bits); }

static int order0(const or_model *m);

uint32_t or_cum(const or_model *m, int32_t r, float mu, float sigma) {
  init_tables();
  float inv_s = 1.0f / sigma;
  if (m->dtype == OR_BF16) {
    float inv_3s = 1.0f / (3.0f * sigma);
    float d = g_lo_bf16[r] - mu;
    float z1 = d * inv_s;
    float z3 = d * inv_3s;
    uint64_t F = (uint64_t)m->we * m->E[r];
    if (!order0(m)) F += (uint64_t)m->w1 * or_phi_q(z1) + (uint64_t)m->w3 * or_phi_q(z3);
    unsigned __int128 num = (unsigned __int128)((1ull << 28) - NSYM_BF16) * F;
    unsigned __int128 one = (unsigned __int128)100 << 26;
    return (uint32_t)(num / one) + (uint32_t)r;
  } else {
    float d = g_lo_e4m3[r] - mu;
    float z1 = d * inv_s;
    uint64_t num = (uint64_t)((1u << 16) - NSYM_E4M3) * or_phi_q(z1);
    return (uint32_t)(num >> 26) + (uint32_t)r;
  }
}

int or_cum_all(const or_model *m, float mu, float sigma, uint32_t *cum) {
  int32_t n = or_nsym(m->dtype);
  for (int32_t r = 0; r <= n; ++r) cum[r] = or_cum(m, r, mu, sigma);
  return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Empirical bf16 distribution (R6)                                    */
/* ------------------------------------------------------------------ */

int or_build_ecdf(const uint64_t *counts, uint32_t *E) {
  init_tables();
  unsigned __int128 S = 0, Stot = 0;
  for (int32_t r = 0; r < NSYM_BF16; ++r) Stot += (unsigned __int128)counts[g_bits_bf16[r]] + 1;
  for (int32_t r = 0; r <= NSYM_BF16; ++r) {
    E[r] = (uint32_t)(((unsigned __int128)PHI_ONE * S) / Stot);
    if (r < NSYM_BF16) S += (unsigned __int128)counts[g_bits_bf16[r]] + 1;
  }
  return OR_OK;
}

/* model fingerprint: sum over 32-bit words k of mix(k << 32 | w_k), then mix(h ^ n) */
static uint64_t mix64(uint64_t z) {
  /* SplitMix64 output function (Steele, Lea, Flood, OOPSLA 2014) */
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* R12: the order-0 baseline model (p-hat alone) */
static int order0(const or_model *m) { return m->dtype == OR_BF16 && m->w1 == 0 && m->w3 == 0; }

uint64_t or_model_hash(const or_model *m) {
  uint64_t nsig = order0(m) ? 0 : (uint64_t)m->L * 2 * m->H * m->D;
  uint64_t h = 0, k = 0;
  for (uint64_t i = 0; i < nsig; ++i, ++k) {
    uint32_t w;
    memcpy(&w, &m->sigma[i], 4);
    h += mix64((k << 32) | w);
  }
  if (m->dtype == OR_BF16)
    for (uint64_t i = 0; i <= NSYM_BF16; ++i, ++k) h += mix64((k << 32) | m->E[i]);
  return mix64(h ^ k);
}

/* ------------------------------------------------------------------ */
/* Chunk geometry and lane layout (R8)                                 */
/*                                                                    */
/* KV and mu are [L][2][H][T][D] row-major.  A chunk is one            */
/* (layer, kv, head, token block of Tb tokens): C = Tb*D contiguous    */
/* scalars (the last block of a row may be shorter).  Chunk index =    */
/* ((l*2 + kv)*H + h)*ceil(T/Tb) + tb.  Scalar p of a chunk belongs to */
/* lane (p/8) mod G; a lane's j-th symbol is p = 8(lane + G*(j/8)) +   */
/* j%8.  Round j = every lane's j-th symbol.                           */
/* ------------------------------------------------------------------ */

typedef struct {
  uint64_t base;   /* first scalar of the chunk in the [L][2][H][T][D] tensor */
  uint64_t srow;   /* first sigma of the chunk's (l, kv, h) row */
  uint64_t ngroup; /* groups of 8 scalars in the chunk */
} geom_t;

uint64_t or_num_chunks(const or_model *m) {
  uint64_t ntb = ((uint64_t)m->T + m->Tb - 1) / m->Tb;
  return (uint64_t)m->L * 2 * m->H * ntb;
}

static geom_t chunk_geom(const or_model *m, uint64_t c) {
  uint64_t ntb = ((uint64_t)m->T + m->Tb - 1) / m->Tb;
  uint64_t row = c / ntb, tb = c % ntb;
  uint64_t t0 = tb * m->Tb, tn = (uint64_t)m->T - t0;
  if (tn > (uint64_t)m->Tb) tn = (uint64_t)m->Tb;
  geom_t g;
  g.base = row * (uint64_t)m->T * m->D + t0 * m->D;
  g.srow = row * (uint64_t)m->D;
  g.ngroup = tn * m->D / 8;
  return g;
}

static uint64_t lane_nsym(const geom_t *g, int G, int lane) {
  if ((uint64_t)lane >= g->ngroup) return 0;
  return 8 * ((g->ngroup - lane + G - 1) / G);
}

static uint64_t lane_pos(int G, int lane, uint64_t j) {
  return 8 * ((uint64_t)lane + (uint64_t)G * (j >> 3)) + (j & 7);
}

static uint32_t sym_at(const or_model *m, const void *kv, uint64_t idx) {
  return m->dtype == OR_BF16 ? ((const uint16_t *)kv)[idx] : ((const uint8_t *)kv)[idx];
}

float or_scale_mult(int32_t s) { return (float)exp2((double)(s - 128) / 32.0); }

static double sym_value(const or_model *m, uint32_t sym) {
  return m->dtype == OR_BF16 ? or_bf16_value((uint16_t)sym) : or_e4m3_value((uint8_t)sym);
}

/* R11: one scale byte per 8-channel group of chunk c (the chunk's tokens) */
int or_chunk_scales(const or_model *m, const void *kv, const uint16_t *mu, uint64_t c,
                    uint8_t *scales) {
  init_tables();
  geom_t g = chunk_geom(m, c);
  const uint64_t ntok = 8 * g.ngroup / (uint64_t)m->D;
  for (int32_t grp = 0; grp < m->D / 8; ++grp) {
    uint64_t hist[256];
    memset(hist, 0, sizeof(hist));
    uint64_t n = 0;
    for (uint64_t t = 0; t < ntok; ++t) {
      for (int32_t k = 0; k < 8; ++k) {
        const int32_t d = 8 * grp + k;
        const uint64_t idx = g.base + t * (uint64_t)m->D + (uint64_t)d;
        const float x = (float)sym_value(m, sym_at(m, kv, idx));
        const float muv = mu_value(mu[idx]);
        const float inv = 1.0f / m->sigma[g.srow + (uint64_t)d];
        const float a = fabsf(x - muv) * inv;
        int32_t bin;
        if (!(a > 0.0f)) bin = 0;
        else if (!isfinite(a)) bin = 255;
        else {
          uint32_t b;
          memcpy(&b, &a, 4);
          bin = (int32_t)(b >> 18) - 127 * 32 + 128; /* 32 * log2 with a linear mantissa */
          bin = bin < 0 ? 0 : (bin > 255 ? 255 : bin);
        }
        hist[bin]++;
        n++;
      }
    }
    int32_t med = 0;
    uint64_t acc = 0;
    for (int32_t b = 0; b < 256; ++b) {
      acc += hist[b];
      if (acc >= (n + 1) / 2) {
        med = b;
        break;
      }
    }
    int32_t sc = med + (m->dtype == OR_BF16 ? 18 : 21);
    sc = sc < 0 ? 0 : (sc > 255 ? 255 : sc);
    for (int32_t k = 0; k < 8; ++k)
      if (!or_sigma_valid(m->sigma[g.srow + (uint64_t)(8 * grp + k)] * or_scale_mult(sc))) sc = 128;
    scales[grp] = (uint8_t)sc;
  }
  return OR_OK;
}

static float sigma_eff(const or_model *m, const geom_t *g, const uint8_t *scales, uint64_t p) {
  const uint64_t d = p % (uint64_t)m->D;
  const float s = m->sigma[g->srow + d];
  return m->block_scale ? s * or_scale_mult(scales[d / 8]) : s;
}

static uint64_t scale_words(const or_model *m) {
  return m->block_scale ? (uint64_t)(m->D / 8 + 3) / 4 : 0;
}

int or_model_check(const or_model *m) {
  if (m->dtype != OR_BF16 && m->dtype != OR_E4M3) return OR_ERR_ARG;
  if (m->L <= 0 || m->H <= 0 || m->T <= 0 || m->D <= 0 || m->Tb <= 0) return OR_ERR_ARG;
  if (m->D % 8) return OR_ERR_ARG;
  if (m->G < 1 || m->G > 32 || (m->G & (m->G - 1))) return OR_ERR_ARG;
  if (m->w1 + m->w3 + m->we != 100) return OR_ERR_ARG;
  if (m->block_scale != 0 && m->block_scale != 1) return OR_ERR_ARG;
  if (m->dtype == OR_E4M3 && m->w1 == 0 && m->w3 == 0) return OR_ERR_ARG; /* bf16 only */
  if (order0(m) && m->block_scale) return OR_ERR_ARG;
  if (m->adaptive != 0 && m->adaptive != 1) return OR_ERR_ARG;
  if (m->adaptive && !order0(m)) return OR_ERR_ARG;
  return OR_OK;
}

/* R13: the coding table of chunk c from the row's earlier blocks of kv (for a
   decoder: the cache decoded so far).  P, if given, receives P_b (NSYM_BF16). */
int or_adaptive_table(const or_model *m, const void *kv, uint64_t c, uint32_t *E, uint64_t *P) {
  init_tables();
  const uint64_t ntb = ((uint64_t)m->T + m->Tb - 1) / m->Tb;
  const uint64_t row = c / ntb, b = c % ntb;
  const uint64_t A = 63570, B = 58982;
  uint64_t *Pb = (uint64_t *)malloc(sizeof(uint64_t) * NSYM_BF16);
  uint64_t *C = (uint64_t *)calloc(NSYM_BF16, sizeof(uint64_t));
  uint64_t *W = (uint64_t *)malloc(sizeof(uint64_t) * (uint64_t)m->Tb);
  if (!Pb || !C || !W) { free(Pb); free(C); free(W); return OR_ERR_ARG; }
  for (int32_t r = 0; r < NSYM_BF16; ++r) Pb[r] = (uint64_t)(m->E[r + 1] - m->E[r]) << 6;
  W[m->Tb - 1] = 65536;
  for (int32_t t = m->Tb - 1; t > 0; --t) W[t - 1] = (W[t] * A) >> 16;
  const uint64_t Dk = (W[0] * A) >> 16;
  for (uint64_t blk = 0; blk < b; ++blk) {
    for (int32_t r = 0; r < NSYM_BF16; ++r) C[r] = (C[r] * Dk) >> 16;
    for (uint64_t t = 0; t < (uint64_t)m->Tb; ++t)   /* earlier blocks are whole */
      for (uint64_t d = 0; d < (uint64_t)m->D; ++d) {
        const uint64_t idx = (row * (uint64_t)m->T + blk * m->Tb + t) * m->D + d;
        C[or_rank(OR_BF16, ((const uint16_t *)kv)[idx])] += W[t];
      }
    uint64_t sum = 0;
    for (int32_t r = 0; r < NSYM_BF16; ++r) sum += C[r];
    for (int32_t r = 0; r < NSYM_BF16; ++r) {
      const uint64_t est = (uint64_t)(((unsigned __int128)C[r] << 32) / sum);
      Pb[r] = (B * Pb[r] + (65536 - B) * est) >> 16;
    }
  }
  uint64_t stot = 0;
  for (int32_t r = 0; r < NSYM_BF16; ++r) stot += Pb[r] + 1;
  uint64_t acc = 0;
  for (int32_t r = 0; r <= NSYM_BF16; ++r) {
    E[r] = (uint32_t)(((unsigned __int128)acc << 26) / stot);
    if (r < NSYM_BF16) acc += Pb[r] + 1;
  }
  if (P) memcpy(P, Pb, sizeof(uint64_t) * NSYM_BF16);
  free(Pb); free(C); free(W);
  return OR_OK;
}

/* R13: a copy of m whose E is chunk c's table (E points at the caller's
   NSYM_BF16 + 1 buffer); m itself if the model is not adaptive. */
static const or_model *chunk_model(const or_model *m, const void *hist, uint64_t c,
                                   or_model *copy, uint32_t *E, uint64_t *P, int *rc) {
  *rc = OR_OK;
  if (!m->adaptive) return m;
  *rc = or_adaptive_table(m, hist, c, E, P);
  *copy = *m;
  copy->E = E;
  return copy;
}

/* ------------------------------------------------------------------ */
/* rANS encode of one chunk ([P1] "什么能预测 KV 缓存": (KV, mu, sigma) -> bits) */
/*                                                                    */
/* Symbols are pushed in reverse decode order (rounds descending, lanes */
/* descending); each push may first emit the low 32 bits of the state. */
/* Finally every lane's state is pushed as (hi, lo), lanes descending.  */
/* The chunk's stream is the pushed word list reversed, so it starts    */
/* lo(x_0), hi(x_0), lo(x_1), ... followed by the renormalisation words */
/* in the order the decoder consumes them.                              */
/* ------------------------------------------------------------------ */

int or_encode_chunk(const or_model *m, const void *kv, const uint16_t *mu, uint64_t c,
                    uint32_t *out, uint64_t cap_words, uint64_t *nwords) {
  init_tables();
  int rc = or_model_check(m);
  if (rc) return rc;
  /* R13: the chunk's own table from the row's earlier blocks, then order 0 */
  uint32_t *Ea = m->adaptive ? (uint32_t *)malloc(sizeof(uint32_t) * (NSYM_BF16 + 1)) : NULL;
  or_model ma;
  if (m->adaptive && !Ea) return OR_ERR_ARG;
  m = chunk_model(m, kv, c, &ma, Ea, NULL, &rc);
  if (rc) { free(Ea); return rc; }
  const int M = m->dtype == OR_BF16 ? 28 : 16;
  const int G = m->G;
  geom_t g = chunk_geom(m, c);
  uint64_t n0 = lane_nsym(&g, G, 0);
  uint8_t scales[256];
  if (m->block_scale) or_chunk_scales(m, kv, mu, c, scales);
  const uint64_t nsw = scale_words(m);
  uint64_t cap = 8 * g.ngroup + 2 * (uint64_t)G + nsw;
  uint32_t *stack = (uint32_t *)malloc(sizeof(uint32_t) * cap);
  if (!stack) { free(Ea); return OR_ERR_ARG; }
  uint64_t sp = 0;
  uint64_t x[32];
  for (int l = 0; l < G; ++l) x[l] = STATE_L;

  for (uint64_t jj = n0; jj-- > 0;) {
    for (int l = G - 1; l >= 0; --l) {
      if (jj >= lane_nsym(&g, G, l)) continue;
      uint64_t p = lane_pos(G, l, jj);
      uint64_t idx = g.base + p;
      float sigma = 1.0f, muv = 0.0f;
      if (!order0(m)) {
        sigma = m->sigma[g.srow + p % (uint64_t)m->D];
        muv = mu_value(mu[idx]);
        if (!or_sigma_valid(sigma) || !isfinite(muv)) { free(stack); free(Ea); return OR_ERR_PARAM; }
        sigma = sigma_eff(m, &g, scales, p);
      }
      int32_t r = or_rank(m->dtype, sym_at(m, kv, idx));
      if (r < 0) { free(stack); free(Ea); return OR_ERR_SYMBOL; }
      uint32_t cr = or_cum(m, r, muv, sigma);
      uint32_t freq = or_cum(m, r + 1, muv, sigma) - cr;
      uint64_t xmax = ((STATE_L >> M) << 32) * freq;
      if (x[l] >= xmax) {
        stack[sp++] = (uint32_t)x[l];
        x[l] >>= 32;
      }
      x[l] = ((x[l] / freq) << M) + (x[l] % freq) + cr;
    }
  }
  for (int l = G - 1; l >= 0; --l) {
    stack[sp++] = (uint32_t)(x[l] >> 32);
    stack[sp++] = (uint32_t)x[l];
  }
  /* the scale bytes open the chunk: word w holds groups 4w..4w+3, low byte first */
  for (uint64_t wi = nsw; wi-- > 0;) {
    uint32_t word = 0;
    for (int b = 3; b >= 0; --b) {
      const uint64_t grp = 4 * wi + (uint64_t)b;
      word = (word << 8) | (grp < (uint64_t)(m->D / 8) ? scales[grp] : 0u);
    }
    stack[sp++] = word;
  }
  *nwords = sp;
  if (sp > cap_words) { free(stack); free(Ea); return OR_ERR_CAPACITY; }
  for (uint64_t i = 0; i < sp; ++i) out[i] = stack[sp - 1 - i];
  free(stack);
  free(Ea);
  return OR_OK;
}

/* Largest rank r with cum(r) <= slot, by plain bisection over [0, |alphabet|). */
static int32_t find_rank(const or_model *m, uint32_t slot, float muv, float sigma) {
  int32_t lo = 0, hi = or_nsym(m->dtype); /* cum(lo) <= slot < cum(hi) */
  while (hi - lo > 1) {
    int32_t mid = lo + (hi - lo) / 2;
    if (or_cum(m, mid, muv, sigma) <= slot) lo = mid;
    else hi = mid;
  }
  return lo;
}

static int decode_chunk_with(const or_model *m, const uint32_t *w, uint64_t nwords,
                             const uint16_t *mu, uint64_t c, void *kv_out);

int or_decode_chunk(const or_model *m, const uint32_t *w, uint64_t nwords, const uint16_t *mu,
                    uint64_t c, void *kv_out) {
  init_tables();
  int rc = or_model_check(m);
  if (rc) return rc;
  /* R13: the table is built from the blocks already decoded into kv_out */
  uint32_t *Ea = m->adaptive ? (uint32_t *)malloc(sizeof(uint32_t) * (NSYM_BF16 + 1)) : NULL;
  or_model ma;
  if (m->adaptive && !Ea) return OR_ERR_ARG;
  m = chunk_model(m, kv_out, c, &ma, Ea, NULL, &rc);
  if (!rc) rc = decode_chunk_with(m, w, nwords, mu, c, kv_out);
  free(Ea);
  return rc;
}

static int decode_chunk_with(const or_model *m, const uint32_t *w, uint64_t nwords,
                             const uint16_t *mu, uint64_t c, void *kv_out) {
  const int M = m->dtype == OR_BF16 ? 28 : 16;
  const uint64_t mask = (1ull << M) - 1;
  const int G = m->G;
  geom_t g = chunk_geom(m, c);
  uint64_t n0 = lane_nsym(&g, G, 0);
  const uint64_t nsw = scale_words(m);
  if (nwords < 2 * (uint64_t)G + nsw) return OR_ERR_CORRUPT;
  uint8_t scales[256];
  for (int32_t grp = 0; grp < m->D / 8; ++grp) {
    scales[grp] = (uint8_t)(w[grp / 4] >> (8 * (grp % 4)));
    /* a scale the encoder cannot have chosen (an invalid static sigma is the
       caller's error, reported per symbol below) */
    for (int32_t k = 0; m->block_scale && k < 8; ++k) {
      const float sg = m->sigma[g.srow + (uint64_t)(8 * grp + k)];
      if (or_sigma_valid(sg) && !or_sigma_valid(sg * or_scale_mult(scales[grp])))
        return OR_ERR_CORRUPT;
    }
  }
  const uint32_t *ws = w + nsw;
  uint64_t x[32];
  for (int l = 0; l < G; ++l) x[l] = (uint64_t)ws[2 * l] | ((uint64_t)ws[2 * l + 1] << 32);
  uint64_t cur = 2 * (uint64_t)G + nsw;

  for (uint64_t j = 0; j < n0; ++j) {
    for (int l = 0; l < G; ++l) {
      if (j >= lane_nsym(&g, G, l)) continue;
      uint64_t p = lane_pos(G, l, j);
      uint64_t idx = g.base + p;
      float sigma = 1.0f, muv = 0.0f;
      if (!order0(m)) {
        sigma = m->sigma[g.srow + p % (uint64_t)m->D];
        muv = mu_value(mu[idx]);
        if (!or_sigma_valid(sigma) || !isfinite(muv)) return OR_ERR_PARAM;
        sigma = sigma_eff(m, &g, scales, p);
      }
      uint32_t slot = (uint32_t)(x[l] & mask);
      int32_t r = find_rank(m, slot, muv, sigma);
      uint32_t cr = or_cum(m, r, muv, sigma);
      uint32_t freq = or_cum(m, r + 1, muv, sigma) - cr;
      x[l] = (uint64_t)freq * (x[l] >> M) + slot - cr;
      if (x[l] < STATE_L) {
        if (cur >= nwords) return OR_ERR_CORRUPT;
        x[l] = (x[l] << 32) | w[cur++];
      }
      uint32_t s = or_bits(m->dtype, r);
      if (m->dtype == OR_BF16) ((uint16_t *)kv_out)[idx] = (uint16_t)s;
      else ((uint8_t *)kv_out)[idx] = (uint8_t)s;
    }
  }
  for (int l = 0; l < G; ++l)
    if (x[l] != STATE_L) return OR_ERR_CORRUPT;
  if (cur != nwords) return OR_ERR_CORRUPT;
  return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Container v1 (little-endian):                                       */
/*   64-byte header | u64 offsets[num_chunks + 1] | payload             */
/* header: u32 magic "SKV1", u16 version 1, u8 dtype, u8 M,             */
/*   u32 L, u32 2, u32 H, u32 T, u32 D, u32 Tb, u16 G, u8 vec (8),      */
/*   u8 log2 of the Phi table's steps per unit z (9), u16 Phi range     */
/*   (8), u16 0, u64 num_chunks, u64 payload_bytes, u64 model hash.     */
/* offsets are byte offsets from the payload start; chunk c occupies    */
/* [offsets[c], offsets[c+1]) and is a whole number of 32-bit words.    */
/* ------------------------------------------------------------------ */

static void put16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void put32(uint8_t *p, uint32_t v) { for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i)); }
static void put64(uint8_t *p, uint64_t v) { for (int i = 0; i < 8; ++i) p[i] = (uint8_t)(v >> (8 * i)); }
static uint16_t get16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t get32(const uint8_t *p) {
  uint32_t v = 0;
  for (int i = 3; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}
static uint64_t get64(const uint8_t *p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}

static void write_header(const or_model *m, uint8_t *h, uint64_t nchunks, uint64_t payload) {
  memset(h, 0, 64);
  put32(h + 0, 0x31564B53u); /* "SKV1" */
  put16(h + 4, 1);
  h[6] = (uint8_t)m->dtype;
  h[7] = (uint8_t)(m->dtype == OR_BF16 ? 28 : 16);
  put32(h + 8, (uint32_t)m->L);
  put32(h + 12, 2);
  put32(h + 16, (uint32_t)m->H);
  put32(h + 20, (uint32_t)m->T);
  put32(h + 24, (uint32_t)m->D);
  put32(h + 28, (uint32_t)m->Tb);
  put16(h + 32, (uint16_t)m->G);
  h[34] = 8;
  h[35] = 9;
  put16(h + 36, 8);
  put16(h + 38, (uint16_t)((m->block_scale ? 1 : 0) | (order0(m) ? 2 : 0) |
                           (m->adaptive ? 4 : 0))); /* feature bits */
  put64(h + 40, nchunks);
  put64(h + 48, payload);
  put64(h + 56, or_model_hash(m));
}

uint64_t or_max_encoded_bytes(const or_model *m) {
  uint64_t n = (uint64_t)m->L * 2 * m->H * m->T * m->D;
  uint64_t nc = or_num_chunks(m);
  return 64 + 8 * (nc + 1) + 4 * (n + (2 * (uint64_t)m->G + scale_words(m)) * nc);
}

int or_encode(const or_model *m, const void *kv, const uint16_t *mu, uint8_t *out, uint64_t cap,
              uint64_t *out_bytes) {
  int rc = or_model_check(m);
  if (rc) return rc;
  uint64_t nc = or_num_chunks(m);
  uint64_t head = 64 + 8 * (nc + 1);
  if (cap < head) return OR_ERR_CAPACITY;
  uint64_t pos = 0;
  put64(out + 64, 0);
  for (uint64_t c = 0; c < nc; ++c) {
    uint64_t room = (cap - head - pos) / 4, nw = 0;
    /* words are assembled in a scratch buffer to keep the output byte order explicit */
    geom_t g = chunk_geom(m, c);
    uint64_t need = 8 * g.ngroup + 2 * (uint64_t)m->G + scale_words(m);
    uint32_t *tmp = (uint32_t *)malloc(sizeof(uint32_t) * need);
    if (!tmp) return OR_ERR_ARG;
    rc = or_encode_chunk(m, kv, mu, c, tmp, need, &nw);
    if (rc) { free(tmp); return rc; }
    if (nw > room) { free(tmp); return OR_ERR_CAPACITY; }
    for (uint64_t i = 0; i < nw; ++i) put32(out + head + pos + 4 * i, tmp[i]);
    free(tmp);
    pos += 4 * nw;
    put64(out + 64 + 8 * (c + 1), pos);
  }
  write_header(m, out, nc, pos);
  *out_bytes = head + pos;
  return OR_OK;
}

/* Chunks [c0, c1) of a container (in, in_bytes), each against this oracle's
 * own encoding of that chunk: OR_OK if every chunk's offsets and payload bytes
 * are identical, else OR_ERR_CORRUPT with *bad the first chunk that differs.
 * With c0 = 0 the offset table must start at 0, with c1 = the chunk count it
 * must end at the payload size.  A loop over or_encode_chunk and a byte
 * comparison: no arithmetic of its own (the header is or_check_header's). */
int or_compare_chunks(const or_model *m, const void *kv, const uint16_t *mu, const uint8_t *in,
                      uint64_t in_bytes, uint64_t c0, uint64_t c1, uint64_t *bad) {
  int rc = or_model_check(m);
  if (rc) return rc;
  uint64_t nc = or_num_chunks(m);
  uint64_t head = 64 + 8 * (nc + 1);
  if (in_bytes < head || c1 > nc || c0 > c1) return OR_ERR_ARG;
  uint64_t payload = in_bytes - head;
  *bad = c0;
  if (c0 == 0 && get64(in + 64) != 0) return OR_ERR_CORRUPT;
  *bad = c1 ? c1 - 1 : 0;
  if (c1 == nc && get64(in + 64 + 8 * nc) != payload) return OR_ERR_CORRUPT;
  uint64_t cap = (uint64_t)m->Tb * (uint64_t)m->D + 2 * (uint64_t)m->G + scale_words(m);
  uint32_t *tmp = (uint32_t *)malloc(sizeof(uint32_t) * cap);
  if (!tmp) return OR_ERR_ARG;
  for (uint64_t c = c0; c < c1; ++c) {
    *bad = c;
    uint64_t a = get64(in + 64 + 8 * c), b = get64(in + 64 + 8 * (c + 1)), nw = 0;
    if (b < a || b > payload || (b - a) % 4) { free(tmp); return OR_ERR_CORRUPT; }
    rc = or_encode_chunk(m, kv, mu, c, tmp, cap, &nw);
    if (rc) { free(tmp); return rc; }
    if (nw != (b - a) / 4) { free(tmp); return OR_ERR_CORRUPT; }
    for (uint64_t i = 0; i < nw; ++i)
      if (get32(in + head + a + 4 * i) != tmp[i]) { free(tmp); return OR_ERR_CORRUPT; }
  }
  free(tmp);
  return OR_OK;
}

int or_check_header(const or_model *m, const uint8_t *in, uint64_t in_bytes) {
  if (in_bytes < 64) return OR_ERR_CORRUPT;
  uint8_t want[64];
  uint64_t nc = or_num_chunks(m);
  write_header(m, want, nc, get64(in + 48));
  if (memcmp(want, in, 64) != 0) return OR_ERR_CORRUPT;
  uint64_t head = 64 + 8 * (nc + 1);
  if (in_bytes < head || get64(in + 48) != in_bytes - head) return OR_ERR_CORRUPT;
  return OR_OK;
}

int or_decode(const or_model *m, const uint8_t *in, uint64_t in_bytes, const uint16_t *mu,
              void *kv_out) {
  init_tables();
  int rc = or_model_check(m);
  if (rc) return rc;
  rc = or_check_header(m, in, in_bytes);
  if (rc) return rc;
  uint64_t nc = or_num_chunks(m);
  uint64_t head = 64 + 8 * (nc + 1), payload = in_bytes - head;
  if (get64(in + 64) != 0) return OR_ERR_CORRUPT;
  for (uint64_t c = 0; c < nc; ++c) {
    uint64_t a = get64(in + 64 + 8 * c), b = get64(in + 64 + 8 * (c + 1));
    if (b < a || b > payload || (b - a) % 4) return OR_ERR_CORRUPT;
    uint64_t nw = (b - a) / 4;
    uint32_t *w = (uint32_t *)malloc(sizeof(uint32_t) * (nw ? nw : 1));
    if (!w) return OR_ERR_ARG;
    for (uint64_t i = 0; i < nw; ++i) w[i] = get32(in + head + a + 4 * i);
    rc = or_decode_chunk(m, w, nw, mu, c, kv_out);
    free(w);
    if (rc) return rc;
  }
  if (get64(in + 64 + 8 * nc) != payload) return OR_ERR_CORRUPT;
  return OR_OK;
}

uint64_t or_header_u64(const uint8_t *in, int off) { return get64(in + off); }
uint32_t or_header_u32(const uint8_t *in, int off) { return get32(in + off); }
uint32_t or_header_u16(const uint8_t *in, int off) { return get16(in + off); }

/* ------------------------------------------------------------------ */
/* Ideal bits (R10): -log2 q(x) with q the exact bin mass, binary64.   */
/* [P1] "KV 缓存并非真正随机": with a Dirac-delta source every coded bit */
/* is cross-entropy, so the ideal cost of a scalar is -log2 q(x).      */
/* ------------------------------------------------------------------ */

/* log of the upper tail Q(z) = P(N(0,1) > z) */
double or_log_q(double z) {
  if (z == INFINITY) return -INFINITY;
  if (z == -INFINITY) return 0.0;
  if (z < 37.0) {
    if (z < 0) return log1p(-0.5 * erfc(-z * M_SQRT1_2));
    return log(0.5 * erfc(z * M_SQRT1_2));
  }
  /* Laplace's asymptotic series for the Mills ratio (erfc underflows here) */
  double u = 1.0 / (z * z);
  double series = 1.0 - u + 3 * u * u - 15 * u * u * u + 105 * u * u * u * u;
  return -0.5 * z * z - log(z) - 0.5 * log(2 * M_PI) + log(series);
}

/* log of the mass of N(0,1) on [za, zb] */
double or_log_mass(double za, double zb) {
  if (!(zb > za)) return -INFINITY;
  if (isfinite(za) && isfinite(zb)) {
    double w = zb - za, zm = 0.5 * (za + zb);
    double scale = fabs(zm) > 1.0 ? fabs(zm) : 1.0;
    if (w * scale < 1e-3) {
      /* midpoint rule with its second-order term: error O((w*scale)^4) */
      return -0.5 * zm * zm - 0.5 * log(2 * M_PI) + log(w) +
             log1p((zm * zm - 1.0) * w * w / 24.0);
    }
  }
  if (za >= 0) {
    double a = or_log_q(za), b = or_log_q(zb);
    return a + log(-expm1(b - a));
  }
  if (zb <= 0) {
    double a = or_log_q(-zb), b = or_log_q(-za);
    return a + log(-expm1(b - a));
  }
  /* the bin straddles the mean */
  double qa = isfinite(za) ? 0.5 * erfc(-za * M_SQRT1_2) : 0.0; /* P(Z < za) */
  double qb = isfinite(zb) ? 0.5 * erfc(zb * M_SQRT1_2) : 0.0;  /* P(Z > zb) */
  return log1p(-(qa + qb));
}

static double log_gauss_bin(double lo, double hi, double mu, double s) {
  return or_log_mass((lo - mu) / s, (hi - mu) / s);
}

static double lse3(double a, double b, double c) {
  double m = a > b ? a : b;
  m = m > c ? m : c;
  if (m == -INFINITY) return -INFINITY;
  return m + log(exp(a - m) + exp(b - m) + exp(c - m));
}

double or_ideal_bits_one(const or_model *m, uint32_t sym, uint16_t mu_bits, float sigma) {
  init_tables();
  int32_t r = or_rank(m->dtype, sym);
  if (r < 0) return NAN;
  double muv = or_bf16_value(mu_bits);
  double s = (double)sigma;
  double lo = (double)or_lo(m->dtype, r), hi = (double)or_lo(m->dtype, r + 1);
  if (m->dtype == OR_E4M3) return -log_gauss_bin(lo, hi, muv, s) / M_LN2;
  double lp1 = log(m->w1 / 100.0) + log_gauss_bin(lo, hi, muv, s);
  double lp3 = log(m->w3 / 100.0) + log_gauss_bin(lo, hi, muv, 3.0 * s);
  double stot = 0;
  for (int32_t k = 0; k < NSYM_BF16; ++k) stot += (double)m->counts[g_bits_bf16[k]] + 1.0;
  double lpe = log(m->we / 100.0) + log(((double)m->counts[sym & 0xFFFF] + 1.0) / stot);
  return -lse3(lp1, lp3, lpe) / M_LN2;
}

int or_ideal_bits(const or_model *m, const void *kv, const uint16_t *mu, uint64_t begin,
                  uint64_t end, double *per_scalar, double *total) {
  init_tables();
  int rc = or_model_check(m);
  if (rc) return rc;
  double stot = 0;
  if (m->dtype == OR_BF16 && m->counts)
    for (int32_t k = 0; k < NSYM_BF16; ++k) stot += (double)m->counts[g_bits_bf16[k]] + 1.0;
  uint64_t *Pa = NULL;
  uint32_t *Ea2 = NULL;
  double pa_stot = 0;
  if (m->adaptive) {
    Pa = (uint64_t *)malloc(sizeof(uint64_t) * NSYM_BF16);
    Ea2 = (uint32_t *)malloc(sizeof(uint32_t) * (NSYM_BF16 + 1));
    if (!Pa || !Ea2) { free(Pa); free(Ea2); return OR_ERR_ARG; }
  }
  double acc = 0;
  const uint64_t nc = or_num_chunks(m);
  for (uint64_t c = 0; c < nc; ++c) {
    geom_t g = chunk_geom(m, c);
    const uint64_t c0 = g.base, c1 = g.base + 8 * g.ngroup;
    if (c1 <= begin || c0 >= end) continue;
    uint8_t scales[256];
    if (m->block_scale) or_chunk_scales(m, kv, mu, c, scales);
    if (m->adaptive) {
      if ((rc = or_adaptive_table(m, kv, c, Ea2, Pa))) { free(Pa); free(Ea2); return rc; }
      pa_stot = 0;
      for (int32_t k = 0; k < NSYM_BF16; ++k) pa_stot += (double)Pa[k] + 1.0;
    }
    for (uint64_t i = c0 > begin ? c0 : begin; i < (c1 < end ? c1 : end); ++i) {
      uint32_t sym = sym_at(m, kv, i);
      int32_t r = or_rank(m->dtype, sym);
      if (r < 0) { free(Pa); free(Ea2); return OR_ERR_SYMBOL; }
      if (m->adaptive) { /* R13: q = (P_b + 1) / S_tot of the chunk's model */
        const double bits = -log(((double)Pa[r] + 1.0) / pa_stot) / M_LN2;
        if (per_scalar) per_scalar[i - begin] = bits;
        acc += bits;
        continue;
      }
      if (order0(m)) { /* R12: q = p-hat */
        const double bits = -log(((double)m->counts[sym] + 1.0) / stot) / M_LN2;
        if (per_scalar) per_scalar[i - begin] = bits;
        acc += bits;
        continue;
      }
      float sigma = m->sigma[g.srow + (i - g.base) % (uint64_t)m->D];
      double muv = or_bf16_value(mu[i]);
      if (!or_sigma_valid(sigma) || !isfinite(muv)) { free(Pa); free(Ea2); return OR_ERR_PARAM; }
      sigma = sigma_eff(m, &g, scales, i - g.base);
      double s = (double)sigma;
      double lo = (double)or_lo(m->dtype, r), hi = (double)or_lo(m->dtype, r + 1);
      double bits;
      if (m->dtype == OR_E4M3) {
        bits = -log_gauss_bin(lo, hi, muv, s) / M_LN2;
      } else {
        double lp1 = log(m->w1 / 100.0) + log_gauss_bin(lo, hi, muv, s);
        double lp3 = log(m->w3 / 100.0) + log_gauss_bin(lo, hi, muv, 3.0 * s);
        double lpe = log(m->we / 100.0) + log(((double)m->counts[sym] + 1.0) / stot);
        bits = -lse3(lp1, lp3, lpe) / M_LN2;
      }
      if (per_scalar) per_scalar[i - begin] = bits;
      acc += bits;
    }
  }
  free(Pa);
  free(Ea2);
  *total = acc;
  return OR_OK;
}

/* the rANS code length of a chunk under the coder's own integer model */
int or_model_bits_chunk(const or_model *m, const void *kv, const uint16_t *mu, uint64_t c,
                        double *bits) {
  init_tables();
  int rc;
  uint32_t *Ea = m->adaptive ? (uint32_t *)malloc(sizeof(uint32_t) * (NSYM_BF16 + 1)) : NULL;
  or_model ma;
  if (m->adaptive && !Ea) return OR_ERR_ARG;
  m = chunk_model(m, kv, c, &ma, Ea, NULL, &rc);
  if (rc) { free(Ea); return rc; }
  const int M = m->dtype == OR_BF16 ? 28 : 16;
  geom_t g = chunk_geom(m, c);
  uint8_t scales[256];
  if (m->block_scale) or_chunk_scales(m, kv, mu, c, scales);
  double acc = 0;
  for (uint64_t p = 0; p < 8 * g.ngroup; ++p) {
    uint64_t idx = g.base + p;
    float sigma = order0(m) ? 1.0f : sigma_eff(m, &g, scales, p);
    float muv = order0(m) ? 0.0f : mu_value(mu[idx]);
    int32_t r = or_rank(m->dtype, sym_at(m, kv, idx));
    if (r < 0) { free(Ea); return OR_ERR_SYMBOL; }
    uint32_t freq = or_cum(m, r + 1, muv, sigma) - or_cum(m, r, muv, sigma);
    acc += (double)M - log2((double)freq);
  }
  free(Ea);
  *bits = acc;
  return OR_OK;
}
