/*
 * skv_oracle.h -- interface of the oracle (test infrastructure only; see
 * skv_oracle.c).  Nothing in the CUDA library includes this file.
 */
#ifndef SKV_ORACLE_H
#define SKV_ORACLE_H
#include <stdint.h>

enum { OR_BF16 = 0, OR_E4M3 = 1 };
enum { OR_OK = 0, OR_ERR_ARG = -1, OR_ERR_CAPACITY = -2, OR_ERR_SYMBOL = -3,
       OR_ERR_PARAM = -4, OR_ERR_CORRUPT = -5 };

typedef struct {
  int32_t dtype;                /* OR_BF16 or OR_E4M3 */
  int32_t L, H, T, D;           /* tensor [L][2][H][T][D] */
  int32_t Tb, G;                /* token block, lanes per chunk */
  int32_t w1, w3, we;           /* mixture weights in percent (95, 3, 2) */
  int32_t block_scale;          /* 1: per-(chunk, 8-channel group) sigma scales */
  int32_t adaptive;             /* 1: adaptive order-0 counts per (layer, kv, head) row */
  const float *sigma;           /* [L][2][H][D] */
  const uint32_t *E;            /* bf16: empirical prefix table, 65283 entries */
  const uint64_t *counts;       /* bf16: calibration counts by bit pattern, 65536 */
} or_model;

double or_bf16_value(uint16_t u);
double or_e4m3_value(uint8_t u);
void or_phi_table(uint32_t *T);
int32_t or_nsym(int dtype);
int32_t or_rank(int dtype, uint32_t u);
uint32_t or_bits(int dtype, int32_t r);
float or_lo(int dtype, int32_t r);
uint32_t or_phi_q(float z);
int or_sigma_valid(float s);
uint32_t or_cum(const or_model *m, int32_t r, float mu, float sigma);
int or_cum_all(const or_model *m, float mu, float sigma, uint32_t *cum);
int or_build_ecdf(const uint64_t *counts, uint32_t *E);
uint64_t or_model_hash(const or_model *m);
uint64_t or_num_chunks(const or_model *m);
int or_model_check(const or_model *m);
int or_encode_chunk(const or_model *m, const void *kv, const uint16_t *mu, uint64_t c,
                    uint32_t *out, uint64_t cap_words, uint64_t *nwords);
int or_decode_chunk(const or_model *m, const uint32_t *w, uint64_t nwords, const uint16_t *mu,
                    uint64_t c, void *kv_out);
uint64_t or_max_encoded_bytes(const or_model *m);
int or_encode(const or_model *m, const void *kv, const uint16_t *mu, uint8_t *out, uint64_t cap,
              uint64_t *out_bytes);
int or_check_header(const or_model *m, const uint8_t *in, uint64_t in_bytes);
int or_compare_chunks(const or_model *m, const void *kv, const uint16_t *mu, const uint8_t *in,
                      uint64_t in_bytes, uint64_t c0, uint64_t c1, uint64_t *bad);
int or_decode(const or_model *m, const uint8_t *in, uint64_t in_bytes, const uint16_t *mu,
              void *kv_out);
float or_scale_mult(int32_t s);
int or_chunk_scales(const or_model *m, const void *kv, const uint16_t *mu, uint64_t c,
                    uint8_t *scales);
int or_adaptive_table(const or_model *m, const void *kv, uint64_t c, uint32_t *E, uint64_t *P);
double or_log_q(double z);
double or_log_mass(double za, double zb);
double or_ideal_bits_one(const or_model *m, uint32_t sym, uint16_t mu_bits, float sigma);
int or_ideal_bits(const or_model *m, const void *kv, const uint16_t *mu, uint64_t begin,
                  uint64_t end, double *per_scalar, double *total);
int or_model_bits_chunk(const or_model *m, const void *kv, const uint16_t *mu, uint64_t c,
                        double *bits);

#endif
