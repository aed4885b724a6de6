/*
 * dsa_oracle.h — CPU oracle of the DSA indexer path (TEST INFRASTRUCTURE ONLY).
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load this library. The CUDA product library never includes, links or calls
 * it, and it shares no code with that library.
 *
 * Everything here is plain, slow and written to be checked by eye against
 * the definitions it follows. Floating point work is fp64 on dequantised
 * values, except where a quantised code is decided: that decision is taken
 * in fp32, the precision the quantiser works in.
 */
#ifndef DSA_ORACLE_H
#define DSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORA_HEADS 64
#define ORA_DIM 128
#define ORA_ROPE 64                               /* rotated leading dims (PE subspace) */
#define ORA_BLOCK 64
#define ORA_SLOT_BYTES 132                       /* 128 B FP8 K + 4 B fp32 scale */
#define ORA_PAGE_BYTES (ORA_BLOCK * ORA_SLOT_BYTES) /* 8448 */
#define ORA_FP4_SLOT_BYTES 68                    /* 64 B E2M1 K (2 per byte) + 4 B fp32 scale */
#define ORA_FP4_PAGE_BYTES (ORA_BLOCK * ORA_FP4_SLOT_BYTES) /* 4352 */
#define ORA_FMT_FP8 0
#define ORA_FMT_FP4 1

/* E4M3 (OCP FP8) */
double ora_e4m3_value(uint8_t code);
uint8_t ora_e4m3_encode(float v);

/* ue8m0 group scale and one group's quantisation */
float ora_ue8m0_scale(float amax);
void ora_quant_group(const float *x, int n, uint8_t *codes, float *scale);

/* E2M1 (OCP MX FP4) and the FP4 cache's quantiser */
double ora_e2m1_value(uint8_t code);
uint8_t ora_e2m1_encode(float v);
float ora_ue8m0_scale_e2m1(float amax);
void ora_quant_group_e2m1(const float *x, int n, uint8_t *packed, float *scale);

/* paged cache */
void ora_slot_offsets(int64_t slot, int64_t *k_byte, int64_t *scale_byte);
void ora_slot_offsets_fmt(int64_t slot, int fmt, int64_t *k_byte, int64_t *scale_byte);
int64_t ora_k_quant_write(const uint16_t *k_bf16, int64_t n, const int64_t *slot_mapping,
                          uint8_t *cache, int64_t num_blocks);
int64_t ora_k_quant_write_fmt(const uint16_t *k_bf16, int64_t n, const int64_t *slot_mapping,
                              uint8_t *cache, int64_t num_blocks, int fmt);
void ora_q_quant(const uint16_t *q_bf16, int64_t rows, uint8_t *q_codes, float *q_scale);

/* RoPE on the leading 64 dims (half-split pairs, fp32 steps, bf16 result);
 * returns the number of rows left unrotated (position out of range). */
int64_t ora_rope(const uint16_t *x, int64_t rows, int64_t rows_per_token, const int64_t *positions,
                 const float *cos_sin, int64_t max_pos, uint16_t *out);

/* indexer scores and selection */
void ora_logits_row(const uint8_t *q_codes, const float *q_scale, const float *w,
                    const uint8_t *cache, const int32_t *bt_row, int64_t n_keys,
                    double *out);
void ora_logits_row_fmt(const uint8_t *q_codes, const float *q_scale, const float *w,
                        const uint8_t *cache, int fmt, const int32_t *bt_row, int64_t n_keys,
                        double *out);
void ora_topk_row(const double *scores, int64_t n, int k, int32_t *out);
int64_t ora_indexer(const uint16_t *q_bf16, const float *w, const uint8_t *cache,
                    const int32_t *block_table, int64_t bt_stride,
                    const int32_t *req_id_per_token, const int64_t *positions,
                    const int64_t *rows, int64_t n_rows, int topk,
                    int32_t *topk_out, double *scores_out, int64_t scores_ld);
int64_t ora_indexer_fmt(const uint16_t *q_bf16, const float *w, const uint8_t *cache, int fmt,
                        const int32_t *block_table, int64_t bt_stride,
                        const int32_t *req_id_per_token, const int64_t *positions,
                        const int64_t *rows, int64_t n_rows, int topk,
                        int32_t *topk_out, double *scores_out, int64_t scores_ld);

/* logical -> physical ids, IndexCache schedule */
void ora_convert(const int32_t *logical, int64_t n_tokens, int topk,
                 const int32_t *req_id_per_token, const int32_t *block_table,
                 int64_t bt_stride, int block_size, int block_stride_rows,
                 int32_t *physical, int32_t *valid_counts);
int ora_schedule(int n_layers, int use_index_cache, int freq, int offset,
                 const char *pattern, char *fs_out, int32_t *producer_out);

/* The consumer's gather by physical row (bytes); returns out-of-range ids. */
int64_t ora_gather_rows(const uint8_t *rows, int64_t num_rows, int64_t row_bytes, int64_t row_stride,
                        const int32_t *physical, int64_t n_tokens, int topk, uint8_t *out);

#ifdef __cplusplus
}
#endif
#endif
