/*
 * dsa_oracle.c — CPU oracle of the DSA indexer path (TEST INFRASTRUCTURE ONLY).
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * this code; the CUDA library never calls it and shares nothing with it.
 *
 * Sources, cited below by short name:
 *   [IC] "IndexCache：DeepSeek 稀疏注意力中的跨层索引复用" (atomage.cn): code
 *        snippets of vLLM's DeepSeek-V3.2 indexer — the `Indexer` module and
 *        its `forward`, the FP8 indexer K cache, `SparseAttnIndexer`, the
 *        IndexCache layer schedule and the shared top-k buffer.
 *   [PR] "PR #37735 完整报告" on vLLM's "[Feature]: IndexCache support for DSA
 *        models" (prhub.com.cn): sections 实现拆解, 关键源码片段, 风险与影响.
 *   [IG] "vllm.v1.attention.backends.mla.index_group" API page (docs.vllm.ai):
 *        `SparseMLAIndexGroup._convert_once` and the group builder.
 *   [OCP] OCP 8-bit Floating Point Specification (OFP8), E4M3 encoding.
 *   [MX]  OCP Microscaling Formats (MX) Specification v1.0, the FP4 (E2M1)
 *         element type.
 *
 * Where the pages leave a step open, the reading taken is stated at the
 * function. Arithmetic is fp64 on dequantised values; the two places where
 * floating point decides a code (the group scale and the E4M3 rounding) work
 * in fp32, the precision the quantiser of [IC] works in.
 */
#include "dsa_oracle.h"

#include <fenv.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* E4M3 per [OCP]: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
 * Exponent field 0 holds subnormals (m/8 * 2^-6). S.1111.111 is NaN, there
 * is no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448.       */

double ora_e4m3_value(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* Nearest E4M3 value to v, ties to the even code; finite values beyond 448
 * become +-448 (saturating conversion). The sign of zero is kept. */
uint8_t ora_e4m3_encode(float v) {
  uint8_t sign;
  double a, quantum, q;
  int e;
  if (isnan(v)) return 0x7F;
  sign = signbit(v) ? 0x80 : 0x00;
  a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  /* binade of a; subnormals share the spacing of the lowest normal binade */
  e = ilogb(a);
  if (e < -6) e = -6;
  quantum = ldexp(1.0, e - 3); /* 8 steps per binade */
  q = nearbyint(a / quantum);  /* a/quantum is exact; default mode rounds half to even */
  if (q == 0.0) return sign;
  if (q < 8.0) /* only reachable when e == -6: a subnormal code */
    return sign | (uint8_t)q;
  if (q == 16.0) { /* rounded up into the next binade */
    e += 1;
    q = 8.0;
  }
  return sign | (uint8_t)(((e + 7) << 3) | ((int)q - 8));
}

/* ------------------------------------------------------------------------ */
/* Group scale. [IC] `Indexer.forward` quantises q with one scale per group of
 * `quant_block_size` values using ue8m0 scales; the K cache holds "128 bytes
 * K + 4 bytes FP32 scale" per token, so the group is the whole 128-dim row.
 * Reading taken: scale = amax/448 (fp32), with amax floored at 1e-10, rounded
 * UP to a power of two (ue8m0 = exponent only), so |x/scale| <= 448.          */
static float ue8m0_of(float amax, float qmax) {
  float r;
  int e;
  double m;
  if (!(amax >= 1e-10f)) amax = 1e-10f;
  r = amax / qmax;               /* IEEE fp32 division */
  m = frexp((double)r, &e);      /* r = m * 2^e, m in [0.5, 1) */
  if (m == 0.5) return r;        /* already a power of two */
  return (float)ldexp(1.0, e);   /* next power of two above r */
}

float ora_ue8m0_scale(float amax) { return ue8m0_of(amax, 448.0f); }

void ora_quant_group(const float *x, int n, uint8_t *codes, float *scale) {
  float amax = 0.0f, s;
  int i;
  for (i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  s = ora_ue8m0_scale(amax);
  for (i = 0; i < n; ++i) codes[i] = ora_e4m3_encode(x[i] / s); /* fp32 division */
  *scale = s;
}

/* ------------------------------------------------------------------------ */
/* FP4 indexer cache. [IC] hands `sparse_attn_indexer` a `use_fp4_cache` flag
 * beside `quant_block_size` and `scale_fmt`; the pages print nothing more of
 * the format. Reading taken: the element type is [MX]'s E2M1, and the
 * quantiser is the FP8 cache's with E2M1 in place of E4M3 — one ue8m0 scale
 * per token's 128 values, amax/6 (6 = E2M1's largest magnitude) rounded up to
 * a power of two, codes rounded to nearest-even and saturated. q stays FP8.
 *
 * E2M1 per [MX]: 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit.
 * Exponent field 0 holds the subnormal m * 0.5; there is no infinity or NaN,
 * so the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4 and 6. Codes are 0..15.      */

double ora_e2m1_value(uint8_t code) {
  int sign = (code >> 3) & 1;
  int e = (code >> 1) & 3;
  int m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -mag : mag;
}

/* Nearest E2M1 value to v, ties to the even code; magnitudes beyond 6 become
 * 6 (saturating). The sign of zero is kept. NaN never reaches the quantiser
 * (finite bf16 inputs, |x/scale| <= 6); it is mapped to +6. */
uint8_t ora_e2m1_encode(float v) {
  uint8_t sign;
  double a, quantum, steps;
  int e;
  if (isnan(v)) return 0x7;
  sign = signbit(v) ? 0x8 : 0x0;
  a = fabs((double)v);
  if (a >= 6.0) return sign | 0x7;
  if (!(a > 0.0)) return sign;
  e = ilogb(a);
  if (e < 0) e = 0;               /* the subnormal 0.5 shares the spacing of [1, 2) */
  quantum = ldexp(1.0, e - 1);    /* 2 steps per binade */
  steps = nearbyint(a / quantum); /* exact quotient; default mode rounds half to even */
  if (steps == 0.0) return sign;
  if (steps < 2.0) return sign | 0x1; /* only when e == 0: the subnormal 0.5 */
  if (steps == 4.0) {                 /* rounded up into the next binade */
    e += 1;
    steps = 2.0;
  }
  return sign | (uint8_t)(((e + 1) << 1) | ((int)steps - 2));
}

float ora_ue8m0_scale_e2m1(float amax) { return ue8m0_of(amax, 6.0f); }

/* One group to packed E2M1: element 2i in the low nibble of byte i, element
 * 2i+1 in the high nibble (reading taken: the lower index in the lower bits,
 * as in little-endian packing). n is even. */
void ora_quant_group_e2m1(const float *x, int n, uint8_t *packed, float *scale) {
  float amax = 0.0f, s;
  int i;
  for (i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  s = ora_ue8m0_scale_e2m1(amax);
  for (i = 0; i < n; i += 2)
    packed[i / 2] = (uint8_t)(ora_e2m1_encode(x[i] / s) | (ora_e2m1_encode(x[i + 1] / s) << 4));
  *scale = s;
}

static float bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* fp32 -> bf16, round to nearest even (the model's tensors are bf16). */
static uint16_t bf16_round(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return (uint16_t)((u >> 16) | 0x40u); /* NaN */
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Rotary position embedding of the PE subspace, before the quantiser.
 * "IndexCache：DeepSeek 稀疏注意力中的跨层索引复用", `Indexer.forward`: the first
 * rope_dim = 64 dims of every q head and of the shared K row are rotated by
 * `rotary_emb(positions, q_pe, k_pe)`; the other 64 dims pass through.
 * Reading taken (the pairing is not printed): half-split pairs (i, i+32),
 * i < 32, with the angles of position p given as an input table
 * cos_sin[p*64 + i] = cos, cos_sin[p*64 + 32 + i] = sin;
 *   y[i]    = x[i]*cos - x[i+32]*sin,   y[i+32] = x[i+32]*cos + x[i]*sin,
 * each product and each sum rounded in IEEE fp32 (no fused multiply-add), the
 * result rounded to bf16. Row r belongs to token r / rows_per_token. A row
 * whose position is outside [0, max_pos) is copied unrotated and counted. */
int64_t ora_rope(const uint16_t *x, int64_t rows, int64_t rows_per_token, const int64_t *positions,
                 const float *cos_sin, int64_t max_pos, uint16_t *out) {
  int64_t r, bad = 0;
  for (r = 0; r < rows; ++r) {
    const uint16_t *xr = x + r * ORA_DIM;
    uint16_t *yr = out + r * ORA_DIM;
    const int64_t p = positions[r / rows_per_token];
    int i;
    memcpy(yr, xr, ORA_DIM * sizeof(uint16_t));
    if (p < 0 || p >= max_pos) {
      ++bad;
      continue;
    }
    for (i = 0; i < ORA_ROPE / 2; ++i) {
      const float x1 = bf16_value(xr[i]), x2 = bf16_value(xr[i + ORA_ROPE / 2]);
      const float c = cos_sin[p * ORA_ROPE + i], s = cos_sin[p * ORA_ROPE + ORA_ROPE / 2 + i];
      const float a = x1 * c, b = x2 * s, d = x2 * c, e = x1 * s;
      yr[i] = bf16_round(a - b);
      yr[i + ORA_ROPE / 2] = bf16_round(d + e);
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------ */
/* Paged cache. [IC] `DeepseekV32IndexerBackend.get_kv_cache_shape` gives
 * (num_blocks, block_size, head_size) uint8 with one shared K head, and the
 * FP8 cache snippet a head_size of 128 + 128/128*4 = 132 bytes per slot.
 * Reading taken for the order inside a 64-slot page (8448 B): the 64 K rows
 * of 128 B first, then the 64 fp32 scales.                                  */
void ora_slot_offsets(int64_t slot, int64_t *k_byte, int64_t *scale_byte) {
  ora_slot_offsets_fmt(slot, ORA_FMT_FP8, k_byte, scale_byte);
}

/* The FP4 page (reading taken, as for FP8): the 64 rows of 64 code bytes,
 * then the 64 fp32 scales — 4352 B. */
void ora_slot_offsets_fmt(int64_t slot, int fmt, int64_t *k_byte, int64_t *scale_byte) {
  int64_t page = slot / ORA_BLOCK, off = slot % ORA_BLOCK;
  int64_t row = (fmt == ORA_FMT_FP4) ? ORA_DIM / 2 : ORA_DIM;
  int64_t page_bytes = (fmt == ORA_FMT_FP4) ? ORA_FP4_PAGE_BYTES : ORA_PAGE_BYTES;
  *k_byte = page * page_bytes + off * row;
  *scale_byte = page * page_bytes + ORA_BLOCK * row + off * 4;
}

/* [IC] `SparseAttnIndexer` body: `indexer_k_quant_and_cache(k, kv_cache,
 * slot_mapping, ...)` quantises each token's K and stores it at its slot.
 * A negative slot is a padding token and is skipped. Returns the number of
 * tokens whose slot lies outside the cache (also skipped). */
int64_t ora_k_quant_write(const uint16_t *k_bf16, int64_t n, const int64_t *slot_mapping,
                          uint8_t *cache, int64_t num_blocks) {
  return ora_k_quant_write_fmt(k_bf16, n, slot_mapping, cache, num_blocks, ORA_FMT_FP8);
}

/* The same write into an FP8 (fmt 0) or FP4 (fmt 1) cache. */
int64_t ora_k_quant_write_fmt(const uint16_t *k_bf16, int64_t n, const int64_t *slot_mapping,
                              uint8_t *cache, int64_t num_blocks, int fmt) {
  int64_t i, bad = 0;
  for (i = 0; i < n; ++i) {
    float x[ORA_DIM], s;
    uint8_t codes[ORA_DIM];
    int64_t kb, sb;
    int d;
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    if (slot >= num_blocks * ORA_BLOCK) {
      ++bad;
      continue;
    }
    for (d = 0; d < ORA_DIM; ++d) x[d] = bf16_value(k_bf16[i * ORA_DIM + d]);
    if (fmt == ORA_FMT_FP4)
      ora_quant_group_e2m1(x, ORA_DIM, codes, &s);
    else
      ora_quant_group(x, ORA_DIM, codes, &s);
    ora_slot_offsets_fmt(slot, fmt, &kb, &sb);
    memcpy(cache + kb, codes, (fmt == ORA_FMT_FP4) ? ORA_DIM / 2 : ORA_DIM);
    memcpy(cache + sb, &s, 4);
  }
  return bad;
}

/* [IC] `Indexer.forward`: q viewed as (-1, head_dim) and quantised per group
 * of 128 with ue8m0 scales — one scale per (token, head). */
void ora_q_quant(const uint16_t *q_bf16, int64_t rows, uint8_t *q_codes, float *q_scale) {
  int64_t r;
  for (r = 0; r < rows; ++r) {
    float x[ORA_DIM];
    int d;
    for (d = 0; d < ORA_DIM; ++d) x[d] = bf16_value(q_bf16[r * ORA_DIM + d]);
    ora_quant_group(x, ORA_DIM, q_codes + r * ORA_DIM, q_scale + r);
  }
}

/* ------------------------------------------------------------------------ */
/* Indexer score of one query token against keys s = 0 .. n_keys-1 of its
 * request, written out unfolded in fp64:
 *
 *   I[s] = softmax_scale * H^-1/2 * sum_h w[h] * ReLU( q[h] . k[s] )
 *
 * with q[h] = q_codes[h] * q_scale[h] and k[s] = k_codes[s] * k_scale[s]
 * dequantised. [IC] `Indexer.forward` folds q_scale, softmax_scale and
 * n_head^-0.5 into the head weights before the op; since every factor is
 * positive and ReLU is positively homogeneous, the unfolded sum above is the
 * same quantity. The 64 heads share one K row (MQA: `num_kv_heads=1` in
 * `DeepseekV32IndexerCache.get_kv_cache_spec`). Reading taken for
 * softmax_scale (not printed): head_dim^-1/2. n_keys = position + 1: the key
 * at the query's own position is visible, its K having been written first.  */
void ora_logits_row(const uint8_t *q_codes, const float *q_scale, const float *w,
                    const uint8_t *cache, const int32_t *bt_row, int64_t n_keys,
                    double *out) {
  ora_logits_row_fmt(q_codes, q_scale, w, cache, ORA_FMT_FP8, bt_row, n_keys, out);
}

/* The same score over an FP8 (fmt 0) or FP4 (fmt 1) K cache; only the
 * dequantisation of k[s] differs. */
void ora_logits_row_fmt(const uint8_t *q_codes, const float *q_scale, const float *w,
                        const uint8_t *cache, int fmt, const int32_t *bt_row, int64_t n_keys,
                        double *out) {
  static const double softmax_scale = 0.08838834764831845; /* 1/sqrt(128) */
  static const double head_norm = 0.125;                   /* 1/sqrt(64) */
  double qd[ORA_HEADS][ORA_DIM], kd[ORA_DIM];
  int h, d;
  int64_t s;
  for (h = 0; h < ORA_HEADS; ++h)
    for (d = 0; d < ORA_DIM; ++d)
      qd[h][d] = ora_e4m3_value(q_codes[h * ORA_DIM + d]) * (double)q_scale[h];
  for (s = 0; s < n_keys; ++s) {
    int64_t slot = (int64_t)bt_row[s / ORA_BLOCK] * ORA_BLOCK + s % ORA_BLOCK;
    int64_t kb, sb;
    float ks;
    double total = 0.0;
    ora_slot_offsets_fmt(slot, fmt, &kb, &sb);
    memcpy(&ks, cache + sb, 4);
    for (d = 0; d < ORA_DIM; ++d) {
      double v = (fmt == ORA_FMT_FP4) ? ora_e2m1_value((uint8_t)((cache[kb + d / 2] >> (4 * (d & 1))) & 15))
                                      : ora_e4m3_value(cache[kb + d]);
      kd[d] = v * (double)ks;
    }
    for (h = 0; h < ORA_HEADS; ++h) {
      double dot = 0.0;
      for (d = 0; d < ORA_DIM; ++d) dot += qd[h][d] * kd[d];
      total += (double)w[h] * (dot > 0.0 ? dot : 0.0);
    }
    out[s] = softmax_scale * head_norm * total;
  }
}

/* ------------------------------------------------------------------------ */
/* Top-k of one row: every key ordered by (score descending, index
 * ascending) with a full sort; the first min(k, n) indices, then -1 for the
 * rest ([IC] resets the shared buffer rows to -1 before the indexer fills
 * them). Ties are broken towards the lower index. */
static _Thread_local const double *g_sort_scores; /* the row being sorted by this thread */
static int cmp_desc(const void *a, const void *b) {
  int32_t i = *(const int32_t *)a, j = *(const int32_t *)b;
  double si = g_sort_scores[i], sj = g_sort_scores[j];
  if (si > sj) return -1;
  if (si < sj) return 1;
  return (i < j) ? -1 : (i > j);
}

void ora_topk_row(const double *scores, int64_t n, int k, int32_t *out) {
  int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  int64_t i;
  for (i = 0; i < n; ++i) idx[i] = (int32_t)i;
  g_sort_scores = scores; /* qsort takes no context argument */
  qsort(idx, (size_t)n, sizeof(int32_t), cmp_desc);
  for (i = 0; i < k; ++i) out[i] = (i < n) ? idx[i] : -1;
  free(idx);
}

/* One indexer pass over the listed query rows: quantise each row's q (64
 * heads), score it against the keys [0, position] of its request, select the
 * top-k. scores_out (optional) receives the fp64 scores, row-major with
 * leading dimension scores_ld. Returns 0, or -1 if a row needs more keys than
 * scores_ld holds. */
int64_t ora_indexer(const uint16_t *q_bf16, const float *w, const uint8_t *cache,
                    const int32_t *block_table, int64_t bt_stride,
                    const int32_t *req_id_per_token, const int64_t *positions,
                    const int64_t *rows, int64_t n_rows, int topk,
                    int32_t *topk_out, double *scores_out, int64_t scores_ld) {
  return ora_indexer_fmt(q_bf16, w, cache, ORA_FMT_FP8, block_table, bt_stride, req_id_per_token, positions,
                         rows, n_rows, topk, topk_out, scores_out, scores_ld);
}

int64_t ora_indexer_fmt(const uint16_t *q_bf16, const float *w, const uint8_t *cache, int fmt,
                        const int32_t *block_table, int64_t bt_stride,
                        const int32_t *req_id_per_token, const int64_t *positions,
                        const int64_t *rows, int64_t n_rows, int topk,
                        int32_t *topk_out, double *scores_out, int64_t scores_ld) {
  int64_t i, err = 0;
  for (i = 0; i < n_rows; ++i)
    if (scores_out && positions[rows[i]] + 1 > scores_ld) err = -1;
  if (err) return err;
#pragma omp parallel for schedule(dynamic, 1)
  for (i = 0; i < n_rows; ++i) {
    int64_t t = rows[i];
    int64_t n = positions[t] + 1;
    uint8_t qc[ORA_HEADS * ORA_DIM];
    float qs[ORA_HEADS];
    double *sc = scores_out ? scores_out + i * scores_ld
                            : (double *)malloc(sizeof(double) * (size_t)n);
    ora_q_quant(q_bf16 + t * ORA_HEADS * ORA_DIM, ORA_HEADS, qc, qs);
    ora_logits_row_fmt(qc, qs, w + t * ORA_HEADS, cache, fmt,
                       block_table + (int64_t)req_id_per_token[t] * bt_stride, n, sc);
    ora_topk_row(sc, n, topk, topk_out + i * topk);
    if (!scores_out) free(sc);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Logical -> physical ids. [IG] `_convert_once` maps each request-local
 * token id through the request's block table: block = id / block_size,
 * physical = block_table[req][block] * block_stride_rows + id % block_size;
 * -1 stays -1. The valid count of a row is its number of ids >= 0.
 * block_stride_rows <= 0 means block_size. */
void ora_convert(const int32_t *logical, int64_t n_tokens, int topk,
                 const int32_t *req_id_per_token, const int32_t *block_table,
                 int64_t bt_stride, int block_size, int block_stride_rows,
                 int32_t *physical, int32_t *valid_counts) {
  int64_t t;
  int j;
  if (block_stride_rows <= 0) block_stride_rows = block_size;
  for (t = 0; t < n_tokens; ++t) {
    const int32_t *row = block_table + (int64_t)req_id_per_token[t] * bt_stride;
    int32_t valid = 0;
    for (j = 0; j < topk; ++j) {
      int32_t id = logical[t * topk + j];
      if (id < 0) {
        physical[t * topk + j] = -1;
      } else {
        physical[t * topk + j] = row[id / block_size] * block_stride_rows + id % block_size;
        ++valid;
      }
    }
    if (valid_counts) valid_counts[t] = valid;
  }
}

/* IndexCache layer schedule. [IC] (layer construction snippet) and [PR]
 * (关键源码片段, `DeepseekAttention.__init__`): with IndexCache on, layer l
 * skips its top-k ('S') iff max(l - offset + 1, 0) % freq != 0, offset
 * defaulting to 2 (so max(l-1, 0) % freq); an explicit pattern overrides it,
 * 'S' meaning skip. Without IndexCache every layer is 'F'. An 'S' layer
 * reuses the buffer left by the nearest preceding 'F' layer; producer[l] is
 * that layer (itself for 'F').
 * Validation, stricter than the page ([PR] 风险与影响 notes the length is
 * checked but the characters are not): the pattern must have exactly
 * n_layers characters, each 'F' or 'S', and start with 'F'; freq >= 1 and
 * the freq rule must make layer 0 an 'F' layer.
 * Returns 0, or -1 on invalid input (outputs untouched). */
int ora_schedule(int n_layers, int use_index_cache, int freq, int offset,
                 const char *pattern, char *fs_out, int32_t *producer_out) {
  int l;
  if (n_layers < 0) return -1;
  if (use_index_cache) {
    if (pattern) {
      if ((int)strlen(pattern) != n_layers) return -1;
      for (l = 0; l < n_layers; ++l)
        if (pattern[l] != 'F' && pattern[l] != 'S') return -1;
      if (n_layers > 0 && pattern[0] != 'F') return -1;
    } else {
      int v0 = 1 - offset;
      if (freq < 1) return -1;
      if (v0 < 0) v0 = 0;
      if (n_layers > 0 && v0 % freq != 0) return -1; /* layer 0 would have no producer */
    }
  }
  for (l = 0; l < n_layers; ++l) {
    int skip = 0;
    if (use_index_cache) {
      if (pattern) {
        skip = pattern[l] == 'S';
      } else {
        int v = l - offset + 1;
        if (v < 0) v = 0;
        skip = (v % freq) != 0;
      }
    }
    fs_out[l] = skip ? 'S' : 'F';
    producer_out[l] = skip ? producer_out[l - 1] : l;
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* The consumer's gather of the selected rows: "IndexCache：DeepSeek 稀疏注意力中的跨层
 * 索引复用" — the sparse MLA of every layer of a group reads, for each query
 * token, the KV rows of the k selected keys; "vllm.v1.attention.backends.mla.
 * index_group" converts the ids to physical slots for exactly that read. The
 * row format is not on the pages, so the gather is by bytes: out[t][j] = the
 * row_bytes bytes of physical row physical[t][j] (rows row_stride bytes
 * apart), zeros where the id is -1; an id >= num_rows (or < -1) also gives
 * zeros and is counted. Returns that count. */
int64_t ora_gather_rows(const uint8_t *rows, int64_t num_rows, int64_t row_bytes, int64_t row_stride,
                        const int32_t *physical, int64_t n_tokens, int topk, uint8_t *out) {
  int64_t t, bad = 0;
  int j;
  for (t = 0; t < n_tokens; ++t) {
    for (j = 0; j < topk; ++j) {
      const int32_t id = physical[t * topk + j];
      uint8_t *dst = out + (t * topk + j) * row_bytes;
      if (id >= 0 && id < num_rows) {
        memcpy(dst, rows + (int64_t)id * row_stride, (size_t)row_bytes);
      } else {
        memset(dst, 0, (size_t)row_bytes);
        if (id != -1) ++bad;
      }
    }
  }
  return bad;
}
