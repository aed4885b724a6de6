// kernels.h — host-side launchers of the sm_103a kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsaidx.h"

namespace dsa {

constexpr int kHeads = DSA_HEADS;
constexpr int kDim = DSA_HEAD_DIM;
constexpr int kBlock = DSA_BLOCK_SIZE;
constexpr int kPageBytes = DSA_PAGE_BYTES;
constexpr int kScaleOffset = kBlock * kDim;  // 8192: the 64 fp32 scales follow the 64 K rows
constexpr int kFp4PageBytes = DSA_FP4_PAGE_BYTES;      // FP4 cache: 64 rows of 64 E2M1 bytes, then the scales
constexpr int kFp4ScaleOffset = kBlock * kDim / 2;     // 4096
constexpr int kRope = 64;                    // rotated leading dims of q and K rows

// RoPE fused into the quantiser: cos_sin == nullptr means the rows arrive rotated.
struct RopeArgs {
  const int64_t* positions;  // [tokens]
  const float* cos_sin;      // [max_pos, 64]: cos of the 32 pair angles, then sin
  int64_t max_pos;
};

// Query tokens per block of the prefill segment (decode blocks hold one).
constexpr int kPrefillTok = 4;

// One query block: NTOK consecutive query tokens of one request.
struct QBlock {
  int32_t req;  // request
  int32_t t0;   // first token (row of q / logits)
  int32_t ntok; // tokens in the block (1..NTOK)
  int32_t p0;   // position of the first token; token i sees keys [0, p0 + i]
};

// Slice of the flat (query block, tile) list that one persistent CTA runs.
struct CtaWork {
  int32_t it_begin, it_end;  // items [it_begin, it_end)
  int32_t qb0;               // query block holding it_begin
  int32_t kt0;               // tile of it_begin within that block
};

constexpr int kMaxCtas = 1024;

// Work plan of one kernel segment, in device memory.
struct SegmentPlan {
  QBlock* qb;           // [max_qb]
  int32_t* tile_start;  // [max_qb + 1]: exclusive prefix of 128-key tiles; tile_start[nqb] = total
  int32_t* nqb;         // [1]
  int32_t* req_base;    // [B + 1] scratch
  CtaWork* cta;         // [kMaxCtas]: each CTA's slice, so a CTA starts with one load
  int32_t max_qb;       // capacity of qb / tile_start
};

// Raises func's dynamic shared-memory limit to `bytes` on the current device.
// The attribute is held per device, so it is set once per device: *done has
// one bit per device ordinal (below 64), read and updated under a lock.
cudaError_t raise_smem_limit(const void* func, int bytes, uint64_t* done);

// One bounded pipeline wait that runs out (see dsa_selftest_wait_timeout).
cudaError_t launch_wait_selftest(int32_t* err, cudaStream_t stream);

// fp4: the cache has FP4 pages (E2M1 codes) instead of FP8 pages.
cudaError_t launch_k_quant_write(const void* k, int64_t n, int64_t row_stride, const int64_t* slot_mapping,
                                 uint8_t* cache, int64_t num_blocks, bool fp4, const RopeArgs& rope, int32_t* err,
                                 cudaStream_t stream);
cudaError_t launch_q_quant_fold(const void* q, const float* w, int64_t n_tokens, float softmax_scale,
                                uint8_t* q_fp8, float* q_scale, float* w_folded, const RopeArgs& rope,
                                int32_t* err, cudaStream_t stream);
cudaError_t launch_convert(const int32_t* logical, int64_t n_tokens, int topk, const int32_t* req_id,
                           const int32_t* block_table, int num_reqs, int64_t bt_stride, int stride_rows,
                           int32_t* physical, int32_t* valid_counts, int32_t* err, cudaStream_t stream);

struct PlanArgs {
  const int32_t* qsl;
  const int32_t* seq_lens;
  int num_reqs, num_decodes, num_decode_tokens, num_tokens;
  int64_t bt_stride;
  int grid;  // CTAs of the score kernels
  SegmentPlan pre;  // the prefill segment (the decode score kernel plans its own work)
  int32_t* err;
};


// Fused per-layer prologue: K quant + cache write of the step's tokens, q quant
// with the weight fold, and (when `plan`) the work plan.
struct PrologueArgs {
  const __nv_bfloat16* q;   // [T, 64, 128]
  const void* w;            // [T, w_row_stride]: fp32, or bf16 when w_bf16; the first 64 used
  int64_t w_row_stride;     // elements between the rows of w
  bool w_bf16;
  float softmax_scale;
  uint8_t* q_fp8;           // [T, 64, 128]
  float* w_folded;          // [T, 64]
  const __nv_bfloat16* k_new;     // [T, k_row_stride] (first 128 used) or nullptr
  int64_t k_row_stride;           // elements between the rows of k_new
  const int64_t* slot_mapping;    // [T]
  uint8_t* k_cache;
  int64_t num_blocks;
  bool k_fp4;               // k_cache has FP4 pages
  int n_tokens;
  RopeArgs rope;            // RoPE of q and k_new rows before the quantiser (optional)
  bool plan;
  PlanArgs p;
  uint32_t* hist;      // zeroed here for the score kernel: [hist_rows][kHistBins]
  uint32_t* hist2;     // zeroed here for the select: [hist_rows][kHistBins]
  uint32_t* counters;  // [hist_rows][kRowCounters]
  int hist_rows;
  int num_sms;         // SMs of the device: the grid is one wave
  bool pdl;            // launched as a programmatic dependent of the previous kernel
  int32_t* err;
};

cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t stream);

// Histogram bins of a decode row's scores: the top 11 bits of the
// order-preserving 32-bit key (sign, exponent, 2 mantissa bits).
constexpr int kHistBins = 2048;
constexpr int kHistShift = 21;

// Optional S5 fused into the top-k output: physical ids and valid counts.
struct TopkPhys {
  const int32_t* block_table;
  int64_t bt_stride;
  int stride_rows;
  int32_t* physical;
  int32_t* valid_counts;  // may be nullptr
  int32_t* err;
};

// Per decode row (multi-CTA select): ids placed, boundary-bin candidates,
// the boundary bin, the count above it.
constexpr int kRowCounters = 4;

// Rows up to this many scores are staged in shared memory by the top-k.
constexpr int kTopkRowCap = 12288;

struct LogitsArgs {
  const float* w_folded;
  const uint8_t* k_cache;
  const int32_t* block_table;
  int64_t bt_stride;
  int64_t num_blocks;
  float* logits;
  int64_t ld;
  uint32_t* hist;  // [hist_rows][kHistBins] or nullptr: decode rows' score histograms (zeroed before)
  int hist_rows;
  // request metadata, from which the decode score kernel plans its own slice
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* req_id;
  int num_decodes;
  int num_dec_tokens;
  int32_t* err;
};

struct SelectArgs {
  const float* logits;
  int64_t ld;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* req_id;
  int num_reqs;
  int n_rows;               // decode rows [0, n_rows)
  int topk;
  int32_t* out;             // [T, topk]
  const uint32_t* hist;     // [n_rows][kHistBins]
  uint32_t* counters;       // [n_rows][kRowCounters], zeroed before: ids placed, candidates, b1, count above b1
  uint2* cand;              // [n_rows][ld]: (key, id) of the boundary bin
  uint32_t* hist2;          // [n_rows][kHistBins], zeroed before: the boundary bin's next 11 bits
};

// ntok_per_block = 1 (decode segment: the kernel plans its slice from the
// request metadata in `a`, `plan` is unused) or kPrefillTok (prefill segment,
// `plan` written by the prologue). fp4: the K cache has FP4 pages and tmap_k
// describes them (make_kcache_map with fp4); tmap_s is the pages' scale rows
// (make_kscale_map).
cudaError_t launch_logits(int ntok_per_block, bool fp4, const CUtensorMap* tmap_k, const CUtensorMap* tmap_s,
                          const CUtensorMap* tmap_q, SegmentPlan plan, const LogitsArgs& a, int num_sms,
                          cudaStream_t stream);

// Rows [row_begin, n_tokens): one CTA per row. Rows t < hist_rows take their
// first radix pass from hist (the score kernel's histograms; may be nullptr).
cudaError_t launch_topk(const float* logits, int64_t ld, const int32_t* qsl, const int32_t* seq_lens,
                        const int32_t* req_id, int num_reqs, int row_begin, int n_tokens, int topk, int32_t* out,
                        const TopkPhys* phys, const uint32_t* hist, int hist_rows, cudaStream_t stream);

// Decode rows [0, a.n_rows) whose score histograms the score kernel built:
// one CTA per row when the rows fit one CTA's shared memory; else each row in
// chunks (one CTA per chunk) and a second launch, one CTA per row, resolving
// the boundary bin.
cudaError_t launch_select(const SelectArgs& a, const TopkPhys* phys, int num_sms, cudaStream_t stream);

// The consumer's gather: out[i] = row physical[i] (row_bytes, a multiple of
// 16, from rows row_stride bytes apart), zeros for -1 or out of range.
cudaError_t launch_gather_rows(const uint8_t* rows, int64_t num_rows, int64_t row_bytes, int64_t row_stride,
                               const int32_t* physical, int64_t n_ids, uint8_t* out, int num_sms, int32_t* err,
                               cudaStream_t stream);

}  // namespace dsa
