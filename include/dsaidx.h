/*
 * dsaidx.h — C ABI of the GB300 (sm_103a) DSA sparse-attention indexer with
 * IndexCache cross-layer reuse.
 *
 * The operation is DeepSeek-V3.2's "lightning indexer" as vLLM runs it,
 * described by three web pages, cited by short name:
 *   [IC] "IndexCache：DeepSeek 稀疏注意力中的跨层索引复用" (atomage.cn) —
 *        snippets of `Indexer.forward`, the FP8 indexer K cache
 *        (`DeepseekV32IndexerCache`, `DeepseekV32IndexerBackend`),
 *        `SparseAttnIndexer`, `DeepseekV32IndexerMetadata`, the IndexCache
 *        layer schedule and the shared `topk_indices_buffer`;
 *   [PR] "PR #37735 完整报告" (prhub.com.cn), vLLM "[Feature]: IndexCache
 *        support for DSA models" — sections 实现拆解, 关键源码片段, 风险与影响;
 *   [IG] "vllm.v1.attention.backends.mla.index_group" (docs.vllm.ai) —
 *        `SparseMLAIndexGroup._convert_once`, `SparseMLAIndexGroupBuilder`.
 *
 * Shapes are fixed by the model: H = 64 indexer heads of dim D = 128 sharing
 * one K row per token (MQA), pages of 64 slots.
 *
 * Conventions for every entry point:
 *  - Ownership: the caller owns every buffer. Pointers marked "device" are
 *    device memory of the current CUDA device; "host" pointers are read
 *    during the call only. The library never allocates device memory: the
 *    scratch an entry point needs is a caller buffer of the size that the
 *    matching *_workspace_size() returns.
 *  - Launches are asynchronous on `stream` (NULL = legacy default stream);
 *    a call returns once its kernels are queued.
 *  - Status: every entry point returns DSA_OK (0) or an error code below;
 *    dsa_status_string() names it. Argument errors are found on the host
 *    before anything is launched (nothing is written then).
 *  - Device error word: entry points that take `dev_err` (a device int32,
 *    zeroed by the caller) OR a DSA_DEVERR_* bit into it when the data is
 *    inconsistent — a slot or block id outside the cache, a token id beyond
 *    its block-table row, a wait that ran out of time. The kernel then skips
 *    the offending access (no trap, no fault) and keeps going; results that
 *    depend on the skipped data are unspecified. dev_err may be NULL.
 *  - Alignment: all device pointers 16-byte aligned; the K cache is
 *    num_blocks pages of 8448 bytes (FP8) or, 32-byte aligned, of 4352 bytes
 *    (FP4, DsaBatch.k_cache_format = DSA_KCACHE_FP4).
 */
#ifndef DSAIDX_H
#define DSAIDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dsa_stream_t; /* same type as cudaStream_t */

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

/* ---------------------------------------------------------------- status */
#define DSA_OK 0
#define DSA_EINVAL 1   /* bad argument: shape, pointer, pattern, frequency, size */
#define DSA_ECUDA 2    /* a CUDA runtime/driver call failed */
#define DSA_EDEVICE 3  /* the device error word is nonzero (dsa_check_device_error) */
#define DSA_ENOSPACE 4 /* workspace smaller than *_workspace_size() */
#define DSA_ENODEV 5   /* no sm_103a device / kernel image for this device */

#define DSA_DEVERR_SLOT_RANGE 1u  /* slot_mapping entry >= num_blocks*64 */
#define DSA_DEVERR_BLOCK_RANGE 2u /* block-table entry outside [0, num_blocks) for a visible key */
#define DSA_DEVERR_ID_RANGE 4u    /* top-k id past its request's block-table row */
#define DSA_DEVERR_TIMEOUT 8u     /* a pipeline wait gave up (about 1 s); kernel returned early */
#define DSA_DEVERR_SEQ_RANGE 16u  /* seq_len < q_len, or seq_len beyond the block-table row */
#define DSA_DEVERR_POS_RANGE 32u  /* a RoPE position outside [0, max_pos): the row is left unrotated */

#define DSA_HEADS 64
#define DSA_HEAD_DIM 128
#define DSA_BLOCK_SIZE 64
#define DSA_SLOT_BYTES 132                        /* 128 B FP8 K + 4 B fp32 scale */
#define DSA_PAGE_BYTES (DSA_BLOCK_SIZE * DSA_SLOT_BYTES) /* 8448 */
#define DSA_FP4_SLOT_BYTES 68                             /* 64 B E2M1 K (two per byte) + 4 B fp32 scale */
#define DSA_FP4_PAGE_BYTES (DSA_BLOCK_SIZE * DSA_FP4_SLOT_BYTES) /* 4352 */
#define DSA_KCACHE_FP8 0
#define DSA_KCACHE_FP4 1

DSA_API const char *dsa_status_string(int status);
DSA_API int dsa_version(void); /* major*10000 + minor*100 + patch */

/* Copy the device error word to *out (synchronising `stream`) and return
 * DSA_EDEVICE if it is nonzero, DSA_OK otherwise. */
DSA_API int dsa_check_device_error(const int32_t *dev_err, uint32_t *out, dsa_stream_t stream);

/* Diagnostic, not part of the indexer: one thread waits, with the bounded
 * wait every pipeline of this library uses, on an mbarrier that nothing
 * completes. After about 1 s the wait gives up, ORs DSA_DEVERR_TIMEOUT into
 * *dev_err (device int32) and the kernel returns; the context stays usable.
 * It shows the failure path of the pipelines without a hang or a fault. */
DSA_API int dsa_selftest_wait_timeout(int32_t *dev_err, dsa_stream_t stream);

/* ------------------------------------------------------------ the batch */
/* One step's attention metadata, after [IC] `DeepseekV32IndexerMetadata`
 * (seq_lens, slot_mapping, num_decodes, ...) and the decode-first ordering of
 * [IG] `HiSparseMLAIndexGroup` (decode requests occupy rows [0, num_decodes)).
 * Request r has q_len[r] = query_start_loc[r+1] - query_start_loc[r] query
 * tokens and seq_lens[r] keys in total, this step's tokens included; query
 * token i of request r sits at position seq_lens[r] - q_len[r] + i and sees
 * keys [0, position] (causal, itself included). Key s of request r lives in
 * slot block_table[r*bt_stride + s/64]*64 + s%64 of the paged cache. A step
 * writes the K of its own tokens only, at their own slots (positions
 * [seq_lens[r] - q_len[r], seq_lens[r]) of each request), and no request
 * reads another's pages that the step writes: the decode score kernel may
 * fetch a request's earlier pages while this step's K write is still running. */
typedef struct DsaBatch {
  int32_t num_reqs;          /* B >= 0 */
  int32_t num_decodes;       /* requests [0, num_decodes) are run by the decode kernel */
  int32_t num_decode_tokens; /* query_start_loc[num_decodes] (host copy) */
  int32_t num_tokens;        /* T = query_start_loc[B] (host copy) */
  int32_t max_seq_len;       /* host upper bound of seq_lens[*]; sizes the score rows */
  int64_t bt_stride;       /* row stride of block_table, int32 elements */
  int64_t num_blocks;      /* pages in the K cache */
  const int32_t *query_start_loc;  /* device [B+1] */
  const int32_t *seq_lens;         /* device [B] */
  const int32_t *block_table;      /* device [B, bt_stride] */
  const int32_t *req_id_per_token; /* device [T] */
  int32_t k_cache_format;          /* DSA_KCACHE_FP8 (0) or DSA_KCACHE_FP4: the K cache's pages */
} DsaBatch;

/* ------------------------------------------------- S1: K quant + cache */
/* [IC] `SparseAttnIndexer` body, `indexer_k_quant_and_cache(k, kv_cache,
 * slot_mapping, quant_block_size, scale_fmt)`: each token's 128-dim K row is
 * quantised to FP8 E4M3 with one power-of-two (ue8m0) fp32 scale,
 * scale = 2^ceil(log2(max(amax, 1e-10)/448)), codes = RNE_satfinite(k/scale),
 * and stored at its slot: K bytes at page*8448 + (slot%64)*128, the scale at
 * page*8448 + 8192 + (slot%64)*4 (page = slot/64) — 132 bytes per slot as in
 * the [IC] FP8 cache snippet ("128 bytes K + 4 bytes FP32 scale").
 *   k            device bf16 [n_tokens, k_row_stride] (first 128 used)
 *   slot_mapping device int64 [n_tokens]; -1 = padding token, skipped
 *   k_cache      device uint8 [num_blocks, 8448], written in place
 * Slots >= num_blocks*64 are skipped and flag DSA_DEVERR_SLOT_RANGE. */
DSA_API int dsa_indexer_k_quant_write(const void *k, int64_t n_tokens, int64_t k_row_stride,
                              const int64_t *slot_mapping, uint8_t *k_cache,
                              int64_t num_blocks, int32_t *dev_err, dsa_stream_t stream);

/* ------------------------------------------------ the FP4 indexer K cache */
/* [IC] hands `sparse_attn_indexer` a `use_fp4_cache` flag beside
 * `quant_block_size` and `scale_fmt`; the pages give no more of the format.
 * Reading taken: the element is E2M1 (OCP Microscaling Formats (MX)
 * Specification v1.0, FP4: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) and the
 * quantiser is the FP8 cache's with E2M1 for E4M3 — one ue8m0 scale per
 * token's 128 values, scale = 2^ceil(log2(max(amax, 1e-10)/6)), codes =
 * RNE_satfinite(k/scale). Dim 2i goes to the low nibble and dim 2i+1 to the
 * high nibble of byte i. A page holds the 64 rows of 64 code bytes, then the
 * 64 fp32 scales: K bytes at page*4352 + (slot%64)*64, the scale at
 * page*4352 + 4096 + (slot%64)*4. q stays FP8; the scores multiply E2M1 K by
 * E4M3 q on the tensor cores (one kind::f8f6f4 MMA, the same fp32 sums).
 * Select it for the score calls with DsaBatch.k_cache_format = DSA_KCACHE_FP4.
 *   k_cache   device uint8 [num_blocks, 4352], 32-byte aligned, written
 *   positions, cos_sin, max_pos: as dsa_indexer_k_rope_quant_write, or
 *             cos_sin = NULL (positions unused) for rows that arrive rotated
 * Everything else as dsa_indexer_k_quant_write. */
DSA_API int dsa_indexer_k_quant_write_fp4(const void *k, int64_t n_tokens, int64_t k_row_stride,
                                  const int64_t *positions, const float *cos_sin, int64_t max_pos,
                                  const int64_t *slot_mapping, uint8_t *k_cache,
                                  int64_t num_blocks, int32_t *dev_err, dsa_stream_t stream);

/* ------------------------------------------ RoPE fused into S1 and S2a */
/* [IC] `Indexer.forward` rotates the leading qk_rope_head_dim = 64 dims of
 * every q head and of the shared K row, `rotary_emb(positions, q_pe, k_pe)`,
 * before the quantisation. These calls take un-rotated bf16 rows and rotate
 * them on the way into the quantiser: half-split pairs (i, i+32), i < 32,
 *   y[i] = x[i]*cos - x[i+32]*sin,  y[i+32] = x[i+32]*cos + x[i]*sin,
 * each product and sum rounded in fp32 (no fused multiply-add), the result
 * rounded to bf16 (the model's tensors are bf16), dims 64..127 unchanged.
 *   positions  device int64 [n_tokens]: the token's position
 *   cos_sin    device fp32 [max_pos, 64], 16-byte aligned: row p holds
 *              cos(p*f_i) for i < 32, then sin(p*f_i)
 * A position outside [0, max_pos) leaves the row unrotated and flags
 * DSA_DEVERR_POS_RANGE. Everything else as dsa_indexer_k_quant_write and
 * dsa_indexer_q_quant_fold (q rows of token t all take positions[t]). */
DSA_API int dsa_indexer_k_rope_quant_write(const void *k, int64_t n_tokens, int64_t k_row_stride,
                                   const int64_t *positions, const float *cos_sin, int64_t max_pos,
                                   const int64_t *slot_mapping, uint8_t *k_cache,
                                   int64_t num_blocks, int32_t *dev_err, dsa_stream_t stream);
DSA_API int dsa_indexer_q_rope_quant_fold(const void *q, const float *w, int64_t n_tokens,
                                  const int64_t *positions, const float *cos_sin, int64_t max_pos,
                                  float softmax_scale, uint8_t *q_fp8, float *q_scale,
                                  float *w_folded, int32_t *dev_err, dsa_stream_t stream);

/* --------------------------------------- S2a: q quant + weight folding */
/* [IC] `Indexer.forward`: q viewed as rows of 128 is quantised per row with a
 * ue8m0 scale exactly like K above, and the head weights absorb the scales,
 * w'[t,h] = w[t,h] * q_scale[t,h] * softmax_scale * 64^-0.5 (fp32, in that
 * order).
 *   q        device bf16 [n_tokens, 64, 128] contiguous
 *   w        device fp32 [n_tokens, 64]
 *   q_fp8    device uint8 [n_tokens, 64, 128] (E4M3 codes), written
 *   q_scale  device fp32 [n_tokens, 64] or NULL, written
 *   w_folded device fp32 [n_tokens, 64], written
 *   softmax_scale <= 0 selects 128^-0.5. */
DSA_API int dsa_indexer_q_quant_fold(const void *q, const float *w, int64_t n_tokens,
                             float softmax_scale, uint8_t *q_fp8, float *q_scale,
                             float *w_folded, dsa_stream_t stream);

/* ---------------------------------------- S2b + S3: logits and top-k */
/* Indexer scores over the causal keys of every query token,
 *   I[t,s] = k_scale[s] * sum_h w'[t,h] * ReLU(sum_d q8[t,h,d] * k8[s,d]),
 * FP8 x FP8 products accumulated in fp32 on the tensor cores, then the rows'
 * top-k ([IC]: the op fills `topk_indices_buffer`, whose rows start as -1).
 * topk_out[t, :] receives the request-local key ids of the `topk` largest
 * scores of row t, in no particular order, followed by -1 when the row has
 * fewer than `topk` keys. Every row [0, T) is written.
 *   q_fp8, w_folded  from dsa_indexer_q_quant_fold
 *   k_cache          device uint8 [num_blocks, 8448], or [num_blocks, 4352]
 *                    with batch->k_cache_format = DSA_KCACHE_FP4 (E2M1 K, see
 *                    dsa_indexer_k_quant_write_fp4); must hold every key the
 *                    rows see (write this step's K first, or pass k_new, which
 *                    is then quantised in the cache's format)
 *   topk             1..4096, multiple of 4
 *   topk_out         device int32 [T, topk]
 *   ws, ws_bytes     device scratch of dsa_indexer_workspace_size() bytes
 *   k_new, slot_mapping  optional (both NULL = [IC]'s skip_k_cache_insert):
 *                    this step's bf16 K rows [T,128] and their slots; they are
 *                    quantised into k_cache before any score is computed. */
DSA_API size_t dsa_indexer_workspace_size(const DsaBatch *batch, int32_t topk);
DSA_API int dsa_indexer_logits_topk(const DsaBatch *batch, const uint8_t *q_fp8,
                            const float *w_folded, uint8_t *k_cache, int32_t topk,
                            int32_t *topk_out, void *ws, size_t ws_bytes,
                            const void *k_new, const int64_t *slot_mapping,
                            int32_t *dev_err, dsa_stream_t stream);

/* The steps of the call above, one by one.
 * dsa_indexer_plan splits the batch into work items (query blocks x 128-key
 * tiles) and stores the plan in ws; it depends only on the batch metadata,
 * so one plan serves every layer of a step.
 * dsa_indexer_logits needs a plan in ws (same batch) and writes I[t, s] for
 * s in [0, position_t] to logits[t*logits_ld + s] (fp32; other entries
 * untouched); logits_ld >= max_seq_len.
 * dsa_indexer_topk selects from such a score matrix (ws unused, may be NULL). */
DSA_API int dsa_indexer_plan(const DsaBatch *batch, void *ws, size_t ws_bytes, int32_t *dev_err,
                     dsa_stream_t stream);
DSA_API int dsa_indexer_logits(const DsaBatch *batch, const uint8_t *q_fp8, const float *w_folded,
                       const uint8_t *k_cache, float *logits, int64_t logits_ld,
                       void *ws, size_t ws_bytes, int32_t *dev_err, dsa_stream_t stream);
DSA_API int dsa_indexer_topk(const DsaBatch *batch, const float *logits, int64_t logits_ld,
                     int32_t topk, int32_t *topk_out, void *ws, size_t ws_bytes,
                     dsa_stream_t stream);

/* Measurement aid (not a step of the method): a launch timeline. On the
 * calling host thread, the following calls of dsa_indexer_logits_topk,
 * dsa_indexer_logits and dsa_layer_stack_run record events[0], events[1], ...
 * in order: one before the first kernel of each fused call and one after
 * every kernel they launch, until the n_events handles (cudaEvent_t created by
 * the caller) are used up. Under CUDA-graph capture they become external
 * event nodes. cudaEventElapsedTime between consecutive events then gives each
 * kernel's device time on its own stream. n_events = 0 switches it off;
 * at most 32 events; a NULL handle is DSA_EINVAL. Host-only. */
DSA_API int dsa_set_launch_events(void *const *events, int32_t n_events);

/* dsa_indexer_logits_topk for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a service of this library. Callers
 * that cannot call cudaMalloc or supply a scratch buffer — plugins that are
 * handed only an op's input and output tensors, code whose device memory
 * belongs to a framework allocator it may not call, loops that must not touch
 * an allocator — get the same computation with the scratch taken from a
 * device array of
 * DSA_STATIC_WORKSPACE_BYTES inside the library. Every GPU that loads the
 * library holds that array until the process exits. Arguments are those of
 * dsa_indexer_logits_topk without ws/ws_bytes; the caller still passes all
 * inputs and outputs. Nothing is allocated: no cudaMalloc, no cudaFree, no
 * allocating library call.
 *  - A batch whose dsa_indexer_workspace_size() exceeds
 *    DSA_STATIC_WORKSPACE_BYTES is rejected with DSA_ENOSPACE before any
 *    launch (32 MiB holds, e.g., 81 decode tokens at 32K context or 292 at
 *    8K: their score rows, histograms and boundary candidates).
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *    The address belongs to the device's context: when that context has
 *    changed since (after cudaDeviceReset), the next call looks it up again,
 *    so that call too must come before any capture.
 *  - All calls share the array and it keeps the last call's contents; each
 *    call's first kernel writes the plan and clears the histograms and
 *    counters that must start at zero. Calls whose kernels overlap on the GPU —
 *    on two streams, or from two host threads — race on it: serialise them. */
#define DSA_STATIC_WORKSPACE_BYTES (32u << 20)
DSA_API int dsa_indexer_logits_topk_static(const DsaBatch *batch, const uint8_t *q_fp8,
                                   const float *w_folded, uint8_t *k_cache, int32_t topk,
                                   int32_t *topk_out, const void *k_new,
                                   const int64_t *slot_mapping, int32_t *dev_err,
                                   dsa_stream_t stream);

/* ------------------------------------------ S5: logical -> physical ids */
/* [IG] `SparseMLAIndexGroup._convert_once` (the conversion kernel it calls):
 * physical = block_table[req][id/64] * block_stride_rows + id%64, -1 stays -1;
 * valid_counts[t] = number of ids >= 0 in row t.
 *   logical          device int32 [n_tokens, topk]
 *   req_id_per_token device int32 [n_tokens]
 *   block_table      device int32 [num_reqs, bt_stride]
 *   block_stride_rows  rows per physical block; <= 0 selects 64
 *   physical         device int32 [n_tokens, topk], written
 *   valid_counts     device int32 [n_tokens] or NULL, written
 * An id whose page lies past bt_stride, or a negative block entry, gives -1
 * and flags DSA_DEVERR_ID_RANGE; so does every id of a token whose request
 * lies outside [0, num_reqs) (the block table is not read for it). */
DSA_API int dsa_topk_logical_to_physical(const int32_t *logical, int64_t n_tokens, int32_t topk,
                                 const int32_t *req_id_per_token, const int32_t *block_table,
                                 int32_t num_reqs, int64_t bt_stride, int32_t block_stride_rows,
                                 int32_t *physical, int32_t *valid_counts,
                                 int32_t *dev_err, dsa_stream_t stream);

/* ------------------------------------------------ S4: IndexCache schedule */
/* [IC] layer-construction snippet and [PR] 关键源码片段: with IndexCache on,
 * layer l is 'S' (reuses the previous top-k) iff max(l - offset + 1, 0) % freq
 * != 0 (offset 2 by default, i.e. max(l-1,0) % freq), unless an explicit
 * pattern is given ('F' = compute, 'S' = reuse); with it off every layer is
 * 'F'. producer_out[l] = the 'F' layer whose top-k layer l consumes.
 * Host-only, synchronous. Stricter than the page ([PR] 风险与影响): the
 * pattern must be exactly n_layers characters of 'F'/'S' starting with 'F';
 * freq >= 1; layer 0 must be 'F'. Otherwise DSA_EINVAL and nothing written.
 *   fs_out       host char [n_layers] ('F'/'S', not NUL-terminated)
 *   producer_out host int32 [n_layers] */
DSA_API int dsa_schedule_build(int32_t n_layers, int32_t use_index_cache, int32_t freq,
                       int32_t offset, const char *pattern, char *fs_out,
                       int32_t *producer_out);

/* ------------------------------------ the consumer's gather of the rows */
/* [IC]: the sparse MLA of each layer reads, per query token, the KV rows of the
 * selected keys; [IG] `_convert_once` gives it physical slots for that read.
 * The row format is not on the pages, so this copies bytes:
 *   out[t][j] = rows[physical[t][j] * row_stride .. + row_bytes)
 * and zeros where the id is -1 (rows shorter than k keep -1 in the tail).
 *   rows        device uint8, num_rows rows row_stride bytes apart, 16-byte aligned
 *   row_bytes   bytes per row copied: > 0, a multiple of 16, <= row_stride
 *   row_stride  a multiple of 16
 *   physical    device int32 [n_tokens, topk] (dsa_topk_logical_to_physical,
 *               or phys_buf of the layer runner)
 *   out         device uint8 [n_tokens, topk, row_bytes], 16-byte aligned, written
 * An id outside [-1, num_rows) gives a zero row and flags DSA_DEVERR_ID_RANGE. */
DSA_API int dsa_gather_rows(const uint8_t *rows, int64_t num_rows, int64_t row_bytes, int64_t row_stride,
                            const int32_t *physical, int64_t n_tokens, int32_t topk, uint8_t *out,
                            int32_t *dev_err, dsa_stream_t stream);

/* ------------------------------------------- the layer-schedule runner */
/* One decoding step over a stack of DSA layers with IndexCache: [IC] F/S
 * layer forward and [IG] `SparseMLAIndexGroup` (one group = an F layer and
 * the S layers after it; the leader converts the group's indices once).
 * For every 'F' layer l (per the schedule): quantise this step's K of layer l
 * into its cache, quantise q and fold w, run logits + top-k into topk_buf,
 * convert to physical ids in phys_buf/valid_buf (once for the group). Then
 * for every layer (F or S) the optional consumer is called on the host with
 * the group's buffers, in layer order, after that layer's device work is
 * queued on `stream`; it may enqueue its own work on the stream (the sparse
 * attention that reads the indices). 'S' layers own no indexer inputs: their
 * entries of `layers` are ignored and may be zero.
 * Streams: with decode and prefill rows in the batch, part of each F layer
 * runs on a second stream of the calling host thread (created on the first
 * such call, outside stream capture, and kept with two events for the life of
 * the thread; highest priority): with the step's work given (decode_keys,
 * prefill_pairs below) the decode rows' scores and top-k, forked after the
 * layer's prologue; without it the decode rows' top-k, forked after the
 * scores. It is joined back to `stream` before the layer's consumer call, so
 * every later operation on `stream` sees the layer's complete output. In
 * stream capture the fork and join become graph edges. Without that second
 * stream (capture before the first such call, or a launch timeline set by
 * dsa_set_launch_events) the same kernels run on `stream` one after another.
 * After the first F layer of a call without a consumer, each F layer's first
 * kernel starts as a programmatic dependent of the previous layer's top-k
 * (the inputs of every layer are the caller's, fixed for the call). */
#define DSA_W_FP32 0
#define DSA_W_BF16 1
typedef struct DsaLayerInputs {
  const void *q;        /* device bf16 [T, 64, 128] */
  const void *w;        /* device [T, w_row_stride], the first 64 of a row used: fp32, or bf16 with
                           w_dtype = DSA_W_BF16 (converted exactly to fp32 before the fold) */
  const void *k_new;    /* device bf16 [T, k_row_stride] (first 128 used) or NULL (skip the cache insert) */
  uint8_t *k_cache;     /* device uint8 [num_blocks, 8448], or 4352 with an FP4 batch */
  int64_t k_row_stride; /* elements between k_new rows: 0 = 128, else >= 128 and a multiple of 8 */
  int64_t w_row_stride; /* elements between w rows: 0 = 64, else >= 64 */
  int32_t w_dtype;      /* DSA_W_FP32 (0) or DSA_W_BF16 (1) */
} DsaLayerInputs;
/* [IC] `Indexer.forward` takes k = kw[:, :128] and weights = kw[:, 128:] as
 * column views of one fused projection output kw, bf16 [T, 128 + 64]; pass
 * them as they are: k_new = kw, k_row_stride = 192, w = kw + 128 (elements),
 * w_row_stride = 192, w_dtype = DSA_W_BF16. Zero strides and w_dtype keep the
 * contiguous fp32 layout of the fields above. */

typedef void (*dsa_layer_consumer_fn)(int32_t layer, int32_t producer,
                                      const int32_t *physical, const int32_t *valid_counts,
                                      void *user);

typedef struct DsaStackPlan {
  int32_t n_layers;
  const char *fs;                 /* host [n_layers] from dsa_schedule_build */
  const DsaLayerInputs *layers;   /* host [n_layers] */
  int32_t topk;
  float softmax_scale;            /* <= 0 selects 128^-0.5 */
  int32_t block_stride_rows;      /* for the conversion; <= 0 selects 64 */
  /* RoPE fused into the per-layer prologue (see dsa_indexer_q_rope_quant_fold):
   * rope_cos_sin = NULL means q and k_new arrive already rotated. */
  const int64_t *positions;       /* device int64 [T] */
  const float *rope_cos_sin;      /* device fp32 [rope_max_pos, 64] or NULL */
  int64_t rope_max_pos;
  /* The step's work per segment, counted by the caller from its host copy of
   * the metadata (0 = not given): decode_keys = the sum over the decode
   * tokens of the keys each sees (its position + 1), prefill_pairs = the
   * same sum over the prefill tokens. With both given and neither side too
   * small, every F layer scores the decode rows on a share of the SMs while
   * the prefill rows are scored on the rest (the decode scores are bound by
   * HBM on the whole GPU, the prefill scores by the tensor cores), each
   * segment's top-k following its scores; the share balances the two at
   * per-SM rates measured on GB300. Not used while a launch timeline is set
   * (dsa_set_launch_events times every kernel alone on the whole GPU). */
  int64_t decode_keys;
  int64_t prefill_pairs;
} DsaStackPlan;

DSA_API size_t dsa_layer_stack_workspace_size(const DsaBatch *batch, int32_t topk);
/* The SMs dsa_layer_stack_run would give the decode rows' scores on this
 * device (plan->decode_keys, plan->prefill_pairs and the batch; a launch
 * timeline set on this thread counts), written to *decode_sms; 0 = decode and
 * prefill scores one after the other. Host only, no launch. */
DSA_API int dsa_layer_stack_decode_sms(const DsaStackPlan *plan, const DsaBatch *batch, int32_t *decode_sms);
DSA_API int dsa_layer_stack_run(const DsaStackPlan *plan, const DsaBatch *batch,
                        const int64_t *slot_mapping, int32_t *topk_buf,
                        int32_t *phys_buf, int32_t *valid_buf,
                        dsa_layer_consumer_fn consumer, void *user, void *ws,
                        size_t ws_bytes, int32_t *dev_err, dsa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DSAIDX_H */
