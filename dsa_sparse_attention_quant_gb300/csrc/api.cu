// api.cu — the C ABI declared in include/dsaidx.h: argument checks, workspace
// carving, TMA descriptors and kernel launches. Host code only.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/dsaidx.h"
#include "kernels.h"

using namespace dsa;

namespace {
std::mutex g_attr_mutex;
}  // namespace

cudaError_t dsa::raise_smem_limit(const void* func, int bytes, uint64_t* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const uint64_t bit = uint64_t{1} << dev;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  if (*done & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) *done |= bit;
  return e;
}

namespace {

constexpr int kMaxDevices = 64;

int g_num_sms[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_mutex;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return DSA_OK;
  if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver)
    return DSA_ENODEV;
  return DSA_ECUDA;
}

// SM count of the current device; DSA_ENODEV unless it is an sm_103 part.
int device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ENODEV;
  if (dev < 0 || dev >= kMaxDevices) return DSA_ENODEV;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_num_sms[dev] == 0) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DSA_ENODEV;
    if (major != 10 || minor != 3) return DSA_ENODEV;
    g_num_sms[dev] = n;
  }
  *sms = g_num_sms[dev];
  return DSA_OK;
}

int tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return DSA_ENODEV;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = g_encode;
  return DSA_OK;
}

// K cache as a 3-D tensor {128 K values, 64 slots, num_blocks pages}: one box
// is the 64 K rows of one page, landed with the 128-byte swizzle. FP8 pages
// are read as bytes; FP4 pages with the packed 4-bit type, which lands each
// 64-byte row as 128 bytes (8 code bytes, then an 8-byte gap, per 16 bytes),
// the layout the MMA reads E2M1 operands in. That type wants a 32-byte
// aligned base and strides (64 and 4352 are).
int make_kcache_map(CUtensorMap* m, const uint8_t* cache, int64_t num_blocks, bool fp4) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int st = tensor_map_encoder(&enc);
  if (st != DSA_OK) return st;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(kBlock),
                        static_cast<cuuint64_t>(num_blocks)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(fp4 ? kDim / 2 : kDim),
                           static_cast<cuuint64_t>(fp4 ? kFp4PageBytes : kPageBytes)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kDim), static_cast<cuuint32_t>(kBlock), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                   const_cast<uint8_t*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DSA_OK : DSA_ECUDA;
}

// The K cache's scale rows as a 2-D fp32 tensor {64, num_blocks}: row p is
// page p's 64 scales (after its codes); one-row boxes, for the score kernel's
// tile::gather4 of a tile's two rows.
int make_kscale_map(CUtensorMap* m, const uint8_t* cache, int64_t num_blocks, bool fp4) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int st = tensor_map_encoder(&enc);
  if (st != DSA_OK) return st;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kBlock), static_cast<cuuint64_t>(num_blocks)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(fp4 ? kFp4PageBytes : kPageBytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlock), 1};
  cuuint32_t estr[2] = {1, 1};
  uint8_t* scales = const_cast<uint8_t*>(cache) + (fp4 ? kFp4ScaleOffset : kScaleOffset);
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, scales, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DSA_OK : DSA_ECUDA;
}

// q codes as a 2-D byte tensor {128, T*64}: one box is `rows` head rows.
int make_q_map(CUtensorMap* m, const uint8_t* q, int64_t n_tokens, int rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int st = tensor_map_encoder(&enc);
  if (st != DSA_OK) return st;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(n_tokens * kHeads)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDim)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kDim), static_cast<cuuint32_t>(rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DSA_OK : DSA_ECUDA;
}

int check_batch(const DsaBatch* b) {
  if (b == nullptr) return DSA_EINVAL;
  if (b->num_reqs < 0 || b->num_decodes < 0 || b->num_decodes > b->num_reqs || b->num_tokens < 0)
    return DSA_EINVAL;
  if (b->num_decode_tokens < 0 || b->num_decode_tokens > b->num_tokens) return DSA_EINVAL;
  if (b->num_tokens > 0 && (b->num_reqs == 0 || b->max_seq_len < 1)) return DSA_EINVAL;
  if (b->num_reqs > 0 &&
      (b->query_start_loc == nullptr || b->seq_lens == nullptr || b->block_table == nullptr ||
       b->bt_stride < 1 || b->num_blocks < 1 || b->num_blocks > (int64_t{1} << 31) - 1))
    return DSA_EINVAL;
  if (b->num_tokens > 0 && b->req_id_per_token == nullptr) return DSA_EINVAL;
  if (static_cast<int64_t>(b->num_tokens) * kHeads > (int64_t{1} << 31) - 1) return DSA_EINVAL;
  if (b->k_cache_format != DSA_KCACHE_FP8 && b->k_cache_format != DSA_KCACHE_FP4) return DSA_EINVAL;
  return DSA_OK;
}

bool kcache_fp4(const DsaBatch* b) { return b->k_cache_format == DSA_KCACHE_FP4; }

// The K cache base: 16-byte aligned, 32 for FP4 pages (the packed TMA type).
bool kcache_aligned(const DsaBatch* b, const void* k_cache) {
  return k_cache != nullptr && reinterpret_cast<uintptr_t>(k_cache) % (kcache_fp4(b) ? 32 : 16) == 0;
}

int64_t logits_ld(const DsaBatch* b) {
  return static_cast<int64_t>(align_up(b->max_seq_len > 0 ? b->max_seq_len : 1, 4));
}

// Persistent logits grid: one CTA per SM. The plan and the launch must agree on it.
int grid_ctas(int sms) { return sms < kMaxCtas ? sms : kMaxCtas; }

// Workspace of the indexer: the prefill segment's plan (the decode score kernel
// plans its own work), the score matrix, and for the decode rows the score
// histograms, top-k counters and boundary candidates.
struct IndexerWs {
  SegmentPlan pre;
  float* logits;
  uint32_t* hist;
  uint32_t* hist2;
  uint32_t* counters;
  uint2* cand;
  int hist_rows;
  size_t bytes;
};

IndexerWs carve(const DsaBatch* b, void* base) {
  IndexerWs w{};
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    void* r = p ? p + off : nullptr;
    off = align_up(off + bytes, 256);
    return r;
  };
  const size_t T = static_cast<size_t>(b->num_tokens);
  const size_t B = static_cast<size_t>(b->num_reqs);
  const size_t Td = static_cast<size_t>(b->num_decode_tokens);
  const size_t ld = static_cast<size_t>(logits_ld(b));
  const size_t max_pre = T / kPrefillTok + B + 1;
  w.pre.qb = static_cast<QBlock*>(take(max_pre * sizeof(QBlock)));
  w.pre.tile_start = static_cast<int32_t*>(take((max_pre + 1) * 4));
  w.pre.nqb = static_cast<int32_t*>(take(4));
  w.pre.req_base = static_cast<int32_t*>(take((B + 1) * 4));
  w.pre.cta = static_cast<CtaWork*>(take(kMaxCtas * sizeof(CtaWork)));
  w.pre.max_qb = static_cast<int32_t>(max_pre);
  w.logits = static_cast<float*>(take(T * ld * 4));
  w.hist = static_cast<uint32_t*>(take(Td * kHistBins * 4));
  w.hist2 = static_cast<uint32_t*>(take(Td * kHistBins * 4));
  w.counters = static_cast<uint32_t*>(take(Td * kRowCounters * 4));
  w.cand = static_cast<uint2*>(take(Td * ld * sizeof(uint2)));
  w.hist_rows = static_cast<int>(Td);
  w.bytes = off;
  return w;
}

// The prefill plan for a score kernel of pre_grid CTAs.
PlanArgs plan_args(const DsaBatch* b, const IndexerWs& ws, int pre_grid, int32_t* dev_err) {
  return PlanArgs{b->query_start_loc, b->seq_lens,    b->num_reqs, b->num_decodes, b->num_decode_tokens,
                  b->num_tokens,      b->bt_stride,   pre_grid,    ws.pre,         dev_err};
}

// Prologue with no q: (optional) K quant + cache write, the prefill plan (when
// the batch has prefill requests) for a prefill score kernel of pre_grid CTAs,
// and zeroed decode-row histograms and counters.
PrologueArgs plan_only(const DsaBatch* b, const IndexerWs& ws, int sms, int pre_grid, const void* k_new,
                       const int64_t* slot_mapping, uint8_t* k_cache, int32_t* dev_err) {
  PrologueArgs pa{};
  pa.k_new = static_cast<const __nv_bfloat16*>(k_new);
  pa.k_row_stride = kDim;
  pa.w_row_stride = kHeads;
  pa.slot_mapping = slot_mapping;
  pa.k_cache = k_cache;
  pa.num_blocks = b->num_blocks;
  pa.k_fp4 = kcache_fp4(b);
  pa.n_tokens = b->num_tokens;
  pa.plan = b->num_reqs > b->num_decodes;
  pa.p = plan_args(b, ws, pre_grid, dev_err);
  pa.hist = ws.hist;
  pa.hist2 = ws.hist2;
  pa.counters = ws.counters;
  pa.hist_rows = ws.hist_rows;
  pa.num_sms = sms;
  pa.err = dev_err;
  return pa;
}

// Launch timeline set by dsa_set_launch_events for this host thread: one
// event before the first kernel of each call and one after every kernel.
constexpr int kMaxTimeline = 32;
thread_local cudaEvent_t t_events[kMaxTimeline];
thread_local int t_count = 0;
thread_local int t_next = 0;

int mark(cudaStream_t stream) {
  if (t_next >= t_count) return DSA_OK;
  return from_cuda(cudaEventRecordWithFlags(t_events[t_next++], stream, cudaEventRecordExternal));
}

// Status of a kernel launch, followed by the timeline mark after it.
int launched(cudaError_t e, cudaStream_t stream) {
  const int st = from_cuda(e);
  return st != DSA_OK ? st : mark(stream);
}

// Scores for both segments (the prefill plan is already in ws). With `hist`,
// the decode kernel also accumulates the decode rows' histograms (zeroed before).
int run_logits(const DsaBatch* b, const uint8_t* q_fp8, const float* w_folded, const uint8_t* k_cache,
               float* logits, int64_t ld, const IndexerWs& ws, bool hist, int32_t* dev_err, cudaStream_t stream) {
  if (b->num_tokens == 0) return DSA_OK;
  int sms = 0;
  int st = device_sms(&sms);
  if (st != DSA_OK) return st;
  CUtensorMap mk, ms, mq1, mq4;
  const bool fp4 = kcache_fp4(b);
  if ((st = make_kcache_map(&mk, k_cache, b->num_blocks, fp4)) != DSA_OK) return st;
  if ((st = make_kscale_map(&ms, k_cache, b->num_blocks, fp4)) != DSA_OK) return st;
  LogitsArgs a{w_folded,          k_cache,    b->block_table,   b->bt_stride,   b->num_blocks,
               logits,            ld,         hist ? ws.hist : nullptr,          hist ? ws.hist_rows : 0,
               b->query_start_loc, b->seq_lens, b->req_id_per_token, b->num_decodes, b->num_decode_tokens,
               dev_err};
  if (b->num_decodes > 0) {
    if ((st = make_q_map(&mq1, q_fp8, b->num_tokens, kHeads)) != DSA_OK) return st;
    if ((st = launched(launch_logits(1, fp4, &mk, &ms, &mq1, SegmentPlan{}, a, grid_ctas(sms), stream), stream)) !=
        DSA_OK)
      return st;
  }
  if (b->num_reqs > b->num_decodes) {
    if ((st = make_q_map(&mq4, q_fp8, b->num_tokens, kPrefillTok * kHeads)) != DSA_OK) return st;
    if ((st = launched(launch_logits(kPrefillTok, fp4, &mk, &ms, &mq4, ws.pre, a, grid_ctas(sms), stream), stream)) !=
        DSA_OK)
      return st;
  }
  return DSA_OK;
}

// A second stream of this host thread on one device, with its fork and join
// events: the decode rows' select runs on it beside the prefill rows' top-k.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local SideStream t_side[kMaxDevices];

// The side stream of the current device, created on first use (highest
// priority, so the short select's CTAs are placed first), or nullptr: the
// caller then launches both top-k kernels on its own stream. Not used while a
// launch timeline is set (it times every kernel alone), and never created
// while `stream` is being captured.
SideStream* side_stream(cudaStream_t stream) {
  if (t_count > 0) return nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& ss = t_side[dev];
  if (ss.stream != nullptr) return &ss;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return nullptr;
  }
  int least = 0, greatest = 0;
  SideStream n;
  if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
      cudaStreamCreateWithPriority(&n.stream, cudaStreamNonBlocking, greatest) != cudaSuccess ||
      cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();  // not sticky: fall back to one stream
    if (n.join) cudaEventDestroy(n.join);
    if (n.fork) cudaEventDestroy(n.fork);
    if (n.stream) cudaStreamDestroy(n.stream);
    return nullptr;
  }
  ss = n;
  return &ss;
}

// Top-k of every row from scores built with the decode rows' histograms:
// the decode rows by the select (one CTA per row that fits its shared memory,
// else chunk CTAs and a resolving CTA, pass 1 from the histograms), the
// others by one CTA per row. The two read and write disjoint rows; with
// `side`, when both are present, the select runs on the side stream (forked
// from `stream` after the scores, joined back before return), beside the
// prefill rows' top-k: its CTAs fill only as many SMs as there are decode rows.
int run_topk(const DsaBatch* b, const IndexerWs& ws, int64_t ld, int32_t topk, int32_t* out, const TopkPhys* phys,
             int sms, bool side, cudaStream_t stream) {
  SelectArgs sa{ws.logits, ld, b->query_start_loc, b->seq_lens, b->req_id_per_token, b->num_reqs,
                ws.hist_rows, topk, out, ws.hist, ws.counters, ws.cand, ws.hist2};
  const bool dec = ws.hist_rows > 0, pre = b->num_tokens > ws.hist_rows;
  SideStream* ss = side && dec && pre ? side_stream(stream) : nullptr;
  int st = DSA_OK;
  if (ss != nullptr) {
    if ((st = from_cuda(cudaEventRecord(ss->fork, stream))) != DSA_OK) return st;
    if ((st = from_cuda(cudaStreamWaitEvent(ss->stream, ss->fork, 0))) != DSA_OK) return st;
    // from here on the side stream is joined back whatever fails
    st = from_cuda(launch_select(sa, phys, sms, ss->stream));
    const int r = from_cuda(cudaEventRecord(ss->join, ss->stream));
    if (st == DSA_OK) st = r;
  } else if (dec) {
    st = launched(launch_select(sa, phys, sms, stream), stream);
  }
  if (pre && st == DSA_OK)
    st = launched(launch_topk(ws.logits, ld, b->query_start_loc, b->seq_lens, b->req_id_per_token, b->num_reqs,
                              ws.hist_rows, b->num_tokens, topk, out, phys, nullptr, 0, stream),
                  stream);
  if (ss != nullptr) {
    const int j = from_cuda(cudaStreamWaitEvent(stream, ss->join, 0));
    if (st == DSA_OK) st = j;
  }
  return st;
}

// Per-SM rates of the score kernels on GB300, measured: a decode CTA's K-tile
// pipeline took about 0.34 us per 128-key tile whatever the number of CTAs
// (decode8x128k on 40 to 100 SMs: 47-50 GB/s per SM) with four copies a
// tile, and about 13% less with three (the scale rows by one gather4); on the
// whole GPU the shared HBM holds it to about 0.40 us. The prefill kernel
// scores about 730-890 pairs per us per SM (stack61, prefill4x8k). With these,
// stack61's share is 49 SMs (sweep with three copies a tile: 44 / 47 / 50 / 53
// SMs, 174.6 / 173.0 / 173.0 / 175.6 us per F layer).
constexpr double kDecodeKeysPerSmUs = 425.0;
constexpr double kPrefillPairsPerSmUs = 800.0;
constexpr int kMinSplitSms = 16;

// SMs for the decode rows' scores when they run beside the prefill rows'
// scores, or 0 (one after the other): the share that makes both take the same
// time at the rates above. The decode kernel on the whole GPU is bound by HBM
// at about 35 GB/s per SM, so a share streams K at nearly the HBM rate of the
// whole GPU's while the other SMs compute the prefill: stack61 (64 decodes at
// 32768 keys, a 4096-token prefill; 53 of 152 SMs at four copies a tile)
// 211 -> 193 us per F layer.
int decode_split(const DsaStackPlan* plan, const DsaBatch* b, int sms) {
  if (t_count > 0) return 0;  // a launch timeline times every kernel alone, on the whole GPU
  if (plan->decode_keys <= 0 || plan->prefill_pairs <= 0 || b->num_decodes == 0 || b->num_reqs == b->num_decodes)
    return 0;
  const double wd = static_cast<double>(plan->decode_keys) / kDecodeKeysPerSmUs;
  const double wp = static_cast<double>(plan->prefill_pairs) / kPrefillPairsPerSmUs;
  const int s = static_cast<int>(sms * wd / (wd + wp) + 0.5);
  return (s < kMinSplitSms || s > sms - kMinSplitSms || sms - s > kMaxCtas) ? 0 : s;
}

// One F layer's scores and top-k with the SMs split: the decode rows' scores
// (split CTAs) and select on the side stream, the prefill rows' scores (the
// rest, as planned) and top-k on `stream`, joined back before return. Without
// a side stream (stream capture before its first use) the same launches run
// one after the other on `stream`.
int run_split(const DsaBatch* b, const uint8_t* q_fp8, const float* w_folded, const uint8_t* k_cache,
              const IndexerWs& ws, int64_t ld, int32_t topk, int32_t* out, const TopkPhys* phys, int sms, int split,
              int32_t* dev_err, cudaStream_t stream) {
  CUtensorMap mk, ms, mq1, mq4;
  const bool fp4 = kcache_fp4(b);
  int st;
  if ((st = make_kcache_map(&mk, k_cache, b->num_blocks, fp4)) != DSA_OK) return st;
  if ((st = make_kscale_map(&ms, k_cache, b->num_blocks, fp4)) != DSA_OK) return st;
  if ((st = make_q_map(&mq1, q_fp8, b->num_tokens, kHeads)) != DSA_OK) return st;
  if ((st = make_q_map(&mq4, q_fp8, b->num_tokens, kPrefillTok * kHeads)) != DSA_OK) return st;
  LogitsArgs a{w_folded,          k_cache,     b->block_table,       b->bt_stride,   b->num_blocks,
               ws.logits,         ld,          ws.hist,              ws.hist_rows,
               b->query_start_loc, b->seq_lens, b->req_id_per_token, b->num_decodes, b->num_decode_tokens,
               dev_err};
  SelectArgs sa{ws.logits, ld, b->query_start_loc, b->seq_lens, b->req_id_per_token, b->num_reqs,
                ws.hist_rows, topk, out, ws.hist, ws.counters, ws.cand, ws.hist2};
  SideStream* ss = side_stream(stream);
  cudaStream_t ds = ss != nullptr ? ss->stream : stream;
  if (ss != nullptr) {
    if ((st = from_cuda(cudaEventRecord(ss->fork, stream))) != DSA_OK) return st;
    if ((st = from_cuda(cudaStreamWaitEvent(ss->stream, ss->fork, 0))) != DSA_OK) return st;
  }
  // from here on the side stream is joined back whatever fails
  st = from_cuda(launch_logits(1, fp4, &mk, &ms, &mq1, SegmentPlan{}, a, split, ds));
  if (st == DSA_OK) st = from_cuda(launch_select(sa, phys, sms, ds));
  if (ss != nullptr) {
    const int r = from_cuda(cudaEventRecord(ss->join, ss->stream));
    if (st == DSA_OK) st = r;
  }
  if (st == DSA_OK) st = from_cuda(launch_logits(kPrefillTok, fp4, &mk, &ms, &mq4, ws.pre, a, sms - split, stream));
  if (st == DSA_OK)
    st = from_cuda(launch_topk(ws.logits, ld, b->query_start_loc, b->seq_lens, b->req_id_per_token, b->num_reqs,
                               ws.hist_rows, b->num_tokens, topk, out, phys, nullptr, 0, stream));
  if (ss != nullptr) {
    const int j = from_cuda(cudaStreamWaitEvent(stream, ss->join, 0));
    if (st == DSA_OK) st = j;
  }
  return st;
}

bool topk_ok(int32_t topk) { return topk >= 4 && topk <= 4096 && topk % 4 == 0; }

}  // namespace

extern "C" {

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_EINVAL: return "invalid argument";
    case DSA_ECUDA: return "CUDA call failed";
    case DSA_EDEVICE: return "device reported inconsistent data (see the device error word)";
    case DSA_ENOSPACE: return "workspace too small";
    case DSA_ENODEV: return "no sm_103 device or kernel image";
    default: return "unknown status";
  }
}

int dsa_version(void) { return 301; }

int dsa_selftest_wait_timeout(int32_t* dev_err, dsa_stream_t stream) {
  if (dev_err == nullptr || reinterpret_cast<uintptr_t>(dev_err) % 4 != 0) return DSA_EINVAL;
  int sms;
  int st = device_sms(&sms);
  if (st != DSA_OK) return st;
  return from_cuda(launch_wait_selftest(dev_err, stream));
}

int dsa_check_device_error(const int32_t* dev_err, uint32_t* out, dsa_stream_t stream) {
  if (dev_err == nullptr) return DSA_EINVAL;
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, dev_err, 4, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return from_cuda(e);
  if (out) *out = v;
  return v ? DSA_EDEVICE : DSA_OK;
}

int dsa_indexer_k_quant_write(const void* k, int64_t n_tokens, int64_t k_row_stride, const int64_t* slot_mapping,
                              uint8_t* k_cache, int64_t num_blocks, int32_t* dev_err, dsa_stream_t stream) {
  if (n_tokens < 0 || num_blocks < 1 || k_row_stride < kDim || k_row_stride % 8 != 0) return DSA_EINVAL;
  if (n_tokens == 0) return DSA_OK;
  if (!k || !slot_mapping || !k_cache || !aligned16(k) || !aligned16(k_cache)) return DSA_EINVAL;
  int sms;
  int st = device_sms(&sms);
  if (st != DSA_OK) return st;
  return from_cuda(launch_k_quant_write(k, n_tokens, k_row_stride, slot_mapping, k_cache, num_blocks, false,
                                        RopeArgs{}, dev_err, stream));
}

int dsa_indexer_k_quant_write_fp4(const void* k, int64_t n_tokens, int64_t k_row_stride, const int64_t* positions,
                                  const float* cos_sin, int64_t max_pos, const int64_t* slot_mapping,
                                  uint8_t* k_cache, int64_t num_blocks, int32_t* dev_err, dsa_stream_t stream) {
  if (n_tokens < 0 || num_blocks < 1 || k_row_stride < kDim || k_row_stride % 8 != 0) return DSA_EINVAL;
  if (cos_sin != nullptr && (max_pos < 1 || !positions || !aligned16(cos_sin))) return DSA_EINVAL;
  if (n_tokens == 0) return DSA_OK;
  if (!k || !slot_mapping || !k_cache || !aligned16(k) || reinterpret_cast<uintptr_t>(k_cache) % 32 != 0)
    return DSA_EINVAL;
  int sms;
  int st = device_sms(&sms);
  if (st != DSA_OK) return st;
  const RopeArgs rope = cos_sin ? RopeArgs{positions, cos_sin, max_pos} : RopeArgs{};
  return from_cuda(launch_k_quant_write(k, n_tokens, k_row_stride, slot_mapping, k_cache, num_blocks, true, rope,
                                        dev_err, stream));
}

int dsa_indexer_q_quant_fold(const void* q, const float* w, int64_t n_tokens, float softmax_scale, uint8_t* q_fp8,
                             float* q_scale, float* w_folded, dsa_stream_t stream) {
  if (n_tokens < 0) return DSA_EINVAL;
  if (n_tokens == 0) return DSA_OK;
  if (!q || !w || !q_fp8 || !w_folded || !aligned16(q) || !aligned16(q_fp8)) return DSA_EINVAL;
  int sms;
  int st = device_sms(&sms);
  if (st != DSA_OK) return st;
  if (!(softmax_scale > 0.0f)) softmax_scale = 0.08838834764831845f;  // 128^-1/2
  return from_cuda(launch_q_quant_fold(q, w, n_tokens, softmax_scale, q_fp8, q_scale, w_folded, RopeArgs{}, nullptr,
                                       stream));
}

int dsa_gather_rows(const uint8_t* rows, int64_t num_rows, int64_t row_bytes, int64_t row_stride,
                    const int32_t* physical, int64_t n_tokens, int32_t topk, uint8_t* out, int32_t* dev_err,
                    dsa_stream_t stream) {
  if (num_rows < 0 || row_bytes <= 0 || row_bytes % 16 != 0 || row_stride < row_bytes || row_stride % 16 != 0 ||
      n_tokens < 0 || topk < 1)
    return DSA_EINVAL;
  if (n_tokens == 0) return DSA_OK;
  if (!physical || !out || !aligned16(out) || (num_rows > 0 && (!rows || !aligned16(rows)))) return DSA_EINVAL;
  int sms;
  int st = device_sms(&sms);
  if (st != DSA_OK) return st;
  return from_cuda(launch_gather_rows(rows, num_rows, row_bytes, row_stride, physical, n_tokens * topk, out, sms,
                                      dev_err, stream));
}

int dsa_indexer_k_rope_quant_write(const void* k, int64_t n_tokens, int64_t k_row_stride, const int64_t* positions,
                                   const float* cos_sin, int64_t max_pos, const int64_t* slot_mapping,
                                   uint8_t* k_cache, int64_t num_blocks, int32_t* dev_err, dsa_stream_t stream) {
  if (n_tokens < 0 || num_blocks < 1 || k_row_stride < kDim || k_row_stride % 8 != 0 || max_pos < 1) return DSA_EINVAL;
  if (n_tokens == 0) return DSA_OK;
  if (!k || !slot_mapping || !k_cache || !positions || !cos_sin || !aligned16(k) || !aligned16(k_cache) ||
      !aligned16(cos_sin))
    return DSA_EINVAL;
  int sms;
  int st = device_sms(&sms);
  if (st != DSA_OK) return st;
  return from_cuda(launch_k_quant_write(k, n_tokens, k_row_stride, slot_mapping, k_cache, num_blocks, false,
                                        RopeArgs{positions, cos_sin, max_pos}, dev_err, stream));
}

int dsa_indexer_q_rope_quant_fold(const void* q, const float* w, int64_t n_tokens, const int64_t* positions,
                                  const float* cos_sin, int64_t max_pos, float softmax_scale, uint8_t* q_fp8,
                                  float* q_scale, float* w_folded, int32_t* dev_err, dsa_stream_t stream) {
  if (n_tokens < 0 || max_pos < 1) return DSA_EINVAL;
  if (n_tokens == 0) return DSA_OK;
  if (!q || !w || !q_fp8 || !w_folded || !positions || !cos_sin || !aligned16(q) || !aligned16(q_fp8) ||
      !aligned16(cos_sin))
    return DSA_EINVAL;
  int sms;
  int st = device_sms(&sms);
  if (st != DSA_OK) return st;
  if (!(softmax_scale > 0.0f)) softmax_scale = 0.08838834764831845f;  // 128^-1/2
  return from_cuda(launch_q_quant_fold(q, w, n_tokens, softmax_scale, q_fp8, q_scale, w_folded,
                                       RopeArgs{positions, cos_sin, max_pos}, dev_err, stream));
}

size_t dsa_indexer_workspace_size(const DsaBatch* batch, int32_t topk) {
  (void)topk;
  if (check_batch(batch) != DSA_OK) return 0;
  return carve(batch, nullptr).bytes;
}

int dsa_indexer_plan(const DsaBatch* batch, void* ws, size_t ws_bytes, int32_t* dev_err, dsa_stream_t stream) {
  int st = check_batch(batch);
  if (st != DSA_OK) return st;
  if (batch->num_tokens == 0) return DSA_OK;
  if (!ws || !aligned16(ws)) return DSA_EINVAL;
  IndexerWs w = carve(batch, ws);
  if (ws_bytes < w.bytes) return DSA_ENOSPACE;
  int sms;
  if ((st = device_sms(&sms)) != DSA_OK) return st;
  return from_cuda(launch_prologue(plan_only(batch, w, sms, grid_ctas(sms), nullptr, nullptr, nullptr, dev_err), stream));
}

int dsa_set_launch_events(void* const* events, int32_t n_events) {
  if (n_events < 0 || n_events > kMaxTimeline || (n_events > 0 && events == nullptr)) return DSA_EINVAL;
  for (int32_t i = 0; i < n_events; ++i)
    if (events[i] == nullptr) return DSA_EINVAL;
  for (int32_t i = 0; i < n_events; ++i) t_events[i] = static_cast<cudaEvent_t>(events[i]);
  t_count = n_events;
  t_next = 0;
  return DSA_OK;
}
int dsa_indexer_logits(const DsaBatch* batch, const uint8_t* q_fp8, const float* w_folded, const uint8_t* k_cache,
                       float* logits, int64_t logits_ld, void* ws, size_t ws_bytes, int32_t* dev_err,
                       dsa_stream_t stream) {
  int st = check_batch(batch);
  if (st != DSA_OK) return st;
  if (batch->num_tokens == 0) return DSA_OK;
  if (!q_fp8 || !w_folded || !k_cache || !logits || !ws || logits_ld < batch->max_seq_len) return DSA_EINVAL;
  if (!aligned16(q_fp8) || !aligned16(w_folded) || !kcache_aligned(batch, k_cache) || !aligned16(ws)) return DSA_EINVAL;
  IndexerWs w = carve(batch, ws);
  if (ws_bytes < w.bytes) return DSA_ENOSPACE;
  return run_logits(batch, q_fp8, w_folded, k_cache, logits, logits_ld, w, false, dev_err, stream);
}

int dsa_indexer_topk(const DsaBatch* batch, const float* logits, int64_t logits_ld, int32_t topk, int32_t* topk_out,
                     void* ws, size_t ws_bytes, dsa_stream_t stream) {
  (void)ws;
  (void)ws_bytes;
  int st = check_batch(batch);
  if (st != DSA_OK) return st;
  if (!topk_ok(topk)) return DSA_EINVAL;
  if (batch->num_tokens == 0) return DSA_OK;
  if (!logits || !topk_out || logits_ld < 1) return DSA_EINVAL;
  int sms;
  if ((st = device_sms(&sms)) != DSA_OK) return st;
  return from_cuda(launch_topk(logits, logits_ld, batch->query_start_loc, batch->seq_lens,
                               batch->req_id_per_token, batch->num_reqs, 0, batch->num_tokens, topk, topk_out,
                               nullptr, nullptr, 0, stream));
}

int dsa_indexer_logits_topk(const DsaBatch* batch, const uint8_t* q_fp8, const float* w_folded, uint8_t* k_cache,
                            int32_t topk, int32_t* topk_out, void* ws, size_t ws_bytes, const void* k_new,
                            const int64_t* slot_mapping, int32_t* dev_err, dsa_stream_t stream) {
  int st = check_batch(batch);
  if (st != DSA_OK) return st;
  if (!topk_ok(topk)) return DSA_EINVAL;
  if ((k_new == nullptr) != (slot_mapping == nullptr)) return DSA_EINVAL;
  if (batch->num_tokens == 0) return DSA_OK;
  if (!q_fp8 || !w_folded || !k_cache || !topk_out || !ws) return DSA_EINVAL;
  if (!aligned16(q_fp8) || !aligned16(w_folded) || !kcache_aligned(batch, k_cache) || !aligned16(ws) || !aligned16(topk_out))
    return DSA_EINVAL;
  IndexerWs w = carve(batch, ws);
  if (ws_bytes < w.bytes) return DSA_ENOSPACE;
  if (k_new != nullptr && !aligned16(k_new)) return DSA_EINVAL;
  int sms;
  if ((st = device_sms(&sms)) != DSA_OK) return st;
  // one launch: this step's K into the cache (if given), the plan, zeroed histograms
  if ((st = mark(stream)) != DSA_OK) return st;
  st = launched(launch_prologue(plan_only(batch, w, sms, grid_ctas(sms), k_new, slot_mapping, k_cache, dev_err), stream),
                stream);
  if (st != DSA_OK) return st;
  const int64_t ld = logits_ld(batch);
  st = run_logits(batch, q_fp8, w_folded, k_cache, w.logits, ld, w, true, dev_err, stream);
  if (st != DSA_OK) return st;
  return run_topk(batch, w, ld, topk, topk_out, nullptr, sms, false, stream);
}

int dsa_topk_logical_to_physical(const int32_t* logical, int64_t n_tokens, int32_t topk,
                                 const int32_t* req_id_per_token, const int32_t* block_table, int32_t num_reqs,
                                 int64_t bt_stride, int32_t block_stride_rows, int32_t* physical,
                                 int32_t* valid_counts, int32_t* dev_err, dsa_stream_t stream) {
  if (n_tokens < 0 || !topk_ok(topk) || bt_stride < 1 || num_reqs < 0) return DSA_EINVAL;
  if (n_tokens == 0) return DSA_OK;
  if (!logical || !req_id_per_token || !block_table || !physical || !aligned16(logical) || !aligned16(physical))
    return DSA_EINVAL;
  if (n_tokens > 0x7FFFFFFF) return DSA_EINVAL;
  int sms;
  int st = device_sms(&sms);
  if (st != DSA_OK) return st;
  if (block_stride_rows <= 0) block_stride_rows = kBlock;
  return from_cuda(launch_convert(logical, n_tokens, topk, req_id_per_token, block_table, num_reqs, bt_stride,
                                  block_stride_rows, physical, valid_counts, dev_err, stream));
}

int dsa_schedule_build(int32_t n_layers, int32_t use_index_cache, int32_t freq, int32_t offset, const char* pattern,
                       char* fs_out, int32_t* producer_out) {
  if (n_layers < 0 || (n_layers > 0 && (fs_out == nullptr || producer_out == nullptr))) return DSA_EINVAL;
  if (use_index_cache) {
    if (pattern != nullptr) {
      if (static_cast<int64_t>(std::strlen(pattern)) != n_layers) return DSA_EINVAL;
      for (int32_t l = 0; l < n_layers; ++l)
        if (pattern[l] != 'F' && pattern[l] != 'S') return DSA_EINVAL;
      if (n_layers > 0 && pattern[0] != 'F') return DSA_EINVAL;
    } else {
      if (freq < 1) return DSA_EINVAL;
      const int32_t first = 1 - offset > 0 ? 1 - offset : 0;
      if (n_layers > 0 && first % freq != 0) return DSA_EINVAL;
    }
  }
  int32_t producer = 0;
  for (int32_t l = 0; l < n_layers; ++l) {
    bool full = true;
    if (use_index_cache) {
      if (pattern != nullptr) {
        full = pattern[l] == 'F';
      } else {
        const int64_t v = static_cast<int64_t>(l) - offset + 1;
        full = (v > 0 ? v : 0) % freq == 0;
      }
    }
    if (full) producer = l;
    fs_out[l] = full ? 'F' : 'S';
    producer_out[l] = producer;
  }
  return DSA_OK;
}

size_t dsa_layer_stack_workspace_size(const DsaBatch* batch, int32_t topk) {
  if (check_batch(batch) != DSA_OK) return 0;
  const size_t T = static_cast<size_t>(batch->num_tokens);
  size_t bytes = align_up(T * kHeads * kDim, 256) + align_up(T * kHeads * 4, 256);
  return bytes + dsa_indexer_workspace_size(batch, topk);
}

int dsa_layer_stack_decode_sms(const DsaStackPlan* plan, const DsaBatch* batch, int32_t* decode_sms) {
  if (plan == nullptr || decode_sms == nullptr) return DSA_EINVAL;
  int st = check_batch(batch);
  if (st != DSA_OK) return st;
  int sms = 0;
  if ((st = device_sms(&sms)) != DSA_OK) return st;
  *decode_sms = batch->num_tokens > 0 ? decode_split(plan, batch, sms) : 0;
  return DSA_OK;
}

int dsa_layer_stack_run(const DsaStackPlan* plan, const DsaBatch* batch, const int64_t* slot_mapping,
                        int32_t* topk_buf, int32_t* phys_buf, int32_t* valid_buf, dsa_layer_consumer_fn consumer,
                        void* user, void* ws, size_t ws_bytes, int32_t* dev_err, dsa_stream_t stream) {
  int st = check_batch(batch);
  if (st != DSA_OK) return st;
  if (plan == nullptr || plan->n_layers < 0 || (plan->n_layers > 0 && (plan->fs == nullptr || plan->layers == nullptr)))
    return DSA_EINVAL;
  if (!topk_ok(plan->topk)) return DSA_EINVAL;
  if (plan->n_layers > 0 && plan->fs[0] != 'F') return DSA_EINVAL;
  if (plan->rope_cos_sin != nullptr &&
      (plan->positions == nullptr || plan->rope_max_pos < 1 || !aligned16(plan->rope_cos_sin)))
    return DSA_EINVAL;
  for (int32_t l = 0; l < plan->n_layers; ++l) {
    const char c = plan->fs[l];
    if (c != 'F' && c != 'S') return DSA_EINVAL;
    if (c == 'F' && batch->num_tokens > 0) {
      const DsaLayerInputs& L = plan->layers[l];
      if (!L.q || !L.w || !L.k_cache || !aligned16(L.q) || !kcache_aligned(batch, L.k_cache)) return DSA_EINVAL;
      if (L.k_new != nullptr && (slot_mapping == nullptr || !aligned16(L.k_new))) return DSA_EINVAL;
      if (L.w_dtype != DSA_W_FP32 && L.w_dtype != DSA_W_BF16) return DSA_EINVAL;
      const int64_t ks = L.k_row_stride > 0 ? L.k_row_stride : kDim;
      const int64_t wst = L.w_row_stride > 0 ? L.w_row_stride : kHeads;
      if (L.k_row_stride < 0 || ks < kDim || ks % 8 != 0 || L.w_row_stride < 0 || wst < kHeads) return DSA_EINVAL;
      if (reinterpret_cast<uintptr_t>(L.w) % (L.w_dtype == DSA_W_BF16 ? 2 : 4) != 0) return DSA_EINVAL;
    }
  }
  if (batch->num_tokens > 0 && (!topk_buf || !phys_buf || !ws || !aligned16(ws))) return DSA_EINVAL;
  if (ws_bytes < dsa_layer_stack_workspace_size(batch, plan->topk)) return DSA_ENOSPACE;
  const size_t T = static_cast<size_t>(batch->num_tokens);
  uint8_t* q8 = static_cast<uint8_t*>(ws);
  float* wf = reinterpret_cast<float*>(q8 + align_up(T * kHeads * kDim, 256));
  void* iws = reinterpret_cast<uint8_t*>(wf) + align_up(T * kHeads * 4, 256);
  IndexerWs w = carve(batch, iws);
  const int64_t ld = logits_ld(batch);
  int sms = 0;
  if (batch->num_tokens > 0 && (st = device_sms(&sms)) != DSA_OK) return st;
  const float softmax_scale = plan->softmax_scale > 0.0f ? plan->softmax_scale : 0.08838834764831845f;
  // decode and prefill scores side by side on split SMs, when the caller gave the work
  const int split = batch->num_tokens > 0 ? decode_split(plan, batch, sms) : 0;
  bool planned = false;
  int32_t producer = 0;
  for (int32_t l = 0; l < plan->n_layers; ++l) {
    if (plan->fs[l] == 'F') {
      producer = l;
      if (batch->num_tokens > 0) {
        const DsaLayerInputs& L = plan->layers[l];
        // one launch: this layer's K into its cache, q quant + weight fold, and
        // (first F layer only: the batch layout is the same for every layer) the
        // prefill plan
        // (histograms and counters of the decode rows zeroed for this layer's top-k)
        PrologueArgs pa = plan_only(batch, w, sms, split > 0 ? sms - split : grid_ctas(sms), L.k_new, slot_mapping,
                                    L.k_cache, dev_err);
        pa.q = static_cast<const __nv_bfloat16*>(L.q);
        pa.w = L.w;
        pa.w_bf16 = L.w_dtype == DSA_W_BF16;
        pa.w_row_stride = L.w_row_stride > 0 ? L.w_row_stride : kHeads;
        pa.k_row_stride = L.k_row_stride > 0 ? L.k_row_stride : kDim;
        pa.softmax_scale = softmax_scale;
        pa.rope = RopeArgs{plan->positions, plan->rope_cos_sin, plan->rope_max_pos};
        pa.q_fp8 = q8;
        pa.w_folded = wf;
        pa.plan = pa.plan && !planned;
        pa.pdl = planned && consumer == nullptr;  // the previous kernel is then this library's top-k
        if ((st = mark(stream)) != DSA_OK) return st;
        st = launched(launch_prologue(pa, stream), stream);
        if (st != DSA_OK) return st;
        planned = true;
        // S3 with S5 fused into its output pass: logical ids, physical ids, valid counts
        TopkPhys tp{batch->block_table, batch->bt_stride,
                    plan->block_stride_rows > 0 ? plan->block_stride_rows : kBlock, phys_buf, valid_buf, dev_err};
        if (split > 0) {
          st = run_split(batch, q8, wf, L.k_cache, w, ld, plan->topk, topk_buf, &tp, sms, split, dev_err, stream);
        } else {
          st = run_logits(batch, q8, wf, L.k_cache, w.logits, ld, w, true, dev_err, stream);
          if (st == DSA_OK) st = run_topk(batch, w, ld, plan->topk, topk_buf, &tp, sms, true, stream);
        }
        if (st != DSA_OK) return st;
      }
    }
    if (consumer != nullptr) consumer(l, producer, phys_buf, valid_buf, user);
  }
  return DSA_OK;
}

}  // extern "C"
