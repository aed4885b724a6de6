// topk.cu — S3: per-row top-k of the indexer scores (sm_103a), optionally
// fused with S5 (logical -> physical ids).
//
// "IndexCache：DeepSeek 稀疏注意力中的跨层索引复用" (atomage.cn): the indexer op
// resets the rows of the shared `topk_indices_buffer` to -1 and fills each
// row with the ids of the `index_topk` highest-scoring keys. A row with fewer
// visible keys than k keeps -1 in the tail. "vllm.v1.attention.backends.mla.
// index_group" (`_convert_once`): the consumers want physical slots,
// block_table[req][id/64] * block_stride_rows + id%64, and the count of valid
// ids per row; when asked, each selected id is converted as it is written.
//
// Both kernels are exact radix selects (select.cuh); ids are emitted in no
// particular order.
//  * topk_kernel: one CTA per row. Pass 1 comes from the histogram the score
//    kernel built when there is one (decode rows), else from the row. Rows
//    that fit the launch's staging area are staged once in shared memory;
//    longer rows are re-read from L2. Prefill rows run in 256-thread CTAs,
//    several per SM; decode rows of up to 32768 scores in 1024-thread CTAs.
//  * select_kernel + resolve_kernel: decode rows longer than that. Several
//    CTAs per row place the keys above the boundary bin and collect the
//    boundary bin's keys with their next-level histogram; a second launch,
//    one CTA per row, resolves the boundary bin on those candidates only.
#include "select.cuh"

namespace dsa {

constexpr int kRowThreads = 256;  // topk_kernel: small CTAs, so that several rows run per SM
// Boundary-bin keys a staged row gathers (a larger bin takes the exact
// fallback over the row). With k = 2048 and rows of 8192 keys a CTA then
// needs 55 KB of shared memory, and four run per SM.
constexpr int kStagedCandCap = 768;

// Visible keys of row t (clipped to ld); *req = its request.
__device__ __forceinline__ int row_length(int t, const int32_t* qsl, const int32_t* seq_lens, const int32_t* req_id,
                                          int num_reqs, int64_t ld, int* req) {
  const int r = __ldg(req_id + t);
  *req = r;
  if (r < 0 || r >= num_reqs) return 0;
  const int q0 = __ldg(qsl + r), ql = __ldg(qsl + r + 1) - q0;
  int n = __ldg(seq_lens + r) - ql + (t - q0) + 1;
  n = n < 0 ? 0 : n;
  return n > ld ? static_cast<int>(ld) : n;
}

struct PhysOut {
  const int32_t* block_table;  // nullptr: logical ids only
  int64_t bt_stride;
  int stride_rows;
  int32_t* physical;
  int32_t* valid_counts;
  int32_t* err;
};

PhysOut phys_out(const TopkPhys* phys) {
  PhysOut po{};
  if (phys != nullptr) {
    po.block_table = phys->block_table;
    po.bt_stride = phys->bt_stride;
    po.stride_rows = phys->stride_rows;
    po.physical = phys->physical;
    po.valid_counts = phys->valid_counts;
    po.err = phys->err;
  }
  return po;
}

// Output of row t (request r): logical ids, and physical slots when asked.
__device__ __forceinline__ RowOut row_out(const PhysOut& po, int32_t* out, int topk, int t, int r, int num_reqs) {
  RowOut o;
  o.orow = out + static_cast<int64_t>(t) * topk;
  const bool phys = po.block_table != nullptr && r >= 0 && r < num_reqs;
  o.prow = phys ? po.physical + static_cast<int64_t>(t) * topk : nullptr;
  o.bt_row = phys ? po.block_table + static_cast<int64_t>(r) * po.bt_stride : nullptr;
  o.bt_stride = po.bt_stride;
  o.stride_rows = po.stride_rows;
  return o;
}

// Shapes of the per-row top-k: 256-thread CTAs, several per SM, for the many
// rows of a prefill; 1024-thread CTAs, one per SM, that stage rows of up to
// 32768 scores, for the few long rows of a decode batch.
template <int NT>
struct RowCfg {
  static constexpr int kStageMax = NT == 1024 ? 32768 : kTopkRowCap;  // scores staged per row, at most
  static constexpr int kCand = NT == 1024 ? 4096 : kStagedCandCap;    // boundary-bin candidates staged
  static constexpr int kLoads = NT == 1024 ? 8 : 12;                  // float4 loads in flight per thread
};

// One CTA per row (rows row_begin + blockIdx.x). Shared memory, sized by the
// launch: the histogram, kCand boundary-bin candidates (keys, ids), the row's
// ids (topk, rounded up to 4) and a staging area of stage_cap keys. A row of
// at most stage_cap keys is staged there once; a longer row is re-read from
// L2 and the staging area holds up to stage_cap / 2 candidates instead. The
// choice is made per row, so the short prefill rows of a batch whose score
// rows are long (decode requests at long context) still stage.
template <int NT>
__global__ void __launch_bounds__(NT, NT == 1024 ? 1 : 4) topk_kernel(const float* __restrict__ logits, int64_t ld,
                                                                      const int32_t* qsl, const int32_t* seq_lens,
                                                                      const int32_t* req_id, int num_reqs,
                                                                      int row_begin, int topk,
                                                                      int32_t* __restrict__ out, PhysOut po,
                                                                      const uint32_t* hist_g, int hist_rows,
                                                                      int stage_cap) {
  using R = RowCfg<NT>;
  extern __shared__ __align__(16) uint32_t sh[];
  uint32_t* hist = sh;
  uint32_t* oid = sh + kSelBins + 2 * R::kCand;
  uint32_t* keys = oid + ((topk + 3) & ~3);
  __shared__ SelState s;
  __shared__ int32_t bts[R::kStageMax / kBlock];

  // rows in reverse: within a request the later tokens see more keys, so the
  // longest rows are placed first and the short ones fill the tail (prefill4x8k
  // top-k 565 -> 546 us). The request metadata and the block table are inputs
  // of the step: read them while the score kernel may still run.
  const int t = row_begin + static_cast<int>(gridDim.x - 1 - blockIdx.x);
  const int tid = threadIdx.x;
  int r;
  const int n = row_length(t, qsl, seq_lens, req_id, num_reqs, ld, &r);
  const bool staged = n <= stage_cap;
  RowOut o = row_out(po, out, topk, t, r, num_reqs);
  // a staged row's block-table row, for emit: one entry per thread, loaded
  // into a register here and stored to shared memory after the staging loads,
  // so that its latency overlaps theirs (prefill4x8k top-k 427 -> 417 us)
  static_assert(R::kStageMax / kBlock <= NT, "one block-table entry per thread");
  const int cap = po.bt_stride < R::kStageMax / kBlock ? static_cast<int>(po.bt_stride) : R::kStageMax / kBlock;
  const int pages = staged && o.prow != nullptr && n > topk ? min((n + kBlock - 1) / kBlock, cap) : 0;
  const int32_t bt_page = tid < pages ? __ldg(o.bt_row + tid) : -1;
  if (pages > 0) o.bt_row = bts;
  pdl_wait();  // the scores come from the previous kernel
  pdl_launch_dependents();
  bool bad = false;
  if (o.prow != nullptr && po.valid_counts != nullptr && tid == 0) po.valid_counts[t] = n < topk ? n : topk;
  if (n <= topk) {
    write_short_row(n, topk, o, &bad);
    if (bad) flag_error(po.err, DSA_DEVERR_ID_RANGE);
    return;
  }
  const float* lrow = logits + static_cast<int64_t>(t) * ld;
  const bool have_hist = hist_g != nullptr && t < hist_rows;
  if (have_hist) {
    const uint4* hrow = reinterpret_cast<const uint4*>(hist_g + static_cast<int64_t>(t) * kSelBins);
    for (int b = tid; b < kSelBins / 4; b += NT) reinterpret_cast<uint4*>(hist)[b] = __ldcg(hrow + b);
  } else {
    for (int b = tid; b < kSelBins / 4; b += NT) reinterpret_cast<uint4*>(hist)[b] = make_uint4(0, 0, 0, 0);
  }
  // rows are 16-byte aligned (ld is a multiple of 4): float4 loads, several in flight per thread
  const float4* l4 = reinterpret_cast<const float4*>(lrow);
  const int n4 = (n + 3) >> 2;
  if (staged) {
    select_staged_init<NT>(oid, topk, s);
    if (!have_hist) __syncthreads();  // the zeroed histogram, before the staging pass counts into it
    constexpr int U = R::kLoads;
    for (int base = 0; base < n4; base += U * NT) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i4 = base + u * NT + tid;
        v[u] = i4 < n4 ? __ldcg(l4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i4 = base + u * NT + tid;
        if (i4 < n4) {
          const uint4 k = make_uint4(f32_key(v[u].x), f32_key(v[u].y), f32_key(v[u].z), f32_key(v[u].w));
          reinterpret_cast<uint4*>(keys)[i4] = k;
          if (!have_hist) {  // pass 1 while staging: the row's keys below n
            const int i = 4 * i4;
            atomicAdd(&hist[k.x >> kHistShift], 1u);
            if (i + 1 < n) atomicAdd(&hist[k.y >> kHistShift], 1u);
            if (i + 2 < n) atomicAdd(&hist[k.z >> kHistShift], 1u);
            if (i + 3 < n) atomicAdd(&hist[k.w >> kHistShift], 1u);
          }
        }
      }
    }
    if (tid < pages) bts[tid] = bt_page;
    __syncthreads();
    select_row_staged<NT>(keys, n, hist, sh + kSelBins, sh + kSelBins + R::kCand, oid, topk, R::kCand, o, s, &bad);
  } else if constexpr (NT <= 512) {  // (the 1024-thread launch stages every row: stage_cap >= ld)
    __syncthreads();
    if (!have_hist) {  // pass 1 from L2, eight float4 loads in flight per thread
      for (int base = 0; base < n4; base += 8 * NT) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i4 = base + u * NT + tid;
          v[u] = i4 < n4 ? __ldcg(l4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = 4 * (base + u * NT + tid);
          if (i < n) atomicAdd(&hist[f32_key(v[u].x) >> kHistShift], 1u);
          if (i + 1 < n) atomicAdd(&hist[f32_key(v[u].y) >> kHistShift], 1u);
          if (i + 2 < n) atomicAdd(&hist[f32_key(v[u].z) >> kHistShift], 1u);
          if (i + 3 < n) atomicAdd(&hist[f32_key(v[u].w) >> kHistShift], 1u);
        }
      }
      __syncthreads();
    }
    // the staging area holds the boundary bin's candidates instead
    const int cap = stage_cap / 2;
    select_row<NT>([&](int i) -> uint32_t { return f32_key(__ldcg(lrow + i)); }, n, hist, keys, keys + cap, oid,
                   topk, static_cast<uint32_t>(cap), o, s, &bad);
  }
  if (bad) flag_error(po.err, DSA_DEVERR_ID_RANGE);
}

// Keys staged per row by the 256-thread launch: the whole row when the score
// rows fit kTopkRowCap, else 8192 (four CTAs per SM at k = 2048); longer rows
// are re-read from L2.
constexpr int kLongRowStage = 8192;

template <int NT>
static cudaError_t launch_topk_rows(const float* logits, int64_t ld, const int32_t* qsl, const int32_t* seq_lens,
                                    const int32_t* req_id, int num_reqs, int row_begin, int n_tokens, int topk,
                                    int32_t* out, const TopkPhys* phys, const uint32_t* hist, int hist_rows,
                                    int stage_cap, cudaStream_t stream) {
  using R = RowCfg<NT>;
  const int rows = n_tokens - row_begin;
  if (rows <= 0) return cudaSuccess;
  const int ids = (topk + 3) & ~3;
  const int smem = (kSelBins + 2 * R::kCand + ids + stage_cap) * 4;
  static uint64_t configured = 0;  // the largest layout: k = kMaxTopk, stage_cap = kStageMax
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(topk_kernel<NT>),
                                   (kSelBins + 2 * R::kCand + kMaxTopk + R::kStageMax) * 4, &configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(topk_kernel<NT>, dim3(rows), dim3(NT), smem, stream, logits, ld, qsl, seq_lens, req_id, num_reqs,
                    row_begin, topk, out, phys_out(phys), hist, hist_rows, stage_cap);
}

cudaError_t launch_topk(const float* logits, int64_t ld, const int32_t* qsl, const int32_t* seq_lens,
                        const int32_t* req_id, int num_reqs, int row_begin, int n_tokens, int topk, int32_t* out,
                        const TopkPhys* phys, const uint32_t* hist, int hist_rows, cudaStream_t stream) {
  const int stage_cap = ld <= kTopkRowCap ? static_cast<int>((ld + 3) & ~3) : kLongRowStage;
  return launch_topk_rows<kRowThreads>(logits, ld, qsl, seq_lens, req_id, num_reqs, row_begin, n_tokens, topk, out,
                                       phys, hist, hist_rows, stage_cap, stream);
}

// ---------------------------------------------------------------------------
// Decode rows longer than one CTA stages: two launches. select_kernel: CTA
// (c, t) takes scores [c*chunk, (c+1)*chunk) of row t. Pass 1 is the score
// kernel's histogram of the row, so every chunk knows the boundary bin b1 at
// once: it places its keys above b1 (one global reservation per CTA), appends
// its b1 keys to the row's candidate list (another), and adds their next 11
// bits to the row's second-level histogram. resolve_kernel, one CTA per row,
// then finds the k-th key from that histogram (and, when its sub-bin is not
// taken whole, a third level over the sub-bin's candidates) and places the
// boundary keys. The kernel boundary replaces a completion counter and the
// row's last CTA resolving on its own.
// 1024 threads: the chain of dependent loads, scans and reservations is
// latency-bound, and more threads per CTA keep more of each chunk's loads in
// flight (decode8x128k step 49.8 us at 512, 47.3 at 1024, 56.1 at 256).
constexpr int kSelectThreads = 1024;

__global__ void __launch_bounds__(kSelectThreads) select_kernel(SelectArgs a, PhysOut po, int chunk) {
  extern __shared__ __align__(16) uint32_t sh[];
  uint32_t* hist = sh;              // kSelBins: pass 1, then this chunk's second-level histogram
  uint32_t* keys = sh + kSelBins;   // chunk: the chunk's keys
  uint32_t* ids = keys + chunk;     // chunk: its ids above the boundary bin, in order
  __shared__ SelState s;
  __shared__ uint32_t s_base_up, s_base_eq;
  __shared__ int32_t sbt[8192 / kBlock];  // the chunk's block-table entries (chunk <= 8192)

  const int t = blockIdx.y;
  const int c = blockIdx.x;
  const int tid = threadIdx.x;
  int r;
  const int n = row_length(t, a.qsl, a.seq_lens, a.req_id, a.num_reqs, a.ld, &r);  // inputs of the step
  const RowOut o = row_out(po, a.out, a.topk, t, r, a.num_reqs);
  // the chunk's pages of the request's block-table row, for its ids' physical
  // slots: loaded into a register now, stored beside the keys (decode8x128k
  // step 45.4 -> 44.7 us against a global load per emitted id)
  const int p0 = c * chunk / kBlock;
  const int npg = chunk / kBlock;
  const int32_t bt_page =
      o.prow != nullptr && tid < npg ? (p0 + tid < o.bt_stride ? __ldg(o.bt_row + p0 + tid) : -1) : -1;
  pdl_wait();  // the scores come from the previous kernel
  pdl_launch_dependents();
  const int chunks = n > 0 ? (n + chunk - 1) / chunk : 1;
  if (c >= chunks) return;
  bool bad = false;
  if (n <= a.topk) {
    if (c == 0) {
      if (o.prow != nullptr && po.valid_counts != nullptr && tid == 0) po.valid_counts[t] = n;
      write_short_row(n, a.topk, o, &bad);
      if (bad) flag_error(po.err, DSA_DEVERR_ID_RANGE);
    }
    return;
  }
  if (c == 0 && o.prow != nullptr && po.valid_counts != nullptr && tid == 0) po.valid_counts[t] = a.topk;
  uint32_t* cnt = a.counters + static_cast<int64_t>(t) * kRowCounters;
  uint2* crow = a.cand + static_cast<int64_t>(t) * a.ld;
  const int lo = c * chunk;
  const int len = min(n, lo + chunk) - lo;

  // the row's histogram and the chunk's keys, loads issued together
  const uint4* hrow = reinterpret_cast<const uint4*>(a.hist + static_cast<int64_t>(t) * kSelBins);
  for (int b = tid; b < kSelBins / 4; b += kSelectThreads) reinterpret_cast<uint4*>(hist)[b] = __ldcg(hrow + b);
  {
    const float4* l4 = reinterpret_cast<const float4*>(a.logits + static_cast<int64_t>(t) * a.ld + lo);
    const int n4 = (len + 3) >> 2;  // lo and ld are multiples of 4
    for (int base = 0; base < n4; base += 4 * kSelectThreads) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i4 = base + u * kSelectThreads + tid;
        v[u] = i4 < n4 ? __ldcg(l4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i4 = base + u * kSelectThreads + tid;
        if (i4 < n4) reinterpret_cast<uint4*>(keys)[i4] =
            make_uint4(f32_key(v[u].x), f32_key(v[u].y), f32_key(v[u].z), f32_key(v[u].w));
      }
    }
  }
  if (tid == 0) {  // defaults if the histogram were inconsistent with the row
    s.bin = 0;
    s.above = 0;
  }
  if (tid < npg) sbt[tid] = bt_page;
  __syncthreads();
  find_bin<kSelectThreads>(hist, static_cast<uint32_t>(a.topk), s);
  const uint32_t b1 = static_cast<uint32_t>(s.bin);
  if (c == 0 && tid == 0) {  // the boundary for the resolving launch
    cnt[2] = b1;
    cnt[3] = s.above;
  }
  // pass 1 is read (find_bin ends with a barrier): the array takes this
  // chunk's second-level histogram
  for (int b = tid; b < kSelBins; b += kSelectThreads) hist[b] = 0;

  // thread ranges of 4*q keys (q odd), one packed scan for the offsets
  int q4 = ((len + kSelectThreads - 1) / kSelectThreads + 3) >> 2;
  q4 += (q4 & 1) ^ 1;
  const int tl = tid * 4 * q4, th = min(len, tl + 4 * q4);
  const uint4* k4 = reinterpret_cast<const uint4*>(keys);
  int c_up = 0, c_eq = 0;
  for (int i = tl; i < th; i += 4) {
    const uint4 v = k4[i >> 2];
    const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t bin = kk[u] >> kHistShift;
      const bool in = i + u < th;
      c_up += in && bin > b1;
      c_eq += in && bin == b1;
    }
  }
  uint32_t total;  // counts <= chunk <= 8192
  const uint32_t excl =
      block_excl_sum<kSelectThreads>((static_cast<uint32_t>(c_up) << 16) | static_cast<uint32_t>(c_eq), s.sm, &total);
  const uint32_t total_up = total >> 16, total_eq = total & 0xffffu;
  if (tid == 0) {
    s_base_up = total_up ? atomicAdd(&cnt[0], total_up) : 0;
    s_base_eq = total_eq ? atomicAdd(&cnt[1], total_eq) : 0;
  }
  uint32_t p_up = excl >> 16, p_eq = excl & 0xffffu;
  __syncthreads();
  const uint32_t base_eq = s_base_eq;
  for (int i = tl; i < th; i += 4) {
    const uint4 v = k4[i >> 2];
    const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t bin = kk[u] >> kHistShift;
      if (i + u < th) {
        if (bin > b1) {
          ids[p_up++] = static_cast<uint32_t>(lo + i + u);
        } else if (bin == b1) {
          atomicAdd(&hist[(kk[u] >> 10) & (kSelBins - 1)], 1u);
          if (base_eq + p_eq < static_cast<uint32_t>(a.ld))
            crow[base_eq + p_eq] = make_uint2(kk[u], static_cast<uint32_t>(lo + i + u));
          ++p_eq;
        }
      }
    }
  }
  __syncthreads();
  // this chunk's ids above the bin, coalesced, at its reserved positions of the
  // row; its second-level counts added to the row's
  const uint32_t base_up = s_base_up;
  for (uint32_t j = tid; j < total_up; j += kSelectThreads) {
    const uint32_t pos = base_up + j;
    if (pos >= static_cast<uint32_t>(a.topk)) continue;
    const int id = static_cast<int>(ids[j]);
    o.orow[pos] = id;
    if (o.prow != nullptr) {  // the id's page lies in this chunk: [p0, p0 + npg)
      const int32_t blk = sbt[id / kBlock - p0];
      if (blk < 0) bad = true;
      o.prow[pos] = blk < 0 ? -1 : blk * o.stride_rows + id % kBlock;
    }
  }
  if (total_eq > 0) {
    uint32_t* h2 = a.hist2 + static_cast<int64_t>(t) * kSelBins;
    for (int b = tid; b < kSelBins; b += kSelectThreads)
      if (hist[b]) atomicAdd(h2 + b, hist[b]);
  }
  if (bad) flag_error(po.err, DSA_DEVERR_ID_RANGE);
}

// One CTA per long decode row: the boundary keys, from the candidates and the
// second-level histogram the chunk CTAs left. The row's candidates are staged
// in shared memory when they fit (kCandCap), else read from the list.
constexpr int kResolveBt = 2048;  // block-table entries a resolving CTA stages

__global__ void __launch_bounds__(kSelectThreads) resolve_kernel(SelectArgs a, PhysOut po) {
  __shared__ __align__(16) uint32_t hist[kSelBins];
  __shared__ uint2 cands[kCandCap];
  __shared__ SelState s;
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  int r;
  const int n = row_length(t, a.qsl, a.seq_lens, a.req_id, a.num_reqs, a.ld, &r);
  RowOut o = row_out(po, a.out, a.topk, t, r, a.num_reqs);
  // the row's block-table entries, for its ids' physical slots, staged while
  // the chunk CTAs run when they fit (rows of up to 131072 keys; decode8x128k
  // step 44.9 -> 44.2 us)
  extern __shared__ int32_t rbt[];
  const int pages = (n + kBlock - 1) / kBlock;
  if (o.prow != nullptr && n > a.topk && pages <= kResolveBt) {
    for (int p = tid; p < pages; p += kSelectThreads) rbt[p] = p < o.bt_stride ? __ldg(o.bt_row + p) : -1;
    o.bt_row = rbt;
  }
  pdl_wait();  // the chunk CTAs' placements, candidates and counts
  pdl_launch_dependents();
  if (n <= a.topk) return;  // written whole by the row's first chunk
  bool bad = false;
  const uint32_t* cnt = a.counters + static_cast<int64_t>(t) * kRowCounters;
  const uint2* crow = a.cand + static_cast<int64_t>(t) * a.ld;
  const uint32_t b1 = __ldcg(cnt + 2), above = __ldcg(cnt + 3);
  const uint32_t m = min(__ldcg(cnt + 1), static_cast<uint32_t>(a.ld));
  const uint32_t need = static_cast<uint32_t>(a.topk) - above;  // 1 <= need <= m
  const bool staged = m <= static_cast<uint32_t>(kCandCap);
  const uint4* h2 = reinterpret_cast<const uint4*>(a.hist2 + static_cast<int64_t>(t) * kSelBins);
  for (int b = tid; b < kSelBins / 4; b += kSelectThreads) reinterpret_cast<uint4*>(hist)[b] = __ldcg(h2 + b);
  if (staged)
    for (uint32_t j = tid; j < m; j += kSelectThreads) cands[j] = __ldcg(crow + j);
  if (tid == 0) {
    s.bin = 0;
    s.above = 0;
    s.cnt = above;
    s.eq = 0;
  }
  __syncthreads();
  auto cand_at = [&](uint32_t j) -> uint2 { return staged ? cands[j] : __ldcg(crow + j); };
  // take every candidate (level 1), every candidate whose next 11 bits are
  // >= b2 (level 2), or every candidate above T and need3 equal to T (level 3)
  int level = 1;
  uint32_t lo2 = 0, T = 0, need3 = 0;
  if (m != need) {
    find_bin<kSelectThreads>(hist, need, s);
    const uint32_t b2 = static_cast<uint32_t>(s.bin);
    const uint32_t need2 = need - s.above;
    const uint32_t p2 = (b1 << 11) | b2;  // the top 22 bits of the k-th key
    lo2 = p2 << 10;
    level = 2;
    if (hist[b2] != need2) {
      __syncthreads();
      for (int b = tid; b < kSelBins; b += kSelectThreads) hist[b] = 0;
      if (tid == 0) {
        s.bin = 0;
        s.above = 0;
      }
      __syncthreads();
      for (uint32_t j = tid; j < m; j += kSelectThreads) {
        const uint32_t k = cand_at(j).x;
        if ((k >> 10) == p2) atomicAdd(&hist[k & 1023u], 1u);
      }
      __syncthreads();
      find_bin<kSelectThreads>(hist, need2, s);
      T = lo2 | static_cast<uint32_t>(s.bin);
      need3 = need2 - s.above;
      level = 3;
    }
  }
  for (uint32_t j0 = 0; j0 < m; j0 += kSelectThreads) {
    const uint32_t j = j0 + tid;
    const uint2 kv = j < m ? cand_at(j) : make_uint2(0u, 0u);
    const bool in = j < m && (kv.x >> kHistShift) == b1;
    const bool up = in && (level == 1 || (level == 2 ? kv.x >= lo2 : kv.x > T));
    const bool tie = in && level == 3 && kv.x == T;
    const uint32_t tq = warp_reserve(tie, &s.eq);
    const bool take = up || (tie && tq < need3);
    const uint32_t pos = warp_reserve(take, &s.cnt);
    if (take && pos < static_cast<uint32_t>(a.topk)) emit(o, pos, static_cast<int>(kv.y), &bad);
  }
  if (bad) flag_error(po.err, DSA_DEVERR_ID_RANGE);
}

cudaError_t launch_select(const SelectArgs& a, const TopkPhys* phys, int num_sms, cudaStream_t stream) {
  if (a.n_rows <= 0) return cudaSuccess;
  // rows of up to 32768 scores: one 1024-thread CTA per row stages the whole
  // row; cross-CTA exchanges (global reservations, or a thread-block cluster's
  // distributed shared memory) measured slower for these (decode32 step 27.6
  // and 24.6 against 22.7 us)
  if (a.ld <= RowCfg<1024>::kStageMax)
    return launch_topk_rows<1024>(a.logits, a.ld, a.qsl, a.seq_lens, a.req_id, a.num_reqs, 0, a.n_rows, a.topk, a.out,
                                  phys, a.hist, a.n_rows, static_cast<int>((a.ld + 3) & ~3), stream);
  // longer rows: chunks of the row in independent CTAs, then one CTA per row
  // for the boundary; chunks of 1024..8192 scores, the smallest that keeps
  // every row's chunks within about two CTAs per SM
  int chunk = 1024;
  while (chunk < 8192 && static_cast<int64_t>(a.n_rows) * a.ld / chunk > 2 * static_cast<int64_t>(num_sms)) chunk *= 2;
  const int max_smem = (kSelBins + 2 * 8192) * 4;
  static uint64_t configured = 0;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(select_kernel), max_smem, &configured);
  if (e != cudaSuccess) return e;
  const int64_t chunks = (a.ld + chunk - 1) / chunk;
  dim3 grid(static_cast<unsigned>(chunks < 1 ? 1 : chunks), static_cast<unsigned>(a.n_rows));
  const PhysOut po = phys_out(phys);
  e = launch_pdl(select_kernel, grid, dim3(kSelectThreads), (kSelBins + 2 * chunk) * 4, stream, a, po, chunk);
  if (e != cudaSuccess) return e;
  static uint64_t configured_res = 0;
  e = raise_smem_limit(reinterpret_cast<const void*>(resolve_kernel), kResolveBt * 4, &configured_res);
  if (e != cudaSuccess) return e;
  return launch_pdl(resolve_kernel, dim3(a.n_rows), dim3(kSelectThreads), kResolveBt * 4, stream, a, po);
}

}  // namespace dsa
