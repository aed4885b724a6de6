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
// Both kernels are exact radix selects over order-preserving 32-bit keys of
// the fp32 scores (a > b iff key(a) > key(b)); ids are emitted in no
// particular order.
//  * topk_kernel: one CTA per row; up to three histogram rounds (11, 11 and
//    10 bits) narrow down the k-th largest key, then one pass emits every key
//    above it and as many equal keys as are still needed. Rows that fit are
//    staged once in shared memory; longer rows are re-read from L2.
//  * select_kernel: decode rows, whose first-round histogram (top 11 bits)
//    the score kernel already accumulated. Several CTAs per row emit the keys
//    above the boundary bin and collect the boundary bin's keys; the last CTA
//    of the row to finish resolves the boundary bin with the two remaining
//    rounds on those candidates only.
#include "common.cuh"
#include "kernels.h"

namespace dsa {

constexpr int kTopkThreads = 512;
constexpr int kBins = 2048;
constexpr int kSelectChunk = 8192;  // scores per select CTA
static_assert(kBins == kHistBins, "first-round histogram width");

__device__ __forceinline__ int row_length(int t, const int32_t* qsl, const int32_t* seq_lens, const int32_t* req_id,
                                          int num_reqs, int64_t ld, int* req) {
  const int r = req_id[t];
  *req = r;
  if (r < 0 || r >= num_reqs) return 0;
  const int q0 = qsl[r], ql = qsl[r + 1] - q0;
  int n = seq_lens[r] - ql + (t - q0) + 1;
  n = n < 0 ? 0 : n;
  return n > ld ? static_cast<int>(ld) : n;
}

// Bin b, scanning from the top, at which the count reaches `need`; *above = count in bins > b.
__device__ void find_bin(const uint32_t* hist, uint32_t need, int* s_bin, uint32_t* s_above, uint32_t* sm) {
  constexpr int kPer = kBins / kTopkThreads;  // 4 bins per thread
  const int tid = threadIdx.x;
  const int lane = tid & 31, wid = tid >> 5;
  // thread i owns bins [kBins - kPer*(i+1), kBins - kPer*i): thread 0 holds the top bins
  const int hi = kBins - kPer * tid;
  uint32_t local = 0;
#pragma unroll
  for (int b = 0; b < kPer; ++b) local += hist[hi - 1 - b];
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sm[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    uint32_t x = lane < kTopkThreads / 32 ? sm[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t v = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += v;
    }
    if (lane < kTopkThreads / 32) sm[lane] = x;
  }
  __syncthreads();
  incl += wid > 0 ? sm[wid - 1] : 0;
  uint32_t above = incl - local;
  if (above < need && need <= incl) {
    for (int b = 0; b < kPer; ++b) {
      const uint32_t c = hist[hi - 1 - b];
      if (above + c >= need) {
        *s_bin = hi - 1 - b;
        *s_above = above;
        break;
      }
      above += c;
    }
  }
  __syncthreads();
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

__device__ __forceinline__ void emit(int32_t* orow, int32_t* prow, const int32_t* bt_row, int64_t bt_stride,
                                     int stride_rows, uint32_t pos, int id, bool* bad) {
  orow[pos] = id;
  if (prow != nullptr) {
    const int64_t page = id / kBlock;
    const int32_t blk = page < bt_stride ? bt_row[page] : -1;  // global, or the row staged in shared memory
    if (blk < 0) *bad = true;
    prow[pos] = blk < 0 ? -1 : blk * stride_rows + id % kBlock;
  }
}

// Rows with at most k keys: every key, then -1.
__device__ void write_short_row(int n, int topk, int32_t* orow, int32_t* prow, const int32_t* bt_row,
                                const PhysOut& po, bool* bad) {
  for (int i = threadIdx.x; i < topk; i += blockDim.x) {
    if (i < n) {
      emit(orow, prow, bt_row, po.bt_stride, po.stride_rows, i, i, bad);
    } else {
      orow[i] = -1;
      if (prow != nullptr) prow[i] = -1;
    }
  }
}

// Warp-aggregated slot reservation: lanes with `take` get consecutive slots of *ctr.
__device__ __forceinline__ uint32_t warp_reserve(bool take, uint32_t* ctr) {
  const unsigned mask = __ballot_sync(0xffffffffu, take);
  if (mask == 0) return 0;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(mask) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(ctr, static_cast<uint32_t>(__popc(mask)));
  base = __shfl_sync(0xffffffffu, base, leader);
  return base + static_cast<uint32_t>(__popc(mask & ((1u << lane) - 1u)));
}

constexpr int kCandCap = 4096;  // boundary-bin keys gathered in shared memory

// One CTA per row. Round 1 (top 11 bits) comes from the histogram the score
// kernel built when there is one, else from the row. One pass then emits
// every key above the boundary bin and gathers the boundary bin's keys; the
// remaining two rounds and the final choice run on those keys only (or, if
// the bin holds more than kCandCap keys, on the row filtered to the bin).
template <bool kStaged>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ logits, int64_t ld,
                                                            const int32_t* qsl, const int32_t* seq_lens,
                                                            const int32_t* req_id, int num_reqs, int row_begin,
                                                            int topk, int32_t* __restrict__ out, PhysOut po,
                                                            const uint32_t* hist_g, int hist_rows) {
  extern __shared__ uint32_t sh[];
  uint32_t* hist = sh;
  uint32_t* ckey = sh + kBins;
  uint32_t* cidx = ckey + kCandCap;
  uint32_t* keys = cidx + kCandCap;
  __shared__ uint32_t sm[32];
  __shared__ int s_bin;
  __shared__ uint32_t s_above, s_cnt, s_eq;
  __shared__ int32_t bts[kTopkRowCap / kBlock];

  pdl_wait();  // the scores come from the previous kernel
  pdl_launch_dependents();
  const int t = row_begin + blockIdx.x;
  const int tid = threadIdx.x;
  int r;
  const int n = row_length(t, qsl, seq_lens, req_id, num_reqs, ld, &r);
  int32_t* orow = out + static_cast<int64_t>(t) * topk;
  int32_t* prow = po.block_table != nullptr ? po.physical + static_cast<int64_t>(t) * topk : nullptr;
  const int32_t* bt_row = po.block_table != nullptr && r >= 0 && r < num_reqs
                              ? po.block_table + static_cast<int64_t>(r) * po.bt_stride
                              : nullptr;
  if (bt_row == nullptr) prow = nullptr;
  bool bad = false;
  if (prow != nullptr && po.valid_counts != nullptr && tid == 0) po.valid_counts[t] = n < topk ? n : topk;
  const float* lrow = logits + static_cast<int64_t>(t) * ld;
  if (n <= topk) {
    write_short_row(n, topk, orow, prow, bt_row, po, &bad);
    if (bad) flag_error(po.err, DSA_DEVERR_ID_RANGE);
    return;
  }
  if constexpr (kStaged) {
    // rows are 16-byte aligned (ld is a multiple of 4): float4 loads, four in flight per thread
    const float4* l4 = reinterpret_cast<const float4*>(lrow);
    const int n4 = (n + 3) >> 2;
    for (int base = 0; base < n4; base += 4 * kTopkThreads) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i4 = base + u * kTopkThreads + tid;
        v[u] = i4 < n4 ? __ldg(l4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = 4 * (base + u * kTopkThreads + tid);
        if (i < n) keys[i] = f32_key(v[u].x);
        if (i + 1 < n) keys[i + 1] = f32_key(v[u].y);
        if (i + 2 < n) keys[i + 2] = f32_key(v[u].z);
        if (i + 3 < n) keys[i + 3] = f32_key(v[u].w);
      }
    }
    // the request's block-table row, for the id conversion in emit
    if (bt_row != nullptr) {
      const int cap = po.bt_stride < kTopkRowCap / kBlock ? static_cast<int>(po.bt_stride) : kTopkRowCap / kBlock;
      const int pages = min((n + kBlock - 1) / kBlock, cap);
      for (int p = tid; p < pages; p += kTopkThreads) bts[p] = __ldg(bt_row + p);
      bt_row = bts;
    }
  }
  auto key_at = [&](int i) -> uint32_t {
    if constexpr (kStaged) return keys[i];
    else return f32_key(__ldg(lrow + i));
  };

  // round 1
  const bool have_hist = hist_g != nullptr && t < hist_rows;
  if (have_hist) {
    const uint4* hrow = reinterpret_cast<const uint4*>(hist_g + static_cast<int64_t>(t) * kBins);
    for (int b = tid; b < kBins / 4; b += kTopkThreads) reinterpret_cast<uint4*>(hist)[b] = __ldcg(hrow + b);
  } else {
    for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
  }
  if (tid == 0) {
    s_bin = 0;
    s_above = 0;
    s_cnt = 0;
    s_eq = 0;
  }
  __syncthreads();
  if (!have_hist) {
    for (int i = tid; i < n; i += kTopkThreads) atomicAdd(&hist[key_at(i) >> kHistShift], 1u);
    __syncthreads();
  }
  find_bin(hist, static_cast<uint32_t>(topk), &s_bin, &s_above, sm);
  const uint32_t b1 = static_cast<uint32_t>(s_bin);
  uint32_t need = static_cast<uint32_t>(topk) - s_above;
  const bool gather = hist[b1] <= static_cast<uint32_t>(kCandCap);

  // one pass: keys above the boundary bin go out, the bin's keys are gathered
  for (int base = 0; base < n; base += kTopkThreads) {
    const int i = base + tid;
    const uint32_t key = i < n ? key_at(i) : 0u;
    const uint32_t bin = key >> kHistShift;
    const bool up = i < n && bin > b1;
    const uint32_t p = warp_reserve(up, &s_cnt);
    if (up && p < static_cast<uint32_t>(topk)) emit(orow, prow, bt_row, po.bt_stride, po.stride_rows, p, i, &bad);
    if (gather) {
      const bool eq = i < n && bin == b1;
      const uint32_t q = warp_reserve(eq, &s_eq);
      if (eq && q < static_cast<uint32_t>(kCandCap)) {
        ckey[q] = key;
        cidx[q] = static_cast<uint32_t>(i);
      }
    }
  }
  __syncthreads();
  // the boundary bin: candidates j < m, with key and id
  const uint32_t m = gather ? min(s_eq, static_cast<uint32_t>(kCandCap)) : static_cast<uint32_t>(n);
  auto cand_key = [&](uint32_t j) -> uint32_t { return gather ? ckey[j] : key_at(static_cast<int>(j)); };
  auto cand_id = [&](uint32_t j) -> int { return gather ? static_cast<int>(cidx[j]) : static_cast<int>(j); };
  uint32_t prefix = b1;
  int shift = kHistShift;
  const int shifts[2] = {10, 0};
  const int widths[2] = {11, 10};
  if (hist[b1] != need) {  // else the whole bin is taken
    for (int lvl = 0; lvl < 2; ++lvl) {
      const uint32_t mask = (1u << widths[lvl]) - 1u;
      __syncthreads();
      for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
      if (tid == 0) {
        s_bin = 0;
        s_above = 0;
      }
      __syncthreads();
      for (uint32_t j = tid; j < m; j += kTopkThreads) {
        const uint32_t k = cand_key(j);
        if ((k >> shift) == prefix) atomicAdd(&hist[(k >> shifts[lvl]) & mask], 1u);
      }
      __syncthreads();
      find_bin(hist, need, &s_bin, &s_above, sm);
      const int b = s_bin;
      need -= s_above;
      prefix = (prefix << widths[lvl]) | static_cast<uint32_t>(b);
      shift = shifts[lvl];
      if (hist[b] == need) break;
    }
  }
  __syncthreads();
  if (tid == 0) s_eq = 0;
  __syncthreads();
  for (uint32_t j = tid; j < m; j += kTopkThreads) {
    const uint32_t k = cand_key(j);
    if ((k >> kHistShift) != b1) continue;  // row fallback: only the boundary bin
    const uint32_t pk = k >> shift;
    bool take = pk > prefix;
    if (!take && pk == prefix) take = atomicAdd(&s_eq, 1u) < need;
    if (take) {
      const uint32_t pos = atomicAdd(&s_cnt, 1u);
      if (pos < static_cast<uint32_t>(topk))
        emit(orow, prow, bt_row, po.bt_stride, po.stride_rows, pos, cand_id(j), &bad);
    }
  }
  if (bad) flag_error(po.err, DSA_DEVERR_ID_RANGE);
}

cudaError_t launch_topk(const float* logits, int64_t ld, const int32_t* qsl, const int32_t* seq_lens,
                        const int32_t* req_id, int num_reqs, int row_begin, int n_tokens, int topk, int32_t* out,
                        const TopkPhys* phys, const uint32_t* hist, int hist_rows, cudaStream_t stream) {
  const int rows = n_tokens - row_begin;
  if (rows <= 0) return cudaSuccess;
  const PhysOut po = phys_out(phys);
  const int base_smem = (kBins + 2 * kCandCap) * 4;
  if (ld <= kTopkRowCap) {
    const int smem = base_smem + kTopkRowCap * 4;
    static bool configured = false;
    if (!configured) {
      cudaError_t e = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      configured = true;
    }
    return launch_pdl(topk_kernel<true>, dim3(rows), dim3(kTopkThreads), smem, stream, logits, ld, qsl, seq_lens,
                      req_id, num_reqs, row_begin, topk, out, po, hist, hist_rows);
  } else {
    static bool configured = false;
    if (!configured) {
      cudaError_t e =
          cudaFuncSetAttribute(topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, base_smem);
      if (e != cudaSuccess) return e;
      configured = true;
    }
    return launch_pdl(topk_kernel<false>, dim3(rows), dim3(kTopkThreads), base_smem, stream, logits, ld, qsl,
                      seq_lens, req_id, num_reqs, row_begin, topk, out, po, hist, hist_rows);
  }
}

// ---------------------------------------------------------------------------
// Multi-CTA select for decode rows.


__global__ void __launch_bounds__(kTopkThreads) select_kernel(SelectArgs a, PhysOut po) {
  extern __shared__ uint32_t sh[];
  uint32_t* hist = sh;               // kBins
  uint2* cands = reinterpret_cast<uint2*>(sh + kBins);  // staged candidates (finishing CTA)
  __shared__ uint32_t sm[32];
  __shared__ int s_bin;
  __shared__ uint32_t s_above, s_cnt, s_eq;
  __shared__ int s_last;

  pdl_wait();  // the scores come from the previous kernel
  pdl_launch_dependents();
  const int t = blockIdx.y;
  const int c = blockIdx.x;
  const int tid = threadIdx.x;
  int r;
  const int n = row_length(t, a.qsl, a.seq_lens, a.req_id, a.num_reqs, a.ld, &r);
  const int chunks = n > 0 ? (n + kSelectChunk - 1) / kSelectChunk : 1;
  if (c >= chunks) return;
  int32_t* orow = a.out + static_cast<int64_t>(t) * a.topk;
  int32_t* prow = po.block_table != nullptr ? po.physical + static_cast<int64_t>(t) * a.topk : nullptr;
  const int32_t* bt_row = po.block_table != nullptr && r >= 0 && r < a.num_reqs
                              ? po.block_table + static_cast<int64_t>(r) * po.bt_stride
                              : nullptr;
  if (bt_row == nullptr) prow = nullptr;
  bool bad = false;
  if (n <= a.topk) {
    if (c == 0) {
      if (prow != nullptr && po.valid_counts != nullptr && tid == 0) po.valid_counts[t] = n;
      write_short_row(n, a.topk, orow, prow, bt_row, po, &bad);
      if (bad) flag_error(po.err, DSA_DEVERR_ID_RANGE);
    }
    return;
  }
  if (c == 0 && prow != nullptr && po.valid_counts != nullptr && tid == 0) po.valid_counts[t] = a.topk;
  uint32_t* cnt = a.counters + static_cast<int64_t>(t) * kRowCounters;
  uint2* crow = a.cand + static_cast<int64_t>(t) * a.ld;
  const float* lrow = a.logits + static_cast<int64_t>(t) * a.ld;

  // boundary bin of the first round, from the histogram the score kernel built
  const uint32_t* hrow = a.hist + static_cast<int64_t>(t) * kBins;
  for (int b = tid; b < kBins / 4; b += kTopkThreads)
    reinterpret_cast<uint4*>(hist)[b] = __ldcg(reinterpret_cast<const uint4*>(hrow) + b);
  if (tid == 0) {  // defaults if the histogram were inconsistent with the row
    s_bin = 0;
    s_above = 0;
  }
  __syncthreads();
  find_bin(hist, static_cast<uint32_t>(a.topk), &s_bin, &s_above, sm);
  const uint32_t b1 = static_cast<uint32_t>(s_bin);
  const uint32_t above = s_above;

  // this chunk: emit keys above the boundary bin, collect the boundary bin's
  // keys. Count in shared memory first, reserve the row slots with one global
  // atomic per CTA, then write (no global atomics inside the loop).
  const int lo = c * kSelectChunk;
  const int hi = min(n, lo + kSelectChunk);
  uint32_t* ckeys = sh + kBins;  // the chunk's keys (kSelectChunk), shared with `cands` below
  if (tid == 0) {
    s_cnt = 0;
    s_eq = 0;
  }
  {  // stage the chunk's keys: 16-byte loads, four in flight per thread (lo is a multiple of 4)
    const float4* l4 = reinterpret_cast<const float4*>(lrow + lo);
    const int n4 = (hi - lo + 3) >> 2;
    for (int b4 = 0; b4 < n4; b4 += 4 * kTopkThreads) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i4 = b4 + u * kTopkThreads + tid;
        v[u] = i4 < n4 ? __ldg(l4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i4 = b4 + u * kTopkThreads + tid;
        if (i4 < n4) {
          ckeys[4 * i4] = f32_key(v[u].x);
          ckeys[4 * i4 + 1] = f32_key(v[u].y);
          ckeys[4 * i4 + 2] = f32_key(v[u].z);
          ckeys[4 * i4 + 3] = f32_key(v[u].w);
        }
      }
    }
  }
  __syncthreads();
  for (int base = lo; base < hi; base += kTopkThreads) {
    const int i = base + tid;
    const uint32_t key = i < hi ? ckeys[i - lo] : 0u;
    const uint32_t bin = key >> kHistShift;
    const uint32_t n_up = __popc(__ballot_sync(0xffffffffu, i < hi && bin > b1));
    const uint32_t n_eq = __popc(__ballot_sync(0xffffffffu, i < hi && bin == b1));
    if ((tid & 31) == 0) {
      if (n_up) atomicAdd(&s_cnt, n_up);
      if (n_eq) atomicAdd(&s_eq, n_eq);
    }
  }
  __syncthreads();
  __shared__ uint32_t s_base_up, s_base_eq;
  if (tid == 0) {
    s_base_up = s_cnt ? atomicAdd(&cnt[0], s_cnt) : 0;
    s_base_eq = s_eq ? atomicAdd(&cnt[1], s_eq) : 0;
    s_cnt = 0;
    s_eq = 0;
  }
  __syncthreads();
  for (int base = lo; base < hi; base += kTopkThreads) {
    const int i = base + tid;
    const uint32_t key = i < hi ? ckeys[i - lo] : 0;
    const uint32_t bin = key >> kHistShift;
    const bool up = i < hi && bin > b1;
    const bool eq = i < hi && bin == b1;
    const uint32_t p_up = s_base_up + warp_reserve(up, &s_cnt);
    const uint32_t p_eq = s_base_eq + warp_reserve(eq, &s_eq);
    if (up && p_up < static_cast<uint32_t>(a.topk))
      emit(orow, prow, bt_row, po.bt_stride, po.stride_rows, p_up, i, &bad);
    if (eq && p_eq < static_cast<uint32_t>(a.ld)) crow[p_eq] = make_uint2(key, static_cast<uint32_t>(i));
  }
  // the last CTA of the row to finish resolves the boundary bin
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(&cnt[2], 1u) == static_cast<uint32_t>(chunks - 1);
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    const uint32_t m = min(__ldcg(&cnt[1]), static_cast<uint32_t>(a.ld));
    uint32_t need = static_cast<uint32_t>(a.topk) - above;  // 1 <= need <= m
    const bool staged = m <= kTopkRowCap / 2;
    if (staged) {
      for (uint32_t j = tid; j < m; j += kTopkThreads) cands[j] = __ldcg(crow + j);
      __syncthreads();
    }
    auto cand_at = [&](uint32_t j) -> uint2 { return staged ? cands[j] : __ldcg(crow + j); };
    uint32_t prefix = b1;
    int shift = kHistShift;
    const int shifts[2] = {10, 0};
    const int widths[2] = {11, 10};
    for (int lvl = 0; lvl < 2; ++lvl) {
      const uint32_t mask = (1u << widths[lvl]) - 1u;
      for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
      if (tid == 0) {
        s_bin = 0;
        s_above = 0;
      }
      __syncthreads();
      for (uint32_t j = tid; j < m; j += kTopkThreads) {
        const uint32_t k = cand_at(j).x;
        if ((k >> shift) == prefix) atomicAdd(&hist[(k >> shifts[lvl]) & mask], 1u);
      }
      __syncthreads();
      find_bin(hist, need, &s_bin, &s_above, sm);
      const int b = s_bin;
      need -= s_above;
      prefix = (prefix << widths[lvl]) | static_cast<uint32_t>(b);
      shift = shifts[lvl];
      const bool whole = hist[b] == need;
      __syncthreads();
      if (whole) break;
    }
    if (tid == 0) s_eq = 0;
    __syncthreads();
    for (uint32_t j = tid; j < m; j += kTopkThreads) {
      const uint2 kv = cand_at(j);
      const uint32_t pk = kv.x >> shift;
      bool take = pk > prefix;
      if (!take && pk == prefix) take = atomicAdd(&s_eq, 1u) < need;
      if (take) {
        const uint32_t pos = atomicAdd(&cnt[0], 1u);
        if (pos < static_cast<uint32_t>(a.topk))
          emit(orow, prow, bt_row, po.bt_stride, po.stride_rows, pos, static_cast<int>(kv.y), &bad);
      }
    }
    (void)s_cnt;
  }
  if (bad) flag_error(po.err, DSA_DEVERR_ID_RANGE);
}

cudaError_t launch_select(const SelectArgs& a, const TopkPhys* phys, cudaStream_t stream) {
  if (a.n_rows <= 0) return cudaSuccess;
  const int smem = kBins * 4 + (kTopkRowCap / 2) * 8;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t chunks = (a.ld + kSelectChunk - 1) / kSelectChunk;
  dim3 grid(static_cast<unsigned>(chunks < 1 ? 1 : chunks), static_cast<unsigned>(a.n_rows));
  return launch_pdl(select_kernel, grid, dim3(kTopkThreads), smem, stream, a, phys_out(phys));
}

}  // namespace dsa
