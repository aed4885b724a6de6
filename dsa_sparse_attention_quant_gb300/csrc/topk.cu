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
// Exact radix select over order-preserving 32-bit keys of the fp32 scores: up
// to three histogram rounds (11, 11 and 10 bits) narrow down the k-th largest
// key; a final pass emits every key above it and as many keys equal to it as
// are still needed. A round stops early once its boundary bin is needed whole.
// Rows that fit (<= kRowCap scores) are staged once in shared memory; longer
// rows are re-read from global memory (L2) in each round.
#include "common.cuh"
#include "kernels.h"

namespace dsa {

constexpr int kTopkThreads = 512;
constexpr int kBins = 2048;
constexpr int kRowCap = 12288;  // scores staged in shared memory: 48 KB

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

__device__ __forceinline__ void emit(int32_t* orow, int32_t* prow, const int32_t* bt_row, int64_t bt_stride,
                                     int stride_rows, uint32_t pos, int id, bool* bad) {
  orow[pos] = id;
  if (prow != nullptr) {
    const int64_t page = id / kBlock;
    const int32_t blk = page < bt_stride ? __ldg(bt_row + page) : -1;
    if (blk < 0) *bad = true;
    prow[pos] = blk < 0 ? -1 : blk * stride_rows + id % kBlock;
  }
}

template <bool kStaged>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ logits, int64_t ld,
                                                            const int32_t* qsl, const int32_t* seq_lens,
                                                            const int32_t* req_id, int num_reqs, int topk,
                                                            int32_t* __restrict__ out, PhysOut po) {
  extern __shared__ uint32_t sh[];
  uint32_t* hist = sh;
  uint32_t* keys = sh + kBins;
  __shared__ uint32_t sm[32];
  __shared__ int s_bin;
  __shared__ uint32_t s_above, s_cnt, s_eq;

  const int t = blockIdx.x;
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
    for (int i = tid; i < topk; i += kTopkThreads) {
      if (i < n) {
        emit(orow, prow, bt_row, po.bt_stride, po.stride_rows, i, i, &bad);
      } else {
        orow[i] = -1;
        if (prow != nullptr) prow[i] = -1;
      }
    }
    if (bad) flag_error(po.err, DSA_DEVERR_ID_RANGE);
    return;
  }
  if constexpr (kStaged) {
    for (int i = tid; i < n; i += kTopkThreads) keys[i] = f32_key(lrow[i]);
  }
  auto key_at = [&](int i) -> uint32_t {
    if constexpr (kStaged) return keys[i];
    else return f32_key(__ldg(lrow + i));
  };

  uint32_t need = static_cast<uint32_t>(topk);
  uint32_t prefix = 0;  // selected high bits of the threshold key
  int shift = 32;       // prefix = threshold >> shift
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int lvl = 0; lvl < 3; ++lvl) {
    const int sh_l = shifts[lvl];
    const uint32_t mask = (1u << widths[lvl]) - 1u;
    for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kTopkThreads) {
      const uint32_t k = key_at(i);
      if (lvl == 0 || (k >> shift) == prefix) atomicAdd(&hist[(k >> sh_l) & mask], 1u);
    }
    __syncthreads();
    find_bin(hist, need, &s_bin, &s_above, sm);
    const int b = s_bin;
    need -= s_above;
    prefix = (lvl == 0) ? static_cast<uint32_t>(b) : ((prefix << widths[lvl]) | static_cast<uint32_t>(b));
    shift = sh_l;
    const bool whole = hist[b] == need;
    __syncthreads();
    if (whole) break;
  }
  if (tid == 0) {
    s_cnt = 0;
    s_eq = 0;
  }
  __syncthreads();
  for (int i = tid; i < n; i += kTopkThreads) {
    const uint32_t pk = key_at(i) >> shift;  // shift < 32 here
    uint32_t pos = 0xFFFFFFFFu;
    if (pk > prefix) {
      pos = atomicAdd(&s_cnt, 1u);
    } else if (pk == prefix && atomicAdd(&s_eq, 1u) < need) {
      pos = atomicAdd(&s_cnt, 1u);
    }
    if (pos < static_cast<uint32_t>(topk)) emit(orow, prow, bt_row, po.bt_stride, po.stride_rows, pos, i, &bad);
  }
  if (bad) flag_error(po.err, DSA_DEVERR_ID_RANGE);
}

cudaError_t launch_topk(const float* logits, int64_t ld, const int32_t* qsl, const int32_t* seq_lens,
                        const int32_t* req_id, int num_reqs, int n_tokens, int topk, int32_t* out,
                        const TopkPhys* phys, cudaStream_t stream) {
  if (n_tokens <= 0) return cudaSuccess;
  PhysOut po{};
  if (phys != nullptr) {
    po.block_table = phys->block_table;
    po.bt_stride = phys->bt_stride;
    po.stride_rows = phys->stride_rows;
    po.physical = phys->physical;
    po.valid_counts = phys->valid_counts;
    po.err = phys->err;
  }
  if (ld <= kRowCap) {
    const int smem = (kBins + kRowCap) * 4;
    static bool configured = false;
    if (!configured) {
      cudaError_t e = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      configured = true;
    }
    topk_kernel<true><<<n_tokens, kTopkThreads, smem, stream>>>(logits, ld, qsl, seq_lens, req_id, num_reqs, topk,
                                                                out, po);
  } else {
    topk_kernel<false><<<n_tokens, kTopkThreads, kBins * 4, stream>>>(logits, ld, qsl, seq_lens, req_id, num_reqs,
                                                                       topk, out, po);
  }
  return cudaGetLastError();
}

}  // namespace dsa
