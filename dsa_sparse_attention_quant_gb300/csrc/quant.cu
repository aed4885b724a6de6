// quant.cu — S1 (K quantisation fused with the paged-cache write) and S2a
// (q quantisation with the head-weight fold), sm_103a.
//
// Both follow "IndexCache：DeepSeek 稀疏注意力中的跨层索引复用" (atomage.cn):
// the `SparseAttnIndexer` body calls `indexer_k_quant_and_cache(k, kv_cache,
// slot_mapping, quant_block_size, scale_fmt)`, and `Indexer.forward` quantises
// q per 128-value group with ue8m0 scales and folds q_scale, softmax_scale and
// n_head^-0.5 into the head weights. With a cos/sin table, the rows are first
// rotated on their leading 64 dims (RoPE, as `Indexer.forward` applies
// `rotary_emb` before quantising). One warp handles one 128-value row: each
// lane loads 8 bytes (4 bf16), the warp reduces amax with shuffles, and the
// 32 lanes store 128 contiguous code bytes (64 for the FP4 cache) — fully
// coalesced, one pass over HBM in each direction.
#include "common.cuh"
#include "kernels.h"

namespace dsa {

__global__ void __launch_bounds__(256) k_quant_write_kernel(const __nv_bfloat16* __restrict__ k, int64_t n,
                                                            int64_t row_stride,
                                                            const int64_t* __restrict__ slot_mapping,
                                                            uint8_t* __restrict__ cache, int64_t num_blocks,
                                                            bool fp4, RopeArgs rope, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < n; t += warps) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;  // padding token
    if (slot >= num_blocks * kBlock) {
      if (lane == 0) flag_error(err, DSA_DEVERR_SLOT_RANGE);
      continue;
    }
    uint2 raw = __ldg(reinterpret_cast<const uint2*>(k + t * row_stride) + lane);
    if (rope.cos_sin != nullptr) {
      const float* cs = rope_row(rope, t, err, lane);  // warp-uniform
      if (cs != nullptr) raw = rope_row_lane(raw, cs);
    }
    quant_store_k_row(cache, slot, raw, fp4, lane);
  }
}

__global__ void __launch_bounds__(256) q_quant_fold_kernel(const __nv_bfloat16* __restrict__ q,
                                                           const float* __restrict__ w, int64_t rows,
                                                           float softmax_scale, uint8_t* __restrict__ q_fp8,
                                                           float* __restrict__ q_scale,
                                                           float* __restrict__ w_folded, RopeArgs rope,
                                                           int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    uint2 raw = __ldg(reinterpret_cast<const uint2*>(q + r * kDim) + lane);
    if (rope.cos_sin != nullptr) {
      const float* cs = rope_row(rope, r / kHeads, err, lane);  // warp-uniform
      if (cs != nullptr) raw = rope_row_lane(raw, cs);
    }
    float s;
    const uint32_t codes = quant_row_lane(raw, &s);
    reinterpret_cast<uint32_t*>(q_fp8 + r * kDim)[lane] = codes;
    if (lane == 0) {
      if (q_scale != nullptr) q_scale[r] = s;
      // ((w * q_scale) * softmax_scale) * n_head^-0.5, each product rounded to fp32
      w_folded[r] = __fmul_rn(__fmul_rn(__fmul_rn(__ldg(w + r), s), softmax_scale), 0.125f);
    }
  }
}

// S5: one CTA per query row, each thread converts four ids per step.
__global__ void __launch_bounds__(256) convert_kernel(const int32_t* __restrict__ logical, int64_t n_tokens,
                                                      int topk, const int32_t* __restrict__ req_id,
                                                      const int32_t* __restrict__ block_table, int num_reqs,
                                                      int64_t bt_stride, int stride_rows,
                                                      int32_t* __restrict__ physical,
                                                      int32_t* __restrict__ valid_counts, int32_t* err) {
  const int64_t t = blockIdx.x;
  if (t >= n_tokens) return;
  const int r = __ldg(req_id + t);
  const bool req_ok = r >= 0 && r < num_reqs;  // else every id of the row is flagged and left -1
  const int32_t* bt_row = block_table + static_cast<int64_t>(req_ok ? r : 0) * bt_stride;
  const int4* in = reinterpret_cast<const int4*>(logical + t * topk);
  int4* out = reinterpret_cast<int4*>(physical + t * topk);
  int valid = 0;
  bool bad = false;
  for (int j = threadIdx.x; j < topk / 4; j += blockDim.x) {
    int4 v = __ldg(in + j);
    int ids[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int id = ids[e];
      int p = -1;
      if (id >= 0) {
        const int64_t page = id / kBlock;
        const int32_t blk = req_ok && page < bt_stride ? __ldg(bt_row + page) : -1;
        if (blk >= 0) {
          p = blk * stride_rows + id % kBlock;
          ++valid;
        } else {
          bad = true;
        }
      }
      ids[e] = p;
    }
    out[j] = make_int4(ids[0], ids[1], ids[2], ids[3]);
  }
  if (bad) flag_error(err, DSA_DEVERR_ID_RANGE);
  if (valid_counts != nullptr) {  // uniform across the block
    __shared__ int warp_sums[8];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) valid += __shfl_xor_sync(0xffffffffu, valid, o);
    if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = valid;
    __syncthreads();
    if (threadIdx.x == 0) {
      int s = 0;
      for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) s += warp_sums[i];
      valid_counts[t] = s;
    }
  }
}

static int grid_for_rows(int64_t rows, int warps_per_block) {
  int64_t blocks = (rows + warps_per_block - 1) / warps_per_block;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

cudaError_t launch_k_quant_write(const void* k, int64_t n, int64_t row_stride, const int64_t* slot_mapping,
                                 uint8_t* cache, int64_t num_blocks, bool fp4, const RopeArgs& rope, int32_t* err,
                                 cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  k_quant_write_kernel<<<grid_for_rows(n, 8), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(k), n,
                                                                row_stride, slot_mapping, cache, num_blocks, fp4,
                                                                rope, err);
  return cudaGetLastError();
}

cudaError_t launch_q_quant_fold(const void* q, const float* w, int64_t n_tokens, float softmax_scale,
                                uint8_t* q_fp8, float* q_scale, float* w_folded, const RopeArgs& rope, int32_t* err,
                                cudaStream_t stream) {
  const int64_t rows = n_tokens * kHeads;
  if (rows <= 0) return cudaSuccess;
  q_quant_fold_kernel<<<grid_for_rows(rows, 8), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(q), w, rows,
                                                                  softmax_scale, q_fp8, q_scale, w_folded, rope,
                                                                  err);
  return cudaGetLastError();
}

// The failure path of a pipeline wait: an mbarrier that nothing completes,
// waited on with the bounded wait of the pipelines; after the limit the wait
// flags DSA_DEVERR_TIMEOUT and the kernel returns.
__global__ void wait_selftest_kernel(int32_t* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(&bar, 1);
  fence_barrier_init();
  mbar_wait(&bar, 0, &abort_flag, err);  // no arrival: gives up after kWaitLimitNs
}

cudaError_t launch_wait_selftest(int32_t* err, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

cudaError_t launch_convert(const int32_t* logical, int64_t n_tokens, int topk, const int32_t* req_id,
                           const int32_t* block_table, int num_reqs, int64_t bt_stride, int stride_rows,
                           int32_t* physical, int32_t* valid_counts, int32_t* err, cudaStream_t stream) {
  if (n_tokens <= 0) return cudaSuccess;
  convert_kernel<<<static_cast<unsigned>(n_tokens), 256, 0, stream>>>(logical, n_tokens, topk, req_id,
                                                                      block_table, num_reqs, bt_stride,
                                                                      stride_rows, physical, valid_counts, err);
  return cudaGetLastError();
}

}  // namespace dsa
