// gather.cu — the consumer's gather of the selected rows (sm_103a).
//
// "IndexCache：DeepSeek 稀疏注意力中的跨层索引复用" (atomage.cn): the sparse MLA
// of every layer in a group reads, for each query token, the KV rows of the
// `index_topk` selected keys; "vllm.v1.attention.backends.mla.index_group"
// (`_convert_once`) turns the ids into physical slots for exactly that read.
// The row format is not on the pages, so this gathers bytes: out[t][j] = the
// row_bytes bytes of physical row physical[t][j], zeros where the id is -1 (a
// row shorter than k) or out of range (flagged).
//
// The output is a flat array of 16-byte chunks; consecutive threads copy
// consecutive chunks of a row, so the reads of a row and all writes are
// coalesced, and every thread keeps four chunks in flight. HBM-bound: one
// read and one write of each selected row.
#include "common.cuh"
#include "kernels.h"

namespace dsa {

constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 4;

__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(const uint8_t* __restrict__ rows,
                                                                     int64_t num_rows, int64_t chunks_per_row,
                                                                     int64_t row_stride,
                                                                     const int32_t* __restrict__ physical,
                                                                     int64_t total_chunks, uint4* __restrict__ out,
                                                                     int32_t* err) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kGatherThreads;
  bool bad = false;
  for (int64_t c0 = static_cast<int64_t>(blockIdx.x) * kGatherThreads * kGatherUnroll + threadIdx.x;
       c0 < total_chunks; c0 += stride * kGatherUnroll) {
    uint4 v[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int64_t c = c0 + static_cast<int64_t>(u) * kGatherThreads;
      v[u] = make_uint4(0, 0, 0, 0);
      if (c < total_chunks) {
        const int64_t r = c / chunks_per_row;
        const int32_t id = __ldg(physical + r);
        if (id >= 0 && id < num_rows) {
          v[u] = __ldg(reinterpret_cast<const uint4*>(rows + static_cast<int64_t>(id) * row_stride) +
                       (c - r * chunks_per_row));
        } else if (id != -1) {
          bad = true;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int64_t c = c0 + static_cast<int64_t>(u) * kGatherThreads;
      if (c < total_chunks) out[c] = v[u];
    }
  }
  if (bad) flag_error(err, DSA_DEVERR_ID_RANGE);
}

cudaError_t launch_gather_rows(const uint8_t* rows, int64_t num_rows, int64_t row_bytes, int64_t row_stride,
                               const int32_t* physical, int64_t n_ids, uint8_t* out, int num_sms, int32_t* err,
                               cudaStream_t stream) {
  const int64_t cpr = row_bytes / 16;
  const int64_t total = n_ids * cpr;
  if (total <= 0) return cudaSuccess;
  const int64_t per_cta = static_cast<int64_t>(kGatherThreads) * kGatherUnroll;
  int64_t grid = (total + per_cta - 1) / per_cta;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;  // eight 256-thread CTAs per SM; the rest loops
  if (grid > cap) grid = cap;
  gather_rows_kernel<<<static_cast<unsigned>(grid), kGatherThreads, 0, stream>>>(
      rows, num_rows, cpr, row_stride, physical, total, reinterpret_cast<uint4*>(out), err);
  return cudaGetLastError();
}

}  // namespace dsa
