// logits.cu — S2b: indexer scores on the tcgen05 tensor cores (sm_103a).
//
// Computes, for every query token t and every key s it may see (s <= position),
//   I[t,s] = k_scale[s] * sum_h w'[t,h] * ReLU( sum_d q8[t,h,d] * k8[s,d] ),
// the score of DeepSeek-V3.2's indexer as run in "IndexCache：DeepSeek 稀疏注意力
// 中的跨层索引复用" (atomage.cn): 64 FP8 query heads against one shared FP8 K
// row per token (`Indexer.forward`, MQA cache of `DeepseekV32IndexerCache`),
// with q_scale, softmax_scale and n_head^-0.5 already folded into w'.
//
// Mapping onto Blackwell:
//  * M = 128 keys per tile (two 64-slot pages, each fetched by one TMA box
//    through the block table), N = 64 heads x NTOK query tokens, K = 128
//    (four kind::f8f6f4 MMAs of K=32). The head reduction is then local to
//    one TMEM lane (= one key), so the epilogue needs no shuffles.
//  * The work of a launch is a flat list of (query block, key tile) items; each
//    persistent CTA takes one contiguous, equally sized slice of it, so the
//    load is balanced to one tile whatever the mix of lengths.
//  * Warp roles: warp 0 issues TMA (K pages, K scales, q block, w' block),
//    warp 1 issues the MMAs, the remaining warps read TMEM and apply
//    ReLU, the w' reduction and the K scale, and store fp32 scores.
//  * Every wait is bounded in time (DSA_DEVERR_TIMEOUT, then an orderly exit).
#include "common.cuh"
#include "kernels.h"

namespace dsa {

// ------------------------------------------------------------------ logits
template <int NTOK>
struct LogitsCfg {
  static constexpr int N = 64 * NTOK;                     // MMA N: heads x tokens
  static constexpr int kStages = NTOK == 1 ? 8 : 6;       // K-tile ring
  static constexpr int kAcc = NTOK == 1 ? 4 : 2;          // TMEM accumulator ring
  static constexpr int kEpiWG = 2;                        // epilogue warpgroups (take tiles in turn)
  static constexpr int kEpiWarps = 4 * kEpiWG;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr uint32_t kTmemCols = N * kAcc;         // 256 or 512
  static constexpr int kStageBytes = 17 * 1024;           // 2 x 8 KB K pages, 2 x 256 B scales, 1 KB aligned
  static constexpr int kScaleOff = 16384;
  static constexpr int kQBytes = N * kDim;
  static constexpr int kWBytes = NTOK * kHeads * 4;
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffW = kOffQ + 2 * kQBytes;
  static constexpr int kOffBar = kOffW + 2 * kWBytes;
  static constexpr int kNumBars = 2 * kStages + 4 + 2 * kAcc + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // decode: one score histogram per epilogue warp (first radix round of the top-k)
  static constexpr int kHistBytes = NTOK == 1 ? kEpiWarps * kHistBins * 4 : 0;
  static constexpr int kOffHist = (kOffMisc + 16 + 127) / 128 * 128;
  static constexpr int kSmemBytes = kOffHist + kHistBytes + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t kIdesc = f8_idesc(128, N);
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation must be a power of two");
};

__device__ __forceinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, unsigned long long deadline) {
  const uint32_t addr = smem_u32(bar);
  while (!mbar_try_wait(addr, parity)) {
    if (global_ns() > deadline) return false;
  }
  return true;
}

template <int NTOK>
__global__ void __launch_bounds__(LogitsCfg<NTOK>::kThreads, 1)
    logits_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                  SegmentPlan plan, LogitsArgs a) {
  using C = LogitsCfg<NTOK>;
  constexpr int S = C::kStages;
  constexpr int A = C::kAcc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + S;
  uint64_t* qfull = empty + S;
  uint64_t* qempty = qfull + 2;
  uint64_t* tfull = qempty + 2;
  uint64_t* tempty = tfull + A;
  uint64_t* done = tempty + A;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1 + 4);  // MMA commit + the 4 epilogue warps that read the tile's scales
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], 1 + C::kEpiWarps);
    }
    for (int c = 0; c < A; ++c) {
      mbar_init(&tfull[c], 1);
      mbar_init(&tempty[c], 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_q);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Everything above may overlap the previous kernel of the stream (programmatic
  // dependent launch); the plan, q codes, weights and K cache are read below.
  pdl_wait();
  pdl_launch_dependents();
  const CtaWork cw = plan.cta[blockIdx.x];  // this CTA's slice, laid out by the plan kernel
  const int it_begin = cw.it_begin;         // an empty slice runs no loop iteration below
  const int it_end = cw.it_end;
  const int j0 = cw.qb0;  // first query block of this CTA's slice

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int j = j0;
    QBlock qb = plan.qb[j];
    int jt_end = plan.tile_start[j + 1];
    int kt = cw.kt0;
    int qcount = 0, n = 0, npages = 0, batch = -1;
    int32_t cur_ids = -1, nxt_ids = -1;
    const int32_t* bt_row = nullptr;
    bool new_qb = true;
    for (int it = it_begin; it < it_end; ++it, ++n, ++kt) {
      if (it == jt_end) {
        ++j;
        qb = plan.qb[j];
        jt_end = plan.tile_start[j + 1];
        kt = 0;
        new_qb = true;
      }
      if (new_qb) {
        const int qs = qcount & 1;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&qempty[qs], ((qcount >> 1) & 1) ^ 1, abort_flag, a.err);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&qfull[qs], C::kQBytes + qb.ntok * kHeads * 4);
          tma_load_2d(smem + C::kOffQ + qs * C::kQBytes, &tmap_q, &qfull[qs], 0, qb.t0 * kHeads);
          bulk_load(smem + C::kOffW + qs * C::kWBytes, a.w_folded + static_cast<int64_t>(qb.t0) * kHeads,
                    qb.ntok * kHeads * 4, &qfull[qs]);
        }
        ++qcount;
        npages = (qb.p0 + qb.ntok + kBlock - 1) / kBlock;
        bt_row = a.block_table + static_cast<int64_t>(qb.req) * a.bt_stride;
        batch = (2 * kt) >> 5;
        const int p = batch * 32 + lane;
        cur_ids = p < npages ? __ldg(bt_row + p) : -1;
        nxt_ids = p + 32 < npages ? __ldg(bt_row + p + 32) : -1;
        new_qb = false;
      }
      const int stage = n % S;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&empty[stage], ((n / S) & 1) ^ 1, abort_flag, a.err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (((2 * kt) >> 5) != batch) {  // moved into the next batch of 32 page ids
        ++batch;
        cur_ids = nxt_ids;
        const int p = (batch + 1) * 32 + lane;
        nxt_ids = p < npages ? __ldg(bt_row + p) : -1;
      }
      const int id0 = __shfl_sync(0xffffffffu, cur_ids, (2 * kt) & 31);
      const int id1 = __shfl_sync(0xffffffffu, cur_ids, (2 * kt + 1) & 31);
      if (lane == 0) {
        uint8_t* st = smem + stage * C::kStageBytes;
        const bool in1 = 2 * kt + 1 < npages;
        const bool v0 = id0 >= 0 && id0 < a.num_blocks;
        const bool v1 = in1 && id1 >= 0 && id1 < a.num_blocks;
        if (!v0 || (in1 && !v1)) flag_error(a.err, DSA_DEVERR_BLOCK_RANGE);
        mbar_arrive_expect_tx(&full[stage], (v0 ? 8192 + 256 : 0) + (v1 ? 8192 + 256 : 0));
        if (v0) {
          tma_load_3d(st, &tmap_k, &full[stage], 0, 0, id0);
          bulk_load(st + C::kScaleOff, a.k_cache + static_cast<int64_t>(id0) * kPageBytes + kScaleOffset, 256,
                    &full[stage]);
        }
        if (v1) {
          tma_load_3d(st + 8192, &tmap_k, &full[stage], 0, 0, id1);
          bulk_load(st + C::kScaleOff + 256, a.k_cache + static_cast<int64_t>(id1) * kPageBytes + kScaleOffset,
                    256, &full[stage]);
        }
      }
    }
    if (lane == 0 && *abort_flag) {
      // let copies already issued land before the CTA's shared memory goes away
      const unsigned long long deadline = global_ns() + kWaitLimitNs;
      for (int m = (n > S ? n - S : 0); m < n; ++m) mbar_wait_until(&full[m % S], (m / S) & 1, deadline);
      mbar_wait_until(&qfull[(qcount - 1) & 1], ((qcount - 1) >> 1) & 1, deadline);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int j = j0;
      int jt_end = plan.tile_start[j + 1];
      int qcount = 0, qs = 0, n = 0;
      bool new_qb = true;
      for (int it = it_begin; it < it_end; ++it, ++n) {
        if (it == jt_end) {
          ++j;
          jt_end = plan.tile_start[j + 1];
          new_qb = true;
        }
        if (new_qb) {
          qs = qcount & 1;
          if (!mbar_wait(&qfull[qs], (qcount >> 1) & 1, abort_flag, a.err)) break;
          ++qcount;
          new_qb = false;
        }
        const int stage = n % S;
        const int acc = n % A;
        if (!mbar_wait(&full[stage], (n / S) & 1, abort_flag, a.err)) break;
        if (!mbar_wait(&tempty[acc], ((n / A) & 1) ^ 1, abort_flag, a.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * C::N);
        const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
        const uint32_t sb = smem_u32(smem + C::kOffQ + qs * C::kQBytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f8(d, sw128_kmajor_desc(sa + 32 * k), sw128_kmajor_desc(sb + 32 * k), C::kIdesc, k > 0 ? 1u : 0u);
        mma_commit(&empty[stage]);
        mma_commit(&tfull[acc]);
        if (it + 1 == jt_end || it + 1 == it_end) mma_commit(&qempty[qs]);
      }
      mma_commit(done);  // completes once every MMA issued above has finished
      mbar_wait_until(done, 0, global_ns() + kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int g = (warp - 2) >> 2;        // warpgroup: takes every kEpiWG-th tile
    const int quarter = warp & 3;         // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;  // key within the tile
    int j = j0;
    QBlock qb = plan.qb[j];
    int jt_end = plan.tile_start[j + 1];
    int kt = cw.kt0;
    int qcount = 0, qs = 0, n = 0;
    bool new_qb = true, aborted = false;
    float wr[NTOK == 1 ? kHeads : 1];
    // decode rows: this warp's histogram of the keys of its stored scores,
    // added to the row's global histogram when the warp leaves the row
    uint32_t* whist = reinterpret_cast<uint32_t*>(smem + C::kOffHist) + (warp - 2) * kHistBins;
    bool use_hist = false;
    auto flush_hist = [&](int row_t) {
      __syncwarp();
      uint32_t* dst = a.hist + static_cast<int64_t>(row_t) * kHistBins;
      for (int b = lane; b < kHistBins; b += 32) {
        const uint32_t v = whist[b];
        if (v != 0) atomicAdd(dst + b, v);
      }
    };
    for (int it = it_begin; it < it_end; ++it, ++n, ++kt) {
      if (it == jt_end) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[qs]);  // done with this q/w' buffer
        if constexpr (NTOK == 1) {
          if (use_hist) flush_hist(qb.t0);
        }
        ++j;
        qb = plan.qb[j];
        jt_end = plan.tile_start[j + 1];
        kt = 0;
        new_qb = true;
      }
      if (new_qb) {
        qs = qcount & 1;
        if (!mbar_wait(&qfull[qs], (qcount >> 1) & 1, abort_flag, a.err)) {
          aborted = true;
          break;
        }
        ++qcount;
        new_qb = false;
        if constexpr (NTOK == 1) {
          const float4* wsrc = reinterpret_cast<const float4*>(smem + C::kOffW + qs * C::kWBytes);
#pragma unroll
          for (int h = 0; h < kHeads / 4; ++h) {
            const float4 v = wsrc[h];
            wr[4 * h] = v.x;
            wr[4 * h + 1] = v.y;
            wr[4 * h + 2] = v.z;
            wr[4 * h + 3] = v.w;
          }
          use_hist = a.hist != nullptr && qb.t0 < a.hist_rows;
          if (use_hist) {
            uint4* z = reinterpret_cast<uint4*>(whist);
            for (int b = lane; b < kHistBins / 4; b += 32) z[b] = make_uint4(0, 0, 0, 0);
            __syncwarp();
          }
        }
      }
      if ((n % C::kEpiWG) != g) continue;
      const int stage = n % S;
      const int acc = n % A;
      if (!mbar_wait(&tfull[acc], (n / A) & 1, abort_flag, a.err) ||
          !mbar_wait(&full[stage], (n / S) & 1, abort_flag, a.err)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const float kscale =
          reinterpret_cast<const float*>(smem + stage * C::kStageBytes + C::kScaleOff)[row];
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      const int key = kt * 128 + row;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * C::N;
#pragma unroll
      for (int tok = 0; tok < NTOK; ++tok) {
        if (tok < qb.ntok) {
          const float* wt;
          if constexpr (NTOK == 1) {
            wt = wr;
          } else {
            wt = reinterpret_cast<const float*>(smem + C::kOffW + qs * C::kWBytes) + tok * kHeads;
          }
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[32];
            tmem_ld32(tbase + tok * kHeads + half * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 32; h += 2) {
              s0 = fmaf(wt[half * 32 + h], fmaxf(v[h], 0.f), s0);
              s1 = fmaf(wt[half * 32 + h + 1], fmaxf(v[h + 1], 0.f), s1);
            }
          }
          if (key <= qb.p0 + tok && key < a.ld) {
            const float score = (s0 + s1) * kscale;
            a.logits[static_cast<int64_t>(qb.t0 + tok) * a.ld + key] = score;
            if constexpr (NTOK == 1) {
              if (use_hist) atomicAdd(&whist[f32_key(score) >> kHistShift], 1u);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
    __syncwarp();
    if (!aborted) {
      if (lane == 0) mbar_arrive(&qempty[qs]);
      if constexpr (NTOK == 1) {
        if (use_hist) flush_hist(qb.t0);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int NTOK>
static cudaError_t launch_logits_t(const CUtensorMap* tmap_k, const CUtensorMap* tmap_q, SegmentPlan plan,
                                   const LogitsArgs& a, int num_sms, cudaStream_t stream) {
  using C = LogitsCfg<NTOK>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(logits_kernel<NTOK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_pdl(logits_kernel<NTOK>, dim3(num_sms), dim3(C::kThreads), C::kSmemBytes, stream, *tmap_k, *tmap_q,
                    plan, a);
}

cudaError_t launch_logits(int ntok_per_block, const CUtensorMap* tmap_k, const CUtensorMap* tmap_q,
                          SegmentPlan plan, const LogitsArgs& a, int num_sms, cudaStream_t stream) {
  if (ntok_per_block == 1) return launch_logits_t<1>(tmap_k, tmap_q, plan, a, num_sms, stream);
  return launch_logits_t<4>(tmap_k, tmap_q, plan, a, num_sms, stream);
}

}  // namespace dsa
