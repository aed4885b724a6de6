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
//    with warp 2 sharing the K tiles; warp 1 (and warp 3 for decode) issues
//    the MMAs; the remaining warps read TMEM and apply ReLU, the w'
//    reduction and the K scale, and store fp32 scores.
//  * Decode rows also get their score histogram (pass 1 of the top-k radix
//    select), so the top-k never scans a decode row to find its boundary bin.
//  * Every wait is bounded in time (DSA_DEVERR_TIMEOUT, then an orderly exit).
#include "common.cuh"
#include "kernels.h"

namespace dsa {

// ------------------------------------------------------------------ logits
// FP4: the K cache holds E2M1 codes (4352-byte pages). The TMA box of a page
// is then read with the packed 4-bit type, which lands each row as 128 bytes
// in shared memory (8 code bytes and an 8-byte gap per 16-byte chunk, the
// same 128-byte swizzle) and completes 4096 transaction bytes — the global
// bytes it read. The MMA, the epilogue and the shared-memory layout are the
// FP8 cache's.
template <int NTOK, bool FP4>
struct LogitsCfg {
  static constexpr int N = 64 * NTOK;                     // MMA N: heads x tokens
  static constexpr int kStages = NTOK == 1 ? 8 : 6;       // K-tile ring
  // TMEM accumulator ring: as many N-column accumulators as fit in the 512
  // columns, at most four.
  static constexpr int kAcc = 512 / N < 4 ? 512 / N : 4;
  // Epilogue: teams take the tiles in turn, each team one or two warpgroups
  // that split a tile's tokens (two tokens, 128 columns, per warpgroup), one
  // team per accumulator. A decode team is one warpgroup and two teams suffice
  // (their scores ran no faster with more). Prefill blocks of four tokens
  // (two 256-column accumulators, two teams of two warpgroups) ran faster than
  // blocks of two (four teams, each K tile read twice as often).
  static constexpr int kTeamWG = NTOK <= 2 ? 1 : NTOK / 2;  // warpgroups per team
  static constexpr int kTeams = NTOK == 1 ? 2 : kAcc;
  static constexpr int kEpiWG = kTeams * kTeamWG;
  static constexpr int kTokPerWG = NTOK / kTeamWG;          // tokens of a tile one warpgroup reduces
  static constexpr int kEpiWarps = 4 * kEpiWG;
  // K-tile producers: warp 0 (which also loads the q / w' blocks) and warp 2.
  // Tile n is issued by producer n % kProducers: one issuing thread sustained
  // only about one page copy per 0.2 us whatever its size (8448-byte FP8 and
  // 4352-byte FP4 pages alike), which capped the tile rate (decode8x128k step
  // 54.4 -> 50.9 us with two issuers, prefill4x8k scores 1319 -> 1194 us;
  // three or four measured the same as two on decode).
  // MMA issuers: warp 1 and, for decode, warp 3; tile n is issued by MMA
  // warp n % kMmaWarps into accumulator n % kAcc. A decode tile is only four
  // small MMAs, and one thread's issue loop (waits, four MMAs, commit) took
  // about 0.38 us per tile while the tensor pipe idled.
  // The epilogue warpgroups follow.
  static constexpr int kProducers = 2;
  static constexpr int kMmaWarps = NTOK == 1 ? 2 : 1;
  static constexpr int kEpiWarp0 = kProducers + kMmaWarps;
  static constexpr int kThreads = 32 * kEpiWarp0 + 32 * kEpiWarps;
  static constexpr uint32_t kTmemCols = N * kAcc;         // 256 (decode) or 512 (prefill)
  static constexpr int kStageBytes = 17 * 1024;           // 2 x 8 KB K pages, 4 x 256 B scale rows (gather4)
  static constexpr int kScaleOff = 16384;
  static constexpr int kQBytes = N * kDim;
  static constexpr int kWBytes = NTOK * kHeads * 4;
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffW = kOffQ + 2 * kQBytes;
  static constexpr int kOffBar = kOffW + 2 * kWBytes;
  static constexpr int kNumBars = 2 * kStages + 4 + 2 * kAcc + 1 + kEpiWG;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffMeta = kOffMisc + 16;  // 2 QMeta (2 x 24 B), the slice (4 ints), scan scratch (33 ints)
  // decode: one score histogram per epilogue warpgroup (first radix pass of the top-k)
  static constexpr int kHistBytes = NTOK == 1 ? kEpiWG * kHistBins * 4 : 0;
  static constexpr int kOffHist = (kOffMeta + 2 * 24 + 4 * 4 + 33 * 4 + 127) / 128 * 128;
  static constexpr int kSmemBytes = kOffHist + kHistBytes + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t kIdesc = f8_idesc(128, N, FP4);
  static constexpr int64_t kPage = FP4 ? kFp4PageBytes : kPageBytes;     // bytes per K-cache page
  static constexpr uint32_t kCodeTx = FP4 ? 4096 : 8192;                  // code bytes a page's tensor copy lands
  static constexpr uint32_t kScaleTx = 4 * 256;                           // a tile's gather4 of four scale rows
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation must be a power of two");
  static_assert(kAcc % kMmaWarps == 0, "each MMA warp owns every kMmaWarps-th accumulator");
};

__device__ __forceinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, unsigned long long deadline) {
  const uint32_t addr = smem_u32(bar);
  while (!mbar_try_wait(addr, parity)) {
    if (global_ns() > deadline) return false;
  }
  return true;
}

// The query block whose q / w' tile a q buffer holds, written by the producer
// before it arrives on the buffer's barrier, read by the MMA and epilogue warps.
struct QMeta {
  QBlock qb;
  int32_t tiles;  // tiles of the block inside this CTA's slice
  int32_t kt0;    // the first of them
};

// Decode query block of token t (one token per block): request, position and
// number of 128-key tiles; 0 tiles when the request metadata is inconsistent.
// *first_new = position of the request's first token of this step: pages
// below first_new / 64 hold no slot written in this step.
__device__ __forceinline__ int decode_block(const LogitsArgs& a, int t, QBlock* out, int* first_new = nullptr) {
  // one token per decode request is the common case (request t): its
  // metadata is loaded beside req_id[t] instead of after it
  const int r = __ldg(a.req_id + t);
  const bool spec = t < a.num_decodes;
  int q0 = spec ? __ldg(a.qsl + t) : 0, q1 = spec ? __ldg(a.qsl + t + 1) : 0, sl = spec ? __ldg(a.seq_lens + t) : 0;
  QBlock b{r, t, 1, 0};
  int tiles = 0, fn = 0;
  if (r >= 0 && r < a.num_decodes) {
    if (r != t) {
      q0 = __ldg(a.qsl + r);
      q1 = __ldg(a.qsl + r + 1);
      sl = __ldg(a.seq_lens + r);
    }
    if (t >= q0 && t < q1 && sl >= q1 - q0 && static_cast<int64_t>(sl) <= a.bt_stride * kBlock) {
      fn = sl - (q1 - q0);
      b.p0 = fn + (t - q0);
      tiles = (b.p0 + 1 + 127) / 128;
    }
  }
  *out = b;
  if (first_new != nullptr) *first_new = fn;
  return tiles;
}

// Decode segment: this CTA's slice {it_begin, it_end, first token, first tile}
// of the flat (token, tile) list, computed by the whole CTA from the request
// metadata. slice[] is shared memory; scan[] is block-scan scratch.
__device__ void decode_slice(const LogitsArgs& a, int* slice, int* scan) {
  const int T = a.num_dec_tokens;
  const int nt = blockDim.x, tid = threadIdx.x;
  if (blockIdx.x == 0 && tid == 0 && (__ldg(a.qsl) != 0 || __ldg(a.qsl + a.num_decodes) != T))
    flag_error(a.err, DSA_DEVERR_SEQ_RANGE);
  if (tid == 0) {
    slice[2] = 0;
    slice[3] = 0;
  }
  // pass 1: the segment's tile count (and, when the tokens fit in one chunk,
  // each thread's exclusive prefix, so no second pass is needed)
  int total = 0, tot, my_tiles = 0, my_prefix = 0;
  for (int c0 = 0; c0 < T; c0 += nt) {
    const int t = c0 + tid;
    QBlock b;
    const int tiles = t < T ? decode_block(a, t, &b) : 0;
    if (t < T && tiles == 0 && blockIdx.x == 0) flag_error(a.err, DSA_DEVERR_SEQ_RANGE);
    const int incl = block_scan_incl(tiles, scan, &tot);
    my_tiles = tiles;
    my_prefix = total + incl - tiles;
    total += tot;
  }
  const int b0 = static_cast<int>(static_cast<int64_t>(total) * blockIdx.x / gridDim.x);
  const int b1 = static_cast<int>(static_cast<int64_t>(total) * (blockIdx.x + 1) / gridDim.x);
  if (tid == 0) {
    slice[0] = b0;
    slice[1] = b1;
  }
  if (b0 < b1) {
    if (T <= nt) {
      if (tid < T && my_tiles > 0 && my_prefix <= b0 && b0 < my_prefix + my_tiles) {
        slice[2] = tid;
        slice[3] = b0 - my_prefix;
      }
    } else {
      int carry = 0;
      for (int c0 = 0; c0 < T; c0 += nt) {
        const int t = c0 + tid;
        QBlock b;
        const int tiles = t < T ? decode_block(a, t, &b) : 0;
        const int incl = block_scan_incl(tiles, scan, &tot);
        const int s = carry + incl - tiles;
        if (t < T && tiles > 0 && s <= b0 && b0 < s + tiles) {
          slice[2] = t;
          slice[3] = b0 - s;
        }
        carry += tot;
      }
    }
  }
  __syncthreads();
}

template <int NTOK, bool FP4>
__global__ void __launch_bounds__(LogitsCfg<NTOK, FP4>::kThreads, 1)
    logits_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_s,
                  const __grid_constant__ CUtensorMap tmap_q,
                  SegmentPlan plan, LogitsArgs a) {
  using C = LogitsCfg<NTOK, FP4>;
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
  uint64_t* wgbar = done + 1;  // per epilogue warpgroup: its 4 warps meet around the histogram
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  QMeta* qmeta = reinterpret_cast<QMeta*>(smem + C::kOffMeta);
  int* slice = reinterpret_cast<int*>(smem + C::kOffMeta + 2 * sizeof(QMeta));
  int* scan = slice + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool is_producer = warp == 0 || (warp >= 2 && warp < 1 + C::kProducers);
  const bool is_mma = warp == 1 || (warp >= 1 + C::kProducers && warp < C::kEpiWarp0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      // the tile's epilogue warps, after its MMAs completed (tfull) and they read its scales
      mbar_init(&empty[s], 4 * C::kTeamWG);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], C::kMmaWarps + C::kEpiWarps);
    }
    for (int c = 0; c < A; ++c) {
      mbar_init(&tfull[c], 1);
      mbar_init(&tempty[c], 4 * C::kTeamWG);
    }
    mbar_init(done, C::kMmaWarps);
    for (int g = 0; g < C::kEpiWG; ++g) mbar_init(&wgbar[g], 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_s);
    prefetch_tmap(&tmap_q);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // This CTA's slice. Everything before pdl_wait() may overlap the previous
  // kernel of the stream (programmatic dependent launch): the decode slice
  // needs only the request metadata, an input of the step, and the producer
  // may already fetch K pages that hold no slot written in this step. The q
  // codes, the weights, the new K rows and the prefill plan are read after it.
  int it_begin, it_end, j0, kt0;
  if constexpr (NTOK == 1) {
    decode_slice(a, slice, scan);
    it_begin = slice[0];
    it_end = slice[1];
    j0 = slice[2];
    kt0 = slice[3];
  } else {
    pdl_wait();
    const CtaWork cw = plan.cta[blockIdx.x];
    it_begin = cw.it_begin;
    it_end = cw.it_end;
    j0 = cw.qb0;
    kt0 = cw.kt0;
  }
  const int items = it_end - it_begin;  // tiles of this CTA (an empty slice runs no loop)
  pdl_launch_dependents();
  if constexpr (NTOK == 1) {
    if (!is_producer) pdl_wait();  // the producers wait after their early loads
  }

  // Issue the loads of tile kt of a block (pages 2kt, 2kt+1) into a stage:
  // each page's codes by a tensor copy, and both pages' scale rows by one
  // gather4 of the scale map (rows id0, id1, id0, id1; the last two land in the
  // stage's spare kilobyte, unread). Three copies a tile instead of four: in a
  // streaming probe on 40 SMs the per-SM page rate rose from 50.5 to 60.7 GB/s
  // (the copy issue rate, not the bytes, bounds a CTA's K pipeline). A missing
  // or invalid page's scale row is replaced by a valid one: its keys are not
  // stored.
  auto issue_tile = [&](int stage, int kt, int npages, int id0, int id1) {
    uint8_t* st = smem + stage * C::kStageBytes;
    const bool in1 = 2 * kt + 1 < npages;
    const bool v0 = id0 >= 0 && id0 < a.num_blocks;
    const bool v1 = in1 && id1 >= 0 && id1 < a.num_blocks;
    if (!v0 || (in1 && !v1)) flag_error(a.err, DSA_DEVERR_BLOCK_RANGE);
    const int g0 = v0 ? id0 : 0, g1 = v1 ? id1 : g0;
    mbar_arrive_expect_tx(&full[stage], (v0 ? C::kCodeTx : 0) + (v1 ? C::kCodeTx : 0) + C::kScaleTx);
    if (v0) tma_load_3d(st, &tmap_k, &full[stage], 0, 0, id0);
    if (v1) tma_load_3d(st + 8192, &tmap_k, &full[stage], 0, 0, id1);
    tma_gather4_2d(st + C::kScaleOff, &tmap_s, &full[stage], g0, g1, g0, g1);
  };

  if (is_producer) {
    // ------------------------------------------------------------ producers
    const int pi = warp == 0 ? 0 : warp - 1;  // this producer issues tiles n with n % np == pi
    constexpr int np = C::kProducers;
    auto block_at = [&](int j, QBlock* qb, int* first_new) -> int {  // block j and its tile count
      if constexpr (NTOK == 1) {
        return decode_block(a, j, qb, first_new);
      } else {
        *qb = plan.qb[j];
        *first_new = 0;
        return plan.tile_start[j + 1] - plan.tile_start[j];
      }
    };
    int j = j0, kt = kt0, n = 0, qcount = 0;
    bool ok = true;
    QBlock qb{};
    int first_new = 0;
    int block_tiles = items > 0 ? block_at(j, &qb, &first_new) : 0;
    // decode: before the wait, the producers fill the ring with their tiles
    // of the first block whose two pages lie below the first page this step
    // writes (the block table and the lengths are inputs of the step)
    int npre = 0;
    if constexpr (NTOK == 1) {
      const int safe_pages = first_new / kBlock;
      int cnt = min(min(block_tiles - kt, items), S);
      while (cnt > 0 && 2 * (kt + cnt - 1) + 1 >= safe_pages) --cnt;
      if (cnt > 0) {
        const int32_t* bt_row = a.block_table + static_cast<int64_t>(qb.req) * a.bt_stride;
        const int32_t id = lane < 2 * cnt ? __ldg(bt_row + 2 * kt + lane) : -1;
        for (int e = pi; e < cnt; e += np) {
          const int id0 = __shfl_sync(0xffffffffu, id, 2 * e);
          const int id1 = __shfl_sync(0xffffffffu, id, 2 * e + 1);
          if (lane == 0) issue_tile(e, kt + e, 2 * (kt + e) + 2, id0, id1);
        }
      }
      npre = max(cnt, 0);
      pdl_wait();
    }
    while (ok && n < items) {
      const int in_slice = min(block_tiles - kt, items - n);
      if (pi == 0) {  // the block's q codes and w'
        const int qs = qcount & 1;
        int w = 1;
        if (lane == 0) w = mbar_wait(&qempty[qs], ((qcount >> 1) & 1) ^ 1, abort_flag, a.err);
        if (!__shfl_sync(0xffffffffu, w, 0)) break;
        if (lane == 0) {
          qmeta[qs] = QMeta{qb, in_slice, kt};
          mbar_arrive_expect_tx(&qfull[qs], C::kQBytes + qb.ntok * kHeads * 4);
          tma_load_2d(smem + C::kOffQ + qs * C::kQBytes, &tmap_q, &qfull[qs], 0, qb.t0 * kHeads);
          bulk_load(smem + C::kOffW + qs * C::kWBytes, a.w_folded + static_cast<int64_t>(qb.t0) * kHeads,
                    qb.ntok * kHeads * 4, &qfull[qs]);
        }
        ++qcount;
      }
      // page ids of this block, 32 at a time across the warp, one batch ahead
      const int npages = (qb.p0 + qb.ntok + kBlock - 1) / kBlock;
      const int32_t* bt_row = a.block_table + static_cast<int64_t>(qb.req) * a.bt_stride;
      int batch = (2 * kt) >> 5;
      int p = batch * 32 + lane;
      int32_t cur_ids = p < npages ? __ldg(bt_row + p) : -1;
      int32_t nxt_ids = p + 32 < npages ? __ldg(bt_row + p + 32) : -1;
      for (int e = 0; e < in_slice; ++e, ++n, ++kt) {
        if (n < npre || n % np != pi) continue;  // loaded before the wait, or another producer's
        const int stage = n % S;
        int w = 1;
        if (lane == 0) w = mbar_wait(&empty[stage], ((n / S) & 1) ^ 1, abort_flag, a.err);
        if (!__shfl_sync(0xffffffffu, w, 0)) {
          ok = false;
          break;
        }
        while (((2 * kt) >> 5) != batch) {  // moved on to a later batch of 32 page ids
          ++batch;
          cur_ids = nxt_ids;
          p = (batch + 1) * 32 + lane;
          nxt_ids = p < npages ? __ldg(bt_row + p) : -1;
        }
        const int id0 = __shfl_sync(0xffffffffu, cur_ids, (2 * kt) & 31);
        const int id1 = __shfl_sync(0xffffffffu, cur_ids, (2 * kt + 1) & 31);
        if (lane == 0) issue_tile(stage, kt, npages, id0, id1);
      }
      ++j;
      kt = 0;
      if (ok && n < items) block_tiles = block_at(j, &qb, &first_new);
    }
    if (lane == 0 && *abort_flag) {
      // let the copies this producer issued land before the CTA's shared memory goes away
      const unsigned long long deadline = global_ns() + kWaitLimitNs;
      for (int m = (n > S ? n - S : 0); m < n; ++m)
        if (m % np == pi) mbar_wait_until(&full[m % S], (m / S) & 1, deadline);
      for (int m = n; m < npre; ++m)
        if (m % np == pi) mbar_wait_until(&full[m % S], 0, deadline);
      if (pi == 0 && qcount > 0) mbar_wait_until(&qfull[(qcount - 1) & 1], ((qcount - 1) >> 1) & 1, deadline);
    }
  } else if (is_mma) {
    // ------------------------------------------------------------ MMA issuers
    const int mi = warp == 1 ? 0 : warp - C::kProducers;  // issues tiles n with n % kMmaWarps == mi
    if (lane == 0) {
      int n = 0, qcount = 0;
      bool ok = true;
      while (ok && n < items) {
        const int qs = qcount & 1;
        if (!mbar_wait(&qfull[qs], (qcount >> 1) & 1, abort_flag, a.err)) break;
        ++qcount;
        const int in_slice = qmeta[qs].tiles;
        const uint32_t sb = smem_u32(smem + C::kOffQ + qs * C::kQBytes);
        for (int e = 0; e < in_slice; ++e, ++n) {
          if (n % C::kMmaWarps != mi) continue;
          const int stage = n % S;
          const int acc = n % A;
          if (!mbar_wait(&full[stage], (n / S) & 1, abort_flag, a.err) ||
              !mbar_wait(&tempty[acc], ((n / A) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(acc * C::N);
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8(d, sw128_kmajor_desc(sa + 32 * k), sw128_kmajor_desc(sb + 32 * k), C::kIdesc, k > 0 ? 1u : 0u);
          mma_commit(&tfull[acc]);
        }
        if (ok) mma_commit(&qempty[qs]);  // the block's q / w' buffer is free once its MMAs are done
      }
      mma_commit(done);  // completes once every MMA issued above has finished
      mbar_wait_until(done, 0, global_ns() + kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int g = (warp - C::kEpiWarp0) >> 2;          // warpgroup
    const int team = g / C::kTeamWG;                   // takes every kTeams-th tile
    const int tok0 = (g % C::kTeamWG) * C::kTokPerWG;  // the tokens of a tile this warpgroup reduces
    const int quarter = warp & 3;                      // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;               // key within the tile
    const int part = (warp - C::kEpiWarp0) & 3;        // this warp's quarter of the group's histogram bins
    // decode rows: the warpgroup's histogram of the keys of its stored
    // scores, added to the row's global histogram when the group leaves the row
    uint32_t* ghist = reinterpret_cast<uint32_t*>(smem + C::kOffHist) + g * kHistBins;
    uint32_t hphase = 0;
    // the group's 4 warps meet (bounded wait; false once the CTA aborts)
    auto group_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&wgbar[g]);
      int w = 1;
      if (lane == 0) w = mbar_wait(&wgbar[g], hphase & 1, abort_flag, a.err);
      ++hphase;
      return __shfl_sync(0xffffffffu, w, 0) != 0;
    };
    int n = 0, qcount = 0;
    bool ok = true;
    while (ok && n < items) {
      const int qs = qcount & 1;
      if (!mbar_wait(&qfull[qs], (qcount >> 1) & 1, abort_flag, a.err)) break;
      ++qcount;
      const QMeta meta = qmeta[qs];
      const QBlock qb = meta.qb;
      const float* wq = reinterpret_cast<const float*>(smem + C::kOffW + qs * C::kWBytes);  // w' of the block
      bool use_hist = false;
      if constexpr (NTOK == 1) {
        use_hist = a.hist != nullptr && qb.t0 < a.hist_rows;
        if (use_hist) {
          uint4* z = reinterpret_cast<uint4*>(ghist) + part * (kHistBins / 16);
#pragma unroll
          for (int b = lane; b < kHistBins / 16; b += 32) z[b] = make_uint4(0, 0, 0, 0);
          if (!group_sync()) break;
        }
      }
      for (int e = 0; e < meta.tiles; ++e, ++n) {
        if ((n % C::kTeams) != team) continue;
        const int stage = n % S;
        const int acc = n % A;
        if (!mbar_wait(&tfull[acc], (n / A) & 1, abort_flag, a.err) ||
            !mbar_wait(&full[stage], (n / S) & 1, abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float kscale = reinterpret_cast<const float*>(smem + stage * C::kStageBytes + C::kScaleOff)[row];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        const int key = (meta.kt0 + e) * 128 + row;
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * C::N;
        // the warpgroup's tokens in halves of 32 heads: each half's TMEM load
        // is in flight while the previous half is reduced (columns of tokens
        // past the block's end are read too, and not stored)
        auto reduce32 = [&](const uint32_t (&r)[32], const float4* w, uint64_t& s01, uint64_t& s23) {
#pragma unroll
          for (int h = 0; h < 32; h += 4) {
            const float4 w4 = w[h / 4];  // the same address across the warp: one broadcast load
            s01 = fma_f32x2(pack_f32x2(w4.x, w4.y),
                            pack_f32x2(fmaxf(__uint_as_float(r[h]), 0.f), fmaxf(__uint_as_float(r[h + 1]), 0.f)), s01);
            s23 = fma_f32x2(pack_f32x2(w4.z, w4.w),
                            pack_f32x2(fmaxf(__uint_as_float(r[h + 2]), 0.f), fmaxf(__uint_as_float(r[h + 3]), 0.f)),
                            s23);
          }
        };
        uint32_t ra[32], rb[32];
        tmem_ld32(tbase + tok0 * kHeads, ra);
        tmem_wait32(ra);
#pragma unroll
        for (int tt = 0; tt < C::kTokPerWG; ++tt) {
          const int tok = tok0 + tt;
          const float4* wt = reinterpret_cast<const float4*>(wq + tok * kHeads);
          uint64_t s01 = 0, s23 = 0;
          tmem_ld32(tbase + tok * kHeads + 32, rb);
          reduce32(ra, wt, s01, s23);
          tmem_wait32(rb);
          if (tt + 1 < C::kTokPerWG) {
            tmem_ld32(tbase + (tok + 1) * kHeads, ra);
          } else {
            // this warp's last columns are in registers: hand the accumulator
            // back to the MMA before reducing them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
          reduce32(rb, wt + 8, s01, s23);
          if (tt + 1 < C::kTokPerWG) tmem_wait32(ra);
          if (tok < qb.ntok && key <= qb.p0 + tok && key < a.ld) {
            const float2 p01 = unpack_f32x2(s01), p23 = unpack_f32x2(s23);
            const float score = ((p01.x + p01.y) + (p23.x + p23.y)) * kscale;
            a.logits[static_cast<int64_t>(qb.t0 + tok) * a.ld + key] = score;
            if constexpr (NTOK == 1) {
              if (use_hist) atomicAdd(&ghist[f32_key(score) >> kHistShift], 1u);
            }
          }
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[qs]);  // done with this block's q / w' buffer
      if constexpr (NTOK == 1) {
        if (use_hist) {  // the group's adds are done: add its nonzero bins to the row's histogram
          if (!group_sync()) break;
          uint32_t* dst = a.hist + static_cast<int64_t>(qb.t0) * kHistBins + part * (kHistBins / 4);
          const uint4* src = reinterpret_cast<const uint4*>(ghist) + part * (kHistBins / 16);
#pragma unroll
          for (int b = lane; b < kHistBins / 16; b += 32) {
            const uint4 v = src[b];
            if (v.x) atomicAdd(dst + 4 * b, v.x);
            if (v.y) atomicAdd(dst + 4 * b + 1, v.y);
            if (v.z) atomicAdd(dst + 4 * b + 2, v.z);
            if (v.w) atomicAdd(dst + 4 * b + 3, v.w);
          }
          if (!group_sync()) break;  // read before the next block zeroes it
        }
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

template <int NTOK, bool FP4>
static cudaError_t launch_logits_t(const CUtensorMap* tmap_k, const CUtensorMap* tmap_s, const CUtensorMap* tmap_q,
                                   SegmentPlan plan, const LogitsArgs& a, int num_sms, cudaStream_t stream) {
  using C = LogitsCfg<NTOK, FP4>;
  static uint64_t configured = 0;  // devices whose limit is raised
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(logits_kernel<NTOK, FP4>), C::kSmemBytes,
                                   &configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(logits_kernel<NTOK, FP4>, dim3(num_sms), dim3(C::kThreads), C::kSmemBytes, stream, *tmap_k,
                    *tmap_s, *tmap_q, plan, a);
}

cudaError_t launch_logits(int ntok_per_block, bool fp4, const CUtensorMap* tmap_k, const CUtensorMap* tmap_s,
                          const CUtensorMap* tmap_q, SegmentPlan plan, const LogitsArgs& a, int num_sms,
                          cudaStream_t stream) {
  if (ntok_per_block == 1)
    return fp4 ? launch_logits_t<1, true>(tmap_k, tmap_s, tmap_q, plan, a, num_sms, stream)
               : launch_logits_t<1, false>(tmap_k, tmap_s, tmap_q, plan, a, num_sms, stream);
  return fp4 ? launch_logits_t<kPrefillTok, true>(tmap_k, tmap_s, tmap_q, plan, a, num_sms, stream)
             : launch_logits_t<kPrefillTok, false>(tmap_k, tmap_s, tmap_q, plan, a, num_sms, stream);
}

}  // namespace dsa
