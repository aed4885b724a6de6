// plan.cu — work planning for the score kernels, and the fused per-layer
// prologue (K quant + cache write, q quant + weight fold, plan) (sm_103a).
//
// The plan splits every request into query blocks (1 token for the decode
// segment, 4 for the prefill segment), counts the 128-key tiles each block
// scores (keys visible to its last token: causal, [0, position]), and cuts the
// flat list of (block, tile) items into one equal slice per persistent CTA of
// the score kernel, so each CTA starts with a single load. Request metadata
// is staged in shared memory so the lookups are not chains of global loads.
#include "common.cuh"
#include "kernels.h"

namespace dsa {

constexpr int kPlanStage = 2048;  // requests per segment staged in shared memory
constexpr int kBlockCost = 1;     // cost of a query block's q / w' load, in tiles

struct PlanSmem {
  int scan[33];
  int qsl[kPlanStage + 1];
  int sl[kPlanStage];
  int base[kPlanStage + 1];
};

__device__ __forceinline__ QBlock make_qblock(const int* qsl, const int* sl, const int* base, int nreq, int r_begin,
                                              int ntok, int j) {
  int lo = 0, hi = nreq - 1;  // last r with base[r] <= j
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= j) lo = mid; else hi = mid - 1;
  }
  const int jj = j - base[lo];
  const int q0 = qsl[lo], ql = qsl[lo + 1] - q0;
  QBlock b;
  b.req = r_begin + lo;
  b.t0 = q0 + jj * ntok;
  b.ntok = min(ntok, ql - jj * ntok);
  b.p0 = sl[lo] - ql + jj * ntok;
  return b;
}

// Plan requests [r_begin, r_end) into query blocks of up to `ntok` tokens.
__device__ void plan_segment(const int32_t* qsl_g, const int32_t* sl_g, int r_begin, int r_end, int ntok,
                             int num_tokens, int64_t bt_stride, int grid, SegmentPlan P, int32_t* err,
                             PlanSmem& S) {
  const int nreq = r_end - r_begin;
  const bool staged = nreq <= kPlanStage;
  if (staged) {
    for (int i = threadIdx.x; i <= nreq; i += blockDim.x) S.qsl[i] = qsl_g[r_begin + i];
    for (int i = threadIdx.x; i < nreq; i += blockDim.x) S.sl[i] = sl_g[r_begin + i];
    __syncthreads();
  }
  const int* qsl = staged ? S.qsl : qsl_g + r_begin;  // request-relative views
  const int* sl = staged ? S.sl : sl_g + r_begin;
  int* base = staged ? S.base : P.req_base;
  int carry = 0, tot;
  for (int b0 = 0; b0 < nreq; b0 += blockDim.x) {
    const int r = b0 + threadIdx.x;
    int c = 0;
    if (r < nreq) {
      const int ql = qsl[r + 1] - qsl[r];
      const int s = sl[r];
      if (ql < 0 || s < ql || static_cast<int64_t>(s) > bt_stride * kBlock || qsl[r] < 0 ||
          qsl[r + 1] > num_tokens) {
        flag_error(err, DSA_DEVERR_SEQ_RANGE);
      } else {
        c = (ql + ntok - 1) / ntok;
      }
    }
    const int incl = block_scan_incl(c, S.scan, &tot);
    if (r < nreq) base[r] = carry + incl - c;
    carry += tot;
  }
  int nqb = carry;
  if (nqb > P.max_qb) {  // metadata inconsistent with the host sizes: plan nothing
    if (threadIdx.x == 0) flag_error(err, DSA_DEVERR_SEQ_RANGE);
    nqb = 0;
  }
  if (threadIdx.x == 0) {
    base[nreq] = nqb;
    *P.nqb = nqb;
  }
  __syncthreads();
  // pass 1: count the tiles of the segment
  int total = 0;
  for (int b0 = 0; b0 < nqb; b0 += blockDim.x) {
    const int j = b0 + threadIdx.x;
    int tiles = 0;
    if (j < nqb) {
      const QBlock b = make_qblock(qsl, sl, base, nreq, r_begin, ntok, j);
      P.qb[j] = b;
      tiles = (b.p0 + b.ntok + 127) / 128;
    }
    block_scan_incl(tiles, S.scan, &tot);
    total += tot;
  }
  for (int c = threadIdx.x; c < grid; c += blockDim.x) P.cta[c] = CtaWork{0, 0, 0, 0};
  __syncthreads();
  // pass 2: tile prefix, and for every CTA the start of its slice. Slices are
  // equal in cost, where a block costs its tiles plus kBlockCost: a CTA whose
  // blocks hold few tiles (the first blocks of a prefill, one tile each) waits
  // on a q / w' load per block, and with equal tiles it finished last.
  const int64_t W = static_cast<int64_t>(total) + static_cast<int64_t>(nqb) * kBlockCost;
  carry = 0;
  for (int b0 = 0; b0 < nqb; b0 += blockDim.x) {
    const int j = b0 + threadIdx.x;
    int tiles = 0;
    if (j < nqb) {
      const QBlock b = make_qblock(qsl, sl, base, nreq, r_begin, ntok, j);
      tiles = (b.p0 + b.ntok + 127) / 128;
    }
    const int incl = block_scan_incl(tiles, S.scan, &tot);
    if (j < nqb) {
      const int s = carry + incl - tiles;
      P.tile_start[j] = s;
      // block j spans costs [ws, ws + kBlockCost + tiles): its load, then its
      // tiles. CTA c starts at cost floor(W*c/grid): the c whose start lies in
      // that span begin at the tile it falls on (the first, if it falls on the load)
      const int64_t ws = static_cast<int64_t>(s) + static_cast<int64_t>(j) * kBlockCost;
      const int64_t c_lo = (ws * grid + W - 1) / W;
      const int64_t c_hi = ((ws + kBlockCost + tiles) * grid + W - 1) / W - 1;
      for (int64_t c = c_lo; c <= c_hi && c < grid; ++c) {
        const int64_t off = W * c / grid - ws - kBlockCost;
        const int kt = off > 0 ? static_cast<int>(off) : 0;
        P.cta[c] = CtaWork{s + kt, 0, j, kt};
      }
    }
    carry += tot;
  }
  if (threadIdx.x == 0) P.tile_start[nqb] = carry;
  __syncthreads();
  // pass 3: each slice ends where the next begins
  for (int c = threadIdx.x; c < grid; c += blockDim.x)
    P.cta[c].it_end = nqb == 0 ? 0 : (c + 1 < grid ? P.cta[c + 1].it_begin : carry);
  __syncthreads();
}

__device__ void plan_batch(const PlanArgs& p, PlanSmem& S) {
  if (threadIdx.x == 0 && p.qsl[p.num_decodes] != p.num_decode_tokens) flag_error(p.err, DSA_DEVERR_SEQ_RANGE);
  // the decode segment is planned by its score kernel; a segment without
  // requests launches no score kernel
  if (p.num_reqs > p.num_decodes)
    plan_segment(p.qsl, p.seq_lens, p.num_decodes, p.num_reqs, kPrefillTok, p.num_tokens, p.bt_stride, p.grid, p.pre, p.err,
                 S);
}

// ---------------------------------------------------------------------------
// One launch per F layer before the scores: CTA 0 plans (first layer of a
// step only; being first it is dispatched first and overlaps the rest); the
// others quantise the q rows with the weight fold (half a warp per 128-value
// row: 16-byte loads, eight rows per warp in flight), the step's K into the
// cache (a warp per row), and zero the decode rows' score histograms and
// top-k counters. One wave: the grid is the CTAs that fit on the GPU at once
// (four per SM at 256 threads and at most 64 registers), each looping over its
// share. Against a warp per q row (8-byte loads, four rows per warp) and two
// waves, prefill4x8k's prologue took 219 -> 136 us (HBM-bound: 837 MB moved,
// 0.91 of the measured copy bandwidth). Four CTAs of up to 64 registers ran
// 143 -> 137 us against five of 48 (stack61 unchanged); issuing the next
// group's loads before quantising the current one ran 140 us, and 3 us slower
// per stack61 F layer.
// Launched as a programmatic dependent of the previous layer's top-k (pdl), it
// quantises while that top-k's last CTAs run, and waits for it only before
// clearing the decode rows' histograms and counters, which the top-k reads.
constexpr int kPrologueThreads = 256;
constexpr int kPrologueMinCtas = 4;

// FP4: the K cache has FP4 pages (a.k_fp4), fixed per instance so that the
// K store of the other format costs no registers.
template <bool FP4>
__global__ void __launch_bounds__(kPrologueThreads, kPrologueMinCtas) prologue_kernel(PrologueArgs a) {
  extern __shared__ __align__(16) uint8_t plan_smem[];
  pdl_launch_dependents();  // the score kernel may start its set-up now
  if (a.plan && blockIdx.x == 0) {
    plan_batch(a.p, *reinterpret_cast<PlanSmem*>(plan_smem));
    return;
  }
  const int first = a.plan ? 1 : 0;
  const int work_ctas = gridDim.x - first;
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(work_ctas) * (kPrologueThreads / 32);
  const int64_t q_rows = a.q != nullptr ? static_cast<int64_t>(a.n_tokens) * kHeads : 0;
  const int64_t k_rows = a.k_new != nullptr ? a.n_tokens : 0;
  const int64_t z_rows = a.hist != nullptr ? a.hist_rows : 0;
  // jobs: groups of 8 q rows (two rows per 16-byte load of the warp, four
  // loads issued together), then K rows, then zeroing
  constexpr int kGroup = 8;
  const int half = lane >> 4, hl = lane & 15;
  static_assert(kHeads % kGroup == 0, "a group of q rows belongs to one token");
  const int64_t q_groups = (q_rows + kGroup - 1) / kGroup;
  const int64_t jobs = q_groups + k_rows + z_rows;
  for (int64_t j = static_cast<int64_t>(blockIdx.x - first) * (kPrologueThreads / 32) + (threadIdx.x >> 5); j < jobs;
       j += warps) {
    if (j < q_groups) {
      // q_rows is a multiple of 64: every group is whole and heads of one token
      const int64_t r0 = j * kGroup;
      constexpr int kLoads = kGroup / 2;
      uint4 raw[kLoads];
      float wv[kLoads];
#pragma unroll
      for (int u = 0; u < kLoads; ++u) {
        const int64_t r = r0 + 2 * u + half;
        raw[u] = __ldg(reinterpret_cast<const uint4*>(a.q + r * kDim) + hl);
        wv[u] = 0.0f;
        if (hl == 0) {  // w[token][head]: row r is head r % 64 of token r / 64
          const int64_t wi = (r / kHeads) * a.w_row_stride + (r % kHeads);
          wv[u] = a.w_bf16 ? __bfloat162float(__ldg(static_cast<const __nv_bfloat16*>(a.w) + wi))
                           : __ldg(static_cast<const float*>(a.w) + wi);
        }
      }
      if (a.rope.cos_sin != nullptr) {
        const float* cs = rope_row(a.rope, r0 / kHeads, a.err, lane);
        if (cs != nullptr) {
#pragma unroll
          for (int u = 0; u < kLoads; ++u) raw[u] = rope_row_half(raw[u], cs);
        }
      }
#pragma unroll
      for (int u = 0; u < kLoads; ++u) {
        const int64_t r = r0 + 2 * u + half;
        float s;
        const uint2 codes = quant_row_half(raw[u], &s);
        reinterpret_cast<uint2*>(a.q_fp8 + r * kDim)[hl] = codes;
        if (hl == 0) a.w_folded[r] = __fmul_rn(__fmul_rn(__fmul_rn(wv[u], s), a.softmax_scale), 0.125f);
      }
    } else if (j < q_groups + k_rows) {
      const int64_t t = j - q_groups;
      const int64_t slot = __ldg(a.slot_mapping + t);
      if (slot < 0) continue;
      if (slot >= a.num_blocks * kBlock) {
        if (lane == 0) flag_error(a.err, DSA_DEVERR_SLOT_RANGE);
        continue;
      }
      uint2 raw = __ldg(reinterpret_cast<const uint2*>(a.k_new + t * a.k_row_stride) + lane);
      if (a.rope.cos_sin != nullptr) {
        const float* cs = rope_row(a.rope, t, a.err, lane);
        if (cs != nullptr) raw = rope_row_lane(raw, cs);
      }
      quant_store_k_row(a.k_cache, slot, raw, FP4, lane);
    } else {
      // the previous layer's top-k may still read these rows: wait for it
      // (the q codes, the cache rows and the plan above are not read by it)
      pdl_wait();
      const int64_t t = j - q_groups - k_rows;
      uint4* h = reinterpret_cast<uint4*>(a.hist + t * kHistBins);
      uint4* h2 = reinterpret_cast<uint4*>(a.hist2 + t * kHistBins);
#pragma unroll 4
      for (int b = lane; b < kHistBins / 4; b += 32) {
        h[b] = make_uint4(0, 0, 0, 0);
        h2[b] = make_uint4(0, 0, 0, 0);
      }
      if (lane == 0) reinterpret_cast<uint4*>(a.counters)[t] = make_uint4(0, 0, 0, 0);
    }
  }
}

// Prologue CTAs resident on one SM (the occupancy of the instance, with the
// plan's shared memory), found once.
template <bool FP4>
int prologue_resident() {
  static const int n = [] {
    int r = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, prologue_kernel<FP4>, kPrologueThreads, sizeof(PlanSmem)) !=
        cudaSuccess) {
      cudaGetLastError();  // not sticky; leave no error for the launch check
      r = 0;
    }
    return r < 1 ? kPrologueMinCtas : r;
  }();
  return n;
}

cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t stream) {
  if (a.plan && (a.p.grid < 1 || a.p.grid > kMaxCtas)) return cudaErrorInvalidValue;
  const int64_t q_groups = a.q != nullptr ? (static_cast<int64_t>(a.n_tokens) * kHeads + 7) / 8 : 0;
  const int64_t jobs = q_groups + (a.k_new != nullptr ? a.n_tokens : 0) + (a.hist != nullptr ? a.hist_rows : 0);
  int64_t quant = (jobs + kPrologueThreads / 32 - 1) / (kPrologueThreads / 32);  // one job per warp, if it fits
  if (quant < 1) quant = 1;
  const int64_t wave = static_cast<int64_t>(a.num_sms > 0 ? a.num_sms : 1) *
                           (a.k_fp4 ? prologue_resident<true>() : prologue_resident<false>()) - (a.plan ? 1 : 0);
  if (quant > wave) quant = wave > 1 ? wave : 1;  // every CTA resident at once; the rest loops
  const size_t smem = a.plan ? sizeof(PlanSmem) : 0;
  static_assert(sizeof(PlanSmem) <= 48 * 1024, "plan staging fits the default dynamic shared memory");
  const unsigned grid = static_cast<unsigned>(quant + (a.plan ? 1 : 0));
  if (a.pdl)
    return a.k_fp4 ? launch_pdl(prologue_kernel<true>, dim3(grid), dim3(kPrologueThreads), smem, stream, a)
                   : launch_pdl(prologue_kernel<false>, dim3(grid), dim3(kPrologueThreads), smem, stream, a);
  if (a.k_fp4)
    prologue_kernel<true><<<grid, kPrologueThreads, smem, stream>>>(a);
  else
    prologue_kernel<false><<<grid, kPrologueThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
