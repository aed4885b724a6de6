// select.cuh — exact per-row top-k by radix select over order-preserving
// 32-bit keys of fp32 scores (a > b iff key(a) > key(b)), shared by the top-k
// kernels: the per-row top-k and the multi-CTA decode select (sm_103a).
//
// The top-k op of "IndexCache：DeepSeek 稀疏注意力中的跨层索引复用" (atomage.cn)
// fills a row of the shared `topk_indices_buffer` with the ids of the
// `index_topk` highest-scoring keys, -1 past the visible keys; "vllm.v1.
// attention.backends.mla.index_group" (`_convert_once`) gives the consumers
// physical slots, block_table[req][id/64] * block_stride_rows + id%64. Ids are
// emitted in no particular order.
//
// Pass 1 bins the keys by their top 11 bits; the bin holding the k-th
// largest key (the boundary bin) is found by a block-wide scan from the top.
// Every key above that bin is taken in one pass while the bin's keys are
// gathered; two more passes (11 and 10 bits) on the gathered keys find the
// k-th key exactly, and the keys above it plus as many equal keys as are
// still needed are taken. The ids are collected in shared memory and written
// out (with their physical slots) in one coalesced pass.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace dsa {

constexpr int kSelBins = kHistBins;  // 2048: pass-1 bins = the score kernel's histograms
constexpr int kCandCap = 4096;       // most boundary-bin keys ever gathered in shared memory
constexpr int kMaxTopk = 4096;       // largest k the library accepts

// Scalars of one selection, in shared memory.
struct SelState {
  uint32_t sm[33];  // scan scratch
  int bin;
  uint32_t above, cnt, eq;
  uint32_t binc;  // the count in bin `bin`
};

// Bin b, scanning from the top, at which the running count reaches `need`;
// s.above = the count in bins above b, s.binc = the count in b. Ends with
// __syncthreads(), after which hist is no longer read. Each
// thread reads its kPer bins with vector loads (hist 16-byte aligned) and
// searches them in registers (prefill4x8k top-k 546 -> 486 us against one
// scalar load per bin, read twice).
template <int NT, int BINS = kSelBins>
__device__ void find_bin(const uint32_t* hist, uint32_t need, SelState& s) {
  static_assert(NT % 32 == 0 && NT / 32 <= 32, "block size");
  constexpr int kPer = BINS / NT;  // bins per thread; thread 0 holds the top bins
  const int tid = threadIdx.x;
  const int lane = tid & 31, wid = tid >> 5;
  const int hi = BINS - kPer * tid;  // bins [hi - kPer, hi)
  static_assert(kPer * NT == BINS && (kPer % 4 == 0 || kPer <= 2), "vector loads of the thread's bins");
  uint32_t v[kPer];  // v[b] = hist[hi - 1 - b]
  if constexpr (kPer == 1) {
    v[0] = hist[hi - 1];
  } else if constexpr (kPer % 4 == 0) {
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q) {
      const uint4 w = reinterpret_cast<const uint4*>(hist + hi - kPer)[q];
      v[kPer - 1 - 4 * q] = w.x;
      v[kPer - 2 - 4 * q] = w.y;
      v[kPer - 3 - 4 * q] = w.z;
      v[kPer - 4 - 4 * q] = w.w;
    }
  } else {
    const uint2 w = *reinterpret_cast<const uint2*>(hist + hi - 2);
    v[1] = w.x;
    v[0] = w.y;
  }
  uint32_t local = 0;
#pragma unroll
  for (int b = 0; b < kPer; ++b) local += v[b];
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s.sm[wid] = incl;
  __syncthreads();
  // every warp sums the totals of the warps before it (one barrier, not two)
  incl += __reduce_add_sync(0xffffffffu, lane < wid ? s.sm[lane] : 0u);
  uint32_t above = incl - local;
  if (above < need && need <= incl) {
#pragma unroll
    for (int b = 0; b < kPer; ++b) {
      const uint32_t c = v[b];
      if (above + c >= need) {
        s.bin = hi - 1 - b;
        s.above = above;
        s.binc = c;
        break;
      }
      above += c;
    }
  }
  __syncthreads();
}

// Exclusive prefix sum of v over the block and the block's total, with one
// barrier: every warp sums the totals of the warps before it. sm (NT/32
// words) must not be rewritten before a later barrier.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_sum(uint32_t v, uint32_t* sm, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) sm[wid] = incl;
  __syncthreads();
  const uint32_t w = lane < NT / 32 ? sm[lane] : 0u;
  *total = __reduce_add_sync(0xffffffffu, w);
  return incl - v + __reduce_add_sync(0xffffffffu, lane < wid ? w : 0u);
}

// Where a row's ids go: logical ids, and optionally physical slots.
struct RowOut {
  int32_t* orow;          // [topk] logical ids
  int32_t* prow;          // [topk] physical slots, or nullptr
  const int32_t* bt_row;  // the request's block-table row (global or shared memory)
  int64_t bt_stride;
  int stride_rows;
};

// Physical slot of logical id `id` >= 0 through the row's block table; -1,
// flagged, when its page has no block.
__device__ __forceinline__ int32_t phys_of(const RowOut& o, int id, bool* bad) {
  const int64_t page = id / kBlock;
  const int32_t blk = page < o.bt_stride ? o.bt_row[page] : -1;
  if (blk < 0) *bad = true;
  return blk < 0 ? -1 : blk * o.stride_rows + id % kBlock;
}

__device__ __forceinline__ void emit(const RowOut& o, uint32_t pos, int id, bool* bad) {
  o.orow[pos] = id;
  if (o.prow != nullptr) o.prow[pos] = phys_of(o, id, bad);
}

// Whether a row's ids can go out in 16-byte stores: k a multiple of 4 (the
// library requires it) and both output rows 16-byte aligned (required of the
// caller's buffers, checked here as well).
__device__ __forceinline__ bool rows_vec4(const RowOut& o, int topk) {
  return (topk & 3) == 0 && ((reinterpret_cast<uintptr_t>(o.orow) | reinterpret_cast<uintptr_t>(o.prow)) & 15u) == 0;
}

// Rows with at most k visible keys: every key, then -1. Four consecutive ids
// per thread and 16-byte stores: the four lie in one page, so they take one
// block-table entry (prefill4x8k, whose 32768 rows hold 8192 short ones:
// top-k 417 -> 413 us). The same 16-byte stores for the selected ids, four
// block-table lookups per thread, spilled registers in the 256-thread kernel
// and ran slower (425 us).
__device__ __forceinline__ void write_short_row(int n, int topk, const RowOut& o, bool* bad) {
  if (rows_vec4(o, topk)) {
#pragma unroll 2
    for (int i = 4 * static_cast<int>(threadIdx.x); i < topk; i += 4 * static_cast<int>(blockDim.x)) {
      reinterpret_cast<int4*>(o.orow)[i >> 2] =
          make_int4(i < n ? i : -1, i + 1 < n ? i + 1 : -1, i + 2 < n ? i + 2 : -1, i + 3 < n ? i + 3 : -1);
      if (o.prow != nullptr) {
        int4 p = make_int4(-1, -1, -1, -1);
        if (i < n) {
          const int64_t page = i / kBlock;
          const int32_t blk = page < o.bt_stride ? o.bt_row[page] : -1;
          if (blk < 0) *bad = true;
          if (blk >= 0) {
            const int b = blk * o.stride_rows + i % kBlock;
            p = make_int4(b, i + 1 < n ? b + 1 : -1, i + 2 < n ? b + 2 : -1, i + 3 < n ? b + 3 : -1);
          }
        }
        reinterpret_cast<int4*>(o.prow)[i >> 2] = p;
      }
    }
    return;
  }
  for (int i = threadIdx.x; i < topk; i += blockDim.x) {
    if (i < n) {
      emit(o, i, i, bad);
    } else {
      o.orow[i] = -1;
      if (o.prow != nullptr) o.prow[i] = -1;
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

// Ids collected in shared memory go out in one coalesced pass (positions
// never filled, which consistent histograms rule out, become -1).
template <int NT>
__device__ void write_ids(const uint32_t* oid, int topk, const RowOut& o, bool* bad) {
  for (int i = threadIdx.x; i < topk; i += NT) {
    const int id = static_cast<int>(oid[i]);
    if (id >= 0) {
      emit(o, static_cast<uint32_t>(i), id, bad);
    } else {
      o.orow[i] = -1;
      if (o.prow != nullptr) o.prow[i] = -1;
    }
  }
}

// Levels that resolve the key's last 21 bits inside the boundary bin: 11 + 10
// bits with 2048 bins for 1024-thread rows; 8 + 8 + 5 bits with 256 bins (one
// per thread) for 256-thread rows, whose boundary bins hold a few hundred keys
// (prefill4x8k top-k 455 -> 441 us: a 256-bin search costs a fraction of a
// 2048-bin one). Level l bins a key by its kWidth<l> bits from bit kShift<l> up.
template <int NT>
struct Levels {
  static constexpr bool kWide = NT >= 1024;
  static constexpr int kCount = kWide ? 2 : 3;
  static constexpr int kBins = kWide ? kSelBins : 256;
  static constexpr int kShift0 = kWide ? 10 : 13, kShift1 = kWide ? 0 : 5, kShift2 = 0;
  static constexpr int kWidth0 = kWide ? 11 : 8, kWidth1 = kWide ? 10 : 8, kWidth2 = 5;
  __device__ static __forceinline__ uint32_t first_bin(uint32_t key) {
    return (key >> kShift0) & ((1u << kWidth0) - 1u);
  }
};

// Passes 2 and 3 on the boundary bin b1's keys cand_key(0..m) (ids cand_id),
// bin_count of them, of which `need` are still to be taken after the n_up keys
// above the bin; the keys above the k-th and as many ties as needed go to
// put(position, id) at positions n_up, n_up + 1, ... (below topk). hist is
// reused for the levels' histograms. With kFirstBuilt the caller has already
// binned the bin's keys by Levels<NT>::first_bin into hist, reset s.bin,
// s.above, s.cnt = n_up and s.eq = 0, and synchronised; else hist holds pass 1
// on entry.
template <int NT, bool kFirstBuilt, typename CandKey, typename CandId, typename Put>
__device__ void resolve_boundary(CandKey cand_key, CandId cand_id, uint32_t m, uint32_t b1, uint32_t bin_count,
                                 uint32_t need, uint32_t n_up, uint32_t* hist, Put put, int topk, SelState& s) {
  using L = Levels<NT>;
  constexpr int kShifts[3] = {L::kShift0, L::kShift1, L::kShift2};
  constexpr int kWidths[3] = {L::kWidth0, L::kWidth1, L::kWidth2};
  const int tid = threadIdx.x;
  uint32_t prefix = b1;
  int shift = kHistShift;
  if (!kFirstBuilt && tid == 0) {  // ordered before the placement below by the syncs that follow
    s.cnt = n_up;
    s.eq = 0;
  }
  bool synced = kFirstBuilt;
  if (bin_count != need) {  // else the whole bin is taken
    for (int lvl = 0; lvl < L::kCount; ++lvl) {
      const uint32_t mask = (1u << kWidths[lvl]) - 1u;
      if (!kFirstBuilt || lvl > 0) {
        __syncthreads();
        for (int b = tid; b < L::kBins / 4; b += NT) reinterpret_cast<uint4*>(hist)[b] = make_uint4(0, 0, 0, 0);
        if (tid == 0) {
          s.bin = 0;
          s.above = 0;
        }
        __syncthreads();
        for (uint32_t j = tid; j < m; j += NT) {
          const uint32_t k = cand_key(j);
          if ((k >> shift) == prefix) atomicAdd(&hist[(k >> kShifts[lvl]) & mask], 1u);
        }
        __syncthreads();
      }
      find_bin<NT, L::kBins>(hist, need, s);
      synced = true;
      const int b = s.bin;
      need -= s.above;
      prefix = (prefix << kWidths[lvl]) | static_cast<uint32_t>(b);
      shift = kShifts[lvl];
      if (s.binc == need) break;
    }
  }
  if (!synced) __syncthreads();
  for (uint32_t j0 = 0; j0 < m; j0 += NT) {
    const uint32_t j = j0 + tid;
    const uint32_t k = j < m ? cand_key(j) : 0u;
    const bool in_bin = j < m && (k >> kHistShift) == b1;  // row fallback: only the boundary bin
    const uint32_t pk = k >> shift;
    const bool up = in_bin && pk > prefix;
    const bool tie = in_bin && pk == prefix;
    const uint32_t tq = warp_reserve(tie, &s.eq);
    const bool take = up || (tie && tq < need);
    const uint32_t pos = warp_reserve(take, &s.cnt);
    if (take && pos < static_cast<uint32_t>(topk)) put(pos, cand_id(j));
  }
  __syncthreads();
}

// Top `topk` of the n > topk keys key_at(0..n) of one row (read from L2),
// written through o. Warp w owns a contiguous chunk of the row: it counts,
// a scan over the warps gives each its offsets, and it places its keys in
// order, so the reads stay coalesced. hist (shared, kSelBins) holds the
// keys' pass-1 histogram on entry; ckey / cidx (shared, cap each) take
// the boundary bin's keys; oid (shared, topk) collects the ids.
template <int NT, typename KeyAt>
__device__ void select_row(KeyAt key_at, int n, uint32_t* hist, uint32_t* ckey, uint32_t* cidx, uint32_t* oid,
                           int topk, uint32_t cap, const RowOut& o, SelState& s, bool* bad) {
  constexpr int kWarps = NT / 32;
  static_assert(kWarps <= 16, "per-warp counts use s.sm[0..16) and s.sm[16..32)");
  const int tid = threadIdx.x;
  const int lane = tid & 31, wid = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  if (tid == 0) {
    s.bin = 0;
    s.above = 0;
  }
  for (int i = tid; i < topk; i += NT) oid[i] = 0xffffffffu;
  __syncthreads();
  find_bin<NT>(hist, static_cast<uint32_t>(topk), s);
  const uint32_t b1 = static_cast<uint32_t>(s.bin);
  const uint32_t n_up = s.above, bin_count = s.binc;
  const bool gather = bin_count <= cap;

  const int per = ((n + kWarps - 1) / kWarps + 31) & ~31;
  const int lo = wid * per, hi = min(n, lo + per);
  uint32_t c_up = 0, c_eq = 0;
  for (int i0 = lo; i0 < hi; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t bin = i < hi ? key_at(i) >> kHistShift : 0u;
    c_up += __popc(__ballot_sync(0xffffffffu, i < hi && bin > b1));
    c_eq += __popc(__ballot_sync(0xffffffffu, i < hi && bin == b1));
  }
  if (lane == 0) {
    s.sm[wid] = c_up;
    s.sm[16 + wid] = c_eq;
  }
  __syncthreads();
  uint32_t p_up = 0, p_eq = 0, total_eq = 0;
#pragma unroll
  for (int v = 0; v < kWarps; ++v) {
    const uint32_t u = s.sm[v], e = s.sm[16 + v];
    if (v < wid) {
      p_up += u;
      p_eq += e;
    }
    total_eq += e;
  }
  for (int i0 = lo; i0 < hi; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < hi ? key_at(i) : 0u;
    const uint32_t bin = key >> kHistShift;
    const bool up = i < hi && bin > b1;
    const bool eq = i < hi && bin == b1;
    const uint32_t m_up = __ballot_sync(0xffffffffu, up);
    const uint32_t m_eq = __ballot_sync(0xffffffffu, eq);
    const uint32_t q_up = p_up + __popc(m_up & lt_mask);
    const uint32_t q_eq = p_eq + __popc(m_eq & lt_mask);
    if (up && q_up < static_cast<uint32_t>(topk)) oid[q_up] = static_cast<uint32_t>(i);
    if (gather && eq && q_eq < cap) {
      ckey[q_eq] = key;
      cidx[q_eq] = static_cast<uint32_t>(i);
    }
    p_up += __popc(m_up);
    p_eq += __popc(m_eq);
  }
  __syncthreads();
  // the boundary bin: candidates j < m (or, past cap, the row filtered to the bin)
  const uint32_t m = gather ? min(total_eq, cap) : static_cast<uint32_t>(n);
  resolve_boundary<NT, false>([&](uint32_t j) -> uint32_t { return gather ? ckey[j] : key_at(static_cast<int>(j)); },
                              [&](uint32_t j) -> uint32_t { return gather ? cidx[j] : j; }, m, b1, bin_count,
                              static_cast<uint32_t>(topk) - n_up, n_up, hist,
                              [&](uint32_t pos, uint32_t id) { oid[pos] = id; }, topk, s);
  write_ids<NT>(oid, topk, o, bad);
  __syncthreads();
}

// Before the staging pass's closing __syncthreads() of a row that
// select_row_staged will take: the ids' slots emptied, the scan state reset.
template <int NT>
__device__ __forceinline__ void select_staged_init(uint32_t* oid, int topk, SelState& s) {
  if (threadIdx.x == 0) {
    s.bin = 0;
    s.above = 0;
  }
  for (int i = threadIdx.x; i < topk / 4; i += NT) reinterpret_cast<uint4*>(oid)[i] = make_uint4(~0u, ~0u, ~0u, ~0u);
}

// Top `topk` of the kTopkRowCap >= n > topk keys staged in shared memory
// (keys, 16-byte aligned), written through o; select_staged_init ran before
// the sync that ended the staging. Thread i owns a contiguous range of 4*q
// keys (q odd: the 16-byte loads of a warp hit distinct banks); one block
// scan of the packed counts gives every thread its offsets. In 1024-thread
// rows the placement pass also bins the boundary bin's keys for the first
// resolving level, into hist, which pass 1 no longer needs once the boundary
// bin is known: one pass and three barriers fewer (decode32 top-k 11.8 ->
// 11.2 us). 256-thread rows gather a few hundred candidates, and a pass over
// them costs less than the counts in the placement (prefill4x8k top-k 430
// against 433 us).
template <int NT>
__device__ void select_row_staged(const uint32_t* keys, int n, uint32_t* hist, uint32_t* ckey, uint32_t* cidx,
                                  uint32_t* oid, int topk, uint32_t cap, const RowOut& o, SelState& s, bool* bad) {
  using L = Levels<NT>;
  constexpr bool kFuse = L::kWide;
  const int tid = threadIdx.x;
  find_bin<NT>(hist, static_cast<uint32_t>(topk), s);
  const uint32_t b1 = static_cast<uint32_t>(s.bin);
  const uint32_t n_up = s.above, bin_count = s.binc;
  const bool gather = bin_count <= cap;
  // hist is no longer read: clear it for the first level (ordered before the
  // placement's counts by the scan's barrier)
  if constexpr (kFuse)
    for (int b = tid; b < L::kBins / 4; b += NT) reinterpret_cast<uint4*>(hist)[b] = make_uint4(0, 0, 0, 0);

  int q4 = ((n + NT - 1) / NT + 3) >> 2;
  q4 += (q4 & 1) ^ 1;  // odd
  const int lo = tid * 4 * q4, hi = min(n, lo + 4 * q4);
  const uint4* k4 = reinterpret_cast<const uint4*>(keys);
  int c_up = 0, c_eq = 0;
  for (int i = lo; i < hi; i += 4) {
    const uint4 v = k4[i >> 2];
    const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t bin = kk[c] >> kHistShift;
      const bool in = i + c < hi;
      c_up += in && bin > b1;
      c_eq += in && bin == b1;
    }
  }
  // counts <= kTopkRowCap < 2^16: up in the high half, boundary-bin keys in the low
  uint32_t total;
  const uint32_t excl = block_excl_sum<NT>((static_cast<uint32_t>(c_up) << 16) | static_cast<uint32_t>(c_eq), s.sm, &total);
  uint32_t p_up = excl >> 16, p_eq = excl & 0xffffu;
  const uint32_t total_eq = total & 0xffffu;
  if (tid == 0) {  // every thread read s.bin, s.above and s.binc before the scan's barrier
    s.bin = 0;
    s.above = 0;
    s.cnt = n_up;
    s.eq = 0;
  }
  for (int i = lo; i < hi; i += 4) {
    const uint4 v = k4[i >> 2];
    const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // predicated: 484 -> 455 us (prefill4x8k) against nested branches
      const uint32_t bin = kk[c] >> kHistShift;
      const bool in = i + c < hi;
      const bool up = in && bin > b1;
      const bool in_bin = in && bin == b1;
      const bool eq = in_bin && gather;
      if (up && p_up < static_cast<uint32_t>(topk)) oid[p_up] = static_cast<uint32_t>(i + c);
      if (kFuse && in_bin) atomicAdd(&hist[L::first_bin(kk[c])], 1u);
      if (eq && p_eq < cap) {
        ckey[p_eq] = kk[c];
        cidx[p_eq] = static_cast<uint32_t>(i + c);
      }
      p_up += up ? 1u : 0u;
      p_eq += eq ? 1u : 0u;
    }
  }
  __syncthreads();
  const uint32_t m = gather ? min(total_eq, cap) : static_cast<uint32_t>(n);
  resolve_boundary<NT, kFuse>([&](uint32_t j) -> uint32_t { return gather ? ckey[j] : keys[j]; },
                              [&](uint32_t j) -> uint32_t { return gather ? cidx[j] : j; }, m, b1, bin_count,
                              static_cast<uint32_t>(topk) - n_up, n_up, hist,
                              [&](uint32_t pos, uint32_t id) { oid[pos] = id; }, topk, s);
  write_ids<NT>(oid, topk, o, bad);
  __syncthreads();
}

}  // namespace dsa
