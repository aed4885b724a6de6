// common.cuh — device helpers shared by the sm_103a kernels of the DSA indexer:
// the ue8m0/E4M3 group quantiser, the device error word, and thin inline-PTX
// wrappers for mbarriers (every wait bounded in time), TMA bulk copies and
// tcgen05 (TMEM allocation, MMA, commit, loads).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsaidx.h"
#include "kernels.h"

namespace dsa {

// Wall-clock limit of any spin on an mbarrier before the kernel gives up,
// flags DSA_DEVERR_TIMEOUT and unwinds.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// Programmatic dependent launch: wait until the previous kernel of the stream
// has completed and its memory is visible (a no-op when the launch did not
// opt in), and let the next kernel of the stream start its own set-up.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kernel` so that it may start while the previous kernel of the
// stream is still running; the kernel calls pdl_wait() before it reads that
// kernel's results. Stream capture keeps the relation as a programmatic edge.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

__device__ __forceinline__ void flag_error(int32_t* err, uint32_t bit) {
  if (err != nullptr) atomicOr(reinterpret_cast<unsigned int*>(err), bit);
}

// ---------------------------------------------------------------------------
// Group quantiser (one 128-value row = one group). The scale is
// max(amax,1e-10)/448 in IEEE fp32, rounded up to a power of two; codes are
// x/scale rounded to nearest-even E4M3 with saturation. x * 2^-e equals
// x / 2^e exactly (same real value, same rounding), so multiplying by the
// exact reciprocal reproduces the division.
//
// The scale without the division, for amax holding a bf16 value (every input
// the quantiser sees is bf16) or the floor 1e-10: it is the smallest power of
// two 2^e >= RN(amax/448). RN(x) <= 2^e iff x <= 2^e (1 + 2^-24) (the tie
// goes to the even 2^e), and no bf16 value lies in (448*2^e, 448*2^e (1 +
// 2^-24)], so 2^e is the smallest power of two with 448*2^e >= amax. With
// amax = m*2^E (1 <= m < 2) and 448 = 1.75*2^8, that is e = E - 8, plus one
// when m > 1.75. The floor 1e-10 = 1.718*2^-34 gives 2^-42, far from a
// boundary. (The pinned CPU oracle divides; the GPU tests compare every scale
// bit for bit, boundary cases included.)
__device__ __forceinline__ float ue8m0_scale(float amax) {
  amax = fmaxf(amax, 1e-10f);
  const uint32_t u = __float_as_uint(amax);
  const uint32_t be = u >> 23;  // biased exponent; amax >= 0
  if (be == 255u) return __uint_as_float(0x7F800000u);  // amax = +inf
  return __uint_as_float((be - 8u + ((u & 0x7FFFFFu) > 0x600000u ? 1u : 0u)) << 23);
}

// The FP4 cache's scale: the smallest power of two 2^e >= RN(amax/6). With
// amax = m*2^E (1 <= m < 2) and 6 = 1.5*2^2 that is e = E - 2, plus one when
// m > 1.5. RN cannot move the quotient across the power of two: for m <= 1.5
// amax/6 <= 2^(E-2) exactly, and for m >= 1.5 + 2^-23 the quotient is at
// least 2^(E-2) (1 + 2^-23/1.5), which rounds to 2^(E-2) (1 + 2^-23). The
// floor 1e-10 = 1.718*2^-34 gives 2^-35.
__device__ __forceinline__ float ue8m0_scale_e2m1(float amax) {
  amax = fmaxf(amax, 1e-10f);
  const uint32_t u = __float_as_uint(amax);
  const uint32_t be = u >> 23;
  if (be == 255u) return __uint_as_float(0x7F800000u);  // amax = +inf
  return __uint_as_float((be - 2u + ((u & 0x7FFFFFu) > 0x400000u ? 1u : 0u)) << 23);
}

// 2^-e for a normal power of two s = 2^e (|e| <= 126).
__device__ __forceinline__ float pow2_reciprocal(float s) {
  uint32_t e = __float_as_uint(s) >> 23;
  return __uint_as_float((254u - e) << 23);
}

// Four fp32 values -> four E4M3 codes, first value in the lowest byte.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One warp quantises one 128-value bf16 row: lane i holds values 4i..4i+3.
// Returns the packed codes of this lane and the row's scale.
__device__ __forceinline__ uint32_t quant_row_lane(uint2 raw, float* scale_out) {
  __nv_bfloat162 p0 = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
  __nv_bfloat162 p1 = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
  float2 f0 = __bfloat1622float2(p0);
  float2 f1 = __bfloat1622float2(p1);
  float amax = fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
  amax = warp_max(amax);
  float s = ue8m0_scale(amax);
  float inv = pow2_reciprocal(s);
  *scale_out = s;
  return e4m3x4(f0.x * inv, f0.y * inv, f1.x * inv, f1.y * inv);
}

// The same quantiser on half a warp: lanes 16h..16h+15 hold one row, lane i of
// the half values 8i..8i+7 (one 16-byte load), so a warp load moves two rows.
// Returns this lane's 8 codes (first value in the lowest byte) and the row's
// scale.
__device__ __forceinline__ uint2 quant_row_half(uint4 raw, float* scale_out) {
  const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
  float f[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[k]));
    f[2 * k] = p.x;
    f[2 * k + 1] = p.y;
  }
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[k]));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));  // within the half
  const float s = ue8m0_scale(amax);
  const float inv = pow2_reciprocal(s);
  *scale_out = s;
  return make_uint2(e4m3x4(f[0] * inv, f[1] * inv, f[2] * inv, f[3] * inv),
                    e4m3x4(f[4] * inv, f[5] * inv, f[6] * inv, f[7] * inv));
}

// Four fp32 values -> four E2M1 codes (nearest-even, saturating), first value
// in the lowest nibble.
__device__ __forceinline__ uint32_t e2m1x4(float a, float b, float c, float d) {
  const __nv_fp4x2_storage_t lo = __nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest);
  const __nv_fp4x2_storage_t hi = __nv_cvt_float2_to_fp4x2(make_float2(c, d), __NV_E2M1, cudaRoundNearest);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 8);
}

// quant_row_lane for the FP4 cache: the 4 E2M1 codes of this lane (16 bits).
__device__ __forceinline__ uint32_t quant_row_lane_e2m1(uint2 raw, float* scale_out) {
  const float2 f0 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.x));
  const float2 f1 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.y));
  float amax = fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
  amax = warp_max(amax);
  const float s = ue8m0_scale_e2m1(amax);
  const float inv = pow2_reciprocal(s);
  *scale_out = s;
  return e2m1x4(f0.x * inv, f0.y * inv, f1.x * inv, f1.y * inv);
}

// S1's store: quantise the K row a warp holds (lane i: values 4i..4i+3) and
// write it at `slot` of an FP8 cache (8448-byte pages: 128 code bytes per
// row) or an FP4 cache (4352-byte pages: 64 code bytes per row), the fp32
// scale after the page's 64 rows.
__device__ __forceinline__ void quant_store_k_row(uint8_t* cache, int64_t slot, uint2 raw, bool fp4, int lane) {
  const int off = static_cast<int>(slot % kBlock);
  float s;
  if (fp4) {
    const uint32_t codes = quant_row_lane_e2m1(raw, &s);
    uint8_t* page = cache + (slot / kBlock) * kFp4PageBytes;
    reinterpret_cast<uint16_t*>(page + off * (kDim / 2))[lane] = static_cast<uint16_t>(codes);
    if (lane == 0) *reinterpret_cast<float*>(page + kFp4ScaleOffset + off * 4) = s;
  } else {
    const uint32_t codes = quant_row_lane(raw, &s);
    uint8_t* page = cache + (slot / kBlock) * kPageBytes;
    reinterpret_cast<uint32_t*>(page + off * kDim)[lane] = codes;
    if (lane == 0) *reinterpret_cast<float*>(page + kScaleOffset + off * 4) = s;
  }
}

// RoPE of the leading 64 dims of one 128-value bf16 row held by a warp (lane
// i: values 4i..4i+3): dim i < 32 pairs with dim i + 32, which sits on lane
// i/4 + 8. y[i] = x[i]*c - x[i+32]*s, y[i+32] = x[i+32]*c + x[i]*s, each
// product and sum rounded in fp32 (no contraction), the result rounded to
// bf16. cs: the position's row of the cos/sin table (64 floats, 16-byte
// aligned: cos of the 32 pair angles, then their sin). All lanes must call.
__device__ __forceinline__ uint2 rope_row_lane(uint2 raw, const float* cs) {
  const int lane = threadIdx.x & 31;
  const uint2 other = make_uint2(__shfl_xor_sync(0xffffffffu, raw.x, 8), __shfl_xor_sync(0xffffffffu, raw.y, 8));
  if (lane >= 16) return raw;
  const int i0 = 4 * (lane & 7);
  const float4 c = __ldg(reinterpret_cast<const float4*>(cs + i0));
  const float4 s = __ldg(reinterpret_cast<const float4*>(cs + 32 + i0));
  const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  const float2 y01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&other.x));
  const float2 y23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&other.y));
  const float x[4] = {x01.x, x01.y, x23.x, x23.y}, y[4] = {y01.x, y01.y, y23.x, y23.y};
  const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {s.x, s.y, s.z, s.w};
  float r[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    // lanes 0-7 hold x[i] (partner x[i+32]); lanes 8-15 hold x[i+32] (partner x[i])
    const float a = __fmul_rn(x[u], cc[u]), b = __fmul_rn(y[u], ss[u]);
    r[u] = lane < 8 ? __fsub_rn(a, b) : __fadd_rn(a, b);
  }
  const __nv_bfloat162 lo = __floats2bfloat162_rn(r[0], r[1]), hi = __floats2bfloat162_rn(r[2], r[3]);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

// rope_row_lane for the half-warp layout of quant_row_half: dim i < 32 sits on
// lane i/8 of the half and pairs with dim i + 32 on lane i/8 + 4; the same
// rounding (each product and sum in fp32, the result to bf16). All lanes must
// call.
__device__ __forceinline__ uint4 rope_row_half(uint4 raw, const float* cs) {
  const int hl = threadIdx.x & 15;
  const uint32_t ow[4] = {__shfl_xor_sync(0xffffffffu, raw.x, 4), __shfl_xor_sync(0xffffffffu, raw.y, 4),
                          __shfl_xor_sync(0xffffffffu, raw.z, 4), __shfl_xor_sync(0xffffffffu, raw.w, 4)};
  if (hl >= 8) return raw;  // dims 64..127 are not rotated
  const int i0 = 8 * (hl & 3);
  const float4 c0 = __ldg(reinterpret_cast<const float4*>(cs + i0));
  const float4 c1 = __ldg(reinterpret_cast<const float4*>(cs + i0 + 4));
  const float4 s0 = __ldg(reinterpret_cast<const float4*>(cs + 32 + i0));
  const float4 s1 = __ldg(reinterpret_cast<const float4*>(cs + 36 + i0));
  const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    // lanes 0-3 hold x[i] (partner x[i+32]); lanes 4-7 hold x[i+32] (partner x[i])
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[k]));
    const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[k]));
    const float a0 = __fmul_rn(x.x, cc[2 * k]), b0 = __fmul_rn(y.x, ss[2 * k]);
    const float a1 = __fmul_rn(x.y, cc[2 * k + 1]), b1 = __fmul_rn(y.y, ss[2 * k + 1]);
    const float r0 = hl < 4 ? __fsub_rn(a0, b0) : __fadd_rn(a0, b0);
    const float r1 = hl < 4 ? __fsub_rn(a1, b1) : __fadd_rn(a1, b1);
    const __nv_bfloat162 p = __floats2bfloat162_rn(r0, r1);
    out[k] = *reinterpret_cast<const uint32_t*>(&p);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// The row of the cos/sin table for a position, or nullptr (no rotation:
// table absent, or the position out of range, which is flagged).
__device__ __forceinline__ const float* rope_row(const RopeArgs& r, int64_t token, int32_t* err, int lane) {
  if (r.cos_sin == nullptr) return nullptr;
  const int64_t p = __ldg(r.positions + token);
  if (p < 0 || p >= r.max_pos) {
    if (lane == 0) flag_error(err, DSA_DEVERR_POS_RANGE);
    return nullptr;
  }
  return r.cos_sin + p * kRope;
}

// ---------------------------------------------------------------------------
// Shared-memory addresses and mbarriers.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete. Gives up after kWaitLimitNs,
// flags DSA_DEVERR_TIMEOUT, raises the CTA's abort flag and returns false.
// Returns false at once if the abort flag is already up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* err) {
  uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(addr, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      flag_error(err, DSA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor) loads into this CTA's shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, uint64_t* bar, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, uint64_t* bar, int32_t c0, int32_t c1,
                                            int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Four one-row boxes of a 2-D tensor map at rows y0..y3 (column 0), landing
// one after the other in shared memory (tile::gather4).
__device__ __forceinline__ void tma_gather4_2d(void* dst, const void* tmap, uint64_t* bar, int32_t y0, int32_t y1,
                                               int32_t y2, int32_t y3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(0), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
      : "memory");
}

// Untiled bulk copy global -> shared (both 16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA and loads.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle (rows of 128 bytes, 8-row groups 1024 bytes apart), the
// layout a TMA load with CU_TENSOR_MAP_SWIZZLE_128B produces.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);      // start address
  d |= static_cast<uint64_t>(1) << 16;                      // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;              // stride byte offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1) << 46;                      // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::f8f6f4 -> fp32, both operands
// K-major, M x N tile. B is E4M3; A is E4M3 (format 0) or, with a_e2m1, E2M1
// (format 5), which the MMA reads from shared memory with each 16-byte chunk
// holding 16 codes in its first 8 bytes (the image a TMA load of the
// 16U4_ALIGN16B type lands); the K step stays 32 elements = 32 bytes.
__host__ __device__ constexpr uint32_t f8_idesc(int M, int N, bool a_e2m1 = false) {
  return (1u << 4)                                  // D format: fp32
         | ((a_e2m1 ? 5u : 0u) << 7) | (0u << 10)   // A format, B format: E4M3
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Two fp32 lanes in one 64-bit register pair, and the packed fused
// multiply-add on them (two independent fma.rn, one instruction).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes; the registers are
// valid only after tmem_wait32 on them.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// Waits for this thread's TMEM loads; the operands tie r's later uses to the wait.
__device__ __forceinline__ void tmem_wait32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Block-wide inclusive prefix sum of v; *total = the block's sum. sm: 33 ints of shared memory.
__device__ __forceinline__ int block_scan_incl(int v, int* sm, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) sm[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int x = lane < nw ? sm[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += n;
    }
    if (lane < nw) sm[lane] = x;
  }
  __syncthreads();
  const int res = v + (wid > 0 ? sm[wid - 1] : 0);
  *total = sm[nw - 1];
  __syncthreads();
  return res;
}

// Order-preserving map of fp32 to uint32: a > b  <=>  key(a) > key(b).
__device__ __forceinline__ uint32_t f32_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace dsa
