// Shared pieces of the quantised-KV decode kernels: the page-unit geometry of
// the shared-memory ring, mma.sync and conversion helpers, the value-table
// addressing, and the producer lane that streams a split's K and V units
// through the ring (the mbarrier and TMA helpers are in tma_ptx.cuh).
#pragma once

#include "lynx_internal.cuh"
#include "tma_ptx.cuh"

#include <cuda.h>
#include <cuda_fp16.h>
#include <math_constants.h>

namespace lynx {

namespace {

constexpr int kConsumers = 8;
constexpr int kConsumerThreads = kConsumers * 32;
constexpr int kThreadsQ = (kConsumers + 1) * 32;
constexpr int kRows = 4;
constexpr int kWsPerCta = kRows * kH + 2 * kRows;

template <bool FULL, int STAGES = 3>
struct QGeo {
  static constexpr int kStages = STAGES;
  static constexpr int kUnit = FULL ? 2 * kPlaneBytes + kMetaBytes : kPlaneBytes + kMetaBytes;
  static constexpr int kResOff = kPlaneBytes;
  static constexpr int kMetaOff = FULL ? 2 * kPlaneBytes : kPlaneBytes;
};
static_assert(QGeo<false>::kUnit % 1024 == 0 && QGeo<true>::kUnit % 1024 == 0,
              "ring slots must keep the 1024-byte alignment of swizzled tiles");

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// largest of a warp's non-negative (or +0 / +inf) floats in one reduction: for
// such floats the bit patterns order as unsigned integers
__device__ __forceinline__ float warp_max_nonneg(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
template <typename T>
__device__ __forceinline__ T lds(const uint8_t* smem, uint32_t off) {
  return *reinterpret_cast<const T*>(smem + off);
}

// ---------------------------------------------------------------- tensor-core helpers

__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// TF32 head (low 13 mantissa bits cleared) and the exact float32 remainder
__device__ __forceinline__ uint32_t tf32_hi(float x) { return __float_as_uint(x) & 0xFFFFE000u; }
__device__ __forceinline__ uint32_t tf32_lo(float x) {
  return __float_as_uint(x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u));
}

// fp16 pair, `lo` in the low half (the lower k index of a fragment register)
__device__ __forceinline__ uint32_t h2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t h2(__half lo, __half hi) {
  const __half2 v = __halves2half2(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// table offset for byte j of `word`: the byte in bits 8..15, the lane's copy
// offset (< 256) in bits 0..7
__device__ __forceinline__ uint32_t byte_sel(uint32_t j) { return 0x5504u | (j << 4); }
__device__ __forceinline__ uint32_t lut_off(uint32_t word, uint32_t lane_off, uint32_t sel) {
  return prmt(word, lane_off, sel);
}

// full codes (anchor nibble | residual nibble << 4) of the even and of the odd
// tokens of the four bytes of an anchor word and its residual word
__device__ __forceinline__ void full_codes(uint32_t wa, uint32_t wr, uint32_t& ev, uint32_t& od) {
  ev = (wa & 0x0F0F0F0Fu) | ((wr << 4) & 0xF0F0F0F0u);
  od = ((wa >> 4) & 0x0F0F0F0Fu) | (wr & 0xF0F0F0F0u);
}

// Producer lane of a decode CTA: streams the K and V units of pages
// [p_begin, p_begin + np) of one page-table row through the kStages-slot ring.
// Unit u (K of page u/2 for even u, V for odd u) goes to slot u % kStages once
// the consumers released that slot's previous unit.  An out-of-range page id
// is reported (status 2) and page 0 read instead.  A wait that gives up sets
// status 1 and the CTA's abort flag.  Before returning, the lane waits
// (bounded) until every copy it issued has landed: a unit older than the last
// kStages was consumed before its slot was reused, so only those last units
// can still be in flight, whether the consumers finished or gave up early.
// first_id is the page id pt_row[p_begin], read by the caller ahead of time
// (e.g. together with the context length) so that the first copy waits on one
// global load less; the table entry of every later page is read once, for its
// K unit.
template <bool FULL, int STAGES = 3>
__device__ void produce_units(const DecodeArgs& a, const int32_t* pt_row, int p_begin, int np, int first_id,
                              uint32_t s_ring, uint32_t bar_full, uint32_t bar_empty,
                              const CUtensorMap* tm_ka, const CUtensorMap* tm_va,
                              const CUtensorMap* tm_kr, const CUtensorMap* tm_vr, int* s_flag) {
  using G = QGeo<FULL, STAGES>;
  constexpr int kSt = G::kStages;
  const int skip = a.inject_skip - 1;   // -1: no unit is skipped
  int u_end = 0;                        // units attempted
  bool ok = true;
  int64_t id = first_id;
  for (int u = 0; u < 2 * np; ++u) {
    const int st = u % kSt;
    if (u >= kSt && !mbar_wait(bar_empty + 8 * st, ((u / kSt) - 1) & 1, a.wait_ns)) {
      ok = false;
      break;
    }
    u_end = u + 1;
    const int p = p_begin + (u >> 1);
    const bool is_v = (u & 1) != 0;
    if (u >= 2 && !is_v) id = pt_row[p];
    if (u == skip) continue;   // test hook: this unit's copy is never issued
    if (id < 0 || id >= a.n_pool) {
      atomicExch(a.status, 2);
      id = 0;
    }
    const uint32_t dst = s_ring + st * G::kUnit;
    const uint32_t bar = bar_full + 8 * st;
    const uint32_t meta_bytes = 4u * (uint32_t)a.meta_floats;   // <= kMetaBytes, a multiple of 16
    mbar_expect_tx(bar, G::kMetaOff + meta_bytes);
    tma_tile_g2s(dst, is_v ? tm_va : tm_ka, 0, (int)(id * kH), bar);
    if (FULL) tma_tile_g2s(dst + G::kResOff, is_v ? tm_vr : tm_kr, 0, (int)(id * kH), bar);
    bulk_g2s(dst + G::kMetaOff, (is_v ? a.v_meta : a.k_meta) + id * a.meta_floats, meta_bytes, bar);
  }
  if (!ok) {
    atomicExch(a.status, 1);
    *s_flag = 1;
  }
  for (int u = u_end - 1; u >= 0 && u >= u_end - kSt; --u)
    if (u != skip) mbar_wait(bar_full + 8 * (u % kSt), (u / kSt) & 1, a.wait_ns);
}

}  // namespace
}  // namespace lynx
