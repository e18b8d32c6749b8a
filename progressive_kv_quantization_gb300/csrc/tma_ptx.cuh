// PTX helpers for mbarriers, bulk copies and 2-D TMA tile loads, and the
// host-side tensor maps built over the library's inputs.  Every wait on an
// mbarrier is bounded: it gives up after two seconds so that a kernel can
// record an error and return instead of hanging.
#pragma once

#include "lynx_internal.cuh"

#include <cuda.h>

namespace lynx {

// 2-D tensor map over a pool of 4-bit planes (rows of 128 bytes, one 128 x 128
// tile per page, 128-byte swizzle); false if the driver refuses it
bool plane_map(CUtensorMap* m, const uint8_t* pool, int64_t n_pool);

// 2-D tensor map over a pool of BF16 pages [n_pool][128][256] (rows of 512
// bytes), boxes of 64 tokens x 128 channels (four per page), 128-byte swizzle;
// false if the driver refuses it
bool bf16_page_map(CUtensorMap* m, const uint16_t* pool, int64_t n_pool);

// 2-D tensor map over token-major BF16 KV (row t = token t, row_elems valid
// elements, stride elements between rows), boxes of 64 channels x 256 tokens,
// no swizzle, zero fill past the last token; false if the driver refuses it
// (x not 16-byte aligned, stride not a multiple of 8, sizes out of range)
bool token_map(CUtensorMap* m, const void* x, int64_t n_tokens, int64_t row_elems, int64_t stride);

namespace {

constexpr unsigned long long kWaitNs = kDefaultWaitNs;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// one poll that may suspend the thread for up to hint_ns; a suspended thread
// resumes as soon as the phase completes, and issues nothing meanwhile
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
constexpr uint32_t kPollHintNs = 100000u;   // a waiting thread sleeps in polls of up to 100 us
// gives up after limit_ns (clock checked after every poll) or 2^26 polls
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 26); ++i) {
    if (mbar_try_wait_hint(bar, parity, kPollHintNs)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
  return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_tile_g2s(uint32_t dst, const CUtensorMap* map, int x, int y,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
}  // namespace
}  // namespace lynx
