// lynx_reconstruct kernels: the Anchor-phase and Residual-phase dequantisation
// of the Lynx paper (§4.2; inverse compander of Eq. (4)).
//
// Work mapping.  One warp owns one channel row (256 tokens) of a page; lane L
// owns tokens 8L .. 8L+7, which are one 32-bit word of each 4-bit plane
// (coalesced 128-byte warp loads) and 16 bytes of BF16 output (coalesced
// 512-byte warp stores).  The per-element inverse compander is a table
// lookup in shared memory with one copy of the table per lane (entry e of
// lane L at word e*32 + L), so a warp's lookups never share a bank.  The two
// affine steps are fused multiply-adds:
//   x = fmaf(fmaf(S*l(I_hat), sigma+eps, mu), gamma_scale+eps, gamma_min).

#include "lynx_internal.cuh"

#include <cuda_bf16.h>

namespace lynx {
namespace {

template <bool kFull, bool kF32>
__global__ void __launch_bounds__(256)
reconstruct_kernel(const uint32_t* __restrict__ anchor, const uint32_t* __restrict__ residual,
                   const float* __restrict__ meta, int64_t n_rows, void* __restrict__ out,
                   const LutTables lut) {
  constexpr int kEntries = kFull ? 256 : 16;
  __shared__ float s_lut[kEntries * 32];
  for (int i = threadIdx.x; i < kEntries * 32; i += blockDim.x)
    s_lut[i] = kFull ? lut.full[i >> 5] : lut.anc16[i >> 5];
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const float eps = lut.eps;
  const float* lut_lane = s_lut + lane;

  // the next row's words and metadata are loaded before the current row is
  // computed, so each warp keeps one row of loads in flight
  struct RowIn {
    uint32_t wa, wr;
    float gmin, gs, mu, sg;
  };
  auto load_row = [&](int64_t row) {
    RowIn r;
    r.wa = __ldg(anchor + row * 32 + lane);
    r.wr = kFull ? __ldg(residual + row * 32 + lane) : 0u;
    const int64_t page = row >> 7;
    const int ch = (int)(row & 127);
    const int blk = lane >> 2;
    const float* mp = meta + page * kMetaFloats;
    r.gmin = __ldg(mp + ch);
    r.gs = __ldg(mp + kH + ch);
    r.mu = __ldg(mp + kMetaMuOff + blk * kH + ch);
    r.sg = __ldg(mp + kMetaSigmaOff + blk * kH + ch);
    return r;
  };
  int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  RowIn nxt{};
  if (row < n_rows) nxt = load_row(row);
  for (; row < n_rows; row += n_warps) {
    const RowIn cur = nxt;
    if (row + n_warps < n_rows) nxt = load_row(row + n_warps);
    const uint32_t wa = cur.wa, wr = cur.wr;
    const float gmin = cur.gmin;
    const float dg = __fadd_rn(cur.gs, eps);
    const float mu = cur.mu;
    const float ds = __fadd_rn(cur.sg, eps);

    float xv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t code = (wa >> (4 * k)) & 0xFu;
      if (kFull) code |= ((wr >> (4 * k)) & 0xFu) << 4;
      const float l = lut_lane[code * 32];
      xv[k] = __fmaf_rn(__fmaf_rn(l, ds, mu), dg, gmin);
    }
    if (kF32) {
      float4* o = reinterpret_cast<float4*>(out) + row * 64 + lane * 2;
      o[0] = make_float4(xv[0], xv[1], xv[2], xv[3]);
      o[1] = make_float4(xv[4], xv[5], xv[6], xv[7]);
    } else {
      uint32_t pk[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(xv[2 * j], xv[2 * j + 1]);
        pk[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      reinterpret_cast<uint4*>(out)[row * 32 + lane] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
}

template <bool kFull, bool kF32>
cudaError_t launch(const uint8_t* anchor, const uint8_t* residual, const float* meta,
                   int64_t n_pages, void* out, const LutTables* lut, cudaStream_t s) {
  const int64_t n_rows = n_pages * kH;
  const int threads = 256;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reconstruct_kernel<kFull, kF32>, threads, 0);
  if (per_sm < 1) per_sm = 1;
  const int64_t max_blocks = (int64_t)device_sm_count() * per_sm;
  const int64_t need = (n_rows + 7) / 8;
  const int blocks = (int)(need < max_blocks ? need : max_blocks);
  reconstruct_kernel<kFull, kF32><<<blocks, threads, 0, s>>>(
      reinterpret_cast<const uint32_t*>(anchor), reinterpret_cast<const uint32_t*>(residual), meta,
      n_rows, out, *lut);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reconstruct(const uint8_t* anchor, const uint8_t* residual, const float* meta,
                               int64_t n_pages, void* out, int out_dtype, const LutTables* lut,
                               cudaStream_t s) {
  const bool full = residual != nullptr;
  const bool f32 = out_dtype == LYNX_OUT_F32;
  if (full) {
    return f32 ? launch<true, true>(anchor, residual, meta, n_pages, out, lut, s)
               : launch<true, false>(anchor, residual, meta, n_pages, out, lut, s);
  }
  return f32 ? launch<false, true>(anchor, residual, meta, n_pages, out, lut, s)
             : launch<false, false>(anchor, residual, meta, n_pages, out, lut, s);
}

}  // namespace lynx
