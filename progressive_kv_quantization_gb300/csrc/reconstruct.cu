// lynx_reconstruct kernels: the Anchor-phase and Residual-phase dequantisation
// of the Lynx paper (§4.2; inverse compander of Eq. (4)).
//
// Work mapping.  A CTA of 8 warps takes 8 consecutive channel rows of a page
// (a row octet) at a time; warp w owns row w, lane L owns tokens 8L .. 8L+7,
// which are one 32-bit word of each 4-bit plane (coalesced 128-byte warp
// loads) and 16 bytes of BF16 output (coalesced 512-byte warp stores).  The
// octet's chunk-major metadata (mu[8 chunks][8 rows], sigma likewise: eight
// 32-byte runs each) is loaded once by the CTA into shared memory, double
// buffered with one barrier per octet; the next octet's plane words and
// metadata are loaded before the current octet is computed.  The inverse
// compander is a shared-memory table lookup with one copy of the table per
// lane (entry e of lane L at word e*32 + L), so lookups never share a bank.
// The two affine steps are fused multiply-adds, two tokens at a time:
//   x = fmaf(fmaf(S*l(I_hat), sigma+eps, mu), gamma_scale+eps, gamma_min).

#include "lynx_internal.cuh"

#include <cuda_bf16.h>

namespace lynx {
namespace {

template <bool kFull, bool kF32>
__global__ void __launch_bounds__(256)
reconstruct_kernel(const uint32_t* __restrict__ anchor, const uint32_t* __restrict__ residual,
                   const float* __restrict__ meta, int64_t n_octets, void* __restrict__ out,
                   const LutTables lut) {
  constexpr int kEntries = kFull ? 256 : 16;
  __shared__ float s_lut[kEntries * 32];
  __shared__ float s_meta[2][4][64];       // [buffer][gmin, gscale, mu, sigma][chunk * 8 + row]
  for (int i = threadIdx.x; i < kEntries * 32; i += blockDim.x)
    s_lut[i] = kFull ? lut.full[i >> 5] : lut.anc16[i >> 5];

  const int tid = threadIdx.x;
  const int w = tid >> 5;
  const int lane = tid & 31;
  const float eps = lut.eps;
  const float* lut_lane = s_lut + lane;

  // metadata of octet o: thread tid < 128 loads one value (kind = tid >> 5 ... see below)
  auto load_meta = [&](int64_t o) {
    float v = 0.0f;
    if (tid < 144) {
      const float* mp = meta + (o >> 4) * kMetaFloats;
      const int ch0 = 8 * (int)(o & 15);
      if (tid < 64) {                      // mu[chunk][row]
        v = __ldg(mp + kMetaMuOff + (tid >> 3) * kH + ch0 + (tid & 7));
      } else if (tid < 128) {              // sigma[chunk][row]
        const int i = tid - 64;
        v = __ldg(mp + kMetaSigmaOff + (i >> 3) * kH + ch0 + (i & 7));
      } else {                             // gamma_min[row], gamma_scale[row]
        const int i = tid - 128;
        v = __ldg(mp + (i >> 3) * kH + ch0 + (i & 7));
      }
    }
    return v;
  };
  auto store_meta = [&](int buf, float v) {
    if (tid < 64) s_meta[buf][2][tid] = v;
    else if (tid < 128) s_meta[buf][3][tid - 64] = v;
    else if (tid < 144) s_meta[buf][(tid - 128) >> 3][tid & 7] = v;
  };

  const int64_t stride = gridDim.x;
  int64_t o = blockIdx.x;
  uint32_t wa_n = 0, wr_n = 0;
  if (o < n_octets) {
    store_meta(0, load_meta(o));
    const int64_t row = 8 * o + w;
    wa_n = __ldg(anchor + row * 32 + lane);
    if (kFull) wr_n = __ldg(residual + row * 32 + lane);
  }
  __syncthreads();
  int buf = 0;
  for (; o < n_octets; o += stride, buf ^= 1) {
    const int64_t row = 8 * o + w;
    const uint32_t wa = wa_n, wr = wr_n;
    const int64_t on = o + stride;
    float mnext = 0.0f;
    if (on < n_octets) {
      mnext = load_meta(on);
      wa_n = __ldg(anchor + (8 * on + w) * 32 + lane);
      if (kFull) wr_n = __ldg(residual + (8 * on + w) * 32 + lane);
    }
    const int blk = lane >> 2;
    const float gmin = s_meta[buf][0][w];
    const float dgv = __fadd_rn(s_meta[buf][1][w], eps);
    const float muv = s_meta[buf][2][blk * 8 + w];
    const float dsv = __fadd_rn(s_meta[buf][3][blk * 8 + w], eps);
    const float2 ds2 = make_float2(dsv, dsv), mu2 = make_float2(muv, muv);
    const float2 dg2 = make_float2(dgv, dgv), gm2 = make_float2(gmin, gmin);
    float2 xv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t c0 = (wa >> (8 * k)) & 0xFu, c1 = (wa >> (8 * k + 4)) & 0xFu;
      if (kFull) {
        c0 |= ((wr >> (8 * k)) & 0xFu) << 4;
        c1 |= ((wr >> (8 * k + 4)) & 0xFu) << 4;
      }
      const float2 l = make_float2(lut_lane[c0 * 32], lut_lane[c1 * 32]);
      xv[k] = __ffma2_rn(__ffma2_rn(l, ds2, mu2), dg2, gm2);
    }
    if (kF32) {
      float4* op = reinterpret_cast<float4*>(out) + row * 64 + lane * 2;
      op[0] = make_float4(xv[0].x, xv[0].y, xv[1].x, xv[1].y);
      op[1] = make_float4(xv[2].x, xv[2].y, xv[3].x, xv[3].y);
    } else {
      uint32_t pk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(xv[k].x, xv[k].y);
        pk[k] = *reinterpret_cast<const uint32_t*>(&h);
      }
      reinterpret_cast<uint4*>(out)[row * 32 + lane] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    if (on < n_octets) store_meta(buf ^ 1, mnext);
    __syncthreads();
  }
}

template <bool kFull, bool kF32>
cudaError_t launch(const uint8_t* anchor, const uint8_t* residual, const float* meta,
                   int64_t n_pages, void* out, const LutTables* lut, cudaStream_t s) {
  const int64_t n_octets = n_pages * (kH / 8);
  const int threads = 256;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reconstruct_kernel<kFull, kF32>, threads, 0);
  if (per_sm < 1) per_sm = 1;
  const int64_t max_blocks = (int64_t)device_sm_count() * per_sm;
  const int blocks = (int)(n_octets < max_blocks ? n_octets : max_blocks);
  reconstruct_kernel<kFull, kF32><<<blocks, threads, 0, s>>>(
      reinterpret_cast<const uint32_t*>(anchor), reinterpret_cast<const uint32_t*>(residual), meta,
      n_octets, out, *lut);
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
