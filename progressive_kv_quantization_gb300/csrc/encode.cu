// lynx_encode_pages kernel: Algorithm 1 of the Lynx paper (§4.1, Stages 1-4)
// in one pass over BF16 KV pages.
//
// Work mapping.  One warp owns four channel rows of a page (a "row group");
// lane L owns chunk (L & 7) of row (L >> 3), i.e. 32 consecutive tokens =
// 64 contiguous bytes, loaded as four 16-byte read-only loads.  The page-level
// min/max of a row is a 3-step xor shuffle over its 8 lanes; the chunk mean is
// the lane's own left-to-right sum of its 32 values, which is the order the
// code definition fixes.  Each lane then writes 16 bytes of the Anchor plane,
// 16 bytes of the Residual plane and its chunk's (mu, sigma); a warp's plane
// stores are contiguous 512-byte runs.  The next row group's 64 bytes are prefetched
// into registers while the current one is processed.
//
// Exactness.  Every Stage 1-2 step is a single correctly rounded float32
// operation written with explicit _rn intrinsics (no contraction).  Each
// division x / d by a per-row or per-chunk divisor d uses r = RN(1/d), then
// q = RN(x r) corrected by one FMA residual step, q' = RN(q + r (x - q d))
// (Markstein's FMA division correction), which returns the correctly rounded
// quotient.  The Stage 3 code round(127 ln(1+alpha a)/ln(1+alpha)) is first
// estimated with the hardware log2; when the estimate lies within a safety
// margin of a rounding edge the code is decided exactly from the threshold
// table (the smallest float32 of each code).

#include "lynx_internal.cuh"

namespace lynx {
namespace {

__device__ __forceinline__ float div_rn_by(float x, float d, float r) {
  const float q = __fmul_rn(x, r);
  const float e = __fmaf_rn(-q, d, x);
  return __fmaf_rn(e, r, q);
}

__device__ __forceinline__ int quantise_mag(float a, const float* __restrict__ s_thr, float c_lg2,
                                            float alpha, float edge) {
  const float y = __fmul_rn(c_lg2, __log2f(__fmaf_rn(alpha, a, 1.0f)));
  const float r = rintf(y);
  int I = __float2int_rn(r);
  if (fabsf(y - r) > edge) {
    I = min(max(I, 0), 127);
    I += (a >= s_thr[I + 1] ? 1 : 0) - (a < s_thr[I] ? 1 : 0);
  }
  return min(max(I, 0), 127);
}

__device__ __forceinline__ void load_chunk(const uint4* __restrict__ src, uint4 (&raw)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) raw[k] = __ldg(src + k);
}

__global__ void __launch_bounds__(256)
encode_kernel(const uint4* __restrict__ x, int64_t n_groups, uint4* __restrict__ anchor,
              uint4* __restrict__ residual, float* __restrict__ meta, const EncodeTables tab) {
  __shared__ float s_thr[129];
  for (int i = threadIdx.x; i < 129; i += blockDim.x) s_thr[i] = tab.thr[i];
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const float eps = tab.eps;

  uint4 raw[4];
  if (g < n_groups) load_chunk(x + g * 128 + lane * 4, raw);

  for (; g < n_groups; g += n_warps) {
    float v[32];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * k + 2 * j] = __uint_as_float(w[j] << 16);
        v[8 * k + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
    const int64_t g_next = g + n_warps;
    if (g_next < n_groups) load_chunk(x + g_next * 128 + lane * 4, raw);

    // ---- Stage 1: per-channel page min / scale
    float mn = v[0], mx = v[0];
#pragma unroll
    for (int t = 1; t < 32; ++t) {
      mn = fminf(mn, v[t]);
      mx = fmaxf(mx, v[t]);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const float gscale = __fsub_rn(mx, mn);
    const float dg = __fadd_rn(gscale, eps);
    const float rg = __frcp_rn(dg);
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] = div_rn_by(__fsub_rn(v[t], mn), dg, rg);

    // ---- Stage 2: chunk mean and max deviation
    float s = v[0];
#pragma unroll
    for (int t = 1; t < 32; ++t) s = __fadd_rn(s, v[t]);
    const float mu = __fmul_rn(s, 0.03125f);
    float sigma = 0.0f;
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      v[t] = __fsub_rn(v[t], mu);
      sigma = fmaxf(sigma, fabsf(v[t]));
    }
    const float ds = __fadd_rn(sigma, eps);
    const float rs = __frcp_rn(ds);

    // ---- Stages 3-4: code, split, pack
    uint32_t pa[4] = {0u, 0u, 0u, 0u}, pr[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const float xf = div_rn_by(v[t], ds, rs);
      const int I = quantise_mag(fabsf(xf), s_thr, tab.c_lg2, tab.alpha, tab.edge);
      const int q8 = (xf < 0.0f) ? ~I : I;                // sign-aware 8-bit code
      const uint32_t an = (uint32_t)(q8 >> 4) & 0xFu;      // anchor nibble
      const uint32_t rn = (uint32_t)(7 - I) & 0xFu;        // residual 16(I>>4)+7-I, mod 16
      pa[t >> 3] |= an << (4 * (t & 7));
      pr[t >> 3] |= rn << (4 * (t & 7));
    }
    anchor[g * 32 + lane] = make_uint4(pa[0], pa[1], pa[2], pa[3]);
    residual[g * 32 + lane] = make_uint4(pr[0], pr[1], pr[2], pr[3]);

    const int64_t page = g >> 5;
    const int rgrp = (int)(g & 31);
    float* mp = meta + page * kMetaFloats;
    const int ch = 4 * rgrp + (lane >> 3);
    if ((lane & 7) == 0) {
      mp[ch] = mn;
      mp[kH + ch] = gscale;
    }
    mp[kMetaMuOff + (lane & 7) * kH + ch] = mu;
    mp[kMetaSigmaOff + (lane & 7) * kH + ch] = sigma;
  }
}

}  // namespace

cudaError_t launch_encode(const void* x, int64_t n_pages, uint8_t* anchor, uint8_t* residual,
                          float* meta, const EncodeTables* tab, cudaStream_t s) {
  const int64_t n_groups = n_pages * 32;
  const int threads = 256;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_kernel, threads, 0);
  if (per_sm < 1) per_sm = 1;
  const int64_t max_blocks = (int64_t)device_sm_count() * per_sm;
  const int64_t need = (n_groups + 7) / 8;
  const int blocks = (int)(need < max_blocks ? need : max_blocks);
  encode_kernel<<<blocks, threads, 0, s>>>(static_cast<const uint4*>(x), n_groups,
                                          reinterpret_cast<uint4*>(anchor),
                                          reinterpret_cast<uint4*>(residual), meta, *tab);
  return cudaGetLastError();
}

}  // namespace lynx
