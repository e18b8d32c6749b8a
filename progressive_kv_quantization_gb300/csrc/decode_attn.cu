// Split-K plumbing shared by the decode attention kernels (the attention of
// the Lynx paper's §2.1, run on the draft KV of the Anchor phase, on the full
// codes of the verification pass (§4.2-4.3) and on plain BF16 pages): the
// split plan, the combine kernel that merges a call's splits with their
// log-sum-exps, the merge of two attention results over disjoint key sets,
// and the dispatch of a decode call to its kernels.
//
// Grid of every decode kernel: x = split of the sequence's pages, y = (KV
// head, tile of query rows), z = sequence.  A query row is one (draft token,
// query head) pair of the GQA group that shares the KV head.  Each CTA writes,
// per 4-row group of its rows, its unnormalised output, maximum and
// denominator to the workspace; decode_combine_kernel merges the splits.

#include "lynx_internal.cuh"

#include <math_constants.h>

namespace lynx {
namespace {

constexpr int kRows = 4;
constexpr int kWsPerCta = kRows * kH + 2 * kRows;   // o[4][128], m[4], l[4]

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

// Merge the splits of one query row: grid (n_rg * 4, Hkv, B), 128 threads
// (thread d = output channel d).  The splits' maxima and denominators are
// gathered by all threads at once (split s by thread s mod 128) and reduced
// across the block; each split's weight 2^(m_s - m*) goes to shared memory;
// then thread d sums its channel over the splits in order, eight loads in
// flight.  A split that saw no key (m_s = -inf) has weight 0 and its partial
// output is not read into the sum.
constexpr int kMaxSplits = 1024;

__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeArgs a) {
  __shared__ float s_w[kMaxSplits];
  __shared__ float s_red[2][4];
  allow_dependent_launch();
  wait_prerequisite_grids();
  const int r = blockIdx.x & 3;
  const int rg = blockIdx.x >> 2;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int row = rg * kRows + r;
  if (row >= a.T * a.G) return;
  const int t = row / a.G, hq = h * a.G + row % a.G;
  const int d = threadIdx.x;
  const int warp = d >> 5, lane = d & 31;
  const int n = a.n_splits;
  const int64_t cta0 = (((int64_t)b * a.Hkv + h) * a.n_rg + rg) * n;
  const float* ws = a.ws + cta0 * kWsPerCta;
  const int64_t o_idx = (((int64_t)b * a.T + t) * a.Hq + hq);

  float mloc = -CUDART_INF_F;
  for (int s = d; s < n; s += kH) mloc = fmaxf(mloc, ws[(int64_t)s * kWsPerCta + kRows * kH + r]);
  mloc = warp_max(mloc);
  if (lane == 0) s_red[0][warp] = mloc;
  __syncthreads();
  const float mstar = fmaxf(fmaxf(s_red[0][0], s_red[0][1]), fmaxf(s_red[0][2], s_red[0][3]));
  if (mstar == -CUDART_INF_F) {
    a.out[o_idx * kH + d] = 0.0f;
    if (d == 0 && a.lse) a.lse[o_idx] = -CUDART_INF_F;
    return;
  }
  float lloc = 0.0f;
  for (int s = d; s < n; s += kH) {
    const float* w = ws + (int64_t)s * kWsPerCta;
    const float ms = w[kRows * kH + r];
    const float f = (ms == -CUDART_INF_F) ? 0.0f : exp2f(ms - mstar);
    s_w[s] = f;
    if (f != 0.0f) lloc = fmaf(w[kRows * kH + kRows + r], f, lloc);
  }
  lloc = warp_sum(lloc);
  if (lane == 0) s_red[1][warp] = lloc;
  __syncthreads();
  const float l = (s_red[1][0] + s_red[1][1]) + (s_red[1][2] + s_red[1][3]);

  const float* od = ws + r * kH + d;
  float o = 0.0f;
  int s = 0;
  for (; s + 32 <= n; s += 32) {
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = od[(int64_t)(s + k) * kWsPerCta];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float f = s_w[s + k];
      o = (f != 0.0f) ? fmaf(v[k], f, o) : o;
    }
  }
  for (; s + 8 <= n; s += 8) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = od[(int64_t)(s + k) * kWsPerCta];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float f = s_w[s + k];
      o = (f != 0.0f) ? fmaf(v[k], f, o) : o;
    }
  }
  for (; s < n; ++s) {
    const float f = s_w[s];
    const float v = od[(int64_t)s * kWsPerCta];
    o = (f != 0.0f) ? fmaf(v, f, o) : o;
  }
  a.out[o_idx * kH + d] = o / l;
  if (d == 0 && a.lse) a.lse[o_idx] = (mstar + log2f(l)) * 0.6931471805599453f;
}

// Log-sum-exp merge of two attention results over disjoint key sets: one warp
// per row, lane L holds channels 4L..4L+3.
__global__ void __launch_bounds__(256)
attn_merge_kernel(const float* __restrict__ oa, const float* __restrict__ la,
                  const float* __restrict__ ob, const float* __restrict__ lb, int64_t rows,
                  float* o, float* lse) {
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += n_warps) {
    const float a = la[r], b = lb[r];
    const float m = fmaxf(a, b);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = -CUDART_INF_F;
    if (m != -CUDART_INF_F) {
      const float wa = (a == -CUDART_INF_F) ? 0.0f : expf(a - m);
      const float wb = (b == -CUDART_INF_F) ? 0.0f : expf(b - m);
      const float s = wa + wb;
      const float4 x = reinterpret_cast<const float4*>(oa + r * kH)[lane];
      const float4 y = reinterpret_cast<const float4*>(ob + r * kH)[lane];
      v = make_float4((wa * x.x + wb * y.x) / s, (wa * x.y + wb * y.y) / s, (wa * x.z + wb * y.z) / s,
                      (wa * x.w + wb * y.w) / s);
      l = m + logf(s);
    }
    __syncwarp();   // every lane has read row r before it is overwritten in place
    reinterpret_cast<float4*>(o + r * kH)[lane] = v;
    if (lane == 0) lse[r] = l;
  }
}

cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s);

// The combine of a decode call, launched as a programmatic dependent of the
// decode kernel just issued on s (it waits for that grid inside the kernel).
cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s) {
  return launch_programmatic(decode_combine_kernel, dim3(a.n_rg * kRows, a.Hkv, a.B), dim3(kH), 0, s, a);
}

}  // namespace

DecodePlan plan_decode(int B, int T, int Hq, int Hkv, int max_pages, int mode) {
  DecodePlan pl{};
  const int G = Hq / Hkv;
  pl.n_rg = (T * G + kRows - 1) / kRows;
  const int64_t units = (int64_t)B * Hkv * pl.n_rg;
  // CTAs per split: the quantised kernels take 8, 16 or 32 query rows per CTA
  const int q_rows = mode == kModeBf16         ? bf16_rows_per_cta(T * G)
                     : use_tc_rows(T * G)        ? tc_rows_per_cta(T * G, mode == kModeFull)
                                                 : kNarrowRows;
  const int64_t cta_units = (int64_t)B * Hkv * ((T * G + q_rows - 1) / q_rows);
  const int64_t resident = device_sm_count();   // one CTA per SM (shared-memory bound)
  int best_s = 1;
  double best = 1e300;
  const int s_max = max_pages < kMaxSplits ? max_pages : kMaxSplits;
  for (int s = 1; s <= s_max; ++s) {
    const int pps = (max_pages + s - 1) / s;
    const int s_eff = (max_pages + pps - 1) / pps;
    if (s_eff != s) continue;
    const int64_t ctas = cta_units * s_eff;
    const int64_t waves = (ctas + resident - 1) / resident;
    const double cost = (double)waves * (pps + 2.0);
    if (cost < best - 1e-9) {
      best = cost;
      best_s = s_eff;
    }
  }
  pl.n_splits = best_s;
  pl.pages_per_split = (max_pages + best_s - 1) / best_s;
  pl.ws_bytes = (size_t)units * pl.n_splits * kWsPerCta * sizeof(float);
  return pl;
}

cudaError_t launch_attn_merge(const float* oa, const float* la, const float* ob, const float* lb,
                              int64_t rows, float* o, float* lse, cudaStream_t s) {
  const int64_t blocks = (rows + 7) / 8;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  attn_merge_kernel<<<(int)(blocks < cap ? blocks : cap), 256, 0, s>>>(oa, la, ob, lb, rows, o, lse);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, int mode, const LutTables* lut, cudaStream_t s) {
  const cudaError_t e = mode == kModeBf16 ? launch_decode_bf16(a, s) : launch_decode_quant(a, mode == kModeFull, lut, s);
  if (e != cudaSuccess) return e;
  return launch_combine(a, s);
}

}  // namespace lynx
