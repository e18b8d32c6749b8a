// lynx_decode_attn kernels: split-K flash decoding over Lynx-encoded KV pages
// (the attention of the Lynx paper's §2.1 run by the decode instance on the
// draft KV of the Anchor phase and on the full codes of the verification pass,
// §4.2-4.3), plus the same attention over plain BF16 pages as a baseline.
//
// Grid: x = split of the sequence's pages, y = (KV head, group of 4 query
// rows), z = sequence.  A query row is one (draft token, query head) pair of
// the GQA group that shares the KV head.  Each CTA (256 threads) walks its
// pages one at a time, keeping an online softmax; a second kernel merges the
// splits with their log-sum-exps.
//
// Staging.  A page's K unit (packed plane(s) + metadata, or the BF16 page) and
// V unit are copied into a ring of shared-memory slots with 1-D bulk async
// copies (cp.async.bulk) completing on one mbarrier per slot; every wait on a
// slot is bounded in time and, if it gives up, the CTA records an error in
// the device status word, drains its outstanding copies and exits.
//
// Dequantisation in registers without materialising K or V.  With
// A = gamma_min + (gamma_scale+eps) mu and B = (gamma_scale+eps)(sigma+eps)
// per (channel d, 32-token chunk b), every key element is A + B * l~ where
// l~ = S l(I_hat) is a table value of the code, so
//   q.k_t = sum_d q_d A_{d,b} + sum_d (q_d B_{d,b}) l~_{d,t}
//   sum_t p_t v_{d,t} = A_{d,b} sum_{t in b} p_t + B_{d,b} sum_{t in b} p_t l~_{d,t}.
// The per-element work is a code -> l~ table lookup (one lookup yields both
// tokens of a byte for the anchor stream) and packed float2 FMAs (FFMA2); the
// per-chunk factors are applied once per 32 tokens.
//
// K phase: warp w covers channels 16w..16w+15, lane L tokens 8L..8L+7; the 8
// warps' partial logits meet in shared memory.  V phase: lane L covers chunk
// (L & 7) of channels 16w + (L >> 3) + 4k, k = 0..3, accumulating its own
// partial outputs across pages; lanes of one channel are reduced at the end.

#include "lynx_internal.cuh"
#include "tma_ptx.cuh"

#include <cuda_bf16.h>
#include <math_constants.h>

namespace lynx {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 4;
constexpr int kWsPerCta = kRows * kH + 2 * kRows;   // o[4][128], m[4], l[4]

template <int MODE>
struct Geo;
template <>
struct Geo<kModeAnchor> {
  static constexpr int kStages = 4;
  static constexpr int kUnit = kPlaneBytes + kMetaBytes;
  static constexpr int kResOff = 0;
  static constexpr int kMetaOff = kPlaneBytes;
  static constexpr int kLutBytes = 256 * 16 * 8;   // byte -> float2, 16 copies
  static constexpr int kCoefBytes = kH * kChunks * 8 * 4;
};
template <>
struct Geo<kModeFull> {
  static constexpr int kStages = 2;
  static constexpr int kUnit = 2 * kPlaneBytes + kMetaBytes;
  static constexpr int kResOff = kPlaneBytes;
  static constexpr int kMetaOff = 2 * kPlaneBytes;
  static constexpr int kLutBytes = 256 * 32 * 4;   // code -> float, 32 copies
  static constexpr int kCoefBytes = kH * kChunks * 8 * 4;
};
template <>
struct Geo<kModeBf16> {
  static constexpr int kStages = 2;
  static constexpr int kUnit = kPageElems * 2;
  static constexpr int kResOff = 0;
  static constexpr int kMetaOff = 0;
  static constexpr int kLutBytes = 0;
  static constexpr int kCoefBytes = kH * 8 * 4;     // duplicated scaled queries
};

template <int MODE>
struct Layout {
  using G = Geo<MODE>;
  static constexpr int kRing = 0;
  static constexpr int kLut = kRing + G::kStages * G::kUnit;
  static constexpr int kPart = kLut + G::kLutBytes;           // [8 warps][4 rows][64 float4]
  static constexpr int kCoef = kPart + 8 * kRows * kP * 4;
  static constexpr int kConstK = kCoef + G::kCoefBytes;       // [8 chunks][4 rows]
  static constexpr int kPs01 = kConstK + kChunks * kRows * 4; // [16 pairs][8 chunks] float4
  static constexpr int kPs23 = kPs01 + 16 * 8 * 16;
  static constexpr int kPb = kPs23 + 16 * 8 * 16;             // [2 halves][8 chunks][4 rows]
  static constexpr int kRedMax = kPb + 2 * kChunks * kRows * 4;  // [2 halves][4 rows]
  static constexpr int kRedSum = kRedMax + 2 * kRows * 4;
  static constexpr int kQs = kRedSum + 2 * kRows * 4;         // [128 d][4 rows]
  static constexpr int kBar = kQs + kH * kRows * 4;
  static constexpr int kTotal = kBar + G::kStages * 8;
};

static_assert(Layout<kModeAnchor>::kTotal <= 232448, "shared memory");
static_assert(Layout<kModeFull>::kTotal <= 232448, "shared memory");
static_assert(Layout<kModeBf16>::kTotal <= 232448, "shared memory");

// ---------------------------------------------------------------- PTX helpers

// (mbarrier, bulk-copy and bounded-wait helpers: tma_ptx.cuh)

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

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

// ------------------------------------------------------------------ kernel

template <int MODE>
__device__ __forceinline__ void issue_unit(const DecodeArgs& a, int u, int p_begin,
                                           const int32_t* __restrict__ pt_row, uint8_t* ring,
                                           uint32_t bar0) {
  using G = Geo<MODE>;
  const int slot = u % G::kStages;
  const int p = p_begin + (u >> 1);
  const bool is_v = (u & 1) != 0;
  int64_t id = pt_row[p];
  if (id < 0 || id >= a.n_pool) {   // invalid page id: record it, read page 0 instead
    atomicExch(a.status, 2);
    id = 0;
  }
  const uint32_t dst = smem_u32(ring + slot * G::kUnit);
  const uint32_t bar = bar0 + slot * 8;
  mbar_expect_tx(bar, G::kUnit);
  if (MODE == kModeBf16) {
    const uint16_t* src = (is_v ? a.v_bf16 : a.k_bf16) + id * kPageElems;
    bulk_g2s(dst, src, G::kUnit, bar);
  } else {
    const uint8_t* anc = (is_v ? a.v_anc : a.k_anc) + id * kPlaneBytes;
    const float* meta = (is_v ? a.v_meta : a.k_meta) + id * kMetaFloats;
    bulk_g2s(dst, anc, kPlaneBytes, bar);
    if (MODE == kModeFull) {
      const uint8_t* res = (is_v ? a.v_res : a.k_res) + id * kPlaneBytes;
      bulk_g2s(dst + G::kResOff, res, kPlaneBytes, bar);
    }
    bulk_g2s(dst + G::kMetaOff, meta, kMetaBytes, bar);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
decode_split_kernel(const DecodeArgs a, const LutTables lut) {
  using G = Geo<MODE>;
  using S = Layout<MODE>;
  constexpr int kSt = G::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem + S::kRing;
  float* s_part = reinterpret_cast<float*>(smem + S::kPart);
  float* s_coef = reinterpret_cast<float*>(smem + S::kCoef);
  float* s_constk = reinterpret_cast<float*>(smem + S::kConstK);
  float4* s_ps01 = reinterpret_cast<float4*>(smem + S::kPs01);
  float4* s_ps23 = reinterpret_cast<float4*>(smem + S::kPs23);
  float* s_pb = reinterpret_cast<float*>(smem + S::kPb);
  float* s_redmax = reinterpret_cast<float*>(smem + S::kRedMax);
  float* s_redsum = reinterpret_cast<float*>(smem + S::kRedSum);
  float* s_qs = reinterpret_cast<float*>(smem + S::kQs);
  const uint32_t bar0 = smem_u32(smem + S::kBar);

  const int tid = threadIdx.x;
  const int w = tid >> 5;
  const int L = tid & 31;
  const int split = blockIdx.x;
  const int h = blockIdx.y / a.n_rg;
  const int rg = blockIdx.y % a.n_rg;
  const int b = blockIdx.z;
  const int64_t cta = ((int64_t)b * gridDim.y + blockIdx.y) * a.n_splits + split;
  const int TG = a.T * a.G;
  const int max_keys = a.max_pages * kP;

  wait_prerequisite_grids();   // every global-memory access of this kernel follows it
  int ctx = a.ctx_len[b];
  if (ctx < 0 || ctx > max_keys) {
    if (tid == 0) atomicExch(a.status, 3);
    ctx = ctx < 0 ? 0 : max_keys;
  }
  int nvis[kRows];
  int max_vis = 0;
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int row = rg * kRows + r;
    int n = 0;
    if (row < TG) n = a.causal ? ctx - a.T + row / a.G + 1 : ctx;
    n = n < 0 ? 0 : n;
    nvis[r] = n;
    max_vis = max(max_vis, n);
  }
  const int n_pages = (max_vis + kP - 1) / kP;
  const int p_begin = split * a.pages_per_split;
  const int np = max(min(p_begin + a.pages_per_split, n_pages) - p_begin, 0);
  const int n_units = 2 * np;
  const int32_t* pt_row = a.page_table + ((int64_t)b * a.Hkv + h) * a.max_pages;

  // queries, scaled by sm_scale * log2(e): s_qs[d][r]
  for (int i = tid; i < kH * kRows; i += kThreads) {
    const int d = i >> 2, r = i & 3, row = rg * kRows + r;
    float v = 0.0f;
    if (row < TG) {
      const int t = row / a.G, hq = h * a.G + row % a.G;
      const uint16_t bits = a.q[(((int64_t)b * a.T + t) * a.Hq + hq) * kH + d];
      v = __uint_as_float((uint32_t)bits << 16) * a.scale_log2;
    }
    s_qs[i] = v;
  }
  if (MODE == kModeAnchor) {
    float2* lut2 = reinterpret_cast<float2*>(smem + S::kLut);
    for (int i = tid; i < 256 * 16; i += kThreads) lut2[i] = lut.anc_pair[i >> 4];
  } else if (MODE == kModeFull) {
    float* lutf = reinterpret_cast<float*>(smem + S::kLut);
    for (int i = tid; i < 256 * 32; i += kThreads) lutf[i] = lut.full[i >> 5];
  }
  if (tid == 0) {
    for (int s = 0; s < kSt; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (MODE == kModeBf16) {
    // duplicated query pairs (q_r, q_r) for the packed FMAs: s_coef[d][8]
    for (int i = tid; i < kH * 8; i += kThreads) s_coef[i] = s_qs[(i >> 3) * 4 + ((i & 7) >> 1)];
  }
  int issued = 0;
  if (tid == 0) {
    for (; issued < kSt && issued < n_units; ++issued)
      issue_unit<MODE>(a, issued, p_begin, pt_row, ring, bar0);
  }

  float m_run[kRows], l_run[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    m_run[r] = -CUDART_INF_F;
    l_run[r] = 0.0f;
  }
  float O[4][kRows];
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int r = 0; r < kRows; ++r) O[k][r] = 0.0f;

  const float eps = a.eps;
  const int blk_k = L >> 2;          // K phase: chunk of this lane's tokens
  const int blk_v = L & 7;           // V phase: chunk owned by this lane
  const int c4 = L >> 3;             // V phase: channel offset within the warp's 16
  bool failed = false;
  int consumed = 0;

  for (int i = 0; i < np; ++i) {
    const int p = p_begin + i;
    const int uK = 2 * i, uV = 2 * i + 1;
    const uint8_t* unitK = ring + (uK % kSt) * G::kUnit;
    const uint8_t* unitV = ring + (uV % kSt) * G::kUnit;

    // ---------------- K unit: per-chunk coefficients
    if (!mbar_wait(bar0 + 8 * (uK % kSt), (uK / kSt) & 1)) failed = true;
    if (MODE != kModeBf16 && !failed) {
      const float* km = reinterpret_cast<const float*>(unitK + G::kMetaOff);
      const int blk = w;
      float cp[kRows] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int d = 4 * L + j;
        const float gmin = km[d];
        const float dg = __fadd_rn(km[kH + d], eps);
        const float mu = km[kMetaMuOff + blk * kH + d];
        const float ds = __fadd_rn(km[kMetaSigmaOff + blk * kH + d], eps);
        const float A = __fmaf_rn(dg, mu, gmin);
        const float Bc = __fmul_rn(dg, ds);
        const float4 q = reinterpret_cast<const float4*>(s_qs)[d];
        float4* cf = reinterpret_cast<float4*>(s_coef) + (d * kChunks + blk) * 2;
        cf[0] = make_float4(q.x * Bc, q.x * Bc, q.y * Bc, q.y * Bc);
        cf[1] = make_float4(q.z * Bc, q.z * Bc, q.w * Bc, q.w * Bc);
        cp[0] = __fmaf_rn(q.x, A, cp[0]);
        cp[1] = __fmaf_rn(q.y, A, cp[1]);
        cp[2] = __fmaf_rn(q.z, A, cp[2]);
        cp[3] = __fmaf_rn(q.w, A, cp[3]);
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) cp[r] = warp_sum(cp[r]);
      if (L == 0) reinterpret_cast<float4*>(s_constk)[blk] = make_float4(cp[0], cp[1], cp[2], cp[3]);
    }
    if (__syncthreads_or(failed)) {
      failed = true;
      break;
    }

    // ---------------- K phase: partial logits of 16 channels x 8 tokens x 4 rows
    {
      float2 acc[kRows][4];
#pragma unroll
      for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[r][k] = make_float2(0.f, 0.f);
      if (MODE == kModeBf16) {
        const uint4* kp = reinterpret_cast<const uint4*>(unitK);
        const float4* qd = reinterpret_cast<const float4*>(s_coef);
#pragma unroll 4
        for (int dd = 0; dd < 16; ++dd) {
          const int d = 16 * w + dd;
          const uint4 kv = kp[d * 32 + L];
          const float4 q01 = qd[d * 2], q23 = qd[d * 2 + 1];
          const float2 qq[4] = {make_float2(q01.x, q01.y), make_float2(q01.z, q01.w),
                                make_float2(q23.x, q23.y), make_float2(q23.z, q23.w)};
          const uint32_t wv[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 kk = make_float2(bf16lo(wv[k]), bf16hi(wv[k]));
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[r][k] = __ffma2_rn(qq[r], kk, acc[r][k]);
          }
        }
      } else {
        const uint32_t* pa = reinterpret_cast<const uint32_t*>(unitK);
        const uint32_t* pr = reinterpret_cast<const uint32_t*>(unitK + G::kResOff);
        const float4* cf = reinterpret_cast<const float4*>(s_coef);
        const float2* lut2 = reinterpret_cast<const float2*>(smem + S::kLut) + (L & 15);
        const float* lutf = reinterpret_cast<const float*>(smem + S::kLut) + L;
#pragma unroll 4
        for (int dd = 0; dd < 16; ++dd) {
          const int d = 16 * w + dd;
          const uint32_t wa = pa[d * 32 + L];
          const uint32_t wr = (MODE == kModeFull) ? pr[d * 32 + L] : 0u;
          const float4 c01 = cf[(d * kChunks + blk_k) * 2];
          const float4 c23 = cf[(d * kChunks + blk_k) * 2 + 1];
          const float2 cc[4] = {make_float2(c01.x, c01.y), make_float2(c01.z, c01.w),
                                make_float2(c23.x, c23.y), make_float2(c23.z, c23.w)};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float2 lv;
            if (MODE == kModeAnchor) {
              lv = lut2[((wa >> (8 * k)) & 0xFFu) * 16];
            } else {
              const uint32_t c0 = ((wa >> (8 * k)) & 0xFu) | (((wr >> (8 * k)) & 0xFu) << 4);
              const uint32_t c1 = ((wa >> (8 * k + 4)) & 0xFu) | (((wr >> (8 * k + 4)) & 0xFu) << 4);
              lv = make_float2(lutf[c0 * 32], lutf[c1 * 32]);
            }
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[r][k] = __ffma2_rn(cc[r], lv, acc[r][k]);
          }
        }
      }
      // partials: s_part[w][r][64 float4]; tokens 8L..8L+3 at float4 L, 8L+4..8L+7 at 32+L
      float4* pp = reinterpret_cast<float4*>(s_part) + w * kRows * 64;
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        pp[r * 64 + L] = make_float4(acc[r][0].x, acc[r][0].y, acc[r][1].x, acc[r][1].y);
        pp[r * 64 + 32 + L] = make_float4(acc[r][2].x, acc[r][2].y, acc[r][3].x, acc[r][3].y);
      }
    }
    fence_proxy_async();
    __syncthreads();
    ++consumed;
    if (tid == 0 && issued < n_units) {
      issue_unit<MODE>(a, issued, p_begin, pt_row, ring, bar0);
      ++issued;
    }

    // ---------------- softmax: thread -> (row r = tid / 64, float4 q = tid % 64)
    float corr[kRows];
    {
      const int r = tid >> 6;
      const int qv = tid & 63;
      const int half = qv >> 5;           // tokens 8j + 4*half + 0..3, j = qv & 31
      const int j = qv & 31;
      const float4* pp = reinterpret_cast<const float4*>(s_part);
      float4 s = pp[r * 64 + qv];
#pragma unroll
      for (int ww = 1; ww < 8; ++ww) {
        const float4 t = pp[(ww * kRows + r) * 64 + qv];
        s.x += t.x; s.y += t.y; s.z += t.z; s.w += t.w;
      }
      const int blk = j >> 2;
      if (MODE != kModeBf16) {
        const float c = s_constk[blk * kRows + r];
        s.x += c; s.y += c; s.z += c; s.w += c;
      }
      const int tok0 = p * kP + 8 * j + 4 * half;
      int my_nvis = nvis[0];
#pragma unroll
      for (int rr = 1; rr < kRows; ++rr) my_nvis = (r == rr) ? nvis[rr] : my_nvis;
      float sv[4] = {s.x, s.y, s.z, s.w};
      float mloc = -CUDART_INF_F;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (tok0 + e >= my_nvis) sv[e] = -CUDART_INF_F;
        mloc = fmaxf(mloc, sv[e]);
      }
      mloc = warp_max(mloc);
      if (L == 0) s_redmax[half * kRows + r] = mloc;
      __syncthreads();
      float mnew[kRows];
      float my_m = 0.0f;
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr) {
        mnew[rr] = fmaxf(m_run[rr], fmaxf(s_redmax[rr], s_redmax[kRows + rr]));
        corr[rr] = (mnew[rr] == -CUDART_INF_F) ? 1.0f : exp2f(m_run[rr] - mnew[rr]);
        my_m = (r == rr) ? mnew[rr] : my_m;
      }
      float pv[4];
      float psum = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pv[e] = (sv[e] == -CUDART_INF_F) ? 0.0f : exp2f(sv[e] - my_m);
        psum += pv[e];
      }
      // chunk sums (4 lanes share a chunk within this half) and row sums
      float csum = psum + __shfl_xor_sync(0xffffffffu, psum, 1);
      csum += __shfl_xor_sync(0xffffffffu, csum, 2);
      if ((j & 3) == 0) s_pb[(half * kChunks + blk) * kRows + r] = csum;
      const float rsum = warp_sum(psum);
      if (L == 0) s_redsum[half * kRows + r] = rsum;
      // probabilities for the V phase: pairs m = 4(j%4) + 2*half + {0,1} of chunk blk
      float* p01 = reinterpret_cast<float*>(s_ps01);
      float* p23 = reinterpret_cast<float*>(s_ps23);
      float* dst = (r < 2) ? p01 : p23;
      const int comp = (r & 1) * 2;
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int m = 4 * (j & 3) + 2 * half + e2;
        *reinterpret_cast<float2*>(dst + (m * kChunks + blk) * 4 + comp) =
            make_float2(pv[2 * e2], pv[2 * e2 + 1]);
      }
      __syncthreads();
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr) {
        l_run[rr] = l_run[rr] * corr[rr] + s_redsum[rr] + s_redsum[kRows + rr];
        m_run[rr] = mnew[rr];
      }
    }

    // ---------------- V phase
    if (!mbar_wait(bar0 + 8 * (uV % kSt), (uV / kSt) & 1)) failed = true;
    if (!failed) {
      float pb[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r)
        pb[r] = s_pb[blk_v * kRows + r] + s_pb[(kChunks + blk_v) * kRows + r];
      float2 acc[4][kRows];
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int r = 0; r < kRows; ++r) acc[k][r] = make_float2(0.f, 0.f);
      if (MODE == kModeBf16) {
        const uint4* vp = reinterpret_cast<const uint4*>(unitV);
        // 4 pieces of 8 tokens; the piece order is rotated per lane so that the
        // 8 lanes of a quarter-warp hit 8 different 16-byte bank groups
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int piece = (jj + (blk_v >> 1)) & 3;
          uint4 vv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int ch = 16 * w + c4 + 4 * k;
            vv[k] = vp[ch * 32 + blk_v * 4 + piece];
          }
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int m = 4 * piece + e2;
            const float4 a01 = s_ps01[m * kChunks + blk_v];
            const float4 a23 = s_ps23[m * kChunks + blk_v];
            const float2 pr[4] = {make_float2(a01.x, a01.y), make_float2(a01.z, a01.w),
                                  make_float2(a23.x, a23.y), make_float2(a23.z, a23.w)};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t wv = (e2 == 0) ? vv[k].x : (e2 == 1) ? vv[k].y : (e2 == 2) ? vv[k].z : vv[k].w;
              const float2 v2 = make_float2(bf16lo(wv), bf16hi(wv));
#pragma unroll
              for (int r = 0; r < kRows; ++r) acc[k][r] = __ffma2_rn(pr[r], v2, acc[k][r]);
            }
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int r = 0; r < kRows; ++r) O[k][r] = O[k][r] * corr[r] + (acc[k][r].x + acc[k][r].y);
      } else {
        const uint4* pa = reinterpret_cast<const uint4*>(unitV);
        const uint4* pr4 = reinterpret_cast<const uint4*>(unitV + G::kResOff);
        const float* vm = reinterpret_cast<const float*>(unitV + G::kMetaOff);
        const float2* lut2 = reinterpret_cast<const float2*>(smem + S::kLut) + (L & 15);
        const float* lutf = reinterpret_cast<const float*>(smem + S::kLut) + L;
        uint4 va[4], vr[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int ch = 16 * w + c4 + 4 * k;
          va[k] = pa[ch * 8 + blk_v];
          vr[k] = (MODE == kModeFull) ? pr4[ch * 8 + blk_v] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float4 a01 = s_ps01[m * kChunks + blk_v];
          const float4 a23 = s_ps23[m * kChunks + blk_v];
          const float2 pp[4] = {make_float2(a01.x, a01.y), make_float2(a01.z, a01.w),
                                make_float2(a23.x, a23.y), make_float2(a23.z, a23.w)};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t wa = (m < 4) ? va[k].x : (m < 8) ? va[k].y : (m < 12) ? va[k].z : va[k].w;
            const uint32_t byte = (wa >> (8 * (m & 3))) & 0xFFu;
            float2 lv;
            if (MODE == kModeAnchor) {
              lv = lut2[byte * 16];
            } else {
              const uint32_t wr = (m < 4) ? vr[k].x : (m < 8) ? vr[k].y : (m < 12) ? vr[k].z : vr[k].w;
              const uint32_t rb = (wr >> (8 * (m & 3))) & 0xFFu;
              const uint32_t c0 = (byte & 0xFu) | ((rb & 0xFu) << 4);
              const uint32_t c1 = (byte >> 4) | (rb & 0xF0u);
              lv = make_float2(lutf[c0 * 32], lutf[c1 * 32]);
            }
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[k][r] = __ffma2_rn(pp[r], lv, acc[k][r]);
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int ch = 16 * w + c4 + 4 * k;
          const float gmin = vm[ch];
          const float dg = __fadd_rn(vm[kH + ch], eps);
          const float mu = vm[kMetaMuOff + blk_v * kH + ch];
          const float ds = __fadd_rn(vm[kMetaSigmaOff + blk_v * kH + ch], eps);
          const float A = __fmaf_rn(dg, mu, gmin);
          const float Bc = __fmul_rn(dg, ds);
#pragma unroll
          for (int r = 0; r < kRows; ++r)
            O[k][r] = O[k][r] * corr[r] + A * pb[r] + Bc * (acc[k][r].x + acc[k][r].y);
        }
      }
    }
    fence_proxy_async();
    if (__syncthreads_or(failed)) {
      failed = true;
      break;
    }
    ++consumed;
    if (tid == 0 && issued < n_units) {
      issue_unit<MODE>(a, issued, p_begin, pt_row, ring, bar0);
      ++issued;
    }
  }

  if (failed) {
    // drain this CTA's outstanding copies (bounded), record the error, leave
    if (tid == 0) {
      atomicExch(a.status, 1);
      for (int u = consumed; u < issued; ++u) mbar_wait(bar0 + 8 * (u % kSt), (u / kSt) & 1);
    }
    return;
  }

  allow_dependent_launch();   // the split combine may be scheduled once every CTA is here
  // reduce the 8 chunk lanes of each channel, write this split's partials
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      float v = O[k][r];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      O[k][r] = v;
    }
  float* ws = a.ws + cta * kWsPerCta;
  if (blk_v == 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int ch = 16 * w + c4 + 4 * k;
#pragma unroll
      for (int r = 0; r < kRows; ++r) ws[r * kH + ch] = O[k][r];
    }
  }
  if (tid < kRows) {
    ws[kRows * kH + tid] = m_run[tid];
    ws[kRows * kH + kRows + tid] = l_run[tid];
  }
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

template <int MODE>
cudaError_t launch_mode(const DecodeArgs& a, const LutTables* lut, cudaStream_t s) {
  constexpr int kSmem = Layout<MODE>::kTotal;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  dim3 grid(a.n_splits, a.Hkv * a.n_rg, a.B);
  const cudaError_t e = launch_programmatic(decode_split_kernel<MODE>, grid, dim3(kThreads), kSmem, s, a, *lut);
  if (e != cudaSuccess) return e;
  return launch_combine(a, s);
}

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
  const bool quant = mode != kModeBf16;
  const int q_rows = !quant ? kRows : use_tc_rows(T * G) ? tc_rows_per_cta(T * G, mode == kModeFull) : kNarrowRows;
  const int64_t cta_units = quant ? (int64_t)B * Hkv * ((T * G + q_rows - 1) / q_rows) : units;
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
  if (mode == kModeBf16) return launch_mode<kModeBf16>(a, lut, s);
  const cudaError_t e = launch_decode_quant(a, mode == kModeFull, lut, s);
  if (e != cudaSuccess) return e;
  return launch_combine(a, s);
}

}  // namespace lynx
