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
// stores are contiguous 512-byte runs.  The next row group's 64 bytes are
// prefetched into registers while the current one is processed.
//
// Exactness.  Every Stage 1-2 step is a single correctly rounded float32
// operation (packed two-wide where the values come in pairs; no contraction).
// Each division x / d by a per-row or per-chunk divisor d uses r = RN(1/d),
// then q = RN(x r) corrected by one FMA residual step, q' = RN(q + r (x - q d))
// (Markstein's FMA division correction), which returns the correctly rounded
// quotient.  The Stage 2 quotient |x_c| / (sigma + eps) feeds only the code
// decision: the estimate takes alpha |x_f| as |x_c| RN(alpha r), inside the fused
// multiply-add that forms 1 + alpha |x_f| (relative error below 2^-23; one
// product per chunk), and the correctly rounded quotient is formed where the
// code is decided from the threshold table.  sigma = max_t |x_n,t - mu| is taken as
// max(RN(x_n(max x) - mu), RN(mu - x_n(min x))): every step from x to
// x_n - mu is a monotone rounding, so the extreme deviations sit at the
// chunk's extreme inputs and the value is the same.  The Stage 3 code
// round(127 ln(1+alpha a)/ln(1+alpha)) is estimated with the hardware log2
// and rounded by adding 1.5 * 2^23; when the estimate lies within a safety
// margin of a rounding edge the code is decided exactly from the threshold
// table (the smallest float32 of each code).
//
// Packing.  The lane's 32 codes sit in the low bytes of the rounded floats;
// byte permutes gather the even and the odd tokens of each group of eight into
// two words (and the sign bytes likewise, straight from the float sign bits),
// and two masked logic steps form the anchor nibbles ((S>0 ? I : ~I) >> 4) and
// the residual nibbles ((7 - I) mod 16 = (I ^ 7) & 15) of all eight tokens,
// even tokens in the low and odd tokens in the high nibbles.

#include "lynx_internal.cuh"
#include "tma_ptx.cuh"

#include <cuda_bf16.h>

namespace lynx {
namespace {

constexpr float kMagic = 12582912.0f;     // 1.5 * 2^23: x + kMagic rounds x to an integer
constexpr uint32_t kMagicBits = 0x4B400000u;

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// (x_lo + c, x_hi + c) for the two BF16 values of w, each one float32
// addition of the exactly converted BF16 value (mixed-precision add)
__device__ __forceinline__ float2 sub_min_bf16x2(uint32_t w, float c) {
  float2 r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %3;\n\tadd.rn.f32.bf16 %1, hi, %3;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "r"(w), "f"(c));
  return r;
}

// correctly rounded x / d for a pair, given r = RN(1/d) and nd = -d
__device__ __forceinline__ float2 div2(float2 x, float2 nd, float2 r) {
  const float2 q = __fmul2_rn(x, r);
  const float2 e = __ffma2_rn(q, nd, x);
  return __ffma2_rn(e, r, q);
}

__device__ __forceinline__ float div1(float x, float d, float r) {
  const float q = __fmul_rn(x, r);
  const float e = __fmaf_rn(-q, d, x);
  return __fmaf_rn(e, r, q);
}

// max(a, b, c) in one instruction (three-input max of sm_100 and later)
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// bytes 0 of w0..w3 -> one word
__device__ __forceinline__ uint32_t gather4(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
  return prmt(prmt(w0, w1, 0x0040u), prmt(w2, w3, 0x0040u), 0x5410u);
}

// sign bytes (0xFF where the float is negative, else 0) of x0..x3 -> one word.
// The selector nibbles 0xB / 0xF replicate the sign bit of byte 3 of each
// operand.  A centred value x_n - mu is never -0 (round-to-nearest gives +0
// for equal operands), so the sign bit is the test x < 0.
__device__ __forceinline__ uint32_t signs4(float x0, float x1, float x2, float x3) {
  return prmt(prmt(__float_as_uint(x0), __float_as_uint(x1), 0x00FBu),
              prmt(__float_as_uint(x2), __float_as_uint(x3), 0x00FBu), 0x5410u);
}

struct QuantConsts {
  float2 alpha2, c2;
  float edge;
};

// Stage 3 for eight magnitudes a (pairs): the rounded code of each lands in the
// low byte of ib[e] (the bits of code + 1.5 * 2^23, the fused c lg + 1.5 * 2^23
// rounding c lg to an integer).  The estimate y = c * log2(1 + alpha a) is off
// by less than 0.5 - edge; when any of the
// eight lies within that margin of a rounding edge, all eight are decided
// exactly: with I0 = round(y) and j = I0 + (y > I0), the code is
// j - 1 + (a >= thr[j]), thr[k] being the smallest float32 with code k.
// exact_a(e) returns the correctly rounded magnitude of element e; the rule
// compares it with the thresholds, while the estimate may start from a value
// within a relative 2^-22 of it (the margin covers that).
template <int LEVELS = 127, typename ExactA>
__device__ __forceinline__ void quantise8(const float2 (&a)[4], uint32_t (&ib)[8],
                                          const float* __restrict__ s_thr, const QuantConsts& qc,
                                          ExactA exact_a) {
  const float2 one2 = f2(1.0f), mone2 = f2(-1.0f), magic2 = f2(kMagic);
  float2 d[4];
  float dmax = 0.0f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 tt = __ffma2_rn(qc.alpha2, a[u], one2);
    const float2 lg = make_float2(__log2f(tt.x), __log2f(tt.y));
    const float2 r = __ffma2_rn(qc.c2, lg, magic2);             // c lg rounded to an integer, + 1.5 2^23
    const float2 nry = __ffma2_rn(r, mone2, magic2);             // -round(c lg), exact
    d[u] = __ffma2_rn(qc.c2, lg, nry);                           // c lg - round(c lg)
    ib[2 * u] = __float_as_uint(r.x);
    ib[2 * u + 1] = __float_as_uint(r.y);
    dmax = max3(dmax, fabsf(d[u].x), fabsf(d[u].y));
  }
  if (dmax > qc.edge) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float de = (e & 1) ? d[e >> 1].y : d[e >> 1].x;
      const float ae = exact_a(e);
      const int I0 = min(max((int)(ib[e] - kMagicBits), 0), LEVELS);
      const int j = I0 + (de > 0.0f ? 1 : 0);
      ib[e] = kMagicBits + (uint32_t)(j - 1 + (ae >= s_thr[j] ? 1 : 0));
    }
  }
}

__device__ __forceinline__ void load_chunk(const uint4* __restrict__ src, uint4 (&raw)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) raw[k] = __ldg(src + k);
}

// Extremes of one channel chunk: w[t] holds tokens 2t (low half) and 2t + 1
// (high half) as BF16; with PARTIAL only the first nc tokens count (min +inf,
// max -inf when there are none).
template <bool PARTIAL>
__device__ __forceinline__ void chunk_extremes(const uint32_t (&w)[16], int nc, float& cmn, float& cmx) {
  uint32_t wmin[16], wmax[16];   // the pairs with padding replaced by +inf / -inf (PARTIAL)
  if (PARTIAL) {
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const bool lo = 2 * t < nc, hi = 2 * t + 1 < nc;
      wmin[t] = (lo ? (w[t] & 0xFFFFu) : 0x7F80u) | (hi ? (w[t] & 0xFFFF0000u) : 0x7F800000u);
      wmax[t] = (lo ? (w[t] & 0xFFFFu) : 0xFF80u) | (hi ? (w[t] & 0xFFFF0000u) : 0xFF800000u);
    }
  }
  // on the packed BF16 pairs (exact)
  __nv_bfloat162 bmn = *reinterpret_cast<const __nv_bfloat162*>(PARTIAL ? &wmin[0] : &w[0]);
  __nv_bfloat162 bmx = *reinterpret_cast<const __nv_bfloat162*>(PARTIAL ? &wmax[0] : &w[0]);
#pragma unroll
  for (int t = 1; t < 16; ++t) {
    bmn = __hmin2(bmn, *reinterpret_cast<const __nv_bfloat162*>(PARTIAL ? &wmin[t] : &w[t]));
    bmx = __hmax2(bmx, *reinterpret_cast<const __nv_bfloat162*>(PARTIAL ? &wmax[t] : &w[t]));
  }
  cmn = fminf(__low2float(bmn), __high2float(bmn));
  cmx = fmaxf(__low2float(bmx), __high2float(bmx));
}

// Output forms of the codes of a chunk; kOutSplitBits + A: the split stream
// with an A-bit Anchor and an (8 - A)-bit Residual (2 <= A <= 6)
enum CodeOut { kOutSplit = 0, kOutInt8 = 1, kOutInt4 = 2, kOutSplitBits = 10 };

// OR a `bits`-wide code into a chunk's little-endian bit string held in words
// w[0..], at bit position pos (compile-time after unrolling)
template <int BITS>
__device__ __forceinline__ void put_bits(uint32_t* w, int pos, uint32_t code) {
  const int wi = pos >> 5, sh = pos & 31;
  w[wi] |= code << sh;
  if (sh + BITS > 32) w[wi + 1] |= code >> (32 - sh);
}

// Stages 1-4 of one channel chunk (32 tokens, w as in chunk_extremes), given
// the row's gamma_min mn and maximum mx and the chunk's extremes cmn, cmx:
// the chunk's codes and its gamma_scale, mu and sigma.  PARTIAL: only the
// first nc tokens are valid (statistics over them; padding gets code 0 with a
// positive sign).  OUT: kOutSplit -> out[0..3] the packed anchor words,
// out[4..7] the packed residual words (16 bytes each); kOutInt8 -> out[0..7]
// the 32 signed bytes S > 0 ? I : -I - 1 in token order; kOutInt4 -> out[0..3]
// the sign-aware nibbles of the 7-level codes (qc, s_thr then describe 7
// levels), two per byte, low nibble = even token; kOutSplitBits + A ->
// out[0..A-1] the chunk's A-bit Anchors as a little-endian bit string (token t
// at bits A t ..), out[A..7] its (8 - A)-bit Residuals likewise: Anchor
// = q8 >> R, Residual = V 2^R + 2^(R-1) - 1 - I with q8 = S > 0 ? I : -I - 1,
// V = I >> R, R = 8 - A (the 4+4 form is the paper's split).
template <bool PARTIAL, int OUT = kOutSplit>
__device__ __forceinline__ void encode_chunk(const uint32_t (&w)[16], int nc, float mn, float mx, float cmn,
                                             float cmx, float eps, const float* __restrict__ s_thr,
                                             const QuantConsts& qc, uint32_t (&out)[8], float& gscale,
                                             float& mu, float& sigma) {
  // ---- Stage 1: x_n = (x - gamma_min) / (gamma_scale + eps)
  gscale = __fsub_rn(mx, mn);
  const float dg = __fadd_rn(gscale, eps);
  const float rg = __frcp_rn(dg);
  const float2 nmn2 = f2(-mn), ndg2 = f2(-dg), rg2 = f2(rg);
  float2 xn[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    if (PARTIAL) {
      float2 v = make_float2(__uint_as_float(w[t] << 16), __uint_as_float(w[t] & 0xFFFF0000u));
      // padding enters no operation: it becomes gamma_min, so x_n = 0 exactly
      v.x = 2 * t < nc ? v.x : mn;
      v.y = 2 * t + 1 < nc ? v.y : mn;
      xn[t] = div2(__fadd2_rn(v, nmn2), ndg2, rg2);
    } else {
      xn[t] = div2(sub_min_bf16x2(w[t], -mn), ndg2, rg2);
    }
  }

  // ---- Stage 2: mu (left-to-right sum), sigma, x_f
  float s = xn[0].x;
  s = __fadd_rn(s, xn[0].y);
#pragma unroll
  for (int t = 1; t < 16; ++t) {
    s = __fadd_rn(s, xn[t].x);
    s = __fadd_rn(s, xn[t].y);
  }
  // (PARTIAL: padding adds exact zeros, so s is the left-to-right sum of the valid x_n)
  mu = __fmul_rn(s, 0.03125f);
  if (PARTIAL && nc < 32) mu = nc == 0 ? 0.0f : div1(s, (float)nc, __frcp_rn((float)nc));
  const float xn_max = div1(__fsub_rn(cmx, mn), dg, rg);
  const float xn_min = div1(__fsub_rn(cmn, mn), dg, rg);
  sigma = fmaxf(__fsub_rn(xn_max, mu), __fsub_rn(mu, xn_min));
  if (PARTIAL && nc == 0) sigma = 0.0f;
  const float ds = __fadd_rn(sigma, eps);
  const float rs = __frcp_rn(ds);
  const float2 nmu2 = f2(-mu);
  // Stage 3's magnitude enters the estimate as |x_c| (alpha / (sigma + eps)): one
  // product per chunk instead of one per element
  const QuantConsts qcs{f2(__fmul_rn(qc.alpha2.x, rs)), qc.c2, qc.edge};

  // ---- Stages 3-4, eight tokens at a time: codes in the low byte of the
  // rounded floats, sign masks, then split and pack
  if (OUT >= kOutSplitBits) {
#pragma unroll
    for (int k = 0; k < 8; ++k) out[k] = 0u;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t ib[8];
    float xs[8];   // centred values (for their signs)
    float2 a[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = 4 * q + u;
      float2 xc = __fadd2_rn(xn[t], nmu2);
      if (PARTIAL) {   // padding: x_c = +0, hence code 0 with a positive sign
        xc.x = 2 * t < nc ? xc.x : 0.0f;
        xc.y = 2 * t + 1 < nc ? xc.y : 0.0f;
      }
      xs[2 * u] = xc.x;
      xs[2 * u + 1] = xc.y;
      a[u] = make_float2(fabsf(xc.x), fabsf(xc.y));
    }
    // the exact |x_f| = RN(|x_c| / (sigma + eps)) only where the code is decided from the table
    quantise8<OUT == kOutInt4 ? 7 : 127>(a, ib, s_thr, qcs, [&](int e) { return div1(fabsf(xs[e]), ds, rs); });
    if constexpr (OUT >= kOutSplitBits) {
      constexpr int A = OUT - kOutSplitBits, R = 8 - A;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int t = 8 * q + e;
        const uint32_t I = ib[e] & 0xFFu;
        const bool neg = __float_as_uint(xs[e]) >> 31;
        const uint32_t q8 = neg ? (~I & 0xFFu) : I;
        const uint32_t anc = (uint32_t)(((int32_t)(q8 << 24) >> (24 + R)) & ((1 << A) - 1));
        const uint32_t ihat = ((I >> R) << R) + (1u << (R - 1)) - 1u;
        const uint32_t res = (ihat - I) & ((1u << R) - 1u);
        put_bits<A>(out, A * t, anc);
        put_bits<R>(out + A, R * t, res);
      }
      continue;
    }
    // codes I (0..127) and sign bytes S of the even tokens 0, 2, 4, 6 and odd tokens 1, 3, 5, 7
    const uint32_t Ie = gather4(ib[0], ib[2], ib[4], ib[6]), Io = gather4(ib[1], ib[3], ib[5], ib[7]);
    const uint32_t Se = signs4(xs[0], xs[2], xs[4], xs[6]), So = signs4(xs[1], xs[3], xs[5], xs[7]);
    if (OUT == kOutSplit) {
      // byte m of a packed word: token 2m in the low nibble, token 2m + 1 in the high nibble.
      // anchor nibble (S>0 ? I : ~I) >> 4 = ((I >> 4) ^ S) & 15; residual (7 - I) mod 16 = (I ^ 7) & 15
      out[q] = (((Ie >> 4) ^ Se) & 0x0F0F0F0Fu) | ((Io ^ So) & 0xF0F0F0F0u);
      out[4 + q] = ((Ie ^ 0x07070707u) & 0x0F0F0F0Fu) | (((Io << 4) ^ 0x70707070u) & 0xF0F0F0F0u);
    } else if (OUT == kOutInt8) {
      // S > 0 ? I : ~I per byte, even and odd tokens interleaved back into token order
      const uint32_t e8 = Ie ^ Se, o8 = Io ^ So;
      out[2 * q] = prmt(e8, o8, 0x5140u);
      out[2 * q + 1] = prmt(e8, o8, 0x7362u);
    } else {
      // 7-level code I4 in 0..7: (S>0 ? I4 : ~I4) & 15, the 4-bit two's complement of S>0 ? I4 : -I4 - 1
      out[q] = ((Ie ^ Se) & 0x0F0F0F0Fu) | (((Io ^ So) << 4) & 0xF0F0F0F0u);
    }
  }
}

// PARTIAL: valid[page] (clamped to 0..256) tokens of each page are valid; the
// statistics cover them only, padding tokens get code 0 with a positive sign,
// and a chunk without valid tokens gets mu = sigma = 0 (a partial last page of
// a sequence).  With 256 valid tokens the result is the full-page one.
template <bool PARTIAL>
__global__ void __launch_bounds__(256, 2)
encode_kernel(const uint4* __restrict__ x, int64_t n_groups, uint4* __restrict__ anchor,
              uint4* __restrict__ residual, float* __restrict__ meta, const EncodeTables tab,
              const int32_t* __restrict__ valid) {
  __shared__ float s_thr[129];
  for (int i = threadIdx.x; i < 129; i += blockDim.x) s_thr[i] = tab.thr[i];
  __syncthreads();
  // launched as a programmatic dependent: every global-memory access follows
  // the wait for the kernel ahead in the stream, and the next kernel may be
  // scheduled at once (its CTAs take the SMs as this grid's CTAs leave them)
  wait_prerequisite_grids();
  allow_dependent_launch();

  const int lane = threadIdx.x & 31;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const float eps = tab.eps;
  const QuantConsts qc{f2(tab.alpha), f2(tab.c_lg2), tab.edge};

  uint4 raw[4];
  if (g < n_groups) load_chunk(x + g * 128 + lane * 4, raw);

  for (; g < n_groups; g += n_warps) {
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w[4 * k] = raw[k].x;
      w[4 * k + 1] = raw[k].y;
      w[4 * k + 2] = raw[k].z;
      w[4 * k + 3] = raw[k].w;
    }
    const int64_t g_next = g + n_warps;
    if (g_next < n_groups) load_chunk(x + g_next * 128 + lane * 4, raw);

    // valid tokens of the page and of this lane's chunk
    int v_page = 256, nc = 32;
    if (PARTIAL) {
      v_page = min(max(__ldg(valid + (g >> 5)), 0), 256);
      nc = min(max(v_page - 32 * (lane & 7), 0), 32);
    }
    // ---- chunk and row extremes
    float cmn, cmx;
    chunk_extremes<PARTIAL>(w, nc, cmn, cmx);
    float mn = cmn, mx = cmx;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (PARTIAL && v_page == 0) {   // an empty page: gamma_min = gamma_scale = 0
      mn = 0.0f;
      mx = 0.0f;
    }

    uint32_t o[8];
    float gscale, mu, sigma;
    encode_chunk<PARTIAL>(w, nc, mn, mx, cmn, cmx, eps, s_thr, qc, o, gscale, mu, sigma);
    anchor[g * 32 + lane] = make_uint4(o[0], o[1], o[2], o[3]);
    residual[g * 32 + lane] = make_uint4(o[4], o[5], o[6], o[7]);

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

// Token-major input, the layout of paged attention: token t's 128 channels of
// head h at x[t * stride + h * 128 ..].  Page (h, j) = tokens 256 j .. 256 j +
// 255 of head h, written as page h * n_pp + j; the last page of a head may be
// partial (statistics over its valid tokens, as encode_kernel<true>).
//
// Work mapping: one CTA per page (grid-stride); warp w owns chunk w (tokens
// 32 w .. 32 w + 31 of the page); the channels are taken in four quarters,
// lane L owning channel 32 q + L of quarter q: its 32 tokens are 32 two-byte
// loads (a warp reads 64 contiguous bytes of a token row; the rest of the row's
// line serves the other quarters from cache).  The row extremes of a channel
// join its 8 chunks' extremes through shared memory (double-buffered by
// quarter, one barrier per quarter); then each lane runs Stages 1-4 on its
// channel chunk exactly as encode_kernel does.  One launch covers pages
// j_begin .. j_begin + j_count - 1 of every head: the full pages (PARTIAL =
// false) or the ragged last pages (PARTIAL = true).  (Staging each warp's 32
// token rows in shared memory with 8-byte loads first was measured slower.)
template <bool PARTIAL>
__global__ void __launch_bounds__(256, 2)
encode_tokens_kernel(const uint16_t* __restrict__ x, int64_t n_tokens, int n_heads, int n_pp, int j_begin,
                     int j_count, int64_t stride, uint4* __restrict__ anchor, uint4* __restrict__ residual,
                     float* __restrict__ meta, const EncodeTables tab) {
  __shared__ float s_thr[129];
  __shared__ float s_mn[2][8][32], s_mx[2][8][32];
  for (int i = threadIdx.x; i < 129; i += blockDim.x) s_thr[i] = tab.thr[i];
  __syncthreads();

  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const float eps = tab.eps;
  const QuantConsts qc{f2(tab.alpha), f2(tab.c_lg2), tab.edge};
  int buf = 0;

  const int64_t n_items = (int64_t)n_heads * j_count;
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int64_t h = item / j_count;
    const int64_t j = j_begin + item % j_count;
    const int64_t page = h * n_pp + j;
    const int64_t t0 = j * 256;
    const int v = PARTIAL ? (int)min(n_tokens - t0, (int64_t)256) : 256;
    const int nc = PARTIAL ? min(max(v - 32 * w, 0), 32) : 32;
#pragma unroll 1
    for (int q = 0; q < 4; ++q, buf ^= 1) {
      const int c = 32 * q + lane;
      // the chunk's 32 values of channel c as BF16 pairs (token 2t low, 2t + 1 high)
      const uint16_t* src = x + (t0 + 32 * w) * stride + h * kH + c;
      uint32_t w16[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) w16[i] = (!PARTIAL || i < nc) ? (uint32_t)__ldg(src + i * stride) : 0u;
      uint32_t wv[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) wv[t] = w16[2 * t] | (w16[2 * t + 1] << 16);

      float cmn, cmx;
      chunk_extremes<PARTIAL>(wv, nc, cmn, cmx);
      s_mn[buf][w][lane] = cmn;
      s_mx[buf][w][lane] = cmx;
      __syncthreads();
      float mn = s_mn[buf][0][lane], mx = s_mx[buf][0][lane];
#pragma unroll
      for (int k = 1; k < 8; ++k) {
        mn = fminf(mn, s_mn[buf][k][lane]);
        mx = fmaxf(mx, s_mx[buf][k][lane]);
      }

      uint32_t o[8];
      float gscale, mu, sigma;
      encode_chunk<PARTIAL>(wv, nc, mn, mx, cmn, cmx, eps, s_thr, qc, o, gscale, mu, sigma);
      anchor[(page * kH + c) * 8 + w] = make_uint4(o[0], o[1], o[2], o[3]);
      residual[(page * kH + c) * 8 + w] = make_uint4(o[4], o[5], o[6], o[7]);
      float* mp = meta + page * kMetaFloats;
      if (w == 0) {
        mp[c] = mn;
        mp[kH + c] = gscale;
      }
      mp[kMetaMuOff + w * kH + c] = mu;
      mp[kMetaSigmaOff + w * kH + c] = sigma;
    }
  }
}

// Token-major input staged through shared memory by TMA.  An item is one half
// page: 64 channels (64 h-local channels 64 k .. 64 k + 63 of head h) x the
// page's 256 tokens, one 32 KB box [256 tokens][64 channels] with 128-byte
// rows, loaded by one TMA copy into a three-slot ring; thread 0 keeps the
// ring full.  Warp w owns chunk w (tokens 32 w .. 32 w + 31); lane L owns the
// channel pair 2L, 2L + 1 of the half: one 4-byte shared load per token gives
// both channels' values, and a byte permute turns two such words (tokens 2i,
// 2i + 1) into the two channels' token pairs, the register form encode_chunk
// takes.  At a fixed token the 32 lanes read 128 contiguous bytes (no bank
// conflict).  The row extremes join the 8 chunks' extremes through shared
// memory (double-buffered by item parity, one barrier per item; the slot is
// handed back to TMA at that barrier, once every lane holds its values).
// Tokens past n_tokens arrive as zeros and count as padding (PARTIAL).
constexpr int kTokSlots = 3;
constexpr int kTokBox = 256 * 64 * 2;
constexpr int kTokSmem = kTokSlots * kTokBox + 64;

template <bool PARTIAL>
__global__ void __launch_bounds__(256, 2)
encode_tokens_tma_kernel(const __grid_constant__ CUtensorMap tm, int64_t n_tokens, int n_heads, int n_pp,
                         int j_begin, int j_count, uint4* __restrict__ anchor, uint4* __restrict__ residual,
                         float* __restrict__ meta, const EncodeTables tab, int* __restrict__ status,
                         unsigned long long wait_ns, bool skip_first) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_thr[129];
  __shared__ float2 s_mn[2][8][32], s_mx[2][8][32];   // [parity][chunk][lane]: channels 2L, 2L + 1
  const uint32_t ring = smem_u32(smem);
  const uint32_t bars = ring + kTokSlots * kTokBox;
  const int tid = threadIdx.x;
  const int w = tid >> 5;
  const int lane = tid & 31;
  const int64_t n_items = (int64_t)n_heads * j_count * 2;

  // item -> (head, page, half): consecutive items are the two halves of a page
  auto coords = [&](int64_t item, int64_t& h, int64_t& j, int& half) {
    half = (int)(item & 1);
    const int64_t hp = item >> 1;
    h = hp / j_count;
    j = j_begin + hp % j_count;
  };
  auto issue = [&](int64_t item, int slot) {
    int64_t h, j;
    int half;
    coords(item, h, j, half);
    const uint32_t bar = bars + 8 * slot;
    mbar_expect_tx(bar, kTokBox);
    tma_tile_g2s(ring + slot * kTokBox, &tm, (int)(h * kH + 64 * half), (int)(j * 256), bar);
  };

  if (tid == 0) {
    for (int k = 0; k < kTokSlots; ++k) mbar_init(bars + 8 * k, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = tid; i < 129; i += blockDim.x) s_thr[i] = tab.thr[i];
  __syncthreads();
  if (tid == 0)
    for (int k = 0; k < kTokSlots; ++k)   // (test hook: skip_first leaves the first item uncopied)
      if (blockIdx.x + (int64_t)k * gridDim.x < n_items && !(skip_first && k == 0))
        issue(blockIdx.x + (int64_t)k * gridDim.x, k);

  const float eps = tab.eps;
  const QuantConsts qc{f2(tab.alpha), f2(tab.c_lg2), tab.edge};
  int k = 0;
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x, ++k) {
    const int slot = k % kTokSlots, par = k & 1;
    const bool ok = mbar_wait(bars + 8 * slot, (uint32_t)((k / kTokSlots) & 1), wait_ns);
    if (__syncthreads_or(!ok)) {
      // a copy never landed: record it, wait (bounded) for the copies in flight, leave
      if (tid == 0) {
        atomicExch(status, 1);
        for (int u = 1; u < kTokSlots; ++u)
          if (item + (int64_t)u * gridDim.x < n_items)
            mbar_wait(bars + 8 * ((k + u) % kTokSlots), (uint32_t)(((k + u) / kTokSlots) & 1), wait_ns);
      }
      return;
    }
    int64_t h, j;
    int half;
    coords(item, h, j, half);
    const int64_t page = h * n_pp + j;
    const int64_t t0 = j * 256;
    const int v = PARTIAL ? (int)min(n_tokens - t0, (int64_t)256) : 256;
    const int nc = PARTIAL ? min(max(v - 32 * w, 0), 32) : 32;

    // the chunk's 32 tokens of channels 2L and 2L + 1 as BF16 token pairs
    const uint8_t* tile = smem + slot * kTokBox + (32 * w) * 128 + 4 * lane;
    uint32_t wa[16], wb[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t e = *reinterpret_cast<const uint32_t*>(tile + (2 * i) * 128);
      const uint32_t o = *reinterpret_cast<const uint32_t*>(tile + (2 * i + 1) * 128);
      wa[i] = prmt(e, o, 0x5410u);
      wb[i] = prmt(e, o, 0x7632u);
    }
    float2 cmn, cmx;
    chunk_extremes<PARTIAL>(wa, nc, cmn.x, cmx.x);
    chunk_extremes<PARTIAL>(wb, nc, cmn.y, cmx.y);
    s_mn[par][w][lane] = cmn;
    s_mx[par][w][lane] = cmx;
    __syncthreads();
    // every lane holds its values: the slot takes the item kTokSlots ahead
    if (tid == 0 && item + (int64_t)kTokSlots * gridDim.x < n_items)
      issue(item + (int64_t)kTokSlots * gridDim.x, slot);
    float2 mn = s_mn[par][0][lane], mx = s_mx[par][0][lane];
#pragma unroll
    for (int c = 1; c < 8; ++c) {
      const float2 a = s_mn[par][c][lane], b = s_mx[par][c][lane];
      mn = make_float2(fminf(mn.x, a.x), fminf(mn.y, a.y));
      mx = make_float2(fmaxf(mx.x, b.x), fmaxf(mx.y, b.y));
    }
    float* mp = meta + page * kMetaFloats;
    auto encode_one = [&](const uint32_t (&wv)[16], float rmn, float rmx, float chmn, float chmx, int c) {
      uint32_t o[8];
      float gscale, mu, sigma;
      encode_chunk<PARTIAL>(wv, nc, rmn, rmx, chmn, chmx, eps, s_thr, qc, o, gscale, mu, sigma);
      anchor[(page * kH + c) * 8 + w] = make_uint4(o[0], o[1], o[2], o[3]);
      residual[(page * kH + c) * 8 + w] = make_uint4(o[4], o[5], o[6], o[7]);
      if (w == 0) {
        mp[c] = rmn;
        mp[kH + c] = gscale;
      }
      mp[kMetaMuOff + w * kH + c] = mu;
      mp[kMetaSigmaOff + w * kH + c] = sigma;
    };
    const int c0 = 64 * half + 2 * lane;
    encode_one(wa, mn.x, mx.x, cmn.x, cmx.x, c0);
    encode_one(wb, mn.y, mx.y, cmn.y, cmx.y, c0 + 1);
  }
}

// Single-precision Lynx variants (the paper's §6.1 "Lynx-INT8" / "Lynx-INT4":
// Algorithm 1 at one precision, no split stream), full pages, with the work
// mapping of encode_kernel.  OUT = kOutInt8: one signed byte per token
// (S > 0 ? I : -I - 1), 256 bytes per channel row; kOutInt4: Stage 3 with 7
// levels (tab describes them), the sign-aware nibble per token, 128 bytes per
// row.  The metadata is Lynx's.
template <int OUT>
__global__ void __launch_bounds__(256, 2)
encode_variant_kernel(const uint4* __restrict__ x, int64_t n_groups, uint4* __restrict__ codes,
                      float* __restrict__ meta, const EncodeTables tab) {
  __shared__ float s_thr[129];
  for (int i = threadIdx.x; i < 129; i += blockDim.x) s_thr[i] = tab.thr[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const float eps = tab.eps;
  const QuantConsts qc{f2(tab.alpha), f2(tab.c_lg2), tab.edge};
  for (int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; g < n_groups; g += n_warps) {
    uint4 raw[4];
    load_chunk(x + g * 128 + lane * 4, raw);
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w[4 * k] = raw[k].x;
      w[4 * k + 1] = raw[k].y;
      w[4 * k + 2] = raw[k].z;
      w[4 * k + 3] = raw[k].w;
    }
    float cmn, cmx;
    chunk_extremes<false>(w, 32, cmn, cmx);
    float mn = cmn, mx = cmx;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    uint32_t o[8];
    float gscale, mu, sigma;
    encode_chunk<false, OUT>(w, 32, mn, mx, cmn, cmx, eps, s_thr, qc, o, gscale, mu, sigma);
    if (OUT == kOutInt8) {   // row group g: 4 rows of 256 bytes; lane = chunk (lane & 7) of row (lane >> 3)
      codes[g * 64 + 2 * lane] = make_uint4(o[0], o[1], o[2], o[3]);
      codes[g * 64 + 2 * lane + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
      codes[g * 32 + lane] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    const int64_t page = g >> 5;
    float* mp = meta + page * kMetaFloats;
    const int ch = 4 * (int)(g & 31) + (lane >> 3);
    if ((lane & 7) == 0) {
      mp[ch] = mn;
      mp[kH + ch] = gscale;
    }
    mp[kMetaMuOff + (lane & 7) * kH + ch] = mu;
    mp[kMetaSigmaOff + (lane & 7) * kH + ch] = sigma;
  }
}

// The split stream with an A-bit Anchor (2 <= A <= 6), full pages, work mapping
// of encode_kernel: a channel row of the Anchor plane holds 8 chunks x 4A
// bytes, of the Residual plane 8 x 4(8 - A); lane = chunk (lane & 7) of row
// (lane >> 3) of the warp's row group.
template <int A>
__global__ void __launch_bounds__(256, 2)
encode_split_kernel(const uint4* __restrict__ x, int64_t n_groups, uint32_t* __restrict__ anchor,
                    uint32_t* __restrict__ residual, float* __restrict__ meta, const EncodeTables tab) {
  constexpr int R = 8 - A;
  __shared__ float s_thr[129];
  for (int i = threadIdx.x; i < 129; i += blockDim.x) s_thr[i] = tab.thr[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const float eps = tab.eps;
  const QuantConsts qc{f2(tab.alpha), f2(tab.c_lg2), tab.edge};
  for (int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; g < n_groups; g += n_warps) {
    uint4 raw[4];
    load_chunk(x + g * 128 + lane * 4, raw);
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w[4 * k] = raw[k].x;
      w[4 * k + 1] = raw[k].y;
      w[4 * k + 2] = raw[k].z;
      w[4 * k + 3] = raw[k].w;
    }
    float cmn, cmx;
    chunk_extremes<false>(w, 32, cmn, cmx);
    float mn = cmn, mx = cmx;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    uint32_t o[8];
    float gscale, mu, sigma;
    encode_chunk<false, kOutSplitBits + A>(w, 32, mn, mx, cmn, cmx, eps, s_thr, qc, o, gscale, mu, sigma);
    const int64_t row = (g >> 5) * kH + 4 * (g & 31) + (lane >> 3);   // channel row of the pool
    const int k = lane & 7;
#pragma unroll
    for (int i = 0; i < A; ++i) anchor[row * 8 * A + A * k + i] = o[i];
#pragma unroll
    for (int i = 0; i < R; ++i) residual[row * 8 * R + R * k + i] = o[A + i];
    float* mp = meta + (g >> 5) * kMetaFloats;
    const int ch = 4 * (int)(g & 31) + (lane >> 3);
    if (k == 0) {
      mp[ch] = mn;
      mp[kH + ch] = gscale;
    }
    mp[kMetaMuOff + k * kH + ch] = mu;
    mp[kMetaSigmaOff + k * kH + ch] = sigma;
  }
}

// Uniform INT-b per channel row of a page (the baseline of the paper's §2.3 and
// §6.1): S = RN((max - min) / (2^b - 1)), Q = rint(RN((x - min) / S)) clamped to
// 0 .. 2^b - 1 (Q = 0 when S = 0), each division correctly rounded (reciprocal
// and one FMA correction step).  Codes: BITS = 8 one byte per token (256 bytes
// per row), BITS = 4 two per byte, low nibble = even token; meta[page] =
// min[128], scale[128].  Work mapping of encode_kernel.
template <int BITS>
__global__ void __launch_bounds__(256)
uniform_encode_kernel(const uint4* __restrict__ x, int64_t n_groups, uint4* __restrict__ codes,
                      float* __restrict__ meta) {
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const float levels = (float)((1 << BITS) - 1);
  for (int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; g < n_groups; g += n_warps) {
    uint4 raw[4];
    load_chunk(x + g * 128 + lane * 4, raw);
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w[4 * k] = raw[k].x;
      w[4 * k + 1] = raw[k].y;
      w[4 * k + 2] = raw[k].z;
      w[4 * k + 3] = raw[k].w;
    }
    float mn, mx;
    chunk_extremes<false>(w, 32, mn, mx);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const float sc = __fdiv_rn(__fsub_rn(mx, mn), levels);
    const float rs = __frcp_rn(sc);
    const float2 nmn2 = f2(-mn), nsc2 = f2(-sc), rs2 = f2(rs);
    uint32_t q[32];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const float2 v = make_float2(__uint_as_float(w[t] << 16), __uint_as_float(w[t] & 0xFFFF0000u));
      const float2 tq = div2(__fadd2_rn(v, nmn2), nsc2, rs2);
      q[2 * t] = sc > 0.0f ? (uint32_t)min(max(__float2int_rn(tq.x), 0), (1 << BITS) - 1) : 0u;
      q[2 * t + 1] = sc > 0.0f ? (uint32_t)min(max(__float2int_rn(tq.y), 0), (1 << BITS) - 1) : 0u;
    }
    if (BITS == 8) {
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        o[k] = q[4 * k] | (q[4 * k + 1] << 8) | (q[4 * k + 2] << 16) | (q[4 * k + 3] << 24);
      codes[g * 64 + 2 * lane] = make_uint4(o[0], o[1], o[2], o[3]);
      codes[g * 64 + 2 * lane + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t wd = 0u;
#pragma unroll
        for (int b = 0; b < 8; ++b) wd |= q[8 * k + b] << (4 * b);
        o[k] = wd;
      }
      codes[g * 32 + lane] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if ((lane & 7) == 0) {
      const int64_t page = g >> 5;
      const int ch = 4 * (int)(g & 31) + (lane >> 3);
      meta[page * 256 + ch] = mn;
      meta[page * 256 + kH + ch] = sc;
    }
  }
}

// Stage 3 alone on float32 magnitudes (|a|, expected in [0, 1]): one 8-value group per thread.
__global__ void __launch_bounds__(256)
quantize_kernel(const float* __restrict__ a, int64_t n, uint8_t* __restrict__ codes,
                const EncodeTables tab) {
  __shared__ float s_thr[129];
  for (int i = threadIdx.x; i < 129; i += blockDim.x) s_thr[i] = tab.thr[i];
  __syncthreads();
  const QuantConsts qc{f2(tab.alpha), f2(tab.c_lg2), tab.edge};
  const int64_t n_groups = (n + 7) / 8;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < n_groups;
       g += (int64_t)gridDim.x * blockDim.x) {
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int64_t i = g * 8 + e;
      v[e] = i < n ? fminf(fabsf(a[i]), 1.0f) : 0.0f;
    }
    float2 av[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) av[u] = make_float2(v[2 * u], v[2 * u + 1]);
    uint32_t ib[8];
    quantise8(av, ib, s_thr, qc, [&](int e) { return v[e]; });
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int64_t i = g * 8 + e;
      if (i < n) codes[i] = (uint8_t)(ib[e] & 0xFFu);
    }
  }
}

}  // namespace

template <bool PARTIAL>
cudaError_t launch_encode_t(const void* x, int64_t n_pages, uint8_t* anchor, uint8_t* residual,
                            float* meta, const EncodeTables* tab, const int32_t* valid, cudaStream_t s) {
  const int64_t n_groups = n_pages * 32;
  const int threads = 256;
  static int per_sm = 0;   // resident CTAs per SM (a property of the kernel)
  if (per_sm == 0) {
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_kernel<PARTIAL>, threads, 0);
    if (per_sm < 1) per_sm = 1;
  }
  const int64_t max_blocks = (int64_t)device_sm_count() * per_sm;
  const int64_t need = (n_groups + 7) / 8;
  const int blocks = (int)(need < max_blocks ? need : max_blocks);
  return launch_programmatic(encode_kernel<PARTIAL>, dim3(blocks), dim3(threads), 0, s,
                             static_cast<const uint4*>(x), n_groups, reinterpret_cast<uint4*>(anchor),
                             reinterpret_cast<uint4*>(residual), meta, *tab, valid);
}

cudaError_t launch_encode(const void* x, int64_t n_pages, uint8_t* anchor, uint8_t* residual,
                          float* meta, const EncodeTables* tab, const int32_t* valid, cudaStream_t s) {
  return valid ? launch_encode_t<true>(x, n_pages, anchor, residual, meta, tab, valid, s)
               : launch_encode_t<false>(x, n_pages, anchor, residual, meta, tab, nullptr, s);
}

template <bool PARTIAL>
cudaError_t launch_tokens_t(const void* x, int64_t n_tokens, int n_heads, int n_pp, int j_begin, int j_count,
                            int64_t stride, uint8_t* anchor, uint8_t* residual, float* meta,
                            const EncodeTables* tab, cudaStream_t s) {
  const int64_t n_items = (int64_t)n_heads * j_count;
  if (n_items == 0) return cudaSuccess;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_tokens_kernel<PARTIAL>, 256, 0);
  if (per_sm < 1) per_sm = 1;
  const int64_t max_blocks = (int64_t)device_sm_count() * per_sm;
  const int blocks = (int)(n_items < max_blocks ? n_items : max_blocks);
  encode_tokens_kernel<PARTIAL><<<blocks, 256, 0, s>>>(static_cast<const uint16_t*>(x), n_tokens, n_heads, n_pp,
                                                      j_begin, j_count, stride, reinterpret_cast<uint4*>(anchor),
                                                      reinterpret_cast<uint4*>(residual), meta, *tab);
  return cudaGetLastError();
}

template <bool PARTIAL>
cudaError_t launch_tokens_tma(const CUtensorMap& tm, int64_t n_tokens, int n_heads, int n_pp, int j_begin,
                              int j_count, uint8_t* anchor, uint8_t* residual, float* meta,
                              const EncodeTables* tab, unsigned long long wait_ns, bool skip_first,
                              cudaStream_t s) {
  const int64_t n_items = (int64_t)n_heads * j_count * 2;
  if (n_items == 0) return cudaSuccess;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(encode_tokens_tma_kernel<PARTIAL>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kTokSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int64_t max_blocks = (int64_t)device_sm_count() * 2;
  const int blocks = (int)(n_items < max_blocks ? n_items : max_blocks);
  encode_tokens_tma_kernel<PARTIAL><<<blocks, 256, kTokSmem, s>>>(
      tm, n_tokens, n_heads, n_pp, j_begin, j_count, reinterpret_cast<uint4*>(anchor),
      reinterpret_cast<uint4*>(residual), meta, *tab, device_status_ptr(), wait_ns, skip_first);
  return cudaGetLastError();
}

// Token-major encode: through the TMA-staged kernel when the input admits a
// tensor map (16-byte aligned, token stride a multiple of 8 elements), else
// through the kernel that reads the channels straight from global memory.
cudaError_t launch_encode_tokens(const void* x, int64_t n_tokens, int n_heads, int64_t stride,
                                 uint8_t* anchor, uint8_t* residual, float* meta, const EncodeTables* tab,
                                 unsigned long long wait_ns, bool skip_first, cudaStream_t s) {
  const int n_pp = (int)((n_tokens + 255) / 256);
  const int n_full = (int)(n_tokens / 256);
  CUtensorMap tm;
  if (token_map(&tm, x, n_tokens, (int64_t)n_heads * kH, stride)) {
    cudaError_t e = launch_tokens_tma<false>(tm, n_tokens, n_heads, n_pp, 0, n_full, anchor, residual, meta,
                                            tab, wait_ns, skip_first, s);
    if (e != cudaSuccess || n_full == n_pp) return e;
    return launch_tokens_tma<true>(tm, n_tokens, n_heads, n_pp, n_full, 1, anchor, residual, meta, tab, wait_ns,
                                   skip_first, s);
  }
  cudaError_t e = launch_tokens_t<false>(x, n_tokens, n_heads, n_pp, 0, n_full, stride, anchor, residual, meta,
                                         tab, s);
  if (e != cudaSuccess || n_full == n_pp) return e;
  return launch_tokens_t<true>(x, n_tokens, n_heads, n_pp, n_full, 1, stride, anchor, residual, meta, tab, s);
}

cudaError_t launch_encode_variant(const void* x, int64_t n_pages, int variant, uint8_t* codes, float* meta,
                                  const EncodeTables* tab, cudaStream_t s) {
  const int64_t n_groups = n_pages * 32;
  const int64_t need = (n_groups + 7) / 8;
  const auto* xp = static_cast<const uint4*>(x);
  auto* cp = reinterpret_cast<uint4*>(codes);
  int per_sm = 0;
  switch (variant) {
    case kVariantLynxInt8:
    case kVariantLynxInt4: {
      const bool i8 = variant == kVariantLynxInt8;
      if (i8) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_variant_kernel<kOutInt8>, 256, 0);
      else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_variant_kernel<kOutInt4>, 256, 0);
      const int64_t cap = (int64_t)device_sm_count() * (per_sm < 1 ? 1 : per_sm);
      const int blocks = (int)(need < cap ? need : cap);
      if (i8) encode_variant_kernel<kOutInt8><<<blocks, 256, 0, s>>>(xp, n_groups, cp, meta, *tab);
      else encode_variant_kernel<kOutInt4><<<blocks, 256, 0, s>>>(xp, n_groups, cp, meta, *tab);
      break;
    }
    case kVariantUniformInt8:
    case kVariantUniformInt4: {
      const bool i8 = variant == kVariantUniformInt8;
      if (i8) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, uniform_encode_kernel<8>, 256, 0);
      else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, uniform_encode_kernel<4>, 256, 0);
      const int64_t cap = (int64_t)device_sm_count() * (per_sm < 1 ? 1 : per_sm);
      const int blocks = (int)(need < cap ? need : cap);
      if (i8) uniform_encode_kernel<8><<<blocks, 256, 0, s>>>(xp, n_groups, cp, meta);
      else uniform_encode_kernel<4><<<blocks, 256, 0, s>>>(xp, n_groups, cp, meta);
      break;
    }
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <int A>
cudaError_t launch_split_t(const void* x, int64_t n_pages, uint8_t* anchor, uint8_t* residual, float* meta,
                           const EncodeTables* tab, cudaStream_t s) {
  const int64_t n_groups = n_pages * 32;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_split_kernel<A>, 256, 0);
  const int64_t cap = (int64_t)device_sm_count() * (per_sm < 1 ? 1 : per_sm);
  const int64_t need = (n_groups + 7) / 8;
  const int blocks = (int)(need < cap ? need : cap);
  encode_split_kernel<A><<<blocks, 256, 0, s>>>(static_cast<const uint4*>(x), n_groups,
                                               reinterpret_cast<uint32_t*>(anchor),
                                               reinterpret_cast<uint32_t*>(residual), meta, *tab);
  return cudaGetLastError();
}

cudaError_t launch_encode_split(const void* x, int64_t n_pages, int anchor_bits, uint8_t* anchor,
                                uint8_t* residual, float* meta, const EncodeTables* tab, cudaStream_t s) {
  switch (anchor_bits) {
    case 2: return launch_split_t<2>(x, n_pages, anchor, residual, meta, tab, s);
    case 3: return launch_split_t<3>(x, n_pages, anchor, residual, meta, tab, s);
    case 4: return launch_split_t<4>(x, n_pages, anchor, residual, meta, tab, s);
    case 5: return launch_split_t<5>(x, n_pages, anchor, residual, meta, tab, s);
    case 6: return launch_split_t<6>(x, n_pages, anchor, residual, meta, tab, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_quantize(const float* a, int64_t n, uint8_t* codes, const EncodeTables* tab,
                            cudaStream_t s) {
  const int64_t groups = (n + 7) / 8;
  const int64_t blocks = (groups + 255) / 256;
  const int grid = (int)(blocks < (int64_t)device_sm_count() * 8 ? blocks : (int64_t)device_sm_count() * 8);
  quantize_kernel<<<grid > 0 ? grid : 1, 256, 0, s>>>(a, n, codes, *tab);
  return cudaGetLastError();
}



}  // namespace lynx
