// lynx_reconstruct kernels: the Anchor-phase and Residual-phase dequantisation
// of the Lynx paper (§4.2; inverse compander of Eq. (4)).  lynx_reconstruct
// and the Lynx-INT4 comparator run reconstruct_staged_kernel (whole pages
// staged by bulk copies, described before it); the Lynx-INT8 comparator's
// one-byte codes run reconstruct_kernel below.
//
// reconstruct_kernel work mapping.  A CTA of 8 warps takes 16 consecutive channel rows of a page
// (a row group) at a time; warp w owns rows w and w+8, lane L owns tokens 8L .. 8L+7,
// which are one 32-bit word of each 4-bit plane (coalesced 128-byte warp
// loads) and 16 bytes of BF16 output (coalesced 512-byte warp stores).  The
// group's chunk-major metadata (mu[8 chunks][16 rows], sigma likewise: eight
// 64-byte runs each) is loaded once by the CTA into shared memory, double
// buffered with one barrier per group; the next group's plane words and
// metadata are loaded before the current group is computed.  The inverse
// compander is a shared-memory table lookup with one copy of the table per
// lane (entry e of lane L at word e*32 + L), so lookups never share a bank.
// The two affine steps are fused multiply-adds, two tokens at a time:
//   x = fmaf(fmaf(S*l(I_hat), sigma+eps, mu), gamma_scale+eps, gamma_min).

#include "lynx_internal.cuh"
#include "tma_ptx.cuh"

#include <cuda_bf16.h>

namespace lynx {
namespace {

// kMode: 0 = Anchor plane alone (16-entry table anc16), 1 = Anchor + Residual
// planes (256-entry table full, code = anchor nibble | residual nibble << 4),
// 2 = one byte per token (Lynx-INT8; 256-entry table full indexed by the byte,
// `anchor` points at the 256-byte rows).
template <int kMode, bool kF32>
__global__ void __launch_bounds__(256)
reconstruct_kernel(const uint32_t* __restrict__ anchor, const uint32_t* __restrict__ residual,
                   const float* __restrict__ meta, int64_t n_groups, void* __restrict__ out,
                   const LutTables lut) {
  constexpr bool kFull = kMode != 0;
  constexpr int kEntries = kFull ? 256 : 16;
  __shared__ float s_lut[kEntries * 32];
  __shared__ float s_meta[2][4][128];      // [buffer][gmin, gscale, mu, sigma][chunk * 16 + row]
  for (int i = threadIdx.x; i < kEntries * 32; i += blockDim.x)
    s_lut[i] = kFull ? lut.full[i >> 5] : lut.anc16[i >> 5];

  // launched as a programmatic dependent: every global-memory access follows
  // the wait for the kernel ahead in the stream, and the next kernel may be
  // scheduled at once (its CTAs take the SMs as this grid's CTAs leave them)
  wait_prerequisite_grids();
  allow_dependent_launch();

  const int tid = threadIdx.x;
  const int w = tid >> 5;
  const int lane = tid & 31;
  const float eps = lut.eps;
  const float* lut_lane = s_lut + lane;

  // metadata of row group o (16 rows of a page): thread tid loads mu / sigma
  // entry tid (chunk tid >> 4, row tid & 15) and threads 0..31 also gamma
  auto load_meta = [&](int64_t o, float& m0, float& m1) {
    const float* mp = meta + (o >> 3) * kMetaFloats;
    const int ch0 = 16 * (int)(o & 7);
    const int i = tid & 127;
    const float* src = mp + (tid < 128 ? kMetaMuOff : kMetaSigmaOff) + (i >> 4) * kH + ch0 + (i & 15);
    m0 = __ldg(src);
    m1 = tid < 32 ? __ldg(mp + (tid >> 4) * kH + ch0 + (tid & 15)) : 0.0f;
  };
  auto store_meta = [&](int buf, float m0, float m1) {
    s_meta[buf][tid < 128 ? 2 : 3][tid & 127] = m0;
    if (tid < 32) s_meta[buf][tid >> 4][tid & 15] = m1;
  };

  const int64_t stride = gridDim.x;
  int64_t o = blockIdx.x;
  uint32_t wa_n[2] = {0u, 0u}, wr_n[2] = {0u, 0u};
  if (o < n_groups) {
    float m0, m1;
    load_meta(o, m0, m1);
    store_meta(0, m0, m1);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t row = 16 * o + w + 8 * h;
      if (kMode == 2) {   // tokens 8L .. 8L+3 and 8L+4 .. 8L+7
        wa_n[h] = __ldg(anchor + row * 64 + 2 * lane);
        wr_n[h] = __ldg(anchor + row * 64 + 2 * lane + 1);
      } else {
        wa_n[h] = __ldg(anchor + row * 32 + lane);
        if (kFull) wr_n[h] = __ldg(residual + row * 32 + lane);
      }
    }
  }
  __syncthreads();
  int buf = 0;
  for (; o < n_groups; o += stride, buf ^= 1) {
    uint32_t wa[2] = {wa_n[0], wa_n[1]}, wr[2] = {wr_n[0], wr_n[1]};
    const int64_t on = o + stride;
    float m0 = 0.0f, m1 = 0.0f;
    if (on < n_groups) {
      load_meta(on, m0, m1);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t row = 16 * on + w + 8 * h;
        if (kMode == 2) {
          wa_n[h] = __ldg(anchor + row * 64 + 2 * lane);
          wr_n[h] = __ldg(anchor + row * 64 + 2 * lane + 1);
        } else {
          wa_n[h] = __ldg(anchor + row * 32 + lane);
          if (kFull) wr_n[h] = __ldg(residual + row * 32 + lane);
        }
      }
    }
    const int blk = lane >> 2;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = w + 8 * h;
      const int64_t row = 16 * o + r;
      const float gmin = s_meta[buf][0][r];
      const float dgv = __fadd_rn(s_meta[buf][1][r], eps);
      const float muv = s_meta[buf][2][blk * 16 + r];
      const float dsv = __fadd_rn(s_meta[buf][3][blk * 16 + r], eps);
      const float2 ds2 = make_float2(dsv, dsv), mu2 = make_float2(muv, muv);
      const float2 dg2 = make_float2(dgv, dgv), gm2 = make_float2(gmin, gmin);
      float2 xv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t c0, c1;
        if (kMode == 2) {   // tokens 2k, 2k + 1: bytes of the two words in token order
          const uint32_t wd = k < 2 ? wa[h] : wr[h];
          c0 = (wd >> (16 * (k & 1))) & 0xFFu;
          c1 = (wd >> (16 * (k & 1) + 8)) & 0xFFu;
        } else {
          c0 = (wa[h] >> (8 * k)) & 0xFu;
          c1 = (wa[h] >> (8 * k + 4)) & 0xFu;
          if (kFull) {
            c0 |= ((wr[h] >> (8 * k)) & 0xFu) << 4;
            c1 |= ((wr[h] >> (8 * k + 4)) & 0xFu) << 4;
          }
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
          const __nv_bfloat162 hv = __floats2bfloat162_rn(xv[k].x, xv[k].y);
          pk[k] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        reinterpret_cast<uint4*>(out)[row * 32 + lane] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    if (on < n_groups) store_meta(buf ^ 1, m0, m1);
    __syncthreads();
  }
}

// The same reconstruction with whole pages staged by bulk copies: one producer
// lane streams each page's Anchor plane (and Residual plane) and its metadata
// record into a shared-memory ring of 6 slots (Anchor only) or 5 (full codes)
// with full / empty mbarriers, every wait bounded; 16 consumer warps turn each
// staged page into BF16 (or float32) rows.  The full-code table keeps 16 copies
// (lane L reads copy L & 15) so that the fifth slot fits.  Consumer warp w takes the rows r = w + 16k (k = 0..7) of the page, and
// its lane group c = L >> 2 (lanes 4c .. 4c+3, tokens 32c .. 32c+31 = chunk c)
// works on row (r + c) mod 128: over the 128 values of r every (row, chunk)
// pair is taken once, and the eight lane groups of a warp read eight different
// rows' metadata, so the per-chunk mu / sigma reads hit eight different banks
// (and the plane words, word (row, L), one bank per lane).
constexpr int kRConsumers = 16;
constexpr int kRThreads = (kRConsumers + 1) * 32;
template <bool kFull> constexpr int kRStagesOf = kFull ? 5 : 6;   // ring slots

template <bool kFull>
struct RLayout {
  static constexpr int kRStages = kRStagesOf<kFull>;
  static constexpr int kUnit = (kFull ? 2 * kPlaneBytes : kPlaneBytes) + kMetaBytes;
  static constexpr int kMetaOff = kFull ? 2 * kPlaneBytes : kPlaneBytes;
  static constexpr int kRing = 0;
  static constexpr int kLut = kRing + kRStages * kUnit;              // float [entries][32 lanes]
  static constexpr int kBar = kLut + (kFull ? 256 * 16 : 16 * 32) * 4;    // full[kRStages], empty[kRStages]
  static constexpr int kFlag = kBar + 2 * kRStages * 8;
  static constexpr int kTotal = kFlag + 16;
};
static_assert(RLayout<true>::kTotal <= 232448, "shared memory (staged reconstruction)");
static_assert(RLayout<false>::kUnit % 16 == 0 && RLayout<true>::kUnit % 16 == 0, "bulk-copy alignment");

template <bool kFull, bool kF32>
__global__ void __launch_bounds__(kRThreads, 1)
reconstruct_staged_kernel(const uint8_t* __restrict__ anchor, const uint8_t* __restrict__ residual,
                          const float* __restrict__ meta, int64_t n_pages, void* __restrict__ out,
                          const LutTables lut, int* __restrict__ status, unsigned long long wait_ns,
                          int skip_unit) {
  using S = RLayout<kFull>;
  constexpr int kRStages = S::kRStages;
  constexpr int kEntries = kFull ? 256 : 16;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t base = smem_u32(smem);
  const uint32_t bar_full = base + S::kBar;
  const uint32_t bar_empty = bar_full + 8 * kRStages;
  int* s_flag = reinterpret_cast<int*>(smem + S::kFlag);
  float* s_lut = reinterpret_cast<float*>(smem + S::kLut);
  if (tid == 0) {
    for (int st = 0; st < kRStages; ++st) {
      mbar_init(bar_full + 8 * st, 1);
      mbar_init(bar_empty + 8 * st, kRConsumers);
    }
    *s_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the value table (kernel parameters only), entry e of lane L at word e * 32 + L
  constexpr int kCopies = kFull ? 16 : 32;
  for (int i = tid; i < kEntries * kCopies; i += kRThreads) s_lut[i] = kFull ? lut.full[i >> 4] : lut.anc16[i >> 5];
  __syncthreads();
  // launched as a programmatic dependent: every global-memory access follows
  // the wait for the kernel ahead in the stream
  wait_prerequisite_grids();
  allow_dependent_launch();

  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int n_mine = first < n_pages ? (int)((n_pages - 1 - first) / stride + 1) : 0;
  if (warp == kRConsumers) {   // ---- producer lane
    if (lane != 0) return;
    int u_end = 0;
    bool ok = true;
    for (int u = 0; u < n_mine; ++u) {
      const int st = u % kRStages;
      if (u >= kRStages && !mbar_wait(bar_empty + 8 * st, ((u / kRStages) - 1) & 1, wait_ns)) {
        ok = false;
        break;
      }
      u_end = u + 1;
      if (u == skip_unit) continue;   // test hook: this page's copy is never issued
      const int64_t page = first + (int64_t)u * stride;
      const uint32_t dst = base + S::kRing + st * S::kUnit;
      const uint32_t bar = bar_full + 8 * st;
      mbar_expect_tx(bar, S::kUnit);
      bulk_g2s(dst, anchor + page * kPlaneBytes, kPlaneBytes, bar);
      if (kFull) bulk_g2s(dst + kPlaneBytes, residual + page * kPlaneBytes, kPlaneBytes, bar);
      bulk_g2s(dst + S::kMetaOff, meta + page * kMetaFloats, kMetaBytes, bar);
    }
    if (!ok) {
      atomicExch(status, 1);
      *reinterpret_cast<volatile int*>(s_flag) = 1;
    }
    // every copy this lane issued has landed before the CTA may exit
    for (int u = u_end - 1; u >= 0 && u >= u_end - kRStages; --u)
      if (u != skip_unit) mbar_wait(bar_full + 8 * (u % kRStages), (u / kRStages) & 1, wait_ns);
    return;
  }

  // ---- consumer warps
  const float eps = lut.eps;
  const float* lut_lane = s_lut + (kFull ? (lane & 15) : lane);
  const int c = lane >> 2;   // the lane group's chunk
  for (int u = 0; u < n_mine; ++u) {
    const int st = u % kRStages;
    const bool got = mbar_wait(bar_full + 8 * st, (u / kRStages) & 1, wait_ns);
    if (__any_sync(0xffffffffu, !got) || *reinterpret_cast<volatile int*>(s_flag) != 0) {
      if (lane == 0) {
        atomicExch(status, 1);
        *reinterpret_cast<volatile int*>(s_flag) = 1;
      }
      break;
    }
    const int64_t page = first + (int64_t)u * stride;
    const uint8_t* unit = smem + S::kRing + st * S::kUnit;
    const uint32_t* pa = reinterpret_cast<const uint32_t*>(unit);
    const uint32_t* pr = reinterpret_cast<const uint32_t*>(unit + kPlaneBytes);
    const float* mt = reinterpret_cast<const float*>(unit + S::kMetaOff);
#pragma unroll 2
    for (int k = 0; k < 8; ++k) {
      const int row = (warp + 16 * k + c) & 127;
      const uint32_t wa = pa[row * 32 + lane];
      const uint32_t wr = kFull ? pr[row * 32 + lane] : 0u;
      const float gmin = mt[row];
      const float dgv = __fadd_rn(mt[kH + row], eps);
      const float muv = mt[kMetaMuOff + c * kH + row];
      const float dsv = __fadd_rn(mt[kMetaSigmaOff + c * kH + row], eps);
      const float2 ds2 = make_float2(dsv, dsv), mu2 = make_float2(muv, muv);
      const float2 dg2 = make_float2(dgv, dgv), gm2 = make_float2(gmin, gmin);
      float2 xv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t c0 = (wa >> (8 * j)) & 0xFu, c1 = (wa >> (8 * j + 4)) & 0xFu;
        if (kFull) {
          c0 |= ((wr >> (8 * j)) & 0xFu) << 4;
          c1 |= ((wr >> (8 * j + 4)) & 0xFu) << 4;
        }
        const float2 l = make_float2(lut_lane[c0 * (kFull ? 16 : 32)], lut_lane[c1 * (kFull ? 16 : 32)]);
        xv[j] = __ffma2_rn(__ffma2_rn(l, ds2, mu2), dg2, gm2);
      }
      const int64_t orow = page * kH + row;
      if (kF32) {
        float4* op = reinterpret_cast<float4*>(out) + orow * 64 + lane * 2;
        op[0] = make_float4(xv[0].x, xv[0].y, xv[1].x, xv[1].y);
        op[1] = make_float4(xv[2].x, xv[2].y, xv[3].x, xv[3].y);
      } else {
        uint32_t pk[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __nv_bfloat162 hv = __floats2bfloat162_rn(xv[j].x, xv[j].y);
          pk[j] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        reinterpret_cast<uint4*>(out)[orow * 32 + lane] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * st);
  }
}

// Uniform INT-b codes (min[128], scale[128] per page): x = fmaf(Q, scale, min).
// One thread per 8 tokens of a row (grid-stride).
template <int BITS, bool kF32>
__global__ void __launch_bounds__(256)
uniform_reconstruct_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ meta, int64_t n_rows,
                           void* __restrict__ out) {
  const int64_t n_items = n_rows * 32;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_items; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i >> 5;
    const int part = (int)(i & 31);
    const float* mp = meta + (row >> 7) * 256;
    const int ch = (int)(row & 127);
    const float mn = __ldg(mp + ch), sc = __ldg(mp + kH + ch);
    uint32_t q[8];
    if (BITS == 8) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(codes + row * 256) + part);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        q[k] = (v.x >> (8 * k)) & 0xFFu;
        q[4 + k] = (v.y >> (8 * k)) & 0xFFu;
      }
    } else {
      const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(codes + row * 128) + part);
#pragma unroll
      for (int k = 0; k < 8; ++k) q[k] = (v >> (4 * k)) & 0xFu;
    }
    float x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = __fmaf_rn((float)q[k], sc, mn);
    if (kF32) {
      float4* op = reinterpret_cast<float4*>(out) + row * 64 + part * 2;
      op[0] = make_float4(x[0], x[1], x[2], x[3]);
      op[1] = make_float4(x[4], x[5], x[6], x[7]);
    } else {
      uint32_t pk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 hv = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
        pk[k] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      reinterpret_cast<uint4*>(out)[row * 32 + part] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
}

// One-byte codes -> two nibble planes: thread i takes 16 codes (tokens 16 m ..
// 16 m + 15 of row r, i = 16 r + m) and writes their low nibbles and their
// high nibbles as 8 bytes each, token 2j in the low half of byte j.
__global__ void __launch_bounds__(256)
split_nibbles_kernel(const uint4* __restrict__ codes, int64_t n_items, uint2* __restrict__ lo,
                     uint2* __restrict__ hi) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_items;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 c = __ldg(codes + i);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t l[4], h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // bytes b0..b3 -> (b0 & 15) | (b1 & 15) << 4 in byte 0, (b2 & 15) | (b3 & 15) << 4 in byte 2
      const uint32_t lw = w[k] & 0x0F0F0F0Fu, hw = (w[k] >> 4) & 0x0F0F0F0Fu;
      l[k] = lw | (lw >> 4);
      h[k] = hw | (hw >> 4);
    }
    auto pack = [](const uint32_t (&v)[4], int k0) {   // bytes 0 and 2 of v[k0], v[k0 + 1]
      return (v[k0] & 0xFFu) | ((v[k0] >> 8) & 0xFF00u) | ((v[k0 + 1] & 0xFFu) << 16) |
             ((v[k0 + 1] << 8) & 0xFF000000u);
    };
    lo[i] = make_uint2(pack(l, 0), pack(l, 2));
    hi[i] = make_uint2(pack(h, 0), pack(h, 2));
  }
}

// the `bits`-wide two's-complement code at bit position pos of a little-endian
// bit string held in words w[], sign-extended
template <int BITS>
__device__ __forceinline__ int get_bits(const uint32_t* w, int pos) {
  const int wi = pos >> 5, sh = pos & 31;
  uint32_t v = w[wi] >> sh;
  if (sh + BITS > 32) v |= w[wi + 1] << (32 - sh);
  return (int)(v << (32 - BITS)) >> (32 - BITS);
}

// The split stream with an A-bit Anchor (2 <= A <= 6): rows of 8 chunks x 4A
// bytes (Anchor) and 8 x 4(8 - A) bytes (Residual), each chunk's codes a
// little-endian bit string.  One thread per (channel row, chunk): 32 tokens.
// Anchor only: x_f from the 2^A-entry table; full: I = V 2^R + 2^(R-1) - 1 -
// Q_res and x_f = S l(I) from the 256-entry table of signed bytes.  Then
// x = fmaf(fmaf(x_f, sigma+eps, mu), gamma_scale+eps, gamma_min) as for the
// 4+4 split.  Tables replicated per lane in shared memory (no bank conflicts).
template <int A, bool FULL, bool kF32>
__global__ void __launch_bounds__(256)
reconstruct_split_kernel(const uint32_t* __restrict__ anchor, const uint32_t* __restrict__ residual,
                         const float* __restrict__ meta, int64_t n_rows, void* __restrict__ out,
                         const SplitTables st, const LutTables lut8) {
  constexpr int R = 8 - A;
  constexpr int kEntries = FULL ? 256 : (1 << A);
  __shared__ float s_lut[kEntries * 32];
  for (int i = threadIdx.x; i < kEntries * 32; i += blockDim.x)
    s_lut[i] = FULL ? lut8.full[i >> 5] : st.anc[i >> 5];
  __syncthreads();
  const float* lut_lane = s_lut + (threadIdx.x & 31);
  const float eps = st.eps;
  const int64_t n_items = n_rows * 8;
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < n_items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = it >> 3;
    const int k = (int)(it & 7);
    uint32_t aw[A], rw[R > 0 ? R : 1];
#pragma unroll
    for (int i = 0; i < A; ++i) aw[i] = __ldg(anchor + row * 8 * A + A * k + i);
    if (FULL) {
#pragma unroll
      for (int i = 0; i < R; ++i) rw[i] = __ldg(residual + row * 8 * R + R * k + i);
    }
    const float* mp = meta + (row >> 7) * kMetaFloats;
    const int ch = (int)(row & 127);
    const float gmin = __ldg(mp + ch);
    const float dg = __fadd_rn(__ldg(mp + kH + ch), eps);
    const float mu = __ldg(mp + kMetaMuOff + k * kH + ch);
    const float ds = __fadd_rn(__ldg(mp + kMetaSigmaOff + k * kH + ch), eps);
    float x[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const int qa = get_bits<A>(aw, A * t);
      float l;
      if (FULL) {
        const int V = qa < 0 ? -qa - 1 : qa;
        const int I = (V << R) + (1 << (R - 1)) - 1 - get_bits<R>(rw, R * t);
        const int q8 = qa < 0 ? -I - 1 : I;
        l = lut_lane[(q8 & 0xFF) * 32];
      } else {
        l = lut_lane[(qa & ((1 << A) - 1)) * 32];
      }
      x[t] = __fmaf_rn(__fmaf_rn(l, ds, mu), dg, gmin);
    }
    if (kF32) {
      float4* op = reinterpret_cast<float4*>(out) + row * 64 + k * 8;
#pragma unroll
      for (int j = 0; j < 8; ++j) op[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
    } else {
      uint4* op = reinterpret_cast<uint4*>(out) + row * 32 + k * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t pk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const __nv_bfloat162 hv = __floats2bfloat162_rn(x[8 * j + 2 * u], x[8 * j + 2 * u + 1]);
          pk[u] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        op[j] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
  }
}

template <int A, bool FULL, bool kF32>
cudaError_t launch_split(const uint8_t* anchor, const uint8_t* residual, const float* meta, int64_t n_pages,
                         void* out, const SplitTables* st, const LutTables* lut8, cudaStream_t s) {
  const int64_t n_rows = n_pages * kH;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reconstruct_split_kernel<A, FULL, kF32>, 256, 0);
  const int64_t cap = (int64_t)device_sm_count() * (per_sm < 1 ? 1 : per_sm);
  const int64_t need = (n_rows * 8 + 255) / 256;
  const int blocks = (int)(need < cap ? need : cap);
  reconstruct_split_kernel<A, FULL, kF32><<<blocks, 256, 0, s>>>(
      reinterpret_cast<const uint32_t*>(anchor), reinterpret_cast<const uint32_t*>(residual), meta, n_rows, out,
      *st, *lut8);
  return cudaGetLastError();
}

template <int A>
cudaError_t launch_split_a(const uint8_t* anchor, const uint8_t* residual, const float* meta, int64_t n_pages,
                           void* out, bool f32, const SplitTables* st, const LutTables* lut8, cudaStream_t s) {
  if (residual)
    return f32 ? launch_split<A, true, true>(anchor, residual, meta, n_pages, out, st, lut8, s)
               : launch_split<A, true, false>(anchor, residual, meta, n_pages, out, st, lut8, s);
  return f32 ? launch_split<A, false, true>(anchor, residual, meta, n_pages, out, st, lut8, s)
             : launch_split<A, false, false>(anchor, residual, meta, n_pages, out, st, lut8, s);
}

template <int kMode, bool kF32>
cudaError_t launch(const uint8_t* anchor, const uint8_t* residual, const float* meta,
                   int64_t n_pages, void* out, const LutTables* lut, cudaStream_t s) {
  const int64_t n_groups = n_pages * (kH / 16);
  const int threads = 256;
  static int per_sm = 0;   // resident CTAs per SM (a property of the kernel)
  if (per_sm == 0) {
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reconstruct_kernel<kMode, kF32>, threads, 0);
    if (per_sm < 1) per_sm = 1;
  }
  const int64_t max_blocks = (int64_t)device_sm_count() * per_sm;
  const int blocks = (int)(n_groups < max_blocks ? n_groups : max_blocks);
  return launch_programmatic(reconstruct_kernel<kMode, kF32>, dim3(blocks), dim3(threads), 0, s,
                             reinterpret_cast<const uint32_t*>(anchor), reinterpret_cast<const uint32_t*>(residual),
                             meta, n_groups, out, *lut);
}

// one CTA per SM (each holds kRStages pages), pages taken round robin
template <bool kFull, bool kF32>
cudaError_t launch_staged(const uint8_t* anchor, const uint8_t* residual, const float* meta, int64_t n_pages,
                          void* out, const LutTables* lut, int* status, cudaStream_t s,
                          unsigned long long wait_ns = kDefaultWaitNs, int skip_unit = -1) {
  constexpr int kSmem = RLayout<kFull>::kTotal;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(reconstruct_staged_kernel<kFull, kF32>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int64_t sms = device_sm_count();
  const int blocks = (int)(n_pages < sms ? n_pages : sms);
  return launch_programmatic(reconstruct_staged_kernel<kFull, kF32>, dim3(blocks), dim3(kRThreads), kSmem, s,
                             anchor, residual, meta, n_pages, out, *lut, status, wait_ns, skip_unit);
}

}  // namespace

cudaError_t launch_split_nibbles(const uint8_t* codes, int64_t n_rows, uint8_t* lo, uint8_t* hi, cudaStream_t s) {
  const int64_t n_items = n_rows * 16;
  const int64_t need = (n_items + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  split_nibbles_kernel<<<(int)(need < cap ? need : cap), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(codes), n_items, reinterpret_cast<uint2*>(lo), reinterpret_cast<uint2*>(hi));
  return cudaGetLastError();
}

cudaError_t launch_reconstruct(const uint8_t* anchor, const uint8_t* residual, const float* meta,
                               int64_t n_pages, void* out, int out_dtype, const LutTables* lut, int* status,
                               unsigned long long wait_ns, int skip_unit, cudaStream_t s) {
  const bool full = residual != nullptr;
  const bool f32 = out_dtype == LYNX_OUT_F32;
  if (full) {
    return f32 ? launch_staged<true, true>(anchor, residual, meta, n_pages, out, lut, status, s, wait_ns, skip_unit)
               : launch_staged<true, false>(anchor, residual, meta, n_pages, out, lut, status, s, wait_ns, skip_unit);
  }
  return f32 ? launch_staged<false, true>(anchor, residual, meta, n_pages, out, lut, status, s, wait_ns, skip_unit)
             : launch_staged<false, false>(anchor, residual, meta, n_pages, out, lut, status, s, wait_ns, skip_unit);
}

cudaError_t launch_reconstruct_split(const uint8_t* anchor, const uint8_t* residual, const float* meta,
                                     int64_t n_pages, int anchor_bits, void* out, int out_dtype,
                                     const SplitTables* st, const LutTables* lut8, cudaStream_t s) {
  const bool f32 = out_dtype == LYNX_OUT_F32;
  switch (anchor_bits) {
    case 2: return launch_split_a<2>(anchor, residual, meta, n_pages, out, f32, st, lut8, s);
    case 3: return launch_split_a<3>(anchor, residual, meta, n_pages, out, f32, st, lut8, s);
    case 4: return launch_split_a<4>(anchor, residual, meta, n_pages, out, f32, st, lut8, s);
    case 5: return launch_split_a<5>(anchor, residual, meta, n_pages, out, f32, st, lut8, s);
    case 6: return launch_split_a<6>(anchor, residual, meta, n_pages, out, f32, st, lut8, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_reconstruct_variant(const uint8_t* codes, const float* meta, int64_t n_pages, int variant,
                                       void* out, int out_dtype, const LutTables* lut, int* status, cudaStream_t s) {
  const bool f32 = out_dtype == LYNX_OUT_F32;
  switch (variant) {
    case kVariantLynxInt8:
      return f32 ? launch<2, true>(codes, nullptr, meta, n_pages, out, lut, s)
                 : launch<2, false>(codes, nullptr, meta, n_pages, out, lut, s);
    case kVariantLynxInt4:   // the Anchor-plane layout with the 7-level table
      return f32 ? launch_staged<false, true>(codes, nullptr, meta, n_pages, out, lut, status, s)
                 : launch_staged<false, false>(codes, nullptr, meta, n_pages, out, lut, status, s);
    case kVariantUniformInt8:
    case kVariantUniformInt4: {
      const int64_t n_rows = n_pages * kH;
      const int64_t blocks_need = (n_rows * 32 + 255) / 256;
      const int64_t cap = (int64_t)device_sm_count() * 8;
      const int blocks = (int)(blocks_need < cap ? blocks_need : cap);
      if (variant == kVariantUniformInt8) {
        if (f32) uniform_reconstruct_kernel<8, true><<<blocks, 256, 0, s>>>(codes, meta, n_rows, out);
        else uniform_reconstruct_kernel<8, false><<<blocks, 256, 0, s>>>(codes, meta, n_rows, out);
      } else {
        if (f32) uniform_reconstruct_kernel<4, true><<<blocks, 256, 0, s>>>(codes, meta, n_rows, out);
        else uniform_reconstruct_kernel<4, false><<<blocks, 256, 0, s>>>(codes, meta, n_rows, out);
      }
      return cudaGetLastError();
    }
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace lynx
