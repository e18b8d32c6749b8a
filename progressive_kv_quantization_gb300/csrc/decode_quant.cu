// Decode / verification attention over Lynx-encoded pages (anchor-only draft
// KV, or anchor + residual full codes), the attention of the Lynx paper's
// §2.1 run on the KV that the Anchor and Residual phases (§4.2-4.3) deliver.
//
// CTA = one (sequence, KV head, group of 4 query rows, split of the pages):
//   warp 8      producer: streams the split's pages through a ring of shared
//               memory slots.  A slot holds one page's K or V unit: the 4-bit
//               plane(s) as a 2-D TMA tile (128 rows x 128 B, 128-byte
//               swizzle) and the metadata as a 1-D bulk copy.  Slots are
//               handed over with "full" (TMA -> consumers) and "empty"
//               (8 consumer warps -> producer) mbarriers; every wait is
//               bounded in time.
//   warps 0..7  consumers: warp w owns the 32-token chunk w of every page and
//               runs its own online softmax over those tokens; the 8 warps'
//               (max, sum, output) states merge once at the end.  No block-wide
//               barrier is taken per page.
//
// Dequantisation stays in registers through the per-chunk affine fold
// (A = gamma_min + (gamma_scale+eps) mu, B = (gamma_scale+eps)(sigma+eps)):
//   q.k_t           = sum_d q_d A_d + sum_d (q_d B_d) l~_{d,t}
//   sum_t p_t v_d,t = A_d sum_t p_t + B_d sum_t p_t l~_{d,t}
// with l~ = S l(I_hat) read from a table in shared memory (anchor: one lookup
// per byte gives both tokens' values) and packed float2 FMAs.
//
// K phase, lane (tg = L & 3, cg = L >> 2): tokens 8tg..8tg+7 of the chunk,
// channels cg + 8j (j = 0..15).  With the swizzle (16-byte unit u of row r at
// u ^ (r & 7)) the lane's plane words sit at one per-lane offset plus j * 1024,
// and the 32 lanes hit 32 different banks.  The 8 channel groups' partial
// logits are summed through shared memory.  V phase, lane L: channels
// L + 32k (k = 0..3), all 32 tokens of the chunk (one 16-byte unit per row).

#include "lynx_internal.cuh"

#include <cuda.h>
#include <math_constants.h>

namespace lynx {
namespace {

constexpr int kConsumers = 8;
constexpr int kThreadsQ = (kConsumers + 1) * 32;
constexpr int kRows = 4;
constexpr int kWsPerCta = kRows * kH + 2 * kRows;
constexpr unsigned long long kWaitNs = 2000000000ull;

template <bool FULL>
struct QGeo {
  static constexpr int kStages = 3;
  static constexpr int kUnit = FULL ? 2 * kPlaneBytes + kMetaBytes : kPlaneBytes + kMetaBytes;
  static constexpr int kResOff = kPlaneBytes;
  static constexpr int kMetaOff = FULL ? 2 * kPlaneBytes : kPlaneBytes;
  // anchor: byte -> (value of low nibble, value of high nibble), 32 copies (entry stride 256 B)
  // full:   8-bit code -> value, 32 copies (entry stride 128 B)
  static constexpr int kLutBytes = FULL ? 256 * 32 * 4 : 256 * 32 * 8;
};
static_assert(QGeo<false>::kUnit % 1024 == 0 && QGeo<true>::kUnit % 1024 == 0,
              "ring slots must keep the 1024-byte alignment of swizzled tiles");

// per consumer warp: coefficients [128][4 rows] f32, partial logits [8 groups][32] f32x4,
// probabilities [16 pairs] f32x4 for rows 0-1 and 2-3
constexpr int kWarpCoef = 0;
constexpr int kWarpPart = kWarpCoef + kH * 4 * 4;
constexpr int kWarpPs01 = kWarpPart + 8 * 32 * 16;
constexpr int kWarpPs23 = kWarpPs01 + 16 * 16;
constexpr int kWarpBytes = kWarpPs23 + 16 * 16;

template <bool FULL>
struct QLayout {
  using G = QGeo<FULL>;
  static constexpr int kRing = 0;
  static constexpr int kLut = kRing + G::kStages * G::kUnit;
  static constexpr int kWarps = kLut + G::kLutBytes;
  static constexpr int kQs = kWarps + kConsumers * kWarpBytes;     // [128][4] f32
  static constexpr int kFlag = kQs + kH * kRows * 4;
  static constexpr int kBar = kFlag + 16;                          // full[S], empty[S]
  static constexpr int kTotal = kBar + 2 * G::kStages * 8;
  static constexpr int kAlloc = kTotal + 1024;                     // room to align the base
  // end-of-kernel merge area (reuses the ring): m[8][4], l[8][4], o[8][4][128]
  static constexpr int kMergeM = 0;
  static constexpr int kMergeL = kMergeM + kConsumers * kRows * 4;
  static constexpr int kMergeO = kMergeL + kConsumers * kRows * 4;
  static_assert(kMergeO + kConsumers * kRows * kH * 4 <= G::kStages * G::kUnit, "merge area");
};
static_assert(QLayout<false>::kAlloc <= 232448, "shared memory (anchor)");
static_assert(QLayout<true>::kAlloc <= 232448, "shared memory (full)");

// ---------------------------------------------------------------- PTX helpers

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
// gives up after kWaitNs (clock checked every 256 polls) or 2^26 polls
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 26); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && global_ns() - t0 > kWaitNs) return false;
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
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
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

// value pair (l~ of token 2m, l~ of token 2m+1) for one anchor byte, or for
// one anchor byte and the matching residual byte
template <bool FULL>
__device__ __forceinline__ float2 lut_pair(const uint8_t* lut_lane, uint32_t a_word, uint32_t r_word,
                                           int k) {
  if (!FULL) {
    // entry stride 256 B: offset = byte k of a_word placed in bits 8..15
    const uint32_t off = prmt(a_word, 0u, 0x4404u | ((uint32_t)k << 4));
    return lds<float2>(lut_lane, off);
  } else {
    const uint32_t ab = (a_word >> (8 * k)) & 0xFFu;
    const uint32_t rb = (r_word >> (8 * k)) & 0xFFu;
    const uint32_t c0 = (ab & 0xFu) | ((rb & 0xFu) << 4);
    const uint32_t c1 = (ab >> 4) | (rb & 0xF0u);
    return make_float2(lds<float>(lut_lane, c0 << 7), lds<float>(lut_lane, c1 << 7));
  }
}

template <bool FULL>
__global__ void __launch_bounds__(kThreadsQ, 1)
decode_quant_kernel(const DecodeArgs a, const LutTables lut,
                    const __grid_constant__ CUtensorMap tm_ka, const __grid_constant__ CUtensorMap tm_va,
                    const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_vr) {
  using G = QGeo<FULL>;
  using S = QLayout<FULL>;
  constexpr int kSt = G::kStages;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (swizzled TMA tiles need it)
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_u32);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int L = tid & 31;
  const int split = blockIdx.x;
  const int h = blockIdx.y / a.n_rg;
  const int rg = blockIdx.y % a.n_rg;
  const int b = blockIdx.z;
  const int64_t cta = ((int64_t)b * gridDim.y + blockIdx.y) * a.n_splits + split;
  const int TG = a.T * a.G;
  const int max_keys = a.max_pages * kP;

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

  const uint32_t s_ring = base + S::kRing;       // shared-window addresses (for TMA)
  const uint32_t bar_full = base + S::kBar;
  const uint32_t bar_empty = bar_full + 8 * kSt;
  int* s_flag = reinterpret_cast<int*>(smem + S::kFlag);

  // ---- prologue: scaled queries, replicated value table, barriers
  for (int i = tid; i < kH * kRows; i += kThreadsQ) {
    const int d = i >> 2, r = i & 3, row = rg * kRows + r;
    float v = 0.0f;
    if (row < TG) {
      const int t = row / a.G, hq = h * a.G + row % a.G;
      const uint16_t bits = a.q[(((int64_t)b * a.T + t) * a.Hq + hq) * kH + d];
      v = __uint_as_float((uint32_t)bits << 16) * a.scale_log2;
    }
    reinterpret_cast<float*>(smem + S::kQs)[i] = v;
  }
  if (!FULL) {
    float2* l2 = reinterpret_cast<float2*>(smem + S::kLut);
    for (int i = tid; i < 256 * 32; i += kThreadsQ) l2[i] = lut.anc_pair[i >> 5];
  } else {
    float* l1 = reinterpret_cast<float*>(smem + S::kLut);
    for (int i = tid; i < 256 * 32; i += kThreadsQ) l1[i] = lut.full[i >> 5];
  }
  if (tid == 0) {
    for (int s = 0; s < kSt; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kConsumers);
    }
    *s_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  float m_run[kRows], l_run[kRows];
  float O[4][kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    m_run[r] = -CUDART_INF_F;
    l_run[r] = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) O[k][r] = 0.0f;
  }

  if (warp == kConsumers) {
    // ================= producer
    if (L == 0) {
      int issued = 0;
      bool ok = true;
      for (int u = 0; u < n_units; ++u) {
        const int s = u % kSt;
        if (u >= kSt && !mbar_wait(bar_empty + 8 * s, ((u / kSt) - 1) & 1)) {
          ok = false;
          break;
        }
        const int p = p_begin + (u >> 1);
        const bool is_v = (u & 1) != 0;
        int64_t id = pt_row[p];
        if (id < 0 || id >= a.n_pool) {
          atomicExch(a.status, 2);
          id = 0;
        }
        const uint32_t dst = s_ring + s * G::kUnit;
        const uint32_t bar = bar_full + 8 * s;
        mbar_expect_tx(bar, G::kUnit);
        tma_tile_g2s(dst, is_v ? &tm_va : &tm_ka, 0, (int)(id * kH), bar);
        if (FULL) tma_tile_g2s(dst + G::kResOff, is_v ? &tm_vr : &tm_kr, 0, (int)(id * kH), bar);
        bulk_g2s(dst + G::kMetaOff, (is_v ? a.v_meta : a.k_meta) + id * kMetaFloats, kMetaBytes, bar);
        ++issued;
      }
      if (!ok) {
        atomicExch(a.status, 1);
        *s_flag = 1;
        // drain: the newest issue of every slot must land before the CTA leaves
        for (int u = issued - 1; u >= 0 && u >= issued - kSt; --u)
          mbar_wait(bar_full + 8 * (u % kSt), (u / kSt) & 1);
      }
    }
  } else {
    // ================= consumers: warp `warp` owns chunk `warp` of every page
    const int w = warp;
    // offsets from smem
    const uint32_t s_w = S::kWarps + w * kWarpBytes;
    const uint32_t s_coef = s_w + kWarpCoef;
    const uint32_t s_part = s_w + kWarpPart;
    const uint32_t s_ps01 = s_w + kWarpPs01;
    const uint32_t s_ps23 = s_w + kWarpPs23;
    const uint32_t s_qs = S::kQs;
    const int tg = L & 3, cg = L >> 2;
    // K phase: plane word of (row cg + 8j, unit w ^ cg, word tg) = k_off + j * 1024
    const uint32_t k_off = cg * 128 + ((w ^ cg) << 4) + 4 * tg;
    const uint8_t* lut_lane = smem + S::kLut + (FULL ? 4 * L : 8 * L);
    const float eps = a.eps;
    bool failed = false;

    for (int i = 0; i < np && !failed; ++i) {
      const int p = p_begin + i;
      const int uK = 2 * i, uV = 2 * i + 1;
      const int sK = uK % kSt, sV = uV % kSt;
      const uint32_t unitK = S::kRing + sK * G::kUnit;   // offsets from smem
      const uint32_t unitV = S::kRing + sV * G::kUnit;

      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sK, (uK / kSt) & 1));
      if (failed) break;

      // ---- per-chunk key coefficients: coef[d] = (q_r B_d, q_r B_d) pairs, constK_r = sum q_r A_d
      float ck[kRows] = {0.f, 0.f, 0.f, 0.f};
      {
        const uint32_t km = unitK + G::kMetaOff;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int d = L + 32 * k;
          const float gmin = lds<float>(smem, km + 4 * d);
          const float dg = __fadd_rn(lds<float>(smem, km + 4 * (kH + d)), eps);
          const float mu = lds<float>(smem, km + 4 * (kMetaMuOff + w * kH + d));
          const float ds = __fadd_rn(lds<float>(smem, km + 4 * (kMetaSigmaOff + w * kH + d)), eps);
          const float A = __fmaf_rn(dg, mu, gmin);
          const float Bc = __fmul_rn(dg, ds);
          const float4 q = lds<float4>(smem, s_qs + 16 * d);
          *reinterpret_cast<float4*>(smem + s_coef + 16 * d) =
              make_float4(q.x * Bc, q.y * Bc, q.z * Bc, q.w * Bc);
          ck[0] = __fmaf_rn(q.x, A, ck[0]);
          ck[1] = __fmaf_rn(q.y, A, ck[1]);
          ck[2] = __fmaf_rn(q.z, A, ck[2]);
          ck[3] = __fmaf_rn(q.w, A, ck[3]);
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) ck[r] = warp_sum(ck[r]);
      }
      __syncwarp();

      // ---- K phase: 16 channels x 8 tokens x 4 rows per lane
      {
        float2 acc[kRows][4];
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
          for (int k = 0; k < 4; ++k) acc[r][k] = make_float2(0.f, 0.f);
        const uint32_t pa = unitK + k_off;
        const uint32_t cbase = s_coef + 16 * cg;
#pragma unroll 4
        for (int j = 0; j < 16; ++j) {
          const uint32_t wa = lds<uint32_t>(smem, pa + j * 1024);
          const uint32_t wr = FULL ? lds<uint32_t>(smem, pa + G::kResOff + j * 1024) : 0u;
          const float4 c = lds<float4>(smem, cbase + j * 128);       // channel cg + 8j, rows 0-3
          const float2 cc[4] = {make_float2(c.x, c.x), make_float2(c.y, c.y),
                                make_float2(c.z, c.z), make_float2(c.w, c.w)};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 lv = lut_pair<FULL>(lut_lane, wa, wr, k);
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[r][k] = __ffma2_rn(cc[r], lv, acc[r][k]);
          }
        }
        // partial logits -> part[cg][32 tokens] (float4 over rows), xor-swizzled slots
        const int f = (tg + 4 * (cg & 1)) & 7;
#pragma unroll
        for (int e8 = 0; e8 < 8; ++e8) {
          const int k = e8 >> 1;
          const float4 v = (e8 & 1) ? make_float4(acc[0][k].y, acc[1][k].y, acc[2][k].y, acc[3][k].y)
                                    : make_float4(acc[0][k].x, acc[1][k].x, acc[2][k].x, acc[3][k].x);
          const int slot = cg * 32 + 8 * tg + (e8 ^ f);
          *reinterpret_cast<float4*>(smem + s_part + 16 * slot) = v;
        }
      }
      __syncwarp();
      // every read of the K unit is done: hand the slot back
      if (L == 0) mbar_arrive(bar_empty + 8 * sK);

      // ---- logits of token L (of this chunk) for the 4 rows
      float s4[kRows];
      {
        const int tgo = L >> 3, e8 = L & 7;
        float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int f = (tgo + 4 * (c & 1)) & 7;
          const float4 v = lds<float4>(smem, s_part + 16 * (c * 32 + 8 * tgo + (e8 ^ f)));
          acc4.x += v.x;
          acc4.y += v.y;
          acc4.z += v.z;
          acc4.w += v.w;
        }
        s4[0] = acc4.x + ck[0];
        s4[1] = acc4.y + ck[1];
        s4[2] = acc4.z + ck[2];
        s4[3] = acc4.w + ck[3];
      }
      // ---- online softmax over this chunk's 32 tokens
      float corr[kRows], pb[kRows], pv[kRows];
      const int pos = p * kP + 32 * w + L;
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const float sr = (pos < nvis[r]) ? s4[r] : -CUDART_INF_F;
        const float mnew = fmaxf(m_run[r], warp_max(sr));
        corr[r] = (mnew == -CUDART_INF_F) ? 1.0f : exp2f(m_run[r] - mnew);
        pv[r] = (sr == -CUDART_INF_F) ? 0.0f : exp2f(sr - mnew);
        l_run[r] = l_run[r] * corr[r] + pv[r];
        m_run[r] = mnew;
        pb[r] = warp_sum(pv[r]);
      }
      {
        float* p01 = reinterpret_cast<float*>(smem + s_ps01);
        float* p23 = reinterpret_cast<float*>(smem + s_ps23);
        const int m = L >> 1, e = L & 1;
        p01[4 * m + e] = pv[0];
        p01[4 * m + 2 + e] = pv[1];
        p23[4 * m + e] = pv[2];
        p23[4 * m + 2 + e] = pv[3];
      }
      __syncwarp();

      // ---- V unit
      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sV, (uV / kSt) & 1));
      if (failed) break;
      {
        const uint32_t vm = unitV + G::kMetaOff;
        uint4 va[4], vr[4];
        float Av[4], Bv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int d = L + 32 * k;
          const uint32_t off = d * 128 + ((w ^ (d & 7)) << 4);
          va[k] = lds<uint4>(smem, unitV + off);
          vr[k] = FULL ? lds<uint4>(smem, unitV + G::kResOff + off) : make_uint4(0u, 0u, 0u, 0u);
          const float gmin = lds<float>(smem, vm + 4 * d);
          const float dg = __fadd_rn(lds<float>(smem, vm + 4 * (kH + d)), eps);
          const float mu = lds<float>(smem, vm + 4 * (kMetaMuOff + w * kH + d));
          const float ds = __fadd_rn(lds<float>(smem, vm + 4 * (kMetaSigmaOff + w * kH + d)), eps);
          Av[k] = __fmaf_rn(dg, mu, gmin);
          Bv[k] = __fmul_rn(dg, ds);
        }
        __syncwarp();
        if (L == 0) mbar_arrive(bar_empty + 8 * sV);

        float2 acc[4][kRows];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int r = 0; r < kRows; ++r) acc[k][r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float4 a01 = lds<float4>(smem, s_ps01 + 16 * m);
          const float4 a23 = lds<float4>(smem, s_ps23 + 16 * m);
          const float2 pp[4] = {make_float2(a01.x, a01.y), make_float2(a01.z, a01.w),
                                make_float2(a23.x, a23.y), make_float2(a23.z, a23.w)};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t wa = (m < 4) ? va[k].x : (m < 8) ? va[k].y : (m < 12) ? va[k].z : va[k].w;
            const uint32_t wr = (m < 4) ? vr[k].x : (m < 8) ? vr[k].y : (m < 12) ? vr[k].z : vr[k].w;
            const float2 lv = lut_pair<FULL>(lut_lane, wa, wr, m & 3);
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[k][r] = __ffma2_rn(pp[r], lv, acc[k][r]);
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int r = 0; r < kRows; ++r)
            O[k][r] = O[k][r] * corr[r] + Av[k] * pb[r] + Bv[k] * (acc[k][r].x + acc[k][r].y);
      }
    }
    if (failed && L == 0) {
      atomicExch(a.status, 1);
      *s_flag = 1;
    }
  }

  // ================= merge the 8 chunk states of this CTA (the ring is idle now)
  __syncthreads();
  const bool any_failed = *reinterpret_cast<volatile int*>(s_flag) != 0;
  if (any_failed) return;
  float* mm = reinterpret_cast<float*>(smem + S::kMergeM);
  float* ml = reinterpret_cast<float*>(smem + S::kMergeL);
  float* mo = reinterpret_cast<float*>(smem + S::kMergeO);
  if (warp < kConsumers) {
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const float lw = warp_sum(l_run[r]);
      if (L == 0) {
        mm[warp * kRows + r] = m_run[r];
        ml[warp * kRows + r] = lw;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) mo[(warp * kRows + r) * kH + L + 32 * k] = O[k][r];
    }
  }
  __syncthreads();
  float* ws = a.ws + cta * kWsPerCta;
  for (int i = tid; i < kRows * kH; i += kThreadsQ) {
    const int r = i / kH, d = i % kH;
    float mstar = -CUDART_INF_F;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) mstar = fmaxf(mstar, mm[ww * kRows + r]);
    float o = 0.0f, l = 0.0f;
    if (mstar != -CUDART_INF_F) {
#pragma unroll
      for (int ww = 0; ww < kConsumers; ++ww) {
        const float mw = mm[ww * kRows + r];
        if (mw == -CUDART_INF_F) continue;
        const float f = exp2f(mw - mstar);
        o += mo[(ww * kRows + r) * kH + d] * f;
        l += ml[ww * kRows + r] * f;
      }
    }
    ws[r * kH + d] = o;
    if (d == 0) {
      ws[kRows * kH + r] = mstar;
      ws[kRows * kH + kRows + r] = l;
    }
  }
}

// ======================================================================
// Tensor-core variant for 16 query rows per CTA (verification: T draft tokens
// x G heads).  Same producer / ring / chunk-per-warp skeleton; the two
// contractions of a chunk run as TF32 mma.sync m16n8k8 with float32
// accumulation:
//   S[16 rows x 32 tokens] = Q . K^T      (A = Q, exact in TF32: BF16 inputs)
//   O^T[128 x 16 rows]    += V^T . P^T     (per chunk, in the online softmax)
// K and V are dequantised in registers (k = A + B l~, float32) and split into
// a TF32 high part (low 13 mantissa bits cleared) and the float32 remainder,
// so each product keeps ~21 bits: S = Q k_hi + Q k_lo, O += v_hi p_hi +
// v_lo p_hi + v_hi p_lo.
// Token orders: the K side uses two n-tiles per 16 tokens, one holding the even
// and one the odd tokens, so one table lookup per packed byte (two tokens of a
// channel) feeds both tiles.  The V side orders the 8 k-slots of each step so
// that slots (t, t+4) are the two tokens of one byte; with that order the
// probabilities a lane needs for its B fragment are exactly the S accumulator
// entries it already holds.
// ======================================================================

constexpr int kMmaRows = 16;
constexpr int kWarpMmaAB = 0;                       // float2 (A, B) per channel: K side then V side
constexpr int kWarpMmaBytes = 2 * kH * 8;

template <bool FULL>
struct MLayout {
  using G = QGeo<FULL>;
  static constexpr int kRing = 0;
  static constexpr int kLut = kRing + G::kStages * G::kUnit;
  static constexpr int kWarps = kLut + G::kLutBytes;
  static constexpr int kQ = kWarps + kConsumers * kWarpMmaBytes;   // uint4 [16 k-steps][32 lanes]
  static constexpr int kFlag = kQ + 16 * 32 * 16;
  static constexpr int kBar = kFlag + 16;
  static constexpr int kTotal = kBar + 2 * G::kStages * 8;
  static constexpr int kAlloc = kTotal + 1024;
  // merge area (reuses the ring): m[8][16], l[8][16], o[8][16][128]
  static constexpr int kMergeM = 0;
  static constexpr int kMergeL = kMergeM + kConsumers * kMmaRows * 4;
  static constexpr int kMergeO = kMergeL + kConsumers * kMmaRows * 4;
  static_assert(kMergeO + kConsumers * kMmaRows * kH * 4 <= G::kStages * G::kUnit, "merge area");
};
static_assert(MLayout<false>::kAlloc <= 232448, "shared memory (anchor, mma)");
static_assert(MLayout<true>::kAlloc <= 232448, "shared memory (full, mma)");

__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t tf32_hi(float x) { return __float_as_uint(x) & 0xFFFFE000u; }
__device__ __forceinline__ uint32_t tf32_lo(float x) {
  return __float_as_uint(x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u));
}

// l~ pair of the packed byte `byte_sel` (0..3) of word a_word (and r_word)
template <bool FULL>
__device__ __forceinline__ float2 lut_pair_sel(const uint8_t* lut_lane, uint32_t a_word,
                                               uint32_t r_word, uint32_t sel_anchor, int k) {
  if (!FULL) {
    return lds<float2>(lut_lane, prmt(a_word, 0u, sel_anchor));
  } else {
    const uint32_t ab = (a_word >> (8 * k)) & 0xFFu;
    const uint32_t rb = (r_word >> (8 * k)) & 0xFFu;
    const uint32_t c0 = (ab & 0xFu) | ((rb & 0xFu) << 4);
    const uint32_t c1 = (ab >> 4) | (rb & 0xF0u);
    return make_float2(lds<float>(lut_lane, c0 << 7), lds<float>(lut_lane, c1 << 7));
  }
}

template <bool FULL>
__global__ void __launch_bounds__(kThreadsQ, 1)
decode_mma_kernel(const DecodeArgs a, const LutTables lut,
                  const __grid_constant__ CUtensorMap tm_ka, const __grid_constant__ CUtensorMap tm_va,
                  const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_vr) {
  using G = QGeo<FULL>;
  using S = MLayout<FULL>;
  constexpr int kSt = G::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_u32);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int L = tid & 31;
  const int g = L >> 2, t = L & 3;
  const int split = blockIdx.x;
  const int n_rg16 = (a.n_rg + 3) / 4;
  const int h = blockIdx.y / n_rg16;
  const int rg16 = blockIdx.y % n_rg16;
  const int b = blockIdx.z;
  const int TG = a.T * a.G;
  const int max_keys = a.max_pages * kP;

  int ctx = a.ctx_len[b];
  if (ctx < 0 || ctx > max_keys) {
    if (tid == 0) atomicExch(a.status, 3);
    ctx = ctx < 0 ? 0 : max_keys;
  }
  // visible keys of row r of this CTA
  auto n_visible = [&](int r) {
    const int row = rg16 * kMmaRows + r;
    if (row >= TG) return 0;
    const int n = a.causal ? ctx - a.T + row / a.G + 1 : ctx;
    return n < 0 ? 0 : n;
  };
  int max_vis = 0;
  for (int r = 0; r < kMmaRows; ++r) max_vis = max(max_vis, n_visible(r));
  const int nv_g = n_visible(g), nv_g8 = n_visible(g + 8);
  const int n_pages = (max_vis + kP - 1) / kP;
  const int p_begin = split * a.pages_per_split;
  const int np = max(min(p_begin + a.pages_per_split, n_pages) - p_begin, 0);
  const int n_units = 2 * np;
  const int32_t* pt_row = a.page_table + ((int64_t)b * a.Hkv + h) * a.max_pages;

  const uint32_t s_ring = base + S::kRing;
  const uint32_t bar_full = base + S::kBar;
  const uint32_t bar_empty = bar_full + 8 * kSt;
  int* s_flag = reinterpret_cast<int*>(smem + S::kFlag);

  if (!FULL) {
    float2* l2 = reinterpret_cast<float2*>(smem + S::kLut);
    for (int i = tid; i < 256 * 32; i += kThreadsQ) l2[i] = lut.anc_pair[i >> 5];
  } else {
    float* l1 = reinterpret_cast<float*>(smem + S::kLut);
    for (int i = tid; i < 256 * 32; i += kThreadsQ) l1[i] = lut.full[i >> 5];
  }
  if (tid == 0) {
    for (int st = 0; st < kSt; ++st) {
      mbar_init(bar_full + 8 * st, 1);
      mbar_init(bar_empty + 8 * st, kConsumers);
    }
    *s_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Q as TF32 A fragments (BF16 values are exact in TF32): entry (ks, lane) holds
  // Q[g][8ks+t], Q[g+8][8ks+t], Q[g][8ks+t+4], Q[g+8][8ks+t+4]
  for (int i = tid; i < 16 * 32 * 4; i += kThreadsQ) {
    const int e = i & 3, ln = (i >> 2) & 31, ks = i >> 7;
    const int row = rg16 * kMmaRows + (ln >> 2) + 8 * (e & 1);
    const int d = 8 * ks + (ln & 3) + 4 * (e >> 1);
    uint32_t v = 0u;
    if (row < TG)
      v = (uint32_t)a.q[(((int64_t)b * a.T + row / a.G) * a.Hq + h * a.G + row % a.G) * kH + d] << 16;
    reinterpret_cast<uint32_t*>(smem + S::kQ)[i] = v;
  }
  __syncthreads();

  // running softmax state of rows g and g+8 (log2 units), output accumulators O^T
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_run[2] = {0.f, 0.f};
  float O[8][2][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) O[mt][nt][e] = 0.f;

  if (warp == kConsumers) {
    // ================= producer (as in decode_quant_kernel)
    if (L == 0) {
      int issued = 0;
      bool ok = true;
      for (int u = 0; u < n_units; ++u) {
        const int st = u % kSt;
        if (u >= kSt && !mbar_wait(bar_empty + 8 * st, ((u / kSt) - 1) & 1)) {
          ok = false;
          break;
        }
        const int p = p_begin + (u >> 1);
        const bool is_v = (u & 1) != 0;
        int64_t id = pt_row[p];
        if (id < 0 || id >= a.n_pool) {
          atomicExch(a.status, 2);
          id = 0;
        }
        const uint32_t dst = s_ring + st * G::kUnit;
        const uint32_t bar = bar_full + 8 * st;
        mbar_expect_tx(bar, G::kUnit);
        tma_tile_g2s(dst, is_v ? &tm_va : &tm_ka, 0, (int)(id * kH), bar);
        if (FULL) tma_tile_g2s(dst + G::kResOff, is_v ? &tm_vr : &tm_kr, 0, (int)(id * kH), bar);
        bulk_g2s(dst + G::kMetaOff, (is_v ? a.v_meta : a.k_meta) + id * kMetaFloats, kMetaBytes, bar);
        ++issued;
      }
      if (!ok) {
        atomicExch(a.status, 1);
        *s_flag = 1;
        for (int u = issued - 1; u >= 0 && u >= issued - kSt; --u)
          mbar_wait(bar_full + 8 * (u % kSt), (u / kSt) & 1);
      }
    }
  } else {
    const int w = warp;
    const uint32_t s_ab = S::kWarps + w * kWarpMmaBytes;   // float2 [128]: (A_d, B_d)
    const uint8_t* lut_lane = smem + S::kLut + (FULL ? 4 * L : 8 * L);
    const float eps = a.eps;
    const float sc = a.scale_log2;
    bool failed = false;

    auto prep_ab = [&](uint32_t unit) {
      const uint32_t mt = unit + G::kMetaOff;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int d = L + 32 * k;
        const float gmin = lds<float>(smem, mt + 4 * d);
        const float dg = __fadd_rn(lds<float>(smem, mt + 4 * (kH + d)), eps);
        const float mu = lds<float>(smem, mt + 4 * (kMetaMuOff + w * kH + d));
        const float ds = __fadd_rn(lds<float>(smem, mt + 4 * (kMetaSigmaOff + w * kH + d)), eps);
        *reinterpret_cast<float2*>(smem + s_ab + 8 * d) =
            make_float2(__fmaf_rn(dg, mu, gmin), __fmul_rn(dg, ds));
      }
    };

    for (int i = 0; i < np && !failed; ++i) {
      const int p = p_begin + i;
      const int uK = 2 * i, uV = 2 * i + 1;
      const int sK = uK % kSt, sV = uV % kSt;
      const uint32_t unitK = S::kRing + sK * G::kUnit;
      const uint32_t unitV = S::kRing + sV * G::kUnit;

      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sK, (uK / kSt) & 1));
      if (failed) break;
      prep_ab(unitK);
      __syncwarp();

      // ---- S = Q K^T for the chunk: per 16-token group q16, tile A = even tokens, tile B = odd
      float sA[2][4], sB[2][4];
#pragma unroll
      for (int q16 = 0; q16 < 2; ++q16)
#pragma unroll
        for (int e = 0; e < 4; ++e) sA[q16][e] = sB[q16][e] = 0.f;
      {
        // byte 8*q16 + g of the chunk's 16-byte unit: word 2*q16 + (g >> 2), byte g & 3
        const uint32_t sel = 0x4404u | ((uint32_t)(g & 3) << 4);
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const uint4 qf = lds<uint4>(smem, S::kQ + (ks * 32 + L) * 16);
          const int c0 = 8 * ks + t, c1 = c0 + 4;
          const float2 ab0 = lds<float2>(smem, s_ab + 8 * c0);
          const float2 ab1 = lds<float2>(smem, s_ab + 8 * c1);
          const uint32_t r0 = unitK + c0 * 128 + ((w ^ (c0 & 7)) << 4);
          const uint32_t r1 = unitK + c1 * 128 + ((w ^ (c1 & 7)) << 4);
#pragma unroll
          for (int q16 = 0; q16 < 2; ++q16) {
            const uint32_t woff = 4 * (2 * q16 + (g >> 2));
            const uint32_t wa0 = lds<uint32_t>(smem, r0 + woff);
            const uint32_t wa1 = lds<uint32_t>(smem, r1 + woff);
            const uint32_t wr0 = FULL ? lds<uint32_t>(smem, r0 + G::kResOff + woff) : 0u;
            const uint32_t wr1 = FULL ? lds<uint32_t>(smem, r1 + G::kResOff + woff) : 0u;
            const float2 l0 = lut_pair_sel<FULL>(lut_lane, wa0, wr0, sel, g & 3);
            const float2 l1 = lut_pair_sel<FULL>(lut_lane, wa1, wr1, sel, g & 3);
            const float2 k0 = __ffma2_rn(l0, make_float2(ab0.y, ab0.y), make_float2(ab0.x, ab0.x));
            const float2 k1 = __ffma2_rn(l1, make_float2(ab1.y, ab1.y), make_float2(ab1.x, ab1.x));
            // tile A (token 2g of the group): rows c0, c1 at even token; tile B: odd token
            mma_tf32(sA[q16], qf.x, qf.y, qf.z, qf.w, tf32_hi(k0.x), tf32_hi(k1.x));
            mma_tf32(sA[q16], qf.x, qf.y, qf.z, qf.w, tf32_lo(k0.x), tf32_lo(k1.x));
            mma_tf32(sB[q16], qf.x, qf.y, qf.z, qf.w, tf32_hi(k0.y), tf32_hi(k1.y));
            mma_tf32(sB[q16], qf.x, qf.y, qf.z, qf.w, tf32_lo(k0.y), tf32_lo(k1.y));
          }
        }
      }
      __syncwarp();
      if (L == 0) mbar_arrive(bar_empty + 8 * sK);

      // ---- online softmax: lane holds rows g (sX[.][0..1]) and g+8 (sX[.][2..3]),
      // tokens 16 q16 + 4t + {0 (A,0/2), 1 (B,0/2), 2 (A,1/3), 3 (B,1/3)}
      float pr[2][2][4];   // [q16][row half][token 4t+j], log2-scaled then exp'd
      float corr[2];
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        const int nv = rh ? nv_g8 : nv_g;
        float mloc = -CUDART_INF_F;
#pragma unroll
        for (int q16 = 0; q16 < 2; ++q16) {
          const int tok0 = p * kP + 32 * w + 16 * q16 + 4 * t;
          const float v4[4] = {sA[q16][2 * rh], sB[q16][2 * rh], sA[q16][2 * rh + 1], sB[q16][2 * rh + 1]};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float sv = (tok0 + j < nv) ? v4[j] * sc : -CUDART_INF_F;
            pr[q16][rh][j] = sv;
            mloc = fmaxf(mloc, sv);
          }
        }
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
        const float mnew = fmaxf(m_run[rh], mloc);
        corr[rh] = (mnew == -CUDART_INF_F) ? 1.0f : exp2f(m_run[rh] - mnew);
        float ps = 0.f;
#pragma unroll
        for (int q16 = 0; q16 < 2; ++q16)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float sv = pr[q16][rh][j];
            const float pv = (sv == -CUDART_INF_F) ? 0.f : exp2f(sv - mnew);
            pr[q16][rh][j] = pv;
            ps += pv;
          }
        l_run[rh] = l_run[rh] * corr[rh] + ps;
        m_run[rh] = mnew;
      }
      // rescale O^T columns: column 2t + e of n-tile nt is row 8 nt + 2t + e
      {
        const float c_lo0 = __shfl_sync(0xffffffffu, corr[0], (2 * t) * 4);
        const float c_lo1 = __shfl_sync(0xffffffffu, corr[0], (2 * t + 1) * 4);
        const float c_hi0 = __shfl_sync(0xffffffffu, corr[1], (2 * t) * 4);
        const float c_hi1 = __shfl_sync(0xffffffffu, corr[1], (2 * t + 1) * 4);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          O[mt][0][0] *= c_lo0; O[mt][0][1] *= c_lo1; O[mt][0][2] *= c_lo0; O[mt][0][3] *= c_lo1;
          O[mt][1][0] *= c_hi0; O[mt][1][1] *= c_hi1; O[mt][1][2] *= c_hi0; O[mt][1][3] *= c_hi1;
        }
      }

      // ---- V unit: O^T += V^T P^T, 8 m-tiles of 16 channels x 4 k-steps of 8 tokens
      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sV, (uV / kSt) & 1));
      if (failed) break;
      prep_ab(unitV);
      __syncwarp();
      {
        // P^T fragments (rows on n): b0 = P[row][slot t], b1 = P[row][slot t+4] where for
        // k-step (q16, hh) slots t, t+4 are tokens 16 q16 + 4t + 2hh and + 1
        uint32_t pbh[2][2][2][2], pbl[2][2][2][2];   // [q16][hh][nt][b]
#pragma unroll
        for (int q16 = 0; q16 < 2; ++q16)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              // this lane's B fragment needs row (8 nt + g), tokens 4t + 2hh, 4t + 2hh + 1:
              // those are pr[q16][nt][2hh], pr[q16][nt][2hh + 1] held by the lane itself
              const float p0 = pr[q16][nt][2 * hh], p1 = pr[q16][nt][2 * hh + 1];
              pbh[q16][hh][nt][0] = tf32_hi(p0);
              pbh[q16][hh][nt][1] = tf32_hi(p1);
              pbl[q16][hh][nt][0] = tf32_lo(p0);
              pbl[q16][hh][nt][1] = tf32_lo(p1);
            }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int c0 = 16 * mt + g, c1 = c0 + 8;
          const float2 ab0 = lds<float2>(smem, s_ab + 8 * c0);
          const float2 ab1 = lds<float2>(smem, s_ab + 8 * c1);
          const uint32_t r0 = unitV + c0 * 128 + ((w ^ (c0 & 7)) << 4);
          const uint32_t r1 = unitV + c1 * 128 + ((w ^ (c1 & 7)) << 4);
          const uint4 va0 = lds<uint4>(smem, r0), va1 = lds<uint4>(smem, r1);
          uint4 vr0 = make_uint4(0u, 0u, 0u, 0u), vr1 = vr0;
          if (FULL) {
            vr0 = lds<uint4>(smem, r0 + G::kResOff);
            vr1 = lds<uint4>(smem, r1 + G::kResOff);
          }
#pragma unroll
          for (int q16 = 0; q16 < 2; ++q16)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              // byte 8 q16 + 2t + hh of the chunk: word 2 q16 + (t >> 1), byte 2 (t & 1) + hh
              const int bsel = 2 * (t & 1) + hh;
              const uint32_t a0w = (q16 == 0) ? ((t >> 1) ? va0.y : va0.x) : ((t >> 1) ? va0.w : va0.z);
              const uint32_t a1w = (q16 == 0) ? ((t >> 1) ? va1.y : va1.x) : ((t >> 1) ? va1.w : va1.z);
              const uint32_t r0w = (q16 == 0) ? ((t >> 1) ? vr0.y : vr0.x) : ((t >> 1) ? vr0.w : vr0.z);
              const uint32_t r1w = (q16 == 0) ? ((t >> 1) ? vr1.y : vr1.x) : ((t >> 1) ? vr1.w : vr1.z);
              const uint32_t sel = 0x4404u | ((uint32_t)bsel << 4);
              const float2 l0 = lut_pair_sel<FULL>(lut_lane, a0w, r0w, sel, bsel);
              const float2 l1 = lut_pair_sel<FULL>(lut_lane, a1w, r1w, sel, bsel);
              const float2 v0 = __ffma2_rn(l0, make_float2(ab0.y, ab0.y), make_float2(ab0.x, ab0.x));
              const float2 v1 = __ffma2_rn(l1, make_float2(ab1.y, ab1.y), make_float2(ab1.x, ab1.x));
              // A fragment: a0 = (c0, slot t) = v0.x, a1 = (c1, slot t) = v1.x,
              //             a2 = (c0, slot t+4) = v0.y, a3 = (c1, slot t+4) = v1.y
              const uint32_t h0 = tf32_hi(v0.x), h1 = tf32_hi(v1.x), h2 = tf32_hi(v0.y), h3 = tf32_hi(v1.y);
              const uint32_t o0 = tf32_lo(v0.x), o1 = tf32_lo(v1.x), o2 = tf32_lo(v0.y), o3 = tf32_lo(v1.y);
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
                mma_tf32(O[mt][nt], h0, h1, h2, h3, pbh[q16][hh][nt][0], pbh[q16][hh][nt][1]);
                mma_tf32(O[mt][nt], o0, o1, o2, o3, pbh[q16][hh][nt][0], pbh[q16][hh][nt][1]);
                mma_tf32(O[mt][nt], h0, h1, h2, h3, pbl[q16][hh][nt][0], pbl[q16][hh][nt][1]);
              }
            }
        }
      }
      __syncwarp();
      if (L == 0) mbar_arrive(bar_empty + 8 * sV);
    }
    if (failed && L == 0) {
      atomicExch(a.status, 1);
      *s_flag = 1;
    }
  }

  // ================= merge the 8 chunk states (ring idle)
  __syncthreads();
  if (*reinterpret_cast<volatile int*>(s_flag) != 0) return;
  float* mm = reinterpret_cast<float*>(smem + S::kMergeM);
  float* ml = reinterpret_cast<float*>(smem + S::kMergeL);
  float* mo = reinterpret_cast<float*>(smem + S::kMergeO);
  if (warp < kConsumers) {
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      float lw = l_run[rh];
      lw += __shfl_xor_sync(0xffffffffu, lw, 1);
      lw += __shfl_xor_sync(0xffffffffu, lw, 2);
      if (t == 0) {
        mm[warp * kMmaRows + g + 8 * rh] = m_run[rh];
        ml[warp * kMmaRows + g + 8 * rh] = lw;
      }
    }
    // O^T[channel][row]: m-tile mt rows 16 mt + g (+8), n-tile nt columns 8 nt + 2t (+1)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int r0 = 8 * nt + 2 * t;
        const int c0 = 16 * mt + g;
        mo[(warp * kMmaRows + r0) * kH + c0] = O[mt][nt][0];
        mo[(warp * kMmaRows + r0 + 1) * kH + c0] = O[mt][nt][1];
        mo[(warp * kMmaRows + r0) * kH + c0 + 8] = O[mt][nt][2];
        mo[(warp * kMmaRows + r0 + 1) * kH + c0 + 8] = O[mt][nt][3];
      }
  }
  __syncthreads();
  // write the 16 rows as four 4-row groups in the split workspace layout
  for (int i = tid; i < kMmaRows * kH; i += kThreadsQ) {
    const int r = i / kH, d = i % kH;
    const int rg4 = rg16 * 4 + r / 4;
    if (rg4 >= a.n_rg) continue;
    float mstar = -CUDART_INF_F;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) mstar = fmaxf(mstar, mm[ww * kMmaRows + r]);
    float o = 0.0f, l = 0.0f;
    if (mstar != -CUDART_INF_F) {
#pragma unroll
      for (int ww = 0; ww < kConsumers; ++ww) {
        const float mw = mm[ww * kMmaRows + r];
        if (mw == -CUDART_INF_F) continue;
        const float f = exp2f(mw - mstar);
        o += mo[(ww * kMmaRows + r) * kH + d] * f;
        l += ml[ww * kMmaRows + r] * f;
      }
    }
    const int64_t cta = (((int64_t)b * a.Hkv + h) * a.n_rg + rg4) * a.n_splits + split;
    float* ws = a.ws + cta * kWsPerCta;
    ws[(r % 4) * kH + d] = o * 1.0f;
    if (d == 0) {
      ws[kRows * kH + (r % 4)] = mstar;
      ws[kRows * kH + kRows + (r % 4)] = l;
    }
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D map over a pool of 4-bit planes: rows of 128 bytes, one 128 x 128 tile per page
bool plane_map(CUtensorMap* m, const uint8_t* pool, int64_t n_pool) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {128, (cuuint64_t)n_pool * kH};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(pool), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FULL>
cudaError_t launch_q(const DecodeArgs& a, const LutTables* lut, cudaStream_t s) {
  constexpr int kSmem = QLayout<FULL>::kAlloc;
  constexpr int kSmemM = MLayout<FULL>::kAlloc;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_quant_kernel<FULL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_mma_kernel<FULL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemM);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  CUtensorMap tka, tva, tkr, tvr;
  if (n_pool_too_large(a.n_pool)) return cudaErrorInvalidValue;
  if (!plane_map(&tka, a.k_anc, a.n_pool) || !plane_map(&tva, a.v_anc, a.n_pool))
    return cudaErrorInvalidValue;
  if (FULL) {
    if (!plane_map(&tkr, a.k_res, a.n_pool) || !plane_map(&tvr, a.v_res, a.n_pool))
      return cudaErrorInvalidValue;
  } else {
    tkr = tka;
    tvr = tva;
  }
  if (use_mma_rows(a.T * a.G)) {
    const int n_rg16 = (a.n_rg + 3) / 4;
    dim3 grid(a.n_splits, a.Hkv * n_rg16, a.B);
    decode_mma_kernel<FULL><<<grid, kThreadsQ, kSmemM, s>>>(a, *lut, tka, tva, tkr, tvr);
  } else {
    dim3 grid(a.n_splits, a.Hkv * a.n_rg, a.B);
    decode_quant_kernel<FULL><<<grid, kThreadsQ, kSmem, s>>>(a, *lut, tka, tva, tkr, tvr);
  }
  return cudaGetLastError();
}

}  // namespace

// query rows per (sequence, KV head) from which the tensor-core kernel is used
bool use_mma_rows(int rows) { return rows >= 12; }

// the TMA row coordinate (page id * 128) is a signed 32-bit value
bool n_pool_too_large(int64_t n_pool) { return n_pool <= 0 || n_pool * kH > ((int64_t)1 << 31) - 1; }

cudaError_t launch_decode_quant(const DecodeArgs& a, bool full, const LutTables* lut, cudaStream_t s) {
  return full ? launch_q<true>(a, lut, s) : launch_q<false>(a, lut, s);
}

}  // namespace lynx
