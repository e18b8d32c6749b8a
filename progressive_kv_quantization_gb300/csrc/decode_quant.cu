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
// logits are summed by a shuffle reduce-scatter (xor 16, 8, 4) that leaves
// lane (tg, cg) with token 8tg + cg.  V phase, lane L: channels
// L + 32k (k = 0..3), all 32 tokens of the chunk (one 16-byte unit per row).

#include "decode_common.cuh"

namespace lynx {
namespace {

// per consumer warp: coefficients [128][4 rows] f32, probabilities [16 pairs] f32x4
// for rows 0-1 and 2-3
constexpr int kWarpCoef = 0;
constexpr int kWarpPs01 = kWarpCoef + kH * 4 * 4;
constexpr int kWarpPs23 = kWarpPs01 + 16 * 16;
constexpr int kWarpBytes = kWarpPs23 + 16 * 16;

// ring slots of the CUDA-core kernel: 4 for the anchor planes (more bytes in
// flight; shared memory allows it), 3 for the full codes
template <bool FULL>
constexpr int kStagesQ = FULL ? 3 : 4;

template <bool FULL>
struct QLayout {
  using G = QGeo<FULL, kStagesQ<FULL>>;
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

// value pair (l~ of token 2m, l~ of token 2m+1) for one anchor byte, or for
// one anchor byte and the matching residual byte
// lut points at the table; lane_off is the lane's copy offset (8L anchor, 4L full)
template <bool FULL>
__device__ __forceinline__ float2 lut_pair(const uint8_t* lut, uint32_t lane_off, uint32_t a_word,
                                           uint32_t r_word, int k) {
  if (!FULL) {
    // entry stride 256 B: byte k of a_word in bits 8..15, the lane's offset (< 256) in bits 0..7
    const uint32_t off = prmt(a_word, lane_off, 0x5504u | ((uint32_t)k << 4));
    return lds<float2>(lut, off);
  } else {
    const uint32_t ab = (a_word >> (8 * k)) & 0xFFu;
    const uint32_t rb = (r_word >> (8 * k)) & 0xFFu;
    const uint32_t c0 = (ab & 0xFu) | ((rb & 0xFu) << 4);
    const uint32_t c1 = (ab >> 4) | (rb & 0xF0u);
    return make_float2(lds<float>(lut, lane_off + (c0 << 7)), lds<float>(lut, lane_off + (c1 << 7)));
  }
}

template <bool FULL>
__global__ void __launch_bounds__(kThreadsQ, 1)
decode_quant_kernel(const DecodeArgs a, const LutTables lut,
                    const __grid_constant__ CUtensorMap tm_ka, const __grid_constant__ CUtensorMap tm_va,
                    const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_vr) {
  using G = QGeo<FULL, kStagesQ<FULL>>;
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
    if (L == 0)
      produce_units<FULL, kStagesQ<FULL>>(a, pt_row, p_begin, np, s_ring, bar_full, bar_empty, &tm_ka, &tm_va, &tm_kr,
                          &tm_vr, s_flag);
  } else {
    // ================= consumers: warp `warp` owns chunk `warp` of every page
    const int w = warp;
    // offsets from smem
    const uint32_t s_w = S::kWarps + w * kWarpBytes;
    const uint32_t s_coef = s_w + kWarpCoef;
    const uint32_t s_ps01 = s_w + kWarpPs01;
    const uint32_t s_ps23 = s_w + kWarpPs23;
    const uint32_t s_qs = S::kQs;
    const int tg = L & 3, cg = L >> 2;
    // K phase: plane word of (row cg + 8j, unit w ^ cg, word tg) = k_off + j * 1024
    const uint32_t k_off = cg * 128 + ((w ^ cg) << 4) + 4 * tg;
    const uint8_t* lut = smem + S::kLut;
    const uint32_t lane_off = FULL ? 4u * L : 8u * L;
    const float eps = a.eps;
    float4 qd[4];   // scaled queries of channels L + 32k, rows 0-3
#pragma unroll
    for (int k = 0; k < 4; ++k) qd[k] = lds<float4>(smem, s_qs + 16 * (L + 32 * k));
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
          const float4 q = qd[k];
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
      float s4[kRows];   // logits of token 8tg + cg of this chunk
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
            const float2 lv = lut_pair<FULL>(lut, lane_off, wa, wr, k);
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[r][k] = __ffma2_rn(cc[r], lv, acc[r][k]);
          }
        }
        // Reduce the partial logits (row r, token 8tg + e8; e8 = 2k (+1 for .y)) over
        // the 8 lanes of equal tg (lane bits 2..4) while scattering them: each xor
        // exchange halves the token range a lane keeps, so that lane (tg, cg) ends
        // with the four rows of token 8tg + cg.
        const bool b2 = (cg & 4) != 0, b1 = (cg & 2) != 0, b0 = (cg & 1) != 0;
        float w4[kRows][4];
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = (e & 1) ? acc[r][e >> 1].y : acc[r][e >> 1].x;          // token e
            const float hi = (e & 1) ? acc[r][2 + (e >> 1)].y : acc[r][2 + (e >> 1)].x;   // token 4 + e
            w4[r][e] = (b2 ? hi : lo) + __shfl_xor_sync(0xffffffffu, b2 ? lo : hi, 16);
          }
        float w2[kRows][2];
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            w2[r][e] = (b1 ? w4[r][2 + e] : w4[r][e]) +
                       __shfl_xor_sync(0xffffffffu, b1 ? w4[r][e] : w4[r][2 + e], 8);
#pragma unroll
        for (int r = 0; r < kRows; ++r)
          s4[r] = (b0 ? w2[r][1] : w2[r][0]) + __shfl_xor_sync(0xffffffffu, b0 ? w2[r][0] : w2[r][1], 4) +
                  ck[r];
      }
      __syncwarp();
      // every read of the K unit is done: hand the slot back
      if (L == 0) mbar_arrive(bar_empty + 8 * sK);

      // ---- online softmax over this chunk's 32 tokens
      float corr[kRows], pb[kRows], pv[kRows];
      const int tok = 8 * tg + cg;
      const int pos = p * kP + 32 * w + tok;
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
        const int m = tok >> 1, e = tok & 1;
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
            const float2 lv = lut_pair<FULL>(lut, lane_off, wa, wr, m & 3);
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

template <bool FULL>
cudaError_t launch_q(const DecodeArgs& a, const LutTables* lut, cudaStream_t s) {
  constexpr int kSmem = QLayout<FULL>::kAlloc;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_quant_kernel<FULL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
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
  dim3 grid(a.n_splits, a.Hkv * a.n_rg, a.B);
  decode_quant_kernel<FULL><<<grid, kThreadsQ, kSmem, s>>>(a, *lut, tka, tva, tkr, tvr);
  return cudaGetLastError();
}

}  // namespace

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

// the TMA row coordinate (page id * 128) is a signed 32-bit value
bool n_pool_too_large(int64_t n_pool) { return n_pool <= 0 || n_pool * kH > ((int64_t)1 << 31) - 1; }

cudaError_t launch_decode_quant(const DecodeArgs& a, bool full, const LutTables* lut, cudaStream_t s) {
  if (use_tc_rows(a.T * a.G)) return launch_decode_tc(a, full, lut, s);
  return full ? launch_q<true>(a, lut, s) : launch_q<false>(a, lut, s);
}

}  // namespace lynx
