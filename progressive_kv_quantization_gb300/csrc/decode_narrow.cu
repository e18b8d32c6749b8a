// Tensor-core decode attention over Lynx-encoded pages for a few query rows per
// KV head: the draft decode (T = 1, the Anchor-only KV of the Lynx paper's
// §4.2) and short verifications, the attention of §2.1 with 8 query rows per
// CTA taking the n = 8 dimension of the mma.sync tiles (rows past T x Hq/Hkv
// are zero).
//
// CTA skeleton as in the wider verification kernel: a producer lane streams
// the split's K and V page units through a 3-slot shared-memory ring (2-D TMA
// tile for the planes, bulk copy for the metadata); 8 consumer warps, warp w
// owning the 32-token chunk w of every page with its own online softmax; one
// merge of the 8 chunk states at the end.
//
//   K side   S^T[32 tokens x 8 rows] = K Q^T as TF32 m16n8k8: two m-tiles of
//            16 tokens, 16 k-steps of 8 channels.  k = A + B l~ is dequantised
//            in float32 (A = gamma_min + (gamma_scale + eps) mu,
//            B = (gamma_scale + eps)(sigma + eps)) and split into its TF32 head
//            and the float32 remainder, two MMAs (~21-bit products); Q (BF16)
//            is exact in TF32.  Row g of m-tile mi holds token 4g + 2mi and
//            row g + 8 token 4g + 2mi + 1: the two tokens of byte
//            2 (g & 1) + mi of plane word g >> 1, so one table lookup per
//            plane byte gives both rows of a fragment register pair.  No
//            cross-lane reduction follows: the MMA sums the channels.
//   V side   U[128 channels x 8 rows] = l~ P^T as fp16 m16n8k16, two k-steps
//            of 16 tokens per chunk, folded into the output with the chunk's
//            constants (O = O corr + A psum + B U), exactly as in the wider
//            kernel: l~ from a table of fp16 head/remainder pairs (two MMAs,
//            ~22 bits), P in fp16 scaled by 2^10.  Slot order of k-step kv:
//            slots 2t, 2t+1 hold tokens 8t + 4kv + {0, 1}, slots 2t+8, 2t+9
//            hold 8t + 4kv + {2, 3}, so the A fragments are plane bytes as
//            stored.
//
// Lane (g = L >> 2, t = L & 3) holds S of query rows 2t and 2t+1 for tokens
// 4g .. 4g+3 of its chunk, and O of channels 16 mt + g (+ 8) for the same two
// rows, so the per-row softmax statistics a lane needs for its output are its
// own.  The P^T fragments of the V side (row g, tokens 8t + 4kv + 0..3) come
// from lane 4 (2t + kv) + (g >> 1) by shuffles.
//
// Softmax.  A row's running maximum moves only when one of the chunk's scores
// exceeds it by more than 5 in log2 units (a probability factor of 2^5; a warp
// vote, then the rows take their maxima by shuffles), so most pages skip the
// max reduction and the rescale, and the probabilities (x 2^10) stay below
// 2^15, inside fp16.  The chunk's row sums of the fp16 probabilities come from
// one more MMA pair, ones x P^T, instead of a shuffle reduction; they feed
// both the output and the normaliser, so the two see the same probabilities.
//
// Rounding: P is rounded to fp16 (relative 2^-11); everything else keeps at
// least ~21 bits, sums are float32.

#include "decode_common.cuh"

namespace lynx {
namespace {

constexpr int kNr = 8;                 // query rows per CTA
constexpr float kLazyLog2 = 5.0f;      // largest log2 lead of a score over the running maximum
constexpr uint32_t kOnes2 = 0x3C003C00u;   // fp16 pair (1, 1)
constexpr int kNrWarpBytes = kH * 8;   // per warp: float2 (A, B) per channel of the current unit

template <bool FULL>
struct NLayout {
  using G = QGeo<FULL>;
  static constexpr int kRing = 0;
  // Tables, 32 copies (one per lane) in rows of 256 B, row = byte or code.
  //   anchor  kLutK: byte -> (l~ low nibble, l~ high nibble) float2, copy at 8L
  //           kLutV: byte -> fp16 pairs (heads, remainders), copy at 8L
  //   full    kLutK: code -> l~ float, copy at 4L; fp16 (head, remainder) at 128 + 4L
  static constexpr int kLutK = kRing + G::kStages * G::kUnit;
  static constexpr int kLutV = FULL ? kLutK : kLutK + 256 * 256;
  static constexpr int kWarps = kLutV + 256 * 256;
  static constexpr int kQ = kWarps + kConsumers * kNrWarpBytes;   // BF16 pairs [16 k-steps][32 lanes]
  static constexpr int kFlag = kQ + 16 * 32 * 4;
  static constexpr int kBar = kFlag + 16;
  static constexpr int kTotal = kBar + 2 * G::kStages * 8;
  static constexpr int kAlloc = kTotal + 1024;
  // end-of-kernel merge area (reuses the ring): m[8][8], l[8][8], o[8][8][128]
  static constexpr int kMergeM = 0;
  static constexpr int kMergeL = kMergeM + kConsumers * kNr * 4;
  static constexpr int kMergeO = kMergeL + kConsumers * kNr * 4;
  static_assert(kMergeO + kConsumers * kNr * kH * 4 <= G::kStages * G::kUnit, "merge area");
};
static_assert(NLayout<false>::kAlloc <= 232448, "shared memory (anchor, narrow)");
static_assert(NLayout<true>::kAlloc <= 232448, "shared memory (full, narrow)");

// UNI: uniform-code metadata (min, scale per channel row) instead of Lynx's
template <bool FULL, bool UNI>
__global__ void __launch_bounds__(kThreadsQ, 1)
decode_narrow_kernel(const DecodeArgs a, const LutTables lut,
                     const __grid_constant__ CUtensorMap tm_ka, const __grid_constant__ CUtensorMap tm_va,
                     const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_vr) {
  using G = QGeo<FULL>;
  using S = NLayout<FULL>;
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
  const int TG = a.T * a.G;
  const int n_tiles = (TG + kNr - 1) / kNr;
  const int h = blockIdx.y / n_tiles;
  const int row0 = (blockIdx.y % n_tiles) * kNr;
  const int b = blockIdx.z;
  const int max_keys = a.max_pages * kP;

  const uint32_t s_ring = base + S::kRing;
  const uint32_t bar_full = base + S::kBar;
  const uint32_t bar_empty = bar_full + 8 * kSt;
  int* s_flag = reinterpret_cast<int*>(smem + S::kFlag);

  // ---- prologue: barriers first; the producer lane starts streaming pages
  // while the consumer warps fill the value tables and the Q^T fragments
  if (tid == 0) {
    for (int st = 0; st < kSt; ++st) {
      mbar_init(bar_full + 8 * st, 1);
      mbar_init(bar_empty + 8 * st, kConsumers);
    }
    *s_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // value tables (kernel parameters only), by the consumer warps, before the
  // wait on the kernel ahead in the stream: with a programmatic launch this
  // overlaps that kernel's tail
  if (warp < kConsumers) {
    // thread e makes row e of the tables and stores its 32 copies, the copy
    // index rotated by the lane so that a warp's stores hit different banks
    {
      const int e = tid;
      if (!FULL) {
        const float2 v = lut.anc_pair[e];
        const __half hx = __float2half_rn(v.x), hy = __float2half_rn(v.y);
        const __half lx = __float2half_rn(v.x - __half2float(hx));
        const __half ly = __float2half_rn(v.y - __half2float(hy));
        const uint2 pv = make_uint2(h2(hx, hy), h2(lx, ly));
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
          const int ln = (L + k) & 31;
          *reinterpret_cast<float2*>(smem + S::kLutK + e * 256 + 8 * ln) = v;
          *reinterpret_cast<uint2*>(smem + S::kLutV + e * 256 + 8 * ln) = pv;
        }
      } else {
        const float v = lut.full[e];
        const __half hv = __float2half_rn(v);
        const __half lv = __float2half_rn(v - __half2float(hv));
        const uint32_t pv = h2(hv, lv);
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
          const int ln = (L + k) & 31;
          *reinterpret_cast<float*>(smem + S::kLutK + e * 256 + 4 * ln) = v;
          *reinterpret_cast<uint32_t*>(smem + S::kLutK + e * 256 + 128 + 4 * ln) = pv;
        }
      }
    }
  }
  // every global-memory access of this kernel follows this wait
  wait_prerequisite_grids();
  // the producer lane reads its first page id together with the context length
  int first_id = 0;
  if (tid == kConsumers * 32) {
    const int pb = split * a.pages_per_split;
    if (pb < a.max_pages) first_id = a.page_table[((int64_t)b * a.Hkv + h) * a.max_pages + pb];
  }

  int ctx = a.ctx_len[b];
  if (ctx < 0 || ctx > max_keys) {
    if (tid == 0) atomicExch(a.status, 3);
    ctx = ctx < 0 ? 0 : max_keys;
  }
  // keys visible to row r of this CTA (0 for padding rows)
  auto n_visible = [&](int r) {
    const int row = row0 + r;
    if (row >= TG) return 0;
    const int n = a.causal ? ctx - a.T + row / a.G + 1 : ctx;
    return n < 0 ? 0 : n;
  };
  // n_visible does not decrease with the row: the extremes are the CTA's
  // first and last real rows (the grid's row tiles start below TG)
  const int max_vis = n_visible(min(kNr, TG - row0) - 1);
  const int min_vis = n_visible(0);
  const int nv[2] = {n_visible(2 * t), n_visible(2 * t + 1)};   // the lane's query rows
  const int n_pages = (max_vis + kP - 1) / kP;
  const int p_begin = split * a.pages_per_split;
  const int np = max(min(p_begin + a.pages_per_split, n_pages) - p_begin, 0);
  const int32_t* pt_row = a.page_table + ((int64_t)b * a.Hkv + h) * a.max_pages;

  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};   // query rows 2t, 2t + 1
  float l_run[2] = {0.0f, 0.0f};
  // O[mt]: (channel 16 mt + g, rows 2t, 2t+1), (channel 16 mt + g + 8, rows 2t, 2t+1)
  float2 O[8][2];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) O[mt][0] = O[mt][1] = make_float2(0.f, 0.f);

  if (warp == kConsumers) {
    if (L == 0)
      produce_units<FULL>(a, pt_row, p_begin, np, first_id, s_ring, bar_full, bar_empty, &tm_ka, &tm_va, &tm_kr,
                          &tm_vr, s_flag);
  } else {
    // the Q^T fragments; the consumer warps meet at named barrier 1 (the
    // producer warp never takes part in it)
    // entry (ks, lane): query row g' (= lane >> 2), BF16 of channel 8 ks + t' in
    // the low half and of channel 8 ks + t' + 4 in the high half; a BF16 value
    // shifted into the top half of a word is its exact TF32 operand
    for (int i = tid; i < 16 * 32; i += kConsumerThreads) {
      const int ln = i & 31, ks = i >> 5;
      const int row = row0 + (ln >> 2);
      const int d = 8 * ks + (ln & 3);
      uint32_t v = 0u;
      if (row < TG) {
        const uint16_t* qr = a.q + (((int64_t)b * a.T + row / a.G) * a.Hq + h * a.G + row % a.G) * kH;
        v = (uint32_t)qr[d] | ((uint32_t)qr[d + 4] << 16);
      }
      reinterpret_cast<uint32_t*>(smem + S::kQ)[i] = v;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");

    const int w = warp;
    const uint32_t s_ab = S::kWarps + w * kNrWarpBytes;
    const uint32_t lane8 = 8u * L, lane4 = 4u * L, lane4v = 128u + 4u * L;
    // K side: bytes 2 (g & 1) (m-tile 0) and 2 (g & 1) + 1 (m-tile 1) of word g >> 1 of a channel row
    const uint32_t ksel0 = byte_sel(2 * (g & 1)), ksel1 = byte_sel(2 * (g & 1) + 1);
    const uint32_t kword = 4 * (g >> 1);
    // V side: bytes 4t..4t+3 of channel 16 mt + g, word t of its chunk unit
    const uint32_t vofs = g * 128 + ((w ^ g) << 4) + 4 * t;
    // source lanes of the P^T fragments of V k-steps 0 and 1
    const int src0 = 4 * (2 * t) + (g >> 1), src1 = src0 + 4;
    const bool odd_row = (g & 1) != 0;
    const float eps = a.eps;
    const float sc = a.scale_log2;
    bool failed = false;

    // (A, B) of the unit's 128 channels, stored so that the two channels one
    // lane contracts together share a 16-byte slot: key unit, channels c and
    // c + 4 (c & 4 == 0) at slot 8 (c >> 3) + 2 (c & 3); value unit, channels
    // c and c + 8 (c & 8 == 0) at slot 16 (c >> 4) + 2 (c & 7)
    auto prep_ab = [&](uint32_t unit, bool key) {
      const uint32_t mt = unit + G::kMetaOff;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int d = L + 32 * k;
        float2 ab;
        if (UNI) {   // uniform codes: value = min + scale * code in every chunk
          ab = make_float2(lds<float>(smem, mt + 4 * d), lds<float>(smem, mt + 4 * (kH + d)));
        } else {
          const float gmin = lds<float>(smem, mt + 4 * d);
          const float dg = __fadd_rn(lds<float>(smem, mt + 4 * (kH + d)), eps);
          const float mu = lds<float>(smem, mt + 4 * (kMetaMuOff + w * kH + d));
          const float ds = __fadd_rn(lds<float>(smem, mt + 4 * (kMetaSigmaOff + w * kH + d)), eps);
          ab = make_float2(__fmaf_rn(dg, mu, gmin), __fmul_rn(dg, ds));
        }
        const int slot = key ? 8 * (d >> 3) + 2 * (d & 3) + ((d >> 2) & 1)
                             : 16 * (d >> 4) + 2 * (d & 7) + ((d >> 3) & 1);
        *reinterpret_cast<float2*>(smem + s_ab + 8 * slot) = ab;
      }
    };

    for (int i = 0; i < np && !failed; ++i) {
      const int p = p_begin + i;
      const int uK = 2 * i, uV = 2 * i + 1;
      const int sK = uK % kSt, sV = uV % kSt;
      const uint32_t unitK = S::kRing + sK * G::kUnit;
      const uint32_t unitV = S::kRing + sV * G::kUnit;

      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sK, (uK / kSt) & 1, a.wait_ns));
      if (failed) break;
      prep_ab(unitK, true);
      __syncwarp();

      // ---- S^T = K Q^T over 16 k-steps of channels (t, t + 4) + 8 ks
      float sacc[2][4];   // [m-tile][(token even, row 2t), (even, 2t+1), (odd, 2t), (odd, 2t+1)]
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mi][e] = 0.0f;
      // the plane words of all 16 k-steps first, so that no table lookup
      // waits on its word's load
      uint32_t kw[16][2];
      if (!FULL) {
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const int c0 = 8 * ks + t, c1 = c0 + 4;
          kw[ks][0] = lds<uint32_t>(smem, unitK + c0 * 128 + ((w ^ (c0 & 7)) << 4) + kword);
          kw[ks][1] = lds<uint32_t>(smem, unitK + c1 * 128 + ((w ^ (c1 & 7)) << 4) + kword);
        }
      }
#pragma unroll
      for (int ks = 0; ks < 16; ++ks) {
        const uint32_t qw = lds<uint32_t>(smem, S::kQ + (ks * 32 + L) * 4);
        const uint2 qf = make_uint2(qw << 16, qw & 0xFFFF0000u);
        const int c0 = 8 * ks + t, c1 = c0 + 4;
        const float4 ab = lds<float4>(smem, s_ab + 16 * (4 * ks + t));   // (A, B) of c0, c1
        const uint32_t r0 = unitK + c0 * 128 + ((w ^ (c0 & 7)) << 4) + kword;
        const uint32_t r1 = unitK + c1 * 128 + ((w ^ (c1 & 7)) << 4) + kword;
        const uint32_t wa0 = FULL ? lds<uint32_t>(smem, r0) : kw[ks][0];
        const uint32_t wa1 = FULL ? lds<uint32_t>(smem, r1) : kw[ks][1];
        // l~ pairs (even, odd token) of m-tiles 0 and 1 for channels c0, c1
        float2 l00, l01, l10, l11;
        if (!FULL) {
          l00 = lds<float2>(smem, S::kLutK + lut_off(wa0, lane8, ksel0));
          l01 = lds<float2>(smem, S::kLutK + lut_off(wa0, lane8, ksel1));
          l10 = lds<float2>(smem, S::kLutK + lut_off(wa1, lane8, ksel0));
          l11 = lds<float2>(smem, S::kLutK + lut_off(wa1, lane8, ksel1));
        } else {
          uint32_t e0, o0, e1, o1;
          full_codes(wa0, lds<uint32_t>(smem, r0 + G::kResOff), e0, o0);
          full_codes(wa1, lds<uint32_t>(smem, r1 + G::kResOff), e1, o1);
          auto val = [&](uint32_t codes, uint32_t sel) {
            return lds<float>(smem, S::kLutK + lut_off(codes, lane4, sel));
          };
          l00 = make_float2(val(e0, ksel0), val(o0, ksel0));
          l01 = make_float2(val(e0, ksel1), val(o0, ksel1));
          l10 = make_float2(val(e1, ksel0), val(o1, ksel0));
          l11 = make_float2(val(e1, ksel1), val(o1, ksel1));
        }
        const float2 A0 = make_float2(ab.x, ab.x), B0 = make_float2(ab.y, ab.y);
        const float2 A1 = make_float2(ab.z, ab.z), B1 = make_float2(ab.w, ab.w);
        // m-tile mi: a0 = (even token, c0), a1 = (odd token, c0), a2 = (even, c1), a3 = (odd, c1)
        const float2 k0[2] = {__ffma2_rn(l00, B0, A0), __ffma2_rn(l01, B0, A0)};
        const float2 k1[2] = {__ffma2_rn(l10, B1, A1), __ffma2_rn(l11, B1, A1)};
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          mma_tf32(sacc[mi], tf32_hi(k0[mi].x), tf32_hi(k0[mi].y), tf32_hi(k1[mi].x), tf32_hi(k1[mi].y), qf.x,
                   qf.y);
          mma_tf32(sacc[mi], tf32_lo(k0[mi].x), tf32_lo(k0[mi].y), tf32_lo(k1[mi].x), tf32_lo(k1[mi].y), qf.x,
                   qf.y);
        }
      }
      __syncwarp();
      if (L == 0) mbar_arrive(bar_empty + 8 * sK);

      // ---- online softmax of query rows 2t + e over this chunk's 32 tokens:
      // the lane holds token 4g + j (j = 2 mi + hh) at sacc[mi][2 hh + e]; the
      // row's other tokens are in the lanes of equal t (lane bits 2..4)
      const int pos0 = p * kP + 32 * w + 4 * g;
      const bool all_visible = (p + 1) * kP <= min_vis;
      float pr[2][4];   // [e][j], probabilities x 2^10
      float corr[2], mloc[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        mloc[e] = -CUDART_INF_F;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float sv = sacc[j >> 1][2 * (j & 1) + e] * sc;
          if (!all_visible && pos0 + j >= nv[e]) sv = -CUDART_INF_F;
          pr[e][j] = sv;
          mloc[e] = fmaxf(mloc[e], sv);
        }
      }
      // the running maximum moves only when a score of the chunk exceeds it by
      // more than kLazyLog2 (then every row of the warp takes its row maximum);
      // otherwise the probabilities stay below 2^(10 + kLazyLog2), inside fp16
      const bool grow = __any_sync(0xffffffffu, mloc[0] > m_run[0] + kLazyLog2 || mloc[1] > m_run[1] + kLazyLog2);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mnew = m_run[e];
        if (grow) {
          float mr = mloc[e];
          mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, 4));
          mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, 8));
          mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, 16));
          mnew = fmaxf(m_run[e], mr);
        }
        corr[e] = (!grow || mnew == -CUDART_INF_F) ? 1.0f : exp2f(m_run[e] - mnew);
        // p x 2^10 = 2^(s - (m - 10)); a masked score (-inf) gives 0, and a row
        // with no visible score yet (m = -inf) takes reference 0 instead
        const float mref = (mnew == -CUDART_INF_F) ? 0.0f : mnew - 10.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) pr[e][j] = exp2f(pr[e][j] - mref);
        m_run[e] = mnew;
      }
      // P^T fragments: b0 / b1 of k-step kv = row g, tokens 8t + 4kv + {0,1} / {2,3},
      // held by lane 4 (2t + kv) + (g >> 1) as its pairs of row 2 (g >> 1) + (g & 1)
      const uint32_t x00 = h2(pr[0][0], pr[0][1]), x01 = h2(pr[0][2], pr[0][3]);
      const uint32_t x10 = h2(pr[1][0], pr[1][1]), x11 = h2(pr[1][2], pr[1][3]);
      uint32_t pb[2][2];
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const int src = kv ? src1 : src0;
        const uint32_t y00 = __shfl_sync(0xffffffffu, x00, src), y01 = __shfl_sync(0xffffffffu, x01, src);
        const uint32_t y10 = __shfl_sync(0xffffffffu, x10, src), y11 = __shfl_sync(0xffffffffu, x11, src);
        pb[kv][0] = odd_row ? y10 : y00;
        pb[kv][1] = odd_row ? y11 : y01;
      }
      // the chunk's row sums of the fp16 probabilities the V side multiplies,
      // from a 16 x 32 matrix of ones times P^T (every accumulator row holds
      // them; the lane's entries 0 and 1 are its rows 2t and 2t + 1)
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
      mma_f16(ps4, kOnes2, kOnes2, kOnes2, kOnes2, pb[0][0], pb[0][1]);
      mma_f16(ps4, kOnes2, kOnes2, kOnes2, kOnes2, pb[1][0], pb[1][1]);
      const float2 cr = make_float2(corr[0], corr[1]);
      const float2 pss = make_float2(ps4[0], ps4[1]);
      l_run[0] = l_run[0] * corr[0] + pss.x;
      l_run[1] = l_run[1] * corr[1] + pss.y;
      const bool rescale = __any_sync(0xffffffffu, corr[0] != 1.0f || corr[1] != 1.0f);

      // ---- V unit: U = l~ P^T per 16-channel m-tile, folded into O
      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sV, (uV / kSt) & 1, a.wait_ns));
      if (failed) break;
      prep_ab(unitV, false);
      __syncwarp();
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float4 ab = lds<float4>(smem, s_ab + 16 * (8 * mt + g));   // (A, B) of 16 mt + g, + 8
        const uint32_t off = unitV + mt * 2048 + vofs;
        const uint32_t wa0 = lds<uint32_t>(smem, off);
        const uint32_t wa1 = lds<uint32_t>(smem, off + 1024);
        uint32_t e0 = 0, o0 = 0, e1 = 0, o1 = 0;
        if (FULL) {
          full_codes(wa0, lds<uint32_t>(smem, off + G::kResOff), e0, o0);
          full_codes(wa1, lds<uint32_t>(smem, off + 1024 + G::kResOff), e1, o1);
        }
        // (head pair, remainder pair) of byte j of row c0 (c = 0) or c0 + 8 (c = 1)
        auto vpair = [&](int c, uint32_t j) -> uint2 {
          const uint32_t sel = byte_sel(j);
          if (!FULL) return lds<uint2>(smem, S::kLutV + lut_off(c ? wa1 : wa0, lane8, sel));
          const uint32_t he = lds<uint32_t>(smem, S::kLutV + lut_off(c ? e1 : e0, lane4v, sel));
          const uint32_t ho = lds<uint32_t>(smem, S::kLutV + lut_off(c ? o1 : o0, lane4v, sel));
          return make_uint2(prmt(he, ho, 0x5410u), prmt(he, ho, 0x7632u));
        };
        float u[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const uint2 y00 = vpair(0, 2 * kv), y10 = vpair(1, 2 * kv);
          const uint2 y01 = vpair(0, 2 * kv + 1), y11 = vpair(1, 2 * kv + 1);
          mma_f16(u, y00.x, y10.x, y01.x, y11.x, pb[kv][0], pb[kv][1]);
          mma_f16(u, y00.y, y10.y, y01.y, y11.y, pb[kv][0], pb[kv][1]);
        }
        float2 q0 = O[mt][0], q1 = O[mt][1];
        if (rescale) {
          q0 = __fmul2_rn(q0, cr);
          q1 = __fmul2_rn(q1, cr);
        }
        q0 = __ffma2_rn(make_float2(ab.x, ab.x), pss, q0);
        q1 = __ffma2_rn(make_float2(ab.z, ab.z), pss, q1);
        O[mt][0] = __ffma2_rn(make_float2(ab.y, ab.y), make_float2(u[0], u[1]), q0);
        O[mt][1] = __ffma2_rn(make_float2(ab.w, ab.w), make_float2(u[2], u[3]), q1);
      }
      __syncwarp();
      if (L == 0) mbar_arrive(bar_empty + 8 * sV);
    }
    if (failed && L == 0) {
      atomicExch(a.status, 1);
      *s_flag = 1;
    }
  }

  // ================= merge the 8 chunk states (the ring is idle now)
  __syncthreads();
  allow_dependent_launch();   // the split combine may be scheduled once every CTA is here
  if (*reinterpret_cast<volatile int*>(s_flag) != 0) return;
  float* mm = reinterpret_cast<float*>(smem + S::kMergeM);
  float* ml = reinterpret_cast<float*>(smem + S::kMergeL);
  float* mo = reinterpret_cast<float*>(smem + S::kMergeO);
  if (warp < kConsumers) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if (g == 0) {   // every lane of equal t holds the rows' whole-chunk sums
        mm[warp * kNr + 2 * t + e] = m_run[e];
        ml[warp * kNr + 2 * t + e] = l_run[e];
      }
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int r = warp * kNr + 2 * t;
      const int c0 = 16 * mt + g;
      mo[r * kH + c0] = O[mt][0].x;
      mo[(r + 1) * kH + c0] = O[mt][0].y;
      mo[r * kH + c0 + 8] = O[mt][1].x;
      mo[(r + 1) * kH + c0 + 8] = O[mt][1].y;
    }
  }
  __syncthreads();
  for (int i = tid; i < kNr * kH; i += kThreadsQ) {
    const int r = i >> 7, d = i & 127;
    const int row = row0 + r;
    const int rg4 = row >> 2;
    if (rg4 >= a.n_rg) continue;
    float mstar = -CUDART_INF_F;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) mstar = fmaxf(mstar, mm[ww * kNr + r]);
    float o = 0.0f, l = 0.0f;
    if (mstar != -CUDART_INF_F) {
#pragma unroll
      for (int ww = 0; ww < kConsumers; ++ww) {
        const float mw = mm[ww * kNr + r];
        if (mw == -CUDART_INF_F) continue;
        const float f = exp2f(mw - mstar);
        o += mo[(ww * kNr + r) * kH + d] * f;
        l += ml[ww * kNr + r] * f;
      }
    }
    // the 2^10 scale of the probabilities cancels in o / l; remove it from both
    const int64_t cta = (((int64_t)b * a.Hkv + h) * a.n_rg + rg4) * a.n_splits + split;
    float* ws = a.ws + cta * kWsPerCta;
    ws[(row & 3) * kH + d] = o * (1.0f / 1024.0f);
    if (d == 0) {
      ws[kRows * kH + (row & 3)] = mstar;
      ws[kRows * kH + kRows + (row & 3)] = l * (1.0f / 1024.0f);
    }
  }
}

template <bool FULL, bool UNI>
cudaError_t launch_narrow(const DecodeArgs& a, const LutTables* lut, cudaStream_t s) {
  constexpr int kSmem = NLayout<FULL>::kAlloc;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(decode_narrow_kernel<FULL, UNI>,
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
  dim3 grid(a.n_splits, a.Hkv * ((a.T * a.G + kNr - 1) / kNr), a.B);
  return launch_programmatic(decode_narrow_kernel<FULL, UNI>, grid, dim3(kThreadsQ), kSmem, s, a, *lut, tka, tva, tkr,
                             tvr);
}

}  // namespace

cudaError_t launch_decode_narrow(const DecodeArgs& a, bool full, const LutTables* lut, cudaStream_t s) {
  if (a.uniform) return full ? launch_narrow<true, true>(a, lut, s) : launch_narrow<false, true>(a, lut, s);
  return full ? launch_narrow<true, false>(a, lut, s) : launch_narrow<false, false>(a, lut, s);
}

}  // namespace lynx
