// Draft decode attention over Lynx Anchor planes: the 1-token decode of the
// Lynx paper's §4.2 Anchor phase (attention of §2.1 over the Anchor-only KV),
// and any call over Anchor planes with at most 8 query rows per KV head
// (T x Hq/Hkv <= 8 per CTA, the n = 8 dimension of the mma.sync tiles).
//
// CTA: one producer lane streams the split's K and V page units through a
// 6-slot shared-memory ring (2-D TMA tile for the plane, bulk copy for the
// metadata); 8 consumer warps, warp w owning the 32-token chunk w of every
// page with its own online softmax, one merge of the 8 chunk states at the end.
//
// Dequantisation table.  Each of the 256 plane bytes maps to one 32-bit entry
// holding the Anchor values l~ of its two nibbles as 15-bit fixed point,
// u = v + 2^14 with v = rint(l~ F), F = 2^14 - 1 (|l~| <= 1, so 0 < u < 2^15),
// low nibble in bits 0..15.  32 copies, one per lane (conflict-free lookups,
// 4 bytes per byte of plane).
//
//   K side  S^T[32 tokens x 8 rows] = K Q^T as fp16 m16n8k16 (two m-tiles of
//           16 tokens, 8 k-steps of 16 channels).  With k = A + B l~
//           (A = gamma_min + (gamma_scale + eps) mu, B = (gamma_scale + eps)
//           (sigma + eps)) and l~ = (u - 2^14) / F, the chunk's scale is folded
//           into the queries: Q' = q B / F 2^-ek (ek puts |Q'| below 2^15),
//           split into an fp16 head and remainder, so that
//           S = alpha + 2^(ek + 32) sum_c Q'_c u_c 2^-32 with
//           alpha = sum_c q_c (A - B 2^14 / F).  The table's bytes of u enter
//           the MMAs as they are (fp16 subnormals u_hi 2^-24, u_lo 2^-24):
//           u_hi x Q'_head, u_hi x Q'_rem and u_lo x Q'_head 2^-8, three
//           products in three accumulators (~21-bit products).  Row g of m-tile mi holds token 4g + 2mi and
//           row g + 8 token 4g + 2mi + 1, the two tokens of one plane byte.
//   V side  T[128 channels x 8 rows] = sum over the chunk's tokens of
//           u 2^-32 p as fp16 m16n8k16: the two bytes of u are the fp16
//           subnormals u_hi 2^-24 and u_lo 2^-24 (one byte permute each; the
//           zero high byte is the replicated sign of the u_hi byte, which is
//           below 128), multiplied by P and by P 2^-8 into one accumulator.
//           With U = sum l~ p = (2^32 T - 2^14 sum p) / F, the output update
//           is O = O corr + (A - B 2^14 / F) psum + (B 2^32 / F) T.  Slot order
//           of k-step kv:
//           slots 2t, 2t+1 hold tokens 8t + 4kv + {0, 1}, slots 2t+8, 2t+9
//           hold 8t + 4kv + {2, 3}, so an A fragment register is one plane
//           byte's entry.
//
// Lane (g = L >> 2, t = L & 3) holds S of query rows 2t, 2t+1 for tokens
// 4g .. 4g+3 of its chunk, and O of channels 16 mt + g (+ 8) for the same two
// rows, so the per-row softmax statistics a lane needs for its output are its
// own.  The P^T fragments of the V side (row g, tokens 8t + 4kv + 0..3) come
// from lane 4 (2t + kv) + (g >> 1) by shuffles.
//
// Softmax.  A row's running maximum moves only when one of the
// chunk's scores exceeds it by more than 5 in log2 units (a probability factor
// of 2^5; a warp vote, then the rows take their maxima by shuffles), so most
// pages skip the max reduction and the rescale, and the probabilities (x 2^10)
// stay below 2^15, inside fp16.  The row sums of the fp16 probabilities the V
// side multiplies come from one more MMA pair (ones x P^T), so the normaliser
// sums exactly the probabilities the output used.
//
// Rounding: P is rounded to fp16 (relative 2^-11) and l~ to 1 / (2 F) absolute;
// products keep ~21 bits, sums are float32.

#include "decode_common.cuh"

namespace lynx {
namespace {

constexpr int kDRows = 8;                                 // query rows per CTA
constexpr int kDChunks = 8;                               // consumer warps: one per 32-token chunk
constexpr int kDThreads = (kDChunks + 1) * 32;            // + the producer warp: 288
constexpr int kDStages = 6;                               // ring slots
constexpr float kDLazyLog2 = 5.0f;                        // largest log2 lead of a score over the running maximum
constexpr uint32_t kDOnes2 = 0x3C003C00u;                 // fp16 pair (1, 1)
constexpr uint32_t kDP8 = 0x1C001C00u;                    // fp16 pair (2^-8, 2^-8)
constexpr float kDFix = 16383.0f;                         // F: table values v = rint(l~ F), |v| < 2^14
constexpr float kDVsum = 16384.0f / 16383.0f;             // 2^14 / F
constexpr float kDVt = 4294967296.0f / 16383.0f;          // 2^32 / F
constexpr uint32_t kDSelHi = 0xB391u;                     // fp16 pair (u0_hi 2^-24, u1_hi 2^-24)
constexpr uint32_t kDSelLo = 0xB290u;                     // fp16 pair (u0_lo 2^-24, u1_lo 2^-24)
// K side, two entries (channels c, c + 1): fp16 pair (u_hi or u_lo of c, of c + 1)
// for the even (u0) or the odd (u1) token; the zero high bytes replicate the
// sign of a u_hi byte (below 128)
constexpr uint32_t kDSelKEvenHi = 0xD591u;
constexpr uint32_t kDSelKOddHi = 0xF7B3u;
constexpr uint32_t kDSelKEvenLo = 0xD490u;
constexpr uint32_t kDSelKOddLo = 0xF6B2u;

struct DLayout {
  using G = QGeo<false, kDStages>;
  static constexpr int kRing = 0;
  static constexpr int kLut = kRing + kDStages * G::kUnit;           // [byte][256 B]: lane L's copy at 4L
  // per warp: float2 per channel of the current unit, (A', B') for a key unit,
  // (A - B 2^14/F, B 2^32/F) for a value unit
  static constexpr int kAb = kLut + 256 * 256;
  static constexpr int kQ = kAb + kDChunks * kH * 8;                  // Q BF16 pairs [64 channel pairs][8 rows]
  static constexpr int kQmax = kQ + 64 * kDRows * 4;                  // u32: largest |q| (BF16 bits)
  static constexpr int kFlag = kQmax + 16;
  static constexpr int kBar = kFlag + 16;                             // ring full[kDStages], empty[kDStages]
  static constexpr int kTotal = kBar + 2 * kDStages * 8;
  static constexpr int kAlloc = kTotal + 1024;
  // end-of-kernel merge area (reuses the ring): o[8][8][kMergeStride] (each
  // chunk's output rows, already scaled by the chunk's factor 2^(m_w - m*); the
  // padded row stride keeps a warp's stores on 32 banks), then m[8][8],
  // l[8][8], the factors f[8][8] and the rows' (m*, l*) pairs
  static constexpr int kMergeStride = kH + 4;
  static constexpr int kMergeO = 0;
  static constexpr int kMergeM = kMergeO + kDChunks * kDRows * kMergeStride * 4;
  static constexpr int kMergeL = kMergeM + kDChunks * kDRows * 4;
  static constexpr int kMergeF = kMergeL + kDChunks * kDRows * 4;
  static constexpr int kMergeS = kMergeF + kDChunks * kDRows * 4;
  static_assert(kMergeS + kDRows * 8 <= kDStages * G::kUnit, "merge area");
  static_assert(kLut % 1024 == 0, "ring slots keep the 1024-byte alignment of swizzled tiles");
};
static_assert(DLayout::kAlloc <= 232448, "shared memory (draft decode)");

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  __half2 x = *reinterpret_cast<const __half2*>(&a);
  const __half2 y = *reinterpret_cast<const __half2*>(&b);
  x = __hmul2(x, y);
  return *reinterpret_cast<const uint32_t*>(&x);
}

__global__ void __launch_bounds__(kDThreads, 1)
decode_draft_kernel(const DecodeArgs a, const LutTables lut, const __grid_constant__ CUtensorMap tm_ka,
                    const __grid_constant__ CUtensorMap tm_va) {
  using G = QGeo<false, kDStages>;
  using S = DLayout;
  constexpr int kSt = kDStages;
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
  const int n_tiles = (TG + kDRows - 1) / kDRows;
  const int h = blockIdx.y / n_tiles;
  const int row0 = (blockIdx.y % n_tiles) * kDRows;
  const int b = blockIdx.z;
  const int max_keys = a.max_pages * kP;

  const uint32_t s_ring = base + S::kRing;
  const uint32_t bar_full = base + S::kBar;
  const uint32_t bar_empty = bar_full + 8 * kSt;
  int* s_flag = reinterpret_cast<int*>(smem + S::kFlag);
  uint32_t* s_q = reinterpret_cast<uint32_t*>(smem + S::kQ);
  uint32_t* s_qmax = reinterpret_cast<uint32_t*>(smem + S::kQmax);

  // ---- prologue: barriers first; the producer lane starts streaming pages
  // while the consumer warps fill the value table and the queries
  if (tid == 0) {
    for (int st = 0; st < kSt; ++st) {
      mbar_init(bar_full + 8 * st, 1);
      mbar_init(bar_empty + 8 * st, kDChunks);
    }
    *s_flag = 0;
    *s_qmax = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // value table (kernel parameters only), before the wait on the kernel ahead
  // in the stream: with a programmatic launch this overlaps that kernel's tail.
  // Thread e makes entry e and stores its 32 copies, the copy index rotated by
  // the lane so that a warp's stores hit different banks.
  if (tid < 256) {
    // entry e = (value of nibble e & 15, value of nibble e >> 4): lane L reads
    // nibble L & 15's value once (16 parameter addresses per warp instead of 32)
    // and the two values come by shuffles
    const float n16 = lut.anc16[L & 15];
    const float2 v = make_float2(__shfl_sync(0xffffffffu, n16, tid & 15), __shfl_sync(0xffffffffu, n16, (tid >> 4) & 15));
    const int v0 = min(max(__float2int_rn(v.x * kDFix), -16383), 16383);
    const int v1 = min(max(__float2int_rn(v.y * kDFix), -16383), 16383);
    const uint32_t ent = (uint32_t)(v0 + 16384) | ((uint32_t)(v1 + 16384) << 16);
#pragma unroll 8
    for (int k = 0; k < 32; ++k)
      *reinterpret_cast<uint32_t*>(smem + S::kLut + tid * 256 + 4 * ((L + k) & 31)) = ent;
  }
  // every global-memory access of this kernel follows this wait
  wait_prerequisite_grids();
  // the producer lane reads its first page id together with the context length
  int first_id = 0;
  if (tid == kDChunks * 32) {
    const int pb = split * a.pages_per_split;
    if (pb < a.max_pages) first_id = a.page_table[((int64_t)b * a.Hkv + h) * a.max_pages + pb];
  }
  // the query vector of thread i < 128 (row i >> 4, channels 8 (i & 15) .. + 7;
  // zeros for padding rows), requested before the context length is read
  uint4 qx = make_uint4(0u, 0u, 0u, 0u);
  if (tid < kDRows * 16) {
    const int row = row0 + (tid >> 4);
    if (row < TG) {
      const uint16_t* qr = a.q + (((int64_t)b * a.T + row / a.G) * a.Hq + h * a.G + row % a.G) * kH;
      qx = __ldg(reinterpret_cast<const uint4*>(qr) + (tid & 15));
    }
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
  const int max_vis = n_visible(min(kDRows, TG - row0) - 1);
  const int min_vis = n_visible(0);
  const int n_pages = (max_vis + kP - 1) / kP;
  const int p_begin = split * a.pages_per_split;
  const int np = max(min(p_begin + a.pages_per_split, n_pages) - p_begin, 0);
  const int32_t* pt_row = a.page_table + ((int64_t)b * a.Hkv + h) * a.max_pages;
  const float eps = a.eps;

  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};   // query rows 2t, 2t + 1
  float l_run[2] = {0.0f, 0.0f};
  // O[mt] = (channel 16 mt + g, rows 2t, 2t+1), (channel 16 mt + g + 8, rows 2t, 2t+1)
  float2 O[8][2];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) O[mt][0] = O[mt][1] = make_float2(0.f, 0.f);
  bool failed = false;

  if (warp == kDChunks) {
    if (L == 0)
      produce_units<false, kDStages>(a, pt_row, p_begin, np, first_id, s_ring, bar_full, bar_empty, &tm_ka, &tm_va, &tm_ka,
                                     &tm_va, s_flag);
  } else {
    const int w = warp;
    // the query rows as BF16 pairs (the consumer warps meet at named barrier 1):
    // word (pair p, row r) = channels 2p, 2p + 1 of query row r of this CTA (0
    // for padding rows), from the vectors qx loaded above; the CTA's largest |q|
    // sets the fp16 scaling of Q'
    {
      uint32_t qm = 0u;
      if (tid < kDRows * 16) {
        const int r = tid >> 4, v = tid & 15;
        const uint32_t w4[4] = {qx.x, qx.y, qx.z, qx.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s_q[(4 * v + j) * kDRows + r] = w4[j];
          qm = max(qm, max(w4[j] & 0x7FFFu, (w4[j] >> 16) & 0x7FFFu));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) qm = max(qm, __shfl_xor_sync(0xffffffffu, qm, o));
      if (L == 0) atomicMax(s_qmax, qm);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDChunks * 32) : "memory");
    // exponent of the largest |q| (BF16 bits -> power of two above it)
    const int eq = (int)((*s_qmax >> 7) & 0xFFu) - 127 + 1;

    const uint32_t s_ab = S::kAb + w * kH * 8;
    const uint32_t lane4 = 4u * L;
    // K side: bytes 2 (g & 1) (m-tile 0) and 2 (g & 1) + 1 (m-tile 1) of word g >> 1 of a channel row
    const uint32_t ksel0 = byte_sel(2 * (g & 1)), ksel1 = byte_sel(2 * (g & 1) + 1);
    const uint32_t kword = 4 * (g >> 1);
    // V side: bytes 4t..4t+3 of channel 16 mt + g, word t of its chunk unit
    const uint32_t vofs = g * 128 + ((w ^ g) << 4) + 4 * t;
    // source lanes of the P^T fragments of V k-steps 0 and 1
    const int src0 = 4 * (2 * t) + (g >> 1), src1 = src0 + 4;
    const bool odd_row = (g & 1) != 0;
    const int nv[2] = {n_visible(2 * t), n_visible(2 * t + 1)};   // the lane's query rows
    const float sc = a.scale_log2;

    for (int i = 0; i < np && !failed; ++i) {
      const int p = p_begin + i;
      const int uK = 2 * i, uV = 2 * i + 1;
      const int sK = uK % kSt, sV = uV % kSt;
      const uint32_t unitK = S::kRing + sK * G::kUnit;
      const uint32_t unitV = S::kRing + sV * G::kUnit;
      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sK, (uK / kSt) & 1, a.wait_ns));
      if (failed) break;
      // (A', B') of the 128 channels in channel order: A' = A - B 2^14 / F and
      // B' = (B / F) 2^-ek, ek chosen so that |q| B' < 2^15 for every query value
      int ek;
      {
        const uint32_t mt = unitK + G::kMetaOff;
        float A[4], Bf[4], bmax = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int d = L + 32 * k;
          const float gmin = lds<float>(smem, mt + 4 * d);
          const float dg = __fadd_rn(lds<float>(smem, mt + 4 * (kH + d)), eps);
          const float mu = lds<float>(smem, mt + 4 * (kMetaMuOff + w * kH + d));
          const float ds = __fadd_rn(lds<float>(smem, mt + 4 * (kMetaSigmaOff + w * kH + d)), eps);
          const float B = __fmul_rn(dg, ds);
          A[k] = __fmaf_rn(-B, kDVsum, __fmaf_rn(dg, mu, gmin));
          Bf[k] = __fmul_rn(B, 1.0f / kDFix);
          bmax = fmaxf(bmax, fabsf(Bf[k]));
        }
        bmax = warp_max_nonneg(bmax);
        // |q| < 2^eq and |B'| < 2^eb, so |q B' 2^-ek| < 2^15 with ek = eq + eb - 15
        const int eb = (int)((__float_as_uint(bmax) >> 23) & 0xFFu) - 127 + 1;
        ek = min(max(eq + eb - 15, -100), 100);
        const float f = __uint_as_float((uint32_t)(127 - ek) << 23);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<float2*>(smem + s_ab + 8 * (L + 32 * k)) = make_float2(A[k], Bf[k] * f);
      }
      __syncwarp();

      // ---- S^T = K Q^T as fp16 m16n8k16 over 8 k-steps of 16 channels:
      // T = sum_c Q'_c u_c 2^-32 with u = 256 u_hi + u_lo the table value of
      // the code, from the products u_hi 2^-24 x (Q'h + Q'l) and
      // u_lo 2^-24 x Q'h 2^-8; then S = alpha + 2^(ek + 32) T with
      // alpha = sum_c q_c A'_c.  k-slots 2t, 2t+1 / 2t+8, 2t+9 are channels
      // 16 ks + 2t, + 1 / + 8, + 9; row g of m-tile mi is token 4g + 2mi, row
      // g + 8 token 4g + 2mi + 1.
      // [m-tile][(token even, row 2t), (even, 2t+1), (odd, 2t), (odd, 2t+1)]; the
      // three products of a k-step go to three accumulators (shorter MMA
      // dependency chains), summed after the last k-step
      float sacc[2][4], sacc2[2][4], sacc3[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mi][e] = sacc2[mi][e] = sacc3[mi][e] = 0.0f;
      float2 alpha2 = make_float2(0.0f, 0.0f);
      // the plane words of all 8 k-steps first: channels 16 ks + 2t + {0, 1, 8, 9}
      uint32_t kw[8][4];
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int ch = 16 * ks + 2 * t + (c & 1) + 8 * (c >> 1);
          kw[ks][c] = lds<uint32_t>(smem, unitK + ch * 128 + ((w ^ (ch & 7)) << 4) + kword);
        }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        // B fragments: Q' of query row g for channels 16 ks + 2t + {0, 1} (b0) and + {8, 9} (b1)
        const uint32_t qa = s_q[(8 * ks + t) * kDRows + g];
        const uint32_t qb = s_q[(8 * ks + t + 4) * kDRows + g];
        const float4 ab0 = lds<float4>(smem, s_ab + 8 * (16 * ks + 2 * t));
        const float4 ab1 = lds<float4>(smem, s_ab + 8 * (16 * ks + 2 * t + 8));
        const float2 q0 = make_float2(__uint_as_float(qa << 16), __uint_as_float(qa & 0xFFFF0000u));
        const float2 q1 = make_float2(__uint_as_float(qb << 16), __uint_as_float(qb & 0xFFFF0000u));
        alpha2 = __ffma2_rn(q0, make_float2(ab0.x, ab0.z), alpha2);
        alpha2 = __ffma2_rn(q1, make_float2(ab1.x, ab1.z), alpha2);
        const float2 qp0 = __fmul2_rn(q0, make_float2(ab0.y, ab0.w));
        const float2 qp1 = __fmul2_rn(q1, make_float2(ab1.y, ab1.w));
        const __half2 hh0 = __floats2half2_rn(qp0.x, qp0.y), hh1 = __floats2half2_rn(qp1.x, qp1.y);
        const float2 f0 = __half22float2(hh0), f1 = __half22float2(hh1);
        const float2 r0 = __ffma2_rn(f0, make_float2(-1.0f, -1.0f), qp0);
        const float2 r1 = __ffma2_rn(f1, make_float2(-1.0f, -1.0f), qp1);
        const uint32_t bh0 = *reinterpret_cast<const uint32_t*>(&hh0), bh1 = *reinterpret_cast<const uint32_t*>(&hh1);
        const uint32_t bl0 = h2(r0.x, r0.y), bl1 = h2(r1.x, r1.y);
        const uint32_t bs0 = hmul2_bits(bh0, kDP8), bs1 = hmul2_bits(bh1, kDP8);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          const uint32_t sel = mi ? ksel1 : ksel0;
          uint32_t e[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) e[c] = lds<uint32_t>(smem, S::kLut + lut_off(kw[ks][c], lane4, sel));
          // a0 / a1: the even / odd token of channels (c0, c0 + 1); a2 / a3: of (c0 + 8, c0 + 9)
          const uint32_t h0 = prmt(e[0], e[1], kDSelKEvenHi), h1 = prmt(e[0], e[1], kDSelKOddHi);
          const uint32_t h2_ = prmt(e[2], e[3], kDSelKEvenHi), h3 = prmt(e[2], e[3], kDSelKOddHi);
          const uint32_t l0 = prmt(e[0], e[1], kDSelKEvenLo), l1 = prmt(e[0], e[1], kDSelKOddLo);
          const uint32_t l2 = prmt(e[2], e[3], kDSelKEvenLo), l3 = prmt(e[2], e[3], kDSelKOddLo);
          mma_f16(sacc[mi], h0, h1, h2_, h3, bh0, bh1);
          mma_f16(sacc2[mi], h0, h1, h2_, h3, bl0, bl1);
          mma_f16(sacc3[mi], l0, l1, l2, l3, bs0, bs1);
        }
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mi][e] += sacc2[mi][e] + sacc3[mi][e];
      __syncwarp();
      if (L == 0) mbar_arrive(bar_empty + 8 * sK);
      // alpha of query row g: the four lanes of equal g hold its channels; the
      // lane's S rows are 2t and 2t + 1, whose alphas sit in lanes 4 (2t) and 4 (2t + 1)
      float alpha = alpha2.x + alpha2.y;
      alpha += __shfl_xor_sync(0xffffffffu, alpha, 1);
      alpha += __shfl_xor_sync(0xffffffffu, alpha, 2);
      const float al0 = __shfl_sync(0xffffffffu, alpha, 8 * t) * sc;
      const float al1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4) * sc;
      const float tsc = sc * __uint_as_float((uint32_t)min(max(127 + ek + 32, 1), 254) << 23);

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
          float sv = __fmaf_rn(sacc[j >> 1][2 * (j & 1) + e], tsc, e ? al1 : al0);
          if (!all_visible && pos0 + j >= nv[e]) sv = -CUDART_INF_F;
          pr[e][j] = sv;
          mloc[e] = fmaxf(mloc[e], sv);
        }
      }
      // the running maximum moves only when a score of the chunk exceeds it by
      // more than kDLazyLog2 (then every row of the warp takes its row maximum);
      // otherwise the probabilities stay below 2^(10 + kDLazyLog2), inside fp16
      const bool grow =
          __any_sync(0xffffffffu, mloc[0] > m_run[0] + kDLazyLog2 || mloc[1] > m_run[1] + kDLazyLog2);
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
      uint32_t pb[2][2], pl[2][2];   // P, and P 2^-8 (the multiplier of the low bytes)
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const int src = kv ? src1 : src0;
        const uint32_t y00 = __shfl_sync(0xffffffffu, x00, src), y01 = __shfl_sync(0xffffffffu, x01, src);
        const uint32_t y10 = __shfl_sync(0xffffffffu, x10, src), y11 = __shfl_sync(0xffffffffu, x11, src);
        pb[kv][0] = odd_row ? y10 : y00;
        pb[kv][1] = odd_row ? y11 : y01;
        pl[kv][0] = hmul2_bits(pb[kv][0], kDP8);
        pl[kv][1] = hmul2_bits(pb[kv][1], kDP8);
      }
      // the chunk's row sums of the fp16 probabilities, from a 16 x 32 matrix of
      // ones times P^T (every accumulator row holds them; the lane's entries 0
      // and 1 are its rows 2t and 2t + 1)
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
      mma_f16(ps4, kDOnes2, kDOnes2, kDOnes2, kDOnes2, pb[0][0], pb[0][1]);
      mma_f16(ps4, kDOnes2, kDOnes2, kDOnes2, kDOnes2, pb[1][0], pb[1][1]);
      const float2 pss = make_float2(ps4[0], ps4[1]);
      const float2 cr = make_float2(corr[0], corr[1]);
      l_run[0] = l_run[0] * cr.x + pss.x;
      l_run[1] = l_run[1] * cr.y + pss.y;
      const bool rescale = __any_sync(0xffffffffu, cr.x != 1.0f || cr.y != 1.0f);

      // ---- V unit: T = u 2^-32 P^T per 16-channel m-tile, folded into O
      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sV, (uV / kSt) & 1, a.wait_ns));
      if (failed) break;
      // (A - B 2^14/F, B 2^32/F) of the 128 channels, channels c and c + 8
      // (c & 8 == 0) side by side: slot 16 (c >> 4) + 2 (c & 7) + ((c >> 3) & 1)
      {
        const uint32_t mt = unitV + G::kMetaOff;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int d = L + 32 * k;
          const float gmin = lds<float>(smem, mt + 4 * d);
          const float dg = __fadd_rn(lds<float>(smem, mt + 4 * (kH + d)), eps);
          const float mu = lds<float>(smem, mt + 4 * (kMetaMuOff + w * kH + d));
          const float ds = __fadd_rn(lds<float>(smem, mt + 4 * (kMetaSigmaOff + w * kH + d)), eps);
          const float A = __fmaf_rn(dg, mu, gmin), B = __fmul_rn(dg, ds);
          const int slot = 16 * (d >> 4) + 2 * (d & 7) + ((d >> 3) & 1);
          *reinterpret_cast<float2*>(smem + s_ab + 8 * slot) = make_float2(__fmaf_rn(-B, kDVsum, A), __fmul_rn(B, kDVt));
        }
      }
      __syncwarp();
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float4 ab = lds<float4>(smem, s_ab + 16 * (8 * mt + g));   // of 16 mt + g and + 8
        const uint32_t off = unitV + mt * 2048 + vofs;
        const uint32_t wa0 = lds<uint32_t>(smem, off);
        const uint32_t wa1 = lds<uint32_t>(smem, off + 1024);
        float u[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const uint32_t e00 = lds<uint32_t>(smem, S::kLut + lut_off(wa0, lane4, byte_sel(2 * kv)));
          const uint32_t e10 = lds<uint32_t>(smem, S::kLut + lut_off(wa1, lane4, byte_sel(2 * kv)));
          const uint32_t e01 = lds<uint32_t>(smem, S::kLut + lut_off(wa0, lane4, byte_sel(2 * kv + 1)));
          const uint32_t e11 = lds<uint32_t>(smem, S::kLut + lut_off(wa1, lane4, byte_sel(2 * kv + 1)));
          const uint32_t h0 = prmt(e00, e00, kDSelHi), h1 = prmt(e10, e10, kDSelHi);
          const uint32_t h2_ = prmt(e01, e01, kDSelHi), h3 = prmt(e11, e11, kDSelHi);
          const uint32_t l0 = prmt(e00, e00, kDSelLo), l1 = prmt(e10, e10, kDSelLo);
          const uint32_t l2 = prmt(e01, e01, kDSelLo), l3 = prmt(e11, e11, kDSelLo);
          mma_f16(u, h0, h1, h2_, h3, pb[kv][0], pb[kv][1]);
          mma_f16(u, l0, l1, l2, l3, pl[kv][0], pl[kv][1]);
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
  float* mo = reinterpret_cast<float*>(smem + S::kMergeO);
  float* mm = reinterpret_cast<float*>(smem + S::kMergeM);
  float* ml = reinterpret_cast<float*>(smem + S::kMergeL);
  float* mf = reinterpret_cast<float*>(smem + S::kMergeF);
  float2* mrow = reinterpret_cast<float2*>(smem + S::kMergeS);
  constexpr int MS = S::kMergeStride;
  if (warp < kDChunks && g == 0) {   // every lane of equal t holds the rows' maxima and whole-chunk sums
    mm[warp * kDRows + 2 * t] = m_run[0];
    mm[warp * kDRows + 2 * t + 1] = m_run[1];
    ml[warp * kDRows + 2 * t] = l_run[0];
    ml[warp * kDRows + 2 * t + 1] = l_run[1];
  }
  __syncthreads();
  // chunk w's factor of row r, 2^(m_w - m*) (0 where the chunk saw no key of the row)
  if (tid < kDChunks * kDRows) {
    const int r = tid % kDRows;
    float mstar = -CUDART_INF_F;
#pragma unroll
    for (int ww = 0; ww < kDChunks; ++ww) mstar = fmaxf(mstar, mm[ww * kDRows + r]);
    const float mw = mm[tid];
    mf[tid] = (mw == -CUDART_INF_F) ? 0.0f : exp2f(mw - mstar);
  }
  __syncthreads();
  // each row's (m*, l*); each lane's O values, scaled by its chunk's factors,
  // into the chunk's rows of the merge area
  if (tid < kDRows) {
    float mstar = -CUDART_INF_F, l = 0.0f;
#pragma unroll
    for (int ww = 0; ww < kDChunks; ++ww) {
      mstar = fmaxf(mstar, mm[ww * kDRows + tid]);
      l += ml[ww * kDRows + tid] * mf[ww * kDRows + tid];
    }
    mrow[tid] = make_float2(mstar, l);
  }
  if (warp < kDChunks) {
    const float f0 = mf[warp * kDRows + 2 * t], f1 = mf[warp * kDRows + 2 * t + 1];
    float* dst = mo + (warp * kDRows + 2 * t) * MS;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int c0 = 16 * mt + g;
      dst[c0] = O[mt][0].x * f0;
      dst[MS + c0] = O[mt][0].y * f1;
      dst[c0 + 8] = O[mt][1].x * f0;
      dst[MS + c0 + 8] = O[mt][1].y * f1;
    }
  }
  __syncthreads();
  for (int i = tid; i < kDRows * kH; i += kDThreads) {
    const int r = i >> 7, d = i & 127;
    const int row = row0 + r;
    const int rg4 = row >> 2;
    if (rg4 >= a.n_rg) continue;
    float o = 0.0f;
#pragma unroll
    for (int ww = 0; ww < kDChunks; ++ww) o += mo[(ww * kDRows + r) * MS + d];
    const float2 st = mrow[r];
    // the 2^10 scale of the probabilities cancels in o / l; remove it from both
    const int64_t cta = (((int64_t)b * a.Hkv + h) * a.n_rg + rg4) * a.n_splits + split;
    float* ws = a.ws + cta * kWsPerCta;
    ws[(row & 3) * kH + d] = o * (1.0f / 1024.0f);
    if (d == 0) {
      ws[kRows * kH + (row & 3)] = st.x;
      ws[kRows * kH + kRows + (row & 3)] = st.y * (1.0f / 1024.0f);
    }
  }
}

}  // namespace

cudaError_t launch_decode_draft(const DecodeArgs& a, const LutTables* lut, cudaStream_t s) {
  constexpr int kSmem = DLayout::kAlloc;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(decode_draft_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  CUtensorMap tka, tva;
  if (n_pool_too_large(a.n_pool)) return cudaErrorInvalidValue;
  if (!plane_map(&tka, a.k_anc, a.n_pool) || !plane_map(&tva, a.v_anc, a.n_pool)) return cudaErrorInvalidValue;
  dim3 grid(a.n_splits, a.Hkv * ((a.T * a.G + kDRows - 1) / kDRows), a.B);
  return launch_programmatic(decode_draft_kernel, grid, dim3(kDThreads), kSmem, s, a, *lut, tka, tva);
}

}  // namespace lynx
