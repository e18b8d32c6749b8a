// Tensor-core verification attention over Lynx-encoded pages: the attention
// of the Lynx paper (§2.1) run on the KV that the Anchor phase (draft) or the
// Anchor and Residual phases (verification) of §4.2-4.3 deliver, for R = 16
// or R = 32 of the query rows that share one KV head (T tokens x
// Hq/Hkv heads) per CTA.  A 32-row CTA dequantises each key once for 32 rows.
//
// CTA skeleton as in the narrow kernel: a producer lane streams the split's
// K and V page units through a 3-slot shared-memory ring (2-D TMA tile for the
// planes, bulk copy for the metadata); 8 consumer warps, warp w owning the
// 32-token chunk w of every page with its own online softmax; one merge of the
// 8 chunk states at the end.
//
// Each chunk's two contractions run on the tensor cores (mma.sync, float32
// accumulation); the rows sharing one KV head make both a dense contraction.
//
//   K side   S[R rows x 32 tokens] = Q K^T as fp16 m16n8k16 over 8 k-steps of
//            16 channels.  k = A + B l~ is dequantised in float32
//            (A = gamma_min + (gamma_scale + eps) mu,
//            B = (gamma_scale + eps)(sigma + eps), the chunk's affine
//            constants) and split into an fp16 head (the float truncated to 11
//            significant bits) and the fp16-rounded remainder, two MMAs, so each
//            product keeps ~22 bits.  Q (BF16) is exact in fp16.  Both operands
//            are scaled by powers of two to fill fp16's range -- Q by the CTA
//            (largest |q| in [2^14, 2^15)), A and B by the chunk (largest
//            |A| + |B| in [2^14, 2^15)) -- and the scale returns, exactly, in
//            the softmax scale.  Four
//            n-tiles per chunk: column n of n-tile k holds token 4n + k, so
//            lane (g, t) needs bytes 2g and 2g+1 of a channel row, both in one
//            32-bit plane word; its k-slots 2t, 2t+1 and 2t+8, 2t+9 are
//            channels 16 ks + 2t, + 1, + 8, + 9.
//   V side   U[128 channels x R rows] = l~ P^T as fp16 m16n8k16, two k-steps
//            of 16 tokens, then folded into the output with the chunk's
//            constants: O = O corr + A psum + B U.  l~ comes from a table of
//            fp16 head/remainder pairs (two MMAs, ~22 bits); P is fp16, scaled
//            by 2^10 away from fp16 subnormals (O and the row sums carry the
//            2^10, removed once at the end).  The row sums that normalise the
//            output and weight A are those of the same fp16 probabilities (a
//            matrix of ones times P^T), so a dominant key's rounding cancels.
//            Slot order of k-step kv: slots
//            2t, 2t+1 hold tokens 8t + 4kv + {0, 1}, slots 2t+8, 2t+9 hold
//            8t + 4kv + {2, 3}.  With that order the A fragments are packed
//            bytes as stored (both tokens of a byte in one register; bytes
//            4t..4t+3 of a channel row, one plane word, serve both k-steps)
//            and the P fragments are S accumulator entries the lane holds
//            already.
//
// Lane (g = L >> 2, t = L & 3) holds S of rows 8 rh + g (rh = 0 .. R/8 - 1; K
// m-tile rh >> 1, accumulator half rh & 1) for tokens 8t + j (j = 4hh + k:
// entry hh of n-tile k) of its chunk.
//
// Output accumulators.  With R = 16 each consumer warp keeps its chunk's
// O[16 rows x 128 channels] in registers.  With R = 32 they live in tensor
// memory (TMEM): warp w owns 128 columns of the 32 TMEM lanes of quadrant
// w mod 4 (columns 128 (w / 4) ..), lane L one row of them; the 16 values of
// channel tile mt are read (tcgen05.ld), updated and written back
// (tcgen05.st) per page.  Warp 0 allocates the 256 columns and frees them on
// every exit path.
//
// Rounding: P is rounded to fp16 (relative 2^-11); everything else keeps at
// least ~21 bits, sums are float32.

#include "decode_common.cuh"

namespace lynx {
namespace {

constexpr int kTcWarpBytes = kH * 8;   // per warp: float2 (A, B) per channel of the current unit
constexpr int kTmemCols = 256;         // R = 32: 8 warps x 128 columns, 2 warps per lane quadrant

template <bool FULL, int R>
struct TLayout {
  using G = QGeo<FULL>;
  static constexpr int kRing = 0;
  // Tables, 32 copies (one per lane) in rows of 256 B, row = byte or code.
  //   anchor  kLutK: byte -> (l~ low nibble, l~ high nibble) float2, copy at 8L
  //           kLutV: byte -> fp16 pairs (heads, remainders), copy at 8L
  //   full    kLutK: code -> l~ float, copy at 4L; fp16 (head, remainder) at 128 + 4L
  static constexpr int kLutK = kRing + G::kStages * G::kUnit;
  static constexpr int kLutV = FULL ? kLutK : kLutK + 256 * 256;
  static constexpr int kWarps = kLutV + 256 * 256;
  static constexpr int kQ = kWarps + kConsumers * kTcWarpBytes;   // uint4 [R/16][8 k-steps][32 lanes]
  static constexpr int kTmemSlot = kQ + (R / 16) * 8 * 32 * 16;    // u32: TMEM base (R = 32)
  static constexpr int kQmax = kTmemSlot + 4;                       // u32: largest |q| (BF16 bits)
  static constexpr int kFlag = kTmemSlot + 16;
  static constexpr int kBar = kFlag + 16;
  static constexpr int kTotal = kBar + 2 * G::kStages * 8;
  static constexpr int kAlloc = kTotal + 1024;
  // end-of-kernel merge area (reuses the ring and the tables, idle by then):
  // o[8][R][kMergeStride] (each chunk's output rows, already scaled by the
  // chunk's factor 2^(m_w - m*); the padded row stride keeps a warp's stores
  // on 32 banks), then m[8][R], l[8][R], the factors f[8][R] and the rows'
  // (m*, l*) pairs
  static constexpr int kMergeStride = kH + 4;
  static constexpr int kMergeO = 0;
  static constexpr int kMergeM = kMergeO + kConsumers * R * kMergeStride * 4;
  static constexpr int kMergeL = kMergeM + kConsumers * R * 4;
  static constexpr int kMergeF = kMergeL + kConsumers * R * 4;
  static constexpr int kMergeS = kMergeF + kConsumers * R * 4;
  static_assert(kMergeS + R * 8 <= kWarps, "merge area");
};
static_assert(TLayout<false, 16>::kAlloc <= 232448, "shared memory (anchor, tensor core)");
static_assert(TLayout<true, 16>::kAlloc <= 232448, "shared memory (full, tensor core)");
static_assert(TLayout<true, 32>::kAlloc <= 232448, "shared memory (full, tensor core, 32 rows)");
static_assert(TLayout<false, 32>::kAlloc <= 232448, "shared memory (anchor, tensor core, 32 rows)");

// ---- tensor memory (cta_group::1).  Column allocation by one whole warp; the
// allocated base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 16 consecutive 32-bit columns of the lane's TMEM row (shape 32x32b: lane i of
// the warp reads TMEM lane base + i)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
// the loaded registers are valid only after the wait: they are passed through
// it so that no use of them is scheduled before it
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                 "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                 "+r"(v[15])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

constexpr uint32_t kOnes2 = 0x3C003C00u;   // fp16 pair (1, 1)

// UNI: uniform-code metadata (min, scale per channel row) instead of Lynx's
template <bool FULL, int R, bool UNI>
__global__ void __launch_bounds__(kThreadsQ, 1)
decode_tc_kernel(const DecodeArgs a, const LutTables lut,
                 const __grid_constant__ CUtensorMap tm_ka, const __grid_constant__ CUtensorMap tm_va,
                 const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_vr) {
  static_assert(R == 16 || R == 32, "16 or 32 query rows per CTA");
  constexpr bool kTmem = (R == 32);
  constexpr int MT = R / 16;   // K side m-tiles (16 rows each)
  constexpr int NR = R / 8;    // row octets: V side n-tiles, S accumulator halves
  using G = QGeo<FULL>;
  using S = TLayout<FULL, R>;
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
  const int n_tiles = (TG + R - 1) / R;
  const int h = blockIdx.y / n_tiles;
  const int row0 = (blockIdx.y % n_tiles) * R;
  const int b = blockIdx.z;
  const int max_keys = a.max_pages * kP;

  const uint32_t s_ring = base + S::kRing;
  const uint32_t bar_full = base + S::kBar;
  const uint32_t bar_empty = bar_full + 8 * kSt;
  int* s_flag = reinterpret_cast<int*>(smem + S::kFlag);

  // ---- prologue: barriers and TMEM first; the producer lane starts streaming
  // pages while the consumer warps fill the value tables and the Q fragments
  uint32_t* s_qmax = reinterpret_cast<uint32_t*>(smem + S::kQmax);
  if (tid == 0) {
    for (int st = 0; st < kSt; ++st) {
      mbar_init(bar_full + 8 * st, 1);
      mbar_init(bar_empty + 8 * st, kConsumers);
    }
    *s_flag = 0;
    *s_qmax = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (kTmem && warp == 0) {
    tmem_alloc(base + S::kTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  if (kTmem) tmem_fence_before_sync();
  __syncthreads();
  if (kTmem) tmem_fence_after_sync();
  uint32_t tmem = 0u;
  if (kTmem) tmem = *reinterpret_cast<volatile uint32_t*>(smem + S::kTmemSlot);
  // this warp's 128 columns of its lane quadrant
  const uint32_t t_warp = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 128u * (uint32_t)(warp >> 2);
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
  // the consumer threads' query vectors, issued before the context length is
  // read: vector i = (row i >> 4, channels 8 (i & 15) .. + 7), zeros for padding rows
  constexpr int kQPer = R * 16 / kConsumerThreads;   // vectors per consumer thread
  uint4 qv[kQPer];
#pragma unroll
  for (int k = 0; k < kQPer; ++k) {
    const int i = tid + k * kConsumerThreads;
    const int row = row0 + (i >> 4);
    qv[k] = make_uint4(0u, 0u, 0u, 0u);
    if (warp < kConsumers && row < TG) {
      const uint16_t* qr = a.q + (((int64_t)b * a.T + row / a.G) * a.Hq + h * a.G + row % a.G) * kH;
      qv[k] = __ldg(reinterpret_cast<const uint4*>(qr) + (i & 15));
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
  const int max_vis = n_visible(min(R, TG - row0) - 1);
  const int min_vis = n_visible(0);
  int nv[NR];   // visible keys of the lane's rows 8 rh + g
#pragma unroll
  for (int rh = 0; rh < NR; ++rh) nv[rh] = n_visible(8 * rh + g);
  const int n_pages = (max_vis + kP - 1) / kP;
  const int p_begin = split * a.pages_per_split;
  const int np = max(min(p_begin + a.pages_per_split, n_pages) - p_begin, 0);
  const int32_t* pt_row = a.page_table + ((int64_t)b * a.Hkv + h) * a.max_pages;

  // m_run: rows 8 rh + g; l_run: the fp16 probabilities' row sums of rows
  // 8 nt + 2t and 8 nt + 2t + 1 (the layout of the V side's U columns)
  float m_run[NR];
  float2 l_run[NR];
#pragma unroll
  for (int rh = 0; rh < NR; ++rh) {
    m_run[rh] = -CUDART_INF_F;
    l_run[rh] = make_float2(0.0f, 0.0f);
  }
  // R = 16: O[mt][nt][c] = channel 16 mt + g + 8c, rows 8 nt + 2t and 8 nt + 2t + 1
  float2 O[kTmem ? 1 : 8][2][2];
#pragma unroll
  for (int mt = 0; mt < (kTmem ? 1 : 8); ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) O[mt][nt][0] = O[mt][nt][1] = make_float2(0.f, 0.f);

  if (warp == kConsumers) {
    if (L == 0)
      produce_units<FULL>(a, pt_row, p_begin, np, first_id, s_ring, bar_full, bar_empty, &tm_ka, &tm_va, &tm_kr,
                          &tm_vr, s_flag);
  } else {
    // the Q fragments, by the 8 consumer warps only; they meet at named
    // barrier 1 (the producer warp never takes part in it).  The CTA's R query
    // rows are the vectors qv loaded above; the largest |q| sets the fp16 scaling: 2^-eq
    // puts it in [2^14, 2^15) (the other values keep their 8 significant bits
    // unless they are 2^-28 times smaller than it)
    {
      uint32_t qm = 0u;
#pragma unroll
      for (int k = 0; k < kQPer; ++k) {
        const uint32_t w4[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) qm = max(qm, max(w4[j] & 0x7FFFu, (w4[j] >> 16) & 0x7FFFu));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) qm = max(qm, __shfl_xor_sync(0xffffffffu, qm, o));
      if (L == 0) atomicMax(s_qmax, qm);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
    const int eq = min(max((int)((*s_qmax >> 7) & 0xFFu) - 127 - 14, -100), 113);
    const float qscale = __uint_as_float((uint32_t)(127 - eq) << 23);   // 2^-eq
    // fragment entry (mi, ks, lane, e) holds row 16 mi + g' + 8 (e & 1), channels
    // 16 ks + 2t' + 8 (e >> 1) + {0, 1} (lane = 4 g' + t'): word j of vector
    // (r, v) goes to mi = r >> 4, g' = r & 7, e = 2 (v & 1) + ((r >> 3) & 1),
    // ks = v >> 1, t' = j
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = tid + k * kConsumerThreads;
      const int r = i >> 4, v = i & 15;
      const int e = 2 * (v & 1) + ((r >> 3) & 1);
      uint32_t* dst = reinterpret_cast<uint32_t*>(smem + S::kQ) + (((r >> 4) * 8 + (v >> 1)) * 32 + 4 * (r & 7)) * 4 + e;
      const uint32_t w4[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dst[4 * j] = h2(__uint_as_float(w4[j] << 16) * qscale, __uint_as_float(w4[j] & 0xFFFF0000u) * qscale);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");

    const int w = warp;
    const uint32_t s_ab = S::kWarps + w * kTcWarpBytes;
    const uint32_t lane8 = 8u * L, lane4 = 4u * L, lane4v = 128u + 4u * L;
    // K side: bytes 2g (n-tiles 0, 1) and 2g+1 (n-tiles 2, 3) of a channel row,
    // bytes 2 (g & 1) and 2 (g & 1) + 1 of its word g >> 1
    const uint32_t ksel0 = byte_sel(2 * (g & 1)), ksel1 = byte_sel(2 * (g & 1) + 1);
    const uint32_t kword = 4 * (g >> 1);
    // V side: bytes 4t..4t+3 of channel 16 mt + g, word t of its chunk unit
    const uint32_t vofs = g * 128 + ((w ^ g) << 4) + 4 * t;
    const float eps = a.eps;
    const float sc = a.scale_log2;
    const float code_max = UNI ? a.code_max : 1.0f;
    bool failed = false;

    if (kTmem) {   // O = 0 (TMEM contents are undefined after allocation)
      uint32_t z[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) z[k] = 0u;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) tmem_st16(t_warp + 16u * mt, z);
    }

    // (A, B) of the unit's 128 channels; for a key unit scaled by 2^-ek so that
    // the largest |A| + code_max |B| (a bound on |k|) lies in [2^14, 2^15), ek returned
    auto prep_ab = [&](uint32_t unit, bool key) -> int {
      const uint32_t mt = unit + G::kMetaOff;
      float2 ab[4];
      float mx = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int d = L + 32 * k;
        if (UNI) {   // uniform codes: value = min + scale * code in every chunk
          ab[k] = make_float2(lds<float>(smem, mt + 4 * d), lds<float>(smem, mt + 4 * (kH + d)));
        } else {
          const float gmin = lds<float>(smem, mt + 4 * d);
          const float dg = __fadd_rn(lds<float>(smem, mt + 4 * (kH + d)), eps);
          const float mu = lds<float>(smem, mt + 4 * (kMetaMuOff + w * kH + d));
          const float ds = __fadd_rn(lds<float>(smem, mt + 4 * (kMetaSigmaOff + w * kH + d)), eps);
          ab[k] = make_float2(__fmaf_rn(dg, mu, gmin), __fmul_rn(dg, ds));
        }
        // |k| <= |A| + code_max |B| (code_max bounds the table values)
        mx = fmaxf(mx, fabsf(ab[k].x) + code_max * fabsf(ab[k].y));
      }
      int ek = 0;
      if (key) {
        mx = warp_max_nonneg(mx);
        ek = min(max((int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127 - 14, -100), 100);
      }
      const float f = __uint_as_float((uint32_t)(127 - ek) << 23);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        *reinterpret_cast<float2*>(smem + s_ab + 8 * (L + 32 * k)) = make_float2(ab[k].x * f, ab[k].y * f);
      return ek;
    };

    for (int i = 0; i < np && !failed; ++i) {
      const int p = p_begin + i;
      const int uK = 2 * i, uV = 2 * i + 1;
      const int sK = uK % kSt, sV = uV % kSt;
      const uint32_t unitK = S::kRing + sK * G::kUnit;
      const uint32_t unitV = S::kRing + sV * G::kUnit;

      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sK, (uK / kSt) & 1, a.wait_ns));
      if (failed) break;
      const int ek = prep_ab(unitK, true);
      __syncwarp();
      // softmax scale of this chunk's logits: the operands' power-of-two scales return here
      const float sck = sc * __uint_as_float((uint32_t)min(max(127 + ek + eq, 1), 254) << 23);

      // ---- S = Q K^T over 8 k-steps of channels 16 ks + 2t + {0, 1, 8, 9}; n-tile k, column n: token 4n + k
      float sacc[MT][4][4];
#pragma unroll
      for (int mi = 0; mi < MT; ++mi)
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[mi][n][e] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint4 qf[MT];
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) qf[mi] = lds<uint4>(smem, S::kQ + ((mi * 8 + ks) * 32 + L) * 16);
        const int c0 = 16 * ks + 2 * t;   // channels c0, c0 + 1 (b0) and c0 + 8, c0 + 9 (b1)
        const float4 abl = lds<float4>(smem, s_ab + 8 * c0);
        const float4 abh = lds<float4>(smem, s_ab + 8 * (c0 + 8));
        const float2 A[4] = {make_float2(abl.x, abl.x), make_float2(abl.z, abl.z), make_float2(abh.x, abh.x),
                             make_float2(abh.z, abh.z)};
        const float2 B[4] = {make_float2(abl.y, abl.y), make_float2(abl.w, abl.w), make_float2(abh.y, abh.y),
                             make_float2(abh.w, abh.w)};
        // k of tokens 4g + {0, 1} (jb 0) and 4g + {2, 3} (jb 1) of the four channels
        float2 kv[4][2];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int ch = c0 + (c & 1) + 8 * (c >> 1);
          const uint32_t r = unitK + ch * 128 + ((w ^ (ch & 7)) << 4) + kword;
          const uint32_t wa = lds<uint32_t>(smem, r);
          float2 l0, l1;
          if (!FULL) {
            l0 = lds<float2>(smem, S::kLutK + lut_off(wa, lane8, ksel0));
            l1 = lds<float2>(smem, S::kLutK + lut_off(wa, lane8, ksel1));
          } else {
            uint32_t ev, od;
            full_codes(wa, lds<uint32_t>(smem, r + G::kResOff), ev, od);
            auto val = [&](uint32_t codes, uint32_t sel) {
              return lds<float>(smem, S::kLutK + lut_off(codes, lane4, sel));
            };
            l0 = make_float2(val(ev, ksel0), val(od, ksel0));
            l1 = make_float2(val(ev, ksel1), val(od, ksel1));
          }
          kv[c][0] = __ffma2_rn(l0, B[c], A[c]);
          kv[c][1] = __ffma2_rn(l1, B[c], A[c]);
        }
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          // n-tile n = token 4g + n: b0 = channels (c0, c0 + 1), b1 = (c0 + 8, c0 + 9)
          float x[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) x[c] = (n & 1) ? kv[c][n >> 1].y : kv[c][n >> 1].x;
          float hf[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) hf[c] = __uint_as_float(__float_as_uint(x[c]) & 0xFFFFE000u);
          const float2 r01 = __ffma2_rn(make_float2(hf[0], hf[1]), make_float2(-1.0f, -1.0f), make_float2(x[0], x[1]));
          const float2 r23 = __ffma2_rn(make_float2(hf[2], hf[3]), make_float2(-1.0f, -1.0f), make_float2(x[2], x[3]));
          const uint32_t h0 = h2(hf[0], hf[1]), h1 = h2(hf[2], hf[3]);
          const uint32_t lo0 = h2(r01.x, r01.y), lo1 = h2(r23.x, r23.y);
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
            mma_f16(sacc[mi][n], qf[mi].x, qf[mi].y, qf[mi].z, qf[mi].w, h0, h1);
            mma_f16(sacc[mi][n], qf[mi].x, qf[mi].y, qf[mi].z, qf[mi].w, lo0, lo1);
          }
        }
      }
      __syncwarp();
      if (L == 0) mbar_arrive(bar_empty + 8 * sK);

      // ---- online softmax: row 8 rh + g is accumulator half rh & 1 (S entries
      // 2 (rh & 1) + hh) of m-tile rh >> 1; token 8t + j, j = 4 hh + k, sits in n-tile k.
      // One warp vote tells whether any score of the chunk exceeds its row's
      // running maximum; only then are the row maxima taken by shuffles and the
      // output rescaled.  Each probability x 2^10 is one exp2 of a fused
      // multiply-add, 2^(S sck + 10 - m) <= 2^10, a masked score (-inf) giving 0.
      // (Letting the maximum lag by up to 2^5 ran 2% faster, but then a
      // dominant key's fp16 probability is no longer exactly 2^10 and the worst
      // output error on an outlier channel rose from 3.6e-4 to 1.5e-3.)
      const int pos0 = p * kP + 32 * w + 8 * t;
      const bool all_visible = (p + 1) * kP <= min_vis;
      float pr[NR][8];   // [rh][j], raw scores, then probabilities x 2^10
      float smax[NR];    // the lane's largest score of each row (scaled)
#pragma unroll
      for (int rh = 0; rh < NR; ++rh) {
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float sv = sacc[rh >> 1][j & 3][2 * (rh & 1) + (j >> 2)];
          if (!all_visible && pos0 + j >= nv[rh]) sv = -CUDART_INF_F;
          pr[rh][j] = sv;
          mx = fmaxf(mx, sv);
        }
        smax[rh] = mx * sck;   // sck > 0
      }
      bool up = false;
#pragma unroll
      for (int rh = 0; rh < NR; ++rh) up |= smax[rh] > m_run[rh];
      const bool rescale = __any_sync(0xffffffffu, up);
      float corr[NR];
#pragma unroll
      for (int rh = 0; rh < NR; ++rh) {
        float mnew = m_run[rh];
        if (rescale) {
          float mr = smax[rh];
          mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, 1));
          mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, 2));
          mnew = fmaxf(m_run[rh], mr);
        }
        corr[rh] = (!rescale || mnew == -CUDART_INF_F) ? 1.0f : exp2f(m_run[rh] - mnew);
        // a row with no visible score yet (m = -inf) takes the reference 0
        const float nref = (mnew == -CUDART_INF_F) ? 0.0f : 10.0f - mnew;
#pragma unroll
        for (int j = 0; j < 8; ++j) pr[rh][j] = exp2f(__fmaf_rn(pr[rh][j], sck, nref));
        m_run[rh] = mnew;
      }
      // P^T fragments of k-step kv, n-tile nt (rows 8 nt + g): tokens 8t + 4kv + {0,1} and + {2,3}
      uint32_t pb[2][NR][2];
#pragma unroll
      for (int kv = 0; kv < 2; ++kv)
#pragma unroll
        for (int nt = 0; nt < NR; ++nt) {
          pb[kv][nt][0] = h2(pr[nt][4 * kv], pr[nt][4 * kv + 1]);
          pb[kv][nt][1] = h2(pr[nt][4 * kv + 2], pr[nt][4 * kv + 3]);
        }
      // statistics of U's columns, rows 8 nt + 2t + e: the corrections from lane
      // 8t + 4e; the row sums of exactly the fp16 probabilities the V side
      // multiplies, from a matrix of ones times P^T (so the normaliser and the
      // A psum term use the same rounded weights as U)
      float2 cr[NR], pss[NR];
#pragma unroll
      for (int nt = 0; nt < NR; ++nt) {
        cr[nt] = make_float2(1.0f, 1.0f);
        if (rescale)
          cr[nt] = make_float2(__shfl_sync(0xffffffffu, corr[nt], 8 * t),
                               __shfl_sync(0xffffffffu, corr[nt], 8 * t + 4));
        float ps4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_f16(ps4, kOnes2, kOnes2, kOnes2, kOnes2, pb[0][nt][0], pb[0][nt][1]);
        mma_f16(ps4, kOnes2, kOnes2, kOnes2, kOnes2, pb[1][nt][0], pb[1][nt][1]);
        pss[nt] = make_float2(ps4[0], ps4[1]);
        l_run[nt] = __ffma2_rn(l_run[nt], cr[nt], pss[nt]);
      }

      // ---- V unit: U = l~ P^T per 16-channel m-tile, folded into O
      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sV, (uV / kSt) & 1, a.wait_ns));
      if (failed) break;
      prep_ab(unitV, false);
      __syncwarp();
      if (kTmem) tmem_wait_st();   // the previous page's O stores have landed
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t ov[16];   // R = 32: O of channel tile mt, [nt][c][row parity]
        if (kTmem) tmem_ld16(t_warp + 16u * mt, ov);
        const int c0 = 16 * mt + g;
        const float2 ab0 = lds<float2>(smem, s_ab + 8 * c0);
        const float2 ab1 = lds<float2>(smem, s_ab + 8 * (c0 + 8));
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
        float u[NR][4];
#pragma unroll
        for (int nt = 0; nt < NR; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) u[nt][e] = 0.0f;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const uint2 x00 = vpair(0, 2 * kv), x10 = vpair(1, 2 * kv);
          const uint2 x01 = vpair(0, 2 * kv + 1), x11 = vpair(1, 2 * kv + 1);
#pragma unroll
          for (int nt = 0; nt < NR; ++nt) {
            mma_f16(u[nt], x00.x, x10.x, x01.x, x11.x, pb[kv][nt][0], pb[kv][nt][1]);
            mma_f16(u[nt], x00.y, x10.y, x01.y, x11.y, pb[kv][nt][0], pb[kv][nt][1]);
          }
        }
        if (kTmem) tmem_wait_ld(ov);
#pragma unroll
        for (int nt = 0; nt < NR; ++nt) {
          float2 p0, p1;
          if (kTmem) {
            p0 = make_float2(__uint_as_float(ov[4 * nt]), __uint_as_float(ov[4 * nt + 1]));
            p1 = make_float2(__uint_as_float(ov[4 * nt + 2]), __uint_as_float(ov[4 * nt + 3]));
          } else {
            p0 = O[kTmem ? 0 : mt][nt & 1][0];
            p1 = O[kTmem ? 0 : mt][nt & 1][1];
          }
          if (rescale) {
            p0 = __fmul2_rn(p0, cr[nt]);
            p1 = __fmul2_rn(p1, cr[nt]);
          }
          p0 = __ffma2_rn(make_float2(ab0.x, ab0.x), pss[nt], p0);
          p1 = __ffma2_rn(make_float2(ab1.x, ab1.x), pss[nt], p1);
          p0 = __ffma2_rn(make_float2(ab0.y, ab0.y), make_float2(u[nt][0], u[nt][1]), p0);
          p1 = __ffma2_rn(make_float2(ab1.y, ab1.y), make_float2(u[nt][2], u[nt][3]), p1);
          if (kTmem) {
            ov[4 * nt] = __float_as_uint(p0.x);
            ov[4 * nt + 1] = __float_as_uint(p0.y);
            ov[4 * nt + 2] = __float_as_uint(p1.x);
            ov[4 * nt + 3] = __float_as_uint(p1.y);
          } else {
            O[kTmem ? 0 : mt][nt & 1][0] = p0;
            O[kTmem ? 0 : mt][nt & 1][1] = p1;
          }
        }
        if (kTmem) tmem_st16(t_warp + 16u * mt, ov);
      }
      __syncwarp();
      if (L == 0) mbar_arrive(bar_empty + 8 * sV);
    }
    if (kTmem) tmem_wait_st();
    if (failed && L == 0) {
      atomicExch(a.status, 1);
      *s_flag = 1;
    }
  }

  // ================= merge the 8 chunk states (the ring and the tables are idle now)
  if (kTmem) tmem_fence_before_sync();
  __syncthreads();
  if (kTmem) tmem_fence_after_sync();
  allow_dependent_launch();   // the split combine may be scheduled once every CTA is here
  const bool ok = *reinterpret_cast<volatile int*>(s_flag) == 0;
  float* mo = reinterpret_cast<float*>(smem + S::kMergeO);
  float* mm = reinterpret_cast<float*>(smem + S::kMergeM);
  float* ml = reinterpret_cast<float*>(smem + S::kMergeL);
  float* mf = reinterpret_cast<float*>(smem + S::kMergeF);
  float2* mrow = reinterpret_cast<float2*>(smem + S::kMergeS);
  constexpr int MS = S::kMergeStride;
  if (ok && warp < kConsumers) {
#pragma unroll
    for (int rh = 0; rh < NR; ++rh) {
      if (t == 0) mm[warp * R + 8 * rh + g] = m_run[rh];
      if (g == 0) {   // every g holds the row sums of rows 8 rh + 2t, + 1
        ml[warp * R + 8 * rh + 2 * t] = l_run[rh].x;
        ml[warp * R + 8 * rh + 2 * t + 1] = l_run[rh].y;
      }
    }
  }
  __syncthreads();
  // chunk w's factor of row r, 2^(m_w - m*) (0 where the chunk saw no key of the row)
  if (ok && tid < kConsumers * R) {
    const int r = tid % R;
    float mstar = -CUDART_INF_F;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) mstar = fmaxf(mstar, mm[ww * R + r]);
    const float mw = mm[tid];
    mf[tid] = (mw == -CUDART_INF_F) ? 0.0f : exp2f(mw - mstar);
  }
  __syncthreads();
  // each row's (m*, l*); each lane's O values, scaled by its chunk's factors,
  // into the chunk's rows of the merge area
  if (ok && tid < R) {
    float mstar = -CUDART_INF_F, l = 0.0f;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) {
      mstar = fmaxf(mstar, mm[ww * R + tid]);
      l += ml[ww * R + tid] * mf[ww * R + tid];
    }
    mrow[tid] = make_float2(mstar, l);
  }
  if (ok && warp < kConsumers) {
    float2 fr[NR];   // factors of the lane's rows 8 nt + 2t and 8 nt + 2t + 1
#pragma unroll
    for (int nt = 0; nt < NR; ++nt) fr[nt] = make_float2(mf[warp * R + 8 * nt + 2 * t], mf[warp * R + 8 * nt + 2 * t + 1]);
    float* dst = mo + warp * R * MS;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      float2 q[NR][2];   // [nt][c]: channel 16 mt + g + 8c, rows 8 nt + 2t, + 1
      if (kTmem) {
        uint32_t ov[16];
        tmem_ld16(t_warp + 16u * mt, ov);
        tmem_wait_ld(ov);
#pragma unroll
        for (int nt = 0; nt < NR; ++nt) {
          q[nt][0] = make_float2(__uint_as_float(ov[4 * nt]), __uint_as_float(ov[4 * nt + 1]));
          q[nt][1] = make_float2(__uint_as_float(ov[4 * nt + 2]), __uint_as_float(ov[4 * nt + 3]));
        }
      } else {
#pragma unroll
        for (int nt = 0; nt < NR; ++nt) {
          q[nt][0] = O[kTmem ? 0 : mt][nt & 1][0];
          q[nt][1] = O[kTmem ? 0 : mt][nt & 1][1];
        }
      }
#pragma unroll
      for (int nt = 0; nt < NR; ++nt) {
        const int r = 8 * nt + 2 * t;
        const int c0 = 16 * mt + g;
        dst[r * MS + c0] = q[nt][0].x * fr[nt].x;
        dst[(r + 1) * MS + c0] = q[nt][0].y * fr[nt].y;
        dst[r * MS + c0 + 8] = q[nt][1].x * fr[nt].x;
        dst[(r + 1) * MS + c0 + 8] = q[nt][1].y * fr[nt].y;
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < R * kH; i += kThreadsQ) {
    if (!ok) break;
    const int r = i >> 7, d = i & 127;
    const int row = row0 + r;
    const int rg4 = row >> 2;
    if (rg4 >= a.n_rg) continue;
    float o = 0.0f;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) o += mo[(ww * R + r) * MS + d];
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
  // every TMEM access of every warp has completed (each waited for its own
  // loads and stores) before the columns are freed
  if (kTmem) {
    tmem_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
      tmem_fence_after_sync();
      tmem_dealloc(tmem, kTmemCols);
    }
  }
}

// rows per CTA: 32 when more than 16 rows share a KV head (each key is
// dequantised once for 32 rows), else 16
constexpr bool tc_wide(int rows, bool) { return rows > 16; }

template <bool FULL, int R, bool UNI>
cudaError_t launch_tc(const DecodeArgs& a, const LutTables* lut, cudaStream_t s) {
  constexpr int kSmem = TLayout<FULL, R>::kAlloc;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<FULL, R, UNI>,
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
  dim3 grid(a.n_splits, a.Hkv * ((a.T * a.G + R - 1) / R), a.B);
  return launch_programmatic(decode_tc_kernel<FULL, R, UNI>, grid, dim3(kThreadsQ), kSmem, s, a, *lut, tka, tva, tkr,
                             tvr);
}

}  // namespace

bool use_tc_rows(int rows) { return rows >= 12; }
int tc_rows_per_cta(int rows, bool full) { return tc_wide(rows, full) ? 32 : 16; }

cudaError_t launch_decode_tc(const DecodeArgs& a, bool full, const LutTables* lut, cudaStream_t s) {
  const bool wide = tc_wide(a.T * a.G, full);
  if (a.uniform) {
    if (!full) return wide ? launch_tc<false, 32, true>(a, lut, s) : launch_tc<false, 16, true>(a, lut, s);
    return wide ? launch_tc<true, 32, true>(a, lut, s) : launch_tc<true, 16, true>(a, lut, s);
  }
  if (!full) return wide ? launch_tc<false, 32, false>(a, lut, s) : launch_tc<false, 16, false>(a, lut, s);
  return wide ? launch_tc<true, 32, false>(a, lut, s) : launch_tc<true, 16, false>(a, lut, s);
}

}  // namespace lynx
