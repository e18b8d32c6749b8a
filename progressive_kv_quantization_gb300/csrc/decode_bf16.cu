// BF16 decode attention on the tensor cores: the attention of the Lynx
// paper's §2.1 over plain BF16 KV pages, the full-precision baseline that the
// quantised draft and verification passes of §4.2-4.3 are measured against.
// Any number of query rows per KV head, in CTAs of 8 or 16 rows.
//
// CTA: one producer lane streams the split's K and V pages through a 3-slot
// shared-memory ring, each page as four TMA tiles of 64 tokens x 128 channels
// (128-byte rows, 128-byte swizzle); 8 consumer warps, warp w owning the
// 32-token chunk w of every page with its own online softmax, merged once per
// CTA; the split combine merges the CTAs' partials by their log-sum-exps.
//
//   K side   S[16 rows x 32 tokens] = Q K^T as bf16 m16n8k16, query rows as
//            M (rows past the CTA's are zero), four n-tiles of 8 tokens, 8
//            k-steps of 16 channels.  The products of BF16 values are exact and
//            sum in float32.  Q fragments come from shared memory by ldmatrix,
//            the K fragments by ldmatrix.trans from the channel rows of the
//            staged page (a page is stored channel-major, so the transposed
//            8 x 8 blocks are the column-major B operand).
//   V side   U[16 channels x 8 rows] = V P^T per channel tile, two k-steps of
//            16 tokens, accumulated straight into the output O.  The V fragments
//            are the staged channel rows as they are (ldmatrix); P^T is the
//            score accumulators of the K side: entries (0, 1) of n-tile 2 kv
//            and 2 kv + 1 hold row g's tokens 2t, 2t + 1 and 2t + 8, 2t + 9 of
//            k-step kv, the B fragment of the V side in the same lane.  P is
//            split into a bf16 head (the float truncated to 8 significant bits)
//            and the bf16-rounded remainder, two MMAs, ~16-bit products.
//
// Softmax.  A row's running maximum moves only when one of the chunk's scores
// exceeds it by more than 5 in log2 units (a warp vote; the row maxima by
// shuffles only then); probabilities are 2^(s - m), at most 2^5.
//
// Rounding: scores and sums in float32; P to ~16 bits.

#include "decode_common.cuh"

#include <cuda_bf16.h>

namespace lynx {
namespace {

constexpr int kBStages = 3;                   // ring slots
constexpr int kBUnit = kPageElems * 2;        // one BF16 page, 65536 B
constexpr int kBTile = 16384;                 // 64 tokens x 128 channels, 128-byte rows
constexpr int kBQStride = 272;                // bytes per query row in shared memory (256 + 16: conflict-free)
constexpr float kBLazyLog2 = 5.0f;            // largest log2 lead of a score over the running maximum

// NT: 8-row tiles of query rows per CTA (1 or 2)
template <int NT>
struct BLayout {
  static constexpr int kR = 8 * NT;
  static constexpr int kRing = 0;
  static constexpr int kQ = kRing + kBStages * kBUnit;   // [16 rows][kBQStride] bf16, rows past kR zero
  static constexpr int kFlag = kQ + 16 * kBQStride;
  static constexpr int kBar = kFlag + 16;                  // ring full[kBStages], empty[kBStages]
  static constexpr int kTotal = kBar + 2 * kBStages * 8;
  static constexpr int kAlloc = kTotal + 1024;
  // end-of-kernel merge area (reuses the ring): o[8][kR][kMergeStride] (each
  // chunk's output rows scaled by the chunk's factor 2^(m_w - m*)), then
  // m[8][kR], l[8][kR], the factors f[8][kR] and the rows' (m*, l*)
  static constexpr int kMergeStride = kH + 4;
  static constexpr int kMergeO = 0;
  static constexpr int kMergeM = kMergeO + kConsumers * kR * kMergeStride * 4;
  static constexpr int kMergeL = kMergeM + kConsumers * kR * 4;
  static constexpr int kMergeF = kMergeL + kConsumers * kR * 4;
  static constexpr int kMergeS = kMergeF + kConsumers * kR * 4;
  static_assert(kMergeS + kR * 8 <= kBStages * kBUnit, "merge area");
};
static_assert(BLayout<2>::kAlloc <= 232448, "shared memory (BF16 decode)");

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&d)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&d)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// bf16 pairs (x low, y high): the head (x, y truncated to bf16) and the
// bf16-rounded remainders
__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const uint32_t xb = __float_as_uint(x), yb = __float_as_uint(y);
  hi = prmt(xb, yb, 0x7632u);
  const float rx = x - __uint_as_float(xb & 0xFFFF0000u);
  const float ry = y - __uint_as_float(yb & 0xFFFF0000u);
  const __nv_bfloat162 r = __floats2bfloat162_rn(rx, ry);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}

// Producer lane: K and V pages of pages [p_begin, p_begin + np) of one
// page-table row through the ring, four 16 KB tiles per page.  Waits bounded
// as in the quantised kernels' producer; on leaving, waits (bounded) for its
// last copies to land.
__device__ void produce_bf16(const DecodeArgs& a, const int32_t* pt_row, int p_begin, int np, int first_id,
                             uint32_t s_ring, uint32_t bar_full, uint32_t bar_empty, const CUtensorMap* tm_k,
                             const CUtensorMap* tm_v, int* s_flag) {
  const int skip = a.inject_skip - 1;   // -1: no unit is skipped
  int u_end = 0;
  bool ok = true;
  int64_t id = first_id;
  for (int u = 0; u < 2 * np; ++u) {
    const int st = u % kBStages;
    if (u >= kBStages && !mbar_wait(bar_empty + 8 * st, ((u / kBStages) - 1) & 1, a.wait_ns)) {
      ok = false;
      break;
    }
    u_end = u + 1;
    const bool is_v = (u & 1) != 0;
    if (u >= 2 && !is_v) id = pt_row[p_begin + (u >> 1)];
    if (u == skip) continue;   // test hook: this unit's copy is never issued
    if (id < 0 || id >= a.n_pool) {
      atomicExch(a.status, 2);
      id = 0;
    }
    const uint32_t dst = s_ring + st * kBUnit;
    const uint32_t bar = bar_full + 8 * st;
    mbar_expect_tx(bar, kBUnit);
#pragma unroll
    for (int q = 0; q < 4; ++q) tma_tile_g2s(dst + q * kBTile, is_v ? tm_v : tm_k, 64 * q, (int)(id * kH), bar);
  }
  if (!ok) {
    atomicExch(a.status, 1);
    *s_flag = 1;
  }
  for (int u = u_end - 1; u >= 0 && u >= u_end - kBStages; --u)
    if (u != skip) mbar_wait(bar_full + 8 * (u % kBStages), (u / kBStages) & 1, a.wait_ns);
}

template <int NT>
__global__ void __launch_bounds__(kThreadsQ, 1)
decode_bf16_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v) {
  using S = BLayout<NT>;
  constexpr int R = S::kR;
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
  const uint32_t bar_empty = bar_full + 8 * kBStages;
  int* s_flag = reinterpret_cast<int*>(smem + S::kFlag);

  if (tid == 0) {
    for (int st = 0; st < kBStages; ++st) {
      mbar_init(bar_full + 8 * st, 1);
      mbar_init(bar_empty + 8 * st, kConsumers);
    }
    *s_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // every global-memory access of this kernel follows this wait
  wait_prerequisite_grids();
  int first_id = 0;
  if (tid == kConsumers * 32) {
    const int pb = split * a.pages_per_split;
    if (pb < a.max_pages) first_id = a.page_table[((int64_t)b * a.Hkv + h) * a.max_pages + pb];
  }
  // query vector of thread i < 256: row i >> 4 of the 16 (zeros past the CTA's
  // rows and past T x G), channels 8 (i & 15) .. + 7
  uint4 qx = make_uint4(0u, 0u, 0u, 0u);
  if (tid < 256) {
    const int r = tid >> 4;
    const int row = row0 + r;
    if (r < R && row < TG) {
      const uint16_t* qr = a.q + (((int64_t)b * a.T + row / a.G) * a.Hq + h * a.G + row % a.G) * kH;
      qx = __ldg(reinterpret_cast<const uint4*>(qr) + (tid & 15));
    }
  }

  int ctx = a.ctx_len[b];
  if (ctx < 0 || ctx > max_keys) {
    if (tid == 0) atomicExch(a.status, 3);
    ctx = ctx < 0 ? 0 : max_keys;
  }
  auto n_visible = [&](int r) {
    const int row = row0 + r;
    if (row >= TG) return 0;
    const int n = a.causal ? ctx - a.T + row / a.G + 1 : ctx;
    return n < 0 ? 0 : n;
  };
  // n_visible does not decrease with the row: the CTA's first and last real rows
  const int max_vis = n_visible(min(R, TG - row0) - 1);
  const int min_vis = n_visible(0);
  const int n_pages = (max_vis + kP - 1) / kP;
  const int p_begin = split * a.pages_per_split;
  const int np = max(min(p_begin + a.pages_per_split, n_pages) - p_begin, 0);
  const int32_t* pt_row = a.page_table + ((int64_t)b * a.Hkv + h) * a.max_pages;

  // softmax state of the lane's rows 8 nr + g
  float m_run[NT], l_run[NT];
#pragma unroll
  for (int nr = 0; nr < NT; ++nr) {
    m_run[nr] = -CUDART_INF_F;
    l_run[nr] = 0.0f;
  }
  // O[mt][nr] = (channel 16 mt + g, rows 8 nr + 2t, + 1), (channel 16 mt + g + 8, same rows)
  float O[8][NT][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int nr = 0; nr < NT; ++nr)
#pragma unroll
      for (int e = 0; e < 4; ++e) O[mt][nr][e] = 0.0f;
  bool failed = false;

  if (warp == kConsumers) {
    if (L == 0) produce_bf16(a, pt_row, p_begin, np, first_id, s_ring, bar_full, bar_empty, &tm_k, &tm_v, s_flag);
  } else {
    *reinterpret_cast<uint4*>(smem + S::kQ + (tid >> 4) * kBQStride + 16 * (tid & 15)) = qx;
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");

    const int w = warp;
    const float sc = a.scale_log2;
    // ldmatrix roles: lane L gives the address of row L & 7 of matrix L >> 3
    const int lj = L >> 3, lr = L & 7;
    // K and V fragments: channel rows 16 x + 8 (lj & 1) + lr of chunk w's tile
    // (tile w >> 1, 16-byte segments 4 (w & 1) ..); a channel row's segment s
    // is stored at s ^ (channel & 7) = s ^ lr
    const uint32_t frag_row = (uint32_t)(w >> 1) * kBTile + (uint32_t)(8 * (lj & 1) + lr) * 128u;
    const int seg0 = 4 * (w & 1) + (lj >> 1);
    // Q fragments: query row 8 (lj & 1) + lr, channels 16 ks + 8 (lj >> 1) ..
    const uint32_t q_frag = base + S::kQ + (uint32_t)(8 * (lj & 1) + lr) * kBQStride + 16u * (lj >> 1);
    int nv[NT];
#pragma unroll
    for (int nr = 0; nr < NT; ++nr) nv[nr] = n_visible(8 * nr + g);

    for (int i = 0; i < np && !failed; ++i) {
      const int p = p_begin + i;
      const int uK = 2 * i, uV = 2 * i + 1;
      const int sK = uK % kBStages, sV = uV % kBStages;
      const uint32_t unitK = s_ring + sK * kBUnit;
      const uint32_t unitV = s_ring + sV * kBUnit;
      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sK, (uK / kBStages) & 1, a.wait_ns));
      if (failed) break;

      // ---- S = Q K^T: n-tile nt = tokens 8 nt .. 8 nt + 7 of the chunk
      float sacc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t qa[4];
        ldsm_x4(q_frag + 32u * ks, qa);
        const uint32_t krow = unitK + frag_row + (uint32_t)(16 * ks) * 128u;
        uint32_t kb0[4], kb1[4];   // (b0, b1) of n-tiles 0, 1 and of n-tiles 2, 3
        ldsm_x4_t(krow + ((uint32_t)((seg0 + 0) ^ lr) << 4), kb0);
        ldsm_x4_t(krow + ((uint32_t)((seg0 + 2) ^ lr) << 4), kb1);
        mma_bf16(sacc[0], qa, kb0[0], kb0[1]);
        mma_bf16(sacc[1], qa, kb0[2], kb0[3]);
        mma_bf16(sacc[2], qa, kb1[0], kb1[1]);
        mma_bf16(sacc[3], qa, kb1[2], kb1[3]);
      }
      __syncwarp();
      if (L == 0) mbar_arrive(bar_empty + 8 * sK);

      // ---- online softmax of rows 8 nr + g: the lane holds tokens 8 nt + 2t + e
      // at sacc[nt][2 nr + e]
      const int pos0 = p * kP + 32 * w + 2 * t;
      const bool all_visible = (p + 1) * kP <= min_vis;
      float mloc[NT];
#pragma unroll
      for (int nr = 0; nr < NT; ++nr) {
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float sv = sacc[nt][2 * nr + e];
            if (!all_visible && pos0 + 8 * nt + e >= nv[nr]) sv = -CUDART_INF_F;
            sacc[nt][2 * nr + e] = sv;
            mx = fmaxf(mx, sv);
          }
        mloc[nr] = mx * sc;   // sc > 0
      }
      bool up = false;
#pragma unroll
      for (int nr = 0; nr < NT; ++nr) up |= mloc[nr] > m_run[nr] + kBLazyLog2;
      const bool grow = __any_sync(0xffffffffu, up);
      float corr[NT];
#pragma unroll
      for (int nr = 0; nr < NT; ++nr) {
        float mnew = m_run[nr];
        if (grow) {
          float mr = mloc[nr];
          mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, 1));
          mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, 2));
          mnew = fmaxf(m_run[nr], mr);
        }
        corr[nr] = (!grow || mnew == -CUDART_INF_F) ? 1.0f : exp2f(m_run[nr] - mnew);
        // p = 2^(s sc - m); a masked score gives 0, a row with no visible score
        // yet (m = -inf) takes the reference 0
        const float nref = (mnew == -CUDART_INF_F) ? 0.0f : -mnew;
        float ps = 0.0f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pv = exp2f(__fmaf_rn(sacc[nt][2 * nr + e], sc, nref));
            sacc[nt][2 * nr + e] = pv;
            ps += pv;
          }
        l_run[nr] = __fmaf_rn(l_run[nr], corr[nr], ps);   // the lane's tokens; summed at the end
        m_run[nr] = mnew;
      }
      // P^T fragments of k-step kv, rows 8 nr + g: (b0, b1) = tokens 16 kv + 2t, + 1 and
      // 16 kv + 2t + 8, + 9, each as a bf16 head and remainder
      uint32_t ph[2][NT][2], pl[2][NT][2];
#pragma unroll
      for (int kv = 0; kv < 2; ++kv)
#pragma unroll
        for (int nr = 0; nr < NT; ++nr)
#pragma unroll
          for (int j = 0; j < 2; ++j)
            split_bf16x2(sacc[2 * kv + j][2 * nr], sacc[2 * kv + j][2 * nr + 1], ph[kv][nr][j], pl[kv][nr][j]);

      // ---- V unit: O += V P^T per 16-channel tile
      failed = __any_sync(0xffffffffu, !mbar_wait(bar_full + 8 * sV, (uV / kBStages) & 1, a.wait_ns));
      if (failed) break;
      if (grow) {   // rows 8 nr + 2t + e of the lane's outputs: corr held by lanes 8t + 4e
#pragma unroll
        for (int nr = 0; nr < NT; ++nr) {
          const float c0 = __shfl_sync(0xffffffffu, corr[nr], 8 * t);
          const float c1 = __shfl_sync(0xffffffffu, corr[nr], 8 * t + 4);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            O[mt][nr][0] *= c0;
            O[mt][nr][1] *= c1;
            O[mt][nr][2] *= c0;
            O[mt][nr][3] *= c1;
          }
        }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const uint32_t vrow = unitV + frag_row + (uint32_t)(16 * mt) * 128u;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          uint32_t va[4];
          ldsm_x4(vrow + ((uint32_t)((seg0 + 2 * kv) ^ lr) << 4), va);
#pragma unroll
          for (int nr = 0; nr < NT; ++nr) {
            mma_bf16(O[mt][nr], va, ph[kv][nr][0], ph[kv][nr][1]);
            mma_bf16(O[mt][nr], va, pl[kv][nr][0], pl[kv][nr][1]);
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
  if (warp < kConsumers) {
#pragma unroll
    for (int nr = 0; nr < NT; ++nr) {
      float lw = l_run[nr];
      lw += __shfl_xor_sync(0xffffffffu, lw, 1);
      lw += __shfl_xor_sync(0xffffffffu, lw, 2);
      if (t == 0) {
        mm[warp * R + 8 * nr + g] = m_run[nr];
        ml[warp * R + 8 * nr + g] = lw;
      }
    }
  }
  __syncthreads();
  // chunk w's factor of row r, 2^(m_w - m*) (0 where the chunk saw no key of the row)
  if (tid < kConsumers * R) {
    const int r = tid % R;
    float mstar = -CUDART_INF_F;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) mstar = fmaxf(mstar, mm[ww * R + r]);
    const float mw = mm[tid];
    mf[tid] = (mw == -CUDART_INF_F) ? 0.0f : exp2f(mw - mstar);
  }
  __syncthreads();
  if (tid < R) {
    float mstar = -CUDART_INF_F, l = 0.0f;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) {
      mstar = fmaxf(mstar, mm[ww * R + tid]);
      l += ml[ww * R + tid] * mf[ww * R + tid];
    }
    mrow[tid] = make_float2(mstar, l);
  }
  if (warp < kConsumers) {
#pragma unroll
    for (int nr = 0; nr < NT; ++nr) {
      const int r = 8 * nr + 2 * t;
      const float f0 = mf[warp * R + r], f1 = mf[warp * R + r + 1];
      float* dst = mo + (warp * R + r) * MS;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int c0 = 16 * mt + g;
        dst[c0] = O[mt][nr][0] * f0;
        dst[MS + c0] = O[mt][nr][1] * f1;
        dst[c0 + 8] = O[mt][nr][2] * f0;
        dst[MS + c0 + 8] = O[mt][nr][3] * f1;
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < R * kH; i += kThreadsQ) {
    const int r = i >> 7, d = i & 127;
    const int row = row0 + r;
    const int rg4 = row >> 2;
    if (rg4 >= a.n_rg) continue;
    float o = 0.0f;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) o += mo[(ww * R + r) * MS + d];
    const float2 st = mrow[r];
    const int64_t cta = (((int64_t)b * a.Hkv + h) * a.n_rg + rg4) * a.n_splits + split;
    float* ws = a.ws + cta * kWsPerCta;
    ws[(row & 3) * kH + d] = o;
    if (d == 0) {
      ws[kRows * kH + (row & 3)] = st.x;
      ws[kRows * kH + kRows + (row & 3)] = st.y;
    }
  }
}

template <int NT>
cudaError_t launch_bf16(const DecodeArgs& a, cudaStream_t s) {
  constexpr int kSmem = BLayout<NT>::kAlloc;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(decode_bf16_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  CUtensorMap tk, tv;
  if (n_pool_too_large(a.n_pool)) return cudaErrorInvalidValue;
  if (!bf16_page_map(&tk, a.k_bf16, a.n_pool) || !bf16_page_map(&tv, a.v_bf16, a.n_pool))
    return cudaErrorInvalidValue;
  dim3 grid(a.n_splits, a.Hkv * ((a.T * a.G + 8 * NT - 1) / (8 * NT)), a.B);
  return launch_programmatic(decode_bf16_kernel<NT>, grid, dim3(kThreadsQ), kSmem, s, a, tk, tv);
}

}  // namespace

int bf16_rows_per_cta(int rows) { return rows <= 8 ? 8 : 16; }

cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t s) {
  return bf16_rows_per_cta(a.T * a.G) == 8 ? launch_bf16<1>(a, s) : launch_bf16<2>(a, s);
}

}  // namespace lynx
