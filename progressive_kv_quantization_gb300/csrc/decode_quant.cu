// Dispatch of the decode / verification attention over Lynx-encoded pages
// (the attention of the Lynx paper's §2.1 over the KV that the Anchor and
// Residual phases of §4.2-4.3 deliver) to its tensor-core kernels, and the
// TMA tensor maps the decode kernels use to stream the 4-bit planes and the
// BF16 pages.
//
//   fewer than 12 query rows per KV head  decode_draft_kernel over Anchor planes
//                                          with Lynx metadata (the draft decode at
//                                          T = 1), else decode_narrow_kernel;
//                                          8 rows per CTA
//   12 or more                             decode_tc_kernel, 16 or 32 rows per CTA
//                                          (the T-token verification)

#include "decode_common.cuh"

namespace lynx {
namespace {

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

}  // namespace

bool plane_map(CUtensorMap* m, const uint8_t* pool, int64_t n_pool) {
  // a decode loop passes the same pools call after call: the last few maps of
  // this host thread are kept (a map depends only on the address and size)
  struct Entry {
    const uint8_t* pool;
    int64_t n_pool;
    CUtensorMap map;
  };
  constexpr int kEntries = 8;
  thread_local Entry cache[kEntries];
  thread_local int next = 0;
  for (int i = 0; i < kEntries; ++i)
    if (cache[i].pool == pool && cache[i].n_pool == n_pool && pool != nullptr) {
      *m = cache[i].map;
      return true;
    }
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {128, (cuuint64_t)n_pool * kH};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t estr[2] = {1, 1};
  const bool ok = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(pool), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  if (ok) {
    cache[next] = Entry{pool, n_pool, *m};
    next = (next + 1) % kEntries;
  }
  return ok;
}

bool bf16_page_map(CUtensorMap* m, const uint16_t* pool, int64_t n_pool) {
  struct Entry {
    const uint16_t* pool;
    int64_t n_pool;
    CUtensorMap map;
  };
  constexpr int kEntries = 8;
  thread_local Entry cache[kEntries];
  thread_local int next = 0;
  for (int i = 0; i < kEntries; ++i)
    if (cache[i].pool == pool && cache[i].n_pool == n_pool && pool != nullptr) {
      *m = cache[i].map;
      return true;
    }
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {kP, (cuuint64_t)n_pool * kH};
  const cuuint64_t strides[1] = {kP * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  const bool ok = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(pool), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  if (ok) {
    cache[next] = Entry{pool, n_pool, *m};
    next = (next + 1) % kEntries;
  }
  return ok;
}

bool token_map(CUtensorMap* m, const void* x, int64_t n_tokens, int64_t row_elems, int64_t stride) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0 || stride % 8 != 0 || row_elems % 64 != 0) return false;
  // TMA coordinates are signed 32-bit: the channel and token offsets must fit
  if (row_elems > ((int64_t)1 << 31) - 64 || n_tokens > ((int64_t)1 << 31) - 256) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)n_tokens};
  const cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
  const cuuint32_t box[2] = {64, 256};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// the TMA row coordinate (page id * 128) is a signed 32-bit value
bool n_pool_too_large(int64_t n_pool) { return n_pool <= 0 || n_pool * kH > ((int64_t)1 << 31) - 1; }

cudaError_t launch_decode_quant(const DecodeArgs& a, bool full, const LutTables* lut, cudaStream_t s) {
  if (use_tc_rows(a.T * a.G)) return launch_decode_tc(a, full, lut, s);
  if (!full && !a.uniform) return launch_decode_draft(a, lut, s);
  return launch_decode_narrow(a, full, lut, s);
}

}  // namespace lynx
