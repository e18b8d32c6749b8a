// lynx_decode_attn_noalloc: the decode / verification attention of
// lynx_decode_attn for callers that cannot allocate device memory.
//
// Who needs it: code that holds no allocator of its own -- for instance a KV
// transfer connector or deserializer plugin that a serving engine loads with a
// fixed device-memory budget, or a decode loop that must not call
// cudaMalloc / cudaFree because those calls synchronise the device and stall
// the streams it is overlapping.  Such a caller still owns the query, page
// pools, page table, context lengths and outputs, but cannot hand over the
// split-K scratch buffer that lynx_decode_attn takes as `workspace`.
//
// How: the scratch lives in this file's static device array g_noalloc_scratch
// (kNoAllocScratchBytes, 8 MiB, held by every GPU that loads the library until
// the process exits).  In host code that name is only a host-side stand-in for
// the device symbol, so the entry point resolves the array's device address
// with cudaGetSymbolAddress once per device (with that device current, on the
// first call made on it) and passes that address to lynx_decode_attn as the
// workspace.  Nothing here calls cudaMalloc, cudaFree or any allocating routine.

#include <mutex>

#include "lynx_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[64];    // device address of g_noalloc_scratch, per device

}  // namespace

extern "C" int lynx_decode_attn_noalloc(const void* q_bf16, int B, int T, int Hq, int Hkv,
                                        int head_dim, const uint8_t* k_anc, const uint8_t* k_res,
                                        const float* k_meta, const uint8_t* v_anc,
                                        const uint8_t* v_res, const float* v_meta,
                                        int64_t n_pool_pages, const int32_t* page_table,
                                        int max_pages, const int32_t* ctx_len,
                                        const lynx_params_t* params, float sm_scale, int causal,
                                        float* out, float* lse, void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return lynx::set_error(LYNX_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return lynx::set_error(LYNX_ERR_UNSUPPORTED, "device index >= 64");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr)
        return lynx::set_error(LYNX_ERR_CUDA, "cudaGetSymbolAddress of the no-allocation scratch failed");
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  const size_t need = lynx_decode_attn_workspace_size(B, T, Hq, Hkv, head_dim, max_pages);
  if (need > kNoAllocScratchBytes)
    return lynx::set_error(LYNX_ERR_WORKSPACE,
                           "this shape needs more split-K scratch than the 8 MiB the "
                           "no-allocation entry point holds; use lynx_decode_attn");
  return lynx_decode_attn(q_bf16, B, T, Hq, Hkv, head_dim, k_anc, k_res, k_meta, v_anc, v_res,
                          v_meta, n_pool_pages, page_table, max_pages, ctx_len, params, sm_scale,
                          causal, out, lse, scratch, kNoAllocScratchBytes, stream);
}
