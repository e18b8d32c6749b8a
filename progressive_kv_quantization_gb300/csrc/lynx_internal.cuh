// Internal definitions shared by the Lynx CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lynx.h"

namespace lynx {

#ifdef __CUDACC__
// Programmatic dependent launch.  A decode kernel calls allow_dependent_launch()
// when its main loop is done, so that the split-combine kernel behind it in the
// stream is scheduled while the last CTAs finish; the combine calls it as it
// starts, so that the next decode call can fill its value tables meanwhile.
// Each of these kernels calls wait_prerequisite_grids() before its first access
// to global memory; it returns once the kernel ahead in the stream has
// completed and its writes are visible.  Where nothing was launched with the
// programmatic attribute both are no-ops.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_prerequisite_grids() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#endif

// Launch of kernel k on stream s as a programmatic dependent of the kernel
// ahead of it in the stream: k may start once that kernel's CTAs have all
// called allow_dependent_launch() (or exited), and must call
// wait_prerequisite_grids() before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
}


// A kernel's bounded wait on a copy or a peer gives up after this long (ns)
// and records an error instead of hanging.
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;

// Page geometry (H channels x P tokens, C-token chunks).
constexpr int kH = 128;
constexpr int kP = 256;
constexpr int kC = 32;
constexpr int kChunks = kP / kC;                       // 8
constexpr int kPageElems = kH * kP;                    // 32768
constexpr int kPlaneBytes = kH * kP / 2;               // 16384: one 4-bit plane
constexpr int kMetaFloats = 2 * kH + 2 * kH * kChunks; // 2304
constexpr int kMetaBytes = kMetaFloats * 4;            // 9216
constexpr int kMetaMuOff = 2 * kH;                     // mu[8][128] (chunk-major) starts here
constexpr int kMetaSigmaOff = 2 * kH + kH * kChunks;   // sigma[8][128]

// Quantiser tables for one (alpha, eps).  thr[k] (k = 1..127) is the smallest
// float32 f with 127 ln(1 + alpha f)/ln(1 + alpha) >= k - 1/2, so that for a
// float32 magnitude a the rounded code is #{k : a >= thr[k]}.  thr[0] = 0 and
// thr[128] = +inf bracket the search.
struct EncodeTables {
  float thr[129];
  float c_lg2;     // 127 / log2(1 + alpha)
  float alpha;
  float eps;
  float edge;      // |y - rint(y)| above which the code is decided from thr[]
};

// Dequantisation tables: signed inverse-compander values S * l(I_hat),
// rounded to float32.
struct LutTables {
  float2 anc_pair[256];  // anchor byte -> (value of low nibble, value of high nibble)
  float full[256];       // (anchor nibble | residual nibble << 4) -> value
  float anc16[16];       // anchor nibble -> value
  float eps;
};

const EncodeTables* encode_tables(float alpha, float eps);
const LutTables* lut_tables(float alpha, float eps);
// the same for the 7-level Lynx-INT4 codes (thr[0..8]; anc16 / anc_pair hold
// S * l4(I4) of the sign-aware nibble) and for Lynx-INT8 bytes (full[byte] =
// S * l(I) of the signed byte S > 0 ? I : -I - 1)
const EncodeTables* encode_tables4(float alpha, float eps);
const LutTables* lut_tables4(float alpha, float eps);
const LutTables* lut_tables8(float alpha, float eps);
// uniform INT-b codes as table values: anc_pair[byte] = (low nibble, high
// nibble) and anc16[v] = v (bits 4), full[byte] = byte (bits 8)
const LutTables* uniform_tables(int bits);

// anchor-only values of an A-bit Anchor (S * l(V 2^R + 2^(R-1) - 1) for the
// A-bit two's-complement code, 2 <= A <= 6), rounded to float32
struct SplitTables {
  float anc[64];
  float eps;
};
const SplitTables* split_tables(float alpha, float eps, int anchor_bits);

// single-precision variants (values of lynx.h's LYNX_VARIANT_*)
enum Variant { kVariantLynxInt8 = 1, kVariantLynxInt4 = 2, kVariantUniformInt8 = 3, kVariantUniformInt4 = 4 };

int device_sm_count();
int set_error(int status, const char* message);   // records lynx_last_error(), returns status
int* device_status_ptr();   // device address of this device's error word

// Launchers (one per kernel family).  Return cudaGetLastError() of the launch.
cudaError_t launch_encode(const void* x, int64_t n_pages, uint8_t* anchor, uint8_t* residual,
                          float* meta, const EncodeTables* tab, const int32_t* valid, cudaStream_t s);
cudaError_t launch_encode_variant(const void* x, int64_t n_pages, int variant, uint8_t* codes, float* meta,
                                  const EncodeTables* tab, cudaStream_t s);
// rows of 256 one-byte codes -> rows of 128 bytes of low nibbles and of high
// nibbles (token 2j in the low nibble of byte j, 2j + 1 in the high one)
cudaError_t launch_split_nibbles(const uint8_t* codes, int64_t n_rows, uint8_t* lo, uint8_t* hi, cudaStream_t s);
cudaError_t launch_reconstruct_variant(const uint8_t* codes, const float* meta, int64_t n_pages, int variant,
                                       void* out, int out_dtype, const LutTables* lut, int* status, cudaStream_t s);
cudaError_t launch_encode_split(const void* x, int64_t n_pages, int anchor_bits, uint8_t* anchor,
                                uint8_t* residual, float* meta, const EncodeTables* tab, cudaStream_t s);
cudaError_t launch_reconstruct_split(const uint8_t* anchor, const uint8_t* residual, const float* meta,
                                     int64_t n_pages, int anchor_bits, void* out, int out_dtype,
                                     const SplitTables* st, const LutTables* lut8, cudaStream_t s);
// wait_ns bounds the waits of the TMA-staged kernel; skip_first (test hook
// only) makes every CTA of it never copy its first item
cudaError_t launch_encode_tokens(const void* x, int64_t n_tokens, int n_heads, int64_t stride,
                                 uint8_t* anchor, uint8_t* residual, float* meta, const EncodeTables* tab,
                                 unsigned long long wait_ns, bool skip_first, cudaStream_t s);
cudaError_t launch_quantize(const float* a, int64_t n, uint8_t* codes, const EncodeTables* tab,
                            cudaStream_t s);
// wait_ns bounds every wait of the staged kernel; skip_unit >= 0 (test hook
// only) makes the producer of every CTA never copy its page skip_unit
cudaError_t launch_reconstruct(const uint8_t* anchor, const uint8_t* residual, const float* meta,
                               int64_t n_pages, void* out, int out_dtype, const LutTables* lut, int* status,
                               unsigned long long wait_ns, int skip_unit, cudaStream_t s);

enum DecodeMode { kModeAnchor = 0, kModeFull = 1, kModeBf16 = 2 };

struct DecodeArgs {
  const uint16_t* q;
  const uint8_t* k_anc;
  const uint8_t* k_res;
  const float* k_meta;
  const uint8_t* v_anc;
  const uint8_t* v_res;
  const float* v_meta;
  const uint16_t* k_bf16;
  const uint16_t* v_bf16;
  const int32_t* page_table;
  const int32_t* ctx_len;
  float* out;
  float* lse;
  float* ws;
  int* status;
  int64_t n_pool;        // pages in each pool (valid page ids are 0 .. n_pool-1)
  int B, T, Hq, Hkv, G, max_pages;
  int n_rg;              // row groups of 4 query rows per (sequence, KV head)
  int n_splits;
  int pages_per_split;
  float scale_log2;      // sm_scale * log2(e)
  int causal;
  float eps;
  // page metadata: Lynx's (gamma_min, gamma_scale, mu, sigma; kMetaFloats per
  // page) or, with `uniform`, a uniform code's (min[128], scale[128]): the value
  // is min + scale * table value for every chunk
  int uniform;
  int meta_floats;
  float code_max;        // the largest |table value| (1 for Lynx's l~)
  // every bounded wait of the quantised decode kernels gives up after wait_ns
  // nanoseconds (two seconds unless the test hook lynx_test_inject_wait_timeout
  // armed this call); with inject_skip > 0 (test hook only) the producer never
  // issues the copy of unit inject_skip - 1 of its split, so that wait runs out
  unsigned long long wait_ns;
  int inject_skip;
};

struct DecodePlan {
  int n_rg;
  int n_splits;
  int pages_per_split;
  size_t ws_bytes;
};

DecodePlan plan_decode(int B, int T, int Hq, int Hkv, int max_pages, int mode);
bool n_pool_too_large(int64_t n_pool);
// tensor-core decode kernel: used for `rows` = T * (Hq / Hkv) query rows per
// (sequence, KV head) when use_tc_rows(rows); one CTA takes
// tc_rows_per_cta(rows, full) of them.  Fewer rows go to the narrow tensor-core
// kernel, kNarrowRows per CTA.
bool use_tc_rows(int rows);
int tc_rows_per_cta(int rows, bool full);
constexpr int kNarrowRows = 8;
cudaError_t launch_decode_narrow(const DecodeArgs& a, bool full, const LutTables* lut, cudaStream_t s);
// the draft decode kernel: Anchor planes with Lynx metadata and a table of
// values |l~| < 1, fewer than 12 query rows per KV head (8 per CTA)
cudaError_t launch_decode_draft(const DecodeArgs& a, const LutTables* lut, cudaStream_t s);
// BF16 pages (the baseline): one CTA takes bf16_rows_per_cta(rows) query rows
// of a (sequence, KV head), 8 or 16
int bf16_rows_per_cta(int rows);
cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_tc(const DecodeArgs& a, bool full, const LutTables* lut, cudaStream_t s);
cudaError_t launch_decode_quant(const DecodeArgs& a, bool full, const LutTables* lut, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, int mode, const LutTables* lut, cudaStream_t s);
cudaError_t launch_attn_merge(const float* oa, const float* la, const float* ob, const float* lb,
                              int64_t rows, float* o, float* lse, cudaStream_t s);

}  // namespace lynx
