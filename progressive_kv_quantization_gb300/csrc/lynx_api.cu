// C ABI of the Lynx hot path: argument checks, per-(alpha, eps) tables,
// the device error word, and kernel launches.  See include/lynx.h.

#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "lynx_internal.cuh"

namespace lynx {

namespace {

thread_local char g_last_error[512] = "";

// calls of this host thread still to run with the wait time-out injected
// (lynx_test_inject_wait_timeout): token encode, reconstruct and decode
thread_local int g_inject_calls = 0;

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(LYNX_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

int check_params(const lynx_params_t* p) {
  if (p == nullptr) return fail(LYNX_ERR_INVALID_ARG, "params is NULL");
  if (p->H != kH || p->P != kP || p->C != kC)
    return fail(LYNX_ERR_UNSUPPORTED, "unsupported page shape H=%d P=%d C=%d (need 128, 256, 32)",
                p->H, p->P, p->C);
  if (!(p->alpha >= 0.25f && p->alpha <= 1e6f))
    return fail(LYNX_ERR_UNSUPPORTED, "alpha=%g outside [0.25, 1e6]", (double)p->alpha);
  if (!(p->eps > 0.0f && p->eps <= 1e-2f))
    return fail(LYNX_ERR_UNSUPPORTED, "eps=%g outside (0, 1e-2]", (double)p->eps);
  return LYNX_OK;
}

double ell(double y, double alpha) {  // inverse compander ((1+alpha)^(y/127) - 1)/alpha
  return expm1(y / 127.0 * log1p(alpha)) / alpha;
}
double ell4(double y, double alpha) {  // the same for 7 levels ((1+alpha)^(y/7) - 1)/alpha
  return expm1(y / 7.0 * log1p(alpha)) / alpha;
}

// smallest float32 >= x
float round_up_f32(double x) {
  float f = (float)x;
  if ((double)f < x) f = nextafterf(f, INFINITY);
  return f;
}

// Margin around a rounding edge inside which the code is decided from the
// table, for an estimate c * log2(1 + alpha a).  The hardware log2's absolute
// error on [1, 2^20) stays below 2^-21 * max(1, log2(t)) (measured over every
// float32 t in that range: at most 2^-22.5 below 4, 2^-20.9 below 256, 2^-19
// below 2^20); the rounding of 1 + alpha a, of c and of the product add at most
// c * 1e-7 + 1.6e-5; a magnitude estimate within a relative 2^-22 of the exact
// one (the encoder's a = RN(x RN(1/d))) moves the estimate by at most
// c 2^-22 / ln 2 < c * 3.5e-7.  The margin is twice the sum.
float rounding_edge(double c, double alpha) {
  const double L = log2(1.0 + alpha);
  const double err = c * (ldexp(1.0, -21) * (L > 1.0 ? L : 1.0) + 1e-7 + 3.5e-7) + 1.6e-5;
  return (float)(0.5 - 2.0 * err);
}

__device__ int g_status;   // per-device error word set by kernels that give up a wait

std::mutex g_dev_mutex;
int g_sm_count[64];
int* g_status_ptr[64];

int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}

}  // namespace

const EncodeTables* encode_tables(float alpha, float eps) {
  thread_local EncodeTables tab;
  thread_local float cached_alpha = -1.0f, cached_eps = -1.0f;
  if (alpha == cached_alpha && eps == cached_eps) return &tab;
  const double a = alpha;
  tab.thr[0] = 0.0f;
  for (int k = 1; k <= 127; ++k) tab.thr[k] = round_up_f32(ell(k - 0.5, a));   // edge between codes k-1, k
  tab.thr[128] = INFINITY;
  const double c = 127.0 / log2(1.0 + a);
  tab.c_lg2 = (float)c;
  tab.alpha = alpha;
  tab.eps = eps;
  tab.edge = rounding_edge(c, a);
  cached_alpha = alpha;
  cached_eps = eps;
  return &tab;
}

const EncodeTables* encode_tables4(float alpha, float eps) {
  thread_local EncodeTables tab;
  thread_local float cached_alpha = -1.0f, cached_eps = -1.0f;
  if (alpha == cached_alpha && eps == cached_eps) return &tab;
  const double a = alpha;
  tab.thr[0] = 0.0f;
  for (int k = 1; k <= 7; ++k) tab.thr[k] = round_up_f32(ell4(k - 0.5, a));
  for (int k = 8; k <= 128; ++k) tab.thr[k] = INFINITY;
  const double c = 7.0 / log2(1.0 + a);
  tab.c_lg2 = (float)c;
  tab.alpha = alpha;
  tab.eps = eps;
  tab.edge = rounding_edge(c, a);
  cached_alpha = alpha;
  cached_eps = eps;
  return &tab;
}

const LutTables* lut_tables(float alpha, float eps) {
  thread_local LutTables lut;
  thread_local float cached_alpha = -1.0f, cached_eps = -1.0f;
  if (alpha == cached_alpha && eps == cached_eps) return &lut;
  const double a = alpha;
  for (int n = 0; n < 16; ++n) {
    const int q = n >= 8 ? n - 16 : n;           // two's-complement anchor
    const int S = q < 0 ? -1 : 1;
    const int V = S > 0 ? q : -q - 1;
    lut.anc16[n] = (float)(S * ell(16 * V + 7, a));
  }
  for (int c = 0; c < 256; ++c) {
    const int na = c & 15, nr = c >> 4;
    const int qa = na >= 8 ? na - 16 : na;
    const int qr = nr >= 8 ? nr - 16 : nr;
    const int S = qa < 0 ? -1 : 1;
    const int V = S > 0 ? qa : -qa - 1;
    lut.full[c] = (float)(S * ell(16 * V + 7 - qr, a));
  }
  for (int byte = 0; byte < 256; ++byte)
    lut.anc_pair[byte] = make_float2(lut.anc16[byte & 15], lut.anc16[byte >> 4]);
  lut.eps = eps;
  cached_alpha = alpha;
  cached_eps = eps;
  return &lut;
}

const LutTables* lut_tables4(float alpha, float eps) {
  thread_local LutTables lut;
  thread_local float cached_alpha = -1.0f, cached_eps = -1.0f;
  if (alpha == cached_alpha && eps == cached_eps) return &lut;
  const double a = alpha;
  for (int n = 0; n < 16; ++n) {
    const int q = n >= 8 ? n - 16 : n;           // sign-aware nibble S > 0 ? I4 : -I4 - 1
    const int S = q < 0 ? -1 : 1;
    const int I4 = S > 0 ? q : -q - 1;
    lut.anc16[n] = (float)(S * ell4(I4, a));
  }
  for (int c = 0; c < 256; ++c) lut.full[c] = 0.0f;
  for (int byte = 0; byte < 256; ++byte)
    lut.anc_pair[byte] = make_float2(lut.anc16[byte & 15], lut.anc16[byte >> 4]);
  lut.eps = eps;
  cached_alpha = alpha;
  cached_eps = eps;
  return &lut;
}

const LutTables* uniform_tables(int bits) {
  static LutTables t4, t8;
  static bool built = false;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  if (!built) {
    for (int v = 0; v < 16; ++v) t4.anc16[v] = (float)v;
    for (int byte = 0; byte < 256; ++byte) {
      t4.anc_pair[byte] = make_float2((float)(byte & 15), (float)(byte >> 4));
      t4.full[byte] = 0.0f;
      t8.full[byte] = (float)byte;
      t8.anc_pair[byte] = make_float2(0.0f, 0.0f);
    }
    for (int v = 0; v < 16; ++v) t8.anc16[v] = 0.0f;
    t4.eps = t8.eps = 0.0f;
    built = true;
  }
  return bits == 8 ? &t8 : &t4;
}

const LutTables* lut_tables8(float alpha, float eps) {
  thread_local LutTables lut;
  thread_local float cached_alpha = -1.0f, cached_eps = -1.0f;
  if (alpha == cached_alpha && eps == cached_eps) return &lut;
  const double a = alpha;
  for (int b = 0; b < 256; ++b) {
    const int q = b >= 128 ? b - 256 : b;        // signed byte S > 0 ? I : -I - 1
    const int S = q < 0 ? -1 : 1;
    const int I = S > 0 ? q : -q - 1;
    lut.full[b] = (float)(S * ell(I, a));
  }
  for (int n = 0; n < 16; ++n) lut.anc16[n] = 0.0f;
  for (int byte = 0; byte < 256; ++byte) lut.anc_pair[byte] = make_float2(0.0f, 0.0f);
  lut.eps = eps;
  cached_alpha = alpha;
  cached_eps = eps;
  return &lut;
}

const SplitTables* split_tables(float alpha, float eps, int anchor_bits) {
  thread_local SplitTables st;
  thread_local float cached_alpha = -1.0f, cached_eps = -1.0f;
  thread_local int cached_bits = -1;
  if (alpha == cached_alpha && eps == cached_eps && anchor_bits == cached_bits) return &st;
  const int A = anchor_bits, R = 8 - A;
  for (int n = 0; n < 64; ++n) st.anc[n] = 0.0f;
  for (int n = 0; n < (1 << A); ++n) {
    const int q = n >= (1 << (A - 1)) ? n - (1 << A) : n;   // A-bit two's complement
    const int S = q < 0 ? -1 : 1;
    const int V = S > 0 ? q : -q - 1;
    st.anc[n] = (float)(S * ell((V << R) + (1 << (R - 1)) - 1, alpha));
  }
  st.eps = eps;
  cached_alpha = alpha;
  cached_eps = eps;
  cached_bits = anchor_bits;
  return &st;
}

int set_error(int status, const char* message) { return fail(status, "%s", message); }

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lk(g_dev_mutex);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sm_count[dev] = n > 0 ? n : 1;
  }
  return g_sm_count[dev];
}

int* device_status_ptr() {
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mutex);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

}  // namespace lynx

using namespace lynx;

extern "C" {

int lynx_version(void) { return 100; }

const char* lynx_last_error(void) { return g_last_error; }

const char* lynx_status_string(int status) {
  switch (status) {
    case LYNX_OK: return "LYNX_OK";
    case LYNX_ERR_INVALID_ARG: return "LYNX_ERR_INVALID_ARG";
    case LYNX_ERR_UNSUPPORTED: return "LYNX_ERR_UNSUPPORTED";
    case LYNX_ERR_ALIGNMENT: return "LYNX_ERR_ALIGNMENT";
    case LYNX_ERR_WORKSPACE: return "LYNX_ERR_WORKSPACE";
    case LYNX_ERR_CUDA: return "LYNX_ERR_CUDA";
    case LYNX_ERR_DEVICE: return "LYNX_ERR_DEVICE";
    default: return "LYNX_ERR_UNKNOWN";
  }
}

namespace {

int encode_common(const void* x_bf16, int64_t n_pages, const int32_t* valid, const lynx_params_t* params,
                  uint8_t* anchor, uint8_t* residual, float* meta, void* stream, const char* name) {
  g_last_error[0] = '\0';
  int st = check_params(params);
  if (st != LYNX_OK) return st;
  if (n_pages < 0) return fail(LYNX_ERR_INVALID_ARG, "n_pages=%lld < 0", (long long)n_pages);
  if (n_pages == 0) return LYNX_OK;
  if (!x_bf16 || !anchor || !residual || !meta)
    return fail(LYNX_ERR_INVALID_ARG, "NULL buffer pointer");
  if (misaligned(x_bf16) || misaligned(anchor) || misaligned(residual) || misaligned(meta) ||
      (valid && misaligned(valid)))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  if (n_pages > ((int64_t)1 << 40)) return fail(LYNX_ERR_INVALID_ARG, "n_pages too large");
  const EncodeTables* tab = encode_tables(params->alpha, params->eps);
  cudaError_t e = launch_encode(x_bf16, n_pages, anchor, residual, meta, tab, valid,
                                static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, name);
  return LYNX_OK;
}

}  // namespace

int lynx_encode_pages(const void* x_bf16, int64_t n_pages, const lynx_params_t* params,
                      uint8_t* anchor, uint8_t* residual, float* meta, void* stream) {
  return encode_common(x_bf16, n_pages, nullptr, params, anchor, residual, meta, stream,
                       "lynx_encode_pages launch");
}

int lynx_encode_pages_partial(const void* x_bf16, int64_t n_pages, const int32_t* valid_tokens,
                              const lynx_params_t* params, uint8_t* anchor, uint8_t* residual,
                              float* meta, void* stream) {
  if (!valid_tokens && n_pages > 0) {
    g_last_error[0] = '\0';
    return fail(LYNX_ERR_INVALID_ARG, "NULL valid_tokens");
  }
  return encode_common(x_bf16, n_pages, valid_tokens, params, anchor, residual, meta, stream,
                       "lynx_encode_pages_partial launch");
}

int lynx_encode_tokens(const void* x_bf16, int64_t n_tokens, int n_heads, int64_t token_stride,
                       const lynx_params_t* params, uint8_t* anchor, uint8_t* residual, float* meta,
                       void* stream) {
  g_last_error[0] = '\0';
  int st = check_params(params);
  if (st != LYNX_OK) return st;
  if (n_tokens < 0 || n_heads < 0)
    return fail(LYNX_ERR_INVALID_ARG, "n_tokens=%lld, n_heads=%d", (long long)n_tokens, n_heads);
  if (n_tokens == 0 || n_heads == 0) return LYNX_OK;
  if (token_stride < (int64_t)n_heads * 128)
    return fail(LYNX_ERR_INVALID_ARG, "token_stride=%lld < n_heads * 128", (long long)token_stride);
  if (!x_bf16 || !anchor || !residual || !meta) return fail(LYNX_ERR_INVALID_ARG, "NULL buffer pointer");
  if ((reinterpret_cast<uintptr_t>(x_bf16) & 1u) != 0)
    return fail(LYNX_ERR_ALIGNMENT, "x must be 2-byte aligned");
  if (misaligned(anchor) || misaligned(residual) || misaligned(meta))
    return fail(LYNX_ERR_ALIGNMENT, "anchor, residual and meta must be 16-byte aligned");
  if (n_tokens > ((int64_t)1 << 40) || (int64_t)n_heads * ((n_tokens + 255) / 256) > ((int64_t)1 << 40))
    return fail(LYNX_ERR_INVALID_ARG, "too many tokens");
  const EncodeTables* tab = encode_tables(params->alpha, params->eps);
  unsigned long long wait_ns = kDefaultWaitNs;
  bool skip_first = false;
  if (g_inject_calls > 0) {   // test hook, off unless armed
    --g_inject_calls;
    skip_first = true;      // the first item of every CTA is never copied
    wait_ns = 1000000ull;   // and every wait gives up after 1 ms
  }
  cudaError_t e = launch_encode_tokens(x_bf16, n_tokens, n_heads, token_stride, anchor, residual, meta, tab,
                                       wait_ns, skip_first, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lynx_encode_tokens launch");
  return LYNX_OK;
}

int lynx_quantize_magnitudes(const float* a, int64_t n, const lynx_params_t* params,
                             uint8_t* codes, void* stream) {
  g_last_error[0] = '\0';
  int st = check_params(params);
  if (st != LYNX_OK) return st;
  if (n < 0) return fail(LYNX_ERR_INVALID_ARG, "n=%lld < 0", (long long)n);
  if (n == 0) return LYNX_OK;
  if (!a || !codes) return fail(LYNX_ERR_INVALID_ARG, "NULL buffer pointer");
  if (misaligned(a) || misaligned(codes)) return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  const EncodeTables* tab = encode_tables(params->alpha, params->eps);
  cudaError_t e = launch_quantize(a, n, codes, tab, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lynx_quantize_magnitudes launch");
  return LYNX_OK;
}

int lynx_reconstruct(const uint8_t* anchor, const uint8_t* residual, const float* meta,
                     int64_t n_pages, const lynx_params_t* params, void* out, int out_dtype,
                     void* stream) {
  g_last_error[0] = '\0';
  int st = check_params(params);
  if (st != LYNX_OK) return st;
  if (out_dtype != LYNX_OUT_BF16 && out_dtype != LYNX_OUT_F32)
    return fail(LYNX_ERR_INVALID_ARG, "out_dtype=%d (need 0 = BF16 or 1 = F32)", out_dtype);
  if (n_pages < 0) return fail(LYNX_ERR_INVALID_ARG, "n_pages=%lld < 0", (long long)n_pages);
  if (n_pages == 0) return LYNX_OK;
  if (!anchor || !meta || !out) return fail(LYNX_ERR_INVALID_ARG, "NULL buffer pointer");
  if (misaligned(anchor) || (residual && misaligned(residual)) || misaligned(meta) || misaligned(out))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  if (n_pages > ((int64_t)1 << 40)) return fail(LYNX_ERR_INVALID_ARG, "n_pages too large");
  const LutTables* lut = lut_tables(params->alpha, params->eps);
  int* status = device_status_ptr();
  if (!status) return fail(LYNX_ERR_CUDA, "cannot resolve the device status word");
  unsigned long long wait_ns = kDefaultWaitNs;
  int skip_unit = -1;
  if (g_inject_calls > 0) {   // test hook, off unless armed
    --g_inject_calls;
    skip_unit = 0;          // the first page of every CTA is never copied
    wait_ns = 1000000ull;   // and every wait gives up after 1 ms
  }
  cudaError_t e = launch_reconstruct(anchor, residual, meta, n_pages, out, out_dtype, lut, status, wait_ns,
                                     skip_unit, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lynx_reconstruct launch");
  return LYNX_OK;
}

namespace {


int check_decode_shape(int B, int T, int Hq, int Hkv, int head_dim, int max_pages) {
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || max_pages < 1)
    return fail(LYNX_ERR_INVALID_ARG, "B=%d T=%d Hq=%d Hkv=%d max_pages=%d must be >= 1", B, T, Hq,
                Hkv, max_pages);
  if (head_dim != kH) return fail(LYNX_ERR_UNSUPPORTED, "head_dim=%d (need 128)", head_dim);
  // the Lynx paper (§6.1) drafts at most 64 tokens, all verified in one pass
  if (T > 64) return fail(LYNX_ERR_UNSUPPORTED, "T=%d > 64", T);
  if (Hq % Hkv != 0) return fail(LYNX_ERR_INVALID_ARG, "Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
  const int G = Hq / Hkv;
  if (T * G > 256) return fail(LYNX_ERR_UNSUPPORTED, "T*Hq/Hkv=%d > 256", T * G);
  const int n_rg = (T * G + 3) / 4;
  if (B > 65535 || (int64_t)Hkv * n_rg > 65535)
    return fail(LYNX_ERR_UNSUPPORTED, "grid too large (B=%d, Hkv*row_groups=%lld)", B,
                (long long)Hkv * n_rg);
  if ((int64_t)max_pages * kP > 0x7fffffff) return fail(LYNX_ERR_UNSUPPORTED, "max_pages too large");
  return LYNX_OK;
}

int decode_common(DecodeArgs& a, int mode, const void* q, int B, int T, int Hq, int Hkv,
                  int head_dim, int64_t n_pool, const int32_t* page_table, int max_pages,
                  const int32_t* ctx_len, float sm_scale, int causal, float* out, float* lse,
                  void* workspace, size_t ws_bytes, float alpha, float eps, void* stream,
                  bool int4 = false, const LutTables* uniform_lut = nullptr) {
  int st = check_decode_shape(B, T, Hq, Hkv, head_dim, max_pages);
  if (st != LYNX_OK) return st;
  if (!q || !page_table || !ctx_len || !out) return fail(LYNX_ERR_INVALID_ARG, "NULL buffer pointer");
  if (n_pool < 1) return fail(LYNX_ERR_INVALID_ARG, "n_pool_pages=%lld < 1", (long long)n_pool);
  if (misaligned(q) || misaligned(page_table) || misaligned(ctx_len) || misaligned(out) ||
      (lse && misaligned(lse)) || (workspace && misaligned(workspace)))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  if (causal != 0 && causal != 1) return fail(LYNX_ERR_INVALID_ARG, "causal=%d", causal);
  if (!(sm_scale > 0.0f) || !isfinite(sm_scale))
    return fail(LYNX_ERR_INVALID_ARG, "sm_scale=%g must be finite and > 0", (double)sm_scale);
  const DecodePlan pl = plan_decode(B, T, Hq, Hkv, max_pages, mode);
  if (workspace == nullptr || ws_bytes < pl.ws_bytes)
    return fail(LYNX_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", pl.ws_bytes,
                workspace ? ws_bytes : (size_t)0);
  int* status = device_status_ptr();
  if (!status) return fail(LYNX_ERR_CUDA, "cannot resolve the device status word");
  a.q = static_cast<const uint16_t*>(q);
  a.page_table = page_table;
  a.ctx_len = ctx_len;
  a.out = out;
  a.lse = lse;
  a.ws = static_cast<float*>(workspace);
  a.status = status;
  a.n_pool = n_pool;
  a.B = B;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.max_pages = max_pages;
  a.n_rg = pl.n_rg;
  a.n_splits = pl.n_splits;
  a.pages_per_split = pl.pages_per_split;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.causal = causal;
  a.eps = eps;
  if (a.meta_floats == 0) {   // Lynx metadata unless the caller set the uniform form
    a.uniform = 0;
    a.meta_floats = kMetaFloats;
    a.code_max = 1.0f;
  }
  a.wait_ns = kDefaultWaitNs;
  if (g_inject_calls > 0) {   // test hook, off unless armed
    --g_inject_calls;
    a.inject_skip = 2;       // the first V unit of every split is never copied
    a.wait_ns = 1000000ull;  // and every wait gives up after 1 ms
  }
  const LutTables* lut = uniform_lut ? uniform_lut : int4 ? lut_tables4(alpha, eps) : lut_tables(alpha, eps);
  cudaError_t e = launch_decode(a, mode, lut, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lynx_decode_attn launch");
  return LYNX_OK;
}

}  // namespace

size_t lynx_decode_attn_workspace_size(int B, int T, int Hq, int Hkv, int head_dim, int max_pages) {
  if (check_decode_shape(B, T, Hq, Hkv, head_dim, max_pages) != LYNX_OK) return 0;
  // the split count depends on the kind of pages (rows per CTA differ), so the
  // size covers all three
  size_t ws = 0;
  for (int mode : {kModeAnchor, kModeFull, kModeBf16}) {
    const size_t m = plan_decode(B, T, Hq, Hkv, max_pages, mode).ws_bytes;
    ws = m > ws ? m : ws;
  }
  return ws;
}

int lynx_decode_attn(const void* q_bf16, int B, int T, int Hq, int Hkv, int head_dim,
                     const uint8_t* k_anc, const uint8_t* k_res, const float* k_meta,
                     const uint8_t* v_anc, const uint8_t* v_res, const float* v_meta,
                     int64_t n_pool_pages, const int32_t* page_table, int max_pages,
                     const int32_t* ctx_len, const lynx_params_t* params, float sm_scale,
                     int causal, float* out, float* lse, void* workspace, size_t workspace_bytes,
                     void* stream) {
  g_last_error[0] = '\0';
  int st = check_params(params);
  if (st != LYNX_OK) return st;
  if (!k_anc || !k_meta || !v_anc || !v_meta) return fail(LYNX_ERR_INVALID_ARG, "NULL page pool");
  if ((k_res == nullptr) != (v_res == nullptr))
    return fail(LYNX_ERR_INVALID_ARG, "k_res and v_res must both be NULL or both be set");
  if (misaligned(k_anc) || misaligned(k_meta) || misaligned(v_anc) || misaligned(v_meta) ||
      (k_res && misaligned(k_res)) || (v_res && misaligned(v_res)))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  DecodeArgs a{};
  a.k_anc = k_anc;
  a.k_res = k_res;
  a.k_meta = k_meta;
  a.v_anc = v_anc;
  a.v_res = v_res;
  a.v_meta = v_meta;
  const int mode = k_res ? kModeFull : kModeAnchor;
  return decode_common(a, mode, q_bf16, B, T, Hq, Hkv, head_dim, n_pool_pages, page_table,
                       max_pages, ctx_len, sm_scale, causal, out, lse, workspace, workspace_bytes,
                       params->alpha, params->eps, stream);
}

int lynx_decode_attn_int4(const void* q_bf16, int B, int T, int Hq, int Hkv, int head_dim,
                          const uint8_t* k_codes, const float* k_meta, const uint8_t* v_codes,
                          const float* v_meta, int64_t n_pool_pages, const int32_t* page_table, int max_pages,
                          const int32_t* ctx_len, const lynx_params_t* params, float sm_scale, int causal,
                          float* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  g_last_error[0] = '\0';
  int st = check_params(params);
  if (st != LYNX_OK) return st;
  if (!k_codes || !k_meta || !v_codes || !v_meta) return fail(LYNX_ERR_INVALID_ARG, "NULL page pool");
  if (misaligned(k_codes) || misaligned(k_meta) || misaligned(v_codes) || misaligned(v_meta))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  DecodeArgs a{};
  a.k_anc = k_codes;
  a.k_meta = k_meta;
  a.v_anc = v_codes;
  a.v_meta = v_meta;
  return decode_common(a, kModeAnchor, q_bf16, B, T, Hq, Hkv, head_dim, n_pool_pages, page_table, max_pages,
                       ctx_len, sm_scale, causal, out, lse, workspace, workspace_bytes, params->alpha,
                       params->eps, stream, true);
}

int lynx_decode_attn_uniform(const void* q_bf16, int B, int T, int Hq, int Hkv, int head_dim, int bits,
                             const uint8_t* k_lo, const uint8_t* k_hi, const float* k_meta, const uint8_t* v_lo,
                             const uint8_t* v_hi, const float* v_meta, int64_t n_pool_pages,
                             const int32_t* page_table, int max_pages, const int32_t* ctx_len, float sm_scale,
                             int causal, float* out, float* lse, void* workspace, size_t workspace_bytes,
                             void* stream) {
  g_last_error[0] = '\0';
  if (bits != 4 && bits != 8) return fail(LYNX_ERR_INVALID_ARG, "bits=%d (need 4 or 8)", bits);
  if (!k_lo || !k_meta || !v_lo || !v_meta) return fail(LYNX_ERR_INVALID_ARG, "NULL page pool");
  if (bits == 8 && (!k_hi || !v_hi))
    return fail(LYNX_ERR_INVALID_ARG, "bits=8 needs the high-nibble planes k_hi and v_hi");
  if (bits == 4 && (k_hi || v_hi)) return fail(LYNX_ERR_INVALID_ARG, "bits=4 takes no high-nibble planes");
  if (misaligned(k_lo) || misaligned(k_meta) || misaligned(v_lo) || misaligned(v_meta) ||
      (k_hi && misaligned(k_hi)) || (v_hi && misaligned(v_hi)))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  DecodeArgs a{};
  a.k_anc = k_lo;
  a.k_res = k_hi;
  a.k_meta = k_meta;
  a.v_anc = v_lo;
  a.v_res = v_hi;
  a.v_meta = v_meta;
  a.uniform = 1;
  a.meta_floats = 2 * kH;
  a.code_max = bits == 8 ? 255.0f : 15.0f;
  return decode_common(a, bits == 8 ? kModeFull : kModeAnchor, q_bf16, B, T, Hq, Hkv, head_dim, n_pool_pages,
                       page_table, max_pages, ctx_len, sm_scale, causal, out, lse, workspace, workspace_bytes,
                       100.0f, 1e-6f, stream, false, uniform_tables(bits));
}

int lynx_split_nibbles(const uint8_t* codes, int64_t n_rows, uint8_t* lo, uint8_t* hi, void* stream) {
  g_last_error[0] = '\0';
  if (n_rows < 0) return fail(LYNX_ERR_INVALID_ARG, "n_rows=%lld < 0", (long long)n_rows);
  if (n_rows == 0) return LYNX_OK;
  if (!codes || !lo || !hi) return fail(LYNX_ERR_INVALID_ARG, "NULL buffer pointer");
  if (misaligned(codes) || misaligned(lo) || misaligned(hi))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  if (n_rows > ((int64_t)1 << 40)) return fail(LYNX_ERR_INVALID_ARG, "n_rows too large");
  cudaError_t e = launch_split_nibbles(codes, n_rows, lo, hi, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lynx_split_nibbles launch");
  return LYNX_OK;
}

int lynx_encode_variant(const void* x_bf16, int64_t n_pages, int variant, const lynx_params_t* params,
                        uint8_t* codes, float* meta, void* stream) {
  g_last_error[0] = '\0';
  if (variant < LYNX_VARIANT_LYNX_INT8 || variant > LYNX_VARIANT_UNIFORM_INT4)
    return fail(LYNX_ERR_INVALID_ARG, "variant=%d", variant);
  const bool lynx_kind = variant == LYNX_VARIANT_LYNX_INT8 || variant == LYNX_VARIANT_LYNX_INT4;
  if (lynx_kind) {
    int st = check_params(params);
    if (st != LYNX_OK) return st;
  }
  if (n_pages < 0) return fail(LYNX_ERR_INVALID_ARG, "n_pages=%lld < 0", (long long)n_pages);
  if (n_pages == 0) return LYNX_OK;
  if (!x_bf16 || !codes || !meta) return fail(LYNX_ERR_INVALID_ARG, "NULL buffer pointer");
  if (misaligned(x_bf16) || misaligned(codes) || misaligned(meta))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  if (n_pages > ((int64_t)1 << 40)) return fail(LYNX_ERR_INVALID_ARG, "n_pages too large");
  const EncodeTables* tab = nullptr;
  if (variant == LYNX_VARIANT_LYNX_INT8) tab = encode_tables(params->alpha, params->eps);
  if (variant == LYNX_VARIANT_LYNX_INT4) tab = encode_tables4(params->alpha, params->eps);
  cudaError_t e = launch_encode_variant(x_bf16, n_pages, variant, codes, meta, tab,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lynx_encode_variant launch");
  return LYNX_OK;
}

int lynx_reconstruct_variant(const uint8_t* codes, const float* meta, int64_t n_pages, int variant,
                             const lynx_params_t* params, void* out, int out_dtype, void* stream) {
  g_last_error[0] = '\0';
  if (variant < LYNX_VARIANT_LYNX_INT8 || variant > LYNX_VARIANT_UNIFORM_INT4)
    return fail(LYNX_ERR_INVALID_ARG, "variant=%d", variant);
  const bool lynx_kind = variant == LYNX_VARIANT_LYNX_INT8 || variant == LYNX_VARIANT_LYNX_INT4;
  if (lynx_kind) {
    int st = check_params(params);
    if (st != LYNX_OK) return st;
  }
  if (out_dtype != LYNX_OUT_BF16 && out_dtype != LYNX_OUT_F32)
    return fail(LYNX_ERR_INVALID_ARG, "out_dtype=%d (need 0 = BF16 or 1 = F32)", out_dtype);
  if (n_pages < 0) return fail(LYNX_ERR_INVALID_ARG, "n_pages=%lld < 0", (long long)n_pages);
  if (n_pages == 0) return LYNX_OK;
  if (!codes || !meta || !out) return fail(LYNX_ERR_INVALID_ARG, "NULL buffer pointer");
  if (misaligned(codes) || misaligned(meta) || misaligned(out))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  if (n_pages > ((int64_t)1 << 40)) return fail(LYNX_ERR_INVALID_ARG, "n_pages too large");
  const LutTables* lut = nullptr;
  if (variant == LYNX_VARIANT_LYNX_INT8) lut = lut_tables8(params->alpha, params->eps);
  if (variant == LYNX_VARIANT_LYNX_INT4) lut = lut_tables4(params->alpha, params->eps);
  int* status = device_status_ptr();
  if (!status) return fail(LYNX_ERR_CUDA, "cannot resolve the device status word");
  cudaError_t e = launch_reconstruct_variant(codes, meta, n_pages, variant, out, out_dtype, lut, status,
                                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lynx_reconstruct_variant launch");
  return LYNX_OK;
}

int lynx_encode_split(const void* x_bf16, int64_t n_pages, int anchor_bits, const lynx_params_t* params,
                      uint8_t* anchor, uint8_t* residual, float* meta, void* stream) {
  g_last_error[0] = '\0';
  int st = check_params(params);
  if (st != LYNX_OK) return st;
  if (anchor_bits < 2 || anchor_bits > 6)
    return fail(LYNX_ERR_UNSUPPORTED, "anchor_bits=%d outside 2..6", anchor_bits);
  if (n_pages < 0) return fail(LYNX_ERR_INVALID_ARG, "n_pages=%lld < 0", (long long)n_pages);
  if (n_pages == 0) return LYNX_OK;
  if (!x_bf16 || !anchor || !residual || !meta) return fail(LYNX_ERR_INVALID_ARG, "NULL buffer pointer");
  if (misaligned(x_bf16) || misaligned(anchor) || misaligned(residual) || misaligned(meta))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  if (n_pages > ((int64_t)1 << 40)) return fail(LYNX_ERR_INVALID_ARG, "n_pages too large");
  cudaError_t e = launch_encode_split(x_bf16, n_pages, anchor_bits, anchor, residual, meta,
                                      encode_tables(params->alpha, params->eps), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lynx_encode_split launch");
  return LYNX_OK;
}

int lynx_reconstruct_split(const uint8_t* anchor, const uint8_t* residual, const float* meta, int64_t n_pages,
                           int anchor_bits, const lynx_params_t* params, void* out, int out_dtype, void* stream) {
  g_last_error[0] = '\0';
  int st = check_params(params);
  if (st != LYNX_OK) return st;
  if (anchor_bits < 2 || anchor_bits > 6)
    return fail(LYNX_ERR_UNSUPPORTED, "anchor_bits=%d outside 2..6", anchor_bits);
  if (out_dtype != LYNX_OUT_BF16 && out_dtype != LYNX_OUT_F32)
    return fail(LYNX_ERR_INVALID_ARG, "out_dtype=%d (need 0 = BF16 or 1 = F32)", out_dtype);
  if (n_pages < 0) return fail(LYNX_ERR_INVALID_ARG, "n_pages=%lld < 0", (long long)n_pages);
  if (n_pages == 0) return LYNX_OK;
  if (!anchor || !meta || !out) return fail(LYNX_ERR_INVALID_ARG, "NULL buffer pointer");
  if (misaligned(anchor) || misaligned(meta) || misaligned(out) || (residual && misaligned(residual)))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  if (n_pages > ((int64_t)1 << 40)) return fail(LYNX_ERR_INVALID_ARG, "n_pages too large");
  cudaError_t e = launch_reconstruct_split(anchor, residual, meta, n_pages, anchor_bits, out, out_dtype,
                                           split_tables(params->alpha, params->eps, anchor_bits),
                                           lut_tables8(params->alpha, params->eps), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lynx_reconstruct_split launch");
  return LYNX_OK;
}

int lynx_attn_merge(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
                    int64_t rows, int head_dim, float* o, float* lse, void* stream) {
  g_last_error[0] = '\0';
  if (rows < 0) return fail(LYNX_ERR_INVALID_ARG, "rows=%lld < 0", (long long)rows);
  if (head_dim != kH) return fail(LYNX_ERR_UNSUPPORTED, "head_dim=%d (need 128)", head_dim);
  if (rows == 0) return LYNX_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o || !lse)
    return fail(LYNX_ERR_INVALID_ARG, "NULL buffer pointer");
  if (misaligned(o_a) || misaligned(o_b) || misaligned(o) || misaligned(lse_a) || misaligned(lse_b) ||
      misaligned(lse))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  cudaError_t e = launch_attn_merge(o_a, lse_a, o_b, lse_b, rows, o, lse, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lynx_attn_merge launch");
  return LYNX_OK;
}

int lynx_decode_attn_bf16(const void* q_bf16, int B, int T, int Hq, int Hkv, int head_dim,
                          const void* k_pages, const void* v_pages, int64_t n_pool_pages,
                          const int32_t* page_table, int max_pages, const int32_t* ctx_len,
                          float sm_scale, int causal, float* out, float* lse, void* workspace,
                          size_t workspace_bytes, void* stream) {
  g_last_error[0] = '\0';
  if (!k_pages || !v_pages) return fail(LYNX_ERR_INVALID_ARG, "NULL page pool");
  if (misaligned(k_pages) || misaligned(v_pages))
    return fail(LYNX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  DecodeArgs a{};
  a.k_bf16 = static_cast<const uint16_t*>(k_pages);
  a.v_bf16 = static_cast<const uint16_t*>(v_pages);
  return decode_common(a, kModeBf16, q_bf16, B, T, Hq, Hkv, head_dim, n_pool_pages, page_table,
                       max_pages, ctx_len, sm_scale, causal, out, lse, workspace, workspace_bytes,
                       100.0f, 1e-6f, stream);
}

int lynx_test_inject_wait_timeout(int n_calls) {
  g_last_error[0] = '\0';
  if (n_calls < 0) return fail(LYNX_ERR_INVALID_ARG, "n_calls=%d < 0", n_calls);
  g_inject_calls = n_calls;
  return LYNX_OK;
}

int lynx_device_status(void) {
  g_last_error[0] = '\0';
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "lynx_device_status synchronize");
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "lynx_device_status read");
  if (v != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    return fail(LYNX_ERR_DEVICE, "device error word = %d (1: a bounded wait gave up, "
                "2: page id outside the pool, 3: ctx_len outside 0..max_pages*256)", v);
  }
  return LYNX_OK;
}

}  // extern "C"
