/*
 * lynx.h -- C ABI of the GB300 (sm_103a) Lynx hot path.
 *
 * Lynx ("Lynx: Progressive Speculative Quantization for accelerating KV
 * Transfer in Long-Context Inference") splits each KV-cache value into an
 * 8-bit code and ships it as two 4-bit streams: an Anchor (most significant
 * nibble) that is enough for speculative draft decoding, and a Residual
 * (least significant nibble) that restores the full code for verification.
 * This library implements, as CUDA kernels for one GB300 GPU:
 *
 *   lynx_encode_pages     Algorithm 1 of the paper (§4.1): BF16 pages ->
 *                         packed Anchor plane, packed Residual plane, fp32
 *                         metadata.
 *   lynx_reconstruct      the two dequantisation phases of §4.2 (Anchor only:
 *                         draft KV; Anchor + Residual: verification KV).
 *   lynx_decode_attn      softmax(Q K^T * scale) V (§2.1) over the packed
 *                         planes, dequantised in registers; 1 query token
 *                         (draft decode) or T tokens (the parallel
 *                         verification pass of §4.3).
 *   lynx_decode_attn_bf16 the same attention over plain BF16 pages (the
 *                         uncompressed baseline the paper compares against).
 *   lynx_attn_merge       combines attention over two disjoint key sets by
 *                         their log-sum-exps (the drafts' own uncompressed KV
 *                         joined to the verification over the packed cache).
 *   lynx_encode_tokens    Algorithm 1 reading token-major (paged-attention) KV.
 *   lynx_encode_split, lynx_reconstruct_split
 *                         the split stream at other Anchor / Residual widths.
 *   lynx_encode_variant, lynx_reconstruct_variant, lynx_decode_attn_int4,
 *   lynx_decode_attn_uniform, lynx_split_nibbles
 *                         the single-precision comparators of §6.1 (uniform
 *                         INT8 / INT4, Lynx-INT8, Lynx-INT4).
 *
 * ---------------------------------------------------------------------------
 * Data layout (all sizes for H = 128 channels, P = 256 tokens, C = 32):
 *
 *   KV page      One KV head's 128 channels x 256 consecutive tokens, BF16,
 *                channel-major: element (c, t) at index c*256 + t.  65536 B.
 *   Anchor plane Per page uint8[128][128]: byte j of channel row c holds the
 *                4-bit two's-complement anchor of token 2j in its low nibble
 *                and of token 2j+1 in its high nibble (paper §5: two 4-bit
 *                segments per byte).  16384 B per page.
 *   Residual     Same layout, 4-bit two's-complement residual.  16384 B.
 *   Metadata     Per page float32[2304] = gamma_min[128], gamma_scale[128],
 *                mu[8][128], sigma[8][128] (Algorithm 1's metadata; mu and
 *                sigma chunk-major: element [b][c] is chunk b of channel c).
 *                9216 B.
 *   Streams     The paper's §5 serialises each stream as one contiguous block:
 *                the Anchor planes of the pages followed immediately by their
 *                metadata.  Here that block is one caller buffer of
 *                n * (16384 + 9216) bytes: pass its first n * 16384 bytes as
 *                `anchor` and the rest as `meta` (16-byte aligned, as every
 *                offset in it is); the Residual stream is the residual planes.
 *
 * Code definition (per channel c of a page, per token t, chunk b = t / 32):
 *   x_n = (x - gamma_min) / (gamma_scale + eps)              (Stage 1)
 *   mu  = (x_n[32b] + ... + x_n[32b+31]) / 32, summed left to right
 *   sigma = max |x_n - mu| over the chunk
 *   x_f = (x_n - mu) / (sigma + eps)                           (Stage 2)
 *   I   = round(127 ln(1 + alpha |x_f|) / ln(1 + alpha))       (Stage 3, Eq. 3)
 *   S   = -1 if x_f < 0 else +1
 *   anchor   = (S > 0 ? I : -I - 1) >> 4   (arithmetic shift), in [-8, 7]
 *   residual = 16 * (I >> 4) + 7 - I,                          in [-8, 7]
 * Every step of Stages 1-2 is one correctly rounded IEEE float32 operation;
 * the rounding of Stage 3 is decided exactly for the float32 x_f.  The anchor
 * equals Stage 4's sign-aware two's-complement map applied to V = I >> 4; the
 * Round-Half-Down bias (+7) sits at the anchor's reconstruction point 16 V + 7,
 * which keeps both streams within 4 bits (as printed, Stage 4 gives an anchor
 * with 18 levels).
 *
 * Reconstruction:  I_hat = 16 V + 7 (anchor only) or 16 V + 7 - residual,
 *   x_hat = gamma_min + (gamma_scale+eps) * (mu + (sigma+eps) * S * l(I_hat)),
 *   l(y) = ((1 + alpha)^(y/127) - 1) / alpha   (Eq. 4; inverse of Eq. 3).
 *
 * ---------------------------------------------------------------------------
 * Conventions for every entry point:
 *   - Device pointers unless stated.  The caller owns and allocates every
 *     buffer; the library allocates no device or host memory and keeps no
 *     state beyond per-device constant tables.
 *   - Pointers must be 16-byte aligned (LYNX_ERR_ALIGNMENT otherwise).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and never synchronise.  A non-zero return means nothing
 *     was launched, except LYNX_ERR_CUDA, which reports a failed launch.
 *   - Inputs must be finite; NaN or Inf give unspecified codes.
 *   - Supported shapes: H = 128, P = 256, C = 32, head_dim = 128,
 *     0.25 <= alpha <= 1e6, 0 < eps <= 1e-2.  Others return
 *     LYNX_ERR_UNSUPPORTED.
 *   - Thread safety: entry points may be called from several host threads;
 *     lynx_last_error() is per host thread.
 *   - CUDA graphs: the first call of each entry point on a device configures
 *     its kernels (shared-memory limits, the status word's address); every
 *     later call only launches kernels on `stream`, so it may be captured in a
 *     CUDA graph and replayed.  Tensor maps and launch shapes are fixed at
 *     capture: a replay reads the same buffers, page-table and context-length
 *     arrays (whose contents may change between replays within the captured
 *     max_pages and shapes).
 */
#ifndef LYNX_H_
#define LYNX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Method parameters.  Defaults {128, 256, 32, 100.0f, 1e-6f}. */
typedef struct lynx_params {
  int32_t H;      /* channels per page (block size of Algorithm 1); must be 128 */
  int32_t P;      /* tokens per page; must be 256                               */
  int32_t C;      /* tokens per chunk (Stage 2); must be 32                     */
  float alpha;    /* alpha of the compander, Eq. (3)                            */
  float eps;      /* epsilon of Algorithm 1, Stages 1 and 2                     */
} lynx_params_t;

enum {
  LYNX_OK = 0,
  LYNX_ERR_INVALID_ARG = -1,   /* null pointer, negative size, bad enum      */
  LYNX_ERR_UNSUPPORTED = -2,   /* shape or parameter outside the supported set */
  LYNX_ERR_ALIGNMENT = -3,     /* a pointer is not 16-byte aligned           */
  LYNX_ERR_WORKSPACE = -4,     /* workspace missing or too small             */
  LYNX_ERR_CUDA = -5,          /* CUDA runtime error (message in lynx_last_error) */
  LYNX_ERR_DEVICE = -6         /* a kernel gave up a bounded wait (see lynx_device_status) */
};

/* Output element types of lynx_reconstruct. */
enum { LYNX_OUT_BF16 = 0, LYNX_OUT_F32 = 1 };

/* Single-precision variants (paper §6.1: the uniform INT8 / INT4 baselines, and
 * Lynx-INT8 / Lynx-INT4, the hierarchical quantiser of §4.1 at one precision
 * without the split stream; §2.3 for the uniform form).
 *   LYNX_VARIANT_LYNX_INT8     codes [n_pages][128][256] bytes: Algorithm 1's
 *                              signed 8-bit code S > 0 ? I : -I - 1 (its
 *                              arithmetic shift by 4 is the Anchor); meta as
 *                              lynx_encode_pages.  Values = Lynx's full codes.
 *   LYNX_VARIANT_LYNX_INT4     codes [n_pages][128][128] bytes, two per byte (low
 *                              nibble = even token): Algorithm 1 with 7 magnitude
 *                              levels, I4 = round(7 ln(1 + alpha |x_f|) /
 *                              ln(1 + alpha)), as the sign-aware nibble
 *                              S > 0 ? I4 : -I4 - 1; meta as lynx_encode_pages;
 *                              x_f = S ((1 + alpha)^(I4/7) - 1) / alpha.
 *   LYNX_VARIANT_UNIFORM_INT8  codes [n_pages][128][256] bytes, Q in 0..255;
 *   LYNX_VARIANT_UNIFORM_INT4  codes [n_pages][128][128] bytes, Q in 0..15, two
 *                              per byte (low nibble = even token); for both,
 *                              per channel row of a page S = (max - min) /
 *                              (2^b - 1), Q = round((x - min) / S) (0 if S = 0),
 *                              x = min + Q S; meta [n_pages][256] float32 =
 *                              min[128], S[128]. */
enum {
  LYNX_VARIANT_LYNX_INT8 = 1,
  LYNX_VARIANT_LYNX_INT4 = 2,
  LYNX_VARIANT_UNIFORM_INT8 = 3,
  LYNX_VARIANT_UNIFORM_INT4 = 4
};

/* Algorithm 1 (paper §4.1, all four stages) on n_pages BF16 pages.
 *   x_bf16    [n_pages][128][256] BF16 (read only)
 *   anchor    [n_pages][128][128] uint8, written
 *   residual  [n_pages][128][128] uint8, written
 *   meta      [n_pages][2304] float32, written
 * n_pages == 0 is a no-op.  Errors: INVALID_ARG (null pointer with n_pages>0,
 * n_pages<0, null params), UNSUPPORTED, ALIGNMENT, CUDA. */
int lynx_encode_pages(const void* x_bf16, int64_t n_pages, const lynx_params_t* params,
                      uint8_t* anchor, uint8_t* residual, float* meta, void* stream);

/* Algorithm 1 on pages of which only a prefix of tokens is valid (the last,
 * partial page of a sequence; the paper encodes whole pages only).
 *   valid_tokens  [n_pages] int32 (device): page n's tokens 0 .. valid_tokens[n]-1
 *                 are valid; values are clamped to 0..256.
 * The statistics cover the valid tokens only: gamma_min / gamma_scale over
 * them (0 and 0 for an empty page); a chunk's mu is the left-to-right sum of
 * its valid x_n divided by their count (a correctly rounded float32
 * division), sigma the largest |x_n - mu| among them, and mu = sigma = 0 for
 * a chunk without valid tokens.  Padding tokens take no part in any
 * operation (their contents may be anything) and get code 0 with a positive
 * sign (anchor nibble 0, residual nibble 7).  A page with 256 valid tokens is
 * encoded exactly as lynx_encode_pages encodes it.  Other arguments and
 * errors as lynx_encode_pages; INVALID_ARG for a NULL valid_tokens. */
int lynx_encode_pages_partial(const void* x_bf16, int64_t n_pages, const int32_t* valid_tokens,
                              const lynx_params_t* params, uint8_t* anchor, uint8_t* residual,
                              float* meta, void* stream);

/* The split stream at other widths: an A-bit Anchor (sign included) and an
 * R = 8 - A bit Residual of Algorithm 1's 8-bit code, 2 <= A <= 6 (the paper's
 * §8 leaves widths other than 4 + 4 to future work).  With q8 = S > 0 ? I :
 * -I - 1 and V = I >> R:  Anchor = q8 >> R (arithmetic), Anchor-only index
 * V 2^R + 2^(R-1) - 1, Residual = that index - I.  Planes: per channel row 8
 * chunks, each a little-endian bit string of its 32 tokens' two's-complement
 * codes (token t at bits A t .. A t + A - 1), so an Anchor row is 32 A bytes
 * and a Residual row 32 R bytes ([n_pages][128][32 A] and [n_pages][128][32 R]);
 * with A = 4 the planes are exactly those of lynx_encode_pages.  Metadata as
 * lynx_encode_pages.  Errors as lynx_encode_pages; UNSUPPORTED for anchor_bits
 * outside 2..6. */
int lynx_encode_split(const void* x_bf16, int64_t n_pages, int anchor_bits, const lynx_params_t* params,
                      uint8_t* anchor, uint8_t* residual, float* meta, void* stream);

/* Reconstruction of lynx_encode_split's planes (residual == NULL: Anchor only),
 * into out as lynx_reconstruct does (the same float32 arithmetic; with A = 4 the
 * same result).  Errors as lynx_reconstruct; UNSUPPORTED for anchor_bits outside
 * 2..6. */
int lynx_reconstruct_split(const uint8_t* anchor, const uint8_t* residual, const float* meta, int64_t n_pages,
                           int anchor_bits, const lynx_params_t* params, void* out, int out_dtype, void* stream);

/* Encode BF16 pages [n_pages][128][256] (device, 16-byte aligned) into one of
 * the single-precision variants above; codes and meta are caller-allocated
 * device buffers (16-byte aligned) in the variant's layout.  params is read for
 * the Lynx variants (alpha, eps; errors as lynx_encode_pages) and ignored for
 * the uniform ones.  Asynchronous on `stream`.  Errors: INVALID_ARG for an
 * unknown variant, n_pages < 0 or a NULL pointer; ALIGNMENT; n_pages == 0 is a
 * no-op. */
int lynx_encode_variant(const void* x_bf16, int64_t n_pages, int variant, const lynx_params_t* params,
                        uint8_t* codes, float* meta, void* stream);

/* Dequantise a variant's codes and meta into out [n_pages][128][256], BF16
 * (LYNX_OUT_BF16, rounded to nearest even) or float32 (LYNX_OUT_F32).  Lynx
 * variants: fmaf(fmaf(v, sigma+eps, mu), gamma_scale+eps, gamma_min) with v the
 * code's signed inverse-compander value rounded to float32 (as
 * lynx_reconstruct); uniform: fmaf(Q, S, min).  Errors as lynx_encode_variant;
 * INVALID_ARG for an unknown out_dtype.  Lynx-INT4 runs lynx_reconstruct's
 * staged kernel, whose bounded waits set the device status word as there. */
int lynx_reconstruct_variant(const uint8_t* codes, const float* meta, int64_t n_pages, int variant,
                             const lynx_params_t* params, void* out, int out_dtype, void* stream);

/* Algorithm 1 on KV held token-major, the layout of paged attention (the
 * paper's §4.1 encodes pages "complying with paged attention"): element
 * (token t, head h, channel c) of one layer's K or V is
 * x_bf16[t * token_stride + h * 128 + c] (device, BF16, 2-byte aligned;
 * token_stride >= n_heads * 128 elements, so K and V interleaved per token or
 * more heads per row are read in place).  Pages are 256 tokens of one head:
 * page h * n_pp + j (n_pp = ceil(n_tokens / 256)) holds tokens 256 j ..
 * 256 j + 255 of head h and is written to anchor / residual / meta in the
 * layouts of lynx_encode_pages (caller-allocated: n_heads * n_pp pages).  The
 * last page of each head holds the remaining n_tokens - 256 (n_pp - 1) tokens
 * and is encoded over them as lynx_encode_pages_partial does; every other page
 * is encoded exactly as lynx_encode_pages encodes the same 256 tokens.
 * Asynchronous on `stream`.  Speed: when x is 16-byte aligned and
 * token_stride is a multiple of 8 elements the tokens are staged through
 * shared memory by TMA (the fast path); otherwise each channel is gathered
 * from global memory directly (same results, about 30% slower).  Errors:
 * INVALID_ARG for negative counts, a token_stride below n_heads * 128 or a NULL
 * pointer (when there is work); ALIGNMENT for an odd x or outputs not 16-byte
 * aligned; n_tokens == 0 or n_heads == 0 is a no-op. */
int lynx_encode_tokens(const void* x_bf16, int64_t n_tokens, int n_heads, int64_t token_stride,
                       const lynx_params_t* params, uint8_t* anchor, uint8_t* residual, float* meta,
                       void* stream);

/* Stage 3 of Algorithm 1 alone: codes[i] = round(127 ln(1 + alpha |a_i|) /
 * ln(1 + alpha)) in 0..127 for float32 magnitudes |a_i| <= 1 (larger values
 * are clamped to 1), decided exactly for the float32 input as in
 * lynx_encode_pages.  a: n float32 (device), codes: n uint8 (device). */
int lynx_quantize_magnitudes(const float* a, int64_t n, const lynx_params_t* params,
                             uint8_t* codes, void* stream);

/* Dequantisation (paper §4.2: Anchor phase and Residual phase).
 *   residual == NULL selects the anchor-only reconstruction (draft KV);
 *   otherwise the full code is used (verification KV).
 *   out       [n_pages][128][256], BF16 (out_dtype = LYNX_OUT_BF16, rounded
 *             to nearest even from the float32 result) or float32
 *             (LYNX_OUT_F32).  The float32 value is
 *             fmaf(fmaf(S*l(I_hat), sigma+eps, mu), gamma_scale+eps, gamma_min)
 *             with S*l(I_hat) rounded to float32.
 * Errors as for lynx_encode_pages; INVALID_ARG for an unknown out_dtype.  The
 * kernel stages pages through shared memory with bounded waits: a wait that
 * runs out (2 s) sets the device status word that lynx_device_status()
 * reports, and the affected pages' outputs are unspecified. */
int lynx_reconstruct(const uint8_t* anchor, const uint8_t* residual, const float* meta,
                     int64_t n_pages, const lynx_params_t* params, void* out, int out_dtype,
                     void* stream);

/* Split-K decode / verification attention over packed planes (paper §2.1 and
 * §4.2-4.3), dequantising in registers.
 *   q_bf16      [B][T][Hq][128] BF16.  Query head hq attends KV head hq / (Hq/Hkv).
 *   k_anc, v_anc, k_meta, v_meta   page pools (layouts above), indexed by page id.
 *   k_res, v_res  NULL for the draft (anchor-only) KV; both non-NULL for the
 *               full codes.  Mixing is INVALID_ARG.
 *   n_pool_pages  pages in each pool; a page id outside 0..n_pool_pages-1
 *               is not dereferenced: page 0 is read instead and the device
 *               error word is set (see lynx_device_status).
 *   page_table  [B][Hkv][max_pages] int32 page ids (device).  Entries past a
 *               sequence's last page are never read.
 *   ctx_len     [B] int32 (device): keys in each sequence, 0..max_pages*256
 *               (values outside are clamped and set the device error word).
 *   causal      0: every query row sees all ctx_len keys.  1: query token i
 *               (0-based, of T) sees keys 0 .. ctx_len - T + i; a row with no
 *               visible key outputs zeros and lse = -inf.
 *   sm_scale    logit scale (1/sqrt(128) in the paper's formula).
 *   out         [B][T][Hq][128] float32;  lse [B][T][Hq] float32 = natural
 *               log of sum_j exp(sm_scale * q.k_j) (NULL to skip).
 *   workspace   device scratch of at least lynx_decode_attn_workspace_size()
 *               bytes (LYNX_ERR_WORKSPACE otherwise); contents need no
 *               initialisation and are clobbered.
 * All values of every page a sequence touches must be finite, including the
 * positions past ctx_len in its last page.
 * Limits: 1 <= T <= 64 (the paper's cap of 64 draft tokens, §6.1), Hq % Hkv == 0,
 *         T * (Hq/Hkv) <= 256, max_pages >= 1,
 * B <= 65535, Hkv * ceil(T*(Hq/Hkv)/4) <= 65535. */
int lynx_decode_attn(const void* q_bf16, int B, int T, int Hq, int Hkv, int head_dim,
                     const uint8_t* k_anc, const uint8_t* k_res, const float* k_meta,
                     const uint8_t* v_anc, const uint8_t* v_res, const float* v_meta,
                     int64_t n_pool_pages, const int32_t* page_table, int max_pages,
                     const int32_t* ctx_len,
                     const lynx_params_t* params, float sm_scale, int causal,
                     float* out, float* lse, void* workspace, size_t workspace_bytes,
                     void* stream);

/* Same attention over plain BF16 page pools k_pages / v_pages ([id][128][256]). */
int lynx_decode_attn_bf16(const void* q_bf16, int B, int T, int Hq, int Hkv, int head_dim,
                          const void* k_pages, const void* v_pages, int64_t n_pool_pages,
                          const int32_t* page_table, int max_pages, const int32_t* ctx_len,
                          float sm_scale, int causal, float* out, float* lse,
                          void* workspace, size_t workspace_bytes, void* stream);

/* lynx_decode_attn without a caller-supplied workspace, for callers that
 * cannot allocate device memory: a connector or deserializer plugin that a
 * serving engine loads with a fixed memory budget and no allocator, or a
 * decode loop that must not call cudaMalloc / cudaFree because they
 * synchronise the device.  The paper has no counterpart; this is an
 * integration entry point of this library.
 *   Arguments: as lynx_decode_attn, minus workspace and workspace_bytes.
 *   Scratch: a static device array of 8 MiB inside the library, held by every
 *   GPU that loads the library until the process exits.  Shapes whose
 *   lynx_decode_attn_workspace_size() exceeds 8 MiB return
 *   LYNX_ERR_WORKSPACE.  The first call on a device resolves the array's
 *   device address (cudaGetSymbolAddress) with that device current; make that
 *   first call before any stream capture.
 *   No allocation: the call never calls cudaMalloc, cudaFree or any allocating
 *   routine.
 *   Sharing: every call on a device uses the same array, which keeps the last
 *   call's contents (the kernels overwrite all of it that they read, so it
 *   needs no clearing); calls whose kernels overlap on the GPU (different
 *   streams, no ordering between them) race on it and give wrong results.
 *   Device reset: the resolved address is kept for the life of the process;
 *   after cudaDeviceReset (or any reset of the device's primary context) the
 *   library reloads its module and the kept address is stale, so do not use
 *   this entry point on a device after resetting it. */
int lynx_decode_attn_noalloc(const void* q_bf16, int B, int T, int Hq, int Hkv, int head_dim,
                             const uint8_t* k_anc, const uint8_t* k_res, const float* k_meta,
                             const uint8_t* v_anc, const uint8_t* v_res, const float* v_meta,
                             int64_t n_pool_pages, const int32_t* page_table, int max_pages,
                             const int32_t* ctx_len, const lynx_params_t* params, float sm_scale,
                             int causal, float* out, float* lse, void* stream);

/* Decode / verification attention over uniform INT-b pages (paper §6.1's
 * uniform INT8 / INT4 baselines, LYNX_VARIANT_UNIFORM_INT8 / _INT4 codes and
 * their meta: min[128], scale[128] per page), through the same kernels as
 * lynx_decode_attn with x = min + scale * Q for every token of a channel row.
 *   bits 4: k_lo / v_lo are the packed code pools [n][128][128] as
 *     lynx_encode_variant writes them; k_hi, v_hi must be NULL.
 *   bits 8: the one-byte codes split by lynx_split_nibbles: k_lo / v_lo the
 *     low-nibble planes, k_hi / v_hi the high-nibble planes ([n][128][128]
 *     each).
 *   k_meta, v_meta: float32 [n][256].  Other arguments, workspace and errors as
 *   lynx_decode_attn; INVALID_ARG for bits other than 4 and 8 or a missing /
 *   superfluous high-nibble pool. */
int lynx_decode_attn_uniform(const void* q_bf16, int B, int T, int Hq, int Hkv, int head_dim, int bits,
                             const uint8_t* k_lo, const uint8_t* k_hi, const float* k_meta, const uint8_t* v_lo,
                             const uint8_t* v_hi, const float* v_meta, int64_t n_pool_pages,
                             const int32_t* page_table, int max_pages, const int32_t* ctx_len, float sm_scale,
                             int causal, float* out, float* lse, void* workspace, size_t workspace_bytes,
                             void* stream);

/* Rows of 256 one-byte codes (e.g. LYNX_VARIANT_UNIFORM_INT8 codes, n_rows =
 * 128 per page) -> two planes of rows of 128 bytes: lo holds the low nibbles
 * and hi the high nibbles, token 2j in the low half of byte j and token 2j + 1
 * in the high half (the layout of the Anchor and Residual planes).  codes, lo,
 * hi: device, 16-byte aligned, caller-allocated.  Asynchronous on `stream`.
 * Errors: INVALID_ARG for n_rows < 0 or a NULL pointer; ALIGNMENT. */
int lynx_split_nibbles(const uint8_t* codes, int64_t n_rows, uint8_t* lo, uint8_t* hi, void* stream);

/* Decode / verification attention over Lynx-INT4 pages (LYNX_VARIANT_LYNX_INT4
 * codes and meta): the draft-decode kernels of lynx_decode_attn with the
 * 7-level value table.  Arguments, workspace and errors as lynx_decode_attn
 * without a residual pool. */
int lynx_decode_attn_int4(const void* q_bf16, int B, int T, int Hq, int Hkv, int head_dim,
                          const uint8_t* k_codes, const float* k_meta, const uint8_t* v_codes,
                          const float* v_meta, int64_t n_pool_pages, const int32_t* page_table, int max_pages,
                          const int32_t* ctx_len, const lynx_params_t* params, float sm_scale, int causal,
                          float* out, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Merge of two attention results over disjoint key sets.  The verification
 * pass (paper §4.3) also attends to the draft tokens' own K and V, which the
 * caller holds uncompressed (e.g. as a BF16 page read by
 * lynx_decode_attn_bf16); attention over a union of key sets is the
 * log-sum-exp weighted combination of the attention over its parts:
 *   m   = max(lse_a, lse_b),  w_a = e^(lse_a - m),  w_b = e^(lse_b - m)
 *   o   = (w_a o_a + w_b o_b) / (w_a + w_b),   lse = m + ln(w_a + w_b)
 * per row, with natural-log LSEs as lynx_decode_attn returns them.  A row whose
 * lse is -inf in one input takes the other input's row; -inf in both gives
 * o = 0, lse = -inf.
 *   o_a, o_b, o    [rows][head_dim] float32;  lse_a, lse_b, lse  [rows] float32.
 *   o may be o_a or o_b and lse may be lse_a or lse_b (in place); other
 *   overlaps are not allowed.
 * rows == 0 is a no-op.  Errors: INVALID_ARG (null pointer, rows < 0),
 * UNSUPPORTED (head_dim != 128), ALIGNMENT, CUDA. */
int lynx_attn_merge(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
                    int64_t rows, int head_dim, float* o, float* lse, void* stream);

/* Workspace bytes needed by lynx_decode_attn / lynx_decode_attn_bf16 for the
 * given shape on the current device (0 for invalid shapes). */
size_t lynx_decode_attn_workspace_size(int B, int T, int Hq, int Hkv, int head_dim, int max_pages);

/* Test hook (not for production use; off by default): the next n_calls calls
 * of lynx_decode_attn, lynx_decode_attn_bf16, lynx_decode_attn_int4,
 * lynx_decode_attn_uniform, lynx_reconstruct or lynx_encode_tokens made from
 * this host thread run with a fault planted on the host side of the launch:
 * every CTA never issues the copy of its first V page (decode), of its first
 * page (reconstruct) or of its first item (the token encoder's TMA-staged
 * kernel; an input that admits no tensor map takes the other kernel, which
 * has no waits, and the call runs normally), and every bounded wait of those
 * kernels gives up after 1 ms instead of 2 s.  The waits for that copy then run
 * out, the kernel records device error word 1, drains the copies it did
 * issue, frees its tensor memory and returns; the call's outputs are
 * unspecified.  Used to check that a wait that runs out leaves the context
 * usable.  n_calls = 0 disarms it.  The paper has no counterpart.  Errors:
 * INVALID_ARG (n_calls < 0). */
int lynx_test_inject_wait_timeout(int n_calls);

/* Reads and clears the current device's error word, which kernels set when a
 * bounded wait on a TMA transfer gives up.  Synchronises the device.
 * Returns LYNX_OK, LYNX_ERR_DEVICE, or LYNX_ERR_CUDA. */
int lynx_device_status(void);

/* Human-readable name of a status code (static storage). */
const char* lynx_status_string(int status);

/* Detail of the last error returned on this host thread ("" if none). */
const char* lynx_last_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int lynx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LYNX_H_ */
