/*
 * spectra.h -- C ABI of the spectral transform codec for transformer KV
 * caches (sm_103a).
 *
 * Method (page titles and sections):
 *  - "Sintesi Tecnica: SPECTRA" (gist.science, paper 2608.07915):
 *      "Metodologia" items 1-3 -- rotate the cache into the eigenbasis of
 *      its own second-moment (Gram) matrix G = E[h^T h], where channels are
 *      uncorrelated and energy concentrates; importance-weighted bit
 *      allocation; zero-bit channels are dropped.
 *      "La Pipeline di SPECTRA" phase 2 -- reverse water-filling of bits on
 *      the measured marginal variances; phase 3 -- tokens are projected,
 *      quantized per token and appended to a latent cache; full keys and
 *      values are rebuilt on the fly.  "Significato e Rivendicazioni" --
 *      attention directly in the latent space (here: spectra_attn_decode).
 *  - "Technisch Overzicht: Ablatie, Statistische Inferentie en Validatie
 *      voor KV-Cache Compressie" (gist.science, paper 2607.09683),
 *      "Experimentele Opstelling": randomized Walsh-Hadamard rotation with a
 *      data-independent Lloyd-Max codebook (the RWHT basis here), and the
 *      per-head eigenbasis calibrated on representative tokens.
 *
 * Conventions shared by every call:
 *  - All pointers are DEVICE pointers unless stated, caller-allocated and
 *    caller-owned.  The library allocates and frees nothing and keeps no
 *    state between calls: every table it needs lives in the plan.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; 0 = legacy
 *    default stream).  Host-detectable argument errors return a non-OK
 *    status before anything is launched.  Conditions only the device can
 *    see (a non-finite Gram matrix, an unconverged eigensolve, a stream
 *    buffer too small for a head's record) are written to plan->status[h]
 *    and read by the caller after synchronising.
 *  - Caches are row-major [tokens][heads][head_dim]: element (t, h, i) of x
 *    is at x[t * token_stride + h * head_dim + i] (token_stride in
 *    elements, >= heads * head_dim).  head_dim is 64 or 128.
 *  - A "head" is one (layer, kv-head) pair: a multi-layer cache laid out as
 *    [tokens][layers * kv_heads][head_dim] is one call with
 *    heads = layers * kv_heads.
 *
 * Packed-code stream (one per head; the pages print no bit layout, this is
 * the library's own): tokens in groups of 32; with R = sum_c bits[c] and
 * o_c = sum_{c' < c} bits[c'], group g holds R little-endian 32-bit words,
 * and bit (t mod 32) of word g*R + o_c + k is bit k of the code of channel c
 * of token t.  Channels are in eigenvalue-descending order; 0-bit channels
 * take no space.  A stream of T tokens takes spectra_stream_bytes(R, T)
 * bytes (zero-padded to a multiple of 16).
 */
#ifndef SPECTRA_H
#define SPECTRA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPECTRA_API __attribute__((visibility("default")))
#else
#define SPECTRA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* spectra_stream_t; /* == cudaStream_t */

typedef enum {
    SPECTRA_OK = 0,
    SPECTRA_ERR_INVALID_ARG = 1,   /* bad pointer, size, stride or enum   */
    SPECTRA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. d)   */
    SPECTRA_ERR_CUDA = 3,          /* a CUDA runtime call failed           */
    SPECTRA_ERR_NOT_CONVERGED = 4, /* device status: eigensolve gave up    */
    SPECTRA_ERR_TIMEOUT = 5,       /* device status: a bounded wait ran out*/
    SPECTRA_ERR_NONFINITE = 6,     /* device status: NaN/Inf in the input  */
    SPECTRA_ERR_BUFFER = 7         /* device status: stream buffer too small */
} spectra_status;

typedef enum { SPECTRA_BF16 = 0, SPECTRA_F32 = 1 } spectra_dtype;
typedef enum { SPECTRA_BASIS_EIGEN = 0, SPECTRA_BASIS_RWHT = 1 } spectra_basis;
typedef enum { SPECTRA_Q_UNIFORM3S = 0, SPECTRA_Q_LLOYD_GAUSS = 1 } spectra_quant;

/*
 * Per-head codec plan.  Host-side ints describe the shape; every pointer is
 * a caller-owned device buffer of the stated size.
 *   basis_mat [heads][d][d] f32  EIGEN: basis_mat[h][i][c] = component i of
 *                                the eigenvector of channel c (channels in
 *                                eigenvalue-descending order).  Unused by RWHT.
 *   eigvals   [heads][d]    f32  EIGEN: marginal variance of channel c.
 *   signs     [heads][d]    i8   RWHT: the +-1 diagonal D of y = H D x / sqrt(d)
 *                                (random draws supplied by the caller).
 *   bits      [heads][d]    u8   width of channel c, 0..8 (0 = dropped).
 *   rec_bits  [heads]       i32  R_h = sum_c bits[h][c].
 *   derived   spectra_plan_derived_bytes(heads, d) bytes, 256-B aligned:
 *                                tables written by spectra_plan_finalize.
 *   status    [heads]       i32  device status words (see above).
 *   max_rec_bits                 host-side upper bound on every R_h, set by
 *                                spectra_alloc_bits (or by the caller before
 *                                spectra_plan_finalize); sizes the streams.
 */
typedef struct {
    int32_t heads;
    int32_t head_dim;
    int32_t basis;          /* spectra_basis */
    int32_t quant;          /* spectra_quant */
    int32_t max_rec_bits;
    int32_t reserved;
    float* basis_mat;
    float* eigvals;
    int8_t* signs;
    uint8_t* bits;
    int32_t* rec_bits;
    void* derived;
    int32_t* status;
} spectra_plan;

/* Library version (major*10000 + minor*100 + patch). */
SPECTRA_API int spectra_version(void);

/*
 * Kernel family for spectra_encode, spectra_decode and spectra_attn_decode
 * (a process-wide setting; not part of the method, which both families
 * compute in full).  AUTO: the tensor-core kernels where they cover the call
 * (bf16 caches with head_dim 128 for the codec; head_dim 128 with at most 8
 * query heads per kv head for attention, with or without the key-residual
 * sketch), the CUDA-core kernels elsewhere.
 * CUDA_CORE: the CUDA-core kernels only.  TENSOR_CORE: the tensor-core
 * kernels only; a call they do not cover returns SPECTRA_ERR_UNSUPPORTED.
 * The initial value comes from the environment variable SPECTRA_PATH, read
 * once on first use ("generic" -> CUDA_CORE, "tc" -> TENSOR_CORE, unset or
 * anything else -> AUTO).  spectra_set_kernel_family returns
 * SPECTRA_ERR_INVALID_ARG for an unknown value; it is not synchronised with
 * calls in flight on other host threads.
 */
typedef enum {
    SPECTRA_KERNELS_AUTO = 0,
    SPECTRA_KERNELS_CUDA_CORE = 1,
    SPECTRA_KERNELS_TENSOR_CORE = 2
} spectra_kernel_family;
SPECTRA_API spectra_status spectra_set_kernel_family(int family);
SPECTRA_API int spectra_get_kernel_family(void);

/* Human-readable name of a status code (static string, never NULL). */
SPECTRA_API const char* spectra_status_string(spectra_status st);

/* Bytes of the plan's `derived` buffer for `heads` heads of width d. */
SPECTRA_API size_t spectra_plan_derived_bytes(int heads, int head_dim);

/* Bytes of one packed stream of T tokens at R bits per token (zero-padded
 * to a multiple of 16).  0 when R == 0 or T == 0. */
SPECTRA_API size_t spectra_stream_bytes(int32_t rec_bits, int64_t T);

/*
 * spectra_calibrate -- per-head Gram matrix and its eigenbasis.
 * ("Sintesi Tecnica: SPECTRA", "Metodologia" items 1 and 3; "Technisch
 * Overzicht ...", "Experimentele Opstelling": per-head eigenbasis calibrated
 * on representative tokens.)
 *   G_h = (1/n_cal) sum_{t < n_cal} x[t,h,:] x[t,h,:]^T   (uncentred), then
 *   G_h = Q diag(lam) Q^T by cyclic Jacobi, one thread block per head, lam
 *   descending (ties: lower index first), each eigenvector's largest-|.|
 *   component positive (ties: lowest row).
 * x: [n_cal][heads][d] of dtype `dt`, token_stride in elements (for BF16 a
 *   multiple of 8, for F32 a multiple of 4; x 16-byte aligned).
 * Writes plan->basis_mat, plan->eigvals and plan->status[h] (= sweeps used,
 *   or -SPECTRA_ERR_NOT_CONVERGED / -SPECTRA_ERR_NONFINITE).
 * workspace: spectra_calibrate_workspace_bytes(heads, d, n_cal) bytes.
 * gram_out: optional [heads][d][d] f32 copy of G (NULL to skip).
 * max_sweeps: 1..100 (Jacobi sweeps before giving up).
 */
SPECTRA_API size_t spectra_calibrate_workspace_bytes(int heads, int head_dim, int64_t n_cal);
SPECTRA_API spectra_status spectra_calibrate(spectra_plan* plan, const void* x, spectra_dtype dt,
                                 int64_t n_cal, int64_t token_stride, int max_sweeps,
                                 void* workspace, size_t workspace_bytes, float* gram_out,
                                 spectra_stream_t stream);

/*
 * spectra_alloc_bits -- integer reverse water-filling, then finalize.
 * ("Sintesi Tecnica: SPECTRA", "La Pipeline di SPECTRA" phase 2; zero-bit
 * channels dropped, "Metodologia" item 2.)
 * fixed_bits == 0: R_tot = min(floor(avg_bits * d + 1e-9), 8 d) one-bit
 *   increments, each to the channel with the largest eigvals[c] * 4^-b_c
 *   among channels below 8 bits (lowest index on ties; negative eigenvalues
 *   count as 0).  Every head gets exactly R_tot bits.
 * fixed_bits in 1..8: every channel gets fixed_bits (no water-filling; the
 *   RWHT variant and uniform-allocation variants).
 * Writes plan->bits, plan->rec_bits and the derived tables; sets
 * plan->max_rec_bits on the host.
 */
SPECTRA_API spectra_status spectra_alloc_bits(spectra_plan* plan, double avg_bits, int fixed_bits,
                                  spectra_stream_t stream);

/*
 * spectra_alloc_bits_ex -- grouped reverse water-filling over the leading
 * channels, then finalize.  ("Sintesi Tecnica: SPECTRA", "La Pipeline di
 * SPECTRA" phase 2, "Raggruppamento": adjacent latent coordinates share one
 * bit width, keeping the cache append-only and streamable; "Technisch
 * Overzicht ...", "Regime-Specifieke Prestaties": the effective dimension is
 * pruned and the channels past it are left out.)
 * EIGEN plans.  With R_tot = min(floor(avg_bits * d + 1e-9), 8 d): the first
 *   keep[h] channels of head h form floor(keep[h] / group) groups of `group`
 *   consecutive channels (eigenvalue-descending order); every other channel
 *   gets 0 bits.  floor(R_tot / group) one-bit steps (fewer if every kept
 *   group reaches 8 bits), each giving all channels of the group with the
 *   largest Lam_G * 4^-b_G one bit (Lam_G = sum of the group's eigenvalues
 *   clipped at 0, in fp64 in ascending channel order; lowest group on ties).
 *   group = 1 with keep = NULL is spectra_alloc_bits.
 * group: a power of two dividing head_dim.  keep: device int32[heads]
 *   (values clipped to 0..d), or NULL for all channels -- for instance the
 *   d_gap output of spectra_effective_dim.
 * Sets plan->max_rec_bits = group * floor(R_tot / group) on the host.
 */
SPECTRA_API spectra_status spectra_alloc_bits_ex(spectra_plan* plan, double avg_bits, int group,
                                     const int32_t* keep, spectra_stream_t stream);

/*
 * spectra_effective_dim -- effective dimension of each head's spectrum,
 * with spectral-gap pruning.  ("Technisch Overzicht ...", "Regime-Specifieke
 * Prestaties": d_eff follows the calibration budget rather than the true
 * rank, and a single spurious eigenvalue can flip the output, so a spectral-
 * gap criterion prunes the estimate.  The page gives no formula; this is the
 * library's reading.)  On plan->eigvals (descending, clipped at 0):
 *   d_energy[h] = the smallest k with lam_0 + ... + lam_{k-1} >= energy * sum
 *                 (0 for an all-zero spectrum), sums in fp64;
 *   d_gap[h]    = the k in 1 .. min(d_energy, d - 1) with the largest
 *                 lam_{k-1} / lam_k (lam_k = 0 counts as infinite), the
 *                 smallest such k on ties.
 * energy in (0, 1]; d_energy, d_gap: device int32[heads].
 */
SPECTRA_API spectra_status spectra_effective_dim(const spectra_plan* plan, double energy, int32_t* d_energy,
                                     int32_t* d_gap, spectra_stream_t stream);

/*
 * spectra_calibrate_plain -- calibration without rotation (the ablation
 * page's Plain-KV: "Technisch Overzicht ...", "Belangrijkste Bijdragen" 1,
 * scalar quantization without rotation).  basis_mat = identity and
 * eigvals[h][c] = (1/n_cal) sum_t x[t,h,c]^2, the raw coordinates' second
 * moments in their own order; status[h] = 0 (or -SPECTRA_ERR_NONFINITE).
 * x, n_cal, token_stride and the workspace as for spectra_calibrate.
 */
SPECTRA_API spectra_status spectra_calibrate_plain(spectra_plan* plan, const void* x, spectra_dtype dt,
                                       int64_t n_cal, int64_t token_stride, void* workspace,
                                       size_t workspace_bytes, spectra_stream_t stream);

/*
 * spectra_plan_finalize -- recompute rec_bits and the derived tables from a
 * plan whose bits (and eigvals / basis_mat / signs) the caller filled in.
 * plan->max_rec_bits must already bound every R_h.
 */
SPECTRA_API spectra_status spectra_plan_finalize(spectra_plan* plan, spectra_stream_t stream);

/*
 * spectra_encode -- rotate, quantize and bit-pack T tokens of every head.
 * ("Sintesi Tecnica: SPECTRA", "La Pipeline di SPECTRA" phase 3: tokens are
 * projected down, quantized per token and appended to the latent cache.)
 * EIGEN: y_c = sum_i basis_mat[i][c] x_i for channels with bits > 0.
 * RWHT:  y = H D x / sqrt(d) (Sylvester Hadamard, natural order).
 * UNIFORM3S: sigma_c = sqrt(max(eigvals[c], 0)), Delta = 6 sigma_c / 2^b,
 *   code = clamp(floor((y + 3 sigma_c) / Delta), 0, 2^b - 1).
 * LLOYD_GAUSS: code = #{Gaussian Lloyd-Max thresholds tau_k <= y / sigma},
 *   sigma = sigma_c (EIGEN) or ||x|| / sqrt(d) per token (RWHT).
 * x: [T][heads][d] of dtype `dt` (token_stride as in spectra_calibrate).
 * codes: head h's stream starts at codes + h * stream_stride_bytes (16-byte
 *   aligned; stride >= spectra_stream_bytes(plan->max_rec_bits, T)); token 0
 *   of the call is written at the start of that stream.  To append after t0
 *   tokens (t0 a multiple of 128), pass codes + t0 / 32 * 4 * R.
 * norms: RWHT only, f32, norms[h * norms_stride + t] = ||x[t,h,:]||;
 *   NULL otherwise.
 */
SPECTRA_API spectra_status spectra_encode(const spectra_plan* plan, const void* x, spectra_dtype dt,
                              int64_t T, int64_t token_stride, uint8_t* codes,
                              int64_t stream_stride_bytes, float* norms, int64_t norms_stride,
                              spectra_stream_t stream);

/*
 * spectra_encode_kv -- spectra_encode of a layer's keys and values in one
 * call: exactly spectra_encode(kplan, k, ..., k_codes, ..., k_norms, ...)
 * followed by spectra_encode(vplan, v, ..., v_codes, ..., v_norms, ...) on
 * the same stream, with the same codes.  ("Sintesi Tecnica: SPECTRA", "La
 * Pipeline di SPECTRA" phase 3: each token's key and value are projected,
 * quantized and appended.)  kplan and vplan must have the same heads and
 * head_dim (else SPECTRA_ERR_INVALID_ARG); k and v share dt, T and
 * token_stride, the two stream sets share stream_stride_bytes, the norms
 * (RWHT plans) share norms_stride.  When both plans take the tensor-core
 * encode (bf16, d = 128, the same basis and quantizer) the two halves run as
 * one launch, so its fixed cost is paid once; otherwise as two.  Every
 * argument of both halves is checked before anything is launched.
 */
SPECTRA_API spectra_status spectra_encode_kv(const spectra_plan* kplan, const spectra_plan* vplan, const void* k,
                                 const void* v, spectra_dtype dt, int64_t T, int64_t token_stride,
                                 uint8_t* k_codes, uint8_t* v_codes, int64_t stream_stride_bytes,
                                 float* k_norms, float* v_norms, int64_t norms_stride, spectra_stream_t stream);

/*
 * spectra_append -- encode n new tokens of every head at stream positions
 * t0 .. t0+n-1 (any t0: a partly filled 32-token group keeps its earlier
 * tokens).  ("Sintesi Tecnica: SPECTRA", "La Pipeline di SPECTRA" phase 2,
 * "Raggruppamento": the latent cache stays append-only and streamable;
 * phase 3: each new token is projected, quantized and appended.)
 * The same codes as spectra_encode of the whole sequence, token by token.
 * x: [n][heads][d] of dt (token_stride as in spectra_encode); codes: the
 *   streams of spectra_encode (stride >= spectra_stream_bytes(max_rec_bits,
 *   t0 + n)); bits of tokens t0 .. t0+n-1 are overwritten, every other bit
 *   of the streams is kept.  norms (RWHT): norms[h * norms_stride + t0 + i].
 * Tokens up to the next multiple of 128 take a read-modify-write of their
 *   group on CUDA cores; the rest is an ordinary encode at that boundary.
 *   Calls that write the same 32-token group must not overlap on the GPU.
 */
SPECTRA_API spectra_status spectra_append(const spectra_plan* plan, const void* x, spectra_dtype dt, int64_t n,
                              int64_t token_stride, int64_t t0, uint8_t* codes, int64_t stream_stride_bytes,
                              float* norms, int64_t norms_stride, spectra_stream_t stream);

/*
 * spectra_decode -- unpack, dequantize, rotate back.
 * ("Sintesi Tecnica: SPECTRA", "La Pipeline di SPECTRA" phase 3: full keys
 * and values rebuilt on the fly.)
 * UNIFORM3S: y_c = -3 sigma_c + (code + 1/2) Delta; LLOYD_GAUSS:
 *   y_c = sigma * level[b][code]; dropped channels y_c = 0.
 * EIGEN: x_i = sum_c basis_mat[i][c] y_c.   RWHT: x = D H y / sqrt(d).
 * codes/norms as in spectra_encode; x_out: [T][heads][d] of out_dt with
 * token_stride in elements.
 */
SPECTRA_API spectra_status spectra_decode(const spectra_plan* plan, const uint8_t* codes,
                              int64_t stream_stride_bytes, const float* norms,
                              int64_t norms_stride, int64_t T, void* x_out, spectra_dtype out_dt,
                              int64_t token_stride, spectra_stream_t stream);

/*
 * spectra_decode_kv -- spectra_decode of a layer's keys and values in one
 * call: exactly spectra_decode(kplan, k_codes, ..., k_norms, ..., k_out, ...)
 * followed by spectra_decode(vplan, v_codes, ..., v_norms, ..., v_out, ...)
 * on the same stream.  kplan and vplan must have the same heads and
 * head_dim (else SPECTRA_ERR_INVALID_ARG); the stream sets share
 * stream_stride_bytes, the norms norms_stride, the outputs out_dt and
 * token_stride.  One launch when both plans take the tensor-core decode (d =
 * 128, the same basis and quantizer), else two.  Every argument of both
 * halves is checked before anything is launched.
 */
SPECTRA_API spectra_status spectra_decode_kv(const spectra_plan* kplan, const spectra_plan* vplan,
                                 const uint8_t* k_codes, const uint8_t* v_codes, int64_t stream_stride_bytes,
                                 const float* k_norms, const float* v_norms, int64_t norms_stride, int64_t T,
                                 void* k_out, void* v_out, spectra_dtype out_dt, int64_t token_stride,
                                 spectra_stream_t stream);

/*
 * spectra_attn_decode -- one decode step of grouped-query attention read
 * straight from packed K/V streams, computed in the latent basis.
 * ("Sintesi Tecnica: SPECTRA", "Significato e Rivendicazioni": attention
 * directly in the latent space.)
 * For batch b and query head j (kv head h = j / (Hq / Hkv), Hkv =
 * kplan->heads = vplan->heads):
 *   s_t = softmax_scale * <q[b,j], khat_t>,  p = softmax(s),
 *   out[b,j] = sum_t p_t vhat_t,
 * with khat/vhat the spectra_decode reconstructions of the streams; the
 * rotation of q into the K basis and of the latent output back out of the
 * V basis are done by the library (khat, vhat are never written).
 * q: [B][Hq][d] of q_dt.  Streams of (b, h) at k_codes / v_codes +
 *   (b * Hkv + h) * stream_stride_bytes, each holding ctx tokens.
 * norms (RWHT plans only): k_norms / v_norms[(b * Hkv + h) * norms_stride + t].
 * out: [B][Hq][d] f32.
 * workspace: spectra_attn_workspace_bytes(B, Hq, d, ctx) bytes (split-context
 *   partials).
 */
SPECTRA_API size_t spectra_attn_workspace_bytes(int B, int Hq, int head_dim, int64_t ctx);
SPECTRA_API spectra_status spectra_attn_decode(const spectra_plan* kplan, const spectra_plan* vplan,
                                   const void* q, spectra_dtype q_dt, int B, int Hq,
                                   const uint8_t* k_codes, const uint8_t* v_codes,
                                   int64_t stream_stride_bytes, const float* k_norms,
                                   const float* v_norms, int64_t norms_stride, int64_t ctx,
                                   float softmax_scale, float* out, void* workspace,
                                   size_t workspace_bytes, spectra_stream_t stream);

/*
 * spectra_attn_decode_window -- spectra_attn_decode over a cache whose
 * newest win_len tokens are not packed yet: the softmax runs over the ctx
 * packed tokens (reconstructed as by spectra_decode) followed by the win_len
 * uncompressed tokens, out[b,j] = sum over both of p_t v_t.  ("La Pipeline
 * di SPECTRA" phase 3: reconstructed keys and values feed standard
 * attention; the recent window holds tokens not yet appended.)
 * k_win / v_win: [B][win_len][Hkv][d] of win_dt, element (b, t, h, i) at
 *   [(b * win_len + t) * win_token_stride + h * d + i] (stride in elements,
 *   >= Hkv * d); 0 <= win_len <= SPECTRA_ATTN_MAX_WINDOW.  ctx may be 0.
 * Every other argument, the workspace (spectra_attn_workspace_bytes(B, Hq,
 *   d, ctx)) and the statuses as for spectra_attn_decode.
 */
#define SPECTRA_ATTN_MAX_WINDOW 16384
SPECTRA_API spectra_status spectra_attn_decode_window(const spectra_plan* kplan, const spectra_plan* vplan,
                                   const void* q, spectra_dtype q_dt, int B, int Hq,
                                   const uint8_t* k_codes, const uint8_t* v_codes,
                                   int64_t stream_stride_bytes, const float* k_norms,
                                   const float* v_norms, int64_t norms_stride, int64_t ctx,
                                   const void* k_win, const void* v_win, spectra_dtype win_dt,
                                   int64_t win_len, int64_t win_token_stride, float softmax_scale,
                                   float* out, void* workspace, size_t workspace_bytes,
                                   spectra_stream_t stream);

/*
 * spectra_qjl_encode -- 1-bit Johnson-Lindenstrauss sketch of the key
 * residuals.  ("Technisch Overzicht ...", "Experimentele Opstelling" and
 * "Belangrijkste Bijdragen" 1: TQ-QKV, a 1-bit QJL residual sketch on the
 * key path; section 2: on the key path its variance is amplified by the
 * softmax.)  For token t of head h: y = the latent coordinates of x[t,h,:]
 * (as spectra_encode computes them), yhat = the dequantized codes already in
 * the stream, r = y - yhat; bit j = (<s_j, r> >= 0) for the rows s_j of
 * `sketch`, and qjl_norms[h * qjl_norms_stride + t] = ||r||.
 * sketch: device f32 [d][d], row j = s_j, a Gaussian matrix (i.i.d. N(0,1)
 *   entries: the random draw is the caller's).
 * qjl_bits: head h at qjl_bits + h * qjl_stride_bytes, the packed-stream
 *   layout with R = d "planes" (word g*d + j, bit t mod 32 = bit j of token
 *   g*32 + t); stride >= spectra_stream_bytes(d, T).  x, codes, norms as for
 *   spectra_encode; CUDA-core kernel.
 */
SPECTRA_API spectra_status spectra_qjl_encode(const spectra_plan* plan, const float* sketch, const void* x,
                                  spectra_dtype dt, int64_t T, int64_t token_stride, const uint8_t* codes,
                                  int64_t stream_stride_bytes, const float* norms, int64_t norms_stride,
                                  uint8_t* qjl_bits, int64_t qjl_stride_bytes, float* qjl_norms,
                                  int64_t qjl_norms_stride, spectra_stream_t stream);

/*
 * spectra_attn_decode_qjl -- spectra_attn_decode whose key scores carry the
 * QJL estimate of the residual's inner product:
 *   s_t = softmax_scale * (<q, khat_t> + sqrt(pi/2)/d ||r_t|| sum_j <s_j, qt> z_j(t)),
 * qt = the query in the K latent coordinates, z_j = +1 for a set bit, -1
 * otherwise (an unbiased estimate of <q, k_t - khat_t>).
 * k_qjl_bits / k_qjl_norms: the spectra_qjl_encode outputs of every (b, kv
 *   head) stream, at + (b * Hkv + h) * qjl_stride_bytes / qjl_norms_stride.
 * Kernels as for spectra_attn_decode (the sketch term is one more tensor-core
 *   contraction of the level-table kernel); everything else as for
 *   spectra_attn_decode.
 */
SPECTRA_API spectra_status spectra_attn_decode_qjl(const spectra_plan* kplan, const spectra_plan* vplan,
                                   const void* q, spectra_dtype q_dt, int B, int Hq,
                                   const uint8_t* k_codes, const uint8_t* v_codes,
                                   int64_t stream_stride_bytes, const float* k_norms,
                                   const float* v_norms, int64_t norms_stride, int64_t ctx,
                                   const float* sketch, const uint8_t* k_qjl_bits, int64_t qjl_stride_bytes,
                                   const float* k_qjl_norms, int64_t qjl_norms_stride, float softmax_scale,
                                   float* out, void* workspace, size_t workspace_bytes,
                                   spectra_stream_t stream);

/*
 * spectra_selftest_wait -- exercises, on the device, the bounded waits that
 * every kernel of the library uses for its pipeline barriers (not part of
 * the method).  A one-block kernel waits for an mbarrier that nothing ever
 * arrives on: one thread with the busy-spin form, one warp with the
 * suspending form, under one shared abort flag.  After limit_ns the first
 * waiter gives up and raises the flag, and the rest give up on it; the kernel
 * then returns normally, so the context stays usable.
 * status: device int32[2] -- status[0] = -SPECTRA_ERR_TIMEOUT when the wait
 *   gave up (0 if the barrier had completed), status[1] = the number of the
 *   33 waiters that gave up.  elapsed_ns: device uint64 -- how long the
 *   spinning thread waited.  limit_ns in 1 .. 10^10.
 */
SPECTRA_API spectra_status spectra_selftest_wait(uint64_t limit_ns, int32_t* status, uint64_t* elapsed_ns,
                                     spectra_stream_t stream);

/*
 * spectra_attn_decode_noalloc -- spectra_attn_decode for callers that cannot
 * allocate device memory when they run a decode step (code inside an
 * allocator or memory-pool callback, hosts whose device memory belongs to
 * another framework's pool, deployments that forbid allocation after
 * start-up).  The pages have no counterpart: this is a packaging variant of
 * spectra_attn_decode, with the same arguments minus the workspace and the
 * same results.
 * Scratch: a static device array of SPECTRA_ATTN_NOALLOC_SCRATCH_BYTES inside
 *   the library, held by every GPU that loads the library until the process
 *   exits.  A call whose spectra_attn_workspace_bytes(B, Hq, d, ctx) exceeds
 *   it returns SPECTRA_ERR_UNSUPPORTED and launches nothing.  Nothing in the
 *   array needs clearing between calls.
 * Arguments are checked exactly as by spectra_attn_decode (same statuses);
 *   then a call whose spectra_attn_workspace_bytes(B, Hq, d, ctx) exceeds
 *   the array returns SPECTRA_ERR_UNSUPPORTED (ctx == 0 needs no scratch).
 * The first call on a device looks up the array's device address and caches
 *   it.  CUDA may load the library's device code lazily, so that first call
 *   can be the moment the array is created on the device: make it at
 *   start-up, outside any allocator callback and before any stream capture
 *   (a call refused for its size still does the lookup).  The cached address
 *   assumes the device's context lasts as long as the process (no
 *   cudaDeviceReset in between).  Every call shares the one array: calls
 *   whose kernels overlap on the GPU race on it.
 * After that first call on a device, this call allocates nothing (no
 *   cudaMalloc / cudaFree, no allocating library routine).
 */
#define SPECTRA_ATTN_NOALLOC_SCRATCH_BYTES (16u << 20)
SPECTRA_API spectra_status spectra_attn_decode_noalloc(const spectra_plan* kplan, const spectra_plan* vplan,
                                   const void* q, spectra_dtype q_dt, int B, int Hq,
                                   const uint8_t* k_codes, const uint8_t* v_codes,
                                   int64_t stream_stride_bytes, const float* k_norms,
                                   const float* v_norms, int64_t norms_stride, int64_t ctx,
                                   float softmax_scale, float* out, spectra_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SPECTRA_H */
