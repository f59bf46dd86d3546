// spectra_internal.cuh -- shared declarations of the CUDA library (not part
// of the public ABI; see include/spectra.h for the contract).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spectra.h"

namespace spectra {

constexpr int kGroup = 32;          // tokens per bit-plane group (one warp)
constexpr int kMaxBits = 8;         // widest channel code
constexpr int kLmStride = 256;      // row stride of the Lloyd-Max tables

// Bucket grids of the Lloyd-Max encode (codec_tc.cu): width b splits
// [-U_b, U_b) into NB_b = 2^p_b buckets of w_b = 2^-k_b, no wider than the
// smallest gap between two thresholds of the Gaussian tables (0.98, 0.50,
// 0.26, 0.13, 0.067, 0.034, 0.017 for b = 2..8), so a bucket holds at most
// one threshold; every threshold lies in the inner buckets (U_b = 2, 2, 4,
// 4, 4, 4, 4, 8 against largest thresholds 0, 0.98, 1.75, 2.40, 2.98, 3.49,
// 3.96, 4.40).  Entry j of width b (j = 0..NB_b, entry NB_b taking u >= U_b)
// holds (hi, cnt): cnt = #{tau <= left edge j}, hi = the first threshold
// above that edge (+inf if none); code(u) = cnt + (u >= hi).
__host__ __device__ constexpr int bk_shift(int b) { return b <= 1 ? 0 : (b <= 3 ? 1 : b - 2); }   // k_b
__host__ __device__ constexpr int bk_log(int b) { return b <= 7 ? b + 1 : 10; }                       // p_b
__host__ __device__ constexpr int bk_off(int b) { return b <= kMaxBits ? (1 << (b + 1)) - 4 + (b - 1) : 1540; }
constexpr int kBkEntries = 1540;   // sum over b of NB_b + 1
static_assert(bk_off(kMaxBits) + (1 << bk_log(kMaxBits)) + 1 == kBkEntries, "bucket table size");

// ---------------------------------------------------------------------------
// Layout of a plan's `derived` buffer.  Each table starts on a 256-byte
// boundary.  Per head h:
//   chan_off[h][c]  u16  bit offset o_c of channel c inside a token's R bits
//   qscale[h][c]    f32  encode scale: UNIFORM3S 2^b/(6 sigma_c); LLOYD 1/sigma_c
//   rscale[h][c]    f32  decode scale: UNIFORM3S Delta_c;        LLOYD sigma_c
// Shared by every head:
//   lm_level[b-1][k] f32 Gaussian Lloyd-Max level k of width b (ascending)
//   lm_thresh[b-1][k] f32 threshold between levels k-1 and k (k >= 1)
//   lm_bucket[e]     (f32 hi, i32 cnt) bucket table of the Lloyd-Max encode
//   lm_bucket_bad    i32 nonzero when the tables break the buckets' premise
// Tensor-core operand images (codec_tc.cu):
//   enc_img[h]  bf16 basis image for the encode contraction
//   dec_img[h]  bf16 basis image for the decode contraction
//   wmax[h]     i32 widest channel of head h
//   dec_bias[h][i] f32 decode offset of output i (uniform quantizer, widths
//               <= 7: the decode contraction then takes 128 + code)
// ---------------------------------------------------------------------------
struct DerivedLayout {
    size_t chan_off, qscale, rscale, lm_level, lm_thresh, lm_bucket, lm_bucket_bad, enc_img, dec_img, wmax, dec_bias,
        total;
    size_t enc_img_head_bytes, dec_img_head_bytes;
};

// ---------------------------------------------------------------------------
// Bit-plane helpers shared by the codec and attention kernels.
// 8x8 bit transpose of a 64-bit block held as (lo, hi): byte i, bit j
// <-> byte j, bit i.  Three delta swaps (exchange distances 7, 14, 28).
__device__ __forceinline__ void transpose8(uint32_t& lo, uint32_t& hi)
{
    uint32_t t;
    t = (lo ^ (lo >> 7)) & 0x00AA00AAu;  lo ^= t ^ (t << 7);
    t = (hi ^ (hi >> 7)) & 0x00AA00AAu;  hi ^= t ^ (t << 7);
    t = (lo ^ (lo >> 14)) & 0x0000CCCCu; lo ^= t ^ (t << 14);
    t = (hi ^ (hi >> 14)) & 0x0000CCCCu; hi ^= t ^ (t << 14);
    t = (lo ^ (hi << 4)) & 0xF0F0F0F0u;  lo ^= t;  hi ^= t >> 4;
}

// bytes k of four words, in order, as one word
__device__ __forceinline__ uint32_t gather_byte(uint32_t a, uint32_t b, uint32_t c, uint32_t d, int k)
{
    const uint32_t sel = ((4u + k) << 4) | uint32_t(k);
    return __byte_perm(__byte_perm(a, b, sel), __byte_perm(c, d, sel), 0x5410);
}

// Launch with programmatic dependent launch allowed: the kernel's CTAs may
// start (and run their prologue) while the previous kernel in the stream
// finishes; such a kernel calls pdl_wait() before its first global read.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args)
{
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
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Per-head tensor-core operand images (bytes; head_dim 128 only, the
// tensor-core kernels' width).  Encode: three bf16 terms (hi, mid, lo) of
// the transposed basis, or one exact +-1 Hadamard term for RWHT.  Decode:
// two bf16 terms of basis * scale, or one +-1 term for RWHT.  Each term is
// a 128 x 128 bf16 tile in the 128-byte-swizzled K-major layout.
__host__ __device__ inline size_t enc_img_bytes(int d) { return d == 128 ? size_t(3) * d * d * 2 : 0; }
__host__ __device__ inline size_t dec_img_bytes(int d) { return d == 128 ? size_t(2) * d * d * 2 : 0; }

__host__ __device__ inline DerivedLayout derived_layout(int heads, int d)
{
    DerivedLayout L;
    size_t o = 0;
    const size_t hd = size_t(heads) * d;
    L.chan_off = o;  o = align256(o + hd * sizeof(uint16_t));
    L.qscale = o;    o = align256(o + hd * sizeof(float));
    L.rscale = o;    o = align256(o + hd * sizeof(float));
    L.lm_level = o;  o = align256(o + kMaxBits * kLmStride * sizeof(float));
    L.lm_thresh = o; o = align256(o + kMaxBits * kLmStride * sizeof(float));
    L.lm_bucket = o; o = align256(o + kBkEntries * 2 * sizeof(float));
    L.lm_bucket_bad = o; o = align256(o + sizeof(int32_t));
    L.enc_img_head_bytes = enc_img_bytes(d);
    L.dec_img_head_bytes = dec_img_bytes(d);
    L.enc_img = o;   o = align256(o + size_t(heads) * L.enc_img_head_bytes);
    L.dec_img = o;   o = align256(o + size_t(heads) * L.dec_img_head_bytes);
    L.wmax = o;      o = align256(o + size_t(heads) * sizeof(int32_t));
    L.dec_bias = o;  o = align256(o + hd * sizeof(float));
    L.total = o;
    return L;
}

// Device-side view of a plan with derived tables resolved.
struct PlanView {
    int heads, d, basis, quant, max_rec_bits;
    const float* basis_mat;
    const float* eigvals;
    const int8_t* signs;
    const uint8_t* bits;
    const int32_t* rec_bits;
    const uint16_t* chan_off;
    const float* qscale;
    const float* rscale;
    const float* lm_level;
    const float* lm_thresh;
    const float2* lm_bucket;
    const int32_t* lm_bucket_bad;
    const uint8_t* enc_img;
    const uint8_t* dec_img;
    const int32_t* wmax;
    const float* dec_bias;
    int32_t* status;
};

inline PlanView make_view(const spectra_plan* p)
{
    const DerivedLayout L = derived_layout(p->heads, p->head_dim);
    const uint8_t* base = static_cast<const uint8_t*>(p->derived);
    PlanView v;
    v.heads = p->heads;
    v.d = p->head_dim;
    v.basis = p->basis;
    v.quant = p->quant;
    v.max_rec_bits = p->max_rec_bits;
    v.basis_mat = p->basis_mat;
    v.eigvals = p->eigvals;
    v.signs = p->signs;
    v.bits = p->bits;
    v.rec_bits = p->rec_bits;
    v.chan_off = reinterpret_cast<const uint16_t*>(base + L.chan_off);
    v.qscale = reinterpret_cast<const float*>(base + L.qscale);
    v.rscale = reinterpret_cast<const float*>(base + L.rscale);
    v.lm_level = reinterpret_cast<const float*>(base + L.lm_level);
    v.lm_thresh = reinterpret_cast<const float*>(base + L.lm_thresh);
    v.lm_bucket = reinterpret_cast<const float2*>(base + L.lm_bucket);
    v.lm_bucket_bad = reinterpret_cast<const int32_t*>(base + L.lm_bucket_bad);
    v.enc_img = base + L.enc_img;
    v.dec_img = base + L.dec_img;
    v.wmax = reinterpret_cast<const int32_t*>(base + L.wmax);
    v.dec_bias = reinterpret_cast<const float*>(base + L.dec_bias);
    v.status = p->status;
    return v;
}

// Bytes of a packed stream: ceil(T/32) groups of R words, padded to 16 B.
__host__ __device__ inline int64_t stream_bytes(int64_t R, int64_t T)
{
    if (R <= 0 || T <= 0) return 0;
    const int64_t raw = ((T + kGroup - 1) / kGroup) * 4 * R;
    return (raw + 15) / 16 * 16;
}

// Sylvester Hadamard entry H[i][j] = (-1)^popcount(i & j).
__host__ __device__ inline int hadamard_sign(int i, int j)
{
#ifdef __CUDA_ARCH__
    return (__popc(i & j) & 1) ? -1 : 1;
#else
    return (__builtin_popcount(unsigned(i & j)) & 1) ? -1 : 1;
#endif
}

__device__ __forceinline__ float load_elem(const void* p, int dt, int64_t idx)
{
    if (dt == SPECTRA_BF16) {
        const uint16_t u = static_cast<const uint16_t*>(p)[idx];
        return __uint_as_float(uint32_t(u) << 16);
    }
    return static_cast<const float*>(p)[idx];
}

// ----- launchers (defined in the .cu files) --------------------------------
spectra_status launch_gram(const spectra_plan* plan, const void* x, int dt, int64_t n_cal,
                           int64_t token_stride, float* partials, int nchunks, cudaStream_t s);
spectra_status launch_jacobi(const spectra_plan* plan, const float* partials, int nchunks,
                             int64_t n_cal, int max_sweeps, float* gram_out, cudaStream_t s);
spectra_status launch_alloc(const spectra_plan* plan, int R_tot, int fixed_bits, cudaStream_t s);
spectra_status launch_alloc_grouped(const spectra_plan* plan, int R_tot, int group, const int32_t* keep,
                                    cudaStream_t s);
spectra_status launch_effdim(const spectra_plan* plan, double energy, int32_t* d_energy, int32_t* d_gap,
                             cudaStream_t s);
spectra_status launch_plain_calibrate(const spectra_plan* plan, const float* partials, int nchunks, int64_t n_cal,
                                      cudaStream_t s);
spectra_status launch_finalize(const spectra_plan* plan, cudaStream_t s);
spectra_status launch_encode(const spectra_plan* plan, const void* x, int dt, int64_t T,
                             int64_t token_stride, uint8_t* codes, int64_t sstride, float* norms,
                             int64_t nstride, cudaStream_t s);
spectra_status launch_decode(const spectra_plan* plan, const uint8_t* codes, int64_t sstride,
                             const float* norms, int64_t nstride, int64_t T, void* x_out,
                             int out_dt, int64_t token_stride, cudaStream_t s);
// The uncompressed recent window of spectra_attn_decode_window.
struct AttnWindow {
    const void* k;
    const void* v;
    int dt;
    int64_t W, stride;
};
// The key-residual sketch of spectra_attn_decode_qjl.
struct AttnQjl {
    const float* sketch;
    const uint8_t* bits;
    int64_t stride;
    const float* norms;
    int64_t nstride;
};
spectra_status launch_attn(const spectra_plan* kplan, const spectra_plan* vplan, const void* q,
                           int q_dt, int B, int Hq, const uint8_t* kc, const uint8_t* vc,
                           int64_t sstride, const float* kn, const float* vn, int64_t nstride,
                           int64_t ctx, float scale, float* out, void* ws, size_t ws_bytes,
                           cudaStream_t s, const AttnWindow* window = nullptr, const AttnQjl* qjl = nullptr);
size_t attn_workspace_bytes(int B, int Hq, int d, int64_t ctx);
// Host-side argument checks of spectra_attn_decode (everything but the
// workspace), shared by the entry points that run it.
spectra_status attn_validate(const spectra_plan* kplan, const spectra_plan* vplan, const void* q, int q_dt,
                             int B, int Hq, const uint8_t* k_codes, const uint8_t* v_codes,
                             int64_t stream_stride_bytes, const float* k_norms, const float* v_norms,
                             int64_t norms_stride, int64_t ctx, float softmax_scale, const float* out);
int gram_chunks(int heads, int64_t n_cal);

inline spectra_status cuda_status(cudaError_t e)
{
    return e == cudaSuccess ? SPECTRA_OK : SPECTRA_ERR_CUDA;
}

// Dynamic shared-memory opt-in of a kernel; a refused size is reported here
// (SPECTRA_ERR_CUDA) instead of surfacing later as a launch failure.
template <typename Kernel>
inline spectra_status set_smem(Kernel kern, size_t bytes)
{
    return cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)));
}

// Kernel family chosen for encode, decode and attention (process-wide; see
// spectra_set_kernel_family): SPECTRA_KERNELS_AUTO, _CUDA_CORE or _TENSOR_CORE.
int kernel_family();

}  // namespace spectra
