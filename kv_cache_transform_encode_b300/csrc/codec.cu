// codec.cu -- encode/decode on CUDA cores (any dtype, d in {64, 128}, both
// bases, both quantizers).  The bf16 d=128 hot configurations go through the
// tensor-core kernels in codec_tc.cu; this file serves every other case.
//
// "Sintesi Tecnica: SPECTRA", "La Pipeline di SPECTRA" phase 3: tokens are
// projected into the latent basis, quantized per token and appended to the
// latent cache; keys and values are rebuilt on the fly.  "Technisch
// Overzicht ...", "Experimentele Opstelling": randomized Walsh-Hadamard
// rotation (y = H D x / sqrt(d)) with a Lloyd-Max codebook.
//
// One warp per 32-token group (lane = token).  The d x d rotation matrix of
// the head sits in shared memory (rows padded to d+1 floats); EIGEN uses the
// plan's basis, RWHT builds M[i][c] = s_i H[i][c] / sqrt(d), so that both
// bases share y_c = sum_i M[i][c] x_i and x_i = sum_c M[i][c] y_c.  Codes are
// packed with one warp ballot per bit-column, which yields exactly the
// group's bit-plane word.
#include "spectra_internal.cuh"

#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

namespace spectra {

namespace {

constexpr int kWarps = 8;       // encode: warps (32-token groups) per block
constexpr int kDecWarps = 4;    // decode: fewer, to fit the staged words

template <int D>
__device__ void load_matrix(const PlanView& pv, int h, float* M)
{
    constexpr int LD = D + 1;
    if (pv.basis == SPECTRA_BASIS_EIGEN) {
        for (int e = threadIdx.x; e < D * D; e += blockDim.x)
            M[(e / D) * LD + (e % D)] = pv.basis_mat[size_t(h) * D * D + e];
    } else {
        const float inv = rsqrtf(float(D));
        for (int e = threadIdx.x; e < D * D; e += blockDim.x) {
            const int i = e / D, c = e % D;
            M[i * LD + c] = float(pv.signs[size_t(h) * D + i] * hadamard_sign(i, c)) * inv;
        }
    }
}

// count of thresholds tau_1..tau_{L-1} that are <= u (ascending table)
__device__ __forceinline__ int lm_code(const float* th, int b, float u)
{
    int lo = 0;                        // answer in [0, L-1]
    for (int step = 1 << (b - 1); step; step >>= 1)
        if (th[lo + step] <= u) lo += step;
    return lo;
}

// Rotation matrix with rows of exactly D floats, for the register-blocked
// projections below (all lanes read the same row: broadcast, no conflicts).
template <int D>
__device__ void load_matrix_dense(const PlanView& pv, int h, float* M)
{
    if (pv.basis == SPECTRA_BASIS_EIGEN) {
        for (int e = threadIdx.x; e < D * D; e += blockDim.x) M[e] = pv.basis_mat[size_t(h) * D * D + e];
    } else {
        const float inv = rsqrtf(float(D));
        for (int e = threadIdx.x; e < D * D; e += blockDim.x) {
            const int i = e / D, c = e % D;
            M[e] = float(pv.signs[size_t(h) * D + i] * hadamard_sign(i, c)) * inv;
        }
    }
}

// y[j] = sum_i M[i][c0 + j] xr[i] for CB consecutive channels, i ascending
// (each y the same sequential fp32 sum as a channel-at-a-time loop); M dense
// [D][D], xr one token's row in shared memory.
template <int D, int CB>
__device__ __forceinline__ void project_block(const float* M, const float* xr, int c0, float (&y)[CB])
{
#pragma unroll
    for (int j = 0; j < CB; ++j) y[j] = 0.f;
#pragma unroll 4
    for (int i = 0; i < D; ++i) {
        const float xi = xr[i];
        const float4* m = reinterpret_cast<const float4*>(M + i * D + c0);
#pragma unroll
        for (int q = 0; q < CB / 4; ++q) {
            const float4 v = m[q];
            y[4 * q] = fmaf(v.x, xi, y[4 * q]);
            y[4 * q + 1] = fmaf(v.y, xi, y[4 * q + 1]);
            y[4 * q + 2] = fmaf(v.z, xi, y[4 * q + 2]);
            y[4 * q + 3] = fmaf(v.w, xi, y[4 * q + 3]);
        }
    }
}

constexpr int kCB = 8;           // channels per register block

// t0: stream position of row 0 of x (an append; 0 for a whole encode).
// Rows 0..T-1 go to stream tokens t0..t0+T-1; a first group that starts
// before t0 keeps the bits of its earlier tokens (read-modify-write of its
// words), every other group is written whole.
// A block walks groups g = blockIdx.x, + gridDim.x, ...: its warps load the
// group's 32 tokens into shared memory together, then split the channels in
// blocks of kCB (lane = token), so a short append still spreads over all
// warps.  The plane words of a channel block are contiguous in the stream
// (offsets follow channel order) and leave 32 at a time from the lanes that
// hold them.
template <int D>
__global__ void __launch_bounds__(kWarps * 32)
encode_generic_kernel(PlanView pv, const void* __restrict__ x, int dt, int64_t T, int64_t tstride,
                      uint8_t* __restrict__ codes, int64_t sstride, float* __restrict__ norms,
                      int64_t nstride, int64_t t0)
{
    constexpr int LD = D + 1;
    extern __shared__ __align__(16) float smem[];
    float* M = smem;                               // [D][D]
    float* xw = M + D * D;                         // [32][LD] the group's tokens
    float* th = xw + 32 * LD;                      // [8][256] Lloyd-Max thresholds
    float* qsc = th + kMaxBits * kLmStride;        // [D]
    float* isg = qsc + D;                          // [32] RWHT: 1 / sigma of each token
    int* bsh = reinterpret_cast<int*>(isg + 32);   // [D]
    int* osh = bsh + D;                            // [D]

    const int h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = pv.rec_bits[h];
    if (R > pv.max_rec_bits) {
        if (threadIdx.x == 0 && blockIdx.x == 0) pv.status[h] = -SPECTRA_ERR_BUFFER;
        return;
    }
    load_matrix_dense<D>(pv, h, M);
    for (int e = threadIdx.x; e < kMaxBits * kLmStride; e += blockDim.x) th[e] = pv.lm_thresh[e];
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        qsc[c] = pv.qscale[size_t(h) * D + c];
        bsh[c] = pv.bits[size_t(h) * D + c];
        osh[c] = pv.chan_off[size_t(h) * D + c];
    }

    const int64_t g0 = t0 / kGroup;
    const int64_t ngroups = (t0 + T + kGroup - 1) / kGroup - g0;
    const bool rwht = pv.basis == SPECTRA_BASIS_RWHT;
    for (int64_t gi = blockIdx.x; gi < ngroups; gi += gridDim.x) {
        const int64_t g = g0 + gi;                     // stream group
        __syncthreads();                               // the previous group's reads of xw are done
        for (int e = threadIdx.x; e < 32 * D; e += blockDim.x) {
            const int r = e / D, i = e % D;
            const int64_t t = g * kGroup + r - t0;     // row of x
            xw[r * LD + i] = (t >= 0 && t < T) ? load_elem(x, dt, t * tstride + int64_t(h) * D + i) : 0.f;
        }
        __syncthreads();
        const int64_t t = g * kGroup + lane - t0;
        const bool live = t >= 0 && t < T;
        if (rwht) {
            if (warp == 0) {
                float n2 = 0.f;
                for (int i = 0; i < D; ++i) n2 = fmaf(xw[lane * LD + i], xw[lane * LD + i], n2);
                const float nrm = sqrtf(n2);
                if (live) norms[int64_t(h) * nstride + t0 + t] = nrm;
                const float sig = nrm * rsqrtf(float(D));
                isg[lane] = (sig > 0.f) ? 1.f / sig : 0.f;
            }
            __syncthreads();
        }
        const float inv_sig = rwht ? isg[lane] : 0.f;
        // lanes of earlier tokens whose bits stay (first group of an unaligned append)
        const uint32_t keep = (gi == 0 && (t0 % kGroup)) ? ((1u << (t0 % kGroup)) - 1u) : 0u;
        uint32_t* out = reinterpret_cast<uint32_t*>(codes + int64_t(h) * sstride) + g * R;
        auto put = [&](int w, uint32_t v) {
            out[w] = keep ? ((out[w] & keep) | (v & ~keep)) : v;
        };
        for (int cb = warp; cb < D / kCB; cb += kWarps) {
            const int c0 = cb * kCB;
            int any = 0;
#pragma unroll
            for (int j = 0; j < kCB; ++j) any |= bsh[c0 + j];
            if (!any) continue;
            float y[kCB];
            project_block<D, kCB>(M, xw + lane * LD, c0, y);
            const int base = osh[c0];
            uint32_t myword = 0;
            int nb = 0;
#pragma unroll
            for (int j = 0; j < kCB; ++j) {
                const int c = c0 + j, b = bsh[c];
                if (b == 0) continue;
                int code;
                if (pv.quant == SPECTRA_Q_UNIFORM3S) {
                    const float u = fmaf(y[j], qsc[c], float(1 << (b - 1)));
                    code = min(max(__float2int_rd(u), 0), (1 << b) - 1);
                } else {
                    const float s = rwht ? inv_sig : qsc[c];
                    code = lm_code(th + (b - 1) * kLmStride, b, y[j] * s);
                }
                if (!live) code = 0;
                for (int k = 0; k < b; ++k, ++nb) {
                    const uint32_t wv = __ballot_sync(0xffffffffu, (code >> k) & 1);
                    if ((nb & 31) == lane) myword = wv;
                    if ((nb & 31) == 31) put(base + (nb & ~31) + lane, myword);
                }
            }
            if ((nb & 31) != 0 && lane < (nb & 31)) put(base + (nb & ~31) + lane, myword);
        }
    }
}

// A few tokens (decode-step appends): one block per head, thread = channel
// for the rotation and the quantizer (the same arithmetic, in the same order,
// as encode_generic_kernel), then thread = plane word for the read-modify-
// write of bit (t mod 32) of each word of the token's group.  Tokens run one
// after another, so a group shared by several of them is never raced.
template <int D>
__global__ void __launch_bounds__(D)
append_small_kernel(PlanView pv, const void* __restrict__ x, int dt, int64_t n, int64_t tstride,
                    uint8_t* __restrict__ codes, int64_t sstride, float* __restrict__ norms, int64_t nstride,
                    int64_t t0)
{
    __shared__ float xs[D];
    __shared__ int code_s[D];
    __shared__ short plane_c[8 * D];
    __shared__ unsigned char plane_k[8 * D];
    __shared__ float red[D / 32];
    const int h = blockIdx.x, c = threadIdx.x, lane = c & 31, warp = c >> 5;
    const int R = pv.rec_bits[h];
    if (R > pv.max_rec_bits) {
        if (c == 0) pv.status[h] = -SPECTRA_ERR_BUFFER;
        return;
    }
    const int b = pv.bits[size_t(h) * D + c];
    const int o = pv.chan_off[size_t(h) * D + c];
    for (int k = 0; k < b; ++k) {
        plane_c[o + k] = short(c);
        plane_k[o + k] = (unsigned char)k;
    }
    const float qsc = pv.qscale[size_t(h) * D + c];
    uint32_t* words = reinterpret_cast<uint32_t*>(codes + int64_t(h) * sstride);
    for (int64_t i = 0; i < n; ++i) {
        const int64_t t = t0 + i;
        xs[c] = load_elem(x, dt, i * tstride + int64_t(h) * D + c);
        __syncthreads();
        float inv_sig = 0.f;
        if (pv.basis == SPECTRA_BASIS_RWHT) {
            // the generic kernel's sequential sum of squares, by one thread
            if (c == 0) {
                float n2 = 0.f;
                for (int j = 0; j < D; ++j) n2 = fmaf(xs[j], xs[j], n2);
                red[0] = n2;
            }
            __syncthreads();
            const float nrm = sqrtf(red[0]);
            if (c == 0) norms[int64_t(h) * nstride + t] = nrm;
            const float sig = nrm * rsqrtf(float(D));
            inv_sig = (sig > 0.f) ? 1.f / sig : 0.f;
        }
        int code = 0;
        if (b > 0) {
            float y = 0.f;
            if (pv.basis == SPECTRA_BASIS_EIGEN) {
                for (int j = 0; j < D; ++j) y = fmaf(pv.basis_mat[(size_t(h) * D + j) * D + c], xs[j], y);
            } else {
                const float inv = rsqrtf(float(D));
                for (int j = 0; j < D; ++j)
                    y = fmaf(float(pv.signs[size_t(h) * D + j] * hadamard_sign(j, c)) * inv, xs[j], y);
            }
            if (pv.quant == SPECTRA_Q_UNIFORM3S) {
                const float u = fmaf(y, qsc, float(1 << (b - 1)));
                code = min(max(__float2int_rd(u), 0), (1 << b) - 1);
            } else {
                const float sc = (pv.basis == SPECTRA_BASIS_RWHT) ? inv_sig : qsc;
                code = lm_code(pv.lm_thresh + (b - 1) * kLmStride, b, y * sc);
            }
        }
        code_s[c] = code;
        __syncthreads();
        const uint32_t bitm = 1u << (t % kGroup);
        uint32_t* gw = words + (t / kGroup) * R;
        for (int r = c; r < R; r += D) {
            const uint32_t v = (code_s[plane_c[r]] >> plane_k[r]) & 1u;
            gw[r] = v ? (gw[r] | bitm) : (gw[r] & ~bitm);
        }
        __syncthreads();
    }
    (void)lane;
    (void)warp;
}

template <int D>
__global__ void __launch_bounds__(kDecWarps * 32)
decode_generic_kernel(PlanView pv, const uint8_t* __restrict__ codes, int64_t sstride,
                      const float* __restrict__ norms, int64_t nstride, int64_t T,
                      void* __restrict__ xo, int out_dt, int64_t tstride)
{
    constexpr int LD = D + 1;
    extern __shared__ float smem[];
    float* M = smem;                               // [D][LD]
    float* ys = M + D * LD;                        // [kDecWarps][32][LD]
    float* lv = ys + kDecWarps * 32 * LD;             // [8][256] Lloyd-Max levels
    float* rsc = lv + kMaxBits * kLmStride;        // [D]
    int* bsh = reinterpret_cast<int*>(rsc + D);    // [D]
    uint32_t* wsh = reinterpret_cast<uint32_t*>(bsh + D);   // [kDecWarps][8*D]

    const int h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = pv.rec_bits[h];
    if (R > pv.max_rec_bits) {
        if (threadIdx.x == 0 && blockIdx.x == 0) pv.status[h] = -SPECTRA_ERR_BUFFER;
        return;
    }
    load_matrix<D>(pv, h, M);
    for (int e = threadIdx.x; e < kMaxBits * kLmStride; e += blockDim.x) lv[e] = pv.lm_level[e];
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        rsc[c] = pv.rscale[size_t(h) * D + c];
        bsh[c] = pv.bits[size_t(h) * D + c];
    }
    __syncthreads();

    const int64_t ngroups = (T + kGroup - 1) / kGroup;
    const int64_t g = int64_t(blockIdx.x) * kDecWarps + warp;
    if (g >= ngroups) return;
    const uint32_t* in = reinterpret_cast<const uint32_t*>(codes + int64_t(h) * sstride) + g * R;
    uint32_t* ww = wsh + warp * 8 * D;
    for (int e = lane; e < R; e += 32) ww[e] = in[e];
    __syncwarp();
    const int64_t t = g * kGroup + lane;
    float sig_t = 0.f;
    if (pv.basis == SPECTRA_BASIS_RWHT && t < T)
        sig_t = norms[int64_t(h) * nstride + t] * rsqrtf(float(D));
    float* yw = ys + warp * 32 * LD;
    int bc = 0;
    for (int c = 0; c < D; ++c) {
        const int b = bsh[c];
        float y = 0.f;
        if (b > 0) {
            int code = 0;
            for (int k = 0; k < b; ++k, ++bc) code |= int((ww[bc] >> lane) & 1u) << k;
            if (pv.quant == SPECTRA_Q_UNIFORM3S)
                y = rsc[c] * (float(code) + 0.5f - float(1 << (b - 1)));
            else
                y = ((pv.basis == SPECTRA_BASIS_RWHT) ? sig_t : rsc[c]) * lv[(b - 1) * kLmStride + code];
        }
        yw[lane * LD + c] = y;
    }
    __syncwarp();
    for (int r = 0; r < 32; ++r) {
        const int64_t tt = g * kGroup + r;
        if (tt >= T) break;
        for (int i = lane; i < D; i += 32) {
            float acc = 0.f;
            for (int c = 0; c < D; ++c) acc = fmaf(M[i * LD + c], yw[r * LD + c], acc);
            const int64_t o = tt * tstride + int64_t(h) * D + i;
            if (out_dt == SPECTRA_BF16) static_cast<__nv_bfloat16*>(xo)[o] = __float2bfloat16_rn(acc);
            else static_cast<float*>(xo)[o] = acc;
        }
    }
}

template <int D>
size_t enc_smem()
{
    return sizeof(float) * (D * D + 32 * (D + 1) + kMaxBits * kLmStride + D + 32) + sizeof(int) * 2 * D;
}
template <int D>
size_t dec_smem()
{
    return sizeof(float) * (D * (D + 1) + kDecWarps * 32 * (D + 1) + kMaxBits * kLmStride + D) +
           sizeof(int) * D + sizeof(uint32_t) * kDecWarps * 8 * D;
}

}  // namespace

spectra_status launch_encode_generic(const spectra_plan* plan, const void* x, int dt, int64_t T,
                                     int64_t token_stride, uint8_t* codes, int64_t sstride,
                                     float* norms, int64_t nstride, cudaStream_t s, int64_t t0)
{
    const PlanView pv = make_view(plan);
    const int64_t ngroups = (t0 + T + kGroup - 1) / kGroup - t0 / kGroup;
    if (ngroups == 0) return SPECTRA_OK;
    // blocks walk the groups: about two blocks per SM (the residency) over all heads
    const int64_t per_head = std::max<int64_t>(1, (2 * 148 + plan->heads - 1) / plan->heads);
    dim3 grid(unsigned(std::min<int64_t>(ngroups, per_head)), plan->heads);
    if (plan->head_dim == 128) {
        const size_t sm = enc_smem<128>();
        if (spectra_status st = set_smem(encode_generic_kernel<128>, sm)) return st;
        encode_generic_kernel<128><<<grid, kWarps * 32, sm, s>>>(pv, x, dt, T, token_stride, codes,
                                                                 sstride, norms, nstride, t0);
    } else {
        const size_t sm = enc_smem<64>();
        if (spectra_status st = set_smem(encode_generic_kernel<64>, sm)) return st;
        encode_generic_kernel<64><<<grid, kWarps * 32, sm, s>>>(pv, x, dt, T, token_stride, codes,
                                                                sstride, norms, nstride, t0);
    }
    return cuda_status(cudaGetLastError());
}

// 1-bit JL sketch of the key residuals ("Technisch Overzicht ...", TQ-QKV:
// a 1-bit QJL residual sketch on the key path).  Per 32-token group (lane =
// token): y = the latent coordinates of x, yhat = the dequantized codes
// already in the stream, r = y - yhat; bit j of the token is (<s_j, r> >= 0)
// for the rows s_j of the caller's Gaussian matrix S (D x D, latent
// coordinates), written as the group's D bit-plane words (word j, bit t mod
// 32); the residual norm ||r|| per token.  A block walks groups; its warps
// split the channels (for r) and then the rows of S (for the bits) in
// register blocks of kCB, with the rotation and S^T in shared memory.
constexpr int kQjlWarps = 8;

template <int D>
__host__ __device__ constexpr int qjl_st_stride() { return D + 4; }    // S^T rows: 16-byte aligned, few store conflicts

template <int D>
__global__ void __launch_bounds__(kQjlWarps * 32)
qjl_encode_kernel(PlanView pv, const float* __restrict__ S, const void* __restrict__ x, int dt, int64_t T,
                  int64_t tstride, const uint8_t* __restrict__ codes, int64_t sstride,
                  const float* __restrict__ norms, int64_t nstride, uint8_t* __restrict__ qbits, int64_t qstride,
                  float* __restrict__ qnorms, int64_t qnstride)
{
    constexpr int LD = D + 1;
    constexpr int SP = qjl_st_stride<D>();
    extern __shared__ __align__(16) float smem[];
    float* M = smem;                                 // [D][D] rotation
    float* St = M + D * D;                           // [D][SP] St[c][j] = S[j][c]
    float* xw = St + D * SP;                         // [32][LD] the group's tokens
    float* rw = xw + 32 * LD;                        // [32][LD] their residuals
    float* lv = rw + 32 * LD;                        // [8][256] Lloyd-Max levels
    float* rsc = lv + kMaxBits * kLmStride;          // [D]
    float* ysg = rsc + D;                            // [32] RWHT: ||x|| / sqrt(d) of each token
    int* bsh = reinterpret_cast<int*>(ysg + 32);     // [D]
    int* osh = bsh + D;                              // [D]
    uint32_t* ww = reinterpret_cast<uint32_t*>(osh + D);   // [8 D] the group's code words
    const int h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = pv.rec_bits[h];
    if (R > pv.max_rec_bits) return;
    load_matrix_dense<D>(pv, h, M);
    for (int e = threadIdx.x; e < D * D; e += blockDim.x) St[(e % D) * SP + e / D] = S[e];
    for (int e = threadIdx.x; e < kMaxBits * kLmStride; e += blockDim.x) lv[e] = pv.lm_level[e];
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        rsc[c] = pv.rscale[size_t(h) * D + c];
        bsh[c] = pv.bits[size_t(h) * D + c];
        osh[c] = pv.chan_off[size_t(h) * D + c];
    }
    const bool rwht = pv.basis == SPECTRA_BASIS_RWHT;
    const int64_t ngroups = (T + kGroup - 1) / kGroup;
    for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
        __syncthreads();                             // the previous group's buffers are free
        for (int e = threadIdx.x; e < 32 * D; e += blockDim.x) {
            const int r = e / D, i = e % D;
            const int64_t t = g * kGroup + r;
            xw[r * LD + i] = (t < T) ? load_elem(x, dt, t * tstride + int64_t(h) * D + i) : 0.f;
        }
        const uint32_t* words = reinterpret_cast<const uint32_t*>(codes + int64_t(h) * sstride) + g * R;
        for (int e = threadIdx.x; e < R; e += blockDim.x) ww[e] = words[e];
        const int64_t t = g * kGroup + lane;
        const bool live = t < T;
        if (warp == 0) ysg[lane] = (rwht && live) ? norms[int64_t(h) * nstride + t] * rsqrtf(float(D)) : 0.f;
        __syncthreads();
        // r = y - yhat, channels in blocks of kCB
        for (int cb = warp; cb < D / kCB; cb += kQjlWarps) {
            const int c0 = cb * kCB;
            float y[kCB];
            project_block<D, kCB>(M, xw + lane * LD, c0, y);
#pragma unroll
            for (int j = 0; j < kCB; ++j) {
                const int c = c0 + j, b = bsh[c];
                float yh = 0.f;
                if (b > 0) {
                    int code = 0;
                    for (int k = 0; k < b; ++k) code |= int((ww[osh[c] + k] >> lane) & 1u) << k;
                    if (pv.quant == SPECTRA_Q_UNIFORM3S) yh = rsc[c] * (float(code) + 0.5f - float(1 << (b - 1)));
                    else yh = (rwht ? ysg[lane] : rsc[c]) * lv[(b - 1) * kLmStride + code];
                }
                rw[lane * LD + c] = y[j] - yh;
            }
        }
        __syncthreads();
        if (warp == 0) {
            float n2 = 0.f;
            for (int c = 0; c < D; ++c) n2 = fmaf(rw[lane * LD + c], rw[lane * LD + c], n2);
            if (live) qnorms[int64_t(h) * qnstride + t] = sqrtf(n2);
        }
        // a_j = <s_j, r>, rows in blocks of kCB; word j of the group = the signs
        uint32_t* out = reinterpret_cast<uint32_t*>(qbits + int64_t(h) * qstride) + g * D;
        for (int jb = warp; jb < D / kCB; jb += kQjlWarps) {
            const int j0 = jb * kCB;
            float a[kCB];
#pragma unroll
            for (int j = 0; j < kCB; ++j) a[j] = 0.f;
#pragma unroll 4
            for (int c = 0; c < D; ++c) {
                const float rc = rw[lane * LD + c];
                const float4* sv = reinterpret_cast<const float4*>(St + c * SP + j0);
#pragma unroll
                for (int q = 0; q < kCB / 4; ++q) {
                    const float4 v = sv[q];
                    a[4 * q] = fmaf(v.x, rc, a[4 * q]);
                    a[4 * q + 1] = fmaf(v.y, rc, a[4 * q + 1]);
                    a[4 * q + 2] = fmaf(v.z, rc, a[4 * q + 2]);
                    a[4 * q + 3] = fmaf(v.w, rc, a[4 * q + 3]);
                }
            }
            uint32_t mine = 0;
#pragma unroll
            for (int j = 0; j < kCB; ++j) {
                const uint32_t wv = __ballot_sync(0xffffffffu, live && a[j] >= 0.f);
                if (lane == j) mine = wv;
            }
            if (lane < kCB) out[j0 + lane] = mine;
        }
    }
}

template <int D>
size_t qjl_smem()
{
    return sizeof(float) * (D * D + D * qjl_st_stride<D>() + 2 * 32 * (D + 1) + kMaxBits * kLmStride + D + 32) +
           sizeof(int) * 2 * D + sizeof(uint32_t) * 8 * D;
}

spectra_status launch_qjl_encode(const spectra_plan* plan, const float* S, const void* x, int dt, int64_t T,
                                 int64_t token_stride, const uint8_t* codes, int64_t sstride, const float* norms,
                                 int64_t nstride, uint8_t* qbits, int64_t qstride, float* qnorms, int64_t qnstride,
                                 cudaStream_t s)
{
    const PlanView pv = make_view(plan);
    const int64_t ngroups = (T + kGroup - 1) / kGroup;
    if (ngroups == 0) return SPECTRA_OK;
    // one block per SM (the shared-memory footprint) over all heads
    const int64_t per_head = std::max<int64_t>(1, 148 / plan->heads);
    dim3 grid(unsigned(std::min<int64_t>(ngroups, per_head)), plan->heads);
    if (plan->head_dim == 128) {
        if (spectra_status st = set_smem(qjl_encode_kernel<128>, qjl_smem<128>())) return st;
        qjl_encode_kernel<128><<<grid, kQjlWarps * 32, qjl_smem<128>(), s>>>(
            pv, S, x, dt, T, token_stride, codes, sstride, norms, nstride, qbits, qstride, qnorms, qnstride);
    } else {
        if (spectra_status st = set_smem(qjl_encode_kernel<64>, qjl_smem<64>())) return st;
        qjl_encode_kernel<64><<<grid, kQjlWarps * 32, qjl_smem<64>(), s>>>(
            pv, S, x, dt, T, token_stride, codes, sstride, norms, nstride, qbits, qstride, qnorms, qnstride);
    }
    return cuda_status(cudaGetLastError());
}

spectra_status launch_append_small(const spectra_plan* plan, const void* x, int dt, int64_t n, int64_t token_stride,
                                   uint8_t* codes, int64_t sstride, float* norms, int64_t nstride, int64_t t0,
                                   cudaStream_t s)
{
    const PlanView pv = make_view(plan);
    if (plan->head_dim == 128)
        append_small_kernel<128><<<plan->heads, 128, 0, s>>>(pv, x, dt, n, token_stride, codes, sstride, norms,
                                                             nstride, t0);
    else
        append_small_kernel<64><<<plan->heads, 64, 0, s>>>(pv, x, dt, n, token_stride, codes, sstride, norms,
                                                           nstride, t0);
    return cuda_status(cudaGetLastError());
}

spectra_status launch_decode_generic(const spectra_plan* plan, const uint8_t* codes, int64_t sstride,
                                     const float* norms, int64_t nstride, int64_t T, void* x_out,
                                     int out_dt, int64_t token_stride, cudaStream_t s)
{
    const PlanView pv = make_view(plan);
    const int64_t ngroups = (T + kGroup - 1) / kGroup;
    if (ngroups == 0) return SPECTRA_OK;
    dim3 grid(unsigned((ngroups + kDecWarps - 1) / kDecWarps), plan->heads);
    if (plan->head_dim == 128) {
        const size_t sm = dec_smem<128>();
        if (spectra_status st = set_smem(decode_generic_kernel<128>, sm)) return st;
        decode_generic_kernel<128><<<grid, kDecWarps * 32, sm, s>>>(pv, codes, sstride, norms, nstride, T,
                                                                 x_out, out_dt, token_stride);
    } else {
        const size_t sm = dec_smem<64>();
        if (spectra_status st = set_smem(decode_generic_kernel<64>, sm)) return st;
        decode_generic_kernel<64><<<grid, kDecWarps * 32, sm, s>>>(pv, codes, sstride, norms, nstride, T,
                                                                x_out, out_dt, token_stride);
    }
    return cuda_status(cudaGetLastError());
}

}  // namespace spectra
