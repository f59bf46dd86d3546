// attn.cu -- decode-step attention read straight from packed K/V streams,
// computed in the latent bases (CUDA-core path; any plan kind).
//
// "Sintesi Tecnica: SPECTRA", "Significato e Rivendicazioni": the latent
// space opens the way to attention computed directly in it.  With
// khat = B_K yk and vhat = B_V yv (the decode reconstructions),
//   <q, khat_t> = <B_K^T q, yk_t>   and   sum_t p_t vhat_t = B_V sum_t p_t yv_t,
// so scores use the rotated query qt = scale * B_K^T q against the latent
// K coordinates, the softmax-weighted sum runs over latent V coordinates,
// and one rotation by B_V at the end gives the output.
//
// Three launches: (1) qt for every (b, query head); (2) one block per
// (context split, kv head, batch) -- online softmax over tiles of 64 tokens
// for the Hq/Hkv query heads that share the kv head, partial (m, l, acc)
// to the workspace; (3) per (b, query head) merge the splits and rotate back.
#include "spectra_internal.cuh"

#include <cuda_bf16.h>
#include <math.h>
#include <stdlib.h>

#include <algorithm>

namespace spectra {

namespace {

constexpr int kTile = 64;           // tokens per tile (two bit-plane groups)
constexpr int kThreads = 256;
constexpr int kMaxGroup = 8;        // query heads per kv head

__device__ __forceinline__ float basis_entry(const PlanView& pv, int h, int i, int c, int D)
{
    if (pv.basis == SPECTRA_BASIS_EIGEN) return pv.basis_mat[(size_t(h) * D + i) * D + c];
    return float(pv.signs[size_t(h) * D + i] * hadamard_sign(i, c)) * rsqrtf(float(D));
}

// Optional 1-bit JL sketch of the key residuals ("Technisch Overzicht ...",
// TQ-QKV): per (b, kv head) stream, bit-plane words of D sketch bits per
// 32-token group and one residual norm per token; w = S qt per query head.
struct QjlArgs {
    const float* sketch;     // [D][D] Gaussian matrix (row j = s_j), latent coordinates
    const uint8_t* bits;
    int64_t stride;          // bytes between the (b, kv head) bit streams
    const float* norms;
    int64_t nstride;
    float* w;                // [B Hq][D] workspace
};

__global__ void attn_qrot_kernel(PlanView kp, const void* __restrict__ q, int q_dt, int Hq, int Hkv,
                                 float scale, float* __restrict__ qt, QjlArgs qj)
{
    const int D = kp.d;
    const int bj = blockIdx.x, j = bj % Hq;
    const int h = j / (Hq / Hkv);
    extern __shared__ float qs[];
    for (int i = threadIdx.x; i < D; i += blockDim.x) qs[i] = load_elem(q, q_dt, int64_t(bj) * D + i);
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        float a = 0.f;
        for (int i = 0; i < D; ++i) a = fmaf(basis_entry(kp, h, i, c, D), qs[i], a);
        qt[int64_t(bj) * D + c] = scale * a;
    }
    if (qj.bits) {
        __syncthreads();
        for (int j = threadIdx.x; j < D; j += blockDim.x) {
            float a = 0.f;
            for (int c = 0; c < D; ++c) a = fmaf(qj.sketch[j * D + c], qt[int64_t(bj) * D + c], a);
            qj.w[int64_t(bj) * D + j] = a;
        }
    }
}

// Split-context attention on CUDA cores (every plan the tensor-core kernel
// does not cover: Lloyd-Max and RWHT plans, head_dim 64, the QJL
// correction).  One block of 256 threads per (split, kv head, batch); per
// 64-token tile (two bit-plane groups):
//  * unpack: a thread per (group, channel) turns its b plane words into the
//    32 tokens' dequantized latent values y[t][c];
//  * scores: four threads per token, each over a quarter of the channels
//    (c = 4 i + quarter) for all GM query heads at once, reduced by shuffles;
//  * the QJL correction (optional) the same way over the tile's sign bits;
//  * P V: a thread per (channel, token subset) for all GM heads at once.
// Rows of y are D + 4 floats apart (4 mod 32 words): the score reads of a
// warp (8 tokens x 4 quarters) and the unpack / P V accesses (consecutive
// channels) are all free of bank conflicts.  K, the signs and V take turns
// in the one y buffer.
template <int D>
constexpr int ystride() { return D + 4; }
constexpr int kLvs = kLmStride + 1;   // level-table rows 257 floats apart (lanes of different widths)

// rkm, rvm: the plans' widest records (the double-buffered word stages)
template <int D, int GM>
size_t split_smem_t(int rkm, int rvm)
{
    return sizeof(float) * (size_t(2) * D * GM + size_t(kTile) * ystride<D>() + kTile * GM + 3 * GM +
                            kMaxBits * kLvs + 2 * kTile + 2 * D) +
           sizeof(int) * 4 * D + sizeof(uint32_t) * 2 * (2 * size_t(rkm) + 2 * size_t(rvm));
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(uint32_t(__cvta_generic_to_shared(dst))), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// the 32 tokens of group g (stream group g0 + g) of channel c into y[32 g + t][c]
template <int D>
__device__ __forceinline__ void unpack_channel_group(const PlanView& pv, int c, int g, int R, const uint32_t* words,
                                                     const int* bits, const int* off, const float* rsc,
                                                     const float* lv, const float* nrm, int ntok, float* y)
{
    constexpr int LD = ystride<D>();
    const int b = bits[c];
    float* yc = y + (32 * g) * LD + c;
    if (b == 0) {
#pragma unroll 4
        for (int t = 0; t < 32; ++t) yc[t * LD] = 0.f;
        return;
    }
    // the 32 codes as bytes: gather each plane's byte m, then 8 x 8 bit
    // transposes -- X[j] holds the codes of tokens 4 j .. 4 j + 3
    uint32_t pl[kMaxBits];
    const uint32_t* wp = words + g * R + off[c];
#pragma unroll
    for (int k = 0; k < kMaxBits; ++k) pl[k] = k < b ? wp[k] : 0u;
    uint32_t X[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        X[2 * m] = gather_byte(pl[0], pl[1], pl[2], pl[3], m);
        X[2 * m + 1] = gather_byte(pl[4], pl[5], pl[6], pl[7], m);
        transpose8(X[2 * m], X[2 * m + 1]);
    }
    const bool uni = pv.quant == SPECTRA_Q_UNIFORM3S;
    const bool rw = pv.basis == SPECTRA_BASIS_RWHT;
    const float sc = rsc[c], mid = 0.5f - float(1 << (b - 1));
    const float* lvb = lv + (b - 1) * kLvs;
#pragma unroll
    for (int t = 0; t < 32; ++t) {
        const int code = int(__byte_perm(X[t >> 2], 0u, 0x4440u | uint32_t(t & 3)));
        float v;
        if (uni) v = sc * (float(code) + mid);
        else v = (rw ? nrm[32 * g + t] : sc) * lvb[code];
        yc[t * LD] = (32 * g + t < ntok) ? v : 0.f;
    }
}

template <int D, int GM>
__global__ void __launch_bounds__(kThreads, 3)
attn_split_kernel(PlanView kp, PlanView vp, const float* __restrict__ qt, int Hq, int64_t ctx,
                  const uint8_t* __restrict__ kc, const uint8_t* __restrict__ vc, int64_t sstride,
                  const float* __restrict__ kn, const float* __restrict__ vn, int64_t nstride,
                  int nsplit, int split_len, float* __restrict__ part, QjlArgs qj)
{
    constexpr int LD = ystride<D>();
    extern __shared__ __align__(16) float smem[];
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int Hkv = kp.heads, G = Hq / Hkv;
    // records wider than the plans' bound are not read (the streams were sized by it)
    const int RKm = kp.max_rec_bits, RVm = vp.max_rec_bits;
    const int RK = kp.rec_bits[h] <= RKm ? kp.rec_bits[h] : 0, RV = vp.rec_bits[h] <= RVm ? vp.rec_bits[h] : 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    float* qT = smem;                       // [D][GM] q~ transposed (heads >= G zero)
    float* wT = qT + D * GM;                // [D][GM] QJL w = S q~, transposed
    float* y = wT + D * GM;                 // [kTile][LD] K, then the signs, then V
    float* St = y + kTile * LD;             // [kTile][GM] scores, then probabilities
    float* mrow = St + kTile * GM;          // [GM]
    float* lrow = mrow + GM;                // [GM]
    float* alpha = lrow + GM;               // [GM]
    float* lv = alpha + GM;                 // [8][kLvs] Gaussian levels (both plans share them)
    float* nrm = lv + kMaxBits * kLvs;      // [kTile] RWHT norms / sqrt(d) of the tile
    float* qnr = nrm + kTile;               // [kTile] QJL residual norms of the tile
    float* rscK = qnr + kTile;              // [D] per-channel tables of the two plans
    float* rscV = rscK + D;
    int* bitsK = reinterpret_cast<int*>(rscV + D);
    int* bitsV = bitsK + D;
    int* offK = bitsV + D;
    int* offV = offK + D;
    // [2 buffers][2 groups x RKm K words, then 2 groups x RVm V words]: the
    // next tile's words arrive (cp.async) while this tile is computed
    uint32_t* wb = reinterpret_cast<uint32_t*>(offV + D);
    const int WB = 2 * RKm + 2 * RVm;

    for (int e = tid; e < D * GM; e += kThreads) {
        const int c = e / GM, j = e % GM;
        qT[e] = j < G ? qt[(int64_t(b) * Hq + h * G + j) * D + c] : 0.f;
        wT[e] = (qj.bits && j < G) ? qj.w[(int64_t(b) * Hq + h * G + j) * D + c] : 0.f;
    }
    {
        // the Gaussian levels, from whichever plan has them (the tables are the same)
        const float* lsrc = kp.quant == SPECTRA_Q_LLOYD_GAUSS ? kp.lm_level : vp.lm_level;
        for (int e = tid; e < kMaxBits * kLmStride; e += kThreads)
            lv[(e / kLmStride) * kLvs + e % kLmStride] = lsrc[e];
    }
    if (tid < GM) { mrow[tid] = -INFINITY; lrow[tid] = 0.f; }

    const int64_t sid = int64_t(b) * Hkv + h;
    const uint32_t* ks = reinterpret_cast<const uint32_t*>(kc + sid * sstride);
    const uint32_t* vs = reinterpret_cast<const uint32_t*>(vc + sid * sstride);
    const float* knr = kn ? kn + sid * nstride : nullptr;
    const float* vnr = vn ? vn + sid * nstride : nullptr;
    const int64_t s0 = int64_t(split) * split_len;
    const int64_t s1 = min(ctx, s0 + split_len);

    for (int c = tid; c < D; c += kThreads) {
        bitsK[c] = kp.bits[size_t(h) * D + c];
        offK[c] = kp.chan_off[size_t(h) * D + c];
        rscK[c] = kp.rscale[size_t(h) * D + c];
        bitsV[c] = vp.bits[size_t(h) * D + c];
        offV[c] = vp.chan_off[size_t(h) * D + c];
        rscV[c] = vp.rscale[size_t(h) * D + c];
    }
    // the K and V words of the tile at t0 into buffer buf, asynchronously
    auto prefetch = [&](int64_t t0, int buf) {
        uint32_t* wk = wb + buf * WB;
        uint32_t* wv = wk + 2 * RKm;
        const int64_t g0 = t0 / kGroup;
        for (int e = tid; e < 2 * RK; e += kThreads) {
            const int64_t gg = g0 + e / RK;
            if (gg * kGroup < s1) cp_async4(wk + e, ks + gg * RK + (e % RK));
            else wk[e] = 0u;
        }
        for (int e = tid; e < 2 * RV; e += kThreads) {
            const int64_t gg = g0 + e / RV;
            if (gg * kGroup < s1) cp_async4(wv + e, vs + gg * RV + (e % RV));
            else wv[e] = 0u;
        }
        cp_async_commit();
    };
    // RWHT: the tile's norms / sqrt(d)
    auto stage_norms = [&](const PlanView& pv, const float* norms, int64_t t0) {
        if (pv.basis == SPECTRA_BASIS_RWHT)
            for (int t = tid; t < kTile; t += kThreads)
                nrm[t] = (t0 + t < s1) ? norms[t0 + t] * rsqrtf(float(D)) : 0.f;
    };
    auto unpack = [&](const PlanView& pv, int R, int ntok, const uint32_t* words, const int* bits, const int* off,
                      const float* rsc) {
        for (int e = tid; e < 2 * D; e += kThreads)
            unpack_channel_group<D>(pv, e % D, e / D, R, words, bits, off, rsc, lv, nrm, ntok, y);
    };

    // P V: thread = (channel c, token subset); GM heads at once
    constexpr int kSub = kThreads / D;             // token subsets (2 for d = 128, 4 for 64)
    constexpr int kSubTok = kTile / kSub;
    const int pc = tid % D, psub = tid / D;
    float acc[GM];
#pragma unroll
    for (int j = 0; j < GM; ++j) acc[j] = 0.f;
    __syncthreads();

    if (s0 < s1) prefetch(s0, 0);
    int buf = 0;
    for (int64_t t0 = s0; t0 < s1; t0 += kTile, buf ^= 1) {
        const int ntok = int(min(int64_t(kTile), s1 - t0));
        const uint32_t* wk = wb + buf * WB;
        const uint32_t* wv = wk + 2 * RKm;
        if (t0 + kTile < s1) {
            prefetch(t0 + kTile, buf ^ 1);   // the buffer tile - 1 used: free since its last barrier
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        // ---- K: unpack, scores
        stage_norms(kp, knr, t0);
        __syncthreads();
        unpack(kp, RK, ntok, wk, bitsK, offK, rscK);
        __syncthreads();
        const int st = tid >> 2, qd = tid & 3;     // token, channel quarter
        {
            float a[GM];
#pragma unroll
            for (int j = 0; j < GM; ++j) a[j] = 0.f;
            const float* yr = y + st * LD;
#pragma unroll 4
            for (int i = 0; i < D / 4; ++i) {
                const int c = 4 * i + qd;
                const float yv = yr[c];
                const float4* qv = reinterpret_cast<const float4*>(qT + c * GM);
#pragma unroll
                for (int j4 = 0; j4 < GM / 4; ++j4) {
                    const float4 q4 = qv[j4];
                    a[4 * j4] = fmaf(q4.x, yv, a[4 * j4]);
                    a[4 * j4 + 1] = fmaf(q4.y, yv, a[4 * j4 + 1]);
                    a[4 * j4 + 2] = fmaf(q4.z, yv, a[4 * j4 + 2]);
                    a[4 * j4 + 3] = fmaf(q4.w, yv, a[4 * j4 + 3]);
                }
            }
#pragma unroll
            for (int j = 0; j < GM; ++j) {
                a[j] += __shfl_xor_sync(0xffffffffu, a[j], 1);
                a[j] += __shfl_xor_sync(0xffffffffu, a[j], 2);
            }
            if (qd == 0) {
#pragma unroll
                for (int j = 0; j < GM; ++j) St[st * GM + j] = (st < ntok) ? a[j] : -INFINITY;
            }
        }
        if (qj.bits) {
            // QJL correction: + sqrt(pi/2)/d ||r_t|| sum_i w_ji (2 b_i(t) - 1)
            __syncthreads();                          // the scores have read y
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(qj.bits + sid * qj.stride);
            const int64_t g0 = t0 / kGroup;
            for (int e = tid; e < 2 * D; e += kThreads) {
                const int g = e / D, i = e % D;
                const uint32_t w = (32 * g < ntok) ? qw[(g0 + g) * D + i] : 0u;
                float* yc = y + (32 * g) * LD + i;
#pragma unroll 4
                for (int t = 0; t < 32; ++t) yc[t * LD] = ((w >> t) & 1u) ? 1.f : -1.f;
            }
            for (int t = tid; t < kTile; t += kThreads)
                qnr[t] = (t0 + t < s1) ? qj.norms[sid * qj.nstride + t0 + t] : 0.f;
            __syncthreads();
            float a[GM];
#pragma unroll
            for (int j = 0; j < GM; ++j) a[j] = 0.f;
            const float* yr = y + st * LD;
#pragma unroll 4
            for (int i = 0; i < D / 4; ++i) {
                const int c = 4 * i + qd;
                const float zv = yr[c];
                const float4* wv = reinterpret_cast<const float4*>(wT + c * GM);
#pragma unroll
                for (int j4 = 0; j4 < GM / 4; ++j4) {
                    const float4 w4 = wv[j4];
                    a[4 * j4] = fmaf(w4.x, zv, a[4 * j4]);
                    a[4 * j4 + 1] = fmaf(w4.y, zv, a[4 * j4 + 1]);
                    a[4 * j4 + 2] = fmaf(w4.z, zv, a[4 * j4 + 2]);
                    a[4 * j4 + 3] = fmaf(w4.w, zv, a[4 * j4 + 3]);
                }
            }
#pragma unroll
            for (int j = 0; j < GM; ++j) {
                a[j] += __shfl_xor_sync(0xffffffffu, a[j], 1);
                a[j] += __shfl_xor_sync(0xffffffffu, a[j], 2);
            }
            const float cst = 1.25331413731550025f / float(D);   // sqrt(pi / 2) / m, m = d
            if (qd == 0 && st < ntok) {
#pragma unroll
                for (int j = 0; j < GM; ++j) St[st * GM + j] += cst * qnr[st] * a[j];
            }
        }
        __syncthreads();                              // scores complete; y free
        // ---- softmax over the tile, one warp per query head
        if (warp < G) {
            const int j = warp;
            const float x0 = St[lane * GM + j], x1 = St[(lane + 32) * GM + j];
            float mx = fmaxf(x0, x1);
            for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mold = mrow[j];
            const float mnew = fmaxf(mold, mx);
            const float p0 = __expf(x0 - mnew), p1 = __expf(x1 - mnew);
            St[lane * GM + j] = p0;
            St[(lane + 32) * GM + j] = p1;
            float ps = p0 + p1;
            for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            if (lane == 0) {
                const float al = (mold == -INFINITY) ? 0.f : __expf(mold - mnew);
                alpha[j] = al;
                lrow[j] = lrow[j] * al + ps;
                mrow[j] = mnew;
            }
        }
        // ---- V: unpack, P V
        stage_norms(vp, vnr, t0);
        __syncthreads();
        unpack(vp, RV, ntok, wv, bitsV, offV, rscV);
        __syncthreads();
        {
#pragma unroll
            for (int j = 0; j < GM; ++j) acc[j] *= (j < G) ? alpha[j] : 0.f;
            const int tb = psub * kSubTok;
#pragma unroll 4
            for (int t = tb; t < tb + kSubTok; ++t) {
                const float yv = y[t * LD + pc];
                const float4* pv4 = reinterpret_cast<const float4*>(St + t * GM);
#pragma unroll
                for (int j4 = 0; j4 < GM / 4; ++j4) {
                    const float4 p4 = pv4[j4];
                    acc[4 * j4] = fmaf(p4.x, yv, acc[4 * j4]);
                    acc[4 * j4 + 1] = fmaf(p4.y, yv, acc[4 * j4 + 1]);
                    acc[4 * j4 + 2] = fmaf(p4.z, yv, acc[4 * j4 + 2]);
                    acc[4 * j4 + 3] = fmaf(p4.w, yv, acc[4 * j4 + 3]);
                }
            }
        }
        __syncthreads();                              // y, St, the tables free for the next tile
    }
    // token subsets -> one sum per (head, channel), through the y buffer
    float* red = y;                                   // [kSub][GM][D]
#pragma unroll
    for (int j = 0; j < GM; ++j) red[(psub * GM + j) * D + pc] = acc[j];
    __syncthreads();
    float* out = part + ((int64_t(b) * Hq + h * G) * nsplit + split) * (D + 2);
    for (int e = tid; e < G * D; e += kThreads) {
        const int j = e / D, c = e % D;
        float a = 0.f;
#pragma unroll
        for (int u = 0; u < kSub; ++u) a += red[(u * GM + j) * D + c];
        out[int64_t(j) * nsplit * (D + 2) + 2 + c] = a;
    }
    if (tid < G) {
        out[int64_t(tid) * nsplit * (D + 2) + 0] = mrow[tid];
        out[int64_t(tid) * nsplit * (D + 2) + 1] = lrow[tid];
    }
}

// One block per (batch, query head): merge its context splits, then
// out[b, hq] = B_V latent with B_V staged in shared memory (rows padded to
// D + 1 floats: conflict-free row reads).  The split weights exp(m_s - M)
// are computed once; the channel sums read the splits with independent
// loads in flight (the partials live in L2).
// code_domain: the partials hold sum_t p_t z_c(t) with z = code - 2^(b-1)
// (tensor-core path, uniform quantizer); the merged value is dequantized as
// Delta_c (z_mean + 1/2) before the rotation.
__global__ void __launch_bounds__(256)
attn_combine_kernel(PlanView vp, const float* __restrict__ part, int Hq, int nsplit, int code_domain,
                    const float* __restrict__ win, float* __restrict__ out)
{
    const int D = vp.d, Hkv = vp.heads, G = Hq / Hkv;
    const int bq = blockIdx.x, hq = bq % Hq, b = bq / Hq, h = hq / G;
    const int LD = D + 1;
    extern __shared__ float sm[];
    float* Bs = sm;                     // [D][LD]
    float* os = Bs + D * LD;            // [D]
    float* red = os + D;                // [4][D] partial sums
    float* stat = red + 4 * D;          // [1]: L
    float* sc = stat + 4;               // [nsplit] split weights
    const bool eig = vp.basis == SPECTRA_BASIS_EIGEN;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (eig) {
        const float4* src = reinterpret_cast<const float4*>(vp.basis_mat + size_t(h) * D * D);
        for (int e = tid; e < D * D / 4; e += blockDim.x) {
            const float4 v = src[e];
            const int i = (4 * e) / D, c = (4 * e) % D;
            float* d = Bs + i * LD + c;
            d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
        }
    }
    const float* pp = part + (int64_t(b) * Hq + hq) * nsplit * (D + 2);
    if (warp == 0) {
        float M = -INFINITY;
        for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, pp[int64_t(s) * (D + 2)]);
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        // the recent window's partial (m, l, o in the original basis) joins the maximum
        const float mw = win ? win[(int64_t(b) * Hq + hq) * (D + 2)] : -INFINITY;
        M = fmaxf(M, mw);
        float L = 0.f;
        for (int s = lane; s < nsplit; s += 32) {
            const float m = pp[int64_t(s) * (D + 2)];
            const float w = (m != -INFINITY) ? __expf(m - M) : 0.f;
            sc[s] = w;
            L = fmaf(pp[int64_t(s) * (D + 2) + 1], w, L);
        }
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) {
            const float ww = (mw != -INFINITY) ? __expf(mw - M) : 0.f;
            const float Lw = win ? ww * win[(int64_t(b) * Hq + hq) * (D + 2) + 1] : 0.f;
            stat[0] = L + Lw;      // all tokens
            stat[1] = L;           // packed tokens
            stat[2] = ww;          // window weight
        }
    }
    __syncthreads();
    const int nh = int(blockDim.x) / D;          // split phases (2 for d = 128, 4 for d = 64)
    {
        const int c = tid % D, ph = tid / D;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        int s = ph;
        for (; s + 3 * nh < nsplit; s += 4 * nh) {
            const float v0 = pp[int64_t(s) * (D + 2) + 2 + c], v1 = pp[int64_t(s + nh) * (D + 2) + 2 + c];
            const float v2 = pp[int64_t(s + 2 * nh) * (D + 2) + 2 + c], v3 = pp[int64_t(s + 3 * nh) * (D + 2) + 2 + c];
            a0 = fmaf(v0, sc[s], a0);
            a1 = fmaf(v1, sc[s + nh], a1);
            a2 = fmaf(v2, sc[s + 2 * nh], a2);
            a3 = fmaf(v3, sc[s + 3 * nh], a3);
        }
        for (; s < nsplit; s += nh) a0 = fmaf(pp[int64_t(s) * (D + 2) + 2 + c], sc[s], a0);
        red[ph * D + c] = (a0 + a1) + (a2 + a3);
    }
    __syncthreads();
    if (tid < D) {
        const int c = tid;
        float a = 0.f;
        for (int k = 0; k < nh; ++k) a += red[k * D + c];
        const float L = stat[0], Lp = stat[1];
        float y;
        if (code_domain) {
            // a = sum_t p z: the latent value is Delta (z + 1/2)
            const int bc = vp.bits[size_t(h) * D + c];
            y = (bc > 0 && L > 0.f) ? vp.rscale[size_t(h) * D + c] * (a + 0.5f * Lp) / L : 0.f;
        } else {
            y = (L > 0.f) ? a / L : 0.f;
        }
        os[c] = y;
    }
    __syncthreads();
    {
        const int i = tid % D, ph = tid / D, cl = D / nh;   // output i, channel slice ph
        float a = 0.f;
        if (eig) {
            for (int c = ph * cl; c < (ph + 1) * cl; ++c) a = fmaf(Bs[i * LD + c], os[c], a);
        } else {
            for (int c = ph * cl; c < (ph + 1) * cl; ++c) a = fmaf(basis_entry(vp, h, i, c, D), os[c], a);
        }
        red[ph * D + i] = a;
    }
    __syncthreads();
    if (tid < D) {
        float a = 0.f;
        for (int k = 0; k < nh; ++k) a += red[k * D + tid];
        if (win) {
            const float L = stat[0];
            a += (L > 0.f) ? stat[2] * win[(int64_t(b) * Hq + hq) * (D + 2) + 2 + tid] / L : 0.f;
        }
        out[(int64_t(b) * Hq + hq) * D + tid] = a;
    }
}

// The recent window: per (batch, query head), softmax partials over W
// uncompressed tokens in the original basis -- s_t = scale <q, k_t>, m, l and
// o = sum_t exp(s_t - m) v_t -- for the combine, which merges them with the
// packed history's split partials.  k_t / v_t at
// win[(b W + t) * win_stride + h d + i] (bf16 or f32).
__global__ void __launch_bounds__(256)
attn_window_kernel(const void* __restrict__ q, int q_dt, int Hq, int Hkv, int D, const void* __restrict__ kw,
                   const void* __restrict__ vw, int w_dt, int64_t W, int64_t wstride, float scale,
                   float* __restrict__ wpart)
{
    extern __shared__ float wsm[];
    float* qs = wsm;                 // [D]
    float* sc = qs + D;              // [W]
    __shared__ float red[8];
    const int bq = blockIdx.x, hq = bq % Hq, b = bq / Hq, h = hq / (Hq / Hkv);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    for (int i = tid; i < D; i += blockDim.x) qs[i] = scale * load_elem(q, q_dt, int64_t(bq) * D + i);
    __syncthreads();
    // one warp per token: lanes over channels
    float mx = -INFINITY;
    for (int64_t t = warp; t < W; t += nw) {
        const int64_t base = (int64_t(b) * W + t) * wstride + int64_t(h) * D;
        float a = 0.f;
        for (int i = lane; i < D; i += 32) a = fmaf(qs[i], load_elem(kw, w_dt, base + i), a);
        for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) sc[t] = a;
        mx = fmaxf(mx, a);
    }
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < nw; ++w) M = fmaxf(M, red[w]);
    __syncthreads();
    float ls = 0.f;
    for (int64_t t = tid; t < W; t += blockDim.x) {
        const float p = __expf(sc[t] - M);
        sc[t] = p;
        ls += p;
    }
    for (int o = 16; o; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    if (lane == 0) red[warp] = ls;
    __syncthreads();
    float* wp = wpart + int64_t(bq) * (D + 2);
    for (int i = tid; i < D; i += blockDim.x) {
        float o = 0.f;
        for (int64_t t = 0; t < W; ++t) o = fmaf(sc[t], load_elem(vw, w_dt, (int64_t(b) * W + t) * wstride + int64_t(h) * D + i), o);
        wp[2 + i] = o;
    }
    if (tid == 0) {
        float L = 0.f;
        for (int w = 0; w < nw; ++w) L += red[w];
        wp[0] = M;
        wp[1] = L;
    }
}

size_t combine_smem(int D, int nsplit) { return sizeof(float) * (size_t(D) * (D + 1) + 5 * size_t(D) + 4 + nsplit); }


// Context split length, a multiple of 256 tokens (the tensor-core tile):
// about 2048 blocks over the (batch, kv head) pairs -- counted as one kv
// head per four query heads, so the size of the workspace depends on
// (B, Hq, ctx) alone -- and at least 1024 tokens per split.
int split_len_of(int B, int Hq, int64_t ctx)
{
    const int64_t pairs = (int64_t(B) * Hq + 3) / 4;
    int64_t L = (ctx * pairs + 2047) / 2048;
    L = (L + 255) / 256 * 256;
    if (L < 1024) L = 1024;
    if (L > (int64_t(1) << 30)) L = int64_t(1) << 30;
    return int(L);
}
int nsplit_of(int B, int Hq, int64_t ctx)
{
    const int64_t L = split_len_of(B, Hq, ctx);
    return int((ctx + L - 1) / L);
}

}  // namespace

size_t attn_tc_extra_bytes(int B, int Hkv);   // attn_tc.cu
spectra_status launch_attn_tc(const spectra_plan* kplan, const spectra_plan* vplan, const void* q, int q_dt,
                              int B, int Hq, const uint8_t* kc, const uint8_t* vc, int64_t sstride, int64_t ctx,
                              float scale, float* part, int nsplit, int split_len, void* extra,
                              cudaStream_t s, bool* done);
spectra_status launch_attn_lv(const spectra_plan* kplan, const spectra_plan* vplan, const float* qt, int B, int Hq,
                              const uint8_t* kc, const uint8_t* vc, int64_t sstride, const float* kn,
                              const float* vn, int64_t nstride, int64_t ctx, float* part, int nsplit, int split_len,
                              const uint8_t* qbits, int64_t qstride, const float* qnorms, int64_t qnstride,
                              const float* qw, cudaStream_t s, bool* done);   // attn_lv.cu

spectra_status launch_combine(const PlanView& vp, const float* part, int B, int Hq, int nsplit, int code_domain,
                              const float* win, float* out, cudaStream_t s)
{
    const size_t sm = combine_smem(vp.d, nsplit);
    if (spectra_status st = set_smem(attn_combine_kernel, sm)) return st;
    attn_combine_kernel<<<B * Hq, 256, sm, s>>>(vp, part, Hq, nsplit, code_domain, win, out);
    return cuda_status(cudaGetLastError());
}

// [qt (B Hq d f32) | split partials | tensor-core operands (sized for Hkv <= Hq) |
//  recent-window partials (B Hq (d + 2) f32)]
size_t attn_workspace_bytes(int B, int Hq, int d, int64_t ctx)
{
    const size_t qt = align256(sizeof(float) * size_t(B) * Hq * d);
    const size_t part = align256(sizeof(float) * size_t(B) * Hq * nsplit_of(B, Hq, ctx) * (d + 2));
    const size_t win = align256(sizeof(float) * size_t(B) * Hq * (d + 2));
    const size_t qjw = align256(sizeof(float) * size_t(B) * Hq * d);
    return qt + part + attn_tc_extra_bytes(B, Hq) + win + qjw;
}

spectra_status launch_attn(const spectra_plan* kplan, const spectra_plan* vplan, const void* q,
                           int q_dt, int B, int Hq, const uint8_t* kc, const uint8_t* vc,
                           int64_t sstride, const float* kn, const float* vn, int64_t nstride,
                           int64_t ctx, float scale, float* out, void* ws, size_t ws_bytes,
                           cudaStream_t s, const AttnWindow* window, const AttnQjl* qjl)
{
    const int D = kplan->head_dim, Hkv = kplan->heads;
    if (Hq / Hkv > kMaxGroup) return SPECTRA_ERR_UNSUPPORTED;
    const PlanView kp = make_view(kplan), vp = make_view(vplan);
    const int nsplit = ctx > 0 ? nsplit_of(B, Hq, ctx) : 0;
    const int split_len = split_len_of(B, Hq, ctx);
    float* qt = static_cast<float*>(ws);
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                           align256(sizeof(float) * size_t(B) * Hq * D));
    void* extra = reinterpret_cast<uint8_t*>(part) + align256(sizeof(float) * size_t(B) * Hq * nsplit_of(B, Hq, ctx) * (D + 2));
    float* wpart = nullptr;
    if (window && window->W > 0) {
        wpart = reinterpret_cast<float*>(static_cast<uint8_t*>(extra) + attn_tc_extra_bytes(B, Hq));
        const size_t sm = sizeof(float) * (size_t(D) + size_t(window->W));
        if (sm > 227 * 1024) return SPECTRA_ERR_UNSUPPORTED;
        if (spectra_status st = set_smem(attn_window_kernel, sm)) return st;
        attn_window_kernel<<<B * Hq, 256, sm, s>>>(q, q_dt, Hq, Hkv, D, window->k, window->v, window->dt,
                                                   window->W, window->stride, scale, wpart);
        if (spectra_status st = cuda_status(cudaGetLastError())) return st;
    }
    if (nsplit == 0) return launch_combine(vp, part, B, Hq, 0, 0, wpart, out, s);
    QjlArgs qj{nullptr, nullptr, 0, nullptr, 0, nullptr};
    if (qjl) {
        qj.sketch = qjl->sketch;
        qj.bits = qjl->bits;
        qj.stride = qjl->stride;
        qj.norms = qjl->norms;
        qj.nstride = qjl->nstride;
        qj.w = reinterpret_cast<float*>(static_cast<uint8_t*>(extra) + attn_tc_extra_bytes(B, Hq) +
                                        align256(sizeof(float) * size_t(B) * Hq * (D + 2)));
    }
    const int fam = kernel_family();
    bool have_qt = false;
    if (fam != SPECTRA_KERNELS_CUDA_CORE) {
        // the bit-plane kernel (uniform quantizer, eigenbasis, <= 4 query
        // heads per kv head, no sketch), else the level-table kernel (any
        // plan pair, with or without the sketch correction)
        bool done = false;
        spectra_status st = SPECTRA_OK;
        if (!qjl) {
            st = launch_attn_tc(kplan, vplan, q, q_dt, B, Hq, kc, vc, sstride, ctx, scale, part, nsplit, split_len,
                                extra, s, &done);
            if (st) return st;
            if (done) return launch_combine(vp, part, B, Hq, nsplit, 1, wpart, out, s);
        }
        attn_qrot_kernel<<<B * Hq, D, D * sizeof(float), s>>>(kp, q, q_dt, Hq, Hkv, scale, qt, qj);
        if (spectra_status e = cuda_status(cudaGetLastError())) return e;
        have_qt = true;
        st = launch_attn_lv(kplan, vplan, qt, B, Hq, kc, vc, sstride, kn, vn, nstride, ctx, part, nsplit, split_len,
                            qj.bits, qj.stride, qj.norms, qj.nstride, qj.w, s, &done);
        if (st) return st;
        if (done) return launch_combine(vp, part, B, Hq, nsplit, 0, wpart, out, s);
        if (fam == SPECTRA_KERNELS_TENSOR_CORE) return SPECTRA_ERR_UNSUPPORTED;
    }
    if (!have_qt) attn_qrot_kernel<<<B * Hq, D, D * sizeof(float), s>>>(kp, q, q_dt, Hq, Hkv, scale, qt, qj);
    dim3 grid(nsplit, Hkv, B);
    const int rkm = std::max(kplan->max_rec_bits, 1), rvm = std::max(vplan->max_rec_bits, 1);
    auto go = [&](auto kern, size_t sm) -> spectra_status {
        if (spectra_status st = set_smem(kern, sm)) return st;
        kern<<<grid, kThreads, sm, s>>>(kp, vp, qt, Hq, ctx, kc, vc, sstride, kn, vn, nstride, nsplit, split_len,
                                        part, qj);
        return SPECTRA_OK;
    };
    spectra_status gst;
    if (D == 128)
        gst = Hq / Hkv <= 4 ? go(attn_split_kernel<128, 4>, split_smem_t<128, 4>(rkm, rvm))
                            : go(attn_split_kernel<128, 8>, split_smem_t<128, 8>(rkm, rvm));
    else
        gst = Hq / Hkv <= 4 ? go(attn_split_kernel<64, 4>, split_smem_t<64, 4>(rkm, rvm))
                            : go(attn_split_kernel<64, 8>, split_smem_t<64, 8>(rkm, rvm));
    if (gst) return gst;
    if (spectra_status st = cuda_status(cudaGetLastError())) return st;
    return launch_combine(vp, part, B, Hq, nsplit, 0, wpart, out, s);
}

}  // namespace spectra
