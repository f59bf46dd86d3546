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

struct Side {            // per-plan tables staged in shared memory
    int* bits;
    int* off;
    float* rsc;
    uint32_t* words;     // [2][R]
};

template <int D>
__device__ void unpack_tile(const PlanView& pv, const Side& sd, int h, int R, const uint32_t* stream,
                            const float* norms, int64_t t0, int64_t tend, float* y, const float* lv)
{
    constexpr int LD = D + 1;
    // stage the two groups' words
    const int64_t g0 = t0 / kGroup;
    for (int e = threadIdx.x; e < 2 * R; e += blockDim.x) {
        const int64_t gg = g0 + e / R;
        sd.words[e] = (gg * kGroup < tend) ? stream[gg * R + (e % R)] : 0u;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
        const int t = e / D, c = e % D;
        const int b = sd.bits[c];
        float v = 0.f;
        if (b > 0 && t0 + t < tend) {
            const uint32_t* w = sd.words + (t >> 5) * R + sd.off[c];
            int code = 0;
            for (int k = 0; k < b; ++k) code |= int((w[k] >> (t & 31)) & 1u) << k;
            if (pv.quant == SPECTRA_Q_UNIFORM3S)
                v = sd.rsc[c] * (float(code) + 0.5f - float(1 << (b - 1)));
            else {
                const float s = (pv.basis == SPECTRA_BASIS_RWHT)
                                    ? norms[t0 + t] * rsqrtf(float(D)) : sd.rsc[c];
                v = s * lv[(b - 1) * kLmStride + code];
            }
        }
        y[t * LD + c] = v;
    }
    __syncthreads();
}

template <int D>
__global__ void __launch_bounds__(kThreads)
attn_split_kernel(PlanView kp, PlanView vp, const float* __restrict__ qt, int Hq, int64_t ctx,
                  const uint8_t* __restrict__ kc, const uint8_t* __restrict__ vc, int64_t sstride,
                  const float* __restrict__ kn, const float* __restrict__ vn, int64_t nstride,
                  int nsplit, int split_len, float* __restrict__ part, QjlArgs qj)
{
    constexpr int LD = D + 1;
    extern __shared__ float smem[];
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int Hkv = kp.heads, G = Hq / Hkv;
    const int RK = kp.rec_bits[h], RV = vp.rec_bits[h];

    float* qs = smem;                       // [G][D]
    float* yk = qs + kMaxGroup * D;         // [kTile][LD]
    float* yv = yk + kTile * LD;            // [kTile][LD]
    float* S = yv + kTile * LD;             // [G][kTile]
    float* mrow = S + kMaxGroup * kTile;    // [G]
    float* lrow = mrow + kMaxGroup;         // [G]
    float* alpha = lrow + kMaxGroup;        // [G]
    float* lvK = alpha + kMaxGroup;         // [8][256]
    float* lvV = lvK + kMaxBits * kLmStride;
    Side sk, sv;
    sk.rsc = lvV + kMaxBits * kLmStride;
    sv.rsc = sk.rsc + D;
    sk.bits = reinterpret_cast<int*>(sv.rsc + D);
    sv.bits = sk.bits + D;
    sk.off = sv.bits + D;
    sv.off = sk.off + D;
    sk.words = reinterpret_cast<uint32_t*>(sv.off + D);
    sv.words = sk.words + 2 * 8 * D;

    for (int e = threadIdx.x; e < G * D; e += blockDim.x)
        qs[e] = qt[(int64_t(b) * Hq + h * G) * D + e];
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        sk.bits[c] = kp.bits[size_t(h) * D + c];
        sv.bits[c] = vp.bits[size_t(h) * D + c];
        sk.off[c] = kp.chan_off[size_t(h) * D + c];
        sv.off[c] = vp.chan_off[size_t(h) * D + c];
        sk.rsc[c] = kp.rscale[size_t(h) * D + c];
        sv.rsc[c] = vp.rscale[size_t(h) * D + c];
    }
    for (int e = threadIdx.x; e < kMaxBits * kLmStride; e += blockDim.x) {
        lvK[e] = kp.lm_level[e];
        lvV[e] = vp.lm_level[e];
    }
    if (threadIdx.x < kMaxGroup) { mrow[threadIdx.x] = -INFINITY; lrow[threadIdx.x] = 0.f; }

    const int64_t sid = int64_t(b) * Hkv + h;
    const uint32_t* ks = reinterpret_cast<const uint32_t*>(kc + sid * sstride);
    const uint32_t* vs = reinterpret_cast<const uint32_t*>(vc + sid * sstride);
    const float* knr = kn ? kn + sid * nstride : nullptr;
    const float* vnr = vn ? vn + sid * nstride : nullptr;
    const int64_t s0 = int64_t(split) * split_len;
    const int64_t s1 = min(ctx, s0 + split_len);

    // each thread owns outputs (j, c) for e = tid + k*blockDim
    constexpr int kOwn = kMaxGroup * D / kThreads;
    float acc[kOwn];
#pragma unroll
    for (int k = 0; k < kOwn; ++k) acc[k] = 0.f;
    __syncthreads();

    for (int64_t t0 = s0; t0 < s1; t0 += kTile) {
        unpack_tile<D>(kp, sk, h, RK, ks, knr, t0, s1, yk, lvK);
        for (int e = threadIdx.x; e < G * kTile; e += blockDim.x) {
            const int j = e / kTile, t = e % kTile;
            float a = 0.f;
            for (int c = 0; c < D; ++c) a = fmaf(qs[j * D + c], yk[t * LD + c], a);
            S[j * kTile + t] = (t0 + t < s1) ? a : -INFINITY;
        }
        __syncthreads();
        if (qj.bits) {
            // QJL correction: + sqrt(pi/2)/D ||r_t|| sum_i w_ji (2 b_i(t) - 1), w = S_jl qt
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(qj.bits + sid * qj.stride);
            const float* qnr = qj.norms + sid * qj.nstride;
            float* zs = yv;                         // [kTile][LD] signs, free until the V unpack
            const int64_t g0 = t0 / kGroup;
            for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
                const int t = e / D, i = e % D;
                const int64_t gg = g0 + t / kGroup;
                const bool in = t0 + t < s1;
                const uint32_t w = in ? qw[gg * D + i] : 0u;
                zs[t * LD + i] = ((w >> (t & 31)) & 1u) ? 1.f : -1.f;
            }
            __syncthreads();
            const float cst = 1.25331413731550025f / float(D);   // sqrt(pi / 2) / m, m = d
            for (int e = threadIdx.x; e < G * kTile; e += blockDim.x) {
                const int j = e / kTile, t = e % kTile;
                if (t0 + t >= s1) continue;
                const float* wj = qj.w + (int64_t(b) * Hq + h * G + j) * D;
                float a = 0.f;
                for (int i = 0; i < D; ++i) a = fmaf(wj[i], zs[t * LD + i], a);
                S[j * kTile + t] += cst * qnr[t0 + t] * a;
            }
            __syncthreads();
        }
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (warp < G) {
            float mx = fmaxf(S[warp * kTile + lane], S[warp * kTile + lane + 32]);
            for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mold = mrow[warp];
            const float mnew = fmaxf(mold, mx);
            const float p0 = __expf(S[warp * kTile + lane] - mnew);
            const float p1 = __expf(S[warp * kTile + lane + 32] - mnew);
            S[warp * kTile + lane] = p0;
            S[warp * kTile + lane + 32] = p1;
            float ps = p0 + p1;
            for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            if (lane == 0) {
                const float al = (mold == -INFINITY) ? 0.f : __expf(mold - mnew);
                alpha[warp] = al;
                lrow[warp] = lrow[warp] * al + ps;
                mrow[warp] = mnew;
            }
        }
        unpack_tile<D>(vp, sv, h, RV, vs, vnr, t0, s1, yv, lvV);   // syncs inside
#pragma unroll
        for (int k = 0; k < kOwn; ++k) {
            const int e = threadIdx.x + k * kThreads;
            const int j = e / D, c = e % D;
            if (j < G) {
                float a = acc[k] * alpha[j];
                for (int t = 0; t < kTile; ++t) a = fmaf(S[j * kTile + t], yv[t * LD + c], a);
                acc[k] = a;
            }
        }
        __syncthreads();
    }
    float* out = part + ((int64_t(b) * Hq + h * G) * nsplit + split) * (D + 2);
#pragma unroll
    for (int k = 0; k < kOwn; ++k) {
        const int e = threadIdx.x + k * kThreads;
        const int j = e / D, c = e % D;
        if (j < G) out[int64_t(j) * nsplit * (D + 2) + 2 + c] = acc[k];
    }
    if (threadIdx.x < G) {
        out[int64_t(threadIdx.x) * nsplit * (D + 2) + 0] = mrow[threadIdx.x];
        out[int64_t(threadIdx.x) * nsplit * (D + 2) + 1] = lrow[threadIdx.x];
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

template <int D>
size_t split_smem()
{
    return sizeof(float) * (kMaxGroup * D + 2 * kTile * (D + 1) + kMaxGroup * kTile + 3 * kMaxGroup +
                            2 * kMaxBits * kLmStride + 2 * D) +
           sizeof(int) * 4 * D + sizeof(uint32_t) * 2 * 2 * 8 * D;
}

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
    if (fam != SPECTRA_KERNELS_CUDA_CORE && !qjl) {
        bool done = false;
        spectra_status st = launch_attn_tc(kplan, vplan, q, q_dt, B, Hq, kc, vc, sstride, ctx, scale, part, nsplit,
                                           split_len, extra, s, &done);
        if (st) return st;
        if (done) return launch_combine(vp, part, B, Hq, nsplit, 1, wpart, out, s);
        if (fam == SPECTRA_KERNELS_TENSOR_CORE) return SPECTRA_ERR_UNSUPPORTED;
    }
    if (qjl && fam == SPECTRA_KERNELS_TENSOR_CORE) return SPECTRA_ERR_UNSUPPORTED;
    attn_qrot_kernel<<<B * Hq, D, D * sizeof(float), s>>>(kp, q, q_dt, Hq, Hkv, scale, qt, qj);
    dim3 grid(nsplit, Hkv, B);
    if (D == 128) {
        const size_t sm = split_smem<128>();
        if (spectra_status st = set_smem(attn_split_kernel<128>, sm)) return st;
        attn_split_kernel<128><<<grid, kThreads, sm, s>>>(kp, vp, qt, Hq, ctx, kc, vc, sstride, kn, vn,
                                                          nstride, nsplit, split_len, part, qj);
    } else {
        const size_t sm = split_smem<64>();
        if (spectra_status st = set_smem(attn_split_kernel<64>, sm)) return st;
        attn_split_kernel<64><<<grid, kThreads, sm, s>>>(kp, vp, qt, Hq, ctx, kc, vc, sstride, kn, vn,
                                                         nstride, nsplit, split_len, part, qj);
    }
    if (spectra_status st = cuda_status(cudaGetLastError())) return st;
    return launch_combine(vp, part, B, Hq, nsplit, 0, wpart, out, s);
}

}  // namespace spectra
