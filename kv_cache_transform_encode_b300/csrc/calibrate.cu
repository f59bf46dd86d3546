// calibrate.cu -- per-head Gram matrix and its eigenbasis.
//
// "Sintesi Tecnica: SPECTRA", "Metodologia" items 1 and 3: the transform is
// weighted by the activation second moment G = E[h^T h] and the cache is
// rotated into a basis computed from its own statistics, where channels are
// uncorrelated and energy-ordered.  "Technisch Overzicht ...",
// "Experimentele Opstelling": a per-head eigenbasis calibrated on
// representative tokens.
//
// gram_partial_kernel: grid (chunks, heads); each block accumulates the Gram
//   matrix of one contiguous token chunk in fp32 registers (8x8 or 4x4 tile
//   per thread) and writes it to the workspace.  Deterministic: the Jacobi
//   kernel sums the chunk partials in a fixed order.
// jacobi_kernel: one block per head.  The matrix and the rotation
//   accumulator live in shared memory (rows padded to d+1 floats so column
//   accesses are bank-conflict free).  Each round applies d/2 disjoint
//   rotations chosen by the round-robin ("circle") tournament, so a sweep of
//   d-1 rounds visits every pair once; the two-sided update J^T A J is done
//   one 2x2 block at a time in registers (one pass over A per round), the
//   accumulator V J in the same phase.
#include "spectra_internal.cuh"

#include <cooperative_groups.h>
#include <math.h>

#include <algorithm>

namespace spectra {

namespace {

constexpr int kGramThreads = 256;
constexpr int kGramTile = 32;   // tokens staged per iteration

template <int D>
__global__ void __launch_bounds__(kGramThreads)
gram_partial_kernel(const void* __restrict__ x, int dt, int64_t n_cal, int64_t token_stride,
                    int heads, int64_t chunk_len, float* __restrict__ partials)
{
    constexpr int RB = D / 16;      // rows/cols per thread
    __shared__ float xs[kGramTile][D];
    const int chunk = blockIdx.x, h = blockIdx.y;
    const int64_t t_begin = int64_t(chunk) * chunk_len;
    const int64_t t_end = min(n_cal, t_begin + chunk_len);
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;

    float acc[RB][RB];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int c = 0; c < RB; ++c) acc[r][c] = 0.f;

    for (int64_t t0 = t_begin; t0 < t_end; t0 += kGramTile) {
        const int nt = int(min(int64_t(kGramTile), t_end - t0));
        for (int e = threadIdx.x; e < kGramTile * D; e += kGramThreads) {
            const int tt = e / D, i = e % D;
            xs[tt][i] = (tt < nt) ? load_elem(x, dt, (t0 + tt) * token_stride + int64_t(h) * D + i) : 0.f;
        }
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
            float a[RB], b[RB];
#pragma unroll
            for (int r = 0; r < RB; ++r) a[r] = xs[tt][ty * RB + r];
#pragma unroll
            for (int c = 0; c < RB; ++c) b[c] = xs[tt][tx * RB + c];
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int c = 0; c < RB; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
        }
        __syncthreads();
    }
    float* out = partials + (size_t(h) * gridDim.x + chunk) * D * D;
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int c = 0; c < RB; ++c) out[(ty * RB + r) * D + tx * RB + c] = acc[r][c];
}

constexpr int kJacobiThreads = 1024;

__device__ __forceinline__ float block_sum(float v, float* red)
{
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x < 32) {
        s = (l < int(blockDim.x >> 5)) ? red[l] : 0.f;
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (l == 0) red[32] = s;
    }
    __syncthreads();
    return red[32];
}

// Round-robin tournament: in round r, pair k of n players.
__device__ __forceinline__ void rr_pair(int n, int r, int k, int& p, int& q)
{
    auto idx = [&](int j) { return 1 + (j + r) % (n - 1); };
    if (k == 0) { p = 0; q = idx(0); }
    else { p = idx(k); q = idx(n - 1 - k); }
}

template <int D>
__global__ void __launch_bounds__(kJacobiThreads)
jacobi_kernel(const float* __restrict__ partials, int nchunks, float inv_n, int max_sweeps,
              float* __restrict__ basis_out, float* __restrict__ eig_out,
              int32_t* __restrict__ status, float* __restrict__ gram_out)
{
    constexpr int LD = D + 1;
    constexpr int NP = D / 2;
    extern __shared__ float smem[];
    float* A = smem;                 // [D][LD]
    float* V = A + D * LD;           // [D][LD]
    float* sn = V + D * LD;          // [NP] sin
    float* ta = sn + NP;             // [NP] tau = s / (1 + c)
    float* tt = ta + NP;             // [NP] tan
    int* pp = reinterpret_cast<int*>(tt + NP);   // [NP]
    int* qq = pp + NP;                           // [NP]
    float* red = reinterpret_cast<float*>(qq + NP);   // [33]
    int* flag = reinterpret_cast<int*>(red + 33);

    const int h = blockIdx.x;
    const int tid = threadIdx.x;
    if (tid == 0) flag[0] = 0;
    __syncthreads();

    // 1. G = (1/n) sum of chunk partials, fixed order; identity accumulator.
    for (int e = tid; e < D * D; e += blockDim.x) {
        const int i = e / D, j = e % D;
        const float* src = partials + size_t(h) * nchunks * D * D + e;
        float s = 0.f;
        for (int c = 0; c < nchunks; ++c) s += src[size_t(c) * D * D];
        s *= inv_n;
        A[i * LD + j] = s;
        V[i * LD + j] = (i == j) ? 1.f : 0.f;
        if (gram_out) gram_out[size_t(h) * D * D + e] = s;
        if (!isfinite(s)) flag[0] = 1;
    }
    __syncthreads();
    if (flag[0]) {
        for (int e = tid; e < D * D; e += blockDim.x)
            basis_out[size_t(h) * D * D + e] = ((e / D) == (e % D)) ? 1.f : 0.f;
        if (tid < D) eig_out[size_t(h) * D + tid] = 0.f;
        if (tid == 0) status[h] = -SPECTRA_ERR_NONFINITE;
        return;
    }

    // 2. Frobenius norm of G and the sweep loop.
    float loc = 0.f;
    for (int e = tid; e < D * D; e += blockDim.x) {
        const float a = A[(e / D) * LD + (e % D)];
        loc = fmaf(a, a, loc);
    }
    const float fro = sqrtf(block_sum(loc, red));

    int sweeps = 0, converged = 0;
    float prev_off = INFINITY;
    for (;;) {
        loc = 0.f;
        for (int e = tid; e < D * D; e += blockDim.x) {
            const int i = e / D, j = e % D;
            if (i != j) { const float a = A[i * LD + j]; loc = fmaf(a, a, loc); }
        }
        const float off = sqrtf(block_sum(loc, red));
        // converged: below 1e-6 of ||G||, or stalled at the fp32 round-off
        // floor (a full sweep no longer halves it, already below 1e-4 ||G||)
        if (off <= 1e-6f * fro || fro == 0.f || (off > 0.5f * prev_off && off <= 1e-4f * fro)) {
            converged = 1;
            break;
        }
        if (sweeps >= max_sweeps) break;
        prev_off = off;
        ++sweeps;
        for (int r = 0; r < D - 1; ++r) {
            // rotation k annihilates A[p][q] (p = top, q = bottom of pair k).
            // Rutishauser's form: with tau = s / (1 + c), c*x - s*y is
            // evaluated as x - s (y + tau x), which keeps every rotation
            // orthogonal to working precision even when c rounds to 1.
            if (tid < NP) {
                int p, q;
                rr_pair(D, r, tid, p, q);
                const float apq = A[p * LD + q];
                const float app = A[p * LD + p], aqq = A[q * LD + q];
                float t = 0.f, s = 0.f, tau = 0.f;
                if (fabsf(apq) > 1e-30f && fabsf(apq) > 1e-10f * sqrtf(fabsf(app * aqq))) {
                    const float theta = (aqq - app) / (2.f * apq);
                    const float at = fabsf(theta);
                    t = (at > 1e18f) ? 0.5f / at : 1.f / (at + sqrtf(fmaf(at, at, 1.f)));
                    t = (theta >= 0.f) ? t : -t;
                    const float c = 1.f / sqrtf(fmaf(t, t, 1.f));
                    s = t * c;
                    tau = s / (1.f + c);
                }
                sn[tid] = s; ta[tid] = tau; tt[tid] = t; pp[tid] = p; qq[tid] = q;
            }
            __syncthreads();
            // A <- J^T A J, one 2x2 block (pair k rows, pair l cols) at a time
            for (int e = tid; e < NP * NP; e += blockDim.x) {
                const int k = e / NP, l = e % NP;
                const int p = pp[k], q = qq[k], u = pp[l], w = qq[l];
                float a = A[p * LD + u], b = A[p * LD + w], c = A[q * LD + u], d = A[q * LD + w];
                if (k == l) {
                    const float tk = tt[k];
                    a = a - tk * b;          // a_pp - t a_pq
                    d = d + tk * b;          // a_qq + t a_pq
                    b = 0.f;
                    c = 0.f;
                } else {
                    const float sl = sn[l], tl = ta[l], sk = sn[k], tk = ta[k];
                    // columns (u, w) by rotation l
                    float a1 = a - sl * (b + tl * a), b1 = b + sl * (a - tl * b);
                    float c1 = c - sl * (d + tl * c), d1 = d + sl * (c - tl * d);
                    // rows (p, q) by rotation k
                    a = a1 - sk * (c1 + tk * a1);
                    c = c1 + sk * (a1 - tk * c1);
                    b = b1 - sk * (d1 + tk * b1);
                    d = d1 + sk * (b1 - tk * d1);
                }
                A[p * LD + u] = a; A[p * LD + w] = b; A[q * LD + u] = c; A[q * LD + w] = d;
            }
            // V <- V J
            for (int e = tid; e < NP * D; e += blockDim.x) {
                const int k = e / D, i = e % D;
                const int p = pp[k], q = qq[k];
                const float s = sn[k], tau = ta[k];
                const float vp = V[i * LD + p], vq = V[i * LD + q];
                V[i * LD + p] = vp - s * (vq + tau * vp);
                V[i * LD + q] = vq + s * (vp - tau * vq);
            }
            __syncthreads();
        }
    }

    // 3. Sort descending (ties: lower index first), sign-fix, write out.
    int* rank = reinterpret_cast<int*>(sn);   // reuse: needs D ints (sn..ta span 2 NP floats)
    if (tid < D) {
        const float li = A[tid * LD + tid];
        int rk = 0;
        for (int j = 0; j < D; ++j) {
            const float lj = A[j * LD + j];
            rk += (lj > li) || (lj == li && j < tid);
        }
        rank[tid] = rk;
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
    for (int i = warp; i < D; i += nwarps) {
        // largest |V[r][i]|, lowest r on ties
        float best = -1.f;
        int br = 0;
        for (int r = lane; r < D; r += 32) {
            const float a = fabsf(V[r * LD + i]);
            if (a > best) { best = a; br = r; }
        }
        for (int o = 16; o; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int orr = __shfl_xor_sync(0xffffffffu, br, o);
            if (ob > best || (ob == best && orr < br)) { best = ob; br = orr; }
        }
        const float sgn = (V[br * LD + i] < 0.f) ? -1.f : 1.f;
        const int c = rank[i];
        for (int r = lane; r < D; r += 32)
            basis_out[size_t(h) * D * D + size_t(r) * D + c] = sgn * V[r * LD + i];
        if (lane == 0) eig_out[size_t(h) * D + c] = A[i * LD + i];
    }
    if (tid == 0) status[h] = converged ? sweeps : -SPECTRA_ERR_NOT_CONVERGED;
}

// ---------------------------------------------------------------------------
// jacobi128_kernel: cyclic Jacobi for head_dim 128 with the odd-even
// ("caterpillar") ordering, register-blocked.  Round r pairs adjacent
// positions: (2k, 2k+1) when r is even, (2k+1, 2k+2) when r is odd.  Every
// pair's transform is the Jacobi rotation that annihilates A[p][q] followed
// by a swap of the two positions, so after 128 rounds (one sweep) every pair
// of eigen-indices has met exactly once -- the odd-even transposition
// network run with every comparator exchanging.  Because pairs are always
// adjacent, the 128x128 matrix A and the accumulator V stay in registers:
// thread (warp w, lane l) owns the 4x4 blocks A[4w..4w+3][4l..4l+3] and
// V[4w..][4l..].  Column rotations that straddle two blocks take the
// neighbour lane's column by shuffle; row rotations that straddle two warps
// take the neighbour block row from shared memory.  The 64 rotations of a
// round come from the diagonal band (A[i][i], A[i][i+1]), which the owners
// of the diagonal and super-diagonal blocks publish after each round; two
// warps turn the band into rotations while the other thirty apply the
// previous round's rotations to V (V trails A by one round).
// Rutishauser's form (c x - s y evaluated as x - s (y + tau x), tau =
// s / (1 + c)) keeps the transforms orthogonal to working precision.
constexpr int kJ2 = 128;
constexpr int kJacCluster = 4;   // CTAs per head in the cluster Jacobi (4 measured fastest: 2 and 8 are slower)

struct Rot { float s, tau, t; };

__device__ __forceinline__ Rot load_rot(const float4* prm, int k)
{
    const float4 v = prm[k];
    Rot r;
    r.s = v.x;
    r.tau = v.y;
    r.t = v.z;
    return r;
}

// (x, y) <- (s x + c y, c x - s y): rotation then swap, in Rutishauser form
__device__ __forceinline__ void rotswap(float& x, float& y, float s, float tau)
{
    const float xn = fmaf(s, fmaf(-tau, y, x), y);
    const float yn = fmaf(-s, fmaf(tau, x, y), x);
    x = xn;
    y = yn;
}

// the same on two rows at once (packed fp32x2 FMAs)
__device__ __forceinline__ void rotswap2(float2& x, float2& y, float s, float tau)
{
    const float2 S = make_float2(s, s), NS = make_float2(-s, -s);
    const float2 T = make_float2(tau, tau), NT = make_float2(-tau, -tau);
    const float2 u = __ffma2_rn(NT, y, x);
    const float2 v = __ffma2_rn(T, x, y);
    const float2 xn = __ffma2_rn(S, u, y);
    const float2 yn = __ffma2_rn(NS, v, x);
    x = xn;
    y = yn;
}

// Rotation of pair (p, q) from the band: fast-math reciprocal and square
// roots (the rotation only has to be orthogonal, which c = rsqrt(1 + t^2),
// s = t c guarantees to a few ulp whatever small error t carries).
__device__ __forceinline__ float4 band_rotation(float app, float aqq, float apq)
{
    float s = 0.f, tau = 0.f, t = 0.f;
    if (fabsf(apq) > 1e-30f && apq * apq > 1e-20f * fabsf(app * aqq)) {
        const float theta = __fdividef(aqq - app, 2.f * apq);
        const float at = fabsf(theta);
        if (at > 1e18f) {
            t = __fdividef(0.5f, at);
        } else {
            const float q1 = fmaf(at, at, 1.f);
            t = __fdividef(1.f, fmaf(q1, rsqrtf(q1), at));     // 1 / (|theta| + sqrt(theta^2 + 1))
        }
        t = (theta >= 0.f) ? t : -t;
        const float c = rsqrtf(fmaf(t, t, 1.f));
        s = t * c;
        tau = __fdividef(s, 1.f + c);
    }
    return make_float4(s, tau, t, 0.f);
}

// V <- V Q for round parity `par` (columns only; V rows are independent).
__device__ __forceinline__ void v_update(float2 (&v)[2][4], const float4* pr, bool E, int l)
{
    if (E) {
        const Rot c0 = load_rot(pr, 2 * l), c1 = load_rot(pr, 2 * l + 1);
#pragma unroll
        for (int ip = 0; ip < 2; ++ip) {
            rotswap2(v[ip][0], v[ip][1], c0.s, c0.tau);
            rotswap2(v[ip][2], v[ip][3], c1.s, c1.tau);
        }
    } else {
        const bool lf = l > 0, rt = l < 31;
        const Rot cm = load_rot(pr, lf ? 2 * l - 1 : 0), c0 = load_rot(pr, 2 * l), c1 = load_rot(pr, 2 * l + 1);
#pragma unroll
        for (int ip = 0; ip < 2; ++ip) {
            float2 vr, vl;
            vr.x = __shfl_down_sync(0xffffffffu, v[ip][0].x, 1);
            vr.y = __shfl_down_sync(0xffffffffu, v[ip][0].y, 1);
            vl.x = __shfl_up_sync(0xffffffffu, v[ip][3].x, 1);
            vl.y = __shfl_up_sync(0xffffffffu, v[ip][3].y, 1);
            if (rt) {
                float2 x = v[ip][3], y = vr;
                rotswap2(x, y, c1.s, c1.tau);
                v[ip][3] = x;
            }
            if (lf) {
                float2 x = vl, y = v[ip][0];
                rotswap2(x, y, cm.s, cm.tau);
                v[ip][0] = y;
            }
            rotswap2(v[ip][1], v[ip][2], c0.s, c0.tau);
        }
    }
}

__global__ void __launch_bounds__(1024, 1)
jacobi128_kernel(const float* __restrict__ partials, int nchunks, float inv_n, int max_sweeps,
                 float* __restrict__ basis_out, float* __restrict__ eig_out, int32_t* __restrict__ status,
                 float* __restrict__ gram_out)
{
    constexpr int D = kJ2;
    extern __shared__ float smem[];
    float* rowx = smem;                                   // [32][2][D] exchanged block rows
    float* band = rowx + 32 * 2 * D;                      // [2 parity][2][D]: diag, super-diag
    float4* prm = reinterpret_cast<float4*>(band + 4 * D);  // [2 parity][64]
    float* red = reinterpret_cast<float*>(prm + 128);     // [33]

    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31, h = blockIdx.x;
    // a[ip][j] = (A[4w + 2ip][4l + j], A[4w + 2ip + 1][4l + j]); v likewise
    float2 a[2][4], v[2][4];
#define AE(i, j) ((i) & 1 ? a[(i) >> 1][j].y : a[(i) >> 1][j].x)

    // 1. G = (1/n) sum of the chunk partials (fixed order), V = I.
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = 4 * w + i, c = 4 * l + j;
            const float* src = partials + size_t(h) * nchunks * D * D + size_t(r) * D + c;
            float sum = 0.f;
            for (int ch = 0; ch < nchunks; ++ch) sum += src[size_t(ch) * D * D];
            sum *= inv_n;
            AE(i, j) = sum;
            ((i & 1) ? v[i >> 1][j].y : v[i >> 1][j].x) = (r == c) ? 1.f : 0.f;
            if (gram_out) gram_out[size_t(h) * D * D + size_t(r) * D + c] = sum;
            bad |= !isfinite(sum);
        }
    if (__syncthreads_or(bad)) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                basis_out[size_t(h) * D * D + size_t(4 * w + i) * D + 4 * l + j] = (4 * w + i == 4 * l + j) ? 1.f : 0.f;
        if (tid < D) eig_out[size_t(h) * D + tid] = 0.f;
        if (tid == 0) status[h] = -SPECTRA_ERR_NONFINITE;
        return;
    }
    auto publish_band = [&](int par) {
        float* dg = band + par * 2 * D;
        float* sp = dg + D;
        if (w == l) {
            dg[4 * w + 0] = a[0][0].x; dg[4 * w + 1] = a[0][1].y;
            dg[4 * w + 2] = a[1][2].x; dg[4 * w + 3] = a[1][3].y;
            sp[4 * w + 0] = a[0][1].x; sp[4 * w + 1] = a[0][2].y; sp[4 * w + 2] = a[1][3].x;
        }
        if (l == w + 1) sp[4 * w + 3] = a[1][0].y;
    };
    publish_band(0);

    float loc = 0.f;
#pragma unroll
    for (int ip = 0; ip < 2; ++ip)
#pragma unroll
        for (int j = 0; j < 4; ++j) loc += a[ip][j].x * a[ip][j].x + a[ip][j].y * a[ip][j].y;
    const float fro = sqrtf(block_sum(loc, red));

    int sweeps = 0, converged = 0, rounds = 0;
    float prev_off = INFINITY;
    for (;;) {
        loc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (4 * w + i != 4 * l + j) loc = fmaf(AE(i, j), AE(i, j), loc);
        const float off = sqrtf(block_sum(loc, red));
        if (off <= 1e-6f * fro || fro == 0.f || (off > 0.5f * prev_off && off <= 1e-4f * fro)) {
            converged = 1;
            break;
        }
        if (sweeps >= max_sweeps) break;
        prev_off = off;
        ++sweeps;
        for (int r = 0; r < D; ++r, ++rounds) {
            const int par = r & 1;
            const bool E = par == 0;   // pairs (2k, 2k+1)
            __syncthreads();           // band[par] published
            if (w < 2) {
                const int k = tid, p = E ? 2 * k : 2 * k + 1, q = p + 1;
                float4 rt = make_float4(0.f, 0.f, 0.f, 0.f);
                if (q < D) {
                    const float* dg = band + par * 2 * D;
                    rt = band_rotation(dg[p], dg[q], dg[D + p]);
                }
                prm[par * 64 + k] = rt;
            } else if (rounds > 0) {
                v_update(v, prm + (par ^ 1) * 64, !E, l);   // previous round's rotations
            }
            __syncthreads();
            if (w < 2 && rounds > 0) v_update(v, prm + (par ^ 1) * 64, !E, l);
            const float4* pr = prm + par * 64;
            if (E) {
                const Rot r0 = load_rot(pr, 2 * w), r1 = load_rot(pr, 2 * w + 1);     // rows
                const Rot c0 = load_rot(pr, 2 * l), c1 = load_rot(pr, 2 * l + 1);     // columns
                float d00 = 0.f, d11 = 0.f, d01 = 0.f, d22 = 0.f, d33 = 0.f, d23 = 0.f;
                if (w == l) {
                    d00 = a[0][0].x; d11 = a[0][1].y; d01 = a[0][1].x;
                    d22 = a[1][2].x; d33 = a[1][3].y; d23 = a[1][3].x;
                }
#pragma unroll
                for (int ip = 0; ip < 2; ++ip) {
                    rotswap2(a[ip][0], a[ip][1], c0.s, c0.tau);
                    rotswap2(a[ip][2], a[ip][3], c1.s, c1.tau);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    rotswap(a[0][j].x, a[0][j].y, r0.s, r0.tau);
                    rotswap(a[1][j].x, a[1][j].y, r1.s, r1.tau);
                }
                if (w == l) {   // diagonal sub-blocks: exact values
                    a[0][0].x = fmaf(r0.t, d01, d11); a[0][1].y = fmaf(-r0.t, d01, d00);
                    a[0][1].x = 0.f; a[0][0].y = 0.f;
                    a[1][2].x = fmaf(r1.t, d23, d33); a[1][3].y = fmaf(-r1.t, d23, d22);
                    a[1][3].x = 0.f; a[1][2].y = 0.f;
                }
            } else {
                const bool up = w > 0, dn = w < 31, lf = l > 0, rt = l < 31;
                const Rot cm = load_rot(pr, lf ? 2 * l - 1 : 0), c0 = load_rot(pr, 2 * l), c1 = load_rot(pr, 2 * l + 1);
                float d11 = 0.f, d22 = 0.f, d12 = 0.f;
                if (w == l) { d11 = a[0][1].y; d22 = a[1][2].x; d12 = a[0][2].y; }
                // columns: (4l-1, 4l) with the left lane, (4l+1, 4l+2) inside, (4l+3, 4l+4) with the right lane
#pragma unroll
                for (int ip = 0; ip < 2; ++ip) {
                    float2 ar, al;
                    ar.x = __shfl_down_sync(0xffffffffu, a[ip][0].x, 1);
                    ar.y = __shfl_down_sync(0xffffffffu, a[ip][0].y, 1);
                    al.x = __shfl_up_sync(0xffffffffu, a[ip][3].x, 1);
                    al.y = __shfl_up_sync(0xffffffffu, a[ip][3].y, 1);
                    if (rt) {
                        float2 x = a[ip][3], y = ar;
                        rotswap2(x, y, c1.s, c1.tau);
                        a[ip][3] = x;
                    }
                    if (lf) {
                        float2 x = al, y = a[ip][0];
                        rotswap2(x, y, cm.s, cm.tau);
                        a[ip][0] = y;
                    }
                    rotswap2(a[ip][1], a[ip][2], c0.s, c0.tau);
                }
                // rows: (4w-1, 4w) and (4w+3, 4w+4) through shared memory
                float* mine = rowx + w * 2 * D + 4 * l;
                *reinterpret_cast<float4*>(mine) = make_float4(a[0][0].x, a[0][1].x, a[0][2].x, a[0][3].x);
                *reinterpret_cast<float4*>(mine + D) = make_float4(a[1][0].y, a[1][1].y, a[1][2].y, a[1][3].y);
                __syncthreads();
                const Rot rm = load_rot(pr, up ? 2 * w - 1 : 0), r0 = load_rot(pr, 2 * w), r1 = load_rot(pr, 2 * w + 1);
                if (dn) {
                    const float4 b4 = *reinterpret_cast<const float4*>(rowx + (w + 1) * 2 * D + 4 * l);
                    const float bl[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) a[1][j].y = fmaf(r1.s, fmaf(-r1.tau, bl[j], a[1][j].y), bl[j]);
                }
                if (up) {
                    const float4 a4 = *reinterpret_cast<const float4*>(rowx + (w - 1) * 2 * D + D + 4 * l);
                    const float ab[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) a[0][j].x = fmaf(-rm.s, fmaf(rm.tau, ab[j], a[0][j].x), ab[j]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) rotswap(a[0][j].y, a[1][j].x, r0.s, r0.tau);
                if (w == l) {
                    a[0][1].y = fmaf(r0.t, d12, d22); a[1][2].x = fmaf(-r0.t, d12, d11);
                    a[0][2].y = 0.f; a[1][1].x = 0.f;
                }
            }
            publish_band(par ^ 1);
        }
    }
    if (rounds > 0) {   // V trails A by one round: apply the last one
        __syncthreads();
        v_update(v, prm + ((rounds - 1) & 1) * 64, ((rounds - 1) & 1) == 0, l);
    }

    // 2. Sort descending (ties: lower position first), sign-fix, write out.
    __syncthreads();
    constexpr int LD = D + 1;
    float* Vs = smem;                 // [D][LD]
    float* lam = Vs + D * LD;         // [D]
    int* rank = reinterpret_cast<int*>(lam + D);
#pragma unroll
    for (int ip = 0; ip < 2; ++ip)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            Vs[(4 * w + 2 * ip) * LD + 4 * l + j] = v[ip][j].x;
            Vs[(4 * w + 2 * ip + 1) * LD + 4 * l + j] = v[ip][j].y;
        }
    if (w == l) {
        lam[4 * w + 0] = a[0][0].x; lam[4 * w + 1] = a[0][1].y;
        lam[4 * w + 2] = a[1][2].x; lam[4 * w + 3] = a[1][3].y;
    }
#undef AE
    __syncthreads();
    if (tid < D) {
        const float li = lam[tid];
        int rk = 0;
        for (int j = 0; j < D; ++j) {
            const float lj = lam[j];
            rk += (lj > li) || (lj == li && j < tid);
        }
        rank[tid] = rk;
    }
    __syncthreads();
    for (int i = w; i < D; i += 32) {
        float best = -1.f;
        int br = 0;
        for (int rr = l; rr < D; rr += 32) {
            const float av = fabsf(Vs[rr * LD + i]);
            if (av > best) { best = av; br = rr; }
        }
        for (int o = 16; o; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int orr = __shfl_xor_sync(0xffffffffu, br, o);
            if (ob > best || (ob == best && orr < br)) { best = ob; br = orr; }
        }
        const float sgn = (Vs[br * LD + i] < 0.f) ? -1.f : 1.f;
        const int c = rank[i];
        for (int rr = l; rr < D; rr += 32) basis_out[size_t(h) * D * D + size_t(rr) * D + c] = sgn * Vs[rr * LD + i];
        if (l == 0) eig_out[size_t(h) * D + c] = lam[i];
    }
    if (tid == 0) status[h] = converged ? sweeps : -SPECTRA_ERR_NOT_CONVERGED;
}

size_t jacobi128_smem()
{
    const size_t work = sizeof(float) * (32 * 2 * kJ2 + 4 * kJ2) + sizeof(float4) * 128 + sizeof(float) * 33;
    const size_t fin = sizeof(float) * (kJ2 * (kJ2 + 1) + kJ2) + sizeof(int) * kJ2;
    return (work > fin ? work : fin) + 16;
}

// ---------------------------------------------------------------------------
// jacobi128c_kernel<C>: the same odd-even Jacobi spread over a cluster of C
// CTAs per head (distributed shared memory).  CTA r owns block rows
// [NW r, NW r + NW) (NW = 32 / C warps, 4 rows each) of A and V; thread
// (warp, lane) still owns one 4x4 block of each.  Once per round, after a
// cluster barrier, every CTA holds the whole diagonal band (each CTA writes
// its band entries into all CTAs' shared memory) and computes the round's 64
// rotations itself; the block rows that straddle two CTAs in odd rounds are
// sent ahead (as they stand after the previous round) and each receiver
// applies the column rotations to its copy.  Every CTA runs the same rounds
// and takes the same convergence decision (cluster-reduced in a fixed
// order), so every barrier is met by all CTAs.
template <int C>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(1024 / C, 1)
jacobi128c_kernel(const float* partials, int nchunks, float inv_n, int max_sweeps,
                  float* __restrict__ basis_out, float* __restrict__ eig_out, int32_t* __restrict__ status,
                  float* __restrict__ gram_out, float* scratch)
{
    namespace cg = cooperative_groups;
    constexpr int D = kJ2;
    constexpr int NW = 32 / C;                // warps per CTA
    constexpr int NT = 32 * NW;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int hd = blockIdx.x / C;

    extern __shared__ float smem[];
    float* rowx = smem;                                    // [NW][2][D]
    float* band = rowx + NW * 2 * D;                       // [2][2][D]
    float* nbr = band + 4 * D;                             // [2 parity][2: up, down][D]
    float4* prm = reinterpret_cast<float4*>(nbr + 4 * D);  // [2][64]
    float* red = reinterpret_cast<float*>(prm + 128);      // [33]
    float* csum = red + 33;                                // [2][C] cluster partial sums
    float* lamall = csum + 2 * C;                          // [D]
    int* cflag = reinterpret_cast<int*>(lamall + D);       // [C]

    const int tid = threadIdx.x, wl = tid >> 5, l = tid & 31;
    const int w = rank * NW + wl;                          // global block row
    cluster.sync();    // every CTA of the cluster runs before any shared memory is touched remotely
    float2 a[2][4], v[2][4];
#define AE(i, j) ((i) & 1 ? a[(i) >> 1][j].y : a[(i) >> 1][j].x)

    // cluster-wide sum of one float per CTA, identical in every CTA
    int cuse = 0;
    auto cluster_sum = [&](float part) -> float {
        const float tot = block_sum(part, red);
        if (tid < C) *cluster.map_shared_rank(csum + (cuse & 1) * C + rank, tid) = tot;
        cluster.sync();
        float s = 0.f;
        for (int k = 0; k < C; ++k) s += csum[(cuse & 1) * C + k];
        ++cuse;
        return s;
    };

    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = 4 * w + i, c = 4 * l + j;
            const float* src = partials + size_t(hd) * nchunks * D * D + size_t(r) * D + c;
            float sum = 0.f;
            for (int ch = 0; ch < nchunks; ++ch) sum += src[size_t(ch) * D * D];
            sum *= inv_n;
            AE(i, j) = sum;
            ((i & 1) ? v[i >> 1][j].y : v[i >> 1][j].x) = (r == c) ? 1.f : 0.f;
            if (gram_out) gram_out[size_t(hd) * D * D + size_t(r) * D + c] = sum;
            bad |= !isfinite(sum);
        }
    {
        const int bl = __syncthreads_or(bad);
        if (tid < C) *cluster.map_shared_rank(cflag + rank, tid) = bl;
        cluster.sync();
        int any = 0;
        for (int k = 0; k < C; ++k) any |= cflag[k];
        if (any) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    basis_out[size_t(hd) * D * D + size_t(4 * w + i) * D + 4 * l + j] = (4 * w + i == 4 * l + j) ? 1.f : 0.f;
            if (rank == 0 && tid < D) eig_out[size_t(hd) * D + tid] = 0.f;
            if (rank == 0 && tid == 0) status[hd] = -SPECTRA_ERR_NONFINITE;
            return;
        }
    }
    // publish this CTA's band entries (all CTAs) and, before odd rounds, the
    // block rows the neighbour CTAs need
    auto publish = [&](int par, bool rows) {
        if (w == l) {
            const float dv[4] = {a[0][0].x, a[0][1].y, a[1][2].x, a[1][3].y};
            const float sv[3] = {a[0][1].x, a[0][2].y, a[1][3].x};
            for (int k = 0; k < C; ++k) {
                float* dg = cluster.map_shared_rank(band + par * 2 * D, k);
#pragma unroll
                for (int i = 0; i < 4; ++i) dg[4 * w + i] = dv[i];
#pragma unroll
                for (int i = 0; i < 3; ++i) dg[D + 4 * w + i] = sv[i];
            }
        }
        if (l == w + 1) {
            for (int k = 0; k < C; ++k) cluster.map_shared_rank(band + par * 2 * D, k)[D + 4 * w + 3] = a[1][0].y;
        }
        if (rows) {
            if (wl == 0 && rank > 0) {          // my row 0 -> rank-1's "down" row
                float* dst = cluster.map_shared_rank(nbr + (par * 2 + 1) * D, rank - 1) + 4 * l;
                *reinterpret_cast<float4*>(dst) = make_float4(a[0][0].x, a[0][1].x, a[0][2].x, a[0][3].x);
            }
            if (wl == NW - 1 && rank < C - 1) { // my row 3 -> rank+1's "up" row
                float* dst = cluster.map_shared_rank(nbr + (par * 2 + 0) * D, rank + 1) + 4 * l;
                *reinterpret_cast<float4*>(dst) = make_float4(a[1][0].y, a[1][1].y, a[1][2].y, a[1][3].y);
            }
        }
    };
    publish(0, false);

    float loc = 0.f;
#pragma unroll
    for (int ip = 0; ip < 2; ++ip)
#pragma unroll
        for (int j = 0; j < 4; ++j) loc += a[ip][j].x * a[ip][j].x + a[ip][j].y * a[ip][j].y;
    const float fro = sqrtf(cluster_sum(loc));

    // column rotations of one 4-wide row segment (odd round): (4l-1, 4l) with
    // the left lane, (4l+1, 4l+2) inside, (4l+3, 4l+4) with the right lane
    auto col_odd = [&](float (&x)[4], const Rot& cm, const Rot& c0, const Rot& c1) {
        const float xr = __shfl_down_sync(0xffffffffu, x[0], 1);
        const float xl = __shfl_up_sync(0xffffffffu, x[3], 1);
        if (l < 31) x[3] = fmaf(c1.s, fmaf(-c1.tau, xr, x[3]), xr);
        if (l > 0) x[0] = fmaf(-cm.s, fmaf(cm.tau, xl, x[0]), xl);
        rotswap(x[1], x[2], c0.s, c0.tau);
    };

    int sweeps = 0, converged = 0, rounds = 0;
    float prev_off = INFINITY;
    for (;;) {
        loc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (4 * w + i != 4 * l + j) loc = fmaf(AE(i, j), AE(i, j), loc);
        const float off = sqrtf(cluster_sum(loc));
        if (off <= 1e-6f * fro || fro == 0.f || (off > 0.5f * prev_off && off <= 1e-4f * fro)) {
            converged = 1;
            break;
        }
        if (sweeps >= max_sweeps) break;
        prev_off = off;
        ++sweeps;
        for (int r = 0; r < D; ++r, ++rounds) {
            const int par = r & 1;
            const bool E = par == 0;
            cluster.sync();                        // band[par] (and rows) from every CTA visible
            if (wl < 2) {
                const int k = tid, p = E ? 2 * k : 2 * k + 1, q = p + 1;
                float4 rt = make_float4(0.f, 0.f, 0.f, 0.f);
                if (q < D) {
                    const float* dg = band + par * 2 * D;
                    rt = band_rotation(dg[p], dg[q], dg[D + p]);
                }
                prm[par * 64 + k] = rt;
            } else if (rounds > 0) {
                v_update(v, prm + (par ^ 1) * 64, !E, l);
            }
            __syncthreads();
            if (wl < 2 && rounds > 0) v_update(v, prm + (par ^ 1) * 64, !E, l);
            const float4* pr = prm + par * 64;
            if (E) {
                const Rot r0 = load_rot(pr, 2 * w), r1 = load_rot(pr, 2 * w + 1);
                const Rot c0 = load_rot(pr, 2 * l), c1 = load_rot(pr, 2 * l + 1);
                float d00 = 0.f, d11 = 0.f, d01 = 0.f, d22 = 0.f, d33 = 0.f, d23 = 0.f;
                if (w == l) {
                    d00 = a[0][0].x; d11 = a[0][1].y; d01 = a[0][1].x;
                    d22 = a[1][2].x; d33 = a[1][3].y; d23 = a[1][3].x;
                }
#pragma unroll
                for (int ip = 0; ip < 2; ++ip) {
                    rotswap2(a[ip][0], a[ip][1], c0.s, c0.tau);
                    rotswap2(a[ip][2], a[ip][3], c1.s, c1.tau);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    rotswap(a[0][j].x, a[0][j].y, r0.s, r0.tau);
                    rotswap(a[1][j].x, a[1][j].y, r1.s, r1.tau);
                }
                if (w == l) {
                    a[0][0].x = fmaf(r0.t, d01, d11); a[0][1].y = fmaf(-r0.t, d01, d00);
                    a[0][1].x = 0.f; a[0][0].y = 0.f;
                    a[1][2].x = fmaf(r1.t, d23, d33); a[1][3].y = fmaf(-r1.t, d23, d22);
                    a[1][3].x = 0.f; a[1][2].y = 0.f;
                }
            } else {
                const bool up = w > 0, dn = w < 31, lf = l > 0, rt = l < 31;
                const Rot cm = load_rot(pr, lf ? 2 * l - 1 : 0), c0 = load_rot(pr, 2 * l), c1 = load_rot(pr, 2 * l + 1);
                float d11 = 0.f, d22 = 0.f, d12 = 0.f;
                if (w == l) { d11 = a[0][1].y; d22 = a[1][2].x; d12 = a[0][2].y; }
#pragma unroll
                for (int ip = 0; ip < 2; ++ip) {
                    float2 ar, al;
                    ar.x = __shfl_down_sync(0xffffffffu, a[ip][0].x, 1);
                    ar.y = __shfl_down_sync(0xffffffffu, a[ip][0].y, 1);
                    al.x = __shfl_up_sync(0xffffffffu, a[ip][3].x, 1);
                    al.y = __shfl_up_sync(0xffffffffu, a[ip][3].y, 1);
                    if (rt) {
                        float2 x = a[ip][3], y = ar;
                        rotswap2(x, y, c1.s, c1.tau);
                        a[ip][3] = x;
                    }
                    if (lf) {
                        float2 x = al, y = a[ip][0];
                        rotswap2(x, y, cm.s, cm.tau);
                        a[ip][0] = y;
                    }
                    rotswap2(a[ip][1], a[ip][2], c0.s, c0.tau);
                }
                // rows across warps of this CTA: shared memory; across CTAs:
                // the neighbour's row as it stood, column-rotated here
                float* mine = rowx + wl * 2 * D + 4 * l;
                *reinterpret_cast<float4*>(mine) = make_float4(a[0][0].x, a[0][1].x, a[0][2].x, a[0][3].x);
                *reinterpret_cast<float4*>(mine + D) = make_float4(a[1][0].y, a[1][1].y, a[1][2].y, a[1][3].y);
                float ab[4] = {0.f, 0.f, 0.f, 0.f}, bl[4] = {0.f, 0.f, 0.f, 0.f};
                if (wl == 0 && up) {
                    const float4 t4 = *reinterpret_cast<const float4*>(nbr + (par * 2 + 0) * D + 4 * l);
                    ab[0] = t4.x; ab[1] = t4.y; ab[2] = t4.z; ab[3] = t4.w;
                    col_odd(ab, cm, c0, c1);
                }
                if (wl == NW - 1 && dn) {
                    const float4 t4 = *reinterpret_cast<const float4*>(nbr + (par * 2 + 1) * D + 4 * l);
                    bl[0] = t4.x; bl[1] = t4.y; bl[2] = t4.z; bl[3] = t4.w;
                    col_odd(bl, cm, c0, c1);
                }
                __syncthreads();
                const Rot rm = load_rot(pr, up ? 2 * w - 1 : 0), r0 = load_rot(pr, 2 * w), r1 = load_rot(pr, 2 * w + 1);
                if (dn) {
                    if (wl < NW - 1) {
                        const float4 b4 = *reinterpret_cast<const float4*>(rowx + (wl + 1) * 2 * D + 4 * l);
                        bl[0] = b4.x; bl[1] = b4.y; bl[2] = b4.z; bl[3] = b4.w;
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) a[1][j].y = fmaf(r1.s, fmaf(-r1.tau, bl[j], a[1][j].y), bl[j]);
                }
                if (up) {
                    if (wl > 0) {
                        const float4 a4 = *reinterpret_cast<const float4*>(rowx + (wl - 1) * 2 * D + D + 4 * l);
                        ab[0] = a4.x; ab[1] = a4.y; ab[2] = a4.z; ab[3] = a4.w;
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) a[0][j].x = fmaf(-rm.s, fmaf(rm.tau, ab[j], a[0][j].x), ab[j]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) rotswap(a[0][j].y, a[1][j].x, r0.s, r0.tau);
                if (w == l) {
                    a[0][1].y = fmaf(r0.t, d12, d22); a[1][2].x = fmaf(-r0.t, d12, d11);
                    a[0][2].y = 0.f; a[1][1].x = 0.f;
                }
            }
            publish(par ^ 1, E);
        }
    }
    if (rounds > 0) {
        __syncthreads();
        v_update(v, prm + ((rounds - 1) & 1) * 64, ((rounds - 1) & 1) == 0, l);
    }

    // Sort descending (ties: lower position first), sign-fix, write out.  V
    // rows go through global scratch, eigenvalues to every CTA.
    float* Vg = scratch + size_t(hd) * nchunks * D * D;    // [D][D] position-ordered columns
#pragma unroll
    for (int ip = 0; ip < 2; ++ip)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            Vg[size_t(4 * w + 2 * ip) * D + 4 * l + j] = v[ip][j].x;
            Vg[size_t(4 * w + 2 * ip + 1) * D + 4 * l + j] = v[ip][j].y;
        }
    if (w == l) {
        const float dv[4] = {a[0][0].x, a[0][1].y, a[1][2].x, a[1][3].y};
        for (int k = 0; k < C; ++k) {
            float* lm = cluster.map_shared_rank(lamall, k);
#pragma unroll
            for (int i = 0; i < 4; ++i) lm[4 * w + i] = dv[i];
        }
    }
#undef AE
    __threadfence();
    cluster.sync();
    constexpr int CPC = D / C;                 // columns per CTA
    for (int ci = wl; ci < CPC; ci += NW) {
        const int i = rank * CPC + ci;         // position
        const float li = lamall[i];
        int rk = 0;
        for (int j = l; j < D; j += 32) {
            const float lj = lamall[j];
            rk += (lj > li) || (lj == li && j < i);
        }
        for (int o = 16; o; o >>= 1) rk += __shfl_xor_sync(0xffffffffu, rk, o);
        float best = -1.f;
        int br = 0;
        for (int rr = l; rr < D; rr += 32) {
            const float av = fabsf(__ldcg(Vg + size_t(rr) * D + i));   // written by other CTAs: skip L1
            if (av > best) { best = av; br = rr; }
        }
        for (int o = 16; o; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int orr = __shfl_xor_sync(0xffffffffu, br, o);
            if (ob > best || (ob == best && orr < br)) { best = ob; br = orr; }
        }
        const float sgn = (__ldcg(Vg + size_t(br) * D + i) < 0.f) ? -1.f : 1.f;
        for (int rr = l; rr < D; rr += 32)
            basis_out[size_t(hd) * D * D + size_t(rr) * D + rk] = sgn * __ldcg(Vg + size_t(rr) * D + i);
        if (l == 0) eig_out[size_t(hd) * D + rk] = li;
    }
    if (rank == 0 && tid == 0) status[hd] = converged ? sweeps : -SPECTRA_ERR_NOT_CONVERGED;
    cluster.sync();   // no CTA leaves while others may still write into its shared memory
}

template <int C>
size_t jacobi128c_smem()
{
    constexpr int NW = 32 / C;
    return sizeof(float) * (NW * 2 * kJ2 + 4 * kJ2 + 4 * kJ2) + sizeof(float4) * 128 +
           sizeof(float) * (33 + 2 * C + kJ2) + sizeof(int) * C + 16;
}

template <int D>
size_t jacobi_smem()
{
    return sizeof(float) * (2 * D * (D + 1) + 3 * (D / 2)) + sizeof(int) * D + sizeof(float) * 33 + 16;
}

}  // namespace

int gram_chunks(int heads, int64_t n_cal)
{
    const int64_t want = (2 * 148 + heads - 1) / heads;
    const int64_t maxc = (n_cal + kGramTile - 1) / kGramTile;
    return int(std::max<int64_t>(1, std::min<int64_t>(want, maxc)));
}

spectra_status launch_gram(const spectra_plan* plan, const void* x, int dt, int64_t n_cal,
                           int64_t token_stride, float* partials, int nchunks, cudaStream_t s)
{
    const int64_t chunk_len = (n_cal + nchunks - 1) / nchunks;
    dim3 grid(nchunks, plan->heads);
    if (plan->head_dim == 128)
        gram_partial_kernel<128><<<grid, kGramThreads, 0, s>>>(x, dt, n_cal, token_stride,
                                                               plan->heads, chunk_len, partials);
    else
        gram_partial_kernel<64><<<grid, kGramThreads, 0, s>>>(x, dt, n_cal, token_stride,
                                                              plan->heads, chunk_len, partials);
    return cuda_status(cudaGetLastError());
}

spectra_status launch_jacobi(const spectra_plan* plan, const float* partials, int nchunks,
                             int64_t n_cal, int max_sweeps, float* gram_out, cudaStream_t s)
{
    const float inv_n = 1.0f / float(n_cal);
    if (plan->head_dim == 128) {
        // one cluster of kJacCluster CTAs per head; the Gram partials of the
        // head (at least D x D floats) double as the scratch of the final sort
        constexpr int C = kJacCluster;
        const size_t sm = jacobi128c_smem<C>();
        cudaFuncSetAttribute(jacobi128c_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm));
        jacobi128c_kernel<C><<<plan->heads * C, 1024 / C, sm, s>>>(partials, nchunks, inv_n, max_sweeps,
                                                                   plan->basis_mat, plan->eigvals, plan->status,
                                                                   gram_out, const_cast<float*>(partials));
    } else {
        const size_t sm = jacobi_smem<64>();
        cudaFuncSetAttribute(jacobi_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm));
        jacobi_kernel<64><<<plan->heads, kJacobiThreads, sm, s>>>(
            partials, nchunks, inv_n, max_sweeps, plan->basis_mat, plan->eigvals, plan->status, gram_out);
    }
    return cuda_status(cudaGetLastError());
}

}  // namespace spectra
