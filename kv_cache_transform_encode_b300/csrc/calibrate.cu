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
// jacobi1s_kernel (d = 128): one-sided Jacobi on the Cholesky factor of G,
//   a cluster of CTAs per head; see the comment at the kernel.
// jacobi_kernel (d = 64): one block per head.  The matrix and the rotation
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

constexpr int kJ2 = 128;
#ifndef SPECTRA_J1S_CLUSTER
#define SPECTRA_J1S_CLUSTER 8
#endif
constexpr int kJ1sCluster = SPECTRA_J1S_CLUSTER;   // CTAs per head in the one-sided Jacobi (d = 128)

// ------------------------------------------------------------------ one-sided Jacobi
// jacobi1s_kernel<C>: Hestenes' one-sided cyclic Jacobi, spread over a
// cluster of C CTAs per head, on the Cholesky factor of the Gram matrix:
// R^T R = G + delta I (R upper triangular; the small shift delta keeps a
// singular G positive definite in fp32 and changes no eigenvector).  With
// X = R V (X = R, V = I at the start), each rotation of the column pair
// (p, q) makes X_p and X_q orthogonal and applies the same plane rotation
// to V; when every pair is orthogonal, X^T X = V^T (G + delta I) V is
// diagonal, so the columns of V are the eigenvectors of G, with eigenvalues
// lambda_i = |X_i|^2 - delta.  Rotating R rather than G itself keeps the
// convergence of the two-sided method on G (one-sided Jacobi on G behaves
// like two-sided Jacobi on G^2: half again as many sweeps).  The pair order is the
// odd-even ("caterpillar") one with rotation-and-swap: positions (2i, 2i+1)
// in even rounds, (2i+1, 2i+2) in odd rounds, and the rotated columns trade
// places, so every pair meets once in d rounds.  CTA r owns positions
// [r d/C, (r+1) d/C) with their whole columns of Gc and V in shared memory:
// all rotations are local, and in an odd round only the pair that
// straddles two CTAs needs a column from the neighbour, which that
// neighbour pushes into this CTA's shared memory (st.async, counted by an
// mbarrier) at the end of the even round before.  Both CTAs of a straddling
// pair compute its rotation from the same two columns in the same order, so
// they agree bit for bit; each keeps the half that lands in its position.
// The only cluster-wide barriers are once per sweep (convergence) and at
// the ends.
template <int C>
struct J1s {
    static constexpr int D = kJ2;
    static constexpr int PPC = D / C;       // positions (columns) per CTA
    static constexpr int NP = PPC / 2;      // local pairs in an even round
    static constexpr int NW = NP + 1;       // warps: one per pair + the left boundary
};

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(uint32_t(__cvta_generic_to_shared(p))), "r"(rank));
    return r;
}

// 16 bytes into another CTA's shared memory, counted on its mbarrier
__device__ __forceinline__ void st_async_v4(uint32_t raddr, float4 v, uint32_t rbar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(raddr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rbar)
                 : "memory");
}

__device__ __forceinline__ void mbar_init_local(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(uint32_t(__cvta_generic_to_shared(bar))), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(uint32_t(__cvta_generic_to_shared(bar))),
                 "r"(bytes)
                 : "memory");
}

// bounded wait for a phase of a local mbarrier (false after ~2 s)
__device__ __forceinline__ bool mbar_wait_phase(uint64_t* bar, uint32_t parity)
{
    const uint32_t a = uint32_t(__cvta_generic_to_shared(bar));
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((it & 63u) == 0) {
            uint64_t t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            if (it == 0) t0 = t;
            else if (t - t0 > 2000000000ull) return false;
        }
    }
}

// Rotation of the column pair (p, q): lane holds rows 4l..4l+3 of both.
// Returns (s, tau) with tau = s / (1 + c) (Rutishauser's form), or s = 0
// when the pair is already orthogonal to `tol`.  rel = |g| / sqrt(a b).
__device__ __forceinline__ float2 pair_rotation(float4 p, float4 q, float tol, float& rel)
{
    float a = p.x * p.x, b = q.x * q.x, g = p.x * q.x;
    a = fmaf(p.y, p.y, a); b = fmaf(q.y, q.y, b); g = fmaf(p.y, q.y, g);
    a = fmaf(p.z, p.z, a); b = fmaf(q.z, q.z, b); g = fmaf(p.z, q.z, g);
    a = fmaf(p.w, p.w, a); b = fmaf(q.w, q.w, b); g = fmaf(p.w, q.w, g);
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
        g += __shfl_xor_sync(0xffffffffu, g, o);
    }
    const float ab = a * b;
    rel = (ab > 0.f) ? fabsf(g) * rsqrtf(ab) : 0.f;
    // t = tan(theta) = 2 g sgn(d) / (|d| + sqrt(d^2 + 4 g^2)), d = b - a: the
    // smaller root, without the 1 / (2 g) of the textbook form
    const float dd = b - a, g2 = 2.f * g;
    const float h2 = fmaf(dd, dd, g2 * g2);
    const float hyp = h2 * rsqrtf(fmaxf(h2, 1e-37f));
    float t = __fdividef(g2, fabsf(dd) + hyp);
    t = (dd >= 0.f) ? t : -t;
    const float c = rsqrtf(fmaf(t, t, 1.f));
    const bool rot = ab > 0.f && g * g > tol * tol * ab;
    const float s = rot ? t * c : 0.f;
    const float tau = rot ? __fdividef(t * c, 1.f + c) : 0.f;
    return make_float2(s, tau);
}

// p' = c p - s q = p - s (q + tau p);  q' = s p + c q = q + s (p - tau q)
__device__ __forceinline__ float4 rot_p(float4 p, float4 q, float s, float tau)
{
    return make_float4(fmaf(-s, fmaf(tau, p.x, q.x), p.x), fmaf(-s, fmaf(tau, p.y, q.y), p.y),
                       fmaf(-s, fmaf(tau, p.z, q.z), p.z), fmaf(-s, fmaf(tau, p.w, q.w), p.w));
}
__device__ __forceinline__ float4 rot_q(float4 p, float4 q, float s, float tau)
{
    return make_float4(fmaf(s, fmaf(-tau, q.x, p.x), q.x), fmaf(s, fmaf(-tau, q.y, p.y), q.y),
                       fmaf(s, fmaf(-tau, q.z, p.z), q.z), fmaf(s, fmaf(-tau, q.w, p.w), q.w));
}

template <int C>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(32 * J1s<C>::NW, 1)
jacobi1s_kernel(const float* __restrict__ partials, int nchunks, float inv_n, int max_sweeps,
                float* __restrict__ basis_out, float* __restrict__ eig_out, int32_t* __restrict__ status,
                float* __restrict__ gram_out)
{
    namespace cg = cooperative_groups;
    constexpr int D = J1s<C>::D, PPC = J1s<C>::PPC, NP = J1s<C>::NP, NW = J1s<C>::NW;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int hd = blockIdx.x / C;
    const int tid = threadIdx.x, wl = tid >> 5, l = tid & 31;

    extern __shared__ __align__(16) float jsm[];
    float (*Gc)[D] = reinterpret_cast<float (*)[D]>(jsm);               // [PPC][D] columns of X
    float (*Vc)[D] = reinterpret_cast<float (*)[D]>(jsm + PPC * D);     // [PPC][D] columns of V
    float* Am = jsm + 2 * PPC * D;                                      // [D][D + 1] Gram / Cholesky
    __shared__ __align__(16) float rb[2][2][2][D];     // [X, V][side: from left, from right][parity][D]
    __shared__ __align__(8) uint64_t rbar[2][2][2];    // [X, V][side][parity]
    __shared__ float wred[NW];
    __shared__ float cred[2][C];                       // cluster exchange (two slots)
    __shared__ float lamall[D];
    __shared__ int cflag[2][C];
    __shared__ float invd[16];                         // 1 / L[j][j] of the current Cholesky panel

    if (tid == 0) {
        for (int xv = 0; xv < 2; ++xv)
            for (int sd = 0; sd < 2; ++sd)
                for (int pp = 0; pp < 2; ++pp) mbar_init_local(&rbar[xv][sd][pp], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    cluster.sync();    // every CTA of the cluster runs before any shared memory is touched remotely
    constexpr int AS = D + 1;                          // Cholesky row stride (conflict-free columns)
    // the Gram matrix: CTA r sums rows [r d/C, (r+1) d/C) of the chunk
    // partials (fixed order) and writes them into every CTA's copy
    bool bad = false;
    {
        const int rb0 = rank * PPC;
        for (int e = tid; e < PPC * D; e += 32 * NW) {
            const int r = rb0 + e / D, c = e % D;
            const float* src = partials + size_t(hd) * nchunks * D * D + size_t(r) * D + c;
            float sum = 0.f;
            int ch = 0;
            for (; ch + 4 <= nchunks; ch += 4) {
                const float a0 = src[size_t(ch) * D * D], a1 = src[size_t(ch + 1) * D * D];
                const float a2 = src[size_t(ch + 2) * D * D], a3 = src[size_t(ch + 3) * D * D];
                sum += a0; sum += a1; sum += a2; sum += a3;
            }
            for (; ch < nchunks; ++ch) sum += src[size_t(ch) * D * D];
            sum *= inv_n;
            if (gram_out) gram_out[size_t(hd) * D * D + size_t(r) * D + c] = sum;
            bad |= !isfinite(sum);
            for (int k = 0; k < C; ++k) *cluster.map_shared_rank(&Am[r * AS + c], k) = sum;
        }
    }
    {
        const int bl = __syncthreads_or(bad);
        if (tid < C) *cluster.map_shared_rank(&cflag[0][rank], tid) = bl;
        cluster.sync();   // also: every CTA's rows of the Gram matrix have landed everywhere
        int any = 0;
        for (int k = 0; k < C; ++k) any |= cflag[0][k];
        if (any) {
            for (int e = tid; e < PPC * D; e += 32 * NW) {
                const int r = e / PPC, c = rank * PPC + e % PPC;
                basis_out[size_t(hd) * D * D + size_t(r) * D + c] = (r == c) ? 1.f : 0.f;
            }
            if (rank == 0 && tid < D) eig_out[size_t(hd) * D + tid] = 0.f;
            if (rank == 0 && tid == 0) status[hd] = -SPECTRA_ERR_NONFINITE;
            cluster.sync();
            return;
        }
    }

    // G + delta I = L L^T (L lower triangular, in place), R = L^T.  delta is
    // a few fp32 rounding units of the largest diagonal entry times d, so a
    // positive semi-definite G never meets a non-positive pivot.
    float dmax = 0.f;
    for (int i = 0; i < D; ++i) dmax = fmaxf(dmax, Am[i * AS + i]);
    const float delta = 8e-7f * float(D) * dmax;
    for (int i = tid; i < D; i += 32 * NW) Am[i * AS + i] += delta;
    // Blocked right-looking factorization, 16-column panels: warp 0 factors
    // the diagonal block, every thread then solves rows of the panel below
    // it (forward substitution), and 4x4 register tiles apply the rank-16
    // update to the trailing lower triangle (the upper triangle of Am is
    // scratch: it is never read).
    constexpr int NB = 16;
    for (int c0 = 0; c0 < D; c0 += NB) {
        __syncthreads();
        if (wl == 0) {
            for (int j = c0; j < c0 + NB; ++j) {
                const float piv = fmaxf(Am[j * AS + j], 1e-30f);
                const float rs = rsqrtf(piv);
                const int i = j + 1 + l;
                const float lij = (i < c0 + NB) ? Am[i * AS + j] * rs : 0.f;
                __syncwarp();
                if (l == 0) {
                    Am[j * AS + j] = piv * rs;
                    invd[j - c0] = rs;
                }
                if (i < c0 + NB) Am[i * AS + j] = lij;
                __syncwarp();
                for (int e = l; e < NB * NB; e += 32) {
                    const int ii = c0 + e / NB, kk = c0 + e % NB;
                    if (kk > j && kk <= ii) Am[ii * AS + kk] = fmaf(-Am[ii * AS + j], Am[kk * AS + j], Am[ii * AS + kk]);
                }
                __syncwarp();
            }
        }
        __syncthreads();
        for (int i = c0 + NB + tid; i < D; i += 32 * NW) {
            float x[NB];
#pragma unroll
            for (int m = 0; m < NB; ++m) {
                float a = Am[i * AS + c0 + m];
#pragma unroll
                for (int q = 0; q < m; ++q) a = fmaf(-x[q], Am[(c0 + m) * AS + c0 + q], a);
                x[m] = a * invd[m];
                Am[i * AS + c0 + m] = x[m];
            }
        }
        __syncthreads();
        const int n4 = (D - c0 - NB) / 4;
        for (int t = tid; t < n4 * n4; t += 32 * NW) {
            const int ti = t / n4, tk = t % n4;
            if (tk > ti) continue;
            const int i0 = c0 + NB + 4 * ti, k0 = c0 + NB + 4 * tk;
            float acc[4][4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[r][q] = Am[(i0 + r) * AS + k0 + q];
#pragma unroll 4
            for (int m = 0; m < NB; ++m) {
                float li[4], lk[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) { li[r] = Am[(i0 + r) * AS + c0 + m]; lk[r] = Am[(k0 + r) * AS + c0 + m]; }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(-li[r], lk[q], acc[r][q]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) Am[(i0 + r) * AS + k0 + q] = acc[r][q];
        }
    }
    __syncthreads();
    // X = R: column c of R is row c of L (zero past the diagonal); V = I
    for (int e = tid; e < PPC * D; e += 32 * NW) {
        const int cl = e / D, r = e % D, c = rank * PPC + cl;
        Gc[cl][r] = (r <= c) ? Am[c * AS + r] : 0.f;
        Vc[cl][r] = (r == c) ? 1.f : 0.f;
    }
    __syncthreads();

    constexpr float kTol = 2e-6f;      // |X_p . X_q| / (|X_p| |X_q|) below which a pair counts as orthogonal
    int sweeps = 0, converged = 0, failed = 0, cuse = 1;
    float prev_m = INFINITY;
    uint32_t gr = 0;                   // rounds so far (all sweeps)
    float4* G4 = reinterpret_cast<float4*>(&Gc[0][0]);
    float4* V4 = reinterpret_cast<float4*>(&Vc[0][0]);
    constexpr int Q = D / 4;           // float4 per column
    constexpr uint32_t kColBytesH = D * 4; // one column
    // V trails X by one round: in round r a warp rotates the X pair of its
    // round-r role and applies, in the same instructions stream, the rotation
    // it found in round r-1 to the V pair of its round-(r-1) role (nothing
    // reads V before the end, so its updates fill the latency of the X
    // chain).  (ps, ptau): this warp's rotation of the previous round.
    float ps = 0.f, ptau = 0.f;
    auto send_col = [&](int xv, int side, uint32_t kp, uint32_t rk, float4 v) {
        st_async_v4(cluster_map(&rb[xv][side][kp][4 * l], rk), v, cluster_map(&rbar[xv][side][kp], rk));
    };
    auto recv_col = [&](int xv, int side, uint32_t kp, uint32_t ph) -> float4 {
        if (l == 0) mbar_expect(&rbar[xv][side][kp], kColBytesH);
        if (!mbar_wait_phase(&rbar[xv][side][kp], ph)) failed = 1;
        return *reinterpret_cast<const float4*>(&rb[xv][side][kp][4 * l]);
    };
    // even round (or the final V-only step when !dox): X pairs (2w, 2w+1);
    // V of the previous (odd) round: pairs (2w+1, 2w+2), the boundaries
    auto even_round = [&](bool dox, bool dov, uint32_t kx, uint32_t kv) -> float {
        float rel = 0.f;
        const uint32_t kxp = kx & 1, kvp = kv & 1, kvph = (kv >> 1) & 1;
        float2 st = make_float2(0.f, 0.f);
        if (wl < NP) {
            const int P = 2 * wl;
            if (dox) {
                const float4 gp = G4[P * Q + l], gq = G4[(P + 1) * Q + l];
                st = pair_rotation(gp, gq, kTol, rel);
                const float4 gq2 = rot_q(gp, gq, st.x, st.y), gp2 = rot_p(gp, gq, st.x, st.y);
                G4[P * Q + l] = gq2;
                G4[(P + 1) * Q + l] = gp2;
                if (P == 0 && rank > 0) send_col(0, 1, kxp, uint32_t(rank - 1), gq2);
                if (P + 1 == PPC - 1 && rank < C - 1) send_col(0, 0, kxp, uint32_t(rank + 1), gp2);
            }
            if (dov) {
                if (wl < NP - 1) {                       // previous odd local pair (2w+1, 2w+2)
                    const int R = 2 * wl + 1;
                    const float4 vp = V4[R * Q + l], vq = V4[(R + 1) * Q + l];
                    V4[R * Q + l] = rot_q(vp, vq, ps, ptau);
                    V4[(R + 1) * Q + l] = rot_p(vp, vq, ps, ptau);
                } else if (rank < C - 1) {               // previous right boundary
                    const float4 vp = V4[(PPC - 1) * Q + l];
                    const float4 vq = recv_col(1, 1, kvp, kvph);
                    V4[(PPC - 1) * Q + l] = rot_q(vp, vq, ps, ptau);
                }
            }
        } else if (dov && rank > 0) {                    // previous left boundary
            const float4 vq = V4[l];
            const float4 vp = recv_col(1, 0, kvp, kvph);
            V4[l] = rot_p(vp, vq, ps, ptau);
        }
        ps = st.x;
        ptau = st.y;
        return rel;
    };
    // odd round: X pairs (2w+1, 2w+2) and the boundaries; V of the previous
    // (even) round: pairs (2w, 2w+1), whose edge columns go to the neighbours
    auto odd_round = [&](uint32_t kx, uint32_t kv) -> float {
        float rel = 0.f;
        const uint32_t kxp = kx & 1, kxph = (kx >> 1) & 1, kvp = kv & 1;
        float2 st = make_float2(0.f, 0.f);
        if (wl < NP - 1) {
            const int P = 2 * wl + 1;
            const float4 gp = G4[P * Q + l], gq = G4[(P + 1) * Q + l];
            st = pair_rotation(gp, gq, kTol, rel);
            G4[P * Q + l] = rot_q(gp, gq, st.x, st.y);
            G4[(P + 1) * Q + l] = rot_p(gp, gq, st.x, st.y);
        } else if (wl == NP - 1) {
            if (rank < C - 1) {
                const float4 gp = G4[(PPC - 1) * Q + l];
                const float4 gq = recv_col(0, 1, kxp, kxph);
                st = pair_rotation(gp, gq, kTol, rel);
                G4[(PPC - 1) * Q + l] = rot_q(gp, gq, st.x, st.y);
            }
        } else {
            if (rank > 0) {
                const float4 gq = G4[l];
                const float4 gp = recv_col(0, 0, kxp, kxph);
                st = pair_rotation(gp, gq, kTol, rel);
                G4[l] = rot_p(gp, gq, st.x, st.y);
            }
        }
        if (wl < NP) {                                   // previous even pair (2w, 2w+1)
            const int P = 2 * wl;
            const float4 vp = V4[P * Q + l], vq = V4[(P + 1) * Q + l];
            const float4 vq2 = rot_q(vp, vq, ps, ptau), vp2 = rot_p(vp, vq, ps, ptau);
            V4[P * Q + l] = vq2;
            V4[(P + 1) * Q + l] = vp2;
            if (P == 0 && rank > 0) send_col(1, 1, kvp, uint32_t(rank - 1), vq2);
            if (P + 1 == PPC - 1 && rank < C - 1) send_col(1, 0, kvp, uint32_t(rank + 1), vp2);
        }
        ps = st.x;
        ptau = st.y;
        return rel;
    };
    for (;;) {
        if (sweeps >= max_sweeps) break;
        ++sweeps;
        float mrel = 0.f;
        for (int r = 0; r < D; ++r, ++gr) {
            // odd-round index of this round (X) and of the previous one (V)
            const uint32_t kx = gr >> 1, kv = (gr - 1) >> 1;
            if ((gr & 1) == 0) mrel = fmaxf(mrel, even_round(true, gr > 0, kx, kv));
            else mrel = fmaxf(mrel, odd_round(kx, kv));
            __syncthreads();
        }
        // sweep done: cluster-wide max of the pair residuals and the failure flag
        if (l == 0) wred[wl] = failed ? INFINITY : mrel;
        __syncthreads();
        if (tid < C) {
            float m = 0.f;
            for (int w = 0; w < NW; ++w) m = fmaxf(m, wred[w]);
            *cluster.map_shared_rank(&cred[cuse & 1][rank], tid) = m;
        }
        cluster.sync();
        float m = 0.f;
        for (int kk = 0; kk < C; ++kk) m = fmaxf(m, cred[cuse & 1][kk]);
        ++cuse;
        if (m == INFINITY) { failed = 1; break; }
        // converged when no pair needed a rotation, or when this sweep
        // started within the quadratic regime (every pair orthogonal to
        // 1e-3 in the previous sweep: this one has taken them to rounding
        // level, and a further sweep would rotate nothing)
        if (m <= kTol || prev_m <= 1e-3f) { converged = 1; break; }
        prev_m = m;
    }
    if (gr > 0) {   // the last (odd) round's rotations still owe their V update
        even_round(false, true, gr >> 1, (gr - 1) >> 1);
        __syncthreads();
    }

    // eigenvalues (Rayleigh quotients) to every CTA; ranks, sign fix, output
    for (int P = wl; P < PPC; P += NW) {
        const float4 g = G4[P * Q + l];
        const float lam = warp_sum(g.x * g.x + g.y * g.y + g.z * g.z + g.w * g.w) - delta;
        if (l < C) *cluster.map_shared_rank(&lamall[rank * PPC + P], l) = lam;
    }
    cluster.sync();
    for (int P = wl; P < PPC; P += NW) {
        const int i = rank * PPC + P;
        const float li = lamall[i];
        int rk = 0;
        for (int j = l; j < D; j += 32) {
            const float lj = lamall[j];
            rk += (lj > li) || (lj == li && j < i);
        }
        rk = int(warp_sum(float(rk)) + 0.5f);
        const float4 v = V4[P * Q + l];
        float best = fabsf(v.x);
        int br = 4 * l;
        if (fabsf(v.y) > best) { best = fabsf(v.y); br = 4 * l + 1; }
        if (fabsf(v.z) > best) { best = fabsf(v.z); br = 4 * l + 2; }
        if (fabsf(v.w) > best) { best = fabsf(v.w); br = 4 * l + 3; }
        float bv = (br == 4 * l) ? v.x : (br == 4 * l + 1) ? v.y : (br == 4 * l + 2) ? v.z : v.w;
        for (int o = 16; o; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int orr = __shfl_xor_sync(0xffffffffu, br, o);
            const float obv = __shfl_xor_sync(0xffffffffu, bv, o);
            if (ob > best || (ob == best && orr < br)) { best = ob; br = orr; bv = obv; }
        }
        const float sgn = (bv < 0.f) ? -1.f : 1.f;
        float* dst = basis_out + size_t(hd) * D * D + rk;
        dst[size_t(4 * l) * D] = sgn * v.x;
        dst[size_t(4 * l + 1) * D] = sgn * v.y;
        dst[size_t(4 * l + 2) * D] = sgn * v.z;
        dst[size_t(4 * l + 3) * D] = sgn * v.w;
        if (l == 0) eig_out[size_t(hd) * D + rk] = li;
    }
    if (rank == 0 && tid == 0)
        status[hd] = failed ? -SPECTRA_ERR_TIMEOUT : converged ? sweeps : -SPECTRA_ERR_NOT_CONVERGED;
    cluster.sync();   // no CTA leaves while others may still write into its shared memory
}

template <int D>
size_t jacobi_smem()
{
    return sizeof(float) * (2 * D * (D + 1) + 3 * (D / 2)) + sizeof(int) * D + sizeof(float) * 33 + 16;
}

}  // namespace

// Plain-KV calibration ("Technisch Overzicht ...", "Belangrijkste
// Bijdragen" 1: scalar quantization without rotation): the identity basis and
// the raw coordinates' second moments, the Gram diagonal summed from the
// chunk partials in chunk order.
template <int D>
__global__ void __launch_bounds__(D)
plain_calibrate_kernel(const float* __restrict__ partials, int nchunks, float inv_n, float* __restrict__ basis,
                       float* __restrict__ eig, int32_t* __restrict__ status)
{
    const int h = blockIdx.x, c = threadIdx.x;
    float s = 0.f;
    for (int ch = 0; ch < nchunks; ++ch) s += partials[((size_t(h) * nchunks + ch) * D + c) * D + c];
    const float v = s * inv_n;
    eig[size_t(h) * D + c] = v;
    for (int i = 0; i < D; ++i) basis[(size_t(h) * D + i) * D + c] = (i == c) ? 1.f : 0.f;
    const int bad = __syncthreads_or(!isfinite(v));
    if (c == 0) status[h] = bad ? -SPECTRA_ERR_NONFINITE : 0;
}

spectra_status launch_plain_calibrate(const spectra_plan* plan, const float* partials, int nchunks, int64_t n_cal,
                                      cudaStream_t s)
{
    const float inv_n = 1.0f / float(n_cal);
    if (plan->head_dim == 128)
        plain_calibrate_kernel<128><<<plan->heads, 128, 0, s>>>(partials, nchunks, inv_n, plan->basis_mat,
                                                                plan->eigvals, plan->status);
    else
        plain_calibrate_kernel<64><<<plan->heads, 64, 0, s>>>(partials, nchunks, inv_n, plan->basis_mat,
                                                              plan->eigvals, plan->status);
    return cuda_status(cudaGetLastError());
}

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
        // one cluster of kJ1sCluster CTAs per head (one-sided Jacobi on the
        // Cholesky factor); d = 64 keeps the one-block two-sided kernel
        constexpr int C = kJ1sCluster;
        const size_t sm = sizeof(float) * (2 * J1s<C>::PPC * kJ2 + kJ2 * (kJ2 + 1));
        if (spectra_status st = set_smem(jacobi1s_kernel<C>, sm)) return st;
        if (C > 8 && cudaFuncSetAttribute(jacobi1s_kernel<C>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1))
            return SPECTRA_ERR_CUDA;
        jacobi1s_kernel<C><<<plan->heads * C, 32 * J1s<C>::NW, sm, s>>>(partials, nchunks, inv_n, max_sweeps,
                                                                      plan->basis_mat, plan->eigvals, plan->status,
                                                                      gram_out);
    } else {
        const size_t sm = jacobi_smem<64>();
        if (spectra_status st = set_smem(jacobi_kernel<64>, sm)) return st;
        jacobi_kernel<64><<<plan->heads, kJacobiThreads, sm, s>>>(
            partials, nchunks, inv_n, max_sweeps, plan->basis_mat, plan->eigvals, plan->status, gram_out);
    }
    return cuda_status(cudaGetLastError());
}

}  // namespace spectra
