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
        const size_t sm = jacobi_smem<128>();
        cudaFuncSetAttribute(jacobi_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm));
        jacobi_kernel<128><<<plan->heads, kJacobiThreads, sm, s>>>(
            partials, nchunks, inv_n, max_sweeps, plan->basis_mat, plan->eigvals, plan->status, gram_out);
    } else {
        const size_t sm = jacobi_smem<64>();
        cudaFuncSetAttribute(jacobi_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm));
        jacobi_kernel<64><<<plan->heads, kJacobiThreads, sm, s>>>(
            partials, nchunks, inv_n, max_sweeps, plan->basis_mat, plan->eigvals, plan->status, gram_out);
    }
    return cuda_status(cudaGetLastError());
}

}  // namespace spectra
