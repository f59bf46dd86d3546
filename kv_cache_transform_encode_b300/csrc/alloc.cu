// alloc.cu -- integer reverse water-filling, plan finalization and the
// Gaussian Lloyd-Max tables.
//
// "Sintesi Tecnica: SPECTRA", "La Pipeline di SPECTRA" phase 2: reverse
// water-filling on the measured marginal variances -- more bits to
// high-variance latent coordinates, fewer (down to zero) to the rest;
// "Metodologia" item 2: zero-bit channels are dropped.
//
// The greedy rule (R_tot one-bit steps, each to the channel with the largest
// lam_c * 4^-b_c, lowest index on ties) picks, in order, the R_tot largest
// keys of the multiset {lam_c 4^-k : c < d, 0 <= k < 8}: every channel's keys
// fall with k, so a channel's chosen keys are a prefix.  alloc_kernel selects
// those keys directly: one thread per key (thread c*8+k), a bisection on the
// fp64 bit pattern of the R_tot-th largest key (64 block-wide counts), then
// ties at that value broken in thread order, which is (c asc, k asc) -- the
// greedy's tie order.  Keys are exact powers-of-two scalings of fp32
// eigenvalues, so the result is bit-identical to the sequential greedy.
#include "spectra_internal.cuh"

#include <math.h>

namespace spectra {

namespace {

template <int D>
__global__ void __launch_bounds__(D * 8)
alloc_kernel(const float* __restrict__ eig, int R, int fixed_bits, uint8_t* __restrict__ bits_out)
{
    __shared__ int warp_tot[32];
    const int h = blockIdx.x, tid = threadIdx.x;
    const int c = tid >> 3, k = tid & 7;
    const int lane = tid & 31, warp = tid >> 5;
    uint8_t* bo = bits_out + size_t(h) * D;
    if (fixed_bits > 0) {
        if (k == 0) bo[c] = uint8_t(fixed_bits);
        return;
    }
    float lf = eig[size_t(h) * D + c];
    lf = (lf > 0.f) ? lf : 0.f;     // negative or NaN -> 0
    const double key = ldexp(double(lf), -2 * k);
    const unsigned long long kb = static_cast<unsigned long long>(__double_as_longlong(key));

    bool sel = false;
    if (R > 0) {
        // smallest u with #{keys > u} < R  ==  the R-th largest key
        unsigned long long lo = 0ull, hi = 0x7FF0000000000000ull;
        while (lo < hi) {
            const unsigned long long mid = lo + ((hi - lo) >> 1);
            const int gt = __syncthreads_count(kb > mid);
            if (gt < R) hi = mid; else lo = mid + 1;
        }
        const bool gt = kb > lo, eq = kb == lo;
        const int n_gt = __syncthreads_count(gt);
        const int need = R - n_gt;
        // rank of this key among equal keys, in thread order
        const unsigned m = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) warp_tot[warp] = __popc(m);
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w) before += warp_tot[w];
        before += __popc(m & ((1u << lane) - 1u));
        sel = gt || (eq && before < need);
    }
    const unsigned sm = __ballot_sync(0xffffffffu, sel);
    if (k == 0) bo[c] = uint8_t(__popc((sm >> (lane & ~7)) & 0xFFu));
}

// Grouped reverse water-filling ("La Pipeline di SPECTRA" phase 2,
// "Raggruppamento": adjacent latent coordinates share one width), over the
// first keep[h] channels (the rest get 0 bits: the effective-dimension
// pruning of "Technisch Overzicht ...", "Regime-Specifieke Prestaties").
// Groups of g consecutive channels, floor(keep / g) of them; the greedy's
// steps give a whole group one bit each, on the key Lam_G 4^-b with Lam_G the
// group's clipped eigenvalues summed in fp64 in ascending channel order.  The
// same top-`steps` selection as alloc_kernel, over the keys Lam_G 4^-k of the
// kept groups (thread 8 G + k); keys of groups past the kept ones never
// count (they are 0 and come after every kept key in thread order, and
// steps <= 8 * kept groups).
template <int D>
__global__ void __launch_bounds__(D * 8)
alloc_grouped_kernel(const float* __restrict__ eig, int R, int g, const int32_t* __restrict__ keep,
                     uint8_t* __restrict__ bits_out)
{
    __shared__ int warp_tot[32];
    __shared__ double Lam[D];
    const int h = blockIdx.x, tid = threadIdx.x;
    const int G = tid >> 3, k = tid & 7;
    const int lane = tid & 31, warp = tid >> 5;
    int kp = keep ? keep[h] : D;
    kp = kp < 0 ? 0 : (kp > D ? D : kp);
    const int ng = kp / g;                       // kept groups
    const int steps = min(R / g, 8 * ng);
    if (k == 0 && G < ng) {
        double s = 0.0;
        for (int c = G * g; c < (G + 1) * g; ++c) {
            const float lf = eig[size_t(h) * D + c];
            s += double(lf > 0.f ? lf : 0.f);
        }
        Lam[G] = s;
    }
    __syncthreads();
    const double key = (G < ng) ? ldexp(Lam[G], -2 * k) : 0.0;
    const unsigned long long kb = static_cast<unsigned long long>(__double_as_longlong(key));
    bool sel = false;
    if (steps > 0) {
        unsigned long long lo = 0ull, hi = 0x7FF0000000000000ull;
        while (lo < hi) {
            const unsigned long long mid = lo + ((hi - lo) >> 1);
            const int gt = __syncthreads_count(kb > mid);
            if (gt < steps) hi = mid; else lo = mid + 1;
        }
        const bool gt = kb > lo, eq = kb == lo && G < ng;
        const int n_gt = __syncthreads_count(gt);
        const int need = steps - n_gt;
        const unsigned m = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) warp_tot[warp] = __popc(m);
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w) before += warp_tot[w];
        before += __popc(m & ((1u << lane) - 1u));
        sel = (gt && G < ng) || (eq && before < need);
    }
    const unsigned sm = __ballot_sync(0xffffffffu, sel);
    const int width = __popc((sm >> (lane & ~7)) & 0xFFu);
    if (G < D / g)
        for (int c = G * g + k; c < (G + 1) * g; c += 8) bits_out[size_t(h) * D + c] = uint8_t(G < ng ? width : 0);
}

// Effective dimension with spectral-gap pruning ("Technisch Overzicht ...",
// "Regime-Specifieke Prestaties"), one warp per head, lane 0 in fp64:
// d_energy = the smallest k whose leading k clipped eigenvalues hold `energy`
// of their sum; d_gap = the k in 1 .. min(d_energy, d - 1) with the largest
// lam_{k-1} / lam_k (exact cross products; smallest k on ties).
__global__ void effdim_kernel(const float* __restrict__ eig, int d, double energy, int32_t* __restrict__ d_energy,
                              int32_t* __restrict__ d_gap)
{
    const int h = blockIdx.x;
    if (threadIdx.x != 0) return;
    const float* l = eig + size_t(h) * d;
    auto lam = [&](int c) { return double(l[c] > 0.f ? l[c] : 0.f); };
    double tot = 0.0;
    for (int c = 0; c < d; ++c) tot += lam(c);
    int de = 0;
    if (tot > 0.0) {
        double cum = 0.0;
        while (de < d) {
            cum += lam(de);
            ++de;
            if (cum >= energy * tot) break;
        }
    }
    int best = de;
    if (de > 0 && d > 1) {
        const int kmax = de < d - 1 ? de : d - 1;
        best = 1;
        for (int k = 2; k <= kmax; ++k)
            if (lam(k - 1) * lam(best) > lam(best - 1) * lam(k)) best = k;
    }
    d_energy[h] = de;
    d_gap[h] = best;
}

// Per-head offsets, record size and quantizer scales.
template <int D>
__global__ void __launch_bounds__(D)
finalize_kernel(int basis, int quant, int max_rec_bits, const float* __restrict__ eig,
                const uint8_t* __restrict__ bits, int32_t* __restrict__ rec_bits,
                uint16_t* __restrict__ chan_off, float* __restrict__ qscale,
                float* __restrict__ rscale, int32_t* __restrict__ status)
{
    __shared__ int wsum[D / 32];
    const int h = blockIdx.x, c = threadIdx.x, lane = c & 31, warp = c >> 5;
    const int b = bits[size_t(h) * D + c];
    int incl = b;
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int base = 0, total = 0;
    for (int w = 0; w < D / 32; ++w) {
        if (w < warp) base += wsum[w];
        total += wsum[w];
    }
    chan_off[size_t(h) * D + c] = uint16_t(base + incl - b);
    float qs = 1.f, rs = 1.f;
    if (basis == SPECTRA_BASIS_EIGEN && b > 0) {
        float lam = eig[size_t(h) * D + c];
        lam = (lam > 0.f) ? lam : 0.f;
        const float sig = sqrtf(lam);
        if (quant == SPECTRA_Q_UNIFORM3S) {
            const float levels = float(1 << b);
            qs = (sig > 0.f) ? levels / (6.f * sig) : 0.f;
            rs = 6.f * sig / levels;
        } else {
            qs = (sig > 0.f) ? 1.f / sig : 0.f;
            rs = sig;
        }
    }
    qscale[size_t(h) * D + c] = qs;
    rscale[size_t(h) * D + c] = rs;
    if (c == 0) {
        rec_bits[h] = total;
        if (total > max_rec_bits || b > 8) status[h] = -SPECTRA_ERR_BUFFER;
    }
}

// Gaussian Lloyd-Max codebooks for widths 1..8 (one warp per width, one
// block per width).  The optimal levels of N(0,1) are the fixed point of
// Lloyd's map: each level equals the centroid of its cell,
//   c_k = (phi(t_k) - phi(t_{k+1})) / (Phi(t_{k+1}) - Phi(t_k)),
// with thresholds t at the midpoints of adjacent levels.  Solved here by
// Newton's method on G(a) = a - c(a) (tridiagonal Jacobian, Thomas solve)
// with a backtracking line search on max|G| that keeps the levels ordered --
// a different solver from plain Lloyd iteration, reaching the same fixed
// point.  By symmetry only the L/2 positive levels are unknowns.
constexpr int kHalfMax = 128;

// Evaluates G = a - c(a) over the positive half; optionally the Jacobian
// bands.  Returns max |G| over the warp.
__device__ double lm_eval(const double* a, int H, int lane, double* G, double* lo, double* up, double* dg)
{
    const double inv_sqrt2 = 0.70710678118654752440;
    const double inv_sqrt2pi = 0.39894228040143267794;
    double gmax = 0.0;
    for (int k = lane; k < H; k += 32) {
        const double ak = a[k];
        const bool last = (k == H - 1);
        const double tk = (k == 0) ? 0.0 : 0.5 * (a[k - 1] + ak);
        const double tk1 = last ? 0.0 : 0.5 * (ak + a[k + 1]);
        const double Qk = 0.5 * erfc(tk * inv_sqrt2);
        const double Qk1 = last ? 0.0 : 0.5 * erfc(tk1 * inv_sqrt2);
        const double phk = inv_sqrt2pi * exp(-0.5 * tk * tk);
        const double phk1 = last ? 0.0 : inv_sqrt2pi * exp(-0.5 * tk1 * tk1);
        const double P = Qk - Qk1;
        const double c = (phk - phk1) / P;
        const double g = ak - c;
        gmax = fmax(gmax, fabs(g));
        if (G) {
            const double dck = (k >= 1) ? phk * (c - tk) / P : 0.0;      // dc/dt_k
            const double dck1 = last ? 0.0 : phk1 * (tk1 - c) / P;       // dc/dt_{k+1}
            G[k] = g;
            lo[k] = -0.5 * dck;
            up[k] = -0.5 * dck1;
            dg[k] = 1.0 - 0.5 * dck - 0.5 * dck1;
        }
    }
    for (int o = 16; o; o >>= 1) gmax = fmax(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
    return gmax;
}

__global__ void __launch_bounds__(32)
lm_tables_kernel(float* __restrict__ levels, float* __restrict__ thresh)
{
    __shared__ double a[kHalfMax], tr[kHalfMax], f[kHalfMax], lo[kHalfMax], up[kHalfMax], dg[kHalfMax];
    const int lane = threadIdx.x;
    const int b = blockIdx.x + 1, L = 1 << b, H = L >> 1;
    for (int k = lane; k < H; k += 32) a[k] = normcdfinv((H + k + 0.5) / double(L));
    __syncwarp();
    for (int it = 0; it < 100; ++it) {
        const double g0 = lm_eval(a, H, lane, f, lo, up, dg);
        __syncwarp();
        if (g0 < 1e-13) break;
        if (lane == 0) {   // Thomas solve J delta = -G (in place: up <- c', f <- d')
            double m = dg[0];
            up[0] /= m;
            f[0] = -f[0] / m;
            for (int k = 1; k < H; ++k) {
                m = dg[k] - lo[k] * up[k - 1];
                up[k] /= m;
                f[k] = (-f[k] - lo[k] * f[k - 1]) / m;
            }
            for (int k = H - 2; k >= 0; --k) f[k] -= up[k] * f[k + 1];
        }
        __syncwarp();
        double lam = 1.0;
        bool accepted = false;
        for (int ls = 0; ls < 50 && !accepted; ++ls, lam *= 0.5) {
            for (int k = lane; k < H; k += 32) tr[k] = a[k] + lam * f[k];
            __syncwarp();
            bool mono = true;
            for (int k = lane; k < H; k += 32) mono = mono && (tr[k] > ((k == 0) ? 0.0 : tr[k - 1]));
            mono = __all_sync(0xffffffffu, mono);
            if (mono) accepted = lm_eval(tr, H, lane, nullptr, nullptr, nullptr, nullptr) < g0;
            __syncwarp();
        }
        if (!accepted) break;
        for (int k = lane; k < H; k += 32) a[k] = tr[k];
        __syncwarp();
    }
    float* lv = levels + (b - 1) * kLmStride;
    float* th = thresh + (b - 1) * kLmStride;
    for (int k = lane; k < H; k += 32) {
        lv[H + k] = float(a[k]);
        lv[H - 1 - k] = float(-a[k]);
    }
    for (int j = lane; j < L; j += 32) {
        double t;
        if (j == 0) { th[0] = -INFINITY; continue; }
        if (j == H) t = 0.0;
        else if (j > H) t = 0.5 * (a[j - H - 1] + a[j - H]);
        else t = -0.5 * (a[L - j - H - 1] + a[L - j - H]);
        th[j] = float(t);
    }
}

// The bucket table of the Lloyd-Max encode (layout in spectra_internal.cuh)
// from the thresholds, with a check of its premise: no threshold below the
// inner grid or above it, at most one inside any bucket.  One block.
__global__ void __launch_bounds__(256)
lm_bucket_kernel(const float* __restrict__ thresh, float2* __restrict__ tab, int32_t* __restrict__ bad)
{
    bool ok = true;
    for (int e = threadIdx.x; e < kBkEntries; e += blockDim.x) {
        int b = 1;
        while (b < kMaxBits && e >= bk_off(b + 1)) ++b;
        const int j = e - bk_off(b), NB = 1 << bk_log(b), L = 1 << b;
        const float w = ldexpf(1.f, -bk_shift(b));
        const float ej = float(j - NB / 2) * w;                 // left edge (exact)
        const float* tt = thresh + (b - 1) * kLmStride;         // tt[1 .. L-1] ascending
        int cnt = 0;
        for (int step = L >> 1; step; step >>= 1)
            if (tt[cnt + step] <= ej) cnt += step;
        const float hi = cnt + 1 <= L - 1 ? tt[cnt + 1] : INFINITY;
        bool e_ok = hi == hi && hi > ej;
        if (cnt + 2 <= L - 1 && !(tt[cnt + 2] >= ej + w)) e_ok = false;   // two thresholds in one bucket
        if (j == 0 && (cnt != 0 || !(hi >= ej + w))) e_ok = false;          // none below the inner grid
        if (j >= NB - 1 && cnt != L - 1) e_ok = false;                      // none above it
        tab[e] = make_float2(hi, __int_as_float(cnt));
        ok = ok && e_ok;
    }
    const int any_bad = __syncthreads_or(!ok);
    if (threadIdx.x == 0) *bad = any_bad ? 1 : 0;
}

}  // namespace

spectra_status launch_alloc(const spectra_plan* plan, int R_tot, int fixed_bits, cudaStream_t s)
{
    if (plan->head_dim == 128)
        alloc_kernel<128><<<plan->heads, 128 * 8, 0, s>>>(plan->eigvals, R_tot, fixed_bits, plan->bits);
    else
        alloc_kernel<64><<<plan->heads, 64 * 8, 0, s>>>(plan->eigvals, R_tot, fixed_bits, plan->bits);
    return cuda_status(cudaGetLastError());
}

spectra_status launch_alloc_grouped(const spectra_plan* plan, int R_tot, int group, const int32_t* keep,
                                    cudaStream_t s)
{
    if (plan->head_dim == 128)
        alloc_grouped_kernel<128><<<plan->heads, 128 * 8, 0, s>>>(plan->eigvals, R_tot, group, keep, plan->bits);
    else
        alloc_grouped_kernel<64><<<plan->heads, 64 * 8, 0, s>>>(plan->eigvals, R_tot, group, keep, plan->bits);
    return cuda_status(cudaGetLastError());
}

spectra_status launch_effdim(const spectra_plan* plan, double energy, int32_t* d_energy, int32_t* d_gap,
                             cudaStream_t s)
{
    effdim_kernel<<<plan->heads, 32, 0, s>>>(plan->eigvals, plan->head_dim, energy, d_energy, d_gap);
    return cuda_status(cudaGetLastError());
}

spectra_status launch_tc_images(const spectra_plan* plan, cudaStream_t s);   // codec_tc.cu

spectra_status launch_finalize(const spectra_plan* plan, cudaStream_t s)
{
    const PlanView v = make_view(plan);
    uint16_t* co = const_cast<uint16_t*>(v.chan_off);
    float* qs = const_cast<float*>(v.qscale);
    float* rs = const_cast<float*>(v.rscale);
    if (plan->head_dim == 128)
        finalize_kernel<128><<<plan->heads, 128, 0, s>>>(plan->basis, plan->quant, plan->max_rec_bits,
                                                         plan->eigvals, plan->bits, plan->rec_bits, co,
                                                         qs, rs, plan->status);
    else
        finalize_kernel<64><<<plan->heads, 64, 0, s>>>(plan->basis, plan->quant, plan->max_rec_bits,
                                                       plan->eigvals, plan->bits, plan->rec_bits, co,
                                                       qs, rs, plan->status);
    spectra_status st = cuda_status(cudaGetLastError());
    if (st != SPECTRA_OK) return st;
    if (plan->quant == SPECTRA_Q_LLOYD_GAUSS) {
        lm_tables_kernel<<<kMaxBits, 32, 0, s>>>(const_cast<float*>(v.lm_level), const_cast<float*>(v.lm_thresh));
        lm_bucket_kernel<<<1, 256, 0, s>>>(v.lm_thresh, const_cast<float2*>(v.lm_bucket),
                                           const_cast<int32_t*>(v.lm_bucket_bad));
        st = cuda_status(cudaGetLastError());
        if (st != SPECTRA_OK) return st;
    }
    return launch_tc_images(plan, s);
}

}  // namespace spectra
