// api.cu -- the exported C ABI (include/spectra.h): argument validation on
// the host, then launches on the caller's stream.  Nothing here allocates
// device memory or synchronises.
#include "spectra_internal.cuh"

#include <math.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>

using namespace spectra;

namespace spectra {
spectra_status launch_encode_generic(const spectra_plan*, const void*, int, int64_t, int64_t,
                                     uint8_t*, int64_t, float*, int64_t, cudaStream_t, int64_t t0 = 0);
spectra_status launch_gram_tc(const spectra_plan*, const void*, int, int64_t, int64_t, float*, int, cudaStream_t,
                              bool*);
int gram_tc_chunks(int heads, int64_t n_cal);
spectra_status launch_wait_selftest(uint64_t limit_ns, int32_t* out, uint64_t* t_out, cudaStream_t s);
spectra_status launch_qjl_encode(const spectra_plan*, const float*, const void*, int, int64_t, int64_t,
                                 const uint8_t*, int64_t, const float*, int64_t, uint8_t*, int64_t, float*,
                                 int64_t, cudaStream_t);
spectra_status launch_append_small(const spectra_plan*, const void*, int, int64_t, int64_t, uint8_t*, int64_t,
                                   float*, int64_t, int64_t, cudaStream_t);
spectra_status launch_decode_generic(const spectra_plan*, const uint8_t*, int64_t, const float*,
                                     int64_t, int64_t, void*, int, int64_t, cudaStream_t);
spectra_status launch_encode_tc(const spectra_plan*, const void*, int, int64_t, int64_t,
                                uint8_t*, int64_t, float*, int64_t, cudaStream_t, bool*, int64_t g0 = 0);
spectra_status launch_encode_tc_kv(const spectra_plan*, const spectra_plan*, const void*, const void*, int, int64_t,
                                   int64_t, uint8_t*, uint8_t*, int64_t, float*, float*, int64_t, cudaStream_t,
                                   bool*);
spectra_status launch_decode_tc_kv(const spectra_plan*, const spectra_plan*, const uint8_t*, const uint8_t*, int64_t,
                                   const float*, const float*, int64_t, int64_t, void*, void*, int, int64_t,
                                   cudaStream_t, bool*);
spectra_status launch_decode_tc(const spectra_plan*, const uint8_t*, int64_t, const float*,
                                int64_t, int64_t, void*, int, int64_t, cudaStream_t, bool*);
}  // namespace spectra

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kSmallAppend = 8;   // appends of at most this many tokens take the channel-parallel kernel

int elem_size(int dt) { return dt == SPECTRA_BF16 ? 2 : 4; }

bool valid_dtype(int dt) { return dt == SPECTRA_BF16 || dt == SPECTRA_F32; }

spectra_status check_plan(const spectra_plan* p, bool need_tables)
{
    if (!p) return SPECTRA_ERR_INVALID_ARG;
    if (p->heads <= 0 || p->heads > (1 << 20)) return SPECTRA_ERR_INVALID_ARG;
    if (p->head_dim != 64 && p->head_dim != 128) return SPECTRA_ERR_UNSUPPORTED;
    if (p->basis != SPECTRA_BASIS_EIGEN && p->basis != SPECTRA_BASIS_RWHT) return SPECTRA_ERR_INVALID_ARG;
    if (p->quant != SPECTRA_Q_UNIFORM3S && p->quant != SPECTRA_Q_LLOYD_GAUSS) return SPECTRA_ERR_INVALID_ARG;
    if (p->basis == SPECTRA_BASIS_RWHT && p->quant != SPECTRA_Q_LLOYD_GAUSS) return SPECTRA_ERR_UNSUPPORTED;
    if (p->basis == SPECTRA_BASIS_EIGEN && (!p->basis_mat || !p->eigvals)) return SPECTRA_ERR_INVALID_ARG;
    if (p->basis == SPECTRA_BASIS_RWHT && !p->signs) return SPECTRA_ERR_INVALID_ARG;
    if (!p->bits || !p->rec_bits || !p->status) return SPECTRA_ERR_INVALID_ARG;
    if (need_tables) {
        if (!p->derived || (reinterpret_cast<uintptr_t>(p->derived) & 255u)) return SPECTRA_ERR_INVALID_ARG;
        if (p->max_rec_bits < 0 || p->max_rec_bits > 8 * p->head_dim) return SPECTRA_ERR_INVALID_ARG;
    }
    return SPECTRA_OK;
}

spectra_status check_cache(const void* x, int dt, int64_t T, int64_t tstride, int heads, int d)
{
    if (!valid_dtype(dt)) return SPECTRA_ERR_INVALID_ARG;
    if (T < 0) return SPECTRA_ERR_INVALID_ARG;
    if (T == 0) return SPECTRA_OK;
    if (!x || !aligned16(x)) return SPECTRA_ERR_INVALID_ARG;
    if (tstride < int64_t(heads) * d) return SPECTRA_ERR_INVALID_ARG;
    if ((tstride * elem_size(dt)) % 16 != 0) return SPECTRA_ERR_INVALID_ARG;
    return SPECTRA_OK;
}

spectra_status check_streams(const spectra_plan* p, const uint8_t* codes, int64_t sstride, int64_t T,
                             int64_t nstreams)
{
    const int64_t need = stream_bytes(p->max_rec_bits, T);
    if (need == 0) return SPECTRA_OK;
    if (!codes || !aligned16(codes)) return SPECTRA_ERR_INVALID_ARG;
    if (nstreams > 1 && (sstride < need || sstride % 16 != 0)) return SPECTRA_ERR_INVALID_ARG;
    if (nstreams == 1 && sstride != 0 && sstride < need) return SPECTRA_ERR_INVALID_ARG;
    return SPECTRA_OK;
}

// Kernel-family selection for encode, decode and attention.  The process-
// wide value starts from the environment variable SPECTRA_PATH, read once
// (generic = CUDA-core kernels only; tc = tensor-core kernels required, a
// call they do not cover returns SPECTRA_ERR_UNSUPPORTED; unset = tensor
// cores where they apply), and spectra_set_kernel_family changes it.
std::atomic<int> g_family{-1};

int family_from_env()
{
    const char* e = getenv("SPECTRA_PATH");
    if (e && e[0] == 'g') return SPECTRA_KERNELS_CUDA_CORE;
    if (e && e[0] == 't') return SPECTRA_KERNELS_TENSOR_CORE;
    return SPECTRA_KERNELS_AUTO;
}

}  // namespace

spectra_status spectra::attn_validate(const spectra_plan* kplan, const spectra_plan* vplan, const void* q,
                                      int q_dt, int B, int Hq, const uint8_t* k_codes, const uint8_t* v_codes,
                                      int64_t stream_stride_bytes, const float* k_norms, const float* v_norms,
                                      int64_t norms_stride, int64_t ctx, float softmax_scale, const float* out)
{
    spectra_status st;
    if ((st = check_plan(kplan, true))) return st;
    if ((st = check_plan(vplan, true))) return st;
    if (kplan->heads != vplan->heads || kplan->head_dim != vplan->head_dim) return SPECTRA_ERR_INVALID_ARG;
    const int Hkv = kplan->heads;
    if (B <= 0 || Hq <= 0 || Hq % Hkv != 0 || ctx < 0) return SPECTRA_ERR_INVALID_ARG;
    if (!q || !out || !valid_dtype(q_dt) || !isfinite(softmax_scale)) return SPECTRA_ERR_INVALID_ARG;
    if ((st = check_streams(kplan, k_codes, stream_stride_bytes, ctx, int64_t(B) * Hkv))) return st;
    if ((st = check_streams(vplan, v_codes, stream_stride_bytes, ctx, int64_t(B) * Hkv))) return st;
    if (kplan->basis == SPECTRA_BASIS_RWHT && ctx > 0 && (!k_norms || norms_stride < ctx))
        return SPECTRA_ERR_INVALID_ARG;
    if (vplan->basis == SPECTRA_BASIS_RWHT && ctx > 0 && (!v_norms || norms_stride < ctx))
        return SPECTRA_ERR_INVALID_ARG;
    return SPECTRA_OK;
}

int spectra::kernel_family()
{
    int f = g_family.load(std::memory_order_relaxed);
    if (f < 0) {
        int expect = -1;
        g_family.compare_exchange_strong(expect, family_from_env());
        f = g_family.load(std::memory_order_relaxed);
    }
    return f;
}

namespace {

// Gram partials: tcgen05 for bf16 caches with head_dim 128 (unless the
// CUDA-core family is selected), the CUDA-core kernel otherwise.  Returns
// the chunk count through *nch.
spectra_status run_gram(const spectra_plan* plan, const void* x, int dt, int64_t n_cal, int64_t token_stride,
                        float* partials, int* nch, cudaStream_t s)
{
    if (spectra::kernel_family() != SPECTRA_KERNELS_CUDA_CORE) {
        bool done = false;
        *nch = gram_tc_chunks(plan->heads, n_cal);
        spectra_status st = launch_gram_tc(plan, x, dt, n_cal, token_stride, partials, *nch, s, &done);
        if (st || done) return st;
    }
    *nch = gram_chunks(plan->heads, n_cal);
    return launch_gram(plan, x, dt, n_cal, token_stride, partials, *nch, s);
}

}  // namespace

extern "C" {

int spectra_version(void) { return 200; }

spectra_status spectra_set_kernel_family(int family)
{
    if (family != SPECTRA_KERNELS_AUTO && family != SPECTRA_KERNELS_CUDA_CORE &&
        family != SPECTRA_KERNELS_TENSOR_CORE)
        return SPECTRA_ERR_INVALID_ARG;
    g_family.store(family, std::memory_order_relaxed);
    return SPECTRA_OK;
}

int spectra_get_kernel_family(void) { return kernel_family(); }

const char* spectra_status_string(spectra_status st)
{
    switch (st) {
    case SPECTRA_OK: return "ok";
    case SPECTRA_ERR_INVALID_ARG: return "invalid argument";
    case SPECTRA_ERR_UNSUPPORTED: return "unsupported";
    case SPECTRA_ERR_CUDA: return "CUDA error";
    case SPECTRA_ERR_NOT_CONVERGED: return "eigensolve not converged";
    case SPECTRA_ERR_TIMEOUT: return "bounded wait timed out";
    case SPECTRA_ERR_NONFINITE: return "non-finite input";
    case SPECTRA_ERR_BUFFER: return "stream buffer too small";
    }
    return "unknown status";
}

size_t spectra_plan_derived_bytes(int heads, int head_dim)
{
    if (heads <= 0 || (head_dim != 64 && head_dim != 128)) return 0;
    return derived_layout(heads, head_dim).total;
}

size_t spectra_stream_bytes(int32_t rec_bits, int64_t T) { return size_t(stream_bytes(rec_bits, T)); }

size_t spectra_calibrate_workspace_bytes(int heads, int head_dim, int64_t n_cal)
{
    if (heads <= 0 || n_cal <= 0 || (head_dim != 64 && head_dim != 128)) return 0;
    return sizeof(float) * size_t(heads) * gram_chunks(heads, n_cal) * head_dim * head_dim;
}

spectra_status spectra_calibrate(spectra_plan* plan, const void* x, spectra_dtype dt, int64_t n_cal,
                                 int64_t token_stride, int max_sweeps, void* workspace,
                                 size_t workspace_bytes, float* gram_out, spectra_stream_t stream)
{
    spectra_status st = check_plan(plan, false);
    if (st) return st;
    if (plan->basis != SPECTRA_BASIS_EIGEN) return SPECTRA_ERR_INVALID_ARG;
    if (n_cal <= 0 || max_sweeps < 1 || max_sweeps > 100) return SPECTRA_ERR_INVALID_ARG;
    if ((st = check_cache(x, dt, n_cal, token_stride, plan->heads, plan->head_dim))) return st;
    const size_t need = spectra_calibrate_workspace_bytes(plan->heads, plan->head_dim, n_cal);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return SPECTRA_ERR_INVALID_ARG;
    int nch = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = run_gram(plan, x, dt, n_cal, token_stride, static_cast<float*>(workspace), &nch, s))) return st;
    return launch_jacobi(plan, static_cast<float*>(workspace), nch, n_cal, max_sweeps, gram_out, s);
}

spectra_status spectra_plan_finalize(spectra_plan* plan, spectra_stream_t stream)
{
    spectra_status st = check_plan(plan, true);
    if (st) return st;
    return launch_finalize(plan, reinterpret_cast<cudaStream_t>(stream));
}

spectra_status spectra_alloc_bits(spectra_plan* plan, double avg_bits, int fixed_bits,
                                  spectra_stream_t stream)
{
    spectra_status st = check_plan(plan, false);
    if (st) return st;
    if (!plan->derived || (reinterpret_cast<uintptr_t>(plan->derived) & 255u)) return SPECTRA_ERR_INVALID_ARG;
    const int d = plan->head_dim;
    int R;
    if (fixed_bits != 0) {
        if (fixed_bits < 1 || fixed_bits > 8) return SPECTRA_ERR_INVALID_ARG;
        R = fixed_bits * d;
    } else {
        if (!(avg_bits >= 0.0) || !isfinite(avg_bits)) return SPECTRA_ERR_INVALID_ARG;
        if (plan->basis != SPECTRA_BASIS_EIGEN) return SPECTRA_ERR_INVALID_ARG;
        const double r = floor(avg_bits * d + 1e-9);
        R = int(r < 8.0 * d ? r : 8.0 * d);
    }
    plan->max_rec_bits = R;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = launch_alloc(plan, R, fixed_bits, s))) return st;
    return launch_finalize(plan, s);
}

spectra_status spectra_alloc_bits_ex(spectra_plan* plan, double avg_bits, int group, const int32_t* keep,
                                     spectra_stream_t stream)
{
    spectra_status st = check_plan(plan, false);
    if (st) return st;
    if (!plan->derived || (reinterpret_cast<uintptr_t>(plan->derived) & 255u)) return SPECTRA_ERR_INVALID_ARG;
    if (plan->basis != SPECTRA_BASIS_EIGEN) return SPECTRA_ERR_INVALID_ARG;
    const int d = plan->head_dim;
    if (group < 1 || group > d || (group & (group - 1)) || d % group) return SPECTRA_ERR_INVALID_ARG;
    if (!(avg_bits >= 0.0) || !isfinite(avg_bits)) return SPECTRA_ERR_INVALID_ARG;
    const double r = floor(avg_bits * d + 1e-9);
    const int R = int(r < 8.0 * d ? r : 8.0 * d);
    plan->max_rec_bits = (R / group) * group;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = launch_alloc_grouped(plan, R, group, keep, s))) return st;
    return launch_finalize(plan, s);
}

spectra_status spectra_effective_dim(const spectra_plan* plan, double energy, int32_t* d_energy, int32_t* d_gap,
                                     spectra_stream_t stream)
{
    spectra_status st = check_plan(plan, false);
    if (st) return st;
    if (plan->basis != SPECTRA_BASIS_EIGEN || !d_energy || !d_gap) return SPECTRA_ERR_INVALID_ARG;
    if (!(energy > 0.0 && energy <= 1.0)) return SPECTRA_ERR_INVALID_ARG;
    return launch_effdim(plan, energy, d_energy, d_gap, reinterpret_cast<cudaStream_t>(stream));
}

spectra_status spectra_calibrate_plain(spectra_plan* plan, const void* x, spectra_dtype dt, int64_t n_cal,
                                       int64_t token_stride, void* workspace, size_t workspace_bytes,
                                       spectra_stream_t stream)
{
    spectra_status st = check_plan(plan, false);
    if (st) return st;
    if (plan->basis != SPECTRA_BASIS_EIGEN) return SPECTRA_ERR_INVALID_ARG;
    if (n_cal <= 0) return SPECTRA_ERR_INVALID_ARG;
    if ((st = check_cache(x, dt, n_cal, token_stride, plan->heads, plan->head_dim))) return st;
    const size_t need = spectra_calibrate_workspace_bytes(plan->heads, plan->head_dim, n_cal);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return SPECTRA_ERR_INVALID_ARG;
    int nch = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = run_gram(plan, x, dt, n_cal, token_stride, static_cast<float*>(workspace), &nch, s))) return st;
    return launch_plain_calibrate(plan, static_cast<float*>(workspace), nch, n_cal, s);
}

spectra_status spectra_encode(const spectra_plan* plan, const void* x, spectra_dtype dt, int64_t T,
                              int64_t token_stride, uint8_t* codes, int64_t stream_stride_bytes,
                              float* norms, int64_t norms_stride, spectra_stream_t stream)
{
    spectra_status st = check_plan(plan, true);
    if (st) return st;
    if ((st = check_cache(x, dt, T, token_stride, plan->heads, plan->head_dim))) return st;
    if ((st = check_streams(plan, codes, stream_stride_bytes, T, plan->heads))) return st;
    if (plan->basis == SPECTRA_BASIS_RWHT && T > 0) {
        if (!norms || (plan->heads > 1 && norms_stride < T)) return SPECTRA_ERR_INVALID_ARG;
    }
    if (T == 0 || plan->max_rec_bits == 0) {
        if (plan->basis != SPECTRA_BASIS_RWHT || T == 0) return SPECTRA_OK;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int fam = kernel_family();
    if (fam != SPECTRA_KERNELS_CUDA_CORE) {
        bool done = false;
        st = launch_encode_tc(plan, x, dt, T, token_stride, codes, stream_stride_bytes, norms,
                              norms_stride, s, &done);
        if (st || done) return st;
        if (fam == SPECTRA_KERNELS_TENSOR_CORE) return SPECTRA_ERR_UNSUPPORTED;
    }
    return launch_encode_generic(plan, x, dt, T, token_stride, codes, stream_stride_bytes, norms,
                                 norms_stride, s);
}

spectra_status spectra_encode_kv(const spectra_plan* kplan, const spectra_plan* vplan, const void* k, const void* v,
                                 spectra_dtype dt, int64_t T, int64_t token_stride, uint8_t* k_codes,
                                 uint8_t* v_codes, int64_t stream_stride_bytes, float* k_norms, float* v_norms,
                                 int64_t norms_stride, spectra_stream_t stream)
{
    // every argument of both halves is checked before anything is launched
    const spectra_plan* plans[2] = {kplan, vplan};
    const void* xs[2] = {k, v};
    uint8_t* cs[2] = {k_codes, v_codes};
    float* ns[2] = {k_norms, v_norms};
    spectra_status st;
    for (int i = 0; i < 2; ++i) {
        if ((st = check_plan(plans[i], true))) return st;
        if ((st = check_cache(xs[i], dt, T, token_stride, plans[i]->heads, plans[i]->head_dim))) return st;
        if ((st = check_streams(plans[i], cs[i], stream_stride_bytes, T, plans[i]->heads))) return st;
        if (plans[i]->basis == SPECTRA_BASIS_RWHT && T > 0) {
            if (!ns[i] || (plans[i]->heads > 1 && norms_stride < T)) return SPECTRA_ERR_INVALID_ARG;
        }
    }
    if (kplan->heads != vplan->heads || kplan->head_dim != vplan->head_dim) return SPECTRA_ERR_INVALID_ARG;
    if (T == 0) return SPECTRA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (kernel_family() != SPECTRA_KERNELS_CUDA_CORE) {
        bool done = false;
        st = launch_encode_tc_kv(kplan, vplan, k, v, dt, T, token_stride, k_codes, v_codes, stream_stride_bytes,
                                 k_norms, v_norms, norms_stride, s, &done);
        if (st || done) return st;
    }
    // not one launch: the two encodes in turn
    if ((st = spectra_encode(kplan, k, dt, T, token_stride, k_codes, stream_stride_bytes, k_norms, norms_stride,
                             stream)))
        return st;
    return spectra_encode(vplan, v, dt, T, token_stride, v_codes, stream_stride_bytes, v_norms, norms_stride,
                          stream);
}

spectra_status spectra_append(const spectra_plan* plan, const void* x, spectra_dtype dt, int64_t n,
                              int64_t token_stride, int64_t t0, uint8_t* codes, int64_t stream_stride_bytes,
                              float* norms, int64_t norms_stride, spectra_stream_t stream)
{
    spectra_status st = check_plan(plan, true);
    if (st) return st;
    if (t0 < 0) return SPECTRA_ERR_INVALID_ARG;
    if ((st = check_cache(x, dt, n, token_stride, plan->heads, plan->head_dim))) return st;
    if ((st = check_streams(plan, codes, stream_stride_bytes, t0 + n, plan->heads))) return st;
    if (plan->basis == SPECTRA_BASIS_RWHT && n > 0) {
        if (!norms || (plan->heads > 1 && norms_stride < t0 + n)) return SPECTRA_ERR_INVALID_ARG;
    }
    if (n == 0 || plan->max_rec_bits == 0) {
        if (plan->basis != SPECTRA_BASIS_RWHT || n == 0) return SPECTRA_OK;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // tokens up to the next 128-token boundary: read-modify-write of the
    // partly filled group on CUDA cores; the rest is an ordinary encode at a
    // tile-aligned stream position (16 R bytes per 128 tokens)
    const int64_t t_al = std::min<int64_t>(t0 + n, (t0 + 127) / 128 * 128);
    const int fam = kernel_family();
    if (t_al > t0 || fam == SPECTRA_KERNELS_CUDA_CORE) {
        const int64_t nh = fam == SPECTRA_KERNELS_CUDA_CORE ? n : t_al - t0;
        // a few tokens (decode steps): channel-parallel, token by token
        st = nh <= kSmallAppend
                 ? launch_append_small(plan, x, dt, nh, token_stride, codes, stream_stride_bytes, norms,
                                       norms_stride, t0, s)
                 : launch_encode_generic(plan, x, dt, nh, token_stride, codes, stream_stride_bytes, norms,
                                         norms_stride, s, t0);
        if (st) return st;
        if (nh == n) return SPECTRA_OK;
    }
    const int64_t rest = t0 + n - t_al;
    const size_t esz = dt == SPECTRA_BF16 ? 2 : 4;
    const void* xr = static_cast<const uint8_t*>(x) + size_t(t_al - t0) * size_t(token_stride) * esz;
    bool done = false;
    if ((st = launch_encode_tc(plan, xr, dt, rest, token_stride, codes, stream_stride_bytes, norms, norms_stride, s,
                               &done, t_al / 32)))
        return st;
    if (done) return SPECTRA_OK;
    if (fam == SPECTRA_KERNELS_TENSOR_CORE) return SPECTRA_ERR_UNSUPPORTED;
    return launch_encode_generic(plan, xr, dt, rest, token_stride, codes, stream_stride_bytes, norms, norms_stride,
                                 s, t_al);
}

spectra_status spectra_decode(const spectra_plan* plan, const uint8_t* codes, int64_t stream_stride_bytes,
                              const float* norms, int64_t norms_stride, int64_t T, void* x_out,
                              spectra_dtype out_dt, int64_t token_stride, spectra_stream_t stream)
{
    spectra_status st = check_plan(plan, true);
    if (st) return st;
    if ((st = check_cache(x_out, out_dt, T, token_stride, plan->heads, plan->head_dim))) return st;
    if ((st = check_streams(plan, codes, stream_stride_bytes, T, plan->heads))) return st;
    if (plan->basis == SPECTRA_BASIS_RWHT && T > 0) {
        if (!norms || (plan->heads > 1 && norms_stride < T)) return SPECTRA_ERR_INVALID_ARG;
    }
    if (T == 0) return SPECTRA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int fam = kernel_family();
    if (fam != SPECTRA_KERNELS_CUDA_CORE) {
        bool done = false;
        st = launch_decode_tc(plan, codes, stream_stride_bytes, norms, norms_stride, T, x_out, out_dt,
                              token_stride, s, &done);
        if (st || done) return st;
        if (fam == SPECTRA_KERNELS_TENSOR_CORE) return SPECTRA_ERR_UNSUPPORTED;
    }
    return launch_decode_generic(plan, codes, stream_stride_bytes, norms, norms_stride, T, x_out,
                                 out_dt, token_stride, s);
}

spectra_status spectra_decode_kv(const spectra_plan* kplan, const spectra_plan* vplan, const uint8_t* k_codes,
                                 const uint8_t* v_codes, int64_t stream_stride_bytes, const float* k_norms,
                                 const float* v_norms, int64_t norms_stride, int64_t T, void* k_out, void* v_out,
                                 spectra_dtype out_dt, int64_t token_stride, spectra_stream_t stream)
{
    const spectra_plan* plans[2] = {kplan, vplan};
    const uint8_t* cs[2] = {k_codes, v_codes};
    const float* ns[2] = {k_norms, v_norms};
    void* outs[2] = {k_out, v_out};
    spectra_status st;
    for (int i = 0; i < 2; ++i) {
        if ((st = check_plan(plans[i], true))) return st;
        if ((st = check_cache(outs[i], out_dt, T, token_stride, plans[i]->heads, plans[i]->head_dim))) return st;
        if ((st = check_streams(plans[i], cs[i], stream_stride_bytes, T, plans[i]->heads))) return st;
        if (plans[i]->basis == SPECTRA_BASIS_RWHT && T > 0) {
            if (!ns[i] || (plans[i]->heads > 1 && norms_stride < T)) return SPECTRA_ERR_INVALID_ARG;
        }
    }
    if (kplan->heads != vplan->heads || kplan->head_dim != vplan->head_dim) return SPECTRA_ERR_INVALID_ARG;
    if (T == 0) return SPECTRA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (kernel_family() != SPECTRA_KERNELS_CUDA_CORE) {
        bool done = false;
        st = launch_decode_tc_kv(kplan, vplan, k_codes, v_codes, stream_stride_bytes, k_norms, v_norms,
                                 norms_stride, T, k_out, v_out, out_dt, token_stride, s, &done);
        if (st || done) return st;
    }
    if ((st = spectra_decode(kplan, k_codes, stream_stride_bytes, k_norms, norms_stride, T, k_out, out_dt,
                             token_stride, stream)))
        return st;
    return spectra_decode(vplan, v_codes, stream_stride_bytes, v_norms, norms_stride, T, v_out, out_dt,
                          token_stride, stream);
}

size_t spectra_attn_workspace_bytes(int B, int Hq, int head_dim, int64_t ctx)
{
    if (B <= 0 || Hq <= 0 || ctx < 0 || (head_dim != 64 && head_dim != 128)) return 0;
    return attn_workspace_bytes(B, Hq, head_dim, ctx);
}

spectra_status spectra_attn_decode(const spectra_plan* kplan, const spectra_plan* vplan, const void* q,
                                   spectra_dtype q_dt, int B, int Hq, const uint8_t* k_codes,
                                   const uint8_t* v_codes, int64_t stream_stride_bytes,
                                   const float* k_norms, const float* v_norms, int64_t norms_stride,
                                   int64_t ctx, float softmax_scale, float* out, void* workspace,
                                   size_t workspace_bytes, spectra_stream_t stream)
{
    spectra_status st = attn_validate(kplan, vplan, q, q_dt, B, Hq, k_codes, v_codes, stream_stride_bytes,
                                      k_norms, v_norms, norms_stride, ctx, softmax_scale, out);
    if (st) return st;
    const int d = kplan->head_dim;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (ctx == 0)
        return cuda_status(cudaMemsetAsync(out, 0, sizeof(float) * size_t(B) * Hq * d, s));
    const size_t need = attn_workspace_bytes(B, Hq, d, ctx);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return SPECTRA_ERR_INVALID_ARG;
    return launch_attn(kplan, vplan, q, q_dt, B, Hq, k_codes, v_codes, stream_stride_bytes, k_norms,
                       v_norms, norms_stride, ctx, softmax_scale, out, workspace, workspace_bytes, s);
}

spectra_status spectra_attn_decode_window(const spectra_plan* kplan, const spectra_plan* vplan, const void* q,
                                          spectra_dtype q_dt, int B, int Hq, const uint8_t* k_codes,
                                          const uint8_t* v_codes, int64_t stream_stride_bytes,
                                          const float* k_norms, const float* v_norms, int64_t norms_stride,
                                          int64_t ctx, const void* k_win, const void* v_win, spectra_dtype win_dt,
                                          int64_t win_len, int64_t win_token_stride, float softmax_scale,
                                          float* out, void* workspace, size_t workspace_bytes,
                                          spectra_stream_t stream)
{
    spectra_status st = attn_validate(kplan, vplan, q, q_dt, B, Hq, k_codes, v_codes, stream_stride_bytes,
                                      k_norms, v_norms, norms_stride, ctx, softmax_scale, out);
    if (st) return st;
    const int d = kplan->head_dim;
    if (win_len < 0 || win_len > SPECTRA_ATTN_MAX_WINDOW) return SPECTRA_ERR_INVALID_ARG;
    if (win_len > 0) {
        if (!valid_dtype(win_dt) || !k_win || !v_win) return SPECTRA_ERR_INVALID_ARG;
        if (win_token_stride < int64_t(kplan->heads) * d) return SPECTRA_ERR_INVALID_ARG;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (ctx == 0 && win_len == 0)
        return cuda_status(cudaMemsetAsync(out, 0, sizeof(float) * size_t(B) * Hq * d, s));
    const size_t need = attn_workspace_bytes(B, Hq, d, ctx);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return SPECTRA_ERR_INVALID_ARG;
    AttnWindow w{k_win, v_win, int(win_dt), win_len, win_token_stride};
    return launch_attn(kplan, vplan, q, q_dt, B, Hq, k_codes, v_codes, stream_stride_bytes, k_norms, v_norms,
                       norms_stride, ctx, softmax_scale, out, workspace, workspace_bytes, s, &w);
}

spectra_status spectra_qjl_encode(const spectra_plan* plan, const float* sketch, const void* x, spectra_dtype dt,
                                  int64_t T, int64_t token_stride, const uint8_t* codes,
                                  int64_t stream_stride_bytes, const float* norms, int64_t norms_stride,
                                  uint8_t* qjl_bits, int64_t qjl_stride_bytes, float* qjl_norms,
                                  int64_t qjl_norms_stride, spectra_stream_t stream)
{
    spectra_status st = check_plan(plan, true);
    if (st) return st;
    if ((st = check_cache(x, dt, T, token_stride, plan->heads, plan->head_dim))) return st;
    if ((st = check_streams(plan, codes, stream_stride_bytes, T, plan->heads))) return st;
    if (T == 0) return SPECTRA_OK;
    if (!sketch || !qjl_bits || !qjl_norms || !aligned16(qjl_bits)) return SPECTRA_ERR_INVALID_ARG;
    const int64_t need = stream_bytes(plan->head_dim, T);
    if (plan->heads > 1 && (qjl_stride_bytes < need || qjl_stride_bytes % 16 != 0)) return SPECTRA_ERR_INVALID_ARG;
    if (plan->heads > 1 && qjl_norms_stride < T) return SPECTRA_ERR_INVALID_ARG;
    if (plan->basis == SPECTRA_BASIS_RWHT && (!norms || (plan->heads > 1 && norms_stride < T)))
        return SPECTRA_ERR_INVALID_ARG;
    return launch_qjl_encode(plan, sketch, x, dt, T, token_stride, codes, stream_stride_bytes, norms, norms_stride,
                             qjl_bits, qjl_stride_bytes, qjl_norms, qjl_norms_stride,
                             reinterpret_cast<cudaStream_t>(stream));
}

spectra_status spectra_attn_decode_qjl(const spectra_plan* kplan, const spectra_plan* vplan, const void* q,
                                       spectra_dtype q_dt, int B, int Hq, const uint8_t* k_codes,
                                       const uint8_t* v_codes, int64_t stream_stride_bytes, const float* k_norms,
                                       const float* v_norms, int64_t norms_stride, int64_t ctx,
                                       const float* sketch, const uint8_t* k_qjl_bits, int64_t qjl_stride_bytes,
                                       const float* k_qjl_norms, int64_t qjl_norms_stride, float softmax_scale,
                                       float* out, void* workspace, size_t workspace_bytes, spectra_stream_t stream)
{
    spectra_status st = attn_validate(kplan, vplan, q, q_dt, B, Hq, k_codes, v_codes, stream_stride_bytes,
                                      k_norms, v_norms, norms_stride, ctx, softmax_scale, out);
    if (st) return st;
    const int d = kplan->head_dim;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (ctx == 0) return cuda_status(cudaMemsetAsync(out, 0, sizeof(float) * size_t(B) * Hq * d, s));
    if (!sketch || !k_qjl_bits || !k_qjl_norms || !aligned16(k_qjl_bits)) return SPECTRA_ERR_INVALID_ARG;
    if (qjl_stride_bytes < stream_bytes(d, ctx) || qjl_stride_bytes % 16 != 0 || qjl_norms_stride < ctx)
        return SPECTRA_ERR_INVALID_ARG;
    const size_t need = attn_workspace_bytes(B, Hq, d, ctx);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return SPECTRA_ERR_INVALID_ARG;
    AttnQjl qj{sketch, k_qjl_bits, qjl_stride_bytes, k_qjl_norms, qjl_norms_stride};
    return launch_attn(kplan, vplan, q, q_dt, B, Hq, k_codes, v_codes, stream_stride_bytes, k_norms, v_norms,
                       norms_stride, ctx, softmax_scale, out, workspace, workspace_bytes, s, nullptr, &qj);
}

spectra_status spectra_selftest_wait(uint64_t limit_ns, int32_t* status, uint64_t* elapsed_ns,
                                    spectra_stream_t stream)
{
    if (!status || !elapsed_ns || limit_ns == 0 || limit_ns > 10000000000ull) return SPECTRA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(elapsed_ns) & 7u) || (reinterpret_cast<uintptr_t>(status) & 3u))
        return SPECTRA_ERR_INVALID_ARG;
    return launch_wait_selftest(limit_ns, status, elapsed_ns, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
