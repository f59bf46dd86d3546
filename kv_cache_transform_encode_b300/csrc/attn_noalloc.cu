// attn_noalloc.cu -- spectra_attn_decode without a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the point where they run a
// decode step: code running inside an allocator or memory-pool callback
// (calling cudaMalloc there would re-enter the allocator), a host whose
// device memory is wholly owned by another framework's pool, or a deployment
// that forbids any device allocation after start-up.  For them this entry
// point takes its split-context scratch from one file-scope device array that
// is part of the library image, so the call itself allocates nothing.
//
// The first call on each device looks up the array's device address
// (cudaGetSymbolAddress, with that device current) and caches it.  CUDA may
// load this file's module lazily, so that first lookup can be the moment
// the array is created on the device: make the first call on each device at
// start-up, outside any allocator callback and before any stream capture
// (a call that is refused for its size still does the lookup).  Every later
// call allocates nothing.  The cached address assumes the device's context
// lives as long as the process (no cudaDeviceReset in between).
//
// The array (SPECTRA_ATTN_NOALLOC_SCRATCH_BYTES) is created with the
// library's module on every GPU that loads it and stays resident until the
// process exits.  All calls on a device share it: two calls whose kernels
// overlap on the GPU (different streams without ordering between them) race
// on it and give wrong results.  Nothing in it needs clearing between calls:
// every byte a call's kernels read from it was written earlier by the same
// call.
#include "spectra_internal.cuh"

#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_attn_scratch[SPECTRA_ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device.  In host code the
// symbol names a host-side stand-in, never the device buffer, so the address
// is looked up once per device (with that device current) and cached.
spectra_status scratch_address(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPECTRA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess || !p) return SPECTRA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SPECTRA_OK;
}

}  // namespace

extern "C" spectra_status spectra_attn_decode_noalloc(
    const spectra_plan* kplan, const spectra_plan* vplan, const void* q, spectra_dtype q_dt, int B,
    int Hq, const uint8_t* k_codes, const uint8_t* v_codes, int64_t stream_stride_bytes,
    const float* k_norms, const float* v_norms, int64_t norms_stride, int64_t ctx,
    float softmax_scale, float* out, spectra_stream_t stream)
{
    // the same argument checks, in the same order, as spectra_attn_decode
    spectra_status st = spectra::attn_validate(kplan, vplan, q, q_dt, B, Hq, k_codes, v_codes,
                                               stream_stride_bytes, k_norms, v_norms, norms_stride, ctx,
                                               softmax_scale, out);
    if (st != SPECTRA_OK) return st;
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != SPECTRA_OK) return st;
    if (ctx > 0) {   // an empty context only zeroes `out` and needs no scratch
        const size_t need = spectra_attn_workspace_bytes(B, Hq, kplan->head_dim, ctx);
        if (need > size_t(SPECTRA_ATTN_NOALLOC_SCRATCH_BYTES)) return SPECTRA_ERR_UNSUPPORTED;
    }
    return spectra_attn_decode(kplan, vplan, q, q_dt, B, Hq, k_codes, v_codes, stream_stride_bytes,
                               k_norms, v_norms, norms_stride, ctx, softmax_scale, out, scratch,
                               size_t(SPECTRA_ATTN_NOALLOC_SCRATCH_BYTES), stream);
}
