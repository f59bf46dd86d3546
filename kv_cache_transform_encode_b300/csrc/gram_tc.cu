// gram_tc.cu -- per-head Gram matrix on the tensor cores (tcgen05), bf16
// caches with head_dim 128.
//
// "Sintesi Tecnica: SPECTRA", "Metodologia" item 3: the transform is
// weighted by the activation second moment G = E[h^T h]; "Technisch
// Overzicht ...", "Experimentele Opstelling": a per-head eigenbasis
// calibrated on representative tokens.
//
// G_h = sum_t x_t x_t^T is the product X^T X of the calibration tokens.  One
// CTA per (token chunk, head) accumulates its chunk's part in tensor memory:
// per tile of 128 tokens, the four warps write X^T -- row = channel, K =
// token -- into shared memory in the K-major 128-byte-swizzle layout (two
// 64-token blocks), and one thread issues eight tcgen05.mma (M = N = 128,
// K = 16) with that one tile as both operands: D[i][j] += sum_t X^T[i][t]
// X^T[j][t].  bf16 products are exact; the accumulator is fp32.  Two tile
// buffers: the writes of tile k + 1 overlap the MMAs of tile k, and a
// buffer is rewritten only after the commit of the MMAs that read it.  At the
// end each warp reads its 32 accumulator lanes (channels) with tcgen05.ld
// and writes the chunk partial, in the layout the Jacobi kernels sum.
#include "spectra_internal.cuh"
#include "tc_common.cuh"

namespace spectra {

namespace {

using namespace tc;

constexpr int D = 128;
constexpr int TILE = 128;                      // tokens per tile (MMA K per tile)
constexpr uint32_t KBLK = 128 * 128;           // one 64-token block: 128 rows x 128 bytes
constexpr uint32_t OPND = 2 * KBLK;            // one tile: 32 KB
constexpr uint32_t IDESC = idesc_bf16_f32(128, 128);
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads, 1)
gram_tc_kernel(const uint16_t* __restrict__ x, int64_t n_cal, int64_t token_stride, int heads, int64_t chunk_len,
               float* __restrict__ partials)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* tiles = smem;                                      // [2][OPND]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * OPND);
    uint64_t* done = bars;                                      // [2] MMAs of buffer b complete
    uint64_t* fin = bars + 2;                                   // every MMA complete
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 4);
    volatile int* drain_flag = abort_flag + 1;

    const int chunk = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t t_begin = int64_t(chunk) * chunk_len;
    const int64_t t_end = min(n_cal, t_begin + chunk_len);
    const int ntiles = int((t_end - t_begin + TILE - 1) / TILE);

    if (tid == 0) {
        mbar_init(&done[0], 1);
        mbar_init(&done[1], 1);
        mbar_init(fin, 1);
        *abort_flag = 0;
        *drain_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    // thread = (token pair p, channel half hc): tokens 2p, 2p + 1, channels 64 hc ..
    const int p = tid & 63, hc = tid >> 6;
    bool ok = true;
    for (int k = 0; k < ntiles && ok; ++k) {
        const int buf = k & 1;
        // the MMAs that last read this buffer (tile k - 2) are complete
        if (k >= 2) ok = mbar_wait(&done[buf], uint32_t((k - 2) >> 1) & 1u, abort_flag, kWaitNs);
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        const int64_t t0 = t_begin + int64_t(k) * TILE;
        uint8_t* tile = tiles + buf * OPND;
        uint4 a[8], b[8];
        const int64_t ta = t0 + 2 * p, tb = ta + 1;
        const uint4* ra = reinterpret_cast<const uint4*>(x + ta * token_stride + int64_t(h) * D + 64 * hc);
        const uint4* rb = reinterpret_cast<const uint4*>(x + tb * token_stride + int64_t(h) * D + 64 * hc);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            a[q] = ta < t_end ? ra[q] : make_uint4(0u, 0u, 0u, 0u);
            b[q] = tb < t_end ? rb[q] : make_uint4(0u, 0u, 0u, 0u);
        }
        // X^T[i][t] at block (t / 64), row i, byte 2 (t mod 64): tokens 2p, 2p + 1
        // of channel i are one 32-bit word
        const uint32_t kb = uint32_t((2 * p) >> 6), kbytes = uint32_t((2 * p) & 63) * 2;
        const uint32_t* aw = reinterpret_cast<const uint32_t*>(a);
        const uint32_t* bw = reinterpret_cast<const uint32_t*>(b);
#pragma unroll
        for (int w = 0; w < 32; ++w) {
            const int i = 64 * hc + 2 * w;
            const uint32_t lo = __byte_perm(aw[w], bw[w], 0x5410);   // channel i: (t, t + 1)
            const uint32_t hi = __byte_perm(aw[w], bw[w], 0x7632);   // channel i + 1
            *reinterpret_cast<uint32_t*>(tile + kb * KBLK + sw128_offset(uint32_t(i), kbytes)) = lo;
            *reinterpret_cast<uint32_t*>(tile + kb * KBLK + sw128_offset(uint32_t(i + 1), kbytes)) = hi;
        }
        fence_proxy_async_smem();          // generic-proxy writes -> the tensor cores' reads
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t ta_s = smem_u32(tile);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t koff = (kk >> 2) * KBLK + (kk & 3) * 32;
                const uint64_t desc = sdesc_sw128(ta_s + koff);
                mma_bf16_ss(tmem, desc, desc, IDESC, (k | kk) ? 1u : 0u);
            }
            mma_commit(&done[buf]);
        }
    }
    // every issued MMA complete (bounded), then the accumulator out
    if (tid == 0) {
        if (ntiles > 0) mma_commit(fin);
        else mbar_arrive(fin);
    }
    const bool fin_ok = mbar_wait(fin, 0u, drain_flag, kWaitNs);
    tc_fence_after();
    float* out = partials + (size_t(h) * gridDim.x + chunk) * D * D;
    const int i = 32 * warp + lane;
    const bool good = ok && fin_ok && ntiles > 0;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem + (uint32_t(32 * warp) << 16) + uint32_t(32 * cb), r);
        tmem_ld_wait();
        float4* o4 = reinterpret_cast<float4*>(out + size_t(i) * D + 32 * cb);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float4 v;
            v.x = good ? __uint_as_float(r[4 * e]) : (ntiles > 0 ? NAN : 0.f);
            v.y = good ? __uint_as_float(r[4 * e + 1]) : (ntiles > 0 ? NAN : 0.f);
            v.z = good ? __uint_as_float(r[4 * e + 2]) : (ntiles > 0 ? NAN : 0.f);
            v.w = good ? __uint_as_float(r[4 * e + 3]) : (ntiles > 0 ? NAN : 0.f);
            o4[e] = v;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// Self-test of the bounded waits every kernel of the library uses: an
// mbarrier that nothing ever arrives on.  Thread 0 spins on it (the single-
// thread form), warp 1 waits on it (the suspending form), under one shared
// abort flag: the first waiter to pass `limit_ns` raises the flag and every
// other one gives up on it.  out[0] = -SPECTRA_ERR_TIMEOUT when thread 0 gave
// up (0 otherwise), out[1] = how many of the 33 waiters gave up; t_out =
// thread 0's wait in ns.
__global__ void wait_selftest_kernel(uint64_t limit_ns, int32_t* out, uint64_t* t_out)
{
    __shared__ uint64_t bar;
    __shared__ int abort_s;
    __shared__ int gave_up;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_s = 0;
        gave_up = 0;
        fence_mbar_init();
    }
    __syncthreads();
    volatile int* abort_flag = &abort_s;
    const int warp = threadIdx.x >> 5;
    bool ok = true;
    uint64_t t0 = 0, t1 = 0;
    if (threadIdx.x == 0) {
        t0 = globaltimer_ns();
        ok = mbar_spin(&bar, 0u, abort_flag, limit_ns);
        t1 = globaltimer_ns();
    } else if (warp == 1) {
        ok = mbar_wait(&bar, 0u, abort_flag, limit_ns);
    }
    if ((threadIdx.x == 0 || warp == 1) && !ok) atomicAdd(&gave_up, 1);
    __syncthreads();
    if (threadIdx.x == 0) {
        out[0] = ok ? 0 : -SPECTRA_ERR_TIMEOUT;
        out[1] = gave_up;
        *t_out = t1 - t0;
    }
}

}  // namespace

// Chunks of whole 128-token tiles, at most gram_chunks(heads, n_cal) of them
// (the workspace bound).
int gram_tc_chunks(int heads, int64_t n_cal)
{
    const int64_t want = (2 * 148 + heads - 1) / heads;
    const int64_t maxc = (n_cal + TILE - 1) / TILE;
    const int64_t c = want < maxc ? want : maxc;
    return int(c < 1 ? 1 : c);
}

spectra_status launch_wait_selftest(uint64_t limit_ns, int32_t* out, uint64_t* t_out, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 64, 0, s>>>(limit_ns, out, t_out);
    return cuda_status(cudaGetLastError());
}

spectra_status launch_gram_tc(const spectra_plan* plan, const void* x, int dt, int64_t n_cal, int64_t token_stride,
                              float* partials, int nchunks, cudaStream_t s, bool* done)
{
    *done = false;
    if (dt != SPECTRA_BF16 || plan->head_dim != D) return SPECTRA_OK;
    // whole tiles per chunk except the last
    const int64_t tiles = (n_cal + TILE - 1) / TILE;
    const int64_t chunk_len = (tiles + nchunks - 1) / nchunks * TILE;
    const size_t sm = 2 * OPND + 64 + 1024;
    if (spectra_status st = set_smem(gram_tc_kernel, sm)) return st;
    dim3 grid(nchunks, plan->heads);
    gram_tc_kernel<<<grid, kThreads, sm, s>>>(static_cast<const uint16_t*>(x), n_cal, token_stride, plan->heads,
                                             chunk_len, partials);
    *done = true;
    return cuda_status(cudaGetLastError());
}

}  // namespace spectra
