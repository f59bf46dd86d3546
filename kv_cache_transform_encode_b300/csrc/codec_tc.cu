// codec_tc.cu -- tensor-core (tcgen05) encode and decode for bf16 caches
// with head_dim 128, both bases, both quantizers.
//
// "Sintesi Tecnica: SPECTRA", "La Pipeline di SPECTRA" phase 3: tokens are
// projected into the latent basis, quantized per token and appended to the
// latent cache; keys and values are rebuilt on the fly.  "Technisch
// Overzicht ...", "Experimentele Opstelling": randomized Walsh-Hadamard
// rotation with a Lloyd-Max codebook.
//
// Both kernels are persistent (one CTA per SM) and warp-specialised; the
// work list is the (head, 128-token tile) pairs in head-major order, split
// into one contiguous range per CTA, so a CTA reloads its head's operand
// image at most a few times.
//
// Encode, per tile: TMA brings x [128 tokens][128] bf16 into shared memory
// (128-byte swizzle); one thread issues tcgen05.mma with A = the plan's basis
// image (M = 128 channels, K = 128) and B = x (N = 128 tokens) into a TMEM
// accumulator (double-buffered), so TMEM lane = channel, column = token.
// The basis is fp32; it enters the bf16 tensor cores as three bf16 terms
// (hi + mid + lo, 24 significand bits in all) accumulated into the same fp32
// accumulator, so y carries fp32-grade accuracy, which the code-parity band
// (3e-5 sigma) needs.  RWHT uses one exact +-1 term.  Eight epilogue warps
// (lane = channel, two 32-token groups each) quantize without branches (two
// FMAs per value for the uniform quantizer, all channel constants in
// registers), gather each token's code into a byte, and turn the 32 codes
// of a group into the channel's bit-plane words with four 8x8 bit
// transposes -- exactly the stream layout.
//
// Decode, per tile: a bulk copy brings the tile's code words into shared
// memory; eight unpack warps (lane = a pair of channels, one 32-token group
// each) invert the bit transposes, dequantize and write the A operand
// (bf16; for the uniform quantizer the exact odd integer 2 code + 1 - 2^b,
// the scale Delta/2 being folded into the image) in the swizzled layout;
// tcgen05.mma forms x = A * image^T (M = 128 tokens; image = basis * scale
// as bf16 hi + lo; Lloyd-Max levels enter as bf16 hi + lo too); four
// epilogue warps (lane = token) convert the accumulator to the output dtype
// in a swizzled staging buffer that a TMA store writes out (rows past T are
// clipped by the TMA unit).
#include "spectra_internal.cuh"
#include "tc_common.cuh"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <mutex>

namespace spectra {

namespace {

using namespace tc;

constexpr int D = 128;
constexpr int TILE = 128;                 // tokens per tile (MMA M)
constexpr uint32_t OPND = TILE * D * 2;   // one bf16 operand tile: 32 KB
constexpr uint32_t KBLK = TILE * 128;     // one 64-element K block: 16 KB
constexpr uint32_t IDESC = idesc_bf16_f32(128, 128);
constexpr uint64_t kWaitNs = 2000000000ull;

// ------------------------------------------------------------------ helpers
// Work schedule of a persistent CTA over the (head, 128-token tile) items.
// Interleaved (the grid a multiple of the head count): CTA c keeps head
// c mod H and walks tiles j, j + cph, j + 2 cph, ... (j = c / H, cph = CTAs
// per head), so the CTAs of all heads move through the same token range
// together -- each [token][heads][d] row of the cache is read (or written)
// whole at about the same time, which keeps DRAM pages open -- and every
// CTA loads its operand image once.  Contiguous (otherwise): one range of
// the head-major item list per CTA.
// Loops walk the items with first() / next(), which divide only once.
struct Item {
    int h, tile;
};

struct Sched {
    int interleaved, head, j, cph, begin, n, tiles;
    __device__ __forceinline__ int head_of(int k) const { return interleaved ? head : (begin + k) / tiles; }
    __device__ __forceinline__ Item first() const
    {
        return interleaved ? Item{head, j} : Item{begin / tiles, begin % tiles};
    }
    __device__ __forceinline__ void next(Item& it) const
    {
        if (interleaved) {
            it.tile += cph;
        } else if (++it.tile == tiles) {
            it.tile = 0;
            ++it.h;
        }
    }
};

__device__ __forceinline__ Sched make_sched(int heads, int tiles, bool contig = false)
{
    Sched S;
    S.tiles = tiles;
    const int G = int(gridDim.x);
    if (!contig && G >= heads && G % heads == 0) {
        S.interleaved = 1;
        S.cph = G / heads;
        S.head = int(blockIdx.x) % heads;
        S.j = int(blockIdx.x) / heads;
        S.begin = 0;
        S.n = (tiles > S.j) ? (tiles - S.j + S.cph - 1) / S.cph : 0;
    } else {
        const int64_t total = int64_t(heads) * tiles;
        S.interleaved = 0;
        S.cph = S.head = S.j = 0;
        S.begin = int((total * blockIdx.x) / G);
        S.n = int((total * (blockIdx.x + 1)) / G) - S.begin;
    }
    return S;
}

// grid of the persistent kernels: interleaved when the heads fit the SMs
inline int sched_grid(int sms, int heads, int tiles)
{
    if (heads <= sms) {
        const int cph = std::min(sms / heads, tiles);
        return cph * heads;
    }
    return std::min<int64_t>(sms, int64_t(heads) * tiles);
}

// ------------------------------------------------------------------ pack helpers
// low bytes of four words, in order, as one word
__device__ __forceinline__ uint32_t low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Uniform quantizer in two FMA-pipe instructions.  With s = sat(y/(6 sigma)
// + 1/2 + 2^-22) and v = RD(s * L(1 - 2^-22) + 1.5 * 2^23), the low byte of
// v's bit pattern is clamp(floor((y + 3 sigma) / Delta), 0, L - 1): the
// saturation does the clamp, the magic addend puts floor(.) in the low
// mantissa bits, the factor (1 - 2^-22) maps s = 1 to L - 1 and the 2^-22
// offset keeps y = 0 with sigma = 0 in the middle cell.  Decision
// boundaries move by at most 6 sigma 2^-22 (1.4e-6 sigma).
constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23

__device__ __forceinline__ uint32_t quant_uniform(float y, float qk, float cl)
{
    const float s = __saturatef(fmaf(y, qk, 0.5f + 0x1p-22f));
    return __float_as_uint(__fmaf_rd(s, cl, kMagic));
}

// Lloyd-Max code by the plan's bucket table (exact, one shared-memory
// load): s = RD_sat(u 2^(k-p) + 1/2) and floor(s 2^p) (a round-down FMA
// with a magic addend) give the exact bucket of u -- both scales are powers
// of two and rounding down never crosses a multiple of 2^-p -- and then
// code(u) = #{tau <= u} = cnt + (u >= hi): the same count as a search over
// the thresholds, in the same fp32 comparisons.
__device__ __forceinline__ float fma_rm_sat(float a, float b, float c)
{
    float d;
    asm("fma.rm.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ------------------------------------------------------------------ encode
constexpr int ETILE = 256;                        // tokens per encode tile (MMA N)
constexpr uint32_t ESTAGE = ETILE * D * 2;        // x tile, two K blocks: 64 KB
constexpr uint32_t EKBLK = ETILE * 128;           // one 64-element K block: 32 KB
constexpr uint32_t IDESC_E = idesc_bf16_f32(128, ETILE);
constexpr int kEncEpiWarps = 16;
constexpr int kEncThreads = 64 + 32 * kEncEpiWarps;   // producer, MMA, epilogue
constexpr uint32_t kImgCol = 256;                 // TMEM column of the basis image

// One launch encodes one or two segments (the K and V caches of a layer:
// the same shapes, basis and quantizer, each with its own plan, input and
// streams).  Work units are (segment, head) = seg * heads + h.
struct EncParams {
    PlanView pv;           // segment 0
    PlanView pv2;          // segment 1 (nseg == 2)
    int nseg;
    int max_rec;           // widest record over the segments (shared-memory layout)
    int64_t T;
    int64_t g0;            // stream group of token 0 (an append at a 128-token boundary; 0 otherwise)
    int tiles_per_head;
    int stages;
    int contig;            // contiguous work ranges (else interleaved)
    uint8_t* codes;
    int64_t sstride;
    float* norms;
    int64_t nstride;
    uint8_t* codes2;
    int64_t sstride2;
    float* norms2;
    int64_t nstride2;
};

struct EncSmem {            // offsets into dynamic shared memory (1024-aligned base)
    uint32_t xs, img, cb, cbytes, th, red, bars, total;
};

// cbytes: one tile's packed codes (8 groups of R words), double-buffered
__host__ __device__ inline EncSmem enc_smem_layout(int stages, int max_rec_bits, bool lm)
{
    EncSmem L;
    uint32_t o = 0;
    L.xs = o;   o += stages * ESTAGE;
    // the basis image passes through the x stages (all of them idle then)
    L.img = stages >= 3 ? ESTAGE : 0;
    L.cbytes = uint32_t((32 * (max_rec_bits > 0 ? max_rec_bits : 1) + 15) / 16 * 16);
    L.cb = o;   o += 2 * L.cbytes;
    L.th = o;   o += lm ? (kBkEntries * 8 + 15) / 16 * 16 : 0;   // Lloyd-Max bucket table
    L.red = o;  o += (4 * 4 * 32 + kEncEpiWarps * 32) * 4;   // RWHT norm partials and inverses
    L.bars = o; o += 256;
    L.total = o;
    return L;
}

// D[c][t] = sum_i img[c][i] x[t][i] for a 256-token tile: TMEM lane =
// channel, column = token (columns 0..255, one accumulator); the basis
// image (A operand, K-major: lane = channel, two bf16 per column) sits in
// columns 256.. for the whole head.  It reaches TMEM by a bulk copy into
// the idle x stages and tcgen05.cp, issued by the producer and the MMA
// thread.  Epilogue warp (warps 2..17): lane quadrant q = warp & 3
// (channels 32q .. 32q+31), slot gi = (warp - 2) / 4, which takes the
// 32-token groups gi and gi + 4 of every tile.  The accumulator is read
// into registers and released at once, so the MMAs of the next tile overlap
// the quantize / pack of this one.  The packed words of a tile are gathered
// in shared memory (the stream layout of 8 groups) and leave in one bulk
// store.  One epilogue thread watches the accumulator barrier and a named
// barrier wakes the rest.
// LM: Lloyd-Max quantizer; RWHT: Hadamard basis (per-token scale).
// 18 warps put five on two of the four SM sub-partitions, whose register
// files (16 K each) then allow 96 registers a thread.
template <bool LM, bool RWHT>
__global__ void __launch_bounds__(kEncThreads, 1)
encode_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_x2,
                 EncParams P)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr bool lm = LM;
    constexpr bool rwht = RWHT;
    constexpr int NT = RWHT ? 1 : 3;       // bf16 terms of the basis image
    const EncSmem L = enc_smem_layout(P.stages, P.max_rec, lm);
    uint8_t* xs = smem + L.xs;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* full = bars;                 // [stages <= 4]
    uint64_t* empty = bars + 4;            // [stages]
    uint64_t* accfull = bars + 8;
    uint64_t* accempty = bars + 9;
    uint64_t* imgsmem = bars + 10;         // basis image landed in shared memory
    uint64_t* imgcopied = bars + 11;       // ... and copied on to TMEM
    uint64_t* drain = bars + 12;
    uint64_t* rbar = bars + 13;            // [4] RWHT norm rendezvous, one per slot
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 17);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 18);
    volatile int* drain_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = P.pv.heads;
    const Sched S = make_sched(P.nseg * H, P.tiles_per_head, P.contig != 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < P.stages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(accfull, 1);
        mbar_init(accempty, kEncEpiWarps);
        mbar_init(imgsmem, 1);
        mbar_init(imgcopied, 1);
        mbar_init(drain, 1);
        for (int g = 0; g < 4; ++g) mbar_init(&rbar[g], 4);
        *abort_flag = 0;
        *drain_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);      // accumulator: columns 0..255; basis image: 256..447
        tmem_relinquish();
    }
    // the prologue above overlaps the previous kernel; global reads wait for it
    pdl_trigger();
    pdl_wait();
    bool bk_bad = false;            // the plan's tables break the buckets' premise
    if (lm) {
        const float4* src = reinterpret_cast<const float4*>(P.pv.lm_bucket);
        float4* dst = reinterpret_cast<float4*>(smem + L.th);
        for (int e = threadIdx.x; e < kBkEntries / 2; e += blockDim.x) dst[e] = src[e];
        bk_bad = *P.pv.lm_bucket_bad != 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int s = 0, k = 0, j = 0, cur_h = -1, last_s = -1, iss = 0;
            uint32_t ph = 0, last_ph = 0;
            bool img_pending = false;
            Item it = S.first();
            auto issue = [&](const Item& t) {
                mbar_arrive_expect_tx(&full[s], ESTAGE);
                uint8_t* dst = xs + s * ESTAGE;
                const bool s1 = t.h >= H;
                const CUtensorMap* tm = s1 ? &tmap_x2 : &tmap_x;
                const int hh = s1 ? t.h - H : t.h;
                tma_load_3d(dst, tm, &full[s], 0, hh, t.tile * ETILE);
                tma_load_3d(dst + EKBLK, tm, &full[s], 64, hh, t.tile * ETILE);
                last_s = s;
                last_ph = ph;
                ++iss;
                if (++s == P.stages) { s = 0; ph ^= 1u; }
            };
            for (; k < S.n; ++k, S.next(it)) {
                bool pre = false;
                if (it.h != cur_h) {
                    // every tile issued so far consumed: the stages are free
                    if (last_s >= 0 && !mbar_spin(&empty[last_s], last_ph, abort_flag, kWaitNs)) break;
                    mbar_arrive_expect_tx(imgsmem, NT * OPND);
                    const uint8_t* src = it.h >= H ? P.pv2.enc_img + size_t(it.h - H) * enc_img_bytes(D)
                                                   : P.pv.enc_img + size_t(it.h) * enc_img_bytes(D);
                    for (int t = 0; t < NT; ++t) bulk_load(smem + L.img + t * OPND, src + t * OPND, OPND, imgsmem);
                    img_pending = true;
                    // with three stages the image passes through stages 1-2,
                    // so the first tile streams meanwhile
                    if (k == 0 && L.img >= ESTAGE) {
                        issue(it);
                        pre = true;
                    }
                    if (!mbar_spin(imgcopied, j & 1, abort_flag, kWaitNs)) break;
                    img_pending = false;
                    ++j;
                    cur_h = it.h;
                    if (pre) continue;
                }
                if (iss >= P.stages && !mbar_spin(&empty[s], ph ^ 1u, abort_flag, kWaitNs)) break;
                issue(it);
            }
            if (*abort_flag) {   // let copies in flight land before the CTA exits
                for (int i = (iss > P.stages ? iss - P.stages : 0); i < iss; ++i)
                    mbar_wait(&full[i % P.stages], (i / P.stages) & 1, drain_flag, 100000000ull);
                if (img_pending) mbar_wait(imgsmem, j & 1, drain_flag, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA
        if (lane == 0) {
            int j = 0, cur_h = -1, s = 0;
            uint32_t ph = 0;
            bool issued = false;
            const uint64_t dbase = sdesc_sw128(smem_u32(xs));
            const uint64_t ibase = sdesc_sw128(smem_u32(smem + L.img));
            Item it = S.first();
            for (int k = 0; k < S.n; ++k) {
                const int h = it.h;
                S.next(it);
                if (h != cur_h) {
                    // image: shared memory -> TMEM columns 256.. (lane = channel);
                    // the MMAs below read it after the copies (same issuing thread)
                    if (!mbar_spin(imgsmem, j & 1, abort_flag, kWaitNs)) break;
                    tc_fence_after();
#pragma unroll
                    for (int t = 0; t < NT; ++t)
#pragma unroll
                        for (int kc = 0; kc < 8; ++kc)
                            tmem_cp_128x256b(tmem + kImgCol + t * 64 + kc * 8,
                                             ibase + ((t * OPND + (kc >> 2) * KBLK + (kc & 3) * 32) >> 4));
                    mma_commit(imgcopied);
                    issued = true;
                    cur_h = h;
                    ++j;
                }
                if (!mbar_spin(&full[s], ph, abort_flag, kWaitNs)) break;
                if (k > 0 && !mbar_spin(accempty, (k - 1) & 1, abort_flag, kWaitNs)) break;
                tc_fence_after();
                // descriptor start addresses advance in 16-byte units
                const uint64_t db = dbase + uint64_t(s) * (ESTAGE >> 4);
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16_ts(tmem, tmem + kImgCol + t * 64 + kk * 8,
                                    db + ((kk >> 2) * (EKBLK >> 4) + (kk & 3) * 2), IDESC_E, (t | kk) ? 1u : 0u);
                mma_commit(&empty[s]);
                mma_commit(accfull);
                if (++s == P.stages) { s = 0; ph ^= 1u; }
            }
            if (issued) {   // every tcgen05 operation of this CTA done before TMEM is released
                mma_commit(drain);
                mbar_wait(drain, 0, drain_flag, 100000000ull);
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                        // TMEM lane quadrant: channels 32q..
        const int gi = (warp - 2) >> 2;                // slot: token groups gi and gi + 4
        const int c = q * 32 + lane;                   // this thread's channel
        const bool leader = warp == 2 && lane == 0;    // watches the accumulator, issues the stores
        const uint32_t tq = tmem + (uint32_t(q * 32) << 16);
        const float2* tab = reinterpret_cast<const float2*>(smem + L.th);
        float* part = reinterpret_cast<float*>(smem + L.red) + gi * (4 * 32);          // [4 q][32 t]
        float* invs = reinterpret_cast<float*>(smem + L.red) + 4 * 4 * 32 + (warp - 2) * 32;
        int cur_h = -1, R = 0, b = 0, o = 0, bmax = 0, ruse = 0;
        float qk = 0.f, cl = 0.f;
        // Lloyd-Max bucket grid of this channel's width: clamp range, 2^k,
        // m + magic, table offset - the magic's bit pattern
        float bk_a = 0.f, bk_sc = 0.f;
        int bk_base = 0;         // table offset of the width minus the magic's bit pattern
        uint32_t bk_addr = 0u;   // the same as a shared address: first entry - 8 x the magic's bits (wraps)
        bool head_ok = true;
        uint32_t* out = nullptr;
        float* cur_norms = nullptr;            // RWHT: this unit's norms
        // the tile whose codes wait in shared memory for the bulk store
        uint32_t* p_out = nullptr;
        int p_R = 0, p_tile = 0;
        bool p_live = false;

        // leader: tile p_tile's packed words (buffer pb) -> the stream
        auto flush = [&](int pb) {
            if (!p_live) return;
            uint32_t* cb = reinterpret_cast<uint32_t*>(smem + L.cb + pb * L.cbytes);
            const int64_t t0 = int64_t(p_tile) * ETILE;
            const int ng = int(min(int64_t(8), (P.T - t0 + 31) / 32));
            const uint32_t words = uint32_t(ng * p_R);
            const uint32_t bytes = (words * 4 + 15) / 16 * 16;
            for (uint32_t w = words; w < bytes / 4; ++w) cb[w] = 0u;   // stream padding
            fence_proxy_async_smem();
            bulk_store(p_out + int64_t(p_tile) * 8 * p_R, cb, bytes);
            tma_store_commit();
        };

        // RWHT: per-token norms of one 32-token group (r: this channel's 32
        // values); ||x_t||^2 = (1/d) sum_c D[c][t]^2, reduced over the 32
        // columns across this warp's lanes (lane t ends with token t), then
        // over the four lane quadrants through shared memory.  Leaves the
        // inverse norms in invs[]; false when a rendezvous gave up.
        auto rwht_norm = [&](const uint32_t (&r)[32], int64_t tile, int g) -> bool {
            const int64_t t0 = tile * ETILE + g * 32;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * __uint_as_float(r[i]);
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1) {
                const bool up = lane & sh;
#pragma unroll
                for (int i = 0; i < sh; ++i) {
                    const float send = up ? v[i] : v[i + sh];
                    const float keep = up ? v[i + sh] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
                }
            }
            part[q * 32 + lane] = v[0];
            __syncwarp();
            if (lane == 0) mbar_arrive(&rbar[gi]);
            if (!mbar_wait(&rbar[gi], ruse & 1, abort_flag, kWaitNs)) return false;
            ++ruse;
            const float n2 = part[lane] + part[32 + lane] + part[64 + lane] + part[96 + lane];
            const float nrm = sqrtf(n2 * (1.0f / float(D)));
            if (q == 0 && head_ok && t0 + lane < P.T) cur_norms[32 * P.g0 + t0 + lane] = nrm;
            invs[lane] = (nrm > 0.f) ? 1.f / nrm : 0.f;
            __syncwarp();
            // everyone has read part[] before it is written again
            if (lane == 0) mbar_arrive(&rbar[gi]);
            if (!mbar_wait(&rbar[gi], ruse & 1, abort_flag, kWaitNs)) return false;
            ++ruse;
            return true;
        };
        // codes of 32 tokens of this channel -> byte i of the 64-bit block
        // (Y[2m], Y[2m+1]) holds bit i of tokens 8m .. 8m+7
        auto quant8 = [&](uint32_t (&r)[32], uint32_t (&Y)[8]) {
            if (!lm) {
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = quant_uniform(__uint_as_float(r[i]), qk, cl);
            } else if (!bk_bad) {
                // eight lookups in flight at a time (the memory clobber keeps the
                // compiler from hoisting all 32 loads, which needs 64 registers)
                if (rwht) {
#pragma unroll
                    for (int i0 = 0; i0 < 32; i0 += 8) {
#pragma unroll
                        for (int i = i0; i < i0 + 8; ++i) {
                            const float u = __uint_as_float(r[i]) * invs[i];
                            const float sv = fma_rm_sat(u, bk_a, 0.5f);
                            const float2 e = tab[__float_as_int(__fmaf_rd(sv, bk_sc, kMagic)) + bk_base];
                            r[i] = uint32_t(__float_as_int(e.y) + (u >= e.x ? 1 : 0));
                        }
                        asm volatile("" ::: "memory");
                    }
                } else {
                    // eigenbasis: the image already carries 1 / sigma_c, and the
                    // entry's address is the bucket value's bit pattern times 8
                    // plus one per-width base
#pragma unroll
                    for (int i0 = 0; i0 < 32; i0 += 8) {
#pragma unroll
                        for (int i = i0; i < i0 + 8; ++i) {
                            const float u = __uint_as_float(r[i]);
                            const float sv = fma_rm_sat(u, bk_a, 0.5f);
                            const uint32_t bits = __float_as_uint(__fmaf_rd(sv, bk_sc, kMagic));
                            float hi, cnt;
                            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];"
                                         : "=f"(hi), "=f"(cnt)
                                         : "r"(bk_addr + (bits << 3)));
                            r[i] = uint32_t(__float_as_int(cnt) + (u >= hi ? 1 : 0));
                        }
                        asm volatile("" ::: "memory");
                    }
                }
            } else {
                // a table whose premise failed: a binary search over the thresholds
                const float* tb = P.pv.lm_thresh + (b > 0 ? (b - 1) * kLmStride : 0);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float u = rwht ? __uint_as_float(r[i]) * invs[i] : __uint_as_float(r[i]);
                    int lo = 0;
#pragma unroll 1
                    for (int step = b > 0 ? 1 << (b - 1) : 0; step; step >>= 1)
                        if (tb[lo + step] <= u) lo += step;
                    r[i] = uint32_t(lo);
                }
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                Y[2 * m] = low_bytes(r[8 * m], r[8 * m + 1], r[8 * m + 2], r[8 * m + 3]);
                Y[2 * m + 1] = low_bytes(r[8 * m + 4], r[8 * m + 5], r[8 * m + 6], r[8 * m + 7]);
                transpose8(Y[2 * m], Y[2 * m + 1]);
            }
        };
        // the channel's bit-plane words of group g into the tile buffer
        auto store8 = [&](const uint32_t (&Y)[8], uint32_t* cb, int64_t tile, int g) {
            const int64_t t0 = tile * ETILE + g * 32;
            if (t0 >= P.T) return;
            const int64_t nt = P.T - t0;
            const uint32_t live = nt >= 32 ? 0xffffffffu : ((1u << nt) - 1u);
            uint32_t* dst = cb + g * R + o;
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
                if (kb < bmax) {
                    const int hs = kb >> 2;
                    const uint32_t pw = gather_byte(Y[hs], Y[2 + hs], Y[4 + hs], Y[6 + hs], kb & 3) & live;
                    if (kb < b) dst[kb] = pw;
                }
            }
        };

        Item it = S.first();
        for (int k = 0; k < S.n; ++k, S.next(it)) {
            const int h = it.h, tile = it.tile;
            // rendezvous: accumulator k complete; the codes of tile k-1 all in
            // shared memory; the bulk store of tile k-2 done reading its buffer
            if (warp == 2) {
                if (lane == 0) {
                    mbar_spin(accfull, k & 1, abort_flag, kWaitNs);
                    tma_store_wait_read<0>();
                }
                __syncwarp();
                tc_fence_before();
            }
            if (named_barrier_or(1, 32 * kEncEpiWarps, *abort_flag != 0)) break;
            tc_fence_after();
            if (leader) flush((k - 1) & 1);
            if (h != cur_h) {
                cur_h = h;
                const bool s1 = h >= H;                // segment of the unit
                const int hh = s1 ? h - H : h;
                const int32_t* rb = s1 ? P.pv2.rec_bits : P.pv.rec_bits;
                int32_t* st = s1 ? P.pv2.status : P.pv.status;
                R = rb[hh];
                head_ok = R <= (s1 ? P.pv2.max_rec_bits : P.pv.max_rec_bits);
                if (!head_ok && lane == 0) st[hh] = -SPECTRA_ERR_BUFFER;
                b = (s1 ? P.pv2.bits : P.pv.bits)[size_t(hh) * D + c];
                o = (s1 ? P.pv2.chan_off : P.pv.chan_off)[size_t(hh) * D + c];
                const float qs = (s1 ? P.pv2.qscale : P.pv.qscale)[size_t(hh) * D + c];
                // UNIFORM3S: qscale = 2^b / (6 sigma) -> qk = 1 / (6 sigma); LLOYD: 1 / sigma
                qk = lm ? qs : qs / float(1 << b);
                cl = float(1 << b) * (1.0f - 0x1p-22f);
                bmax = __reduce_max_sync(0xffffffffu, b);
                if (lm) {
                    const int bw = b > 0 ? b : 1;
                    bk_a = __int_as_float((127 + bk_shift(bw) - bk_log(bw)) << 23);      // 2^(k-p)
                    bk_sc = __int_as_float((127 + bk_log(bw)) << 23);                    // 2^p
                    bk_base = bk_off(bw) - __float_as_int(kMagic);
                    bk_addr = smem_u32(tab) + 8u * uint32_t(bk_base);
                }
                out = reinterpret_cast<uint32_t*>(s1 ? P.codes2 + int64_t(hh) * P.sstride2
                                                      : P.codes + int64_t(hh) * P.sstride) + P.g0 * R;
                if (rwht) cur_norms = s1 ? P.norms2 + int64_t(hh) * P.nstride2 : P.norms + int64_t(hh) * P.nstride;
            }
            uint32_t* cb = reinterpret_cast<uint32_t*>(smem + L.cb + (k & 1) * L.cbytes);
            const bool live = head_ok && R > 0;
            if (rwht || lm) {
                // one group at a time (the per-token norms and the table
                // lookups need the registers); the accumulator is released
                // after the second read -- these epilogues are longer than the MMAs
                uint32_t r[32], Y[8];
                tmem_ld32(tq + gi * 32, r);
                tmem_ld_wait();
                const bool ok0 = !rwht || rwht_norm(r, tile, gi);
                if (ok0 && live) { quant8(r, Y); store8(Y, cb, tile, gi); }
                tmem_ld32(tq + (gi + 4) * 32, r);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(accempty);
                if (ok0 && (!rwht || rwht_norm(r, tile, gi + 4)) && live) {
                    quant8(r, Y);
                    store8(Y, cb, tile, gi + 4);
                }
            } else {
                uint32_t r0[32], r1[32];
                tmem_ld32(tq + gi * 32, r0);
                tmem_ld32(tq + (gi + 4) * 32, r1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(accempty);      // accumulator read: the next tile's MMAs may start
                if (live) {
                    uint32_t Y[8];
                    quant8(r0, Y);
                    store8(Y, cb, tile, gi);
                    quant8(r1, Y);
                    store8(Y, cb, tile, gi + 4);
                }
            }
            fence_proxy_async_smem();      // this thread's words -> the bulk store
            p_out = out;
            p_R = R;
            p_tile = tile;
            p_live = live;
        }
        // the last tile's codes
        named_barrier(1, 32 * kEncEpiWarps);
        if (leader) {
            if (!*abort_flag && S.n > 0) flush((S.n - 1) & 1);
            tma_store_wait_all<0>();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        for (int kk = 0; kk < S.n; ++kk) {
            const int u = S.head_of(kk);
            (u >= H ? P.pv2.status : P.pv.status)[u >= H ? u - H : u] = -SPECTRA_ERR_TIMEOUT;
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ decode
constexpr int kDecUnpackWarps = 8;
constexpr int kDecEpiWarps = 8;   // two per TMEM lane quadrant, one column half each
constexpr int kDecThreads = 32 * (2 + kDecUnpackWarps + kDecEpiWarps);

// Like the encode: one or two segments (a layer's K and V streams), work
// units (segment, head) = seg * heads + h.
struct DecParams {
    PlanView pv;           // segment 0
    PlanView pv2;          // segment 1 (nseg == 2)
    int nseg;
    int contig;            // contiguous work ranges (else interleaved)
    int64_t T;
    int tiles_per_head;
    int total;
    int nterms;            // image terms: 2 (EIGEN) or 1 (RWHT)
    int na;                // A tiles per stage: 1 (uniform) or 2 (Lloyd-Max hi + lo)
    int astages;           // A stages (1 or 2)
    int cstages;           // code-word stages
    uint32_t cbytes;       // bytes of one code-word stage (16 * max R)
    int out_f32;
    const uint8_t* codes;
    int64_t sstride;
    const float* norms;
    int64_t nstride;
    const uint8_t* codes2;
    const float* norms2;
};

// Lloyd-Max levels in shared memory: one row per width, 257 floats apart, so
// lanes of different widths reading the same code hit different banks
constexpr int kLvStride = kLmStride + 1;

struct DecSmem {
    uint32_t img, as, cs, stg, lv, bias, bars, total;
};

__host__ __device__ inline DecSmem dec_smem_layout(int nterms, int na, int astages, int cstages, uint32_t cbytes,
                                                   bool lm)
{
    DecSmem L;
    uint32_t o = 0;
    L.img = o;  o += nterms * OPND;
    L.as = o;   o += astages * na * OPND;
    L.stg = o;  o += 2 * OPND;
    L.cs = o;   o += cstages * cbytes;
    o = (o + 15) & ~15u;
    L.lv = o;   o += lm ? kMaxBits * kLvStride * 4 : 0;
    L.bias = o; o += kDecEpiWarps * D * 4;        // per epilogue warp: output offsets of the head
    L.bars = o; o += 256;
    L.total = o;
    return L;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}


// Unpack one channel's codes of a 32-token group: planes -> code bytes.
// X[2m], X[2m+1] hold the codes of tokens 8m .. 8m+7, one per byte.
__device__ __forceinline__ void unpack_channel(const uint32_t* words, int o, int b, int bmax, uint32_t (&X)[8])
{
    uint32_t pl[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) pl[k] = (k < bmax && k < b) ? words[o + k] : 0u;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        X[2 * m] = gather_byte(pl[0], pl[1], pl[2], pl[3], m);
        X[2 * m + 1] = gather_byte(pl[4], pl[5], pl[6], pl[7], m);
        transpose8(X[2 * m], X[2 * m + 1]);
    }
}

// The same for widths <= 2: each 4-token nibble of the two planes spreads
// into bytes with one multiply (bit i -> bit 8i), no transposes.
__device__ __forceinline__ void unpack_narrow(const uint32_t* words, int o, int b, uint32_t (&X)[8])
{
    const uint32_t w0 = b > 0 ? words[o] : 0u, w1 = b > 1 ? words[o + 1] : 0u;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t s0 = (((w0 >> (4 * m)) & 0xFu) * 0x00204081u) & 0x01010101u;
        const uint32_t s1 = (((w1 >> (4 * m)) & 0xFu) * 0x00204081u) & 0x01010101u;
        X[m] = s0 | (s1 << 1);
    }
}

// byte t of the 32 codes in X as an integer
__device__ __forceinline__ int code_int(const uint32_t (&X)[8], int t)
{
    return int(__byte_perm(X[t >> 2], 0u, 0x4440u | uint32_t(t & 3)));
}

// byte i of the 32 codes in X as a float (exact): M + code - M
__device__ __forceinline__ float code_byte(const uint32_t (&X)[8], int t)
{
    return __uint_as_float(__byte_perm(X[t >> 2], 0x4B400000u, 0x7650u | uint32_t(t & 3))) - kMagic;
}

template <bool LM>
__global__ void __launch_bounds__(kDecThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_out, const __grid_constant__ CUtensorMap tmap_out2,
                 DecParams P)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr bool lm = LM;
    const bool rwht = P.pv.basis == SPECTRA_BASIS_RWHT;
    const DecSmem L = dec_smem_layout(P.nterms, P.na, P.astages, P.cstages, P.cbytes, lm);
    uint8_t* img = smem + L.img;
    uint8_t* as = smem + L.as;
    uint8_t* cs = smem + L.cs;
    uint8_t* stg = smem + L.stg;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* cfull = bars;          // [cstages <= 4]
    uint64_t* cempty = bars + 4;     // [cstages]
    uint64_t* afull = bars + 8;      // [astages <= 2]
    uint64_t* aempty = bars + 10;    // [astages]
    uint64_t* accfull = bars + 12;   // [2]
    uint64_t* accempty = bars + 14;  // [2]
    uint64_t* imgfull = bars + 16;
    uint64_t* imgempty = bars + 17;
    uint64_t* drain = bars + 18;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 20);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 21);
    volatile int* drain_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = P.pv.heads;
    const Sched S = make_sched(P.nseg * H, P.tiles_per_head, P.contig != 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < P.cstages; ++s) { mbar_init(&cfull[s], 1); mbar_init(&cempty[s], kDecUnpackWarps); }
        for (int s = 0; s < P.astages; ++s) { mbar_init(&afull[s], kDecUnpackWarps); mbar_init(&aempty[s], 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(&accfull[a], 1); mbar_init(&accempty[a], kDecEpiWarps); }
        mbar_init(imgfull, 1);
        mbar_init(imgempty, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        *drain_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 256);
        tmem_relinquish();
    }
    // the prologue above overlaps the previous kernel; global reads wait for it
    pdl_trigger();
    pdl_wait();
    if (lm) {
        float* lv = reinterpret_cast<float*>(smem + L.lv);
        // each level as its bf16 pair (hi = RN(level), lo = RN(level - hi)) in one word
        uint32_t* lvp = reinterpret_cast<uint32_t*>(lv);
        for (int e = threadIdx.x; e < kMaxBits * kLmStride; e += blockDim.x) {
            const float v = P.pv.lm_level[e];
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
            lvp[(e / kLmStride) * kLvStride + e % kLmStride] =
                uint32_t(__bfloat16_as_ushort(hi)) | (uint32_t(__bfloat16_as_ushort(lo)) << 16);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int k = 0, j = 0, cur_h = -1, R = 0;
            int last_issued[4] = {-1, -1, -1, -1};
            int img_issued = 0, cs_i = 0;
            uint32_t cs_ph = 0;
            const uint8_t* hcodes = nullptr;     // this unit's stream
            Item it = S.first();
            for (; k < S.n; ++k, S.next(it)) {
                const int h = it.h, tile = it.tile;
                if (h != cur_h) {
                    if (j > 0 && !mbar_wait(imgempty, (j - 1) & 1, abort_flag, kWaitNs)) break;
                    const uint32_t bytes = P.nterms * OPND;
                    mbar_arrive_expect_tx(imgfull, bytes);
                    const bool s1 = h >= H;
                    const int hh = s1 ? h - H : h;
                    const uint8_t* src = (s1 ? P.pv2.dec_img : P.pv.dec_img) + size_t(hh) * dec_img_bytes(D);
                    for (uint32_t o = 0; o < bytes; o += 32768u) bulk_load(img + o, src + o, 32768u, imgfull);
                    img_issued = j + 1;
                    cur_h = h;
                    R = (s1 ? P.pv2.rec_bits : P.pv.rec_bits)[hh];
                    if (R > (s1 ? P.pv2.max_rec_bits : P.pv.max_rec_bits)) {
                        (s1 ? P.pv2.status : P.pv.status)[hh] = -SPECTRA_ERR_BUFFER;
                        R = 0;
                    }
                    hcodes = s1 ? P.codes2 + int64_t(hh) * P.sstride : P.codes + int64_t(hh) * P.sstride;
                    ++j;
                }
                const int s = cs_i;
                if (k >= P.cstages && !mbar_spin(&cempty[s], cs_ph ^ 1u, abort_flag, kWaitNs)) break;
                if (++cs_i == P.cstages) { cs_i = 0; cs_ph ^= 1u; }
                const int64_t t0 = int64_t(tile) * TILE;
                const int64_t ngroups = min(int64_t(4), (P.T - t0 + 31) / 32);
                const uint32_t bytes = uint32_t((ngroups * 4 * R + 15) / 16 * 16);
                if (bytes > 0) {
                    mbar_arrive_expect_tx(&cfull[s], bytes);
                    bulk_load(cs + s * P.cbytes, hcodes + (t0 / 32) * 4 * R, bytes, &cfull[s]);
                    last_issued[s] = k;
                } else {
                    mbar_arrive(&cfull[s]);
                }
            }
            if (*abort_flag) {
                for (int s = 0; s < P.cstages; ++s)
                    if (last_issued[s] >= 0)
                        mbar_wait(&cfull[s], (last_issued[s] / P.cstages) & 1, drain_flag, 100000000ull);
                if (img_issued > 0) mbar_wait(imgfull, (img_issued - 1) & 1, drain_flag, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA
        if (lane == 0) {
            int k = 0, j = 0, cur_h = -1;
            bool issued = false;
            // products (A term, image term): uniform 2 (ell x hi, ell x lo);
            // EIGEN Lloyd-Max 3 (hi x hi, lo x hi, hi x lo); RWHT 2 (hi, lo x +-1)
            const int npr = !lm ? P.nterms : (!rwht ? 3 : 2);
            const uint32_t pa = !lm ? 0u : (!rwht ? 0x010u : 0x10u);    // nibble pr: A term
            const uint32_t pb = !lm ? 0x10u : (!rwht ? 0x100u : 0x00u); // nibble pr: image term
            int as_i = 0;
            uint32_t as_ph = 0;
            Item it = S.first();
            for (; k < S.n; ++k) {
                const int h = it.h;
                S.next(it);
                if (h != cur_h) {
                    if (!mbar_spin(imgfull, j & 1, abort_flag, kWaitNs)) break;
                    cur_h = h;
                    ++j;
                }
                const int s = as_i, a = k & 1;
                if (!mbar_spin(&afull[s], as_ph, abort_flag, kWaitNs)) break;
                if (++as_i == P.astages) { as_i = 0; as_ph ^= 1u; }
                if (k >= 2 && !mbar_spin(&accempty[a], ((k >> 1) - 1) & 1, abort_flag, kWaitNs)) break;
                tc_fence_after();
                const uint32_t aa = smem_u32(as + s * P.na * OPND);
                const uint32_t ia = smem_u32(img);
                const uint32_t d_tmem = tmem + a * 128;
                for (int pr = 0; pr < npr; ++pr) {
                    const uint32_t at = (pa >> (4 * pr)) & 15u, bt = (pb >> (4 * pr)) & 15u;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t koff = (kk >> 2) * KBLK + (kk & 3) * 32;
                        mma_bf16_ss(d_tmem, sdesc_sw128(aa + at * OPND + koff), sdesc_sw128(ia + bt * OPND + koff),
                                    IDESC, (pr | kk) ? 1u : 0u);
                    }
                }
                issued = true;
                mma_commit(&aempty[s]);
                mma_commit(&accfull[a]);
                const bool head_ends = (k + 1 == S.n) || (it.h != h);
                if (head_ends) mma_commit(imgempty);
            }
            if (issued) {
                mma_commit(drain);
                mbar_wait(drain, 0, drain_flag, 100000000ull);
            }
        }
    } else if (warp < 2 + kDecUnpackWarps) {
        // ---------------------------------------------------------- unpack
        // unit = (group gi, channel half hc); lane handles channels c0 = 64 hc + 2 lane, c0 + 1
        const int u = warp - 2, gi = u >> 1, hc = u & 1;
        const int c0 = 64 * hc + 2 * lane;
        const float* lv = reinterpret_cast<const float*>(smem + L.lv);
        int k = 0, cur_h = -1, R = 0, b0 = 0, b1 = 0, o0 = 0, o1 = 0, bmax = 0;
        float off0 = 0.f, off1 = 0.f;
        bool code_mode = false;
        int u_ci = 0, u_ai = 0;
        uint32_t u_cph = 0, u_aph = 0;
        Item it = S.first();
        for (; k < S.n; ++k, S.next(it)) {
            const int h = it.h, tile = it.tile;
            if (h != cur_h) {
                cur_h = h;
                const bool s1 = h >= H;
                const int hh = s1 ? h - H : h;
                R = (s1 ? P.pv2.rec_bits : P.pv.rec_bits)[hh];
                if (R > (s1 ? P.pv2.max_rec_bits : P.pv.max_rec_bits)) R = 0;
                const uint8_t* bts = s1 ? P.pv2.bits : P.pv.bits;
                const uint16_t* cof = s1 ? P.pv2.chan_off : P.pv.chan_off;
                b0 = bts[size_t(hh) * D + c0];
                b1 = bts[size_t(hh) * D + c0 + 1];
                o0 = cof[size_t(hh) * D + c0];
                o1 = cof[size_t(hh) * D + c0 + 1];
                off0 = 1.0f - float(1 << b0);
                off1 = 1.0f - float(1 << b1);
                bmax = __reduce_max_sync(0xffffffffu, max(b0, b1));
                code_mode = !lm && !rwht && (s1 ? P.pv2.wmax : P.pv.wmax)[hh] <= 7;
            }
            const int sc = u_ci, sa = u_ai;
            if (!mbar_wait(&cfull[sc], u_cph, abort_flag, kWaitNs)) break;
            if (k >= P.astages && !mbar_wait(&aempty[sa], u_aph ^ 1u, abort_flag, kWaitNs)) break;
            if (++u_ci == P.cstages) { u_ci = 0; u_cph ^= 1u; }
            if (++u_ai == P.astages) { u_ai = 0; u_aph ^= 1u; }
            const int64_t t0 = int64_t(tile) * TILE + gi * 32;
            if (t0 < P.T && R > 0) {
                const uint32_t* words = reinterpret_cast<const uint32_t*>(cs + sc * P.cbytes) + gi * R;
                uint32_t X0[8], X1[8];
                if (bmax <= 2) {
                    unpack_narrow(words, o0, b0, X0);
                    unpack_narrow(words, o1, b1, X1);
                } else {
                    unpack_channel(words, o0, b0, bmax, X0);
                    unpack_channel(words, o1, b1, bmax, X1);
                }
                const uint32_t abase = smem_u32(as + sa * P.na * OPND) + hc * KBLK;
                const uint32_t* lv0 = reinterpret_cast<const uint32_t*>(lv) + (b0 > 0 ? (b0 - 1) * kLvStride : 0);
                const uint32_t* lv1 = reinterpret_cast<const uint32_t*>(lv) + (b1 > 0 ? (b1 - 1) * kLvStride : 0);
                if (code_mode) {
                    // (c0, c0+1) of token t as bf16 (128 + code): byte permutes only.
                    // Row r = 32 gi + t; its swizzled chunk depends on r & 7 = t & 7.
                    uint32_t rb[8];
#pragma unroll
                    for (int r8 = 0; r8 < 8; ++r8)
                        rb[r8] = abase + uint32_t(gi * 32) * 128u + ((uint32_t(lane >> 2) ^ uint32_t(r8)) << 4) +
                                 4u * uint32_t(lane & 3);
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const uint32_t lo = __byte_perm(X0[m], X1[m], 0x5140);   // tokens 4m, 4m+1
                        const uint32_t hi = __byte_perm(X0[m], X1[m], 0x7362);   // tokens 4m+2, 4m+3
                        const int t = 4 * m;
                        st_shared_u32(rb[(t + 0) & 7] + uint32_t(t + 0) * 128u, __byte_perm(lo, 0x4343u, 0x5140));
                        st_shared_u32(rb[(t + 1) & 7] + uint32_t(t + 1) * 128u, __byte_perm(lo, 0x4343u, 0x5342));
                        st_shared_u32(rb[(t + 2) & 7] + uint32_t(t + 2) * 128u, __byte_perm(hi, 0x4343u, 0x5140));
                        st_shared_u32(rb[(t + 3) & 7] + uint32_t(t + 3) * 128u, __byte_perm(hi, 0x4343u, 0x5342));
                    }
                } else
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const uint32_t row = uint32_t(gi * 32 + t);
                    const uint32_t addr = abase + row * 128u + ((uint32_t(lane >> 2) ^ (row & 7u)) << 4) +
                                          4u * uint32_t(lane & 3);
                    if (!lm) {
                        const float k0 = code_byte(X0, t), k1 = code_byte(X1, t);
                        // 2 code + 1 - 2^b (odd integer, exact in bf16); 0 for dropped channels
                        const float v0 = b0 ? fmaf(k0, 2.f, off0) : 0.f;
                        const float v1 = b1 ? fmaf(k1, 2.f, off1) : 0.f;
                        st_shared_u32(addr, pack_bf16x2(v0, v1));
                    } else {
                        // the levels' (hi, lo) pairs of channels c0, c0 + 1 -> the hi and lo tiles
                        const uint32_t e0 = b0 ? lv0[code_int(X0, t)] : 0u;
                        const uint32_t e1 = b1 ? lv1[code_int(X1, t)] : 0u;
                        st_shared_u32(addr, __byte_perm(e0, e1, 0x5410));
                        st_shared_u32(addr + OPND, __byte_perm(e0, e1, 0x7632));
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&afull[sa]);
                mbar_arrive(&cempty[sc]);
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        // warp e = warp - 2 - unpack warps: TMEM lane quadrant q = warp & 3
        // (tokens 32q ..), column half ch = e / 4 (outputs 64 ch ..)
        const int q = warp & 3, ch = (warp - 2 - kDecUnpackWarps) >> 2;
        const bool leader = (warp == 2 + kDecUnpackWarps && lane == 0);
        float* bsh = reinterpret_cast<float*>(smem + L.bias) + (warp - 2 - kDecUnpackWarps) * D;
        int k = 0, cur_h = -1, hh = 0;
        bool code_mode = false, s1 = false;   // s1: the unit's segment
        // all the epilogue warps (named barrier 1); the OR of the abort flag
        // makes every warp leave at the same point
        auto rendezvous = [&]() -> bool {
            __syncwarp();
            return !named_barrier_or(1, 32 * kDecEpiWarps, *abort_flag != 0);
        };
        Item it = S.first();
        for (; k < S.n; ++k, S.next(it)) {
            const int h = it.h, tile = it.tile;
            if (h != cur_h) {       // code mode: per-output offsets of this head
                cur_h = h;
                s1 = h >= H;
                hh = s1 ? h - H : h;
                code_mode = !lm && !rwht && (s1 ? P.pv2.wmax : P.pv.wmax)[hh] <= 7;
                const float* db = s1 ? P.pv2.dec_bias : P.pv.dec_bias;
                __syncwarp();
                for (int i = lane; i < D; i += 32) bsh[i] = code_mode ? db[size_t(hh) * D + i] : 0.f;
                __syncwarp();
            }
            const int a = k & 1;
            if (leader) mbar_spin(&accfull[a], (k >> 1) & 1, abort_flag, kWaitNs);
            bool ok = true;
            const int64_t t = int64_t(tile) * TILE + q * 32 + lane;
            float scale = 1.f;
            if (rwht) scale = (t < P.T) ? (s1 ? P.norms2 : P.norms)[int64_t(hh) * P.nstride + t] * (1.0f / float(D)) : 0.f;
            const uint32_t tm = tmem + a * 128 + (uint32_t(q * 32) << 16);
            const uint32_t row = uint32_t(q * 32 + lane);
            const int nrounds = P.out_f32 ? 2 : 1;
            for (int rd = 0; rd < nrounds; ++rd) {
                // staging slot(s) must be free: the stores issued from them earlier have read them
                const int slot = P.out_f32 ? rd : (k & 1);
                if (leader) tma_store_wait_read<1>();
                tc_fence_before();
                if (!(ok = rendezvous())) break;
                tc_fence_after();
                uint8_t* sb = stg + slot * OPND;
                const uint32_t sba = smem_u32(sb);
                if (!P.out_f32) {
                    // 32 columns at a time; the load of the next 32 is in flight
                    // while these are converted (one wait covers both loads)
                    auto convert = [&](const uint32_t (&r)[32], int j) {
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            uint32_t pk[4];
                            const float4 bA = *reinterpret_cast<const float4*>(bsh + 32 * j + c4 * 8);
                            const float4 bB = *reinterpret_cast<const float4*>(bsh + 32 * j + c4 * 8 + 4);
                            const float bb[8] = {bA.x, bA.y, bA.z, bA.w, bB.x, bB.y, bB.z, bB.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                pk[e] = pack_bf16x2(fmaf(__uint_as_float(r[c4 * 8 + 2 * e]), scale, bb[2 * e]),
                                                    fmaf(__uint_as_float(r[c4 * 8 + 2 * e + 1]), scale, bb[2 * e + 1]));
                            const uint32_t off = (j >> 1) * KBLK + sw128_offset(row, (j & 1) * 64 + c4 * 16);
                            st_shared_v4(sba + off, pk[0], pk[1], pk[2], pk[3]);
                        }
                    };
                    uint32_t ra[32], rb[32];
                    tmem_ld32(tm + 64 * ch, ra);
                    tmem_ld_wait();
                    tmem_ld32(tm + 64 * ch + 32, rb);
                    convert(ra, 2 * ch);
                    tmem_ld_wait();
                    // accumulator read: the MMA may reuse it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&accempty[a]);
                    convert(rb, 2 * ch + 1);
                } else {
                    {
                        const int j = ch;
                        uint32_t r[32];
                        tmem_ld32(tm + 64 * rd + 32 * j, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4) {
                            const uint32_t off = j * KBLK + sw128_offset(row, c4 * 16);
                            const float4 bA = *reinterpret_cast<const float4*>(bsh + 64 * rd + 32 * j + 4 * c4);
                            st_shared_v4(sba + off, __float_as_uint(fmaf(__uint_as_float(r[4 * c4]), scale, bA.x)),
                                         __float_as_uint(fmaf(__uint_as_float(r[4 * c4 + 1]), scale, bA.y)),
                                         __float_as_uint(fmaf(__uint_as_float(r[4 * c4 + 2]), scale, bA.z)),
                                         __float_as_uint(fmaf(__uint_as_float(r[4 * c4 + 3]), scale, bA.w)));
                        }
                    }
                }
                if (P.out_f32 && rd == nrounds - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&accempty[a]);
                }
                fence_proxy_async_smem();
                if (!(ok = rendezvous())) break;
                if (leader) {
                    const CUtensorMap* tmo = s1 ? &tmap_out2 : &tmap_out;
                    if (!P.out_f32) {
                        tma_store_3d(tmo, sb, 0, hh, tile * TILE);
                        tma_store_3d(tmo, sb + KBLK, 64, hh, tile * TILE);
                    } else {
                        tma_store_3d(tmo, sb, 64 * rd, hh, tile * TILE);
                        tma_store_3d(tmo, sb + KBLK, 64 * rd + 32, hh, tile * TILE);
                    }
                    tma_store_commit();
                }
            }
            if (!ok) break;
        }
        if (leader) tma_store_wait_all<0>();
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        for (int kk = 0; kk < S.n; ++kk) {
            const int u = S.head_of(kk);
            (u >= H ? P.pv2.status : P.pv.status)[u >= H ? u - H : u] = -SPECTRA_ERR_TIMEOUT;
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ------------------------------------------------------------------ images
// Operand images of one head, in the swizzled K-major layout the MMAs read.
//  encode (B operand, rows = channel c, K = input index i):
//    EIGEN: three bf16 terms of basis[i][c] (hi, mid, lo);  RWHT: s_i H[i][c].
//  decode (B operand, rows = output index i, K = channel c):
//    EIGEN uniform: basis[i][c] * Delta_c / 2;  EIGEN Lloyd-Max: basis[i][c] *
//    sigma_c -- two bf16 terms (hi, lo);  RWHT: s_i H[i][c].
// Decode "code mode" (uniform quantizer, every width <= 7): the A operand is
// the exact bf16 number 128 + code, the image basis[i][c] * Delta_c, and the
// decode adds dec_bias[i] = sum_c basis[i][c] (Delta_c / 2)(1 - 2^b_c)
// - 128 sum_c image[i][c]  (so x_i = sum_c image[i][c] code_c + the affine
// part of the dequantizer).  Otherwise A is the odd integer 2 code + 1 - 2^b
// and the image basis * Delta / 2.
__device__ __forceinline__ float dec_image_value(const PlanView& pv, int h, int i, int c, bool code_mode)
{
    if (pv.basis == SPECTRA_BASIS_RWHT) return float(pv.signs[size_t(h) * D + i] * hadamard_sign(i, c));
    const float sc = pv.rscale[size_t(h) * D + c];
    const float bij = pv.basis_mat[(size_t(h) * D + i) * D + c];
    if (pv.quant != SPECTRA_Q_UNIFORM3S) return bij * sc;
    if (code_mode) return pv.bits[size_t(h) * D + c] > 0 ? bij * sc : 0.f;
    return bij * 0.5f * sc;
}

// grid (heads, D / 16): block (h, part) writes rows [16 part, 16 part + 16)
// of both images of head h and the decode offsets of those output rows.
constexpr int kImgRows = 16;

__global__ void __launch_bounds__(256)
tc_images_kernel(PlanView pv, uint8_t* __restrict__ enc, uint8_t* __restrict__ dec,
                 int32_t* __restrict__ wmax_out, float* __restrict__ bias_out)
{
    const int h = blockIdx.x, r0 = blockIdx.y * kImgRows;
    const bool rwht = pv.basis == SPECTRA_BASIS_RWHT;
    __shared__ int wmax_s;
    if (threadIdx.x == 0) wmax_s = 0;
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += blockDim.x) atomicMax(&wmax_s, int(pv.bits[size_t(h) * D + c]));
    __syncthreads();
    const bool code_mode = !rwht && pv.quant == SPECTRA_Q_UNIFORM3S && wmax_s <= 7;
    if (threadIdx.x == 0 && blockIdx.y == 0) wmax_out[h] = wmax_s;
    uint8_t* e = enc + size_t(h) * enc_img_bytes(D);
    uint8_t* dd = dec + size_t(h) * dec_img_bytes(D);
    for (int idx = threadIdx.x; idx < kImgRows * D; idx += blockDim.x) {
        const int r = r0 + idx / D, kk = idx % D;   // row, K index
        const uint32_t off = (kk >> 6) * KBLK + sw128_offset(r, (kk & 63) * 2);
        // encode: row = channel r, K = input i = kk
        {
            float v;
            if (rwht) v = float(pv.signs[size_t(h) * D + kk] * hadamard_sign(kk, r));
            else v = pv.basis_mat[(size_t(h) * D + kk) * D + r];
            // Lloyd-Max on an eigenbasis: the contraction yields u = y / sigma_c directly
            if (!rwht && pv.quant == SPECTRA_Q_LLOYD_GAUSS) v *= pv.qscale[size_t(h) * D + r];
            const int nt = rwht ? 1 : 3;
            float rem = v;
            for (int t = 0; t < nt; ++t) {
                const __nv_bfloat16 b = __float2bfloat16_rn(rem);
                *reinterpret_cast<__nv_bfloat16*>(e + t * OPND + off) = b;
                rem -= __bfloat162float(b);
            }
        }
        // decode: row = output i = r, K = channel c = kk
        {
            const int nt = rwht ? 1 : 2;
            float rem = dec_image_value(pv, h, r, kk, code_mode);
            for (int t = 0; t < nt; ++t) {
                const __nv_bfloat16 b = __float2bfloat16_rn(rem);
                *reinterpret_cast<__nv_bfloat16*>(dd + t * OPND + off) = b;
                rem -= __bfloat162float(b);
            }
        }
    }
    // per-output offsets of code mode (sums of the rounded image terms):
    // one warp per output row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int ri = warp; ri < kImgRows; ri += blockDim.x >> 5) {
        const int i = r0 + ri;
        float aff = 0.f, img = 0.f;
        if (code_mode) {
            for (int c = lane; c < D; c += 32) {
                const int b = pv.bits[size_t(h) * D + c];
                if (b == 0) continue;
                const float v = dec_image_value(pv, h, i, c, true);
                const __nv_bfloat16 hi = __float2bfloat16_rn(v);
                const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
                img += __bfloat162float(hi) + __bfloat162float(lo);
                aff = fmaf(pv.basis_mat[(size_t(h) * D + i) * D + c] * 0.5f * pv.rscale[size_t(h) * D + c],
                           1.f - float(1 << b), aff);
            }
            for (int o = 16; o; o >>= 1) {
                aff += __shfl_xor_sync(0xffffffffu, aff, o);
                img += __shfl_xor_sync(0xffffffffu, img, o);
            }
        }
        if (lane == 0) bias_out[size_t(h) * D + i] = code_mode ? aff - 128.f * img : 0.f;
    }
}

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    static int cache[64] = {0};
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && cache[dev]) return cache[dev];
    int n = 148;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (dev < 64) cache[dev] = n;
    return n;
}

// [T][heads][128] cache of 2- or 4-byte elements, box [rows tokens][1][64 or 32]
bool make_cache_map(CUtensorMap* m, const void* base, bool f32, int heads, int64_t T, int64_t tstride,
                    int rows = TILE)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const int es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(heads), cuuint64_t(T)};
    cuuint64_t strides[2] = {cuuint64_t(D) * es, cuuint64_t(tstride) * es};
    cuuint32_t box[3] = {cuuint32_t(128 / es), 1u, cuuint32_t(rows)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

constexpr uint32_t kSmemMax = 227 * 1024;

}  // namespace

spectra_status launch_tc_images(const spectra_plan* plan, cudaStream_t s)
{
    if (plan->head_dim != D) return SPECTRA_OK;
    const PlanView pv = make_view(plan);
    tc_images_kernel<<<dim3(plan->heads, D / kImgRows), 256, 0, s>>>(pv, const_cast<uint8_t*>(pv.enc_img), const_cast<uint8_t*>(pv.dec_img),
                                                  const_cast<int32_t*>(pv.wmax), const_cast<float*>(pv.dec_bias));
    return cuda_status(cudaGetLastError());
}

namespace {

// One launch over nseg (1 or 2) segments; returns with *done false (nothing
// launched) when the tensor-core path does not cover the call.
spectra_status encode_tc_segs(const spectra_plan* const* plans, const void* const* xs, int nseg, int dt, int64_t T,
                              int64_t token_stride, uint8_t* const* codes, const int64_t* sstride,
                              float* const* norms, const int64_t* nstride, cudaStream_t s, bool* done, int64_t g0)
{
    *done = false;
    const spectra_plan* plan = plans[0];
    if (dt != SPECTRA_BF16 || plan->head_dim != D || T <= 0) return SPECTRA_OK;
    if (T > (int64_t(1) << 31) - ETILE) return SPECTRA_OK;
    if (nseg == 2) {
        const spectra_plan* p2 = plans[1];
        if (p2->head_dim != D || p2->heads != plan->heads || p2->basis != plan->basis || p2->quant != plan->quant)
            return SPECTRA_OK;
    }
    CUtensorMap m[2];
    for (int i = 0; i < nseg; ++i)
        if (!make_cache_map(&m[i], xs[i], false, plan->heads, T, token_stride, ETILE)) return SPECTRA_OK;
    if (nseg == 1) m[1] = m[0];
    EncParams P;
    P.pv = make_view(plan);
    P.pv2 = nseg == 2 ? make_view(plans[1]) : P.pv;
    P.nseg = nseg;
    P.max_rec = std::max(plan->max_rec_bits, nseg == 2 ? plans[1]->max_rec_bits : 0);
    P.T = T;
    P.g0 = g0;
    P.tiles_per_head = int((T + ETILE - 1) / ETILE);
    const int units = nseg * plan->heads;
    const int64_t total = int64_t(P.tiles_per_head) * units;
    if (total > (int64_t(1) << 31) - 1) return SPECTRA_OK;
    const bool lm = plan->quant == SPECTRA_Q_LLOYD_GAUSS;
    P.stages = 4;
    while (P.stages > 2 && enc_smem_layout(P.stages, P.max_rec, lm).total + 1024 > kSmemMax) --P.stages;
    if (enc_smem_layout(P.stages, P.max_rec, lm).total + 1024 > kSmemMax) return SPECTRA_OK;
    P.codes = codes[0];
    P.sstride = sstride[0];
    P.norms = norms[0];
    P.nstride = nstride[0];
    P.codes2 = codes[nseg - 1];
    P.sstride2 = sstride[nseg - 1];
    P.norms2 = norms[nseg - 1];
    P.nstride2 = nstride[nseg - 1];
    // interleaved schedule (the CTAs of all units read whole token rows at
    // about the same time, which measured ~10% faster per tile) unless
    // contiguous ranges give every CTA over 15% fewer tiles
    const int sms = sm_count();
    int grid = sched_grid(sms, units, P.tiles_per_head);
    P.contig = 0;
    if (units <= sms) {
        const int cph = grid / units;
        const int64_t inter_max = (P.tiles_per_head + cph - 1) / cph;
        const int64_t g2 = std::min<int64_t>(sms, total);
        const int64_t contig_max = (total + g2 - 1) / g2;
        if (contig_max * 115 < inter_max * 100) {
            P.contig = 1;
            grid = int(g2);
        }
    }
    const uint32_t sm = enc_smem_layout(P.stages, P.max_rec, lm).total + 1024;
    const bool rw = plan->basis == SPECTRA_BASIS_RWHT;
    auto kern = lm ? (rw ? encode_tc_kernel<true, true> : encode_tc_kernel<true, false>)
                   : (rw ? encode_tc_kernel<false, true> : encode_tc_kernel<false, false>);
    if (spectra_status st = set_smem(kern, sm)) return st;
    if (cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kEncThreads), sm, s, m[0], m[1], P)) return cuda_status(e);
    *done = true;
    return cuda_status(cudaGetLastError());
}

}  // namespace

spectra_status launch_encode_tc(const spectra_plan* plan, const void* x, int dt, int64_t T, int64_t token_stride,
                                uint8_t* codes, int64_t sstride, float* norms, int64_t nstride, cudaStream_t s,
                                bool* done, int64_t g0)
{
    return encode_tc_segs(&plan, &x, 1, dt, T, token_stride, &codes, &sstride, &norms, &nstride, s, done, g0);
}

spectra_status launch_encode_tc_kv(const spectra_plan* kplan, const spectra_plan* vplan, const void* k,
                                   const void* v, int dt, int64_t T, int64_t token_stride, uint8_t* k_codes,
                                   uint8_t* v_codes, int64_t sstride, float* k_norms, float* v_norms,
                                   int64_t nstride, cudaStream_t s, bool* done)
{
    const spectra_plan* plans[2] = {kplan, vplan};
    const void* xs[2] = {k, v};
    uint8_t* cs[2] = {k_codes, v_codes};
    const int64_t ss[2] = {sstride, sstride};
    float* ns[2] = {k_norms, v_norms};
    const int64_t nss[2] = {nstride, nstride};
    return encode_tc_segs(plans, xs, 2, dt, T, token_stride, cs, ss, ns, nss, s, done, 0);
}

namespace {

// One launch over nseg (1 or 2) segments; *done false when the tensor-core
// path does not cover the call.
spectra_status decode_tc_segs(const spectra_plan* const* plans, const uint8_t* const* codes, int nseg,
                              int64_t sstride, const float* const* norms, int64_t nstride, int64_t T,
                              void* const* outs, int out_dt, int64_t token_stride, cudaStream_t s, bool* done)
{
    *done = false;
    const spectra_plan* plan = plans[0];
    if (plan->head_dim != D || T <= 0) return SPECTRA_OK;
    if (T > (int64_t(1) << 31) - TILE) return SPECTRA_OK;
    if (nseg == 2) {
        const spectra_plan* p2 = plans[1];
        if (p2->head_dim != D || p2->heads != plan->heads || p2->basis != plan->basis || p2->quant != plan->quant)
            return SPECTRA_OK;
    }
    const bool f32 = out_dt == SPECTRA_F32;
    CUtensorMap m[2];
    for (int i = 0; i < nseg; ++i)
        if (!make_cache_map(&m[i], outs[i], f32, plan->heads, T, token_stride)) return SPECTRA_OK;
    if (nseg == 1) m[1] = m[0];
    DecParams P;
    P.pv = make_view(plan);
    P.pv2 = nseg == 2 ? make_view(plans[1]) : P.pv;
    P.nseg = nseg;
    P.T = T;
    P.tiles_per_head = int((T + TILE - 1) / TILE);
    const int units = nseg * plan->heads;
    if (int64_t(P.tiles_per_head) * units > (int64_t(1) << 31) - 1) return SPECTRA_OK;
    P.total = P.tiles_per_head * units;
    const bool lm = plan->quant == SPECTRA_Q_LLOYD_GAUSS;
    P.nterms = plan->basis == SPECTRA_BASIS_RWHT ? 1 : 2;
    P.na = lm ? 2 : 1;
    const int max_rec = std::max(plan->max_rec_bits, nseg == 2 ? plans[1]->max_rec_bits : 0);
    P.cbytes = uint32_t(16 * (max_rec > 0 ? max_rec : 1));
    P.astages = 2;
    P.cstages = 3;
    auto total = [&] { return dec_smem_layout(P.nterms, P.na, P.astages, P.cstages, P.cbytes, lm).total + 1024; };
    while (total() > kSmemMax && P.cstages > 2) --P.cstages;
    while (total() > kSmemMax && P.astages > 1) --P.astages;
    if (total() > kSmemMax) return SPECTRA_OK;
    P.out_f32 = f32 ? 1 : 0;
    P.codes = codes[0];
    P.sstride = sstride;
    P.norms = norms[0];
    P.nstride = nstride;
    P.codes2 = codes[nseg - 1];
    P.norms2 = norms[nseg - 1];
    const uint32_t sm = total();
    auto kern = lm ? decode_tc_kernel<true> : decode_tc_kernel<false>;
    if (spectra_status st = set_smem(kern, sm)) return st;
    // interleaved schedule unless contiguous ranges give every CTA fewer tiles
    const int sms = sm_count();
    int grid = sched_grid(sms, units, P.tiles_per_head);
    P.contig = 0;
    if (units <= sms) {
        const int cph = grid / units;
        const int64_t inter_max = (P.tiles_per_head + cph - 1) / cph;
        const int64_t g2 = std::min<int64_t>(sms, P.total);
        const int64_t contig_max = (P.total + g2 - 1) / g2;
        if (contig_max < inter_max) {
            P.contig = 1;
            grid = int(g2);
        }
    }
    if (cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kDecThreads), sm, s, m[0], m[1], P))
        return cuda_status(e);
    *done = true;
    return cuda_status(cudaGetLastError());
}

}  // namespace

spectra_status launch_decode_tc(const spectra_plan* plan, const uint8_t* codes, int64_t sstride, const float* norms,
                                int64_t nstride, int64_t T, void* x_out, int out_dt, int64_t token_stride,
                                cudaStream_t s, bool* done)
{
    return decode_tc_segs(&plan, &codes, 1, sstride, &norms, nstride, T, &x_out, out_dt, token_stride, s, done);
}

spectra_status launch_decode_tc_kv(const spectra_plan* kplan, const spectra_plan* vplan, const uint8_t* k_codes,
                                   const uint8_t* v_codes, int64_t sstride, const float* k_norms,
                                   const float* v_norms, int64_t nstride, int64_t T, void* k_out, void* v_out,
                                   int out_dt, int64_t token_stride, cudaStream_t s, bool* done)
{
    const spectra_plan* plans[2] = {kplan, vplan};
    const uint8_t* cs[2] = {k_codes, v_codes};
    const float* ns[2] = {k_norms, v_norms};
    void* outs[2] = {k_out, v_out};
    return decode_tc_segs(plans, cs, 2, sstride, ns, nstride, T, outs, out_dt, token_stride, s, done);
}

}  // namespace spectra
