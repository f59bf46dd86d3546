// attn_tc.cu -- decode-step attention over packed K/V streams on the tensor
// cores, computed on the bit planes themselves (uniform quantizer,
// eigenbasis plans, head_dim 128, at most four query heads per kv head).
//
// "Sintesi Tecnica: SPECTRA", "Significato e Rivendicazioni": attention
// computed directly in the latent space.  With the uniform quantizer a
// latent coordinate is yhat_c = Delta_c (code_c - 2^(b-1) + 1/2), and a code
// is the sum of its bit planes, code_c = sum_k 2^k bit_{c,k}.  So with plane
// r = (c, k) of the stream (the stream's own word order, o_c + k),
//   s_j(t) = sum_c qt_jc yhat_c(t) = sum_r V_jr bit_r(t) + C_j,
//     V_jr = qt_jc Delta_c 2^k,   C_j = sum_c qt_jc Delta_c (1/2 - 2^(b_c-1)),
//   sum_t p_j(t) code_c(t) = sum_k 2^k S_{j,(c,k)},  S_jr = sum_t p_j(t) bit_r(t),
// and both contractions are products of a 0/1 matrix -- the packed words
// exactly as stored -- with dense fp16 operands.  No code is ever unpacked.
//
// A bit enters the tensor core as a normal fp16 number.  One byte permute
// moves byte b of a stream word into the high byte of a 16-bit half, so
// token 8 b + j of the word sits at bit q = 8 + j of that half; masking out
// every other bit and ORing a per-position base leaves base_q + bit * d_q:
//   q = 8, 9:    base 2^-14 (exponent 1), bit in the mantissa: d = 2^-16, 2^-15
//   q = 10..14:  base 0, bit alone in the exponent: 2^-14, 2^-13, 2^-11, 2^-7, 2
//   q = 15:      base 1.0, bit in the sign: 1 - 2 bit
// (subnormal operands are avoided: the tensor cores round them coarsely).
// Every row (scores) or token (P V) of a product then carries one known
// affine map of its bits, undone after the MMA or folded into the other
// operand beforehand.
//
//  * Scores (per 32-token group, one warp): m16n8k16 with M = 16 tokens,
//    K = 16 planes, N = 8 = 4 query heads x (hi, lo) fp16 halves of V.  An A
//    register holds two planes of one token: one byte permute of the two
//    plane words per byte, then one mask-and-base per register.  A thread's
//    rows are tokens g, 8 + g, 16 + g, 24 + g, all at q = 8 + g, so
//    sum_r V_r bit_r = (acc - base_q sum_r V_r) / d_q.
//  * P V: m16n8k16 with M = 16 planes, K = 16 tokens, N = 8 = heads x (hi,
//    lo) of P.  An A register holds one plane of tokens s and s + 16: one
//    byte permute of the plane word (bytes 0 and 2, or 1 and 3), then one
//    mask-and-base.  P enters as P' = p c / d_q, so a product is
//    c (p bit + p base_q / d_q); the second term is the same for every plane
//    and is removed with kappa = sum_t p base_q / d_q.
//
// One CTA (8 warps) per (context split, kv head, batch).  Tiles of 256
// tokens (one 32-token group per warp) arrive by bulk copy (the group
// records of K and V, 32 R bytes each) into a ring of shared-memory stages.
// Per tile: each warp scores its group over all K planes; the block takes
// the running maximum per head (barrier 1); each warp writes its tokens'
// probabilities as fp16 hi/lo pairs (barrier 2); each warp then accumulates
// P V for its own slice of the V planes (m-tiles w, w + 8, ...) over the
// whole tile.  The split's (m, l, sum_t p z) per head go to the workspace
// (z = code - 2^(b-1)); the combine kernel of attn.cu merges splits,
// dequantizes and rotates by the V basis.
#include "spectra_internal.cuh"
#include "tc_common.cuh"

#include <cuda_fp16.h>
#include <math.h>

#include <type_traits>

namespace spectra {

namespace {

using namespace tc;

constexpr int D = 128;
constexpr int kGmax = 4;                  // query heads per kv head
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int TT = 32 * kWarps;           // tokens per tile: one group per warp
constexpr int kMaxStages = 4;
constexpr int PSTR = 24;                  // u32 per (group, column) row of the P tile
constexpr int kImgKb = 8 * D / 16;        // k-blocks of the score weights at the widest record
constexpr uint32_t kImgBytesPerHead = kImgKb * 32 * 8;
constexpr uint64_t kWaitNs = 2000000000ull;

// D (16x8 f32) += A (16x16 f16, row) * B (16x8 f16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// ------------------------------------------------------------------ prep
// Per (batch, kv head): qt_j = scale * B_K^T q_j; W_jc = qt_jc Delta_c;
// the score weights V_jr = W_jc 2^k of every plane r = (c, k) as fp16 hi and
// lo parts, laid out as the m16n8k16 B fragments of each 16-plane k-block
// ([kb][lane][b0, b1], column n = 2 j + (0 hi, 1 lo), zero for planes past
// the record and for heads >= G); bias[8] = {C_0..3, sum_r V_0r..V_3r}
// (the sums taken over the fp16 parts exactly as the MMA sees them).
__global__ void __launch_bounds__(kGmax * D)
attn_tc_prep_kernel(PlanView kp, const void* __restrict__ q, int q_dt, int Hq, int G, float scale,
                    uint32_t* __restrict__ img, float* __restrict__ bias)
{
    const int bh = blockIdx.x, Hkv = kp.heads, h = bh % Hkv, b = bh / Hkv;
    const int tid = threadIdx.x, c = tid % D, j = tid / D;   // channel, query head of the group
    extern __shared__ float Bs[];                 // [D][D] basis of head h
    __shared__ float qs[kGmax][D];
    __shared__ float red[2][kGmax][4];
    const int R = min(kp.rec_bits[h], kp.max_rec_bits);
    const int nkb = (max(R, 1) + 15) / 16;
    uint32_t* im = img + size_t(bh) * (kImgBytesPerHead / 4);
    for (int e = tid; e < nkb * 64; e += kGmax * D) im[e] = 0u;
    {
        const float4* src = reinterpret_cast<const float4*>(kp.basis_mat + size_t(h) * D * D);
        float4* dst = reinterpret_cast<float4*>(Bs);
        for (int e = tid; e < D * D / 4; e += kGmax * D) dst[e] = src[e];
    }
    qs[j][c] = (j < G) ? load_elem(q, q_dt, (int64_t(b) * Hq + h * G + j) * D + c) : 0.f;
    __syncthreads();
    float qt = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; ++i) qt = fmaf(Bs[i * D + c], qs[j][i], qt);
    const int bits = kp.bits[size_t(h) * D + c];
    const int off = kp.chan_off[size_t(h) * D + c];
    const float delta = kp.rscale[size_t(h) * D + c];
    const float w = (bits > 0 && j < G && kp.rec_bits[h] <= kp.max_rec_bits) ? qt * scale * delta : 0.f;
    float cj = (bits > 0) ? w * (0.5f - float(1 << (bits - 1))) : 0.f;
    float vs = 0.f;
    __half* ih = reinterpret_cast<__half*>(im);
    for (int k = 0; k < bits && w != 0.f; ++k) {
        const float v = w * float(1 << k);
        const __half hi = __float2half_rn(v);
        const __half lo = __float2half_rn(v - __half2float(hi));
        vs += __half2float(hi) + __half2float(lo);
        const int r = off + k, kb = r >> 4, kk = r & 15;
        const int reg = kk >> 3, tg = (kk & 7) >> 1, hf = kk & 1;
        const int lane_hi = (2 * j) * 4 + tg, lane_lo = (2 * j + 1) * 4 + tg;
        ih[((kb * 32 + lane_hi) * 2 + reg) * 2 + hf] = hi;
        ih[((kb * 32 + lane_lo) * 2 + reg) * 2 + hf] = lo;
    }
    for (int o = 16; o; o >>= 1) {
        cj += __shfl_xor_sync(0xffffffffu, cj, o);
        vs += __shfl_xor_sync(0xffffffffu, vs, o);
    }
    if ((c & 31) == 0) {
        red[0][j][c >> 5] = cj;
        red[1][j][c >> 5] = vs;
    }
    __syncthreads();
    if (tid < 2 * kGmax) {
        const int which = tid / kGmax, jj = tid % kGmax;
        bias[size_t(bh) * 8 + tid] = red[which][jj][0] + red[which][jj][1] + red[which][jj][2] + red[which][jj][3];
    }
}

// ------------------------------------------------------------------ split
struct AttnTcParams {
    PlanView kp, vp;
    int Hq, G, nsplit, split_len, stages;
    int64_t ctx;
    const uint8_t* kc;
    const uint8_t* vc;
    int64_t sstride;
    const uint32_t* img;
    const float* bias;
    float* part;
    uint32_t kst, vst;       // bytes of one stage's K / V words (32 R, rounded to 16) plus padding
};

struct TcSmem {
    uint32_t img, stage, pt, wmax, red, bars, total;
};

__host__ __device__ inline TcSmem tc_smem_layout(int stages, uint32_t kst, uint32_t vst, int nkb)
{
    TcSmem L;
    uint32_t o = 0;
    L.img = o;   o += uint32_t(nkb) * 256;
    L.stage = o; o += uint32_t(stages) * (kst + vst);
    L.pt = o;    o += kWarps * 8 * PSTR * 4;
    L.wmax = o;  o += kWarps * kGmax * 4;
    L.red = o;   o += 2 * kWarps * kGmax * 4;
    L.bars = o;  o += 8 * kMaxStages + 16;
    L.total = o;
    return L;
}

// MTV: V m-tiles per warp (ceil(R_V / 128)).  A record with an even number
// of words starts every group's words 8-byte aligned in shared memory (64-bit
// loads); odd records take 32-bit loads.
// Records up to 256 V planes (MTV <= 2) run three CTAs per SM (24 warps hide
// the latency of the shared-memory loads and MMAs), wider ones two.
template <int MTV>
__global__ void __launch_bounds__(kThreads, MTV <= 2 ? 3 : 2)
attn_tc_split_kernel(AttnTcParams P)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int Hkv = P.kp.heads, G = P.G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, tig = lane & 3;
    const int bh = b * Hkv + h;
    const int S = P.stages;

    const int nkb = (P.kp.max_rec_bits + 15) / 16;
    const TcSmem L = tc_smem_layout(S, P.kst, P.vst, max(nkb, 1));
    uint2* wimg = reinterpret_cast<uint2*>(smem + L.img);
    uint8_t* stage = smem + L.stage;
    uint32_t* pt = reinterpret_cast<uint32_t*>(smem + L.pt);
    float* wmax = reinterpret_cast<float*>(smem + L.wmax);
    float* red = reinterpret_cast<float*>(smem + L.red);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kMaxStages);

    const int64_t t_begin = int64_t(split) * P.split_len;
    const int64_t t_end = min(P.ctx, t_begin + P.split_len);
    const int ntiles = int((t_end - t_begin + TT - 1) / TT);
    // records longer than the plans' bound are not read (the streams were sized by the bound)
    const int RK0 = P.kp.rec_bits[h], RV0 = P.vp.rec_bits[h];
    const int RK = RK0 <= P.kp.max_rec_bits ? RK0 : 0, RV = RV0 <= P.vp.max_rec_bits ? RV0 : 0;
    const int nkbh = (RK + 15) / 16, nmtv = (RV + 15) / 16;
    const int64_t sid = int64_t(b) * Hkv + h;
    const uint8_t* ks = P.kc + sid * P.sstride;
    const uint8_t* vs = P.vc + sid * P.sstride;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        abort_flag[0] = 0;
        abort_flag[1] = 0;
        fence_mbar_init();
    }
    {
        const uint2* src = reinterpret_cast<const uint2*>(P.img + size_t(bh) * (kImgBytesPerHead / 4));
        for (int e = tid; e < nkbh * 32; e += kThreads) wimg[e] = src[e];
    }
    __syncthreads();

    // bulk copies of tile `tile` into its stage: the groups' K and V words
    auto issue = [&](int tile) {
        const int s = tile % S;
        const int64_t t0 = t_begin + int64_t(tile) * TT;
        const int64_t ng = min(int64_t(TT / 32), (t_end - t0 + 31) / 32);
        const uint32_t kb = uint32_t((ng * 4 * RK + 15) / 16 * 16), vb = uint32_t((ng * 4 * RV + 15) / 16 * 16);
        uint8_t* dst = stage + size_t(s) * (P.kst + P.vst);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&full[s], kb + vb);
        if (kb) bulk_load(dst, ks + (t0 / 32) * 4 * RK, kb, &full[s]);
        if (vb) bulk_load(dst + P.kst, vs + (t0 / 32) * 4 * RV, vb, &full[s]);
    };
    int issued = 0;                            // tiles whose copies were issued (thread 0)
    if (tid == 0)
        for (; issued < min(S - 1, ntiles); ++issued) issue(issued);

    // score weights and constants of head tig (this thread's accumulator column pair)
    const float cj = P.bias[size_t(bh) * 8 + tig];
    const float vsum = P.bias[size_t(bh) * 8 + 4 + tig];
    const bool head_ok = tig < G;
    // every row of this thread sits at bit q = 8 + g8 of its half
    const uint32_t mk = (1u << (8 + g8)) | (1u << (24 + g8));
    const uint32_t bk = g8 < 2 ? 0x04000400u : g8 == 7 ? 0x3C003C00u : 0u;
    const float dq = g8 == 0 ? 0x1p-16f : g8 == 1 ? 0x1p-15f : g8 == 2 ? 0x1p-14f : g8 == 3 ? 0x1p-13f
                   : g8 == 4 ? 0x1p-11f : g8 == 5 ? 0x1p-7f : g8 == 6 ? 2.f : -2.f;
    const float bq = g8 < 2 ? 0x1p-14f : g8 == 7 ? 1.f : 0.f;
    const float rs = 1.f / dq;                      // exact: powers of two and -1/2
    const float bsum = bq * vsum;
    // P V: slot 0 holds token pairs at q = 8 + tig, slot 1 at q = 12 + tig
    const uint32_t mv0 = (1u << (8 + tig)) | (1u << (24 + tig));
    const uint32_t mv1 = (1u << (12 + tig)) | (1u << (28 + tig));
    const uint32_t bv0 = tig < 2 ? 0x04000400u : 0u;
    const uint32_t bv1 = tig == 3 ? 0x3C003C00u : 0u;
    // P' = p c / d_q with c = 1/2 for this thread's tokens (q = 8 + g8);
    // beta_q = base_q / d_q feeds kappa
    const float pscale = 0.5f * rs;
    const float beta = bq * rs;
    float acc[MTV][4];
#pragma unroll
    for (int i = 0; i < MTV; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m_run = -INFINITY, l_part = 0.f, k_part = 0.f;
    bool aborted = false;

    for (int tile = 0; tile < ntiles; ++tile) {
        const int s = tile % S;
        const int64_t t0 = t_begin + int64_t(tile) * TT;
        const uint8_t* stg = stage + size_t(s) * (P.kst + P.vst);
        // a give-up is made warp-uniform: the warp-synchronous MMAs below run
        // on whole warps or not at all
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[s], uint32_t(tile / S) & 1u, abort_flag, kWaitNs));

        // ---- scores of this warp's group (tokens t0 + 32 warp ...)
        const int64_t tg0 = t0 + 32 * warp;
        float sc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // tokens g8, g8+8, 16+g8, 24+g8
        if (ok && tg0 < t_end && RK > 0) {
            uint32_t* kwm = reinterpret_cast<uint32_t*>(const_cast<uint8_t*>(stg)) + warp * RK;
            // an even record: merge the group's plane pairs in place, once --
            // words (2i, 2i + 1) become (low halves of both, high halves of
            // both), the tokens 0..15 / 16..31 views the score tiles use (an odd
            // record keeps its words and merges inside the k-loop)
            if (!(RK & 1)) {
                for (int pi = lane; pi < RK / 2; pi += 32) {
                    const uint2 u = reinterpret_cast<const uint2*>(kwm)[pi];
                    reinterpret_cast<uint2*>(kwm)[pi] = make_uint2(__byte_perm(u.x, u.y, 0x5410),
                                                                   __byte_perm(u.x, u.y, 0x7632));
                }
                __syncwarp();
            }
            const uint32_t* kw = kwm;
            // Three accumulator chains per m-tile: the first k-block (the widest
            // channels' planes, which carry the largest terms) alone, then odd and
            // even k-blocks.  The tensor core truncates each accumulation to the
            // running sum's precision; short chains keep that error relative to
            // small partial sums.
            float aA[4] = {0.f, 0.f, 0.f, 0.f}, aB[4] = {0.f, 0.f, 0.f, 0.f};
            float aA2[4] = {0.f, 0.f, 0.f, 0.f}, aB2[4] = {0.f, 0.f, 0.f, 0.f};
            float aA0[4] = {0.f, 0.f, 0.f, 0.f}, aB0[4] = {0.f, 0.f, 0.f, 0.f};
            auto kloop = [&](auto even_tag) {
                constexpr bool EV = decltype(even_tag)::value;
                // one k-block into the chain (ca, cb): l / h hold tokens 0..15 /
                // 16..31 of planes (2 tig, 2 tig + 1) and (2 tig + 8, 2 tig + 9);
                // tokens 0..7 (16..23) reach the high bytes of the halves by a left
                // shift of 8 (a multiply, so it can issue on the FMA pipe), tokens
                // 8..15 (24..31) are already there
                auto kstep = [&](int kb, float (&ca)[4], float (&cb)[4]) {
                    const uint2 wb = wimg[kb * 32 + lane];
                    uint32_t l01, h01, l89, h89;
                    if constexpr (EV) {
                        const uint2 u = *reinterpret_cast<const uint2*>(kw + 16 * kb + 2 * tig);
                        const uint2 v = *reinterpret_cast<const uint2*>(kw + 16 * kb + 2 * tig + 8);
                        l01 = u.x; h01 = u.y; l89 = v.x; h89 = v.y;
                    } else {
                        const uint32_t p0 = kw[16 * kb + 2 * tig], p1 = kw[16 * kb + 2 * tig + 1];
                        const uint32_t p8 = kw[16 * kb + 2 * tig + 8], p9 = kw[16 * kb + 2 * tig + 9];
                        l01 = __byte_perm(p0, p1, 0x5410); h01 = __byte_perm(p0, p1, 0x7632);
                        l89 = __byte_perm(p8, p9, 0x5410); h89 = __byte_perm(p8, p9, 0x7632);
                    }
                    const uint32_t a[4] = {((l01 * 256u) & mk) | bk, (l01 & mk) | bk,
                                           ((l89 * 256u) & mk) | bk, (l89 & mk) | bk};
                    const uint32_t c[4] = {((h01 * 256u) & mk) | bk, (h01 & mk) | bk,
                                           ((h89 * 256u) & mk) | bk, (h89 & mk) | bk};
                    mma16816(ca, a, wb.x, wb.y);
                    mma16816(cb, c, wb.x, wb.y);
                };
                kstep(0, aA0, aB0);
                int kb = 1;
#pragma unroll 1
                for (; kb + 1 < nkbh; kb += 2) {
                    kstep(kb, aA2, aB2);
                    kstep(kb + 1, aA, aB);
                }
                if (kb < nkbh) kstep(kb, aA2, aB2);
            };
            if (RK & 1) kloop(std::false_type{});
            else kloop(std::true_type{});
            float r[4];
            r[0] = aA0[0] + ((aA[0] + aA2[0]) + (aA0[1] + (aA[1] + aA2[1])));
            r[1] = aA0[2] + ((aA[2] + aA2[2]) + (aA0[3] + (aA[3] + aA2[3])));
            r[2] = aB0[0] + ((aB[0] + aB2[0]) + (aB0[1] + (aB[1] + aB2[1])));
            r[3] = aB0[2] + ((aB[2] + aB2[2]) + (aB0[3] + (aB[3] + aB2[3])));
            const int tok[4] = {g8, g8 + 8, 16 + g8, 24 + g8};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float v = (r[e] - bsum) * rs;
                sc[e] = (head_ok && tg0 + tok[e] < t_end) ? v + cj : -INFINITY;
            }
        } else if (ok && tg0 < t_end && head_ok) {
            // zero-bit K record: every score is the constant C_j
            const int tok[4] = {g8, g8 + 8, 16 + g8, 24 + g8};
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[e] = (tg0 + tok[e] < t_end) ? cj : -INFINITY;
        }
        float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (g8 == 0) wmax[warp * kGmax + tig] = mx;
        if (__syncthreads_or(!ok)) {          // barrier 1: tile maxima; stage of tile - 1 free
            aborted = true;
            break;
        }
        if (tid == 0 && issued < ntiles) issue(issued++);

        float tmax = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) tmax = fmaxf(tmax, wmax[w * kGmax + tig]);
        const float m_new = fmaxf(m_run, tmax);
        const float alpha = (m_run == -INFINITY) ? 0.f : __expf(m_run - m_new);
        m_run = m_new;
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = (sc[e] == -INFINITY) ? 0.f : __expf(sc[e] - m_new);
        const float psum = (p[0] + p[1]) + (p[2] + p[3]);
        l_part = l_part * alpha + psum;
        k_part = k_part * alpha + beta * psum;
        {
            // pairs (g8, 16 + g8) -> k-step 0, (8 + g8, 24 + g8) -> k-step 1; pair index g8
            uint32_t* prow = pt + (warp * 8 + 2 * tig) * PSTR + (g8 & 3) * 2 + (g8 >> 2);
#pragma unroll
            for (int ksp = 0; ksp < 2; ++ksp) {
                const float x0 = p[ksp] * pscale, x1 = p[2 + ksp] * pscale;
                const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
                prow[ksp * 8] = pack_half2(__half2float(h0), __half2float(h1));
                prow[PSTR + ksp * 8] = pack_half2(x0 - __half2float(h0), x1 - __half2float(h1));
            }
        }
#pragma unroll
        for (int i = 0; i < MTV; ++i) {
            acc[i][0] *= alpha; acc[i][1] *= alpha; acc[i][2] *= alpha; acc[i][3] *= alpha;
        }
        __syncthreads();                       // barrier 2: the tile's P in shared memory

        // ---- P V over this warp's V planes, all groups of the tile
        if (RV > 0) {
            const uint32_t* vwt = reinterpret_cast<const uint32_t*>(stg + P.kst);
            const int ngv = int(min(int64_t(TT / 32), (t_end - t0 + 31) / 32));
            // two groups at a time into a fresh accumulator per m-tile, added to
            // the running sums with rounding: a plane's sum is scaled by up to
            // 2^7 in the output, so the tensor core's truncating accumulation
            // must not run across the whole split.  Tokens s, s + 16 with s < 8
            // reach the high bytes of the halves by a left shift of 8 (bytes 0,
            // 2); s >= 8 are already there (bytes 1, 3).
            auto vloop = [&](auto even_tag) {
                constexpr bool EV = decltype(even_tag)::value;
                auto pfrag = [&](int g, uint2& pb0, uint2& pb1) {
                    const uint2* pg = reinterpret_cast<const uint2*>(pt + (g * 8 + g8) * PSTR) + tig;
                    pb0 = pg[0];
                    pb1 = pg[4];
                };
                auto vstep = [&](int g, int i, const uint2& pb0, const uint2& pb1, float (&t)[4]) {
                    const uint32_t* vw = vwt + g * RV + 16 * (warp + kWarps * i) + 2 * g8;
                    uint32_t w0, w1;
                    if constexpr (EV) {
                        const uint2 u = *reinterpret_cast<const uint2*>(vw);
                        w0 = u.x; w1 = u.y;
                    } else {
                        w0 = vw[0]; w1 = vw[1];
                    }
                    const uint32_t x0 = w0 * 256u, x1 = w1 * 256u;
                    const uint32_t a0[4] = {(x0 & mv0) | bv0, (x1 & mv0) | bv0, (x0 & mv1) | bv1, (x1 & mv1) | bv1};
                    const uint32_t a1[4] = {(w0 & mv0) | bv0, (w1 & mv0) | bv0, (w0 & mv1) | bv1, (w1 & mv1) | bv1};
                    mma16816(t, a0, pb0.x, pb0.y);
                    mma16816(t, a1, pb1.x, pb1.y);
                };
                int g = 0;
#pragma unroll 1
                for (; g + 1 < ngv; g += 2) {
                    uint2 pa0, pa1, pc0, pc1;
                    pfrag(g, pa0, pa1);
                    pfrag(g + 1, pc0, pc1);
#pragma unroll
                    for (int i = 0; i < MTV; ++i) {
                        if (warp + kWarps * i < nmtv) {
                            float t[4] = {0.f, 0.f, 0.f, 0.f};
                            vstep(g, i, pa0, pa1, t);
                            vstep(g + 1, i, pc0, pc1, t);
                            acc[i][0] += t[0]; acc[i][1] += t[1]; acc[i][2] += t[2]; acc[i][3] += t[3];
                        }
                    }
                }
                if (g < ngv) {
                    uint2 pa0, pa1;
                    pfrag(g, pa0, pa1);
#pragma unroll
                    for (int i = 0; i < MTV; ++i) {
                        if (warp + kWarps * i < nmtv) {
                            float t[4] = {0.f, 0.f, 0.f, 0.f};
                            vstep(g, i, pa0, pa1, t);
                            acc[i][0] += t[0]; acc[i][1] += t[1]; acc[i][2] += t[2]; acc[i][3] += t[3];
                        }
                    }
                }
            };
            if (RV & 1) vloop(std::false_type{});
            else vloop(std::true_type{});
        }
    }

    if (aborted) {
        // let the copies in flight land before the CTA exits (each stage's
        // last issued phase, bounded), then report through the plan's status
        if (tid == 0) {
            for (int st = 0; st < S; ++st) {
                int last = -1;
                for (int t = st; t < issued; t += S) last = t;
                if (last >= 0) mbar_wait(&full[st], uint32_t(last / S) & 1u, abort_flag + 1, 100000000ull);
            }
            P.kp.status[h] = -SPECTRA_ERR_TIMEOUT;
        }
        return;
    }
    __syncthreads();   // every warp is past its last read of the stages and the P tile

    // ---- split partials: S_jr (planes), l_j, then o_jc = sum_k 2^k S_j,(c,k) - 2^(b-1) l_j
    float* Ssm = reinterpret_cast<float*>(stage);           // [kGmax][R_V] (reuses the stages)
#pragma unroll
    for (int i = 0; i < MTV; ++i) {
        const int mt = warp + kWarps * i;
        if (mt < nmtv) {
            const int r = 16 * mt + 2 * g8;
            if (r < RV) Ssm[tig * RV + r] = 2.f * (acc[i][0] + acc[i][1]);
            if (r + 1 < RV) Ssm[tig * RV + r + 1] = 2.f * (acc[i][2] + acc[i][3]);
        }
    }
    float lsum = l_part, ksum = k_part;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
        ksum += __shfl_xor_sync(0xffffffffu, ksum, o);
    }
    if (g8 == 0) {
        red[warp * kGmax + tig] = lsum;
        red[(kWarps + warp) * kGmax + tig] = ksum;
    }
    if (g8 == 0 && warp == 0) wmax[tig] = m_run;
    __syncthreads();
    for (int e = tid; e < kGmax * D; e += kThreads) {
        const int j = e / D, c = e % D;
        if (j >= G) continue;
        float l = 0.f, kap = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            l += red[w * kGmax + j];
            kap += red[(kWarps + w) * kGmax + j];
        }
        const int bc = P.vp.bits[size_t(h) * D + c];
        float o = 0.f;
        if (bc > 0 && RV > 0) {
            const int oc = P.vp.chan_off[size_t(h) * D + c];
            for (int k = bc - 1; k >= 0; --k) o = fmaf(o, 2.f, Ssm[j * RV + oc + k]);
            // each plane sum carries kappa: sum_k 2^k kappa = (2^b - 1) kappa
            o -= float((1 << bc) - 1) * kap + float(1 << (bc - 1)) * l;
        }
        float* bp = P.part + ((int64_t(b) * P.Hq + h * G + j) * P.nsplit + split) * (D + 2);
        bp[2 + c] = o;
        if (c == 0) {
            bp[0] = wmax[j];
            bp[1] = l;
        }
    }
}

}  // namespace

// Workspace of the tensor-core path (inside attn_workspace_bytes):
// [score weight images (B Hkv x 16 KB) | constants (B Hkv x 8 f32)].
size_t attn_tc_extra_bytes(int B, int Hkv)
{
    return align256(size_t(kImgBytesPerHead) * B * Hkv) + align256(sizeof(float) * 8 * size_t(B) * Hkv);
}

spectra_status launch_attn_tc(const spectra_plan* kplan, const spectra_plan* vplan, const void* q, int q_dt, int B,
                              int Hq, const uint8_t* kc, const uint8_t* vc, int64_t sstride, int64_t ctx,
                              float scale, float* part, int nsplit, int split_len, void* extra,
                              cudaStream_t s, bool* done)
{
    *done = false;
    const int Hkv = kplan->heads, G = Hq / Hkv;
    if (kplan->head_dim != D || G > kGmax) return SPECTRA_OK;
    if (kplan->basis != SPECTRA_BASIS_EIGEN || vplan->basis != SPECTRA_BASIS_EIGEN) return SPECTRA_OK;
    if (kplan->quant != SPECTRA_Q_UNIFORM3S || vplan->quant != SPECTRA_Q_UNIFORM3S) return SPECTRA_OK;
    if (split_len % TT != 0) return SPECTRA_OK;
    AttnTcParams P;
    P.kp = make_view(kplan);
    P.vp = make_view(vplan);
    P.Hq = Hq;
    P.G = G;
    P.nsplit = nsplit;
    P.split_len = split_len;
    P.ctx = ctx;
    P.kc = kc;
    P.vc = vc;
    P.sstride = sstride;
    uint32_t* img = static_cast<uint32_t*>(extra);
    float* bias = reinterpret_cast<float*>(static_cast<uint8_t*>(extra) +
                                           align256(size_t(kImgBytesPerHead) * B * Hkv));
    P.img = img;
    P.bias = bias;
    P.part = part;
    const int RKm = kplan->max_rec_bits, RVm = vplan->max_rec_bits;
    // one stage: 8 groups of each record, rounded to 16 bytes, plus 64 bytes
    // for the reads of the last k-block / m-tile past the record
    P.kst = uint32_t((32 * RKm + 15) / 16 * 16 + 64);
    P.vst = uint32_t((32 * RVm + 15) / 16 * 16 + 64);
    const int nkb = max((RKm + 15) / 16, 1);
    // V-side partial sums reuse the stages: kGmax x R_V floats must fit
    auto total = [&](int st) { return tc_smem_layout(st, P.kst, P.vst, nkb).total; };
    const int mtv = (((RVm + 15) / 16) + kWarps - 1) / kWarps;
    // stages that let the kernel's CTAs per SM fit (228 KB per SM, 1 KB of it per CTA reserved)
    const uint32_t fit = mtv <= 2 ? 75 * 1024 : 113 * 1024;
    int st = kMaxStages;
    while (st > 2 && total(st) > fit) --st;
    if (total(st) > 227 * 1024) return SPECTRA_OK;
    if (size_t(st) * (P.kst + P.vst) < sizeof(float) * kGmax * size_t(RVm)) return SPECTRA_OK;
    P.stages = st;
    const size_t sm = total(st);
    if (spectra_status e = set_smem(attn_tc_prep_kernel, sizeof(float) * D * D)) return e;
    attn_tc_prep_kernel<<<B * Hkv, kGmax * D, sizeof(float) * D * D, s>>>(P.kp, q, q_dt, Hq, G, scale, img, bias);
    if (spectra_status e = cuda_status(cudaGetLastError())) return e;
    dim3 grid(nsplit, Hkv, B);
    auto launch = [&](auto kern) -> spectra_status {
        if (spectra_status e = set_smem(kern, sm)) return e;
        kern<<<grid, kThreads, sm, s>>>(P);
        return cuda_status(cudaGetLastError());
    };
    spectra_status e;
    if (mtv <= 1) e = launch(attn_tc_split_kernel<1>);
    else if (mtv <= 2) e = launch(attn_tc_split_kernel<2>);
    else if (mtv <= 4) e = launch(attn_tc_split_kernel<4>);
    else e = launch(attn_tc_split_kernel<8>);
    if (e) return e;
    *done = true;
    return SPECTRA_OK;
}

}  // namespace spectra
