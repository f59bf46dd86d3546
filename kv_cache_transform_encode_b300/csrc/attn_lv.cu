// attn_lv.cu -- decode-step attention over packed K/V streams on the tensor
// cores for every quantizer and either basis (head_dim 128, up to eight
// query heads per kv head): each code is looked up as its dequantized level
// and both contractions run as mma.sync over bf16 (hi, lo) pairs.
//
// "Sintesi Tecnica: SPECTRA", "Significato e Rivendicazioni": attention
// computed in the latent space.  A latent coordinate of token t is
//   yhat_c(t) = a_c n_t lev_{b_c}[code_c(t)],
// lev_b the width-b level table (uniform quantizer: code + 1/2 - 2^(b-1);
// Gaussian Lloyd-Max: the ascending levels), a_c the channel scale (the
// uniform step Delta_c, sigma_c of an eigenbasis Lloyd-Max plan, 1/sqrt(d)
// for an RWHT Lloyd-Max plan) and n_t the token scale (||x_t|| for RWHT
// Lloyd-Max plans -- "Technisch Overzicht ...", "Experimentele Opstelling":
// the rotated vector is coded at its own scale -- else 1).  So
//   s_j(t) = n_t sum_c (qt_jc a_c) lev(code_c(t)),
//   o_jc   = a_c sum_t (p_j(t) n_t) lev(code_c(t)).
//
// A level enters the tensor core as a bf16 (hi, lo) pair in one 32-bit
// register, exactly as a table entry stores it, so one shared-memory load
// per code gives one A-fragment register.  K runs over (code, hi|lo) pairs;
// the other operand (qt a, or p n) is split into bf16 hi and lo parts along
// N and repeated over the pair, so every product keeps about 16 significant
// bits on both sides and the fp32 accumulators see no subnormal operand.
//
//  * Scores, per 32-token group: m16n8k16 with M = 16 tokens, K = 8
//    channels x (hi, lo), N = 4 query heads x (hi, lo).  Thread (g, tg) of
//    a warp reads channels c = tg (mod 4) at tokens g, g+8, g+16, g+24: per
//    plane word one rotate and one masked OR drop the four tokens' bits of
//    plane k in the four bytes of a register -- four codes at once.
//  * P V: M = 16 channels, K = 8 tokens x (hi, lo), N = heads x (hi, lo);
//    thread (g, tg) reads channels c = g (mod 8) at tokens tg (mod 4).
//
// Codes are assembled times 4 (plane k at bit k + 2 of its byte) and every
// width w <= 6 has its level table in a 256-byte slot of its own, so a
// single byte permute of (codes, slot address) is the lookup address.  The
// planes of a step (8 or 16 channels) are read by one straight-line chain
// for the step's widest width, entered by a single jump; a narrower
// channel's extra words (its neighbour's planes, or the slot padding) are
// masked off.  Steps with a 7- or 8-bit channel take the same chain with
// plain codes and a computed address.
//
// The warps are independent: warp w of a CTA takes every eighth 32-token
// group of the CTA's context split and stages its records through two
// cp.async slots of its own, K in one and V in the other: the next group's K
// record (and RWHT norms) lands during this group's softmax and P V, its V
// record during the next group's scores.  Each warp keeps its own online
// softmax (m, l) and value sums (in shared memory, updated once per 16
// channels with the softmax rescale folded in).  The eight states merge once,
// at the end of the split, into the partials the combine kernel of attn.cu
// merges over splits and rotates by the V basis.  Scores are kept in log2
// units (log2 e folded into the weights); the partial's m is converted back.
#include "spectra_internal.cuh"

#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <type_traits>

namespace spectra {

namespace {

constexpr int D = 128;
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kSlot = 64;                  // words of a 256-byte table slot
constexpr int kTabWords = 13 * kSlot;      // widths 0..6 one slot each, width 7 two, width 8 four
constexpr int kPad = 8;                    // slot words past each record (reads up to 7 past a channel)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kQjlScale = 1.25331413731550025f / float(D);   // sqrt(pi / 2) / m, m = d sketch rows

// first word of width w's table (width 0: one zero entry)
__host__ __device__ constexpr int tab_word(int w) { return w <= 7 ? w * kSlot : 9 * kSlot; }

// D (16x8 f32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t bf16_bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
__device__ __forceinline__ float bf16_val(uint32_t u) { return __uint_as_float(u << 16); }

// (hi, lo) of v: hi = bf16(v) in the low half, lo = bf16(v - hi) in the high half
__device__ __forceinline__ uint32_t bf16_pair(float v)
{
    const uint32_t hi = bf16_bits(v);
    return hi | (bf16_bits(v - bf16_val(hi)) << 16);
}
// part y (0 hi, 1 lo) of v in both halves
__device__ __forceinline__ uint32_t bf16_part_dup(float v, int y)
{
    const uint32_t hi = bf16_bits(v);
    const uint32_t u = y ? bf16_bits(v - bf16_val(hi)) : hi;
    return u | (u << 16);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return uint32_t(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// R words of a group record into shared memory (16-byte copies when both
// ends allow them); the warp's lanes split the words
__device__ __forceinline__ void copy_record(uint32_t* dst, const uint8_t* src, int R, int lane)
{
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && (R & 3) == 0) {
        for (int e = lane; e < R / 4; e += 32) cp_async16(smem_u32(dst + 4 * e), src + 16 * e);
    } else {
        for (int e = lane; e < R; e += 32) cp_async4(smem_u32(dst + e), src + 4 * e);
    }
}

// Plane K of two channels (words p0[K], p1[K]) for the four tokens sh + 8 m:
// bit sh + 8 m of the word goes to bit 8 m + K + E of x.
template <int E, int K>
__device__ __forceinline__ void plane2(const uint32_t* p0, const uint32_t* p1, int sh, uint32_t& x0, uint32_t& x1)
{
    if constexpr (K + E < 8) {
        const uint32_t v0 = p0[K], v1 = p1[K];
        x0 |= __funnelshift_r(v0, v0, sh - K - E) & (0x01010101u << (K + E));
        x1 |= __funnelshift_r(v1, v1, sh - K - E) & (0x01010101u << (K + E));
    }
}
// planes 0 .. n-1 of two channels (n warp-uniform, at most 8): one jump into
// a straight-line chain
template <int E>
__device__ __forceinline__ void planes2(const uint32_t* p0, const uint32_t* p1, int n, int sh, uint32_t& x0,
                                        uint32_t& x1)
{
    x0 = 0u;
    x1 = 0u;
    switch (n) {
    case 8: plane2<E, 7>(p0, p1, sh, x0, x1); [[fallthrough]];
    case 7: plane2<E, 6>(p0, p1, sh, x0, x1); [[fallthrough]];
    case 6: plane2<E, 5>(p0, p1, sh, x0, x1); [[fallthrough]];
    case 5: plane2<E, 4>(p0, p1, sh, x0, x1); [[fallthrough]];
    case 4: plane2<E, 3>(p0, p1, sh, x0, x1); [[fallthrough]];
    case 3: plane2<E, 2>(p0, p1, sh, x0, x1); [[fallthrough]];
    case 2: plane2<E, 1>(p0, p1, sh, x0, x1); [[fallthrough]];
    case 1: plane2<E, 0>(p0, p1, sh, x0, x1); [[fallthrough]];
    default: break;
    }
}
// the same for tokens sh + 8 m (x?0) and sh + 4 + 8 m (x?1)
template <int E, int K>
__device__ __forceinline__ void plane4(const uint32_t* p0, const uint32_t* p1, int sh, uint32_t (&x)[4])
{
    if constexpr (K + E < 8) {
        const uint32_t v0 = p0[K], v1 = p1[K], m = 0x01010101u << (K + E);
        x[0] |= __funnelshift_r(v0, v0, sh - K - E) & m;
        x[1] |= __funnelshift_r(v0, v0, sh + 4 - K - E) & m;
        x[2] |= __funnelshift_r(v1, v1, sh - K - E) & m;
        x[3] |= __funnelshift_r(v1, v1, sh + 4 - K - E) & m;
    }
}
template <int E>
__device__ __forceinline__ void planes4(const uint32_t* p0, const uint32_t* p1, int n, int sh, uint32_t (&x)[4])
{
    x[0] = x[1] = x[2] = x[3] = 0u;
    switch (n) {
    case 8: plane4<E, 7>(p0, p1, sh, x); [[fallthrough]];
    case 7: plane4<E, 6>(p0, p1, sh, x); [[fallthrough]];
    case 6: plane4<E, 5>(p0, p1, sh, x); [[fallthrough]];
    case 5: plane4<E, 4>(p0, p1, sh, x); [[fallthrough]];
    case 4: plane4<E, 3>(p0, p1, sh, x); [[fallthrough]];
    case 3: plane4<E, 2>(p0, p1, sh, x); [[fallthrough]];
    case 2: plane4<E, 1>(p0, p1, sh, x); [[fallthrough]];
    case 1: plane4<E, 0>(p0, p1, sh, x); [[fallthrough]];
    default: break;
    }
}
// level pair of the code in byte m of x: codes times 4 (E = 2, widths <= 6,
// the slot address supplies the upper bytes) or plain codes (E = 0)
template <int E>
__device__ __forceinline__ uint32_t level(uint32_t x, uint32_t tad, int m)
{
    if constexpr (E == 2) return lds_u32(__byte_perm(x, tad, 0x7650u | uint32_t(m)));
    else return lds_u32(tad + (((x >> (8 * m)) & 0xffu) << 2));
}

__device__ __forceinline__ bool token_scaled(const PlanView& pv)
{
    return pv.quant == SPECTRA_Q_LLOYD_GAUSS && pv.basis == SPECTRA_BASIS_RWHT;
}
__device__ __forceinline__ float chan_scale(const PlanView& pv, int h, int c)
{
    return token_scaled(pv) ? rsqrtf(float(D)) : pv.rscale[size_t(h) * D + c];
}

struct LvParams {
    PlanView kp, vp;
    const float* qt;          // [B Hq][D] scale * B_K^T q
    const uint8_t* kc;
    const uint8_t* vc;
    int64_t sstride;
    const float* kn;          // RWHT Lloyd-Max plans: per-token norms
    const float* vn;
    int64_t nstride;
    int Hq, G, nsplit, split_len;
    int64_t ctx;
    float* part;
    int sw;                   // words of one record slot
    int nofs;                 // slot offset of the record's norms (after the widest record and its padding)
    // the 1-bit key-residual sketch (kernels with QJ): per (b, kv head) a
    // bit-plane stream of D one-bit rows, the residual norms, and the
    // per-query weights w = S qt
    const uint8_t* qbits;
    int64_t qstride;
    const float* qnorms;
    int64_t qnstride;
    const float* qw;          // [B Hq][D]
};

// Shared memory (after aligning the start to 256 bytes): level tables (K,
// V, and the sketch's -1 / +1), channel descriptors (word offset, table
// address, code masks), per-step widest widths, the score weights (and the
// sketch weights) as B fragments, each warp's P tile and value sums, the
// merge scalars, then the warps' record slots (two each).
template <int NT, bool QJ>
struct LvSmem {
    static constexpr int PS = NT == 1 ? 8 : 24;   // u32 per token row of a P tile (conflict-free reads)
    static constexpr size_t tabK = 0, tabV = tabK + 4 * kTabWords, tabS = tabV + 4 * kTabWords,
                            descK = tabS + 4 * kSlot, descV = descK + 16 * D, bmK = descV + 16 * D,
                            bmV = bmK + 64, wf = bmV + 64, wfq = wf + size_t(8) * NT * 16 * 32,
                            pw = wfq + (QJ ? size_t(8) * NT * 16 * 32 : 0), ob = pw + size_t(4) * kWarps * 32 * PS,
                            mw = ob + size_t(8) * kWarps * NT * 8 * 32, lw = mw + 4 * 64, slots = lw + 4 * 64;
    static size_t total(int sw) { return 256 + slots + size_t(4) * kWarps * 2 * sw; }
};

template <int NT, bool QJ>
__global__ void __launch_bounds__(kThreads, (NT == 1 && !QJ) ? 3 : 2) attn_lv_split_kernel(const LvParams P)
{
    using L = LvSmem<NT, QJ>;
    constexpr int PS = L::PS;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((256u - (smem_u32(smem_raw) & 255u)) & 255u);
    uint32_t* tabK = reinterpret_cast<uint32_t*>(smem + L::tabK);
    uint32_t* tabV = reinterpret_cast<uint32_t*>(smem + L::tabV);
    int4* descK = reinterpret_cast<int4*>(smem + L::descK);
    int4* descV = reinterpret_cast<int4*>(smem + L::descV);
    int* bmK = reinterpret_cast<int*>(smem + L::bmK);     // [16] widest width of channels 8 kb .. 8 kb + 7
    int* bmV = reinterpret_cast<int*>(smem + L::bmV);     // [8] widest width of channels 16 mt .. 16 mt + 15
    uint2* Wf = reinterpret_cast<uint2*>(smem + L::wf);   // [NT][16][32] score-weight fragments
    uint2* Wq = reinterpret_cast<uint2*>(smem + L::wfq);  // [NT][16][32] sketch-weight fragments (QJ)
    uint32_t* tabS = reinterpret_cast<uint32_t*>(smem + L::tabS);   // the sketch's levels -1, +1
    uint32_t* Pw = reinterpret_cast<uint32_t*>(smem + L::pw);
    float2* Ob = reinterpret_cast<float2*>(smem + L::ob); // [8 warps][NT][8 m-tiles][32 lanes]
    float* mw = reinterpret_cast<float*>(smem + L::mw);   // [8 warps][8 heads]
    float* lw = reinterpret_cast<float*>(smem + L::lw);
    uint32_t* slots = reinterpret_cast<uint32_t*>(smem + L::slots);   // [8 warps][K, V][sw]

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tg = lane & 3;
    const PlanView& kp = P.kp;
    const PlanView& vp = P.vp;
    const int G = P.G;
    // records wider than the plans' bound are not read (the streams were sized by it)
    const int RK = kp.rec_bits[h] <= kp.max_rec_bits ? kp.rec_bits[h] : 0;
    const int RV = vp.rec_bits[h] <= vp.max_rec_bits ? vp.rec_bits[h] : 0;
    const bool ktok = token_scaled(kp), vtok = token_scaled(vp);

    // ---- per-CTA tables
    for (int e = tid; e < 2 * kTabWords; e += kThreads) {
        const int side = e / kTabWords, i = e % kTabWords;
        const PlanView& pv = side ? vp : kp;
        const int w = i < 7 * kSlot ? i / kSlot : (i < 9 * kSlot ? 7 : 8);
        const int code = i - tab_word(w);
        uint32_t v = 0u;
        if (w > 0 && code < (1 << w)) {
            const float lev = pv.quant == SPECTRA_Q_LLOYD_GAUSS ? pv.lm_level[(w - 1) * kLmStride + code]
                                                                : float(code) + 0.5f - float(1 << (w - 1));
            v = bf16_pair(lev);
        }
        (side ? tabV : tabK)[i] = v;
    }
    for (int e = tid; e < 2 * D; e += kThreads) {
        const int side = e / D, c = e % D;
        const PlanView& pv = side ? vp : kp;
        const int R = side ? RV : RK;
        int w = pv.bits[size_t(h) * D + c];
        int off = pv.chan_off[size_t(h) * D + c];
        if (w <= 0 || w > kMaxBits || off + w > R) {
            w = 0;
            off = 0;
        }
        const uint32_t mask1 = 0x01010101u * ((1u << w) - 1u);
        const uint32_t tad = smem_u32((side ? tabV : tabK) + tab_word(w));
        (side ? descV : descK)[c] = make_int4(off, int(tad), int(mask1 << 2), int(mask1));
    }
    // score weights W_jc = qt_jc a_c log2(e) as B fragments: lane (g, tg) of
    // k-block kb holds rows (channel 8 kb + tg) and (8 kb + tg + 4), column g
    // = (head 4 nt + g / 2, part g % 2)
    for (int e = tid; e < NT * 16 * 32; e += kThreads) {
        const int nt = e / 512, kb = (e / 32) % 16, ln = e % 32;
        const int gg = ln >> 2, tt = ln & 3, j = 4 * nt + (gg >> 1), y = gg & 1;
        uint2 v = make_uint2(0u, 0u);
        if (j < G) {
            const float* q = P.qt + (int64_t(b) * P.Hq + h * G + j) * D;
            const int c0 = 8 * kb + tt, c1 = c0 + 4;
            v.x = bf16_part_dup(q[c0] * chan_scale(kp, h, c0) * kLog2e, y);
            v.y = bf16_part_dup(q[c1] * chan_scale(kp, h, c1) * kLog2e, y);
        }
        Wf[e] = v;
    }
    if (QJ) {
        // sketch weights w_ji log2(e), laid out like the score weights (row i = sketch row)
        for (int e = tid; e < NT * 16 * 32; e += kThreads) {
            const int nt = e / 512, kb = (e / 32) % 16, ln = e % 32;
            const int gg = ln >> 2, tt = ln & 3, j = 4 * nt + (gg >> 1), y = gg & 1;
            uint2 v = make_uint2(0u, 0u);
            if (j < G) {
                const float* w = P.qw + (int64_t(b) * P.Hq + h * G + j) * D;
                v.x = bf16_part_dup(w[8 * kb + tt] * kLog2e, y);
                v.y = bf16_part_dup(w[8 * kb + tt + 4] * kLog2e, y);
            }
            Wq[e] = v;
        }
        if (tid < kSlot) tabS[tid] = tid == 0 ? bf16_pair(-1.f) : (tid == 1 ? bf16_pair(1.f) : 0u);
    }
    for (int e = tid; e < kWarps * NT * 8 * 32; e += kThreads) Ob[e] = make_float2(0.f, 0.f);
    __syncthreads();
    if (tid < 16) {
        int m = 0;
        for (int i = 0; i < 8; ++i) m = max(m, __popc(uint32_t(descK[8 * tid + i].w) & 0xffu));
        bmK[tid] = m;
    } else if (tid < 24) {
        const int mt = tid - 16;
        int m = 0;
        for (int i = 0; i < 16; ++i) m = max(m, __popc(uint32_t(descV[16 * mt + i].w) & 0xffu));
        bmV[mt] = m;
    }
    __syncthreads();

    const int64_t sid = int64_t(b) * kp.heads + h;
    const uint8_t* ks = P.kc + sid * P.sstride;
    const uint8_t* vs = P.vc + sid * P.sstride;
    const float* knr = ktok ? P.kn + sid * P.nstride : nullptr;
    const float* vnr = vtok ? P.vn + sid * P.nstride : nullptr;
    const int64_t s0 = int64_t(split) * P.split_len;
    const int64_t s1 = min(P.ctx, s0 + P.split_len);
    const int ng = int((s1 - s0 + kGroup - 1) / kGroup);   // s0 is a multiple of 32
    const int64_t g0 = s0 / kGroup;
    uint32_t* const slotK = slots + size_t(warp) * 2 * P.sw;
    uint32_t* const slotV = slotK + P.sw;
    const int noff = P.nofs;         // the record's per-token norms (RWHT Lloyd-Max plans)
    const int qoff = noff + 32;      // K slot (QJ): the sketch record (D words), then its norms
    const float* qnr = QJ ? P.qnorms + sid * P.qnstride : nullptr;
    const uint8_t* qs = QJ ? P.qbits + sid * P.qstride : nullptr;

    // one record (K: side 0, V: side 1) of the warp's it-th group into its
    // slot, with the norms where the plan has them; always commits
    auto issue = [&](int it, int side) {
        const int gi = warp + kWarps * it;
        if (gi < ng) {
            uint32_t* st = side ? slotV : slotK;
            const int64_t grp = g0 + gi;
            if (side) copy_record(st, vs + grp * RV * 4, RV, lane);
            else copy_record(st, ks + grp * RK * 4, RK, lane);
            if (QJ && !side) {
                copy_record(st + qoff, qs + grp * D * 4, D, lane);
                const int64_t t = grp * kGroup + lane;
                float* qn = reinterpret_cast<float*>(st + qoff + D);
                if (t < s1) cp_async4(smem_u32(qn + lane), qnr + t);
                else qn[lane] = 0.f;
            }
            if (side ? vtok : ktok) {
                float* nst = reinterpret_cast<float*>(st + noff);
                const int64_t t = grp * kGroup + lane;
                if (t < s1) cp_async4(smem_u32(nst + lane), (side ? vnr : knr) + t);
                else nst[lane] = 0.f;
            }
        }
        cp_async_commit();
    };

    float m_run[NT], l_run[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m_run[nt] = -INFINITY;
        l_run[nt] = 0.f;
    }
    uint32_t* pw = Pw + warp * 32 * PS;
    float2* ow = Ob + warp * NT * 8 * 32 + lane;

    issue(0, 0);
    issue(0, 1);
#pragma unroll 1
    for (int it = 0; warp + kWarps * it < ng; ++it) {
        cp_async_wait<1>();           // K of this group (its V may still be in flight)
        __syncwarp();                 // the words, copied by every lane, are visible
        const uint32_t* wk = slotK;
        const uint32_t* wv = slotV;
        const float* nk = reinterpret_cast<const float*>(slotK + noff);
        const float* nv = reinterpret_cast<const float*>(slotV + noff);
        const int64_t tb = (g0 + warp + kWarps * it) * kGroup + g;   // token of byte 0

        // ---- scores of the group's 32 tokens
        float sc[NT][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) sc[nt][0][r] = sc[nt][1][r] = 0.f;
        auto score_step = [&](auto e_tag, int kb, int bm) {
            constexpr int E = decltype(e_tag)::value;
            const int4 d0 = descK[8 * kb + tg], d1 = descK[8 * kb + 4 + tg];
            uint32_t x0, x1;
            planes2<E>(wk + d0.x, wk + d1.x, bm, g, x0, x1);
            x0 &= uint32_t(E ? d0.z : d0.w);
            x1 &= uint32_t(E ? d1.z : d1.w);
            const uint32_t t0 = uint32_t(d0.y), t1 = uint32_t(d1.y);
            const uint32_t a00 = level<E>(x0, t0, 0), a01 = level<E>(x0, t0, 1), a02 = level<E>(x0, t0, 2),
                           a03 = level<E>(x0, t0, 3);
            const uint32_t a10 = level<E>(x1, t1, 0), a11 = level<E>(x1, t1, 1), a12 = level<E>(x1, t1, 2),
                           a13 = level<E>(x1, t1, 3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint2 wf = Wf[(nt * 16 + kb) * 32 + lane];
                mma_bf16(sc[nt][0], a00, a01, a10, a11, wf.x, wf.y);
                mma_bf16(sc[nt][1], a02, a03, a12, a13, wf.x, wf.y);
            }
        };
#pragma unroll 1
        for (int kb = 0; kb < 16; ++kb) {
            const int bm = bmK[kb];
            if (bm == 0) continue;
            if (bm <= 6) score_step(std::integral_constant<int, 2>{}, kb, bm);
            else score_step(std::integral_constant<int, 0>{}, kb, bm);
        }

        // the sketch correction: sum_i w_ji z_i(t), z = -1 / +1 for a clear / set bit
        float sq[NT][2][4];
        if (QJ) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) sq[nt][0][r] = sq[nt][1][r] = 0.f;
            const uint32_t* wq = wk + qoff;
            const uint32_t ts = smem_u32(tabS);
#pragma unroll 2
            for (int kb = 0; kb < 16; ++kb) {
                const uint32_t v0 = wq[8 * kb + tg], v1 = wq[8 * kb + 4 + tg];
                const uint32_t x0 = __funnelshift_r(v0, v0, g - 2) & 0x04040404u;
                const uint32_t x1 = __funnelshift_r(v1, v1, g - 2) & 0x04040404u;
                const uint32_t a00 = level<2>(x0, ts, 0), a01 = level<2>(x0, ts, 1), a02 = level<2>(x0, ts, 2),
                               a03 = level<2>(x0, ts, 3);
                const uint32_t a10 = level<2>(x1, ts, 0), a11 = level<2>(x1, ts, 1), a12 = level<2>(x1, ts, 2),
                               a13 = level<2>(x1, ts, 3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint2 wf = Wq[(nt * 16 + kb) * 32 + lane];
                    mma_bf16(sq[nt][0], a00, a01, a10, a11, wf.x, wf.y);
                    mma_bf16(sq[nt][1], a02, a03, a12, a13, wf.x, wf.y);
                }
            }
        }
        // scores of this thread's tokens (g + 8 m), scaled by the K norms,
        // plus sqrt(pi/2)/d ||r_t|| times the sketch correction
        float s[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            s[nt][0] = sc[nt][0][0] + sc[nt][0][1];
            s[nt][1] = sc[nt][0][2] + sc[nt][0][3];
            s[nt][2] = sc[nt][1][0] + sc[nt][1][1];
            s[nt][3] = sc[nt][1][2] + sc[nt][1][3];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (ktok) s[nt][m] *= nk[g + 8 * m];
                if (QJ) {
                    const float* qn = reinterpret_cast<const float*>(wk + qoff + D);
                    const float c = sq[nt][m >> 1][2 * (m & 1)] + sq[nt][m >> 1][2 * (m & 1) + 1];
                    s[nt][m] = fmaf(kQjlScale * qn[g + 8 * m], c, s[nt][m]);
                }
                s[nt][m] = (tb + 8 * m < s1) ? s[nt][m] : -INFINITY;
            }
        }
        __syncwarp();                 // every lane is past its reads of the K slot
        issue(it + 1, 0);             // the next group's K lands during this softmax and P V
        cp_async_wait<1>();           // this group's V
        __syncwarp();

        // ---- online softmax of the warp's own tokens; P tile for P V
        float alpha[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float mx = fmaxf(fmaxf(s[nt][0], s[nt][1]), fmaxf(s[nt][2], s[nt][3]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            // the group has a valid token, so mx is finite; alpha = 0 on the warp's first group
            const float mnew = fmaxf(m_run[nt], mx);
            alpha[nt] = exp2f(m_run[nt] - mnew);
            m_run[nt] = mnew;
            float ps = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float p = exp2f(s[nt][m] - mnew);
                ps += p;
                const float pv = vtok ? p * nv[g + 8 * m] : p;
                const uint32_t hi = bf16_bits(pv), lo = bf16_bits(pv - bf16_val(hi));
                *reinterpret_cast<uint2*>(pw + (g + 8 * m) * PS + 8 * nt + 2 * tg) =
                    make_uint2(hi | (hi << 16), lo | (lo << 16));
            }
            l_run[nt] = l_run[nt] * alpha[nt] + ps;
        }
        __syncwarp();                 // the P tile is complete

        // ---- P V over the group, 16 channels per step
        uint32_t pb[NT][4][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                pb[nt][kb][0] = pw[(8 * kb + tg) * PS + 8 * nt + g];
                pb[nt][kb][1] = pw[(8 * kb + tg + 4) * PS + 8 * nt + g];
            }
        auto value_step = [&](auto e_tag, int mt, int bm) {
            constexpr int E = decltype(e_tag)::value;
            const int4 d0 = descV[16 * mt + g], d1 = descV[16 * mt + 8 + g];
            uint32_t x[4];
            planes4<E>(wv + d0.x, wv + d1.x, bm, tg, x);
            const uint32_t m0 = uint32_t(E ? d0.z : d0.w), m1 = uint32_t(E ? d1.z : d1.w);
            x[0] &= m0;
            x[1] &= m0;
            x[2] &= m1;
            x[3] &= m1;
            const uint32_t t0 = uint32_t(d0.y), t1 = uint32_t(d1.y);
            float c[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                const uint32_t a0 = level<E>(x[0], t0, kb), a1 = level<E>(x[2], t1, kb);
                const uint32_t a2 = level<E>(x[1], t0, kb), a3 = level<E>(x[3], t1, kb);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_bf16(c[nt], a0, a1, a2, a3, pb[nt][kb][0], pb[nt][kb][1]);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float2 o = ow[(nt * 8 + mt) * 32];
                o.x = fmaf(o.x, alpha[nt], c[nt][0] + c[nt][1]);   // channel 16 mt + g
                o.y = fmaf(o.y, alpha[nt], c[nt][2] + c[nt][3]);   // channel 16 mt + 8 + g
                ow[(nt * 8 + mt) * 32] = o;
            }
        };
#pragma unroll 1
        for (int mt = 0; mt < 8; ++mt) {
            const int bm = bmV[mt];
            if (bm == 0) continue;    // zero-width channels: their sums stay 0
            if (bm <= 6) value_step(std::integral_constant<int, 2>{}, mt, bm);
            else value_step(std::integral_constant<int, 0>{}, mt, bm);
        }
        __syncwarp();                 // every lane is past its reads of the V slot
        issue(it + 1, 1);             // the next group's V lands during its scores
    }
    cp_async_wait<0>();               // (only empty groups can remain)

    // ---- merge the warps' states; write the split's partial (m, l, o)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float l = l_run[nt];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        if (g == 0) {
            mw[warp * 8 + 4 * nt + tg] = m_run[nt];
            lw[warp * 8 + 4 * nt + tg] = l;
        }
    }
    __syncthreads();
    for (int e = tid; e < G * D; e += kThreads) {
        const int j = e / D, c = e % D;
        const int nt = j >> 2, jt = j & 3, mt = c >> 4, r = c & 15;
        const int ln = (r & 7) * 4 + jt;                    // lane (g, tg) = (r mod 8, head mod 4)
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mw[w * 8 + j]);
        float l = 0.f, o = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = exp2f(mw[w * 8 + j] - M);   // 0 for a warp without groups
                const float2 ov = Ob[((w * NT + nt) * 8 + mt) * 32 + ln];
                l = fmaf(f, lw[w * 8 + j], l);
                o = fmaf(f, (r < 8) ? ov.x : ov.y, o);
            }
        }
        float* bp = P.part + ((int64_t(b) * P.Hq + h * G + j) * P.nsplit + split) * (D + 2);
        bp[2 + c] = o * chan_scale(vp, h, c);
        if (c == 0) {
            bp[0] = M * kLn2;
            bp[1] = l;
        }
    }
}

}  // namespace

// Attention of any plan pair with head_dim 128 and at most eight query heads
// per kv head, after attn_qrot_kernel has written qt (and, with the sketch,
// qw = S qt); *done is false when the shapes are not covered (nothing
// launched).  qbits null: no sketch correction.
spectra_status launch_attn_lv(const spectra_plan* kplan, const spectra_plan* vplan, const float* qt, int B, int Hq,
                              const uint8_t* kc, const uint8_t* vc, int64_t sstride, const float* kn,
                              const float* vn, int64_t nstride, int64_t ctx, float* part, int nsplit, int split_len,
                              const uint8_t* qbits, int64_t qstride, const float* qnorms, int64_t qnstride,
                              const float* qw, cudaStream_t s, bool* done)
{
    *done = false;
    const int Hkv = kplan->heads, G = Hq / Hkv;
    if (kplan->head_dim != D || vplan->head_dim != D || G < 1 || G > 8) return SPECTRA_OK;
    if (split_len % kGroup != 0) return SPECTRA_OK;
    const int RKm = kplan->max_rec_bits, RVm = vplan->max_rec_bits;
    if (RKm > kMaxBits * D || RVm > kMaxBits * D || RKm < 0 || RVm < 0) return SPECTRA_OK;
    LvParams P;
    P.kp = make_view(kplan);
    P.vp = make_view(vplan);
    P.qt = qt;
    P.kc = kc;
    P.vc = vc;
    P.sstride = sstride;
    P.kn = kn;
    P.vn = vn;
    P.nstride = nstride;
    P.Hq = Hq;
    P.G = G;
    P.nsplit = nsplit;
    P.split_len = split_len;
    P.ctx = ctx;
    P.part = part;
    // a slot: the widest record (16-byte multiple), the padding the plane
    // reads may run into, 32 norms; with the sketch, its record and norms
    const bool qj = qbits != nullptr;
    P.nofs = ((std::max(RKm, RVm) + 3) & ~3) + kPad;
    P.sw = P.nofs + 32 + (qj ? D + 32 : 0);
    P.qbits = qbits;
    P.qstride = qstride;
    P.qnorms = qnorms;
    P.qnstride = qnstride;
    P.qw = qw;
    dim3 grid(nsplit, Hkv, B);
    auto go = [&](auto kern, size_t sm) -> spectra_status {
        if (spectra_status e = set_smem(kern, sm)) return e;
        kern<<<grid, kThreads, sm, s>>>(P);
        if (spectra_status e = cuda_status(cudaGetLastError())) return e;
        *done = true;
        return SPECTRA_OK;
    };
    // as many CTAs per SM as the registers allow, if the shared memory does
    // (228 KB per SM, 1 KB of it per CTA reserved)
    for (int cap : {(G <= 4 && !qj) ? 3 : 2, 2, 1}) {
        const size_t lim = size_t(228 * 1024) / cap - 1024;
        if (!qj) {
            if (G <= 4 && LvSmem<1, false>::total(P.sw) <= lim)
                return go(attn_lv_split_kernel<1, false>, LvSmem<1, false>::total(P.sw));
            if (G > 4 && LvSmem<2, false>::total(P.sw) <= lim)
                return go(attn_lv_split_kernel<2, false>, LvSmem<2, false>::total(P.sw));
        } else {
            if (G <= 4 && LvSmem<1, true>::total(P.sw) <= lim)
                return go(attn_lv_split_kernel<1, true>, LvSmem<1, true>::total(P.sw));
            if (G > 4 && LvSmem<2, true>::total(P.sw) <= lim)
                return go(attn_lv_split_kernel<2, true>, LvSmem<2, true>::total(P.sw));
        }
    }
    return SPECTRA_OK;
}

}  // namespace spectra
