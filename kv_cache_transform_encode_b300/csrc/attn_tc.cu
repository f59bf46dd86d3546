// attn_tc.cu -- decode-step attention over packed K/V streams on the tensor
// cores (uniform quantizer, eigenbasis plans, head_dim 128, at most four
// query heads per kv head).
//
// "Sintesi Tecnica: SPECTRA", "Significato e Rivendicazioni": attention
// computed directly in the latent space.  With the uniform quantizer a
// latent coordinate is yhat_c = (Delta_c / 2)(2 code_c + 1 - 2^b_c), affine
// in the code: with z = code - 2^(b-1) (an exact small integer),
// yhat_c = Delta_c (z_c + 1/2), so
//   s_j(t) = sum_c qt_jc yhat_c(t) = sum_c W_jc z_c(t) + K0_j,
//   W_jc = qt_jc Delta_c,   K0_j = (1/2) sum_c W_jc,
//   sum_t p_j(t) yhat_c(t) = Delta_c (sum_t p_j(t) z_c(t) + l_j / 2),
// and both contractions run on the small integers z.  A code enters the
// tensor core as the fp16 number z: the byte-permute trick gives 1024 +
// code exactly, one packed subtraction of 1024 + 2^(b-1) leaves z, so the
// fp32 accumulators only ever hold sums of small terms.  W and P enter as
// fp16 hi + lo pairs (22 significand bits), so the products carry
// fp32-grade accuracy.
//
// One CTA per (context split, kv head, batch).  Per 128-token tile:
//  1. the tile's K and V code words arrive in shared memory (cp.async,
//     double-buffered);
//  2. eight warps unpack them (per side, warp = 32-token group, lane =
//     channel, over four blocks of 32 channels: the bit-plane words of a
//     group become 32 code bytes through four 8x8 bit transposes, or, where
//     a block is at most 2 bits wide, the two planes are interleaved into
//     even- and odd-token words and each fp16 pair is one shift and one
//     mask), into fp16 tiles L[c][p]; within a 32-token group position
//     2s holds token s and 2s + 1 token s + 16;
//  3. each warp then owns 16 tokens of the tile end to end: scores by
//     mma.sync m16n8k16 (A = L_K^T via ldmatrix.trans, B = [W_hi; W_lo],
//     n = head, hi/lo), an online softmax over its own slice (its running
//     max and sum per head in registers), and P V (A = L_V, channels x the
//     slice's tokens, B = [P_hi; P_lo]) into its own accumulators for all
//     128 channels.  Two block barriers per tile (codes landed, tiles
//     unpacked); the eight slices merge in shared memory at the end.
// The split's (m, l, sum_t p z) go to the workspace; the combine kernel
// of attn.cu merges splits, dequantizes and rotates by the V basis.
#include "spectra_internal.cuh"

#include <cuda_fp16.h>
#include <math.h>

namespace spectra {

namespace {

constexpr int D = 128;
constexpr int TT = 128;                  // tokens per tile
constexpr int LROW = TT * 2 + 16;        // bytes per L row (padded: conflict-free ldmatrix)
constexpr int kThreads = 256;
constexpr int kGmax = 4;                 // query heads per kv head
constexpr int PROW = 24;                 // halves per row of a warp's P tile (conflict-free B loads)

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void transpose8(uint32_t& lo, uint32_t& hi)
{
    uint32_t t;
    t = (lo ^ (lo >> 7)) & 0x00AA00AAu;  lo ^= t ^ (t << 7);
    t = (hi ^ (hi >> 7)) & 0x00AA00AAu;  hi ^= t ^ (t << 7);
    t = (lo ^ (lo >> 14)) & 0x0000CCCCu; lo ^= t ^ (t << 14);
    t = (hi ^ (hi >> 14)) & 0x0000CCCCu; hi ^= t ^ (t << 14);
    t = (lo ^ (hi << 4)) & 0xF0F0F0F0u;  lo ^= t;  hi ^= t >> 4;
}

__device__ __forceinline__ uint32_t gather_byte(uint32_t a, uint32_t b, uint32_t c, uint32_t d, int k)
{
    const uint32_t sel = ((4u + k) << 4) | uint32_t(k);
    return __byte_perm(__byte_perm(a, b, sel), __byte_perm(c, d, sel), 0x5410);
}

// bit planes of one channel for a 32-token group -> 32 code bytes
__device__ __forceinline__ void planes_to_codes(const uint32_t* words, int o, int b, int bmax, uint32_t (&X)[8])
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

__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D (16x8 f32) = A (16x16 f16, row) * B (16x8 f16, col) + C
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                         const float (&c)[4])
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// ------------------------------------------------------------------ prep
// Per (batch, kv head): qt_j = scale * B_K^T q_j, W_jc = qt_jc Delta_c as fp16
// hi/lo rows ([8][D]: rows 0..3 hi, 4..7 lo; heads >= G zero), the sums of
// each row over every 16-channel chunk (the 1024 offsets removed per MMA
// step), and K0_j.
__global__ void __launch_bounds__(kGmax * D)
attn_tc_prep_kernel(PlanView kp, const void* __restrict__ q, int q_dt, int Hq, int G, float scale,
                    __half* __restrict__ wimg, float* __restrict__ bias)
{
    const int bh = blockIdx.x, Hkv = kp.heads, h = bh % Hkv, b = bh / Hkv;
    const int tid = threadIdx.x, c = tid % D, j = tid / D;   // channel, query head of the group
    extern __shared__ float Bs[];                 // [D][D] basis of head h (staged: coalesced 16-B loads)
    __shared__ float qs[kGmax][D];
    __shared__ float red[kGmax][4];
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
    const float delta = kp.rscale[size_t(h) * D + c];
    __half* wr = wimg + size_t(bh) * 8 * D;
    const float qj = qt * scale;
    const float w = (bits > 0 && j < G) ? qj * delta : 0.f;
    const __half hi = __float2half_rn(w);
    const __half lo = __float2half_rn(w - __half2float(hi));
    wr[j * D + c] = hi;
    wr[(kGmax + j) * D + c] = lo;
    // yhat = Delta (z + 1/2): the 1/2 terms of the score, summed over channels
    float k0 = 0.5f * w;
    for (int o = 16; o; o >>= 1) k0 += __shfl_xor_sync(0xffffffffu, k0, o);
    if ((c & 31) == 0) red[j][c >> 5] = k0;
    __syncthreads();
    if (tid < kGmax) bias[size_t(bh) * kGmax + tid] = red[tid][0] + red[tid][1] + red[tid][2] + red[tid][3];
}

// ------------------------------------------------------------------ split
struct AttnTcParams {
    PlanView kp, vp;
    int Hq, G, nsplit, split_len;
    int64_t ctx;
    const uint8_t* kc;
    const uint8_t* vc;
    int64_t sstride;
    const __half* wimg;
    const float* bias;
    float* part;
    uint32_t kbytes, vbytes;   // code-word bytes of one tile (16 R)
};

__global__ void __launch_bounds__(kThreads, 2)
attn_tc_split_kernel(AttnTcParams P)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int Hkv = P.kp.heads, G = P.G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, tig = lane & 3;
    const int bh = b * Hkv + h;

    uint8_t* cw = smem;                                          // [2][kbytes + vbytes]
    const uint32_t cwb = P.kbytes + P.vbytes;
    uint8_t* Lk = cw + 2 * cwb;                                  // [D][LROW]
    uint8_t* Lv = Lk + D * LROW;                                 // [D][LROW]
    __half* Pw = reinterpret_cast<__half*>(Lv + D * LROW);      // per warp [8][PROW]: P of its 16 tokens
    float* mw = reinterpret_cast<float*>(Pw + 8 * 8 * PROW);     // [8 warps][kGmax] running max
    float* lw = mw + 8 * kGmax;                                  // [8 warps][kGmax] running sum

    const int64_t t_begin = int64_t(split) * P.split_len;
    const int64_t t_end = min(P.ctx, t_begin + P.split_len);
    const int ntiles = int((t_end - t_begin + TT - 1) / TT);
    // records larger than the plans' bound are not read (their streams were sized by the bound)
    const int RK0 = P.kp.rec_bits[h], RV0 = P.vp.rec_bits[h];
    const int RK = RK0 <= P.kp.max_rec_bits ? RK0 : 0, RV = RV0 <= P.vp.max_rec_bits ? RV0 : 0;
    const int64_t sid = int64_t(b) * Hkv + h;
    const uint8_t* ks = P.kc + sid * P.sstride;
    const uint8_t* vs = P.vc + sid * P.sstride;

    // unpack role: side (K for warps 0-3, V for 4-7) and 32-token group
    // ug = warp & 3 of the tile, over all 128 channels in four blocks of 32
    // (channel 32 cb + lane).  The wide channels (the leading eigen-
    // directions) sit in block 0, so every warp gets the same mix of one
    // wide and three narrow blocks.  Per block: widths packed 8 bits each
    // (ubp), the widest in the block (ubm), and word offsets 16 bits each.
    const int side = warp >> 2, ug = warp & 3;
    const PlanView& up = side ? P.vp : P.kp;
    uint32_t ubp = 0, ubm = 0, uop01 = 0, uop23 = 0;
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
        const int c = cb * 32 + lane;
        const uint32_t wb = uint32_t(up.bits[size_t(h) * D + c]);
        const uint32_t wo = uint32_t(up.chan_off[size_t(h) * D + c]);
        ubp |= wb << (8 * cb);
        ubm |= uint32_t(__reduce_max_sync(0xffffffffu, wb)) << (8 * cb);
        if (cb < 2) uop01 |= wo << (16 * cb); else uop23 |= wo << (16 * (cb - 2));
    }
    const int uR = side ? RV : RK;

    // score operand B: W rows (n = g8: 0..3 hi, 4..7 lo), k = 16 kb + 2 tig (+8)
    uint32_t wf[8][2];
    {
        const __half* wr = P.wimg + size_t(bh) * 8 * D + g8 * D;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
            wf[kb][0] = *reinterpret_cast<const uint32_t*>(wr + kb * 16 + 2 * tig);
            wf[kb][1] = *reinterpret_cast<const uint32_t*>(wr + kb * 16 + 8 + 2 * tig);
        }
    }
    const float bias0 = P.bias[size_t(bh) * kGmax + ((2 * tig) & 3)];
    const float bias1 = P.bias[size_t(bh) * kGmax + ((2 * tig + 1) & 3)];
    // this warp's share of the output, all 128 channels: m-tile mt holds
    // channels 16 mt + g8 (+8), columns n = 2 tig, 2 tig + 1 (head hi / lo)
    float oacc[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
    // online-softmax state of the warp's token slice, heads j0 = 2 (tig & 1), j0 + 1
    const int j0 = 2 * (tig & 1), j1 = j0 + 1;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    __half* pw = Pw + warp * 8 * PROW;

    auto issue_load = [&](int tile, int buf) {
        const int64_t t0 = t_begin + int64_t(tile) * TT;
        const int64_t ng = min(int64_t(4), (t_end - t0 + 31) / 32);
        const uint32_t nk = uint32_t((ng * 4 * RK + 15) / 16), nv = uint32_t((ng * 4 * RV + 15) / 16);
        uint8_t* dst = cw + buf * cwb;
        const uint8_t* srck = ks + (t0 / 32) * 4 * RK;
        const uint8_t* srcv = vs + (t0 / 32) * 4 * RV;
        for (uint32_t i = tid; i < nk + nv; i += kThreads) {
            if (i < nk) cp_async16(dst + 16 * i, srck + 16 * i);
            else cp_async16(dst + P.kbytes + 16 * (i - nk), srcv + 16 * (i - nk));
        }
        cp_async_commit();
    };
    if (ntiles > 0) issue_load(0, 0);

    for (int tile = 0; tile < ntiles; ++tile) {
        const int buf = tile & 1;
        const int64_t t0 = t_begin + int64_t(tile) * TT;
        cp_async_wait_all();
        __syncthreads();                                   // code words landed; previous tile done
        if (tile + 1 < ntiles) issue_load(tile + 1, buf ^ 1);

        // ---- unpack: one 32-token group per warp, one channel per lane, four channel blocks
        {
            const uint32_t* words = reinterpret_cast<const uint32_t*>(cw + buf * cwb + (side ? P.kbytes : 0));
            uint8_t* L = side ? Lv : Lk;
            const bool live = t0 + 32 * ug < t_end && uR > 0;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                const int ub = int((ubp >> (8 * cb)) & 0xFFu), ubmax = int((ubm >> (8 * cb)) & 0xFFu);
                const int uo = int(((cb < 2 ? uop01 : uop23) >> (16 * (cb & 1))) & 0xFFFFu);
                // v[s] = fp16 pair (1024 + code) for tokens s and s + 16 of the group:
                // the tile keeps each group in that pair order (positions 2s, 2s + 1),
                // the same for K and V, so scores and P V see one consistent order
                uint32_t v[16];
                if (ubmax <= 2) {
                    // widths <= 2 (the block's widest channel): interleave the two
                    // planes once into E (even tokens) and O (odd tokens), 2 bits a
                    // token; tokens s and s + 16 are then bits s and s + 16 of E (or O)
                    uint32_t w0 = 0u, w1 = 0u;
                    if (live) {
                        const uint32_t* wg = words + ug * uR + uo;
                        w0 = ub > 0 ? wg[0] : 0u;
                        w1 = ub > 1 ? wg[1] : 0u;
                    }
                    const uint32_t E = (w0 & 0x55555555u) | ((w1 << 1) & 0xAAAAAAAAu);
                    const uint32_t O = ((w0 >> 1) & 0x55555555u) | (w1 & 0xAAAAAAAAu);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const uint32_t x = (q & 1) ? (O >> (q - 1)) : (E >> q);
                        v[q] = (x & 0x00030003u) | 0x64006400u;
                    }
                } else {
                    uint32_t X[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // byte i of X[m]: code of token 4m + i
                    if (live) planes_to_codes(words + ug * uR, uo, ub, ubmax, X);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const uint32_t sel = uint32_t(q & 3) | (uint32_t(4 + (q & 3)) << 8);
                        v[q] = (__byte_perm(X[q >> 2], X[(q >> 2) + 4], sel) & 0x00FF00FFu) | 0x64006400u;
                    }
                }
                // z = code - 2^(b-1) (0 for dropped channels): (1024 + code) - (1024 + 2^(b-1)), exact in fp16
                const __half2 cz = __float2half2_rn(1024.f + (ub > 0 ? float(1 << (ub - 1)) : 0.f));
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const __half2 z = __hsub2(*reinterpret_cast<const __half2*>(&v[q]), cz);
                    v[q] = *reinterpret_cast<const uint32_t*>(&z);
                }
                uint4* dst = reinterpret_cast<uint4*>(L + (cb * 32 + lane) * LROW + ug * 64);
#pragma unroll
                for (int e = 0; e < 4; ++e) dst[e] = make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
            }
        }
        __syncthreads();

        // ---- per warp, positions 16 warp .. +15 of the tile: scores, online
        // softmax and P V, with no block barrier in between
        const int mi = lane >> 3, ri = lane & 7;
        const int tw = warp * 16;
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kb = 0; kb < 8; kb += 2) {
            uint32_t a[4], a2[4];
            const int k = kb * 16 + (mi >> 1) * 8 + ri, m = tw + (mi & 1) * 8;
            ldsm_x4_t(smem_addr(Lk + k * LROW + m * 2), a);
            ldsm_x4_t(smem_addr(Lk + (k + 16) * LROW + m * 2), a2);
            mma16816(sa, a, wf[kb][0], wf[kb][1], sa);
            mma16816(sb, a2, wf[kb + 1][0], wf[kb + 1][1], sb);
        }
        float sc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            sc[e] = sa[e] + sb[e];
            sc[e] += __shfl_xor_sync(0xffffffffu, sc[e], 2);   // hi + lo columns
        }
        {
            // positions tw + g8 (+8) hold tokens 32 (warp / 2) + (q >> 1) + 16 (q & 1), q the position in the group
            const int qa = (warp & 1) * 16 + g8, qb = qa + 8;
            const int gbase = (warp >> 1) * 32;
            const bool la = t0 + gbase + (qa >> 1) + (qa & 1) * 16 < t_end;
            const bool lb = t0 + gbase + (qb >> 1) + (qb & 1) * 16 < t_end;
            const bool h0 = j0 < G, h1 = j1 < G;
            sc[0] = (la && h0) ? sc[0] + bias0 : -INFINITY;
            sc[1] = (la && h1) ? sc[1] + bias1 : -INFINITY;
            sc[2] = (lb && h0) ? sc[2] + bias0 : -INFINITY;
            sc[3] = (lb && h1) ? sc[3] + bias1 : -INFINITY;
        }
        float x0 = fmaxf(sc[0], sc[2]), x1 = fmaxf(sc[1], sc[3]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o));
        }
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float al0 = (m0 == -INFINITY) ? 0.f : __expf(m0 - n0);
        const float al1 = (m1 == -INFINITY) ? 0.f : __expf(m1 - n1);
        m0 = n0;
        m1 = n1;
        __half ph[4], pl[4];
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float pe = (sc[e] == -INFINITY) ? 0.f : __expf(sc[e] - ((e & 1) ? n1 : n0));
            ph[e] = __float2half_rn(pe);
            pl[e] = __float2half_rn(pe - __half2float(ph[e]));
            const float pq = __half2float(ph[e]) + __half2float(pl[e]);
            if (e & 1) ps1 += pq; else ps0 += pq;
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            ps0 += __shfl_xor_sync(0xffffffffu, ps0, o);
            ps1 += __shfl_xor_sync(0xffffffffu, ps1, o);
        }
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
        // P of the slice as the B operand [n = head hi 0..3 / lo 4..7][k = token]:
        // lanes tig 0/1 write the hi parts of their heads, tig 2/3 the lo parts
        {
            const __half* pv = tig < 2 ? ph : pl;
            const int r0 = (tig < 2 ? 0 : kGmax) + j0;
            pw[r0 * PROW + g8] = pv[0];
            pw[(r0 + 1) * PROW + g8] = pv[1];
            pw[r0 * PROW + g8 + 8] = pv[2];
            pw[(r0 + 1) * PROW + g8 + 8] = pv[3];
        }
        __syncwarp();
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(pw + g8 * PROW + 2 * tig);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(pw + g8 * PROW + 8 + 2 * tig);
        // columns n = 2 tig, 2 tig + 1 are heads j0, j1 (hi for tig < 2, lo otherwise)
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            oacc[mt][0] *= al0; oacc[mt][1] *= al1; oacc[mt][2] *= al0; oacc[mt][3] *= al1;
            uint32_t a[4];
            const int m = mt * 16 + (mi & 1) * 8 + ri, k = tw + (mi >> 1) * 8;
            ldsm_x4(smem_addr(Lv + m * LROW + k * 2), a);
            mma16816(oacc[mt], a, b0, b1, oacc[mt]);
        }
    }
    __syncthreads();   // every warp is past its last read of Lk / Lv

    // merge the eight warps' slices: warp w's partial scaled by exp(m_w - M)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[mt][e] += __shfl_xor_sync(0xffffffffu, oacc[mt][e], 2);   // hi + lo
    float* Ow = reinterpret_cast<float*>(Lk);                    // [8 warps][kGmax][D]
    if (g8 == 0 && tig < 2) {
        mw[warp * kGmax + j0] = m0; mw[warp * kGmax + j1] = m1;
        lw[warp * kGmax + j0] = l0; lw[warp * kGmax + j1] = l1;
    }
    if (tig < 2) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int c0 = mt * 16 + g8, c1 = c0 + 8;
            Ow[(warp * kGmax + j0) * D + c0] = oacc[mt][0];
            Ow[(warp * kGmax + j1) * D + c0] = oacc[mt][1];
            Ow[(warp * kGmax + j0) * D + c1] = oacc[mt][2];
            Ow[(warp * kGmax + j1) * D + c1] = oacc[mt][3];
        }
    }
    __syncthreads();

    // partials: [(b Hq + h G + j) nsplit + split][2 + D]: m, l, sum_t p code
    for (int i = tid; i < kGmax * D; i += kThreads) {
        const int j = i / D, c = i % D;
        if (j >= G) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 8; ++w) M = fmaxf(M, mw[w * kGmax + j]);
        float o = 0.f, l = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const float mv = mw[w * kGmax + j];
            const float f = (mv == -INFINITY) ? 0.f : __expf(mv - M);
            o = fmaf(f, Ow[(w * kGmax + j) * D + c], o);
            l = fmaf(f, lw[w * kGmax + j], l);
        }
        float* bp = P.part + ((int64_t(b) * P.Hq + h * G + j) * P.nsplit + split) * (D + 2);
        bp[2 + c] = o;
        if (c == 0) {
            bp[0] = M;
            bp[1] = l;
        }
    }
}

size_t tc_split_smem(uint32_t kbytes, uint32_t vbytes)
{
    return 2 * size_t(kbytes + vbytes) + 2 * size_t(D) * LROW + sizeof(__half) * 8 * 8 * PROW +
           sizeof(float) * 2 * 8 * kGmax + 64;
}

}  // namespace

// Workspace layout of the tensor-core path (inside attn_workspace_bytes):
// [partials | wimg (B Hkv 8 D fp16) | bias (B Hkv 4 f32)].
size_t attn_tc_extra_bytes(int B, int Hkv)
{
    return align256(sizeof(__half) * size_t(B) * Hkv * 8 * D) + align256(sizeof(float) * size_t(B) * Hkv * kGmax);
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
    __half* wimg = static_cast<__half*>(extra);
    float* bias = reinterpret_cast<float*>(static_cast<uint8_t*>(extra) +
                                           align256(sizeof(__half) * size_t(B) * Hkv * 8 * D));
    P.wimg = wimg;
    P.bias = bias;
    P.part = part;
    P.kbytes = uint32_t(16 * (kplan->max_rec_bits > 0 ? kplan->max_rec_bits : 1));
    P.vbytes = uint32_t(16 * (vplan->max_rec_bits > 0 ? vplan->max_rec_bits : 1));
    const size_t sm = tc_split_smem(P.kbytes, P.vbytes);
    if (sm > 227 * 1024) return SPECTRA_OK;
    if (spectra_status st = set_smem(attn_tc_prep_kernel, sizeof(float) * D * D)) return st;
    attn_tc_prep_kernel<<<B * Hkv, kGmax * D, sizeof(float) * D * D, s>>>(P.kp, q, q_dt, Hq, G, scale, wimg, bias);
    if (spectra_status st = set_smem(attn_tc_split_kernel, sm)) return st;
    dim3 grid(nsplit, Hkv, B);
    attn_tc_split_kernel<<<grid, kThreads, sm, s>>>(P);
    *done = true;
    return cuda_status(cudaGetLastError());
}

}  // namespace spectra
