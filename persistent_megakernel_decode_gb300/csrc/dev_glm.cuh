// GLM FP8 pre-attention block: the three instruction bodies run by the
// consumer warps, and the activation staging of the GEMM tiles.
//
// "MegaRTP megakernel article", section 1: the block is Add+RMSNorm+Quant,
// FP8 GEMMs with 128-wide block scales, RoPE and the cache write-back;
// section 2: after the first kernel, QKV-A, Head-Gate and Indexer-K are
// independent; QKV-A feeds the Q-B (main) and Indexer-Q paths.
//
// FP8 is e4m3 ("fn": bias 7, no infinities, largest finite 448).  At 16 token
// rows the GEMMs are HBM-bound (about 31 flop per weight byte), so they use
// warp-level m16n8k32 e4m3 tensor-core MMAs with the 16 tokens as the M side
// and 8 weight rows as the N side, accumulating each 128-wide K block in the
// MMA and applying its two scales in fp32 registers.
#pragma once
#include <cuda_bf16.h>

#include "dev_common.cuh"

namespace mk {

// e4m3 codes of (lo, hi), lo in the low byte (round to nearest even,
// saturating at +-448)
DEV uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

DEV float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
DEV float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
DEV uint32_t pack_bf16(float lo, float hi) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// D += A * B for A 16 x 32 (rows = tokens), B 32 x 8 (columns = weight rows),
// e4m3 operands, fp32 accumulators
DEV void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Quantise 4 values of a 128-column block whose other 124 values sit in the
// warp's other lanes: scale = amax / 448 (1 for an all-zero block; an IEEE
// division, so the fp32 scale is the correctly rounded one), codes of value
// / scale -- taken as value times the correctly rounded reciprocal, within
// 2^-23 of the quotient, so a code can only differ from the exact quotient's
// rounding where that quotient sits that close to a midpoint between two
// codes.  Returns the 4 codes (first value in the low byte).
DEV uint32_t quant4(const float (&v)[4], float &scale) {
    float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    a = warp_max(a);
    scale = a > 0.f ? a / 448.f : 1.f;
    const float inv = __frcp_rn(scale);
    return e4m3x2(v[0] * inv, v[1] * inv) | (e4m3x2(v[2] * inv, v[3] * inv) << 16);
}

// ---------------------------------------------------------------- A0
// One token row m: h = x + res (the new residual, bf16), RMSNorm of those
// bf16 values, then per 128 columns e4m3 codes and a scale.  Warp w takes the
// 128-column blocks w, w + 8, ...; lane l columns 4l .. 4l + 3 of each.
DEV void glm_a0_task(const KParams &P, const Smem S, const WIns &I, int i, uint32_t &ured,
                                         bool ab) {
    constexpr int BPW = 8;  // blocks per warp: hidden <= 8192
    const int ct = threadIdx.x - CONSUMER_BASE, warp = ct >> 5, lane = ct & 31;
    const int m = F(I, P_ROW0), H = P.H, nb = H >> 7;
    const uint8_t *x = reinterpret_cast<const uint8_t *>(PTR(I, S_GA_X)) + (size_t)m * H * 2;
    const uint8_t *res = reinterpret_cast<const uint8_t *>(PTR(I, S_GA_RES)) + (size_t)m * H * 2;
    const uint8_t *nw = reinterpret_cast<const uint8_t *>(PTR(I, S_GA_NORM));
    uint8_t *rout = reinterpret_cast<uint8_t *>(PTR(I, S_GA_RES_OUT)) + (size_t)m * H * 2;
    uint8_t *qa = reinterpret_cast<uint8_t *>(PTR(I, S_GA_QA)) + (size_t)m * H;
    float *sa = reinterpret_cast<float *>(PTR(I, S_GA_SA)) + (size_t)m * nb;
    // every load first (one round trip), then the arithmetic
    uint2 xv[BPW], rv[BPW], wv[BPW];
#pragma unroll
    for (int j = 0; j < BPW; ++j) {
        const int blk = warp + CONSUMER_WARPS * j, col = blk * 128 + lane * 4;
        const bool in = blk < nb;
        xv[j] = in ? __ldg(reinterpret_cast<const uint2 *>(x + col * 2)) : make_uint2(0u, 0u);
        rv[j] = in ? __ldg(reinterpret_cast<const uint2 *>(res + col * 2)) : make_uint2(0u, 0u);
        wv[j] = in ? __ldg(reinterpret_cast<const uint2 *>(nw + col * 2)) : make_uint2(0u, 0u);
    }
    float h[BPW][4];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < BPW; ++j) {
        const int blk = warp + CONSUMER_WARPS * j, col = blk * 128 + lane * 4;
        h[j][0] = round_bf16(bf16_lo(xv[j].x) + bf16_lo(rv[j].x));
        h[j][1] = round_bf16(bf16_hi(xv[j].x) + bf16_hi(rv[j].x));
        h[j][2] = round_bf16(bf16_lo(xv[j].y) + bf16_lo(rv[j].y));
        h[j][3] = round_bf16(bf16_hi(xv[j].y) + bf16_hi(rv[j].y));
        if (blk < nb && !ab)
            *reinterpret_cast<uint2 *>(rout + col * 2) =
                make_uint2(pack_bf16(h[j][0], h[j][1]), pack_bf16(h[j][2], h[j][3]));
#pragma unroll
        for (int e = 0; e < 4; ++e) ss = fmaf(h[j][e], h[j][e], ss);  // zero past the row's end
    }
    ss = warp_sum(ss);
    trace_stamp(P, i, 9);
    float *red = S.red((int)(ured % NRED));
    ++ured;
    if (lane == 0) red[warp] = ss;
    consumer_bar();
    float tot = 0.f;
#pragma unroll
    for (int k = 0; k < CONSUMER_WARPS; ++k) tot += red[k];
    const float r = rsqrtf(tot / (float)H + P.eps);
    trace_stamp(P, i, 10);
#pragma unroll
    for (int j = 0; j < BPW; ++j) {
        const int blk = warp + CONSUMER_WARPS * j, col = blk * 128 + lane * 4;
        if (blk < nb) {  // warp-uniform
            const float y[4] = {h[j][0] * r * bf16_lo(wv[j].x), h[j][1] * r * bf16_hi(wv[j].x),
                                h[j][2] * r * bf16_lo(wv[j].y), h[j][3] * r * bf16_hi(wv[j].y)};
            float scale;
            const uint32_t codes = quant4(y, scale);
            if (!ab) {
                *reinterpret_cast<uint32_t *>(qa + col) = codes;
                if (lane == 0) sa[blk] = scale;
            }
        }
    }
    trace_stamp(P, i, 12);
}

// ---------------------------------------------------------------- GEMM tile
// out[m, out0 + c] for the M token rows and the tile's NR weight rows n0 + c:
// sum over 128-wide K blocks kb of sa[m, kb] * sw[n / 128, kb] * (a_kb . w_kb),
// rounded to bf16; a RoPE tile (64 columns, the last 64 of a head) then
// rotates pairs (c, c + 32) with the position's table entry and rounds again.
//
// Warp w takes the 8 weight rows (w mod NR/8) * 8 .. + 7 over K split
// KS = 64 / NR ways (part w / (NR/8)).  Within each 64-byte K chunk lane
// (g, t) = (lane / 4, lane % 4) loads 16 contiguous bytes of token rows g and
// g + 8 and of weight row g at offset 16 t, and feeds them to two MMAs: the K
// order inside the chunk is permuted the same way for A and B, which leaves
// the dot products unchanged.  The activation rows are staged in shared
// memory by the activation loader ([16][K + 16] codes, then [16][K / 128]
// scales); weight rows come from the tile's pages, whole rows per page.
template <int NR>
DEV void glm_gemm_task(const KParams &P, const Smem S, const WIns &I, int i, int sl, uint32_t &ring, uint32_t &ured,
                       bool &ab) {
    constexpr int NG = NR / 8, KS = CONSUMER_WARPS / NG;
    const int ct = threadIdx.x - CONSUMER_BASE, warp = ct >> 5, lane = ct & 31;
    const int g = lane >> 2, t = lane & 3, gi = warp % NG, ks = warp / NG;
    const int K = F(I, P_KC), KB = K >> 7, n0 = F(I, P_ROW0), rpp = F(I, P_RPP), npg = F(I, P_NPG);
    const int M = F(I, P_GL_M), ld = F(I, P_GL_LD), out0 = F(I, P_OUT0), rope = F(I, P_GL_ROPE), T = F(I, P_GL_T);
    const float *sw = reinterpret_cast<const float *>(PTR(I, S_GG_SW));
    __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(PTR(I, S_GG_OUT));
    const float2 *rtab = reinterpret_cast<const float2 *>(PTR(I, S_GG_ROPE));
    const int NP = P.num_pages;
    const uint32_t base = ring;
    ring += npg;
    const uint8_t *abuf = reinterpret_cast<const uint8_t *>(S.abuf(sl));
    const int astride = K + 16;
    const float *sa = reinterpret_cast<const float *>(abuf + GLM_MAX_M * astride);
    for (int k = 0; k < npg; ++k)
        if (!ab) ab = !warp_wait_bar(P, S, &S.full()[(base + k) % NP], ((base + k) / NP) & 1, 2, i, MK_OP_GLM_GEMM);
    trace_stamp(P, i, 7);
    const int r = gi * 8 + g;
    const uint8_t *wrow = S.pages() + (size_t)((base + r / rpp) % NP) * P.page_bytes + (size_t)(r % rpp) * K;
    const bool lo_ok = g < M, hi_ok = g + 8 < M;
    const uint8_t *alo = abuf + g * astride, *ahi = abuf + (g + 8) * astride;
    const int kb0 = ks * KB / KS, kb1 = (ks + 1) * KB / KS;
    // the weight scales of this warp's K blocks (at most 32), one per lane
    const float swl = lane < kb1 - kb0 ? __ldg(sw + (size_t)((n0 + gi * 8) >> 7) * KB + kb0 + lane) : 0.f;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    // Two K blocks per iteration and one accumulator set per MMA: eight
    // independent MMAs in flight instead of a chain of four.
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    auto block = [&](int kb, float (&c)[4][4]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int off = kb * 128 + h * 64 + t * 16;
            const uint4 w = *reinterpret_cast<const uint4 *>(wrow + off);
            const uint4 a = lo_ok ? *reinterpret_cast<const uint4 *>(alo + off) : zero;
            const uint4 b = hi_ok ? *reinterpret_cast<const uint4 *>(ahi + off) : zero;
            mma_e4m3(c[2 * h], a.x, b.x, a.y, b.y, w.x, w.y);
            mma_e4m3(c[2 * h + 1], a.z, b.z, a.w, b.w, w.z, w.w);
        }
    };
    auto scale_add = [&](int kb, const float (&c)[4][4]) {
        const float swv = __shfl_sync(FULL, swl, kb - kb0);
        const float s0 = lo_ok ? sa[g * KB + kb] * swv : 0.f;
        const float s1 = hi_ok ? sa[(g + 8) * KB + kb] * swv : 0.f;
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = (c[0][e] + c[1][e]) + (c[2][e] + c[3][e]);
        acc[0] = fmaf(s0, v[0], acc[0]);
        acc[1] = fmaf(s0, v[1], acc[1]);
        acc[2] = fmaf(s1, v[2], acc[2]);
        acc[3] = fmaf(s1, v[3], acc[3]);
    };
    int kb = kb0;
    for (; kb + 2 <= kb1; kb += 2) {
        float c0[4][4] = {}, c1[4][4] = {};
        block(kb, c0);
        block(kb + 1, c1);
        scale_add(kb, c0);
        scale_add(kb + 1, c1);
    }
    if (kb < kb1) {
        float c0[4][4] = {};
        block(kb, c0);
        scale_add(kb, c0);
    }
    __syncwarp();
    trace_stamp(P, i, 9);
    if (lane == 0) {
        for (int k = 0; k < npg; ++k) mbar_arrive(&S.empty()[(base + k) % NP]);
        mbar_arrive(&S.act_empty()[sl]);  // staged rows no longer needed by this warp
    }
    // partials [KS][16][NR] in a reduction buffer (its previous user, NRED
    // buffer uses back, finished before every warp passed a later barrier)
    float *red = S.red((int)(ured % NRED));
    ++ured;
    float *pr = red + ks * GLM_MAX_M * NR;
    const int n = gi * 8 + 2 * t;
    pr[g * NR + n] = acc[0];
    pr[g * NR + n + 1] = acc[1];
    pr[(g + 8) * NR + n] = acc[2];
    pr[(g + 8) * NR + n + 1] = acc[3];
    consumer_bar();
    trace_stamp(P, i, 10);
    if (ab) return;
    for (int e = ct; e < M * NR; e += CONSUMERS) {
        const int m = e / NR, c = e % NR;
        float v = 0.f, o = 0.f;
#pragma unroll
        for (int k = 0; k < KS; ++k) v += red[k * GLM_MAX_M * NR + m * NR + c];
        v = round_bf16(v);
        if (NR == 64 && rope) {
#pragma unroll
            for (int k = 0; k < KS; ++k) o += red[k * GLM_MAX_M * NR + m * NR + (c ^ 32)];
            o = round_bf16(o);
            const float2 cs = rtab[(m % T) * 32 + (c & 31)];
            v = c < 32 ? v * cs.x - o * cs.y : v * cs.x + o * cs.y;
        }
        out[(size_t)m * ld + out0 + c] = __float2bfloat16_rn(v);
    }
}

// ---------------------------------------------------------------- FIN
// One token row m of request m / T at slot pos0 + m % T: q-lora (QKV-A
// columns 0 .. QL-1) re-quantised per 128 columns, one warp per block; the
// latent cache row = kv-lora || RoPE(k_pe); the index cache row = Indexer-K
// with RoPE on its last 64 columns.  With the tensor-core tiles (SUMS) the
// first GEMMs left fp32 sums: FIN reads each value of its row once from
// them, rounds it to bf16 (the GEMM output), stores that and zeroes the sum
// -- the Head-Gate row too.  Every thread loads all its values before any
// store (one round trip); the plan keeps each part within one pass of the
// 256 consumer threads (q-lora <= 16 blocks, kv-lora <= 512, Indexer-K's
// unroped part <= 512, Head-Gate <= 256).
template <bool SUMS>  // the tensor-core instance: the first GEMMs left fp32 sums
DEV void glm_fin_task(const KParams &P, const WIns &I, bool ab) {
    const int ct = threadIdx.x - CONSUMER_BASE, warp = ct >> 5, lane = ct & 31;
    const int m = F(I, P_ROW0), QL = F(I, P_GF_QLORA), KL = F(I, P_GF_KVLORA), ID = F(I, P_GF_IDX);
    const int slots = F(I, P_GF_SLOTS), LDQ = F(I, P_GF_QKVA_LD), T = F(I, P_GL_T), pos0 = F(I, P_GL_POS0);
    const int G = F(I, P_GF_GATE);
    __nv_bfloat16 *qkva = reinterpret_cast<__nv_bfloat16 *>(PTR(I, S_GF_QKVA)) + (size_t)m * LDQ;
    __nv_bfloat16 *ik = reinterpret_cast<__nv_bfloat16 *>(PTR(I, S_GF_IK)) + (size_t)m * ID;
    uint8_t *qb = reinterpret_cast<uint8_t *>(PTR(I, S_GF_QB)) + (size_t)m * QL;
    float *sb = reinterpret_cast<float *>(PTR(I, S_GF_SB)) + (size_t)m * (QL >> 7);
    __nv_bfloat16 *lat = reinterpret_cast<__nv_bfloat16 *>(PTR(I, S_GF_LAT));
    __nv_bfloat16 *idx = reinterpret_cast<__nv_bfloat16 *>(PTR(I, S_GF_IDX));
    const float2 *rtab = reinterpret_cast<const float2 *>(PTR(I, S_GF_ROPE));
    float *fq = SUMS ? reinterpret_cast<float *>(PTR(I, S_GF_FQKVA)) + (size_t)m * LDQ : nullptr;
    float *fi = SUMS ? reinterpret_cast<float *>(PTR(I, S_GF_FIK)) + (size_t)m * ID : nullptr;
    float *fg = SUMS ? reinterpret_cast<float *>(PTR(I, S_GF_FGATE)) + (size_t)m * G : nullptr;
    __nv_bfloat16 *gate = SUMS ? reinterpret_cast<__nv_bfloat16 *>(PTR(I, S_GF_GATE)) + (size_t)m * G : nullptr;
    if (ab) return;
    const int req = m / T, j = m % T, slot = pos0 + j, p = ct & 31, nqb = QL >> 7;
    // what this thread handles: a RoPE pair (threads 0-31 the k_pe slice,
    // 32-63 Indexer-K's last 64), up to two q-lora blocks' 4 values, a
    // kv-lora pair, an unroped Indexer-K pair, a Head-Gate value
    const bool has_rp = ct < 64, has_l = ct * 2 < KL, has_i = ct * 2 < ID - GLM_ROPE, has_g = SUMS && ct < G;
    const int c_rp = ct < 32 ? QL + KL + p : ID - GLM_ROPE + p;  // column in QKV-A (ct < 32) or Indexer-K
    float rp[2] = {0.f, 0.f}, qv[2][4] = {}, lv[2] = {0.f, 0.f}, iv[2] = {0.f, 0.f}, gv = 0.f;
    if constexpr (SUMS) {
        float *fr = ct < 32 ? fq : fi;
        if (has_rp) {
            rp[0] = __ldcg(fr + c_rp);
            rp[1] = __ldcg(fr + c_rp + 32);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int blk = warp + CONSUMER_WARPS * k;
            if (blk < nqb) {
                const float4 x = __ldcg(reinterpret_cast<const float4 *>(fq + blk * 128 + lane * 4));
                qv[k][0] = x.x; qv[k][1] = x.y; qv[k][2] = x.z; qv[k][3] = x.w;
            }
        }
        if (has_l) {
            const float2 x = __ldcg(reinterpret_cast<const float2 *>(fq + QL + ct * 2));
            lv[0] = x.x; lv[1] = x.y;
        }
        if (has_i) {
            const float2 x = __ldcg(reinterpret_cast<const float2 *>(fi + ct * 2));
            iv[0] = x.x; iv[1] = x.y;
        }
        if (has_g) gv = __ldcg(fg + ct);
        // the GEMM outputs: every sum rounded to bf16, stored, and zeroed for the next step
        auto r = [](float &v) { v = round_bf16(v); };
        if (has_rp) {
            __nv_bfloat16 *o = ct < 32 ? qkva : ik;
            r(rp[0]); r(rp[1]);
            o[c_rp] = __float2bfloat16_rn(rp[0]);
            o[c_rp + 32] = __float2bfloat16_rn(rp[1]);
            __stcg(fr + c_rp, 0.f);
            __stcg(fr + c_rp + 32, 0.f);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int blk = warp + CONSUMER_WARPS * k, col = blk * 128 + lane * 4;
            if (blk < nqb) {
                for (int e = 0; e < 4; ++e) r(qv[k][e]);
                *reinterpret_cast<uint2 *>(qkva + col) =
                    make_uint2(pack_bf16(qv[k][0], qv[k][1]), pack_bf16(qv[k][2], qv[k][3]));
                __stcg(reinterpret_cast<float4 *>(fq + col), make_float4(0.f, 0.f, 0.f, 0.f));
            }
        }
        if (has_l) {
            r(lv[0]); r(lv[1]);
            *reinterpret_cast<uint32_t *>(qkva + QL + ct * 2) = pack_bf16(lv[0], lv[1]);
            __stcg(reinterpret_cast<float2 *>(fq + QL + ct * 2), make_float2(0.f, 0.f));
        }
        if (has_i) {
            r(iv[0]); r(iv[1]);
            *reinterpret_cast<uint32_t *>(ik + ct * 2) = pack_bf16(iv[0], iv[1]);
            __stcg(reinterpret_cast<float2 *>(fi + ct * 2), make_float2(0.f, 0.f));
        }
        if (has_g) {
            r(gv);
            gate[ct] = __float2bfloat16_rn(gv);
            __stcg(fg + ct, 0.f);
        }
    } else {
        const unsigned short *br = reinterpret_cast<const unsigned short *>(ct < 32 ? qkva : ik);
        if (has_rp) {
            rp[0] = __uint_as_float((uint32_t)__ldcg(br + c_rp) << 16);
            rp[1] = __uint_as_float((uint32_t)__ldcg(br + c_rp + 32) << 16);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int blk = warp + CONSUMER_WARPS * k;
            if (blk < nqb) {
                const uint2 u = __ldcg(reinterpret_cast<const uint2 *>(qkva + blk * 128 + lane * 4));
                qv[k][0] = bf16_lo(u.x); qv[k][1] = bf16_hi(u.x); qv[k][2] = bf16_lo(u.y); qv[k][3] = bf16_hi(u.y);
            }
        }
        if (has_l) {
            const uint32_t u = __ldcg(reinterpret_cast<const uint32_t *>(qkva + QL + ct * 2));
            lv[0] = bf16_lo(u); lv[1] = bf16_hi(u);
        }
        if (has_i) {
            const uint32_t u = __ldcg(reinterpret_cast<const uint32_t *>(ik + ct * 2));
            iv[0] = bf16_lo(u); iv[1] = bf16_hi(u);
        }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int blk = warp + CONSUMER_WARPS * k, col = blk * 128 + lane * 4;
        if (blk < nqb) {  // warp-uniform
            float scale;
            const uint32_t codes = quant4(qv[k], scale);
            *reinterpret_cast<uint32_t *>(qb + col) = codes;
            if (lane == 0) sb[blk] = scale;
        }
    }
    __nv_bfloat16 *lrow = lat + ((size_t)req * slots + slot) * (KL + GLM_ROPE);
    __nv_bfloat16 *irow = idx + ((size_t)req * slots + slot) * ID;
    if (has_l) *reinterpret_cast<uint32_t *>(lrow + ct * 2) = pack_bf16(lv[0], lv[1]);
    if (has_i) *reinterpret_cast<uint32_t *>(irow + ct * 2) = pack_bf16(iv[0], iv[1]);
    if (has_rp) {
        __nv_bfloat16 *dst = ct < 32 ? lrow + KL : irow + ID - GLM_ROPE;
        const float2 cs = rtab[j * 32 + p];
        dst[p] = __float2bfloat16_rn(rp[0] * cs.x - rp[1] * cs.y);
        dst[p + 32] = __float2bfloat16_rn(rp[1] * cs.x + rp[0] * cs.y);
    }
}

// ---------------------------------------------------------------- staging
// Activation loader, GEMM tiles: after the tile's events were acquired, bulk
// copies of the M activation rows (into rows of K + 16 bytes) and of their
// scales into the activation buffer, completing on the slot's full barrier.
// Returns the bytes in flight (0 if the buffer already holds this input).
DEV uint32_t stage_glm(const KParams &P, const WIns &I, uint8_t *abuf, uint64_t *full) {
    const int lane = threadIdx.x & 31;
    const int K = F(I, P_KC), M = F(I, P_GL_M);
    const uint8_t *xq = reinterpret_cast<const uint8_t *>(PTR(I, S_GG_XQ));
    const uint8_t *xs = reinterpret_cast<const uint8_t *>(PTR(I, S_GG_XS));
    const uint32_t sbytes = (uint32_t)M * (uint32_t)(K >> 7) * 4u;
    const uint32_t bytes = (uint32_t)M * (uint32_t)K + sbytes;
    if (lane == 0) {
        // the acquire of the tile's events (generic proxy) before the bulk reads (async proxy)
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_expect_tx(full, bytes);
        for (int m = 0; m < M; ++m) bulk_g2s_plain(abuf + (size_t)m * (K + 16), xq + (size_t)m * K, (uint32_t)K, full);
        bulk_g2s_plain(abuf + (size_t)GLM_MAX_M * (K + 16), xs, sbytes, full);
    }
    __syncwarp();
    return bytes;
}

}  // namespace mk
