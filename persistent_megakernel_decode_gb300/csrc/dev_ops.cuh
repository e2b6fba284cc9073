// Op bodies of the interpreter: what the activation loader stages for each
// opcode and what the consumer warps compute from the page ring.
//
// GEMV tiles (QKV, O, MLP-up, MLP-down, LM head) follow "CMU 15-779 Lecture 7
// notes", section 5.1 (fused RMSNorm+QKV, O-proj+residual, RMSNorm+up/gate+
// SiLU, down+residual with a counter per K chunk, RMSNorm+LM head); the
// attention task is split over KV positions and the last split of a
// (sequence, kv head) merges the partials (the same section's attention and
// attention-reduction instructions).  RoPE and the KV-cache append sit in the
// attention task's activation stage instead of the QKV epilogue, because a
// QKV tile holds 16 rows of a head and RoPE pairs dimension i with i + D/2.
#pragma once
#include <cuda_fp16.h>

#include <type_traits>

#include "dev_common.cuh"

namespace mk {

// ================================================================ activation stage (one warp)

// RMSNorm-fused ops stage x^ = h * rsqrt(mean(h^2) + eps) * w (fp32); O and
// DOWN stage the attention output / their K chunk of the MLP activation.
// Every load of a round is issued before any is used (up to SC float4 of the
// activation and SC norm-weight quads per lane), so a staging costs a few
// L2 round trips rather than one per loop iteration.
constexpr int SC = 8;

// Batch-1 row-per-warp tiles read x as 8-wide chunks c = lane + 32 k, two
// float4 per chunk.  Staged in natural order, a warp's float4 loads would
// touch 32-byte-strided addresses (two lanes per bank group); the activation
// loader stages those tiles' x "lane-interleaved" instead: float4 q of the
// natural order (chunk q / 2, half q % 2) goes to position
// ((k * 2 + half) * 32 + lane) -- every warp load is then 512 contiguous bytes.
DEV int rpw_perm4(int q) {
    const int c = q >> 1;
    return (((c >> 5) << 1) + (q & 1)) * 32 + (c & 31);
}
// FP8 row-per-warp tiles read x as 16-wide chunks c = lane + 32 k, four
// float4 per chunk: float4 q (chunk q / 4, quarter q % 4) goes to position
// ((k * 4 + quarter) * 32 + lane).
DEV int rpw_perm8(int q) {
    const int c = q >> 2;
    return (((c >> 5) << 2) + (q & 3)) * 32 + (c & 31);
}
// Staging position of float4 q: natural order, or one of the two lane-interleaved orders.
template <bool P8>
DEV int stage_pos(int q, bool perm, bool perm8) {
    if constexpr (P8) {
        if (perm8) return rpw_perm8(q);
    }
    return perm ? rpw_perm4(q) : q;
}

// h * w (w: four bf16) and x * s, elementwise
DEV float4 wmul(float4 x, uint2 w) {
    x.x *= __uint_as_float(w.x << 16);
    x.y *= __uint_as_float(w.x & 0xffff0000u);
    x.z *= __uint_as_float(w.y << 16);
    x.w *= __uint_as_float(w.y & 0xffff0000u);
    return x;
}
DEV float4 fscale(float4 x, float s) {
    x.x *= s;
    x.y *= s;
    x.z *= s;
    x.w *= s;
    return x;
}

template <bool P8 = false>
DEV void stage_copy(const float4 *s4, float4 *d4, int n4, bool perm, bool perm8 = false) {
    const int lane = threadIdx.x & 31;
    for (int base = 0; base < n4; base += 32 * SC) {
        float4 v[SC];
#pragma unroll
        for (int j = 0; j < SC; ++j) {
            const int k = base + lane + 32 * j;
            if (k < n4) v[j] = __ldcg(s4 + k);
        }
#pragma unroll
        for (int j = 0; j < SC; ++j) {
            const int k = base + lane + 32 * j;
            if (k < n4) d4[stage_pos<P8>(k, perm, perm8)] = v[j];
        }
    }
}

// P8 (the FP8 instance): `perm8` stages x in the FP8 tiles' order (rpw_perm8).
template <int MAXB, bool P8 = false>
DEV void stage_gemv(const KParams &P, const WIns &I, float *abuf, bool ab, bool perm, bool perm8 = false) {
    const int lane = threadIdx.x & 31;
    const int opc = F(I, W_OPC);
    const int B = P.B;
    if (opc == MK_OP_QKV || opc == MK_OP_UP || opc == MK_OP_LM) {
        const int H = P.H, n4 = H / 4;
        const float *h = reinterpret_cast<const float *>(
            PTR(I, opc == MK_OP_QKV ? S_QKV_H : opc == MK_OP_UP ? S_UP_H : S_LM_H));
        const uint2 *w4 = reinterpret_cast<const uint2 *>(
            PTR(I, opc == MK_OP_QKV ? S_QKV_NORM : opc == MK_OP_UP ? S_UP_NORM : S_LM_NORM));
        const int snap = F(I, P_SNAP);
        float *hist = nullptr;
        if (snap > 0 && !ab) hist = reinterpret_cast<float *>(PTR(I, opc == MK_OP_QKV ? S_QKV_HIST : S_LM_HIST));
        const bool one_round = n4 <= 32 * SC;
        for (int b = 0; b < B; ++b) {
            const float4 *src = reinterpret_cast<const float4 *>(h + (size_t)b * H);
            float4 *dst = reinterpret_cast<float4 *>(abuf + (size_t)b * H);
            float4 *hs = hist ? reinterpret_cast<float4 *>(hist + ((size_t)(snap - 1) * B + b) * H) : nullptr;
            float ss = 0.f;
            float4 v[SC];
            uint2 ww[SC];
            for (int base = 0; base < n4; base += 32 * SC) {
#pragma unroll
                for (int j = 0; j < SC; ++j) {
                    const int k = base + lane + 32 * j;
                    if (k < n4) {
                        v[j] = __ldcg(src + k);
                        ww[j] = __ldg(w4 + k);
                    }
                }
#pragma unroll
                for (int j = 0; j < SC; ++j) {
                    const int k = base + lane + 32 * j;
                    if (k < n4) {
                        ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
                        if (!one_round) dst[stage_pos<P8>(k, perm, perm8)] = wmul(v[j], ww[j]);
                        if (hs) hs[k] = v[j];
                    }
                }
            }
            ss = warp_sum(ss);
            const float scale = rsqrtf(ss / (float)H + P.eps);
            if (one_round) {
#pragma unroll
                for (int j = 0; j < SC; ++j) {
                    const int k = lane + 32 * j;
                    if (k < n4) dst[stage_pos<P8>(k, perm, perm8)] = fscale(wmul(v[j], ww[j]), scale);
                }
            } else {
                // h * w went to shared memory as each round arrived (the
                // weights are not loaded twice): apply the scale in place, each
                // lane to the positions it wrote, a round's loads issued before
                // its stores
                for (int base = 0; base < n4; base += 32 * (SC / 2)) {
                    float4 y[SC / 2];
#pragma unroll
                    for (int j = 0; j < SC / 2; ++j) {
                        const int k = base + lane + 32 * j;
                        if (k < n4) y[j] = dst[stage_pos<P8>(k, perm, perm8)];
                    }
#pragma unroll
                    for (int j = 0; j < SC / 2; ++j) {
                        const int k = base + lane + 32 * j;
                        if (k < n4) dst[stage_pos<P8>(k, perm, perm8)] = fscale(y[j], scale);
                    }
                }
            }
        }
    } else {
        const int kc = F(I, P_KC);
        const float *src;
        size_t ld;
        if (opc == MK_OP_O) {
            src = reinterpret_cast<const float *>(PTR(I, S_O_IN));
            ld = (size_t)P.Hq * P.D;
        } else {
            src = reinterpret_cast<const float *>(PTR(I, S_DN_IN)) + F(I, P_K0);
            ld = (size_t)P.F;
        }
        for (int b = 0; b < B; ++b)
            stage_copy<P8>(reinterpret_cast<const float4 *>(src + b * ld),
                           reinterpret_cast<float4 *>(abuf + (size_t)b * kc), kc / 4, perm, perm8);
    }
}

// O tiles add their rows of the residual stream; the activation loader stages
// that slice into the slot's tail so the consumers' epilogue reads shared memory.
DEV float *slot_resid(const KParams &P, float *slot) { return slot + (P.act_bytes / 4 - P.B * RESID_ROWS); }
DEV void stage_resid(const KParams &P, const WIns &I, float *slot) {
    const int lane = threadIdx.x & 31;
    const float *hres = reinterpret_cast<const float *>(PTR(I, S_O_HRES));
    const int out0 = F(I, P_OUT0), nrows = F(I, P_NROWS);
    float *resid = slot_resid(P, slot);
    for (int k = lane; k < P.B * RESID_ROWS; k += 32) {
        const int b = k / RESID_ROWS, r = k % RESID_ROWS;
        resid[k] = r < nrows ? __ldcg(hres + (size_t)b * P.H + out0 + r) : 0.f;
    }
}
// Batch 1 (RESID_ROWS <= 32 values): the load is issued before the
// activation's first round and stored after it, so both share a round trip.
DEV float resid_load1(const WIns &I) {
    const int lane = threadIdx.x & 31;
    // (instruction fields are warp shuffles: read them in uniform code)
    const float *hres = reinterpret_cast<const float *>(PTR(I, S_O_HRES));
    const int out0 = F(I, P_OUT0), nrows = min(F(I, P_NROWS), RESID_ROWS);
    return lane < nrows ? __ldcg(hres + out0 + lane) : 0.f;
}
DEV void resid_store1(const KParams &P, float *slot, float v) {
    const int lane = threadIdx.x & 31;
    if (lane < RESID_ROWS) slot_resid(P, slot)[lane] = v;
}
static_assert(RESID_ROWS <= 32, "batch-1 residual staging: one value per lane");

// q (pre-scaled by log2(e)/sqrt(D)), new k and v of one (sequence, kv group):
// q/k RMSNorm (optional), RoPE at the new position (rotate-half pairs,
// theta_i = theta^(-2i/D)), bf16 rounding of the new k/v, and the KV-cache
// append by the split that owns the new position.  Slot layout: q as
// [G][4 quarters][D/4 + 4] (padded against bank conflicts), then k, then v.
// RoPE factors of one position for this lane's dimension pairs, cached by
// the activation loader across attention tasks of the same position.
template <int D>
struct Rope {
    int pos = -1;
    float cs[D / 64], sn[D / 64];
    DEV void at(const KParams &P, int p) {
        if (p == pos) return;
        pos = p;
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int j = 0; j < D / 64; ++j) {
            // angle of pair i in double, reduced mod 2 pi, then a float sincos
            const int i = lane + 32 * j;
            const double inv_freq = exp2(-(2.0 * i / D) * log2((double)P.theta));
            const double ang = (double)p * inv_freq;
            const double two_pi = 6.283185307179586476925286766559;
            const double red = ang - rint(ang / two_pi) * two_pi;
            sincosf((float)red, &sn[j], &cs[j]);
        }
    }
};

template <int D, int GMAX>  // GMAX: bound on the q heads per kv head
DEV void stage_attn(const KParams &P, const WIns &I, float *slot, bool ab, Rope<D> &rope) {
    constexpr int PER = D / 32;
    constexpr int QS = D / 4 + 4;
    const int lane = threadIdx.x & 31;
    const int G = P.Hq / P.Hkv, b = F(I, P_B), g = F(I, P_G);
    const int pos = attn_pos(P, I);
    const int t0 = F(I, P_T0), T = F(I, P_T);
    const float *src = reinterpret_cast<const float *>(PTR(I, S_AT_QKV)) + ((size_t)b * P.Hkv + g) * (G + 2) * D;
    const uint16_t *wq = reinterpret_cast<const uint16_t *>(PTR(I, S_AT_QN));
    const uint16_t *wk = reinterpret_cast<const uint16_t *>(PTR(I, S_AT_KN));
    float *qp = slot;
    float *kn = slot + G * 4 * QS;
    float *vn = kn + D;
    const float qscale = rsqrtf((float)D) * 1.4426950408889634f;
    // every head's values in flight at once
    float x[GMAX + 2][PER];
#pragma unroll
    for (int h = 0; h < GMAX + 2; ++h)
#pragma unroll
        for (int e = 0; e < PER; ++e) x[h][e] = h < G + 2 ? __ldcg(src + (size_t)h * D + lane + 32 * e) : 0.f;
    rope.at(P, pos);
#pragma unroll
    for (int h = 0; h < GMAX + 2; ++h) {
        if (h >= G + 2) continue;
        const bool is_q = h < G, is_k = h == G;
        if (P.qk_norm && (is_q || is_k)) {
            const uint16_t *w = is_q ? wq : wk;
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < PER; ++e) ss += x[h][e] * x[h][e];
            ss = warp_sum(ss);
            const float sc = rsqrtf(ss / (float)D + P.eps);
#pragma unroll
            for (int e = 0; e < PER; ++e) x[h][e] = x[h][e] * sc * bf16_at(w, lane + 32 * e);
        }
        if (is_q || is_k) {
#pragma unroll
            for (int e = 0; e < PER / 2; ++e) {   // element lane+32e pairs with lane+32e+D/2
                const float a = x[h][e], c = x[h][e + PER / 2];
                x[h][e] = a * rope.cs[e] - c * rope.sn[e];
                x[h][e + PER / 2] = a * rope.sn[e] + c * rope.cs[e];
            }
        }
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int d = lane + 32 * e;
            if (is_q) qp[(h * 4 + d / (D / 4)) * QS + d % (D / 4)] = x[h][e] * qscale;
            else if (is_k) kn[d] = round_bf16(x[h][e]);
            else vn[d] = round_bf16(x[h][e]);
        }
    }
    if (!ab && pos >= t0 && pos < t0 + T) {
        __syncwarp();
        const size_t c = (((size_t)b * P.Hkv + g) * P.Smax + pos) * D;
        __nv_bfloat16 *kc = reinterpret_cast<__nv_bfloat16 *>(PTR(I, S_AT_K)) + c;
        __nv_bfloat16 *vc = reinterpret_cast<__nv_bfloat16 *>(PTR(I, S_AT_V)) + c;
        for (int d = lane; d < D; d += 32) {
            kc[d] = __float2bfloat16_rn(kn[d]);
            vc[d] = __float2bfloat16_rn(vn[d]);
        }
    }
}

// ================================================================ consumers (8 warps)

template <int MAXB>
__host__ __device__ constexpr int rows_max() { return MAXB > 4 ? 8 : MAX_TILE_ROWS; }

// x of one consumer thread: its 8-wide K chunks of every sequence.  Batch 1
// keeps them as fp32 pairs for the packed multiply-add (two partial sums per
// row, even and odd columns); larger batches keep plain floats (one sum per
// row and sequence) to stay within the register budget.
template <int MAXB, int NCH>
struct XChunks {
    static constexpr bool PAIRS = MAXB == 1;
    using Acc = std::conditional_t<PAIRS, uint64_t, float>;
    uint64_t v[PAIRS ? NCH : 1][4];
    float f[PAIRS ? 1 : NCH][MAXB][8];
    DEV void load(const float *xs, int ct, int nchunk, int kc, int B) {
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
            const int c = ct + CONSUMERS * j;
#pragma unroll
            for (int b = 0; b < MAXB; ++b) {
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), bb = a;
                if (c < nchunk && b < B) {
                    const float4 *s4 = reinterpret_cast<const float4 *>(xs + (size_t)b * kc + c * 8);
                    a = s4[0];
                    bb = s4[1];
                }
                if constexpr (PAIRS) {
                    v[j][0] = pack2(a.x, a.y); v[j][1] = pack2(a.z, a.w);
                    v[j][2] = pack2(bb.x, bb.y); v[j][3] = pack2(bb.z, bb.w);
                } else {
                    f[j][b][0] = a.x; f[j][b][1] = a.y; f[j][b][2] = a.z; f[j][b][3] = a.w;
                    f[j][b][4] = bb.x; f[j][b][5] = bb.y; f[j][b][6] = bb.z; f[j][b][7] = bb.w;
                }
            }
        }
    }
    DEV static float value(Acc a) {
        if constexpr (PAIRS) return sum2(a);
        else return a;
    }
};

// acc[b] += one weight row chunk . x (sequence b)
template <int MAXB, int NCH>
DEV void row_dot(const uint8_t *wrow, int ct, int nchunk, const XChunks<MAXB, NCH> &x,
                 typename XChunks<MAXB, NCH>::Acc (&acc)[MAXB]) {
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
        const int c = ct + CONSUMERS * j;
        if (c < nchunk) {
            const uint4 w = *reinterpret_cast<const uint4 *>(wrow + c * 16);
            if constexpr (XChunks<MAXB, NCH>::PAIRS) {
                fma2(acc[0], bf16x2_pair(w.x), x.v[j][0]);
                fma2(acc[0], bf16x2_pair(w.y), x.v[j][1]);
                fma2(acc[0], bf16x2_pair(w.z), x.v[j][2]);
                fma2(acc[0], bf16x2_pair(w.w), x.v[j][3]);
            } else {
                float w8[8];
                bf16x8(w, w8);
#pragma unroll
                for (int b = 0; b < MAXB; ++b)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[b] = fmaf(w8[e], x.f[j][b][e], acc[b]);
            }
        }
    }
}

// Branch-free variant: every thread loads a chunk (threads past the row's
// end re-read chunk 0 and zero it with `mask`), so the rows of a page can all
// be in flight at once.
template <int MAXB, int NCH>
DEV void row_dot_nb(const uint8_t *wrow, const int (&off)[NCH], const uint32_t (&mask)[NCH],
                    const XChunks<MAXB, NCH> &x, typename XChunks<MAXB, NCH>::Acc (&acc)[MAXB]) {
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
        uint4 w = *reinterpret_cast<const uint4 *>(wrow + off[j]);
        w.x &= mask[j]; w.y &= mask[j]; w.z &= mask[j]; w.w &= mask[j];
        if constexpr (XChunks<MAXB, NCH>::PAIRS) {
            fma2(acc[0], bf16x2_pair(w.x), x.v[j][0]);
            fma2(acc[0], bf16x2_pair(w.y), x.v[j][1]);
            fma2(acc[0], bf16x2_pair(w.z), x.v[j][2]);
            fma2(acc[0], bf16x2_pair(w.w), x.v[j][3]);
        } else {
            float w8[8];
            bf16x8(w, w8);
#pragma unroll
            for (int b = 0; b < MAXB; ++b)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[b] = fmaf(w8[e], x.f[j][b][e], acc[b]);
        }
    }
}

// One GEMV tile (QKV, O, MLP-up, MLP-down, LM head) split over K: consumer
// thread t holds the 8-wide K chunks t, t + 256, ... of x for every sequence
// in registers (x is read once per tile, 4 bytes per weight column), so each
// warp reads a contiguous 512-byte slice of every weight row.  The tile's rows
// (MLP-up: gate rows, then up rows) lie in its pages in order, RPP to a page
// at most.  Each warp's partial sums are reduced across its lanes with a
// transposed butterfly and parked in one of NRED shared buffers; after a
// hardware barrier of the 8 consumer warps, one warp (rotating) sums the
// partials in warp order and runs the epilogue while the others move on to
// the next instruction.  ONE_PAGE: the whole tile is on one page
// (one wait, one release, one butterfly); otherwise each page is reduced on
// its own.  Returns whether this warp ran the epilogue (wrote global memory).
template <int MAXB, int NCH, int RPP, bool ONE_PAGE>
DEV bool gemv_tile(const KParams &P, const Smem S, const WIns &I, int i, int sl, const float *slot, uint32_t &ring,
                   RingPos &rq, uint32_t &ured, unsigned long long &lm_best, bool &ab) {
    constexpr int RMAX = rows_max<MAXB>();
    constexpr int VT = RMAX * MAXB;            // partials per warp in a reduction buffer: row * MAXB + b
    constexpr int VL = VT >= 32 ? VT / 32 : 1; // epilogue values per lane: v = lane + 32 j
    const int ct = threadIdx.x - CONSUMER_BASE, warp = ct >> 5, lane = ct & 31;
    const int opc = F(I, W_OPC);
    const int kc = F(I, P_KC), nrows = F(I, P_NROWS), npg = F(I, P_NPG);
    const int total = (opc == MK_OP_UP ? 2 : 1) * nrows;
    const int rpp = min(F(I, P_RPP), RPP);
    const int nchunk = kc >> 3, row_bytes = kc * 2;
    const int B = P.B;
    using X = XChunks<MAXB, NCH>;
    X x;
    x.load(S.abuf(sl), ct, nchunk, kc, B);
    // O tiles: the residual values this lane would need in the epilogue, read
    // before the slot is released (any warp may turn out to run the epilogue)
    float resid_v[VL];
#pragma unroll
    for (int j = 0; j < VL; ++j) resid_v[j] = 0.f;
    if (opc == MK_OP_O) {
        const float *rs = slot_resid(P, const_cast<float *>(slot));
#pragma unroll
        for (int j = 0; j < VL; ++j) {
            const int v = lane + 32 * j, r = v / MAXB, b = v % MAXB;
            if (v < VT && b < B && r < nrows) resid_v[j] = rs[b * RESID_ROWS + r];
        }
    }
    if constexpr (!ONE_PAGE) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.act_empty()[sl]);  // activation buffer and slot no longer needed
    }

    // The reduction buffer this tile uses.  Its previous user, NRED GEMV tiles
    // back, has finished its epilogue: the epilogue warp of a tile passes the
    // next GEMV tile's barrier only after it, and every writer of this tile
    // has passed that barrier too.
    const int rb = (int)(ured % NRED);
    const uint32_t use = ured / NRED;
    ++ured;
    float *red = S.red(rb) + warp * VT;
    ring += npg;

    if constexpr (ONE_PAGE) {
        // all RPP rows of the page, unconditionally: the caller guarantees
        // RPP * row_bytes <= page_bytes, and rows past the tile's end (stale
        // page bytes) only feed partials that the epilogue never reads
        int off[NCH];
        uint32_t mask[NCH];
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
            const int c = ct + CONSUMERS * j;
            off[j] = (c < nchunk ? c : 0) * 16;
            mask[j] = c < nchunk ? 0xffffffffu : 0u;
        }
        typename X::Acc acc[RMAX][MAXB];
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
#pragma unroll
            for (int b = 0; b < MAXB; ++b) acc[r][b] = 0;
        if (!ab) ab = !warp_wait_bar(P, S, &S.full()[rq.p], rq.ph, 2, i, opc);
        const uint8_t *page = S.pages() + (size_t)rq.p * P.page_bytes;
#pragma unroll
        for (int r = 0; r < RPP; ++r) row_dot_nb<MAXB, NCH>(page + (size_t)r * row_bytes, off, mask, x, acc[r]);
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&S.empty()[rq.p]);
            mbar_arrive(&S.act_empty()[sl]);  // activation buffer and slot no longer needed
        }
        rq.next(P.num_pages);
        float v[VT];
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
#pragma unroll
            for (int b = 0; b < MAXB; ++b) v[r * MAXB + b] = X::value(acc[r][b]);
        Bfly<VT, 16>::run(v, lane);
        if constexpr (VT >= 32) {
#pragma unroll
            for (int j = 0; j < VT / 32; ++j) red[lane * (VT / 32) + j] = v[j];
        } else {
            if ((lane & (32 / VT - 1)) == 0) red[lane / (32 / VT)] = v[0];
        }
    } else {
        constexpr int VP = RPP * MAXB;
        for (int pg = 0; pg < npg; ++pg) {
            const int r0 = pg * rpp, cnt = min(rpp, total - r0);
            if (!ab) ab = !warp_wait_bar(P, S, &S.full()[rq.p], rq.ph, 2, i, opc);
            const uint8_t *page = S.pages() + (size_t)rq.p * P.page_bytes;
            typename X::Acc acc[RPP][MAXB];
#pragma unroll
            for (int r = 0; r < RPP; ++r) {
#pragma unroll
                for (int b = 0; b < MAXB; ++b) acc[r][b] = 0;
                if (r < cnt) row_dot<MAXB, NCH>(page + (size_t)r * row_bytes, ct, nchunk, x, acc[r]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty()[rq.p]);
            rq.next(P.num_pages);
            float v[VP];
#pragma unroll
            for (int r = 0; r < RPP; ++r)
#pragma unroll
                for (int b = 0; b < MAXB; ++b) v[r * MAXB + b] = X::value(acc[r][b]);
            Bfly<VP, 16>::run(v, lane);
            const int base = r0 * MAXB;
            if constexpr (VP >= 32) {
#pragma unroll
                for (int j = 0; j < VP / 32; ++j) {
                    const int k = lane * (VP / 32) + j;
                    if (k / MAXB < cnt) red[base + k] = v[j];
                }
            } else {
                const int k = lane / (32 / VP);
                if ((lane & (32 / VP - 1)) == 0 && k / MAXB < cnt) red[base + k] = v[0];
            }
        }
    }
    // the 8 consumer warps meet on a hardware barrier (it orders their shared
    // writes before the epilogue's reads); warp `use % 8` runs the epilogue
    consumer_bar();
    if (warp != (int)(use % CONSUMER_WARPS)) return false;

    // epilogue (the last warp): lane handles v = lane + 32 j, i.e. row v / MAXB of sequence v % MAXB
    const float *rall = S.red(rb);
    const int out0 = F(I, P_OUT0);
    const uint64_t ptr_a = PTR(I, opc == MK_OP_QKV ? S_QKV_OUT : opc == MK_OP_O ? S_O_HRES
                                : opc == MK_OP_UP ? S_UP_OUT : opc == MK_OP_DOWN ? S_DN_HRES : S_LM_LOGITS);
    const uint64_t ptr_b = PTR(I, opc == MK_OP_O ? S_O_HMID : S_LM_KEYS);
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < VL; ++j) {
        const int v = lane + 32 * j, r = v / MAXB, b = v % MAXB;
        if (v >= VT || b >= B || r >= nrows || ab) continue;
        float y = 0.f, u = 0.f;
#pragma unroll
        for (int w = 0; w < CONSUMER_WARPS; ++w) y += rall[w * VT + v];
        if (opc == MK_OP_UP) {
#pragma unroll
            for (int w = 0; w < CONSUMER_WARPS; ++w) u += rall[w * VT + nrows * MAXB + v];
        }
        if (opc == MK_OP_QKV) {
            const int G = P.Hq / P.Hkv;
            reinterpret_cast<float *>(ptr_a)[(size_t)b * P.Hkv * (G + 2) * P.D + out0 + r] = y;
        } else if (opc == MK_OP_O) {
            const size_t k = (size_t)b * P.H + out0 + r;
            reinterpret_cast<float *>(ptr_a)[k] = resid_v[j] + y;
            reinterpret_cast<float *>(ptr_b)[k] = resid_v[j] + y;
        } else if (opc == MK_OP_UP) {
            reinterpret_cast<float *>(ptr_a)[(size_t)b * P.F + out0 + r] = y / (1.0f + __expf(-y)) * u;
        } else if (opc == MK_OP_DOWN) {
            atomicAdd(reinterpret_cast<float *>(ptr_a) + (size_t)b * P.H + out0 + r, y);
        } else if (opc == MK_OP_LM) {
            reinterpret_cast<float *>(ptr_a)[(size_t)b * P.V + out0 + r] = y;
            if (y > bv || (y == bv && r < bi)) { bv = y; bi = r; }
        }
    }
    if (opc == MK_OP_LM) {
        // argmax over the tile's rows of each sequence (lowest index on ties);
        // lanes with equal lane % MAXB hold the same sequence
#pragma unroll
        for (int o = 16; o >= MAXB; o >>= 1) {
            const float ov = __shfl_xor_sync(FULL, bv, o);
            const int oi = __shfl_xor_sync(FULL, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane < B && !ab && bi != 0x7fffffff) {
            const unsigned long long key = argmax_key(bv, out0 + bi);
            if (key > lm_best) {  // lane b keeps sequence b's best key of this step
                lm_best = key;
                red_max_u64(reinterpret_cast<unsigned long long *>(ptr_b) + (size_t)I.step * B + lane, key);
            }
        }
    }
    return true;
}

// ---------------------------------------------------------------- tensor-core tiles (batch 2-8, or batch 1 off the row-per-warp path)
// A tile of up to 16 weight rows (MLP-up: 8 gate + 8 up) for every sequence
// as m16n8k16 bf16 MMAs: the weight rows are the MMA's M side, the (up to 8)
// sequences its N side.  Warp w takes K slice [w K/8, (w + 1) K/8) in 64-wide
// chunks; lane (g, t) = (lane / 4, lane % 4) loads 16 contiguous K elements of
// weight rows g and g + 8 and of sequence g's activation at offset 16 t and
// feeds them to four k16 steps (the K order inside a chunk is permuted alike
// for both operands).  The fp32 activation is split into bf16 high and low
// parts (x = hi + lo to 2^-16 relative) and both are multiplied, so the
// products keep fp32-level accuracy.  Partials go to the same reduction
// buffer layout as the split-K path and the same epilogue runs.
DEV uint32_t bf16_pair_rn(float lo, float hi) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}
DEV void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Whether a tile off the batch-1 row-per-warp path takes the tensor-core path.
DEV bool mma_tile(const KParams &P, const WIns &I) {
    const int opc = F(I, W_OPC), kc = F(I, P_KC), rpp = F(I, P_RPP), npg = F(I, P_NPG);
    const int total = (opc == MK_OP_UP ? 2 : 1) * F(I, P_NROWS);
    return kc % (64 * CONSUMER_WARPS) == 0 && total <= 16 && npg <= 2 && rpp >= 8;
}

template <int MAXB>
DEV bool gemv_mma_tile(const KParams &P, const Smem S, const WIns &I, int i, int sl, const float *slot, uint32_t &ring,
                       RingPos &rq, uint32_t &ured, unsigned long long &lm_best, bool &ab) {
    constexpr int RT = 16;                   // rows of the MMA's M side
    constexpr int VT = RT * MAXB;            // partials per warp in a reduction buffer: row * MAXB + b
    constexpr int VL = (VT + 31) / 32;
    const int ct = threadIdx.x - CONSUMER_BASE, warp = ct >> 5, lane = ct & 31;
    const int g = lane >> 2, t = lane & 3;
    const int opc = F(I, W_OPC);
    const int kc = F(I, P_KC), nrows = F(I, P_NROWS), npg = F(I, P_NPG), rpp = F(I, P_RPP);
    const int B = P.B, NP = P.num_pages, row_bytes = 2 * kc;
    const int out0 = F(I, P_OUT0);
    const uint64_t ptr_a = PTR(I, opc == MK_OP_QKV ? S_QKV_OUT : opc == MK_OP_O ? S_O_HRES
                                : opc == MK_OP_UP ? S_UP_OUT : opc == MK_OP_DOWN ? S_DN_HRES : S_LM_LOGITS);
    const uint64_t ptr_b = PTR(I, opc == MK_OP_O ? S_O_HMID : S_LM_KEYS);
    // O tiles: the residual values of this lane's epilogue entries, read
    // before the slot is released (any warp may turn out to run the epilogue)
    float resid_v[VL];
#pragma unroll
    for (int j = 0; j < VL; ++j) resid_v[j] = 0.f;
    if (opc == MK_OP_O) {
        const float *rs = slot_resid(P, const_cast<float *>(slot));
#pragma unroll
        for (int j = 0; j < VL; ++j) {
            const int v = lane + 32 * j, r = v / MAXB, b = v % MAXB;
            if (v < VT && b < B && r < nrows) resid_v[j] = rs[b * RESID_ROWS + r];
        }
    }
    const uint32_t base = ring;
    ring += npg;
    for (int k = 0; k < npg; ++k)
        if (!ab) ab = !warp_wait_bar(P, S, &S.full()[(base + k) % NP], ((base + k) / NP) & 1, 2, i, opc);
    trace_stamp(P, i, 7);
    // rows past the tile's end read stale bytes of its own pages; their
    // results are never stored
    auto row_ptr = [&](int r) -> const uint8_t * {
        const int pg = min(r / rpp, npg - 1);
        return S.pages() + (size_t)((base + pg) % NP) * P.page_bytes + (size_t)(r % rpp) * row_bytes;
    };
    const uint8_t *w0 = row_ptr(g), *w1 = row_ptr(g + 8);
    const bool bok = g < B;
    const float *xb = S.abuf(sl) + (size_t)(bok ? g : 0) * kc;
    const int kw = kc / CONSUMER_WARPS;
    // eight independent accumulator sets (k16 step x high / low part) so that
    // the MMAs of a chunk do not wait on each other
    float acc[8][4];
#pragma unroll
    for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[q][e] = 0.f;
    for (int k0 = warp * kw; k0 < (warp + 1) * kw; k0 += 64) {
        const int off = k0 + 16 * t;
        const uint4 a00 = *reinterpret_cast<const uint4 *>(w0 + off * 2);
        const uint4 a01 = *reinterpret_cast<const uint4 *>(w0 + off * 2 + 16);
        const uint4 a10 = *reinterpret_cast<const uint4 *>(w1 + off * 2);
        const uint4 a11 = *reinterpret_cast<const uint4 *>(w1 + off * 2 + 16);
        float x[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 v = bok ? *reinterpret_cast<const float4 *>(xb + off + 4 * q) : make_float4(0.f, 0.f, 0.f, 0.f);
            x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
        }
        uint32_t bh[8], bl[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float h0 = round_bf16(x[2 * e]), h1 = round_bf16(x[2 * e + 1]);
            bh[e] = bf16_pair_rn(h0, h1);
            bl[e] = bf16_pair_rn(x[2 * e] - h0, x[2 * e + 1] - h1);
        }
        const uint32_t ag[8] = {a00.x, a00.y, a00.z, a00.w, a01.x, a01.y, a01.z, a01.w};
        const uint32_t ag8[8] = {a10.x, a10.y, a10.z, a10.w, a11.x, a11.y, a11.z, a11.w};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            mma_bf16(acc[s], ag[2 * s], ag8[2 * s], ag[2 * s + 1], ag8[2 * s + 1], bh[2 * s], bh[2 * s + 1]);
            mma_bf16(acc[4 + s], ag[2 * s], ag8[2 * s], ag[2 * s + 1], ag8[2 * s + 1], bl[2 * s], bl[2 * s + 1]);
        }
    }
    float ch[4], cl[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        ch[e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
        cl[e] = (acc[4][e] + acc[5][e]) + (acc[6][e] + acc[7][e]);
    }
    __syncwarp();
    trace_stamp(P, i, 9);
    if (lane == 0) {
        for (int k = 0; k < npg; ++k) mbar_arrive(&S.empty()[(base + k) % NP]);
        mbar_arrive(&S.act_empty()[sl]);  // activation buffer and slot no longer needed
    }
    rq.set(ring, NP);
    // the reduction buffer (see gemv_tile for why its previous user is done)
    const int rb = (int)(ured % NRED);
    const uint32_t use = ured / NRED;
    ++ured;
    float *red = S.red(rb) + warp * VT;
    if (2 * t < MAXB) {
        red[g * MAXB + 2 * t] = ch[0] + cl[0];
        red[(g + 8) * MAXB + 2 * t] = ch[2] + cl[2];
    }
    if (2 * t + 1 < MAXB) {
        red[g * MAXB + 2 * t + 1] = ch[1] + cl[1];
        red[(g + 8) * MAXB + 2 * t + 1] = ch[3] + cl[3];
    }
    consumer_bar();
    trace_stamp(P, i, 10);
    if (warp != (int)(use % CONSUMER_WARPS)) return false;
    const float *rall = S.red(rb);
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < VL; ++j) {
        const int v = lane + 32 * j, r = v / MAXB, b = v % MAXB;
        if (v >= VT || b >= B || r >= nrows || ab) continue;
        float y = 0.f, u = 0.f;
#pragma unroll
        for (int w = 0; w < CONSUMER_WARPS; ++w) y += rall[w * VT + v];
        if (opc == MK_OP_UP) {
#pragma unroll
            for (int w = 0; w < CONSUMER_WARPS; ++w) u += rall[w * VT + nrows * MAXB + v];
        }
        if (opc == MK_OP_QKV) {
            const int G = P.Hq / P.Hkv;
            reinterpret_cast<float *>(ptr_a)[(size_t)b * P.Hkv * (G + 2) * P.D + out0 + r] = y;
        } else if (opc == MK_OP_O) {
            const size_t k = (size_t)b * P.H + out0 + r;
            reinterpret_cast<float *>(ptr_a)[k] = resid_v[j] + y;
            reinterpret_cast<float *>(ptr_b)[k] = resid_v[j] + y;
        } else if (opc == MK_OP_UP) {
            reinterpret_cast<float *>(ptr_a)[(size_t)b * P.F + out0 + r] = y / (1.0f + __expf(-y)) * u;
        } else if (opc == MK_OP_DOWN) {
            atomicAdd(reinterpret_cast<float *>(ptr_a) + (size_t)b * P.H + out0 + r, y);
        } else if (opc == MK_OP_LM) {
            reinterpret_cast<float *>(ptr_a)[(size_t)b * P.V + out0 + r] = y;
            if (y > bv || (y == bv && r < bi)) { bv = y; bi = r; }
        }
    }
    if (opc == MK_OP_LM) {
#pragma unroll
        for (int o = 16; o >= MAXB; o >>= 1) {
            const float ov = __shfl_xor_sync(FULL, bv, o);
            const int oi = __shfl_xor_sync(FULL, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane < B && !ab && bi != 0x7fffffff) {
            const unsigned long long key = argmax_key(bv, out0 + bi);
            if (key > lm_best) {
                lm_best = key;
                red_max_u64(reinterpret_cast<unsigned long long *>(ptr_b) + (size_t)I.step * B + lane, key);
            }
        }
    }
    return true;
}

// ---------------------------------------------------------------- batch 1, rows per warp
// Batch-1 GEMV tiles with K a multiple of 256 up to 2048 take the
// row-per-warp path: a tile is NPG pages of 16 rows (or one page of at most
// 16), warp w computes rows w and w + 8 of every page over the whole K,
// holding x (its lane's 8-wide chunks l, l + 32, ...) in registers across
// tiles -- no cross-warp reduction and no barrier.  MLP-up pages hold 8 gate
// rows and their 8 up rows, so a gate row and its up row fall to one warp in
// one page.  Pages are taken one at a time in a loop (one copy of the code
// for any page count) and each page's rows are stored as soon as they are
// summed.
constexpr int RPW_MAX_PAGES = 64;
DEV bool rpw_tile(const KParams &P, const Dec &d) {
    if (P.B != 1 || d.opc < MK_OP_QKV || d.opc > MK_OP_LM || d.opc == MK_OP_ATTN) return false;
    if (d.kc % 256 || d.kc > 2048) return false;
    const bool up = d.opc == MK_OP_UP;
    if (d.npg == 1) return up ? d.nrows == 8 : d.nrows <= 16;
    return d.npg >= 2 && d.npg <= RPW_MAX_PAGES && d.opc != MK_OP_O && P.page_bytes == 32 * d.kc &&
           (up ? d.nrows == 8 * d.npg : d.nrows > 16 * (d.npg - 1) && d.nrows <= 16 * d.npg);
}

// The activation hand-off (activation loader stages, consumers wait) is due
// for every slot except a row-per-warp tile that repeats the previous slot's
// op, K chunk and waits: its input is the one already staged and waited for,
// and x is still in the consumers' registers.  O tiles (their residual rows)
// and snapshotting tiles always take it.  Both sides evaluate this on the same
// instruction stream, so they agree slot by slot.
struct HandoffChain {
    int prev = 0;  // this lane's word of the previous slot
    bool valid = false;
};
template <int FL>
DEV bool needs_handoff(const KParams &P, const WIns &I, const Dec &d, HandoffChain &c) {
    const int lane = threadIdx.x & 31;
    // (the FP8 instance: its e4m3 tiles hold x in registers the same way)
    const bool rpw = (FL == FL_W8 && F(I, P_W8) != 0) || rpw_tile(P, d);
    const bool input_word = lane == W_OPC || lane == W_ROW || lane == W_CNT ||
                            (lane >= W_WAIT && lane < W_SIG) || lane == P_K0 || lane == P_KC;
    const bool same = c.valid && !__any_sync(FULL, input_word && I.w != c.prev);
    const bool skip = rpw && same && d.opc != MK_OP_O && d.snap == 0;
    c.prev = I.w;
    c.valid = rpw;
    return !skip;
}

// x of a consumer lane for the row-per-warp path: chunk k covers columns
// (lane + 32 k) * 8 .. + 8, as fp32 pairs.
struct XRow {
    uint64_t v[8][4];
    long long key = -1;  // op row << 32 | first column of what v holds
};

template <int KG>
DEV void rpw_row(const uint8_t *wrow, int lane, const XRow &x, uint64_t &acc) {
#pragma unroll
    for (int k = 0; k < KG; ++k) {
        const uint4 w = *reinterpret_cast<const uint4 *>(wrow + (lane + 32 * k) * 16);
        fma2(acc, bf16x2_pair(w.x), x.v[k][0]);
        fma2(acc, bf16x2_pair(w.y), x.v[k][1]);
        fma2(acc, bf16x2_pair(w.z), x.v[k][2]);
        fma2(acc, bf16x2_pair(w.w), x.v[k][3]);
    }
}

// Epilogue of the row-per-warp tiles: V row sums per warp (rows w + 8 v),
// reduced across the warp, then stored by op: QKV rows, O rows plus their
// residual (both residual copies), SiLU(gate) x up for MLP-up (the up row of
// gate row r is r + nrows), atomic adds for MLP-down K chunks, logits and the
// running argmax for the LM head.
template <int V>
DEV bool rpw_finish(const KParams &P, const Dec &d, const uint64_t (&acc)[V], const float (&res)[V],
                    unsigned long long &lm_best, bool ab) {
    const int ct = threadIdx.x - CONSUMER_BASE, warp = ct >> 5, lane = ct & 31;
    const int opc = d.opc, nrows = d.nrows, out0 = d.out0;
    const uint64_t ptr_a = d.out, ptr_b = d.out2;
    // after the butterfly, lanes L with L % (32 / V) == 0 hold row w + 8 (L / (32 / V))
    float y[V];
#pragma unroll
    for (int v = 0; v < V; ++v) y[v] = sum2(acc[v]);
    Bfly<V, 16>::run(y, lane);
    constexpr int LPV = 32 / V;
    const int v = lane / LPV, r = warp + 8 * v;
    const bool holder = (lane % LPV) == 0;
    float val = y[0];
    if (opc == MK_OP_UP) {
        // the up row of gate row r is r + nrows: value index v + nrows / 8
        const float u = __shfl_sync(FULL, val, min(31, (v + nrows / 8) * LPV));
        if (holder && !ab && r < nrows) reinterpret_cast<float *>(ptr_a)[out0 + r] = val / (1.0f + __expf(-val)) * u;
        return true;
    }
    float resid = 0.f;
#pragma unroll
    for (int k = 0; k < V; ++k)
        if (k == v) resid = res[k];
    const bool mine = holder && !ab && r < nrows;
    if (opc == MK_OP_QKV) {
        if (mine) reinterpret_cast<float *>(ptr_a)[out0 + r] = val;
    } else if (opc == MK_OP_O) {
        if (mine) {
            reinterpret_cast<float *>(ptr_a)[out0 + r] = resid + val;
            reinterpret_cast<float *>(ptr_b)[out0 + r] = resid + val;
        }
    } else if (opc == MK_OP_DOWN) {
        if (mine) atomicAdd(reinterpret_cast<float *>(ptr_a) + out0 + r, val);
    } else if (opc == MK_OP_LM) {
        if (mine) reinterpret_cast<float *>(ptr_a)[out0 + r] = val;
        // this warp's best row of the tile (lowest index on ties), then the
        // step's running best per warp
        unsigned long long key = mine ? argmax_key(val, out0 + r) : 0ull;
#pragma unroll
        for (int o = 16; o; o >>= 1) key = max(key, __shfl_xor_sync(FULL, key, o));
        if (lane == 0 && key > lm_best && !ab) {
            lm_best = key;
            red_max_u64(reinterpret_cast<unsigned long long *>(ptr_b) + (size_t)d.step, key);
        }
    }
    return true;
}

// KG = K / 256 chunks per lane.  `handoff`: this slot took the activation
// hand-off (the caller waited for activation slot sl); x is reloaded from the
// slot's buffer when its input changed.  Each page: rows w and w + 8 of this
// warp, one butterfly for both (lanes 0 and 16 then hold the two row sums),
// the stores of the op.  Returns true (the warp wrote global memory).
template <int KG>
DEV bool gemv_rpw(const KParams &P, const Smem S, const Dec &d, int i, bool handoff, int sl, const float *slot,
                  XRow &x, uint32_t &ring, RingPos &rq, unsigned long long &lm_best, bool &ab) {
    const int ct = threadIdx.x - CONSUMER_BASE, warp = ct >> 5, lane = ct & 31;
    const int opc = d.opc, row_bytes = d.kc * 2, npg = d.npg, nrows = d.nrows, out0 = d.out0;
    float resid = 0.f;  // O tiles (one page): the residual of this lane's row, w (lane 0) or w + 8 (lane 16)
    if (handoff) {
        const long long key = ((long long)d.row << 32) | (uint32_t)d.k0;
        if (key != x.key) {
            const float4 *xs = reinterpret_cast<const float4 *>(S.abuf(sl));  // lane-interleaved (rpw_perm4)
#pragma unroll
            for (int k = 0; k < KG; ++k) {
                const float4 a = xs[(2 * k) * 32 + lane];
                const float4 c = xs[(2 * k + 1) * 32 + lane];
                x.v[k][0] = pack2(a.x, a.y); x.v[k][1] = pack2(a.z, a.w);
                x.v[k][2] = pack2(c.x, c.y); x.v[k][3] = pack2(c.z, c.w);
            }
            x.key = key;
        }
        if (opc == MK_OP_O) {  // O tiles have at most RESID_ROWS rows
            const int r = warp + (lane >> 4) * 8;
            if (r < RESID_ROWS) resid = slot_resid(P, const_cast<float *>(slot))[r];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.act_empty()[sl]);  // x and the residual rows are in registers
    }
    trace_stamp(P, i, 6);
    float* const out = reinterpret_cast<float *>(d.out);
    float bv = -INFINITY;  // LM head: this lane's best logit of the tile and its row
    int bi = 0;
    for (int pg = 0; pg < npg; ++pg) {
        if (!ab) ab = !warp_wait_bar(P, S, &S.full()[rq.p], rq.ph, 2, i, opc);
        if (pg == 0) trace_stamp(P, i, 7);
        const uint8_t *page = S.pages() + (size_t)rq.p * P.page_bytes;
        uint64_t acc[2] = {0, 0};
        rpw_row<KG>(page + (size_t)warp * row_bytes, lane, x, acc[0]);
        rpw_row<KG>(page + (size_t)(warp + 8) * row_bytes, lane, x, acc[1]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty()[rq.p]);
        rq.next(P.num_pages);
        float y[2] = {sum2(acc[0]), sum2(acc[1])};
        Bfly<2, 16>::run(y, lane);  // lanes 0-15: row w of the page, lanes 16-31: row w + 8
        const float val = y[0];
        if (opc == MK_OP_UP) {
            // gate row 8 pg + w (page slot w) and its up row (slot w + 8)
            const float u = __shfl_sync(FULL, val, 16);
            const int r = 8 * pg + warp;
            if (lane == 0 && !ab && r < nrows) out[out0 + r] = val / (1.0f + __expf(-val)) * u;
            continue;
        }
        const int r = 16 * pg + warp + (lane >> 4) * 8;
        const bool mine = (lane & 15) == 0 && !ab && r < nrows;
        if (opc == MK_OP_QKV) {
            if (mine) out[out0 + r] = val;
        } else if (opc == MK_OP_O) {
            if (mine) {
                out[out0 + r] = resid + val;
                reinterpret_cast<float *>(d.out2)[out0 + r] = resid + val;
            }
        } else if (opc == MK_OP_DOWN) {
            if (mine) atomicAdd(out + out0 + r, val);
        } else {  // LM head
            if (mine) {
                out[out0 + r] = val;
                if (val > bv) { bv = val; bi = r; }  // rows rise with pg: the lowest index wins ties
            }
        }
    }
    ring += npg;
    trace_stamp(P, i, 8);
    if (opc == MK_OP_LM) {
        // this warp's best row of the tile (lowest index on ties), then the
        // step's running best per warp
        unsigned long long key = bv > -INFINITY ? argmax_key(bv, out0 + bi) : 0ull;
#pragma unroll
        for (int o = 16; o; o >>= 1) key = max(key, __shfl_xor_sync(FULL, key, o));
        if (lane == 0 && key > lm_best && !ab) {
            lm_best = key;
            red_max_u64(reinterpret_cast<unsigned long long *>(d.out2) + (size_t)d.step, key);
        }
    }
    trace_stamp(P, i, 9);
    return true;
}

// ---------------------------------------------------------------- batch 1, FP8 rows per warp
// FP8 projections (e4m3 rows of K = 2048, one fp32 scale per 128 x 128
// block): pages of 32 rows (MLP-up: 16 gate rows, then their 16 up rows),
// warp w takes rows w, w + 8, w + 16, w + 24 of every page over the whole K.
// Lane l holds x's 16-wide chunks c = l + 32 k (k < 4; x staged in that
// order, rpw_perm8) in registers, and the scale of each chunk's 128-column
// block -- a tile's rows lie in one 128-row block, so four scales per matrix
// and lane serve the whole tile.  Each chunk: 16 codes to fp32 pairs
// (cvt.rn.f16x2.e4m3x2, exact), 8 packed multiply-adds into a partial, the
// partial times its block scale into the row sum.
DEV uint64_t e4m3x2_pair(uint32_t v) {  // codes in the low 16 bits, the first in the low byte
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)(v & 0xffffu)));
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    return pack2(f.x, f.y);
}
DEV void rpw8_row(const uint8_t *wrow, int lane, const XRow &x, const float (&sc)[4], uint64_t &acc) {
#pragma unroll
    for (int k = 0; k < W8_K / 512; ++k) {
        const uint4 w = *reinterpret_cast<const uint4 *>(wrow + (lane + 32 * k) * 16);
        uint64_t part = 0;
        fma2(part, e4m3x2_pair(w.x), x.v[2 * k][0]);
        fma2(part, e4m3x2_pair(w.x >> 16), x.v[2 * k][1]);
        fma2(part, e4m3x2_pair(w.y), x.v[2 * k][2]);
        fma2(part, e4m3x2_pair(w.y >> 16), x.v[2 * k][3]);
        fma2(part, e4m3x2_pair(w.z), x.v[2 * k + 1][0]);
        fma2(part, e4m3x2_pair(w.z >> 16), x.v[2 * k + 1][1]);
        fma2(part, e4m3x2_pair(w.w), x.v[2 * k + 1][2]);
        fma2(part, e4m3x2_pair(w.w >> 16), x.v[2 * k + 1][3]);
        fma2(acc, part, pack2(sc[k], sc[k]));
    }
}
// This lane's four chunk scales of a matrix for the tile (row block row0 / 128).
DEV void rpw8_scales(const float *s, int row0, int k0, int ktot, int lane, float (&sc)[4]) {
    const float *srow = s + (size_t)(row0 / 128) * (ktot / 128) + k0 / 128;
#pragma unroll
    for (int k = 0; k < 4; ++k) sc[k] = __ldg(srow + (lane + 32 * k) / 8);
}

DEV bool gemv_rpw8(const KParams &P, const Smem S, const WIns &I, const Dec &d, int i, bool handoff, int sl,
                   const float *slot, XRow &x, uint32_t &ring, RingPos &rq, bool &ab) {
    const int ct = threadIdx.x - CONSUMER_BASE, warp = ct >> 5, lane = ct & 31;
    const int opc = d.opc, npg = d.npg, nrows = d.nrows, out0 = d.out0;
    const bool up = opc == MK_OP_UP;
    // block scales: the tile's matrix (QKV: its q, k or v matrix; MLP-up: gate, then up)
    const int row0 = F(I, P_ROW0), ktot = F(I, P_KTOT), mat = opc == MK_OP_QKV ? F(I, P_MAT) : 0;
    const float *s0 = reinterpret_cast<const float *>(PTR(I, S_W8_S0 + mat));
    const float *s1 = reinterpret_cast<const float *>(PTR(I, S_W8_S1));
    float sa[4], sb[4];
    rpw8_scales(s0, row0, d.k0, ktot, lane, sa);
    if (up) rpw8_scales(s1, row0, d.k0, ktot, lane, sb);
    float resid = 0.f;  // O tiles (one page): the residual of this lane's row w + 8 (lane / 8)
    if (handoff) {
        const long long key = ((long long)d.row << 32) | (uint32_t)d.k0 | (1ll << 61);  // (FP8 layout)
        if (key != x.key) {
            const float4 *xs = reinterpret_cast<const float4 *>(S.abuf(sl));  // lane-interleaved (rpw_perm8)
#pragma unroll
            for (int k = 0; k < W8_K / 512; ++k)
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float4 a = xs[(4 * k + h) * 32 + lane];
                    x.v[2 * k + (h >> 1)][(h & 1) * 2] = pack2(a.x, a.y);
                    x.v[2 * k + (h >> 1)][(h & 1) * 2 + 1] = pack2(a.z, a.w);
                }
            x.key = key;
        }
        if (opc == MK_OP_O) {
            const int r = warp + 8 * (lane >> 3);
            if (r < RESID_ROWS) resid = slot_resid(P, const_cast<float *>(slot))[r];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.act_empty()[sl]);  // x and the residual rows are in registers
    }
    trace_stamp(P, i, 6);
    float *const out = reinterpret_cast<float *>(d.out);
    for (int pg = 0; pg < npg; ++pg) {
        if (!ab) ab = !warp_wait_bar(P, S, &S.full()[rq.p], rq.ph, 2, i, opc);
        if (pg == 0) trace_stamp(P, i, 7);
        const uint8_t *page = S.pages() + (size_t)rq.p * P.page_bytes;
        uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 4; ++j)  // MLP-up: rows 0..15 gate (j 0, 1), 16..31 up (j 2, 3)
            rpw8_row(page + (size_t)(warp + 8 * j) * W8_K, lane, x, up && j >= 2 ? sb : sa, acc[j]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty()[rq.p]);
        rq.next(P.num_pages);
        float y[4] = {sum2(acc[0]), sum2(acc[1]), sum2(acc[2]), sum2(acc[3])};
        Bfly<4, 16>::run(y, lane);  // lanes 8 j .. 8 j + 7: row w + 8 j of the page
        const float val = y[0];
        const int j = lane >> 3;
        const bool holder = (lane & 7) == 0;
        if (up) {
            // gate row 16 pg + w + 8 j (j 0, 1) and its up row (page row 16 + w + 8 j: lane 8 j + 16)
            const float u = __shfl_sync(FULL, val, (lane + 16) & 31);
            const int r = 16 * pg + warp + 8 * j;
            if (holder && j < 2 && !ab && r < nrows) out[out0 + r] = val / (1.0f + __expf(-val)) * u;
            continue;
        }
        const int r = W8_ROWS * pg + warp + 8 * j;
        const bool mine = holder && !ab && r < nrows;
        if (opc == MK_OP_QKV) {
            if (mine) out[out0 + r] = val;
        } else if (opc == MK_OP_O) {
            if (mine) {
                out[out0 + r] = resid + val;
                reinterpret_cast<float *>(d.out2)[out0 + r] = resid + val;
            }
        } else {  // MLP-down K chunk
            if (mine) atomicAdd(out + out0 + r, val);
        }
    }
    ring += npg;
    trace_stamp(P, i, 9);
    return true;
}

// Batch-1 tiles whose K (4096) is too long for x in registers, in pages of 8
// rows: warp w computes row w of every page over the whole K, reading its
// lane's 8-wide chunks of x (l, l + 32, ...) from the activation slot in
// shared memory once for all pages of the tile (it waits for both pages
// first; the ring holds three).  The slot is released after the last page, so
// these tiles always take the hand-off.  MLP-up tiles are 8 gate rows (page 0)
// and their 8 up rows (page 1).
constexpr int RPW_WIDE_K = 4096;
DEV bool rpw_wide_tile(const KParams &P, const Dec &d) {
    if (P.B != 1 || d.opc < MK_OP_QKV || d.opc > MK_OP_LM || d.opc == MK_OP_ATTN) return false;
    if (d.kc != RPW_WIDE_K || P.page_bytes != 16 * d.kc || P.num_pages < 2) return false;
    if (d.opc == MK_OP_UP) return d.npg == 2 && d.nrows == 8;
    return d.npg == 1 ? d.nrows <= 8 : d.npg == 2 && d.nrows <= 16;
}

template <int NPG>
DEV bool gemv_rpw_wide(const KParams &P, const Smem S, const Dec &d, int i, int sl, const float *slot,
                       uint32_t &ring, RingPos &rq, unsigned long long &lm_best, bool &ab) {
    constexpr int KG = RPW_WIDE_K / 256;
    const int ct = threadIdx.x - CONSUMER_BASE, warp = ct >> 5, lane = ct & 31;
    const int opc = d.opc, row_bytes = d.kc * 2;
    float res[NPG];
#pragma unroll
    for (int v = 0; v < NPG; ++v) res[v] = 0.f;
    if (opc == MK_OP_O) {
        const float *rs = slot_resid(P, const_cast<float *>(slot));
#pragma unroll
        for (int v = 0; v < NPG; ++v)
            if (warp + 8 * v < RESID_ROWS) res[v] = rs[warp + 8 * v];
    }
    const uint8_t *wrow[NPG];
    int pid[NPG];
#pragma unroll
    for (int pg = 0; pg < NPG; ++pg) {
        if (!ab) ab = !warp_wait_bar(P, S, &S.full()[rq.p], rq.ph, 2, i, opc);
        pid[pg] = rq.p;
        wrow[pg] = S.pages() + (size_t)rq.p * P.page_bytes + (size_t)warp * row_bytes;
        rq.next(P.num_pages);
    }
    const float4 *xs = reinterpret_cast<const float4 *>(S.abuf(sl));  // lane-interleaved (rpw_perm4)
    uint64_t a0[NPG], a1[NPG];
#pragma unroll
    for (int pg = 0; pg < NPG; ++pg) a0[pg] = a1[pg] = 0;
#pragma unroll
    for (int k = 0; k < KG; ++k) {
        const float4 xa = xs[(2 * k) * 32 + lane];
        const float4 xb = xs[(2 * k + 1) * 32 + lane];
        const uint64_t x0 = pack2(xa.x, xa.y), x1 = pack2(xa.z, xa.w), x2 = pack2(xb.x, xb.y), x3 = pack2(xb.z, xb.w);
#pragma unroll
        for (int pg = 0; pg < NPG; ++pg) {
            const uint4 w = *reinterpret_cast<const uint4 *>(wrow[pg] + (lane + 32 * k) * 16);
            fma2(a0[pg], bf16x2_pair(w.x), x0);
            fma2(a1[pg], bf16x2_pair(w.y), x1);
            fma2(a0[pg], bf16x2_pair(w.z), x2);
            fma2(a1[pg], bf16x2_pair(w.w), x3);
        }
    }
    __syncwarp();
    if (lane == 0) {
#pragma unroll
        for (int pg = 0; pg < NPG; ++pg) mbar_arrive(&S.empty()[pid[pg]]);
        mbar_arrive(&S.act_empty()[sl]);  // x and the residual rows are no longer read
    }
    ring += NPG;
    uint64_t acc[NPG];
#pragma unroll
    for (int pg = 0; pg < NPG; ++pg) acc[pg] = pack2(sum2(a0[pg]), sum2(a1[pg]));
    return rpw_finish<NPG>(P, d, acc, res, lm_best, ab);
}

// Split-KV attention of one (sequence, kv group, split).  Each of the 8
// consumer warps is an independent piece of the split: query head w / parts
// of the group over token part w % parts of the split's tokens (parts = 8 /
// group size).  A warp computes its scores (4 lanes per token, log2 units),
// the softmax statistics (max, sum of 2^(s - max)) and P.V for its head,
// writes that partial, and arrives on its head's counter; the warp that
// arrives last for a head merges all of the head's partials (log-sum-exp
// combine).  No barrier inside the task.
// Releases page p after the 8 consumer warps read it.  The tensor-core
// instance's page barriers take one arrival (the MMA commit of a weight
// stage), so there the last of the 8 warps arrives (a shared counter per page).
template <int FL>
DEV void page_release(const Smem S, int p) {
    if constexpr (FL == FL_TC) {
        if (atomicAdd(&S.page_users()[p], 1) == CONSUMER_WARPS - 1) {
            S.page_users()[p] = 0;
            mbar_arrive(&S.empty()[p]);
        }
    } else {
        mbar_arrive(&S.empty()[p]);
    }
}

// Attention, one warp per (q head, token part): head_dim 64, where the
// per-instruction latency matters more than the instruction count.
template <int D, int FL>
DEV void attn_task_heads(const KParams &P, const Smem S, const WIns &I, int i, int sl, const float *slot, uint32_t &ring,
                   bool &ab) {
    constexpr int PER = D / 32;
    constexpr int QS = D / 4 + 4;
    constexpr int DQ = D / 4;
    const int ct = threadIdx.x - CONSUMER_BASE, warp = ct >> 5, lane = ct & 31;
    const int G = P.Hq / P.Hkv, parts = CONSUMER_WARPS / G;
    const int hh = warp / parts, part = warp % parts;  // head within the kv group, token part
    const int b = F(I, P_B), g = F(I, P_G);
    const int split = F(I, P_SPLIT), nsplit = F(I, P_NSPLIT), layer = F(I, P_LAYER);
    const int pos = attn_pos(P, I);
    const int t0 = F(I, P_T0), T = F(I, P_T);
    const int ncache = attn_cached_rows(I, pos);
    const bool has_new = pos >= t0 && pos < t0 + T;
    const int ntot = ncache + (has_new ? 1 : 0);
    const int tp = (T + parts - 1) / parts;
    const int tb = part * tp, te = min(ntot, tb + tp);  // this warp's tokens [tb, te) of the split
    const float *qp = slot, *kn = slot + G * 4 * QS, *vn = kn + D;
    float *sw = S.aux() + warp * tp;  // this warp's scores, then probabilities
    float *part_base = reinterpret_cast<float *>(PTR(I, S_AT_PART));
    float *out = reinterpret_cast<float *>(PTR(I, S_AT_OUT));
    uint32_t *arrive = reinterpret_cast<uint32_t *>(PTR(I, S_AT_ARRIVE));
    const int rpp = P.page_bytes / (D * 2);
    const int npg = attn_pages(T, D, P.page_bytes);  // K pages, then as many V pages
    const uint32_t kring = ring, vring = ring + npg;
    ring = vring + npg;
    // the split's K (V) rows are consecutive rows of its K (V) page(s), rpp
    // (a power of two) to a page; a split spans at most 4 pages of each
    auto page_ptr = [&](uint32_t r) { return S.pages() + (size_t)(r % P.num_pages) * P.page_bytes; };
    const uint8_t *kpage = page_ptr(kring), *vpage = page_ptr(vring);
    const uint8_t *kp1 = page_ptr(kring + 1), *kp2 = page_ptr(kring + 2), *kp3 = page_ptr(kring + 3);
    const uint8_t *vp1 = page_ptr(vring + 1), *vp2 = page_ptr(vring + 2), *vp3 = page_ptr(vring + 3);
    const int rsh = 31 - __clz(rpp);
    auto row_at = [&](bool v, int tk) -> const uint8_t * {
        const int j = tk >> rsh;
        const uint8_t *pg = j == 0 ? (v ? vpage : kpage) : j == 1 ? (v ? vp1 : kp1) : j == 2 ? (v ? vp2 : kp2)
                                                                                        : (v ? vp3 : kp3);
        return pg + (size_t)(tk & (rpp - 1)) * (D * 2);
    };
    for (int k = 0; k < npg; ++k)
        if (!ab) ab = !warp_wait_bar(P, S, &S.full()[(kring + k) % P.num_pages], ((kring + k) / P.num_pages) & 1, 2, i, MK_OP_ATTN);
    trace_stamp(P, i, 6);
    // scores: 8 tokens per round, 4 lanes per token, DQ dims per lane in NC
    // chunks of 8.  Rows are a multiple of 128 bytes apart, so every row
    // starts on bank 0: each lane walks its chunks in a rotated order (by its
    // quarter when D = 128, and by the token's parity) so that the 8 lanes of
    // a quarter-warp phase read 8 different 16-byte bank groups.
    constexpr int NC = DQ / 8;
    const int qtr = lane & 3;
    const int rot = ((NC == 4 ? qtr : 0) + ((lane >> 2) & 1)) % NC;
    uint64_t q2[DQ / 2];  // q as fp32 pairs for packed multiply-adds
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const float *qs = qp + (hh * 4 + qtr) * QS + ((c + rot) % NC) * 8;
        const float4 v0 = *reinterpret_cast<const float4 *>(qs), v1 = *reinterpret_cast<const float4 *>(qs + 4);
        q2[c * 4] = pack2(v0.x, v0.y);
        q2[c * 4 + 1] = pack2(v0.z, v0.w);
        q2[c * 4 + 2] = pack2(v1.x, v1.y);
        q2[c * 4 + 3] = pack2(v1.z, v1.w);
    }
    const int tc = min(te, ncache);  // cached tokens of this warp: [tb, tc); the new token, if ours, is ncache
    float m = -INFINITY;
    for (int t = tb; t < te; t += 8) {
        const int tk = t + (lane >> 2);
        float s0 = 0.f, s1 = 0.f;
        if (tk < tc) {
            const uint8_t *row = row_at(false, tk) + qtr * DQ * 2;
            uint4 kw[DQ / 8];
#pragma unroll
            for (int d = 0; d < DQ / 8; ++d) kw[d] = *reinterpret_cast<const uint4 *>(row + ((d + rot) % NC) * 16);
            uint64_t sa = 0, sb = 0;
#pragma unroll
            for (int d = 0; d < DQ / 8; ++d) {
                fma2(sa, bf16x2_pair(kw[d].x), q2[d * 4]);
                fma2(sb, bf16x2_pair(kw[d].y), q2[d * 4 + 1]);
                fma2(sa, bf16x2_pair(kw[d].z), q2[d * 4 + 2]);
                fma2(sb, bf16x2_pair(kw[d].w), q2[d * 4 + 3]);
            }
            s0 = sum2(sa);
            s1 = sum2(sb);
        } else if (tk < te) {
#pragma unroll
            for (int d = 0; d < DQ; d += 2) {
                const float *kk = kn + qtr * DQ + (((d >> 3) + rot) % NC) * 8 + (d & 7);
                s0 = fmaf(__uint_as_float((uint32_t)q2[d / 2]), kk[0], s0);
                s1 = fmaf(__uint_as_float((uint32_t)(q2[d / 2] >> 32)), kk[1], s1);
            }
        }
        float s = s0 + s1;
        s += __shfl_xor_sync(FULL, s, 1);
        s += __shfl_xor_sync(FULL, s, 2);
        if (tk < te) {
            if (qtr == 0) sw[tk - tb] = s;
            m = fmaxf(m, s);
        }
    }
    m = warp_max(m);
    trace_stamp(P, i, 7);
    __syncwarp();
    if (lane == 0)
        for (int k = 0; k < npg; ++k) page_release<FL>(S, (kring + k) % P.num_pages);
    float l = 0.f;
    for (int t = tb + lane; t < te; t += 32) {
        const float e = exp2f(sw[t - tb] - m);
        sw[t - tb] = e;
        l += e;
    }
    l = warp_sum(l);
    __syncwarp();
    // P.V: lane owns dims lane * PER .. + PER; four accumulator sets so that
    // consecutive tokens' loads and multiply-adds overlap
    for (int k = 0; k < npg; ++k)
        if (!ab) ab = !warp_wait_bar(P, S, &S.full()[(vring + k) % P.num_pages], ((vring + k) / P.num_pages) & 1, 2, i, MK_OP_ATTN);
    trace_stamp(P, i, 8);
    // P.V: lane (token lane tg, dim group dg) sums 8 dims (one 16-byte load
    // of a V row) over tokens tb + tg, tb + tg + TG, ... with packed fp32
    // multiply-adds, two tokens in flight; the TG token lanes are then summed
    // with shuffles.  A warp instruction reads TG whole rows (conflict-free).
    constexpr int NG = D / 8, TG = 32 / NG;
    const int dg = lane % NG, tg = lane / NG;
    uint64_t a0[4] = {0, 0, 0, 0}, a1[4] = {0, 0, 0, 0};
    auto pv8 = [&](uint64_t (&a)[4], float p, const uint8_t *row) {
        const uint4 u = *reinterpret_cast<const uint4 *>(row + dg * 16);
        const uint64_t pp = pack2(p, p);
        fma2(a[0], bf16x2_pair(u.x), pp);
        fma2(a[1], bf16x2_pair(u.y), pp);
        fma2(a[2], bf16x2_pair(u.z), pp);
        fma2(a[3], bf16x2_pair(u.w), pp);
    };
    int t = tb + tg;
    if (npg == 1) {
        for (; t + TG < tc; t += 2 * TG) {
            pv8(a0, sw[t - tb], vpage + (size_t)t * (D * 2));
            pv8(a1, sw[t + TG - tb], vpage + (size_t)(t + TG) * (D * 2));
        }
    } else {
        for (; t + TG < tc; t += 2 * TG) {
            pv8(a0, sw[t - tb], row_at(true, t));
            pv8(a1, sw[t + TG - tb], row_at(true, t + TG));
        }
    }
    if (t < tc) pv8(a0, sw[t - tb], row_at(true, t));
    float o8[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        o8[2 * j] = __uint_as_float((uint32_t)a0[j]) + __uint_as_float((uint32_t)a1[j]);
        o8[2 * j + 1] = __uint_as_float((uint32_t)(a0[j] >> 32)) + __uint_as_float((uint32_t)(a1[j] >> 32));
    }
#pragma unroll
    for (int sft = NG; sft < 32; sft <<= 1)
#pragma unroll
        for (int j = 0; j < 8; ++j) o8[j] += __shfl_xor_sync(FULL, o8[j], sft);
    if (has_new && ncache >= tb && ncache < te) {  // the new token is this warp's
        const float p = sw[ncache - tb];
#pragma unroll
        for (int j = 0; j < 8; ++j) o8[j] = fmaf(p, vn[dg * 8 + j], o8[j]);
    }
    // every lane of a dim group holds its 8 sums: token lane tg keeps the
    // 8 / TG of them it stores (dims dg * 8 + tg * PER ..)
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        float v = o8[e];
#pragma unroll
        for (int k = 1; k < TG; ++k) v = tg == k ? o8[k * PER + e] : v;
        acc[e] = v;
    }
    __syncwarp();
    if (lane == 0) {
        for (int k = 0; k < npg; ++k) page_release<FL>(S, (vring + k) % P.num_pages);
        mbar_arrive(&S.act_empty()[sl]);  // q, k, v of the slot no longer needed by this warp
    }
    trace_stamp(P, i, 9);
    // this warp's partial: (o[D], max, sum) of head (b, g * G + hh), piece split * parts + part
    const int head = g * G + hh, npieces = P.nsplit_max * parts;
    float *pp = part_base + ((size_t)(b * P.Hq + head) * npieces + split * parts + part) * (D + 2);
    if (!ab) {
#pragma unroll
        for (int e = 0; e < PER; ++e) pp[dg * 8 + tg * PER + e] = acc[e];
        if (lane == 0) {
            pp[D] = m;
            pp[D + 1] = l;
        }
    }
    // the acq_rel add is cumulative over this warp's partial (ordered by the
    // warp barrier) and acquires the other pieces' partials
    __syncwarp();
    int last = 0;
    if (lane == 0 && !ab) {
        const uint32_t old = atom_acqrel_add(arrive + ((size_t)layer * P.B + b) * P.Hq + head, 1u);
        last = old == (uint32_t)(I.step + 1) * (uint32_t)(nsplit * parts) - 1u;
    }
    trace_stamp(P, i, 10);
    if (!__shfl_sync(FULL, last, 0)) return;
    __syncwarp();
    // merge: log-sum-exp over the head's pieces, MB at a time so that their
    // L2 round trips overlap
    const float *hb = part_base + (size_t)(b * P.Hq + head) * npieces * (D + 2);
    const int n = nsplit * parts;
    float M = -INFINITY, L = 0.f, o[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = 0.f;
    constexpr int MB = PER <= 2 ? 16 : 8;
    for (int s0 = 0; s0 < n; s0 += MB) {
        float mv[MB], lv[MB], ov[MB][PER];
#pragma unroll
        for (int u = 0; u < MB; ++u) {
            const int sp = s0 + u;
            if (sp < n) {
                const float *ps = hb + (size_t)sp * (D + 2);
                mv[u] = __ldcg(ps + D);
                lv[u] = __ldcg(ps + D + 1);
#pragma unroll
                for (int e = 0; e < PER; ++e) ov[u][e] = __ldcg(ps + lane * PER + e);
            } else {
                mv[u] = -INFINITY;
                lv[u] = 0.f;
#pragma unroll
                for (int e = 0; e < PER; ++e) ov[u][e] = 0.f;
            }
        }
        float Mn = M;
#pragma unroll
        for (int u = 0; u < MB; ++u) Mn = fmaxf(Mn, mv[u]);
        if (Mn == -INFINITY) continue;  // nothing yet
        const float r = exp2f(M - Mn);  // rescale what was accumulated so far
        L *= r;
#pragma unroll
        for (int e = 0; e < PER; ++e) o[e] *= r;
#pragma unroll
        for (int u = 0; u < MB; ++u) {
            const float f = exp2f(mv[u] - Mn);  // 0 for empty pieces
            L += f * lv[u];
#pragma unroll
            for (int e = 0; e < PER; ++e) o[e] += f * ov[u][e];
        }
        M = Mn;
    }
    if constexpr (FL == FL_TC) {
        // the O tiles' input: bf16 high and low rows b and np + b of [2 np, Hq D]
        uint16_t *o16 = reinterpret_cast<uint16_t *>(out);
        const size_t ld = (size_t)P.Hq * D;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const float v = o[e] / L;
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
            o16[(size_t)b * ld + (size_t)head * D + lane * PER + e] = __bfloat16_as_ushort(hi);
            o16[(size_t)(P.np + b) * ld + (size_t)head * D + lane * PER + e] = __bfloat16_as_ushort(lo);
        }
    } else {
#pragma unroll
        for (int e = 0; e < PER; ++e) out[((size_t)b * P.Hq + head) * D + lane * PER + e] = o[e] / L;
    }
}

// Attention of one (sequence, kv head, split of positions).  Each warp takes
// every q head of its kv group (up to 4; with 8 heads per kv head, two groups
// of 4 warps) over its share of the split's tokens, so each K / V row is read
// and converted once per warp, not once per head:
//   scores   8 lanes per token, D / 8 dims per lane, the 4 heads' sums
//            reduce-scattered over the 8 lanes (one head's score per lane);
//   P.V      lane (token lane, group of 8 dims), one 16-byte V load per token
//            for the 4 heads, then reduce-scattered over the token lanes;
//   combine  the warps' pieces (o, max, sum) meet in the split's first V page
//            (after a barrier, so no warp still reads V) and warp h merges head
//            h's pieces into the split's partial; the last split to arrive for
//            a head merges the head's partials (log-sum-exp).
template <int D, int FL>
DEV void attn_task_group(const KParams &P, const Smem S, const WIns &I, int i, int sl, const float *slot, uint32_t &ring,
                   uint32_t &cph, bool &ab) {
    constexpr int PER = D / 32;              // dims per lane in the merges
    constexpr int QS = D / 4 + 4;            // staged q: [head][quarter][QS]
    constexpr int NCH = D / 64;              // 16-byte K chunks per lane and token in the scores
    constexpr int NG = D / 8, TG = 32 / NG;  // P.V: groups of 8 dims, token lanes
    const int ct = threadIdx.x - CONSUMER_BASE, warp = ct >> 5, lane = ct & 31;
    const int G = P.Hq / P.Hkv;
    const int hpw = G < 4 ? G : 4, tw = G <= 4 ? CONSUMER_WARPS : CONSUMER_WARPS / 2;
    const int wh = warp / tw, wt = warp % tw;  // head group (heads wh * hpw ..), token part
    const int b = F(I, P_B), g = F(I, P_G);
    const int split = F(I, P_SPLIT), nsplit = F(I, P_NSPLIT), layer = F(I, P_LAYER);
    const int pos = attn_pos(P, I);
    const int t0 = F(I, P_T0), T = F(I, P_T);
    const int ncache = attn_cached_rows(I, pos);
    const bool has_new = pos >= t0 && pos < t0 + T;
    const int ntot = ncache + (has_new ? 1 : 0);
    const int tp = (T + tw - 1) / tw;
    const int tb = wt * tp, te = min(ntot, tb + tp);  // this warp's tokens [tb, te) of the split
    const int tc = min(te, ncache);                    // cached ones [tb, tc); the new token, if ours, is ncache
    const float *qp = slot, *kn = slot + G * 4 * QS, *vn = kn + D;
    float *sw = S.aux() + warp * hpw * tp;  // this warp's scores, then probabilities: [hpw][tp]
    float *part_base = reinterpret_cast<float *>(PTR(I, S_AT_PART));
    float *out = reinterpret_cast<float *>(PTR(I, S_AT_OUT));
    uint32_t *arrive = reinterpret_cast<uint32_t *>(PTR(I, S_AT_ARRIVE));
    const int rpp = P.page_bytes / (D * 2);
    const int npg = attn_pages(T, D, P.page_bytes);  // K pages, then as many V pages
    const uint32_t kring = ring, vring = ring + npg;
    ring = vring + npg;
    // the split's K (V) rows are consecutive rows of its K (V) page(s), rpp
    // (a power of two) to a page; a split spans at most 4 pages of each
    auto page_ptr = [&](uint32_t r) { return S.pages() + (size_t)(r % P.num_pages) * P.page_bytes; };
    uint8_t *vpage = page_ptr(vring);
    const uint8_t *kpage = page_ptr(kring);
    const uint8_t *kp1 = page_ptr(kring + 1), *kp2 = page_ptr(kring + 2), *kp3 = page_ptr(kring + 3);
    const uint8_t *vp1 = page_ptr(vring + 1), *vp2 = page_ptr(vring + 2), *vp3 = page_ptr(vring + 3);
    const int rsh = 31 - __clz(rpp);
    auto row_at = [&](bool v, int tk) -> const uint8_t * {
        const int j = tk >> rsh;
        const uint8_t *pg = j == 0 ? (v ? vpage : kpage) : j == 1 ? (v ? vp1 : kp1) : j == 2 ? (v ? vp2 : kp2)
                                                                                        : (v ? vp3 : kp3);
        return pg + (size_t)(tk & (rpp - 1)) * (D * 2);
    };
    for (int k = 0; k < npg; ++k)
        if (!ab) ab = !warp_wait_bar(P, S, &S.full()[(kring + k) % P.num_pages], ((kring + k) / P.num_pages) & 1, 2, i, MK_OP_ATTN);
    trace_stamp(P, i, 6);
    // ---- scores.  Lane (tl, dq): token t + tl of a round of 4, dims
    // c * 64 + dq * 8 .. + 8 of each chunk c: the 8 lanes of a token read 128
    // contiguous bytes of its row, a warp 4 rows (conflict-free).
    const int tl = lane >> 3, dq = lane & 7;
    uint64_t q2[4][NCH * 4];  // q of the warp's heads (zero past hpw) as fp32 pairs
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int d0 = c * 64 + dq * 8, hh = wh * hpw + (j < hpw ? j : 0);
            const float *qs = qp + (hh * 4 + d0 / (D / 4)) * QS + d0 % (D / 4);
            float4 v0 = *reinterpret_cast<const float4 *>(qs), v1 = *reinterpret_cast<const float4 *>(qs + 4);
            if (j >= hpw) v0 = v1 = make_float4(0.f, 0.f, 0.f, 0.f);
            q2[j][c * 4] = pack2(v0.x, v0.y);
            q2[j][c * 4 + 1] = pack2(v0.z, v0.w);
            q2[j][c * 4 + 2] = pack2(v1.x, v1.y);
            q2[j][c * 4 + 3] = pack2(v1.z, v1.w);
        }
    // after the reduce-scatter lane dq holds the score of head hown
    const int hown = ((dq >> 2) & 1) * 2 + ((dq >> 1) & 1);
    float mown = -INFINITY;
    for (int t = tb; t < te; t += 4) {
        const int tk = t + tl;
        uint64_t a[4] = {0, 0, 0, 0};
        auto dot = [&](int c, uint64_t k0, uint64_t k1, uint64_t k2, uint64_t k3) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                fma2(a[j], k0, q2[j][c * 4]);
                fma2(a[j], k1, q2[j][c * 4 + 1]);
                fma2(a[j], k2, q2[j][c * 4 + 2]);
                fma2(a[j], k3, q2[j][c * 4 + 3]);
            }
        };
        if (tk < tc) {
            const uint8_t *row = row_at(false, tk) + dq * 16;
            uint4 kw[NCH];
#pragma unroll
            for (int c = 0; c < NCH; ++c) kw[c] = *reinterpret_cast<const uint4 *>(row + c * 128);
#pragma unroll
            for (int c = 0; c < NCH; ++c)
                dot(c, bf16x2_pair(kw[c].x), bf16x2_pair(kw[c].y), bf16x2_pair(kw[c].z), bf16x2_pair(kw[c].w));
        } else if (tk < te) {  // the new token: its k staged in fp32 (bf16-rounded)
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const float *kk = kn + c * 64 + dq * 8;
                const float4 x0 = *reinterpret_cast<const float4 *>(kk), x1 = *reinterpret_cast<const float4 *>(kk + 4);
                dot(c, pack2(x0.x, x0.y), pack2(x0.z, x0.w), pack2(x1.x, x1.y), pack2(x1.z, x1.w));
            }
        }
        float s[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) s[j] = sum2(a[j]);
        // reduce-scatter over the 8 dim lanes: xor 4 keeps heads {0,1} or
        // {2,3}, xor 2 one of the pair, xor 1 completes the sum
        const bool h4 = dq & 4, h2 = dq & 2;
        const float r0 = __shfl_xor_sync(FULL, h4 ? s[0] : s[2], 4);
        const float r1 = __shfl_xor_sync(FULL, h4 ? s[1] : s[3], 4);
        const float u0 = (h4 ? s[2] : s[0]) + r0, u1 = (h4 ? s[3] : s[1]) + r1;
        float v = (h2 ? u1 : u0) + __shfl_xor_sync(FULL, h2 ? u0 : u1, 2);
        v += __shfl_xor_sync(FULL, v, 1);
        if (tk < te && hown < hpw) {
            if ((dq & 1) == 0) sw[hown * tp + tk - tb] = v;
            mown = fmaxf(mown, v);
        }
    }
    mown = fmaxf(mown, __shfl_xor_sync(FULL, mown, 8));
    mown = fmaxf(mown, __shfl_xor_sync(FULL, mown, 16));
    float M[4];  // head j's maximum sits on lanes 2j, 2j + 1
#pragma unroll
    for (int j = 0; j < 4; ++j) M[j] = __shfl_sync(FULL, mown, 2 * j);
    trace_stamp(P, i, 7);
    __syncwarp();
    if (lane == 0)
        for (int k = 0; k < npg; ++k) page_release<FL>(S, (kring + k) % P.num_pages);
    float l4[4] = {0.f, 0.f, 0.f, 0.f};
    for (int t = lane; t < te - tb; t += 32) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (j < hpw) {
                const float e = exp2f(sw[j * tp + t] - M[j]);
                sw[j * tp + t] = e;
                l4[j] += e;
            }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) l4[j] = warp_sum(l4[j]);
    __syncwarp();
    // ---- P.V
    for (int k = 0; k < npg; ++k)
        if (!ab) ab = !warp_wait_bar(P, S, &S.full()[(vring + k) % P.num_pages], ((vring + k) / P.num_pages) & 1, 2, i, MK_OP_ATTN);
    trace_stamp(P, i, 8);
    const int dg = lane % NG, tg = lane / NG;
    uint64_t acc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[j][k] = 0;
    auto pv = [&](int t, const uint8_t *row) {
        const uint4 u = *reinterpret_cast<const uint4 *>(row + dg * 16);
        const uint64_t v0 = bf16x2_pair(u.x), v1 = bf16x2_pair(u.y), v2 = bf16x2_pair(u.z), v3 = bf16x2_pair(u.w);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float p = j < hpw ? sw[j * tp + t - tb] : 0.f;
            const uint64_t pp = pack2(p, p);
            fma2(acc[j][0], v0, pp);
            fma2(acc[j][1], v1, pp);
            fma2(acc[j][2], v2, pp);
            fma2(acc[j][3], v3, pp);
        }
    };
    if (npg == 1) {
        for (int t = tb + tg; t < tc; t += TG) pv(t, vpage + (size_t)t * (D * 2));
    } else {
        for (int t = tb + tg; t < tc; t += TG) pv(t, row_at(true, t));
    }
    // reduce-scatter over the TG token lanes: each lane keeps 8 dims of
    // 4 / TG heads, hk[0 .. 4 / TG) (TG = 2: heads 2 tg, 2 tg + 1; TG = 4:
    // head 2 (tg & 1) + (tg >> 1))
    constexpr int HK = 4 / TG;
    float o[HK][8];
    int hk[HK];
    {
        const bool b0 = tg & 1;
        uint64_t keep[2][4];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint64_t send = b0 ? acc[jj][k] : acc[2 + jj][k];
                const uint64_t mine = b0 ? acc[2 + jj][k] : acc[jj][k];
                const uint64_t r = __shfl_xor_sync(FULL, send, NG);
                keep[jj][k] = pack2(__uint_as_float((uint32_t)mine) + __uint_as_float((uint32_t)r),
                                    __uint_as_float((uint32_t)(mine >> 32)) + __uint_as_float((uint32_t)(r >> 32)));
            }
        if constexpr (TG == 2) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                hk[jj] = 2 * (b0 ? 1 : 0) + jj;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    o[jj][2 * k] = __uint_as_float((uint32_t)keep[jj][k]);
                    o[jj][2 * k + 1] = __uint_as_float((uint32_t)(keep[jj][k] >> 32));
                }
            }
        } else {
            const bool b1 = tg & 2;
            hk[0] = 2 * (b0 ? 1 : 0) + (b1 ? 1 : 0);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint64_t send = b1 ? keep[0][k] : keep[1][k];
                const uint64_t mine = b1 ? keep[1][k] : keep[0][k];
                const uint64_t r = __shfl_xor_sync(FULL, send, 2 * NG);
                o[0][2 * k] = __uint_as_float((uint32_t)mine) + __uint_as_float((uint32_t)r);
                o[0][2 * k + 1] = __uint_as_float((uint32_t)(mine >> 32)) + __uint_as_float((uint32_t)(r >> 32));
            }
        }
    }
    if (has_new && ncache >= tb && ncache < te) {  // the new token is this warp's
#pragma unroll
        for (int jj = 0; jj < HK; ++jj) {
            const float p = hk[jj] < hpw ? sw[hk[jj] * tp + ncache - tb] : 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[jj][e] = fmaf(p, vn[dg * 8 + e], o[jj][e]);
        }
    }
    // ---- combine the warps' pieces in the first V page: [warp][head 0..3][D]
    // fp32 (at most 16 KB, one page); max and sum over the slot's staged q
    // (dead by now; the slot, like the page, is not refilled before every
    // warp has released it)
    consumer_sync(P, S, cph, ab, i);  // no warp reads V, q, k or v any more (a bounded wait)
    float *cb = reinterpret_cast<float *>(vpage);
    float *mlb = const_cast<float *>(slot);  // [warp][head 0..3][2]
#pragma unroll
    for (int jj = 0; jj < HK; ++jj)
        if (hk[jj] < hpw) {
            float4 *dst = reinterpret_cast<float4 *>(cb + (size_t)(warp * 4 + hk[jj]) * D + dg * 8);
            dst[0] = make_float4(o[jj][0], o[jj][1], o[jj][2], o[jj][3]);
            dst[1] = make_float4(o[jj][4], o[jj][5], o[jj][6], o[jj][7]);
        }
    if (lane < hpw) {
        float mj = M[0], lj = l4[0];
#pragma unroll
        for (int j = 1; j < 4; ++j) {
            mj = lane == j ? M[j] : mj;
            lj = lane == j ? l4[j] : lj;
        }
        mlb[(warp * 4 + lane) * 2] = mj;
        mlb[(warp * 4 + lane) * 2 + 1] = lj;
    }
    // the page's next contents arrive by bulk copy (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    consumer_sync(P, S, cph, ab, i);
    const bool merger = warp < G;  // warp h merges head h of the kv group
    if (!merger) {
        __syncwarp();
        if (lane == 0) {
            for (int k = 0; k < npg; ++k) page_release<FL>(S, (vring + k) % P.num_pages);
            mbar_arrive(&S.act_empty()[sl]);  // q, k, v of the slot no longer needed by this warp
        }
        trace_stamp(P, i, 9);
        trace_stamp(P, i, 10);
        return;
    }
    const int jm = warp % hpw, src0 = (warp / hpw) * tw;  // the head's pieces: warps src0 .. src0 + tw
    float Mx = -INFINITY;
    for (int k = 0; k < tw; ++k) Mx = fmaxf(Mx, mlb[((src0 + k) * 4 + jm) * 2]);
    float L = 0.f, om[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) om[e] = 0.f;
    if (Mx != -INFINITY) {
        for (int k = 0; k < tw; ++k) {
            const float f = exp2f(mlb[((src0 + k) * 4 + jm) * 2] - Mx);  // 0 for a warp with no tokens
            L += f * mlb[((src0 + k) * 4 + jm) * 2 + 1];
            const float *ps = cb + (size_t)((src0 + k) * 4 + jm) * D + lane * PER;
#pragma unroll
            for (int e = 0; e < PER; ++e) om[e] = fmaf(f, ps[e], om[e]);
        }
    }
    __syncwarp();
    if (lane == 0) {
        for (int k = 0; k < npg; ++k) page_release<FL>(S, (vring + k) % P.num_pages);
        mbar_arrive(&S.act_empty()[sl]);
    }
    trace_stamp(P, i, 9);
    // the split's partial (o[D], max, sum) of head (b, g * G + warp)
    const int head = g * G + warp;
    float *pp = part_base + ((size_t)(b * P.Hq + head) * P.nsplit_max + split) * (D + 2);
    if (!ab) {
#pragma unroll
        for (int e = 0; e < PER; ++e) pp[lane * PER + e] = om[e];
        if (lane == 0) {
            pp[D] = Mx;
            pp[D + 1] = L;
        }
    }
    // the acq_rel add is cumulative over this warp's partial (ordered by the
    // warp barrier) and acquires the other splits' partials
    __syncwarp();
    int last = 0;
    if (lane == 0 && !ab) {
        const uint32_t old = atom_acqrel_add(arrive + ((size_t)layer * P.B + b) * P.Hq + head, 1u);
        last = old == (uint32_t)(I.step + 1) * (uint32_t)nsplit - 1u;
    }
    trace_stamp(P, i, 10);
    if (!__shfl_sync(FULL, last, 0)) return;
    __syncwarp();
    // merge: log-sum-exp over the head's splits, MB at a time so that their
    // L2 round trips overlap
    const float *hb = part_base + (size_t)(b * P.Hq + head) * P.nsplit_max * (D + 2);
    const int n = nsplit;
    float MM = -INFINITY, LL = 0.f, ov2[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) ov2[e] = 0.f;
    constexpr int MB = PER <= 2 ? 16 : 8;
    for (int s0 = 0; s0 < n; s0 += MB) {
        float mv[MB], lv[MB], ov[MB][PER];
#pragma unroll
        for (int u = 0; u < MB; ++u) {
            const int sp = s0 + u;
            if (sp < n) {
                const float *ps = hb + (size_t)sp * (D + 2);
                mv[u] = __ldcg(ps + D);
                lv[u] = __ldcg(ps + D + 1);
#pragma unroll
                for (int e = 0; e < PER; ++e) ov[u][e] = __ldcg(ps + lane * PER + e);
            } else {
                mv[u] = -INFINITY;
                lv[u] = 0.f;
#pragma unroll
                for (int e = 0; e < PER; ++e) ov[u][e] = 0.f;
            }
        }
        float Mn = MM;
#pragma unroll
        for (int u = 0; u < MB; ++u) Mn = fmaxf(Mn, mv[u]);
        if (Mn == -INFINITY) continue;  // nothing yet
        const float r = exp2f(MM - Mn);  // rescale what was accumulated so far
        LL *= r;
#pragma unroll
        for (int e = 0; e < PER; ++e) ov2[e] *= r;
#pragma unroll
        for (int u = 0; u < MB; ++u) {
            const float f = exp2f(mv[u] - Mn);  // 0 for empty pieces
            LL += f * lv[u];
#pragma unroll
            for (int e = 0; e < PER; ++e) ov2[e] += f * ov[u][e];
        }
        MM = Mn;
    }
    if constexpr (FL == FL_TC) {
        // the O tiles' input: bf16 high and low rows b and np + b of [2 np, Hq D]
        uint16_t *o16 = reinterpret_cast<uint16_t *>(out);
        const size_t ld = (size_t)P.Hq * D;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const float v = ov2[e] / LL;
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
            o16[(size_t)b * ld + (size_t)head * D + lane * PER + e] = __bfloat16_as_ushort(hi);
            o16[(size_t)(P.np + b) * ld + (size_t)head * D + lane * PER + e] = __bfloat16_as_ushort(lo);
        }
    } else {
#pragma unroll
        for (int e = 0; e < PER; ++e) out[((size_t)b * P.Hq + head) * D + lane * PER + e] = ov2[e] / LL;
    }
}

// One attention instruction: the per-head form at head_dim 64, the grouped
// form (fewer loads and conversions per K / V byte) at head_dim 128.  A split
// leaves attn_split_pieces(G, D) partials per head (the workspace's stride).
template <int D, int FL>
DEV void attn_task(const KParams &P, const Smem S, const WIns &I, int i, int sl, const float *slot, uint32_t &ring,
                   uint32_t &cph, bool &ab) {
    if constexpr (D == 64) attn_task_heads<D, FL>(P, S, I, i, sl, slot, ring, ab);
    else attn_task_group<D, FL>(P, S, I, i, sl, slot, ring, cph, ab);
}

DEV void embed_task(const KParams &P, const Smem S, const WIns &I, int i, int sl, bool ab) {
    const int ct = threadIdx.x - CONSUMER_BASE, lane = ct & 31;
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.act_empty()[sl]);
    if (ab) return;
    const uint16_t *E = reinterpret_cast<const uint16_t *>(PTR(I, S_EMB_W));
    float *h = reinterpret_cast<float *>(PTR(I, S_EMB_H));
    int32_t *tokens = reinterpret_cast<int32_t *>(PTR(I, S_EMB_TOK));
    const unsigned long long *keys = reinterpret_cast<const unsigned long long *>(PTR(I, S_EMB_KEYS));
    const int step = I.step;
    const bool host_tokens = (P.flags & MK_RUN_HOST_TOKENS) || step == 0;
    for (int b = 0; b < P.B; ++b) {
        int tok;
        if (host_tokens) tok = __ldcg(tokens + (size_t)step * P.B + b);
        else tok = (int)(0xFFFFFFFFu - (uint32_t)(__ldcg(keys + (size_t)(step - 1) * P.B + b) & 0xFFFFFFFFull));
        if (tok < 0 || tok >= P.V) tok = 0;  // out-of-range ids read row 0 instead of faulting
        if (!host_tokens && ct == 0) tokens[(size_t)step * P.B + b] = tok;
        for (int k = ct; k < P.H; k += CONSUMERS) h[(size_t)b * P.H + k] = bf16_at(E, (size_t)tok * P.H + k);
    }
}

}  // namespace mk
