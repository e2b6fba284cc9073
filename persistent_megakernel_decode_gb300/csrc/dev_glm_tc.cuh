// GLM FP8 GEMMs on the 5th-gen tensor cores (tcgen05, sm_103a).
//
// "MegaRTP megakernel article", section 1: every GEMM of the block is e4m3
// weights x e4m3 activations with fp32 scales per 128-wide K block (the
// activation's per token row, the weight's per 128 x 128 block); section 4:
// a large-M GEMM path with an MMAer warp beside the loaders; section 5:
// single-CTA tcgen05 tiles inside the per-CTA interpreter.
//
// A tile is 128 weight rows (the MMA's M side) x the 16 token rows (its N
// side) over a K range, in stages of 128 K columns -- exactly one scale
// block.  The loader brings each stage's weights (16 KB, one TMA box of
// 128 rows x 128 bytes, 128-byte swizzled) into a page; the activation
// loader brings the tile's whole K range of activation codes (2 KB a stage)
// and the activation scales into the activation slot.  One elected
// thread of the MMA warp issues a stage's four MMAs of K = 32
// (tcgen05.mma.cta_group::1.kind::f8f6f4, e4m3 x e4m3, fp32 accumulate) into
// a fresh TMEM accumulator -- one per stage, four in flight -- so each
// accumulator holds exactly one block's dot products.  Four epilogue warps
// read each block back (tcgen05.ld, one TMEM lane quarter = 32 weight rows
// per warp, the 16 token columns in registers), multiply by that block's
// two scales and add in fp32: the block scales are arbitrary fp32 values,
// so they cannot ride inside the MMA.
//
// The first GEMMs (19 row tiles alone would leave most SMs idle) split K
// over tiles that add their fp32 parts into sum buffers; FIN, which waits
// for all of them anyway, rounds the sums to bf16 and zeroes them for the
// next step.  Whole-K tiles (Q-B, Indexer-Q) round and store their outputs
// themselves, rotating the 64-row halves that are a head's RoPE slice (pairs
// c, c + 32 meet through shared memory).
#pragma once
#include "dev_glm.cuh"
#include "dev_tc.cuh"

namespace mk {

// Instruction descriptor of kind::f8f6f4: e4m3 A and B (K-major), fp32 D,
// M = 128, N = 16 (A / B format code 0 is E4M3).
MK_HD constexpr uint32_t gt_idesc() {
    return (1u << 4)                           // D format: fp32
           | ((uint32_t)(GT_N >> 3) << 17)     // N / 8
           | ((uint32_t)(GT_M >> 4) << 24);    // M / 16
}
DEV void tc_mma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Activation scales of a slot, after the codes: the GEMM's whole [M][K / 128]
// fp32 scale matrix (one bulk copy, no register round trip).
DEV float *gt_slot_scales(const Smem S, int xs) {
    return reinterpret_cast<float *>(S.xslot(xs) + GT_MAX_STAGES * GT_XSTAGE_BYTES);
}

// ---------------------------------------------------------------- loader warp
// Weights of stage s into `page`: rows row0 .. + 127 (zeros past the
// matrix's end), K columns k0 + 128 s .. + 127.  Lane 0; the fields come
// from gt_tile_fields (whole warp).
struct GtTile {
    const void *tw;
    int row0, k0, nst;
};
DEV GtTile gt_tile_fields(const WIns &I) {
    GtTile t;
    t.tw = reinterpret_cast<const void *>(PTR(I, S_GG_TW));
    t.row0 = F(I, P_ROW0);
    t.k0 = F(I, P_K0);
    t.nst = F(I, P_NPG);
    return t;
}
DEV void gt_load_stage(const GtTile &t, int s, uint8_t *page, uint64_t *bar, uint64_t pol) {
    mbar_expect_tx(bar, GT_STAGE_BYTES);
    tma_load_2d(page, t.tw, t.k0 + s * GT_KS, t.row0, bar, pol);
}

// ---------------------------------------------------------------- activation-loader warp
// After the tile's events are met: its activation codes (one TMA box of 16
// rows x 128 bytes per stage) and the activation scale matrix (one bulk
// copy), completing on the slot's full barrier.  `xq` counts the tiles
// staged so far.
DEV void gt_stage_x(const KParams &P, const Smem S, const WIns &I, int i, uint32_t &xq, bool &ab) {
    const int lane = threadIdx.x & 31;
    const int nst = F(I, P_NPG), k0 = F(I, P_K0), KB = F(I, P_KTOT) / GT_KS, M = F(I, P_GL_M);
    const uint32_t xs = xq % GT_XSLOTS, ph = (xq / GT_XSLOTS) & 1;
    ++xq;
    const void *sa = reinterpret_cast<const void *>(PTR(I, S_GG_XS));
    const void *tmap = reinterpret_cast<const void *>(PTR(I, S_GG_TX));
    if (!ab) ab = !warp_wait_bar(P, S, &S.xempty()[xs], ph ^ 1, 1, i, MK_OP_GLM_GEMM);
    if (lane == 0) {
        uint64_t *bar = &S.xfull()[xs];
        if (!ab) {
            const uint64_t pol = evict_last_policy();  // every row tile of the GEMM reads these rows
            const uint32_t sbytes = (uint32_t)(M * KB * 4);
            fence_proxy_async_global();  // codes and scales were written by generic stores; TMA reads them
            mbar_expect_tx(bar, (uint32_t)(nst * GT_XSTAGE_BYTES) + sbytes);
            for (int s = 0; s < nst; ++s)
                tma_load_2d(S.xslot((int)xs) + s * GT_XSTAGE_BYTES, tmap, k0 + s * GT_KS, 0, bar, pol);
            bulk_g2s_plain(gt_slot_scales(S, (int)xs), sa, sbytes, bar);
        } else {
            mbar_arrive(bar);  // aborting: complete the phase empty
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------- consumer warps
// One tile (see the file comment).  Consumer warp TC_MMA_WARP issues the
// MMAs, warps 0..3 read the accumulators back and store, the others only
// keep their positions.  `tc.tiles` counts the accumulator uses (stages) so
// far, `tc.xq` the tiles.  Returns whether this warp wrote global memory.
DEV bool glm_tc_tile(const KParams &P, const Smem S, const WIns &I, int i, uint32_t &ring, TcState &tc, bool &ab) {
    const int ct = threadIdx.x - CONSUMER_BASE, cw = ct >> 5, lane = ct & 31;
    const int nst = F(I, P_NPG);
    const uint32_t xs = tc.xq % GT_XSLOTS, xph = (tc.xq / GT_XSLOTS) & 1;
    const uint32_t a0 = tc.tiles;
    const uint32_t tmem = *S.tmem_slot();
    bool wrote = false;
    if (cw == TC_MMA_WARP) {
        if (!ab) ab = !warp_wait_bar(P, S, &S.xfull()[xs], xph, 2, i, MK_OP_GLM_GEMM);
        const uint32_t xa = saddr(S.xslot((int)xs));
        RingPos wq;
        wq.set(ring, P.num_pages);
        for (int s = 0; s < nst; ++s) {
            const uint32_t a = (a0 + s) % GT_NACC, use = (a0 + s) / GT_NACC;
            if (!ab) ab = !warp_wait_bar(P, S, &S.accempty()[a], (use & 1) ^ 1, 2, i, MK_OP_GLM_GEMM);
            if (!ab) ab = !warp_wait_bar(P, S, &S.full()[wq.p], wq.ph, 2, i, MK_OP_GLM_GEMM);
            tc_fence_after();
            if (lane == 0 && !ab) {
                const uint32_t wa = saddr(S.pages() + (size_t)wq.p * P.page_bytes);
#pragma unroll
                for (int j = 0; j < GT_KS / GT_KSTEP; ++j)  // 32-byte K steps inside the swizzled rows
                    tc_mma_f8(tmem + a * GT_ACC_COLS, tc_desc(wa + j * 32),
                              tc_desc(xa + s * GT_XSTAGE_BYTES + j * 32), gt_idesc(), j != 0 ? 1u : 0u);
            }
            __syncwarp();
            if (lane == 0) {
                // the page is free and the block's sums are ready once these MMAs are done
                if (!ab) {
                    tc_commit(&S.empty()[wq.p]);
                    tc_commit(&S.accfull()[a]);
                } else {
                    mbar_arrive(&S.empty()[wq.p]);
                    mbar_arrive(&S.accfull()[a]);
                }
            }
            wq.next(P.num_pages);
        }
        if (P.trace && lane == 0) P.trace[((size_t)blockIdx.x * P.lmax + i) * 16 + 6] = gtimer();  // last MMAs issued
        if (lane == 0) {  // the MMAs' part of releasing the activation slot
            if (!ab) tc_commit(&S.xempty()[xs]);
            else mbar_arrive(&S.xempty()[xs]);
        }
        __syncwarp();
    } else if (cw < TC_EPI_WARPS) {
        const int row = cw * 32 + lane;  // this thread's weight row in the tile (its TMEM lane)
        const int KB = F(I, P_KTOT) / GT_KS, kb0 = F(I, P_K0) / GT_KS;
        const float *sw = reinterpret_cast<const float *>(PTR(I, S_GG_SW)) + (size_t)(F(I, P_ROW0) / GT_M) * KB + kb0;
        const float swl = lane < nst ? __ldg(sw + lane) : 0.f;  // the weight scale of stage `lane`
        // RoPE tiles: this row's position factors for every token, loaded while the MMAs run
        const int rope = F(I, P_GL_ROPE), T = F(I, P_GL_T), M = F(I, P_GL_M);
        const bool roped = ((rope >> (row >> 6)) & 1) != 0;  // this row's 64-row half is a RoPE slice (warp-uniform)
        const float2 *rtab = reinterpret_cast<const float2 *>(PTR(I, S_GG_ROPE));
        float2 cs[GT_N];
#pragma unroll
        for (int n = 0; n < GT_N; ++n)
            cs[n] = roped && n < M ? rtab[(n % T) * 32 + (row & 31)] : make_float2(1.f, 0.f);
        if (!ab) ab = !warp_wait_bar(P, S, &S.xfull()[xs], xph, 2, i, MK_OP_GLM_GEMM);  // (the scales)
        trace_stamp(P, i, 7);
        const float *sc = gt_slot_scales(S, (int)xs) + kb0;  // [m][KB], from this tile's first block
        float acc[GT_N];
#pragma unroll
        for (int n = 0; n < GT_N; ++n) acc[n] = 0.f;
        for (int s = 0; s < nst; ++s) {
            const uint32_t a = (a0 + s) % GT_NACC, use = (a0 + s) / GT_NACC;
            if (!ab) ab = !warp_wait_bar(P, S, &S.accfull()[a], use & 1, 2, i, MK_OP_GLM_GEMM);
            tc_fence_after();
            uint32_t d[GT_ACC_COLS];
            if (!ab) {
                tmem_ld16(tmem + a * GT_ACC_COLS + ((uint32_t)(cw * 32) << 16), d);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.accempty()[a]);
            if (s == 0) trace_stamp(P, i, 8);
            const float w = __shfl_sync(FULL, swl, s);
            if (!ab) {
#pragma unroll
                for (int n = 0; n < GT_N; ++n)
                    acc[n] = fmaf(w * sc[n * KB + s], __uint_as_float(d[n]), acc[n]);
            }
        }
        trace_stamp(P, i, 9);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.xempty()[xs]);  // the scales are read
        const int nrows = F(I, P_NROWS), out0 = F(I, P_OUT0), ld = F(I, P_GL_LD), sum = F(I, P_GL_SUM);
        __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(PTR(I, S_GG_OUT));
        float *fsum = reinterpret_cast<float *>(PTR(I, S_GG_FSUM));
        const bool ok = !ab && row < nrows;
        if (sum) {
            // this K part into the GEMM's fp32 sums (FIN rounds them once every part is in)
            if (ok) {
#pragma unroll
                for (int n = 0; n < GT_N; ++n)
                    if (n < M) atomicAdd(fsum + (size_t)n * ld + out0 + row, acc[n]);
            }
        } else {
            float v[GT_N];
#pragma unroll
            for (int n = 0; n < GT_N; ++n) v[n] = round_bf16(acc[n]);
            float *ex = reinterpret_cast<float *>(mk_smem + S.o_aux);  // [GT_N][GT_M]
            if (rope) {
#pragma unroll
                for (int n = 0; n < GT_N; ++n) ex[n * GT_M + row] = v[n];
                epi_bar();
            }
            if (ok) {
                const int c = row & 63;
#pragma unroll
                for (int n = 0; n < GT_N; ++n) {
                    if (n >= M) break;
                    float o = v[n];
                    if (roped) {
                        const float pv = ex[n * GT_M + (row ^ 32)];
                        o = c < 32 ? v[n] * cs[n].x - pv * cs[n].y : v[n] * cs[n].x + pv * cs[n].y;
                    }
                    out[(size_t)n * ld + out0 + row] = __float2bfloat16_rn(o);
                }
            }
            if (rope) epi_bar();  // the exchange is read before any warp's next tile writes it
        }
        trace_stamp(P, i, 12);
        wrote = true;
    }
    ring += nst;
    tc.tiles += nst;
    tc.xq += 1;
    return wrote;
}

}  // namespace mk
