// Tensor-core tiles for batched decode (batch 8 .. 16) on sm_103a: 5th-gen
// tensor cores (tcgen05) with accumulators in tensor memory (TMEM), operands
// staged in shared memory by TMA tensor copies.
//
// Where the batch makes a projection a real dense contraction (M = weight
// rows, N = sequences), a GEMV instruction becomes a tile of 128 weight rows
// (two segments of 64 rows, e.g. 64 gate rows and their 64 up rows) over a K
// range, streamed in stages of 128 K columns: the loader warp brings each
// stage's weights (32 KB) into a page of the ring, the activation loader
// brings the matching slice of the input -- bf16 rows, the high and the low
// bf16 part of every fp32 activation value, so x = hi + lo to 2^-16 and the
// products keep fp32-level accuracy -- into a slot of a small activation ring.
// One elected consumer thread issues the stage's 8 MMAs of K = 16
// (tcgen05.mma.cta_group::1.kind::f16, bf16 inputs, fp32 accumulate) from
// shared-memory descriptors into one of two TMEM accumulators and commits
// them to the stage's empty barriers, so the K loop runs through no
// registers.  After the last stage four consumer warps read the 128 x N
// accumulator back (tcgen05.ld, one TMEM lane quarter per warp), add the high
// and low columns and run the op's epilogue.  The large-M GEMM path of the
// "MegaRTP megakernel article" (section 4: a spec registry of compiled GEMM
// paths, an MMAer warp beside the loaders; section 5: single-CTA tcgen05 tiles
// inside the per-CTA interpreter) is the prior art.
//
// Shared-memory layouts are the canonical K-major ones with 128-byte
// swizzling: a box of 64 bf16 columns x R rows lands as R rows of 128 bytes,
// 8-row groups 1024 bytes apart (the stride the descriptors carry), so every
// stage buffer starts 1024-byte aligned.
#pragma once
#include "dev_ops.cuh"

namespace mk {

// (Tile geometry: TC_* in mk_internal.h.)

// ---------------------------------------------------------------- PTX wrappers
// 2-D TMA tensor load of one box into shared memory, completing on `bar`
// (coordinates: x = innermost, in elements; y = row).
DEV void tma_load_2d(void *dst, const void *tmap, int x, int y, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(saddr(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(saddr(bar)), "l"(pol)
        : "memory");
}
// Orders this thread's earlier generic-proxy view of global memory (the
// activation it acquired) before its later async-proxy (TMA) reads.
DEV void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (stride byte offset), leading byte offset unused
// for swizzled K-major operands (encoded 1), descriptor version 1.
DEV uint64_t tc_desc(uint32_t smem_addr) {
    uint64_t d = (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;                 // leading byte offset (16 B, unused)
    d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
    d |= (uint64_t)1 << 46;                 // version
    d |= (uint64_t)2 << 61;                 // 128-byte swizzle
    return d;
}
// Instruction descriptor of kind::f16: bf16 A and B (K-major), fp32 D, M x N.
MK_HD constexpr uint32_t tc_idesc(int m, int n) {
    return (1u << 4)                         // D format: fp32
           | (1u << 7)                       // A format: bf16
           | (1u << 10)                      // B format: bf16
           | ((uint32_t)(n >> 3) << 17)      // N / 8
           | ((uint32_t)(m >> 4) << 24);     // M / 16
}
DEV void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The barrier gets one arrival once every MMA this thread issued so far is done.
DEV void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
                 : "memory");
}
DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Whole warp: allocate / free TMEM columns (power of two >= 32); the address
// is written to shared memory.
DEV void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(dst)), "r"(ncols)
                 : "memory");
}
DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Whole warp: 32 lanes x 16 consecutive 32-bit columns of TMEM (lane i of the
// warp reads TMEM lane (taddr >> 16) + i).
DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
DEV uint64_t evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Named barrier 2 over the TC_EPI_WARPS epilogue warps.
DEV void epi_bar() { asm volatile("bar.sync 2, %0;" ::"n"(TC_EPI_WARPS * 32) : "memory"); }

DEV bool is_gemv_op(int opc) { return opc >= MK_OP_QKV && opc <= MK_OP_LM && opc != MK_OP_ATTN; }

// ---------------------------------------------------------------- loader warp
// Weights of one stage s of a tile into the page at `page`: per 64-column K
// box, segment 0's 64 rows, then segment 1's (rows 0..63 and 64..127 of the
// tile), 8 KB each.  Whole warp; lane 0 issues.
struct TcTile {
    const void *t0, *t1;  // tensor maps of the two segments
    int r0, r1, k0, nst;
};
DEV TcTile tc_tile_fields(const WIns &I) {
    TcTile t;
    t.t0 = reinterpret_cast<const void *>(PTR(I, S_T_W0 + F(I, P_MAT)));
    t.t1 = reinterpret_cast<const void *>(PTR(I, S_T_W0 + F(I, P_S1_MAT)));
    t.r0 = F(I, P_ROW0);
    t.r1 = F(I, P_S1_ROW0);
    t.k0 = F(I, P_K0);
    t.nst = F(I, P_NPG);
    return t;
}
DEV void tc_load_stage(const TcTile &t, int s, uint8_t *page, uint64_t *bar, uint64_t pol) {
    mbar_expect_tx(bar, TC_STAGE_BYTES);
#pragma unroll
    for (int kb = 0; kb < TC_KS / TC_BOX; ++kb) {
        const int x = t.k0 + s * TC_KS + kb * TC_BOX;
        uint8_t *dst = page + kb * (TC_M * 128);
        tma_load_2d(dst, t.t0, x, t.r0, bar, pol);
        tma_load_2d(dst + TC_SEG * 128, t.t1, x, t.r1, bar, pol);
    }
}

// ---------------------------------------------------------------- activation-loader warp
// After the tile's events are met: the input's high/low rows for every stage
// into the activation ring (2 np rows x 64 columns per box, two boxes per
// stage).  `xq` counts the stages staged so far.
DEV void tc_stage_x(const KParams &P, const Smem S, const WIns &I, int i, uint32_t &xq, bool &ab) {
    const int lane = threadIdx.x & 31;
    const int nst = F(I, P_NPG), k0 = F(I, P_K0), opc = F(I, W_OPC), n = 2 * P.np;
    const void *tmap = reinterpret_cast<const void *>(PTR(I, S_T_X));
    const uint64_t pol = evict_last_policy();
    fence_proxy_async_global();  // the activation was written by generic stores; TMA reads it
    for (int s = 0; s < nst; ++s) {
        const uint32_t xs = xq % TC_XSLOTS, ph = (xq / TC_XSLOTS) & 1;
        if (!ab) ab = !warp_wait_bar(P, S, &S.xempty()[xs], ph ^ 1, 1, i, opc);
        if (lane == 0) {
            uint64_t *bar = &S.xfull()[xs];
            if (!ab) {
                mbar_expect_tx(bar, (uint32_t)tc_xstage_bytes(P.np));
                tma_load_2d(S.xslot(xs), tmap, k0 + s * TC_KS, 0, bar, pol);
                tma_load_2d(S.xslot(xs) + n * 128, tmap, k0 + s * TC_KS + TC_BOX, 0, bar, pol);
            } else {
                mbar_arrive(bar);  // aborting: complete the phase empty
            }
        }
        __syncwarp();
        ++xq;
    }
}

// ---------------------------------------------------------------- consumer warps
// What every consumer warp keeps across tensor-core tiles: the tiles so far
// (accumulator tiles & 1, its use tiles >> 1) and the activation stages so far.
struct TcState {
    uint32_t tiles = 0;
    uint32_t xq = 0;
};

// Epilogue of one accumulator row (row = cw * 32 + lane of the tile) for the
// op; y[b] = the row's result for sequence b.  Always reached by all four
// epilogue warps (MLP-up meets on a named barrier).
DEV bool tc_epilogue(const KParams &P, const Smem S, const WIns &I, const Dec &d, int cw, int lane, int a,
                     const float (&y)[TC_MAXB], unsigned long long &lm_best, bool ab) {
    const int row = cw * 32 + lane, B = P.B, np = P.np;
    const int opc = d.opc, out0 = d.out0, nrows = d.nrows;
    if (opc == MK_OP_UP) {
        // rows 0..63 are gate rows, 64..127 their up rows: the up warps hand
        // their values over through shared memory (one buffer per accumulator)
        float *ex = reinterpret_cast<float *>(mk_smem + S.o_aux + P.aux_bytes - NRED * P.red_bytes) -
                    2 * TC_SEG * TC_MAXB + a * TC_SEG * TC_MAXB;
        const int rr = row & (TC_SEG - 1);
        if (row >= TC_SEG) {
#pragma unroll
            for (int b = 0; b < TC_MAXB; ++b) ex[rr * TC_MAXB + b] = y[b];
        }
        epi_bar();
        if (row < TC_SEG && !ab && rr < nrows) {
            uint16_t *act = reinterpret_cast<uint16_t *>(d.out);  // bf16 [2 np][F]: high rows, then low rows
#pragma unroll
            for (int b = 0; b < TC_MAXB; ++b) {
                if (b >= B) break;
                const float g = y[b], u = ex[rr * TC_MAXB + b];
                const float v = g / (1.0f + __expf(-g)) * u;
                const __nv_bfloat16 hi = __float2bfloat16_rn(v);
                const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
                act[(size_t)b * P.F + out0 + rr] = __bfloat16_as_ushort(hi);
                act[(size_t)(np + b) * P.F + out0 + rr] = __bfloat16_as_ushort(lo);
            }
        }
        return true;
    }
    const bool ok = !ab && row < nrows;
    float *out = reinterpret_cast<float *>(d.out);
    if (opc == MK_OP_QKV) {
        const int ldq = P.Hkv * (P.Hq / P.Hkv + 2) * P.D;
        const bool split = d.kc < F(I, P_KTOT);  // K split over tiles: add into the zeroed row
#pragma unroll
        for (int b = 0; b < TC_MAXB; ++b) {
            if (b >= B || !ok) break;
            if (split) atomicAdd(out + (size_t)b * ldq + out0 + row, y[b]);
            else out[(size_t)b * ldq + out0 + row] = y[b];
        }
    } else if (opc == MK_OP_O || opc == MK_OP_DOWN) {  // residual: h += this K range's part
#pragma unroll
        for (int b = 0; b < TC_MAXB; ++b) {
            if (b >= B || !ok) break;
            atomicAdd(out + (size_t)b * P.H + out0 + row, y[b]);
        }
    } else {  // LM head: logits and each sequence's running argmax key
        unsigned long long mine = 0;
#pragma unroll
        for (int b = 0; b < TC_MAXB; ++b) {
            if (b >= B) break;
            if (ok) out[(size_t)b * P.V + out0 + row] = y[b];
            unsigned long long key = ok ? argmax_key(y[b], out0 + row) : 0ull;
#pragma unroll
            for (int o = 16; o; o >>= 1) key = max(key, __shfl_xor_sync(FULL, key, o));
            if (lane == b) mine = key;
        }
        if (lane < B && !ab && mine > lm_best) {
            lm_best = mine;
            red_max_u64(reinterpret_cast<unsigned long long *>(d.out2) + (size_t)d.step * B + lane, mine);
        }
    }
    return true;
}

// One tensor-core tile (see the file comment).  Consumer warp TC_MMA_WARP
// issues the MMAs; warps 0..3 read the accumulator back and store; the others
// only keep their positions.  Every warp advances `ring` and `tc`.  Returns
// whether this warp wrote global memory.
DEV bool tc_tile(const KParams &P, const Smem S, const WIns &I, const Dec &d, int i, uint32_t &ring, TcState &tc,
                 unsigned long long &lm_best, bool &ab) {
    const int ct = threadIdx.x - CONSUMER_BASE, cw = ct >> 5, lane = ct & 31;
    const int nst = d.npg, np = P.np, n = 2 * np;
    const int a = (int)(tc.tiles & 1);
    const uint32_t use = tc.tiles >> 1;
    const uint32_t tmem = *S.tmem_slot() + (uint32_t)(a * TC_ACC_COLS);
    bool wrote = false;
    if (cw == TC_MMA_WARP) {
        if (!ab) ab = !warp_wait_bar(P, S, &S.accempty()[a], (use & 1) ^ 1, 2, i, d.opc);
        tc_fence_after();
        const uint32_t idesc = tc_idesc(TC_M, n);
        RingPos wq;
        wq.set(ring, P.num_pages);
        for (int s = 0; s < nst; ++s) {
            const uint32_t xs = (tc.xq + s) % TC_XSLOTS, xph = ((tc.xq + s) / TC_XSLOTS) & 1;
            if (!ab) ab = !warp_wait_bar(P, S, &S.full()[wq.p], wq.ph, 2, i, d.opc);
            if (!ab) ab = !warp_wait_bar(P, S, &S.xfull()[xs], xph, 2, i, d.opc);
            tc_fence_after();
            if (lane == 0 && !ab) {
                const uint32_t wa = saddr(S.pages() + (size_t)wq.p * P.page_bytes);
                const uint32_t xa = saddr(S.xslot(xs));
#pragma unroll
                for (int j = 0; j < TC_KS / TC_KSTEP; ++j) {
                    const uint32_t kb = j >> 2, kk = (j & 3) * 32;  // TMA box, 32-byte K step inside its rows
                    tc_mma(tmem, tc_desc(wa + kb * (TC_M * 128) + kk), tc_desc(xa + kb * (n * 128) + kk), idesc,
                           (s | j) != 0 ? 1u : 0u);
                }
            }
            __syncwarp();
            if (lane == 0) {
                // the page and the activation slot are free once these MMAs are done
                if (!ab) {
                    tc_commit(&S.empty()[wq.p]);
                    tc_commit(&S.xempty()[xs]);
                } else {
                    mbar_arrive(&S.empty()[wq.p]);
                    mbar_arrive(&S.xempty()[xs]);
                }
            }
            wq.next(P.num_pages);
        }
        if (lane == 0) {
            if (!ab) tc_commit(&S.accfull()[a]);
            else mbar_arrive(&S.accfull()[a]);
        }
        __syncwarp();
    } else if (cw < TC_EPI_WARPS) {
        if (!ab) ab = !warp_wait_bar(P, S, &S.accfull()[a], use & 1, 2, i, d.opc);
        tc_fence_after();
        float y[TC_MAXB];
#pragma unroll
        for (int b = 0; b < TC_MAXB; ++b) y[b] = 0.f;
        if (!ab) {
            // this warp's TMEM lane quarter: tile rows cw * 32 .. + 31
            const uint32_t taddr = tmem + ((uint32_t)(cw * 32) << 16);
            uint32_t h[16], l[16];
            tmem_ld16(taddr, h);
            if (np == 16) tmem_ld16(taddr + 16, l);
            tmem_wait_ld();
#pragma unroll
            for (int b = 0; b < TC_MAXB; ++b) {
                if (np == 16) y[b] = __uint_as_float(h[b]) + __uint_as_float(l[b]);
                else if (b < 8) y[b] = __uint_as_float(h[b]) + __uint_as_float(h[8 + b]);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.accempty()[a]);
        wrote = tc_epilogue(P, S, I, d, cw, lane, a, y, lm_best, ab);
    }
    ring += nst;
    tc.tiles += 1;
    tc.xq += nst;
    return wrote;
}

// RMSNorm of sequence b's residual into bf16 high/low rows b and np + b of
// the normalised-activation buffer (x = hi + lo), by the 8 consumer warps;
// optionally zeroes that sequence's qkv row (the QKV tiles then add their K
// parts) and captures the residual (tests).
DEV void norm_task(const KParams &P, const Smem S, const WIns &I, bool ab) {
    const int ct = threadIdx.x - CONSUMER_BASE, cw = ct >> 5, lane = ct & 31;
    const int b = F(I, P_NB), zero = F(I, P_NZERO), snap = F(I, P_NSNAP);
    const int H = P.H, n4 = H / 4, np = P.np;
    const float4 *h4 = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(PTR(I, S_N_H)) + (size_t)b * H);
    const uint2 *w4 = reinterpret_cast<const uint2 *>(PTR(I, S_N_W));
    uint16_t *xn = reinterpret_cast<uint16_t *>(PTR(I, S_N_XN));
    float *qkv = reinterpret_cast<float *>(PTR(I, S_N_QKV));
    float *hist = reinterpret_cast<float *>(PTR(I, S_N_HIST));
    constexpr int MAXV = 8;  // hidden up to 8192
    float4 v[MAXV];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
        const int k = ct + CONSUMERS * j;
        v[j] = k < n4 ? __ldcg(h4 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
        ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    }
    ss = warp_sum(ss);
    float *red = S.red(0);
    if (lane == 0) red[cw] = ss;
    consumer_bar();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < CONSUMER_WARPS; ++w) tot += red[w];
    const float scale = rsqrtf(tot / (float)H + P.eps);
    if (!ab) {
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            const int k = ct + CONSUMERS * j;
            if (k >= n4) break;
            const uint2 w = __ldg(w4 + k);
            const float e[4] = {v[j].x * scale * __uint_as_float(w.x << 16),
                                v[j].y * scale * __uint_as_float(w.x & 0xffff0000u),
                                v[j].z * scale * __uint_as_float(w.y << 16),
                                v[j].w * scale * __uint_as_float(w.y & 0xffff0000u)};
            uint32_t hi[2], lo[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const __nv_bfloat16 h0 = __float2bfloat16_rn(e[2 * q]), h1 = __float2bfloat16_rn(e[2 * q + 1]);
                const __nv_bfloat16 l0 = __float2bfloat16_rn(e[2 * q] - __bfloat162float(h0));
                const __nv_bfloat16 l1 = __float2bfloat16_rn(e[2 * q + 1] - __bfloat162float(h1));
                hi[q] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                lo[q] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
            }
            *reinterpret_cast<uint2 *>(xn + (size_t)b * H + 4 * k) = make_uint2(hi[0], hi[1]);
            *reinterpret_cast<uint2 *>(xn + (size_t)(np + b) * H + 4 * k) = make_uint2(lo[0], lo[1]);
            if (snap > 0 && hist) reinterpret_cast<float4 *>(hist + ((size_t)(snap - 1) * P.B + b) * H)[k] = v[j];
        }
        if (zero) {
            const int ldq4 = P.Hkv * (P.Hq / P.Hkv + 2) * P.D / 4;
            float4 *q4 = reinterpret_cast<float4 *>(qkv + (size_t)b * ldq4 * 4);
            for (int k = ct; k < ldq4; k += CONSUMERS) q4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    consumer_bar();  // the reduction words are free again
}

}  // namespace mk
