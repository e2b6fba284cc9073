// Persistent decode interpreter for GB300 (sm_103a) and its launch code.
//
// One worker CTA per SM interprets its row of the static instruction queue
// ("MegaRTP megakernel article", sections 3-4; "CMU 15-779 Lecture 7 notes",
// section 4.1).  Warp roles inside a CTA:
//   warp 0  loader: streams each instruction's weight rows (or KV-cache rows)
//           into a ring of shared-memory pages with bulk TMA copies, running
//           ahead of the consumers and never waiting on an event -- weights
//           do not depend on activations ("Lecture 7 notes", section 4.2);
//   warp 1  activation loader: waits on the instruction's event counters
//           with acquire loads right before reading the activation, then
//           stages the activation (RMSNorm-ed where the op fuses it) into one
//           of two activation slots;
//   warps 2-9 consumers: GEMV / attention math from the pages and the slot,
//           write-back, then publish with a release add on the counters.
// Page handoff uses full/empty mbarriers per page; slot handoff uses
// full/empty mbarriers per slot.  Every wait is bounded: on a timeout a role
// records the failure in the workspace, raises a grid-wide abort flag, and
// all roles drain the rest of the queue without waiting or writing, so the
// kernel always returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "dev_glm.cuh"
#include "dev_ops.cuh"
#include "dev_tc.cuh"
#include "dev_glm_tc.cuh"
#include "planner.h"

namespace mk {

// ---------------------------------------------------------------- loader warp
template <int MAXB, int FL>
DEV void loader_role(const KParams &P, const Smem S, const int32_t *myq) {
    constexpr bool POOLS = fl_pools(FL, MAXB);
    const int lane = threadIdx.x & 31;
    const uint64_t pol = evict_first_policy();
    uint32_t ring = 0, rp = 0, rph = 0;  // pages issued; ring position and its use parity
    int cseq = 0;                        // attention-pool claims posted so far
    const int NP = P.num_pages, PS = P.page_bytes;
    WIns I;
    fetch_init(I, P, myq);
    for (I.step = P.step; I.step < P.step + P.nsteps; ++I.step)
    for (int i = 0; i < P.lmax; ++i) {
        if (cta_aborting(S)) goto drain;
        if (lane < 4 && i + 4 + lane < P.lmax) prefetch_l2(myq + (size_t)(i + 4 + lane) * W_WORDS);
        fetch(I, P, myq, i);
        const int opc = F(I, W_OPC);
        if (!ins_valid<FL>(P, I)) {
            if (lane == 0) raise_error(P, S, MK_ERR_DEVICE_CHECK, i, -1, 0, 0, opc, 0);
            goto drain;
        }
        if constexpr (FL == FL_TC || FL == FL_GLMTC) {
            if (FL == FL_TC ? is_gemv_op(opc) : opc == MK_OP_GLM_GEMM) {  // tensor-core tile: one page per stage
                TcTile t{};
                GtTile g{};
                if (FL == FL_TC) t = tc_tile_fields(I);
                else {
                    g = gt_tile_fields(I);
                    t.nst = g.nst;
                }
                if (P.trace && lane == 0) P.trace[((size_t)blockIdx.x * P.lmax + i) * 16 + 4] = gtimer();
                bool stop = false;
                for (int s = 0; s < t.nst; ++s) {
                    if (!warp_wait_bar(P, S, &S.empty()[rp], rph ^ 1, 0, i, opc)) {
                        stop = true;
                        break;
                    }
                    if (lane == 0) {
                        if (FL == FL_TC) tc_load_stage(t, s, S.pages() + (size_t)rp * PS, &S.full()[rp], pol);
                        else gt_load_stage(g, s, S.pages() + (size_t)rp * PS, &S.full()[rp], pol);
                    }
                    __syncwarp();
                    ++ring;
                    if (++rp == (uint32_t)NP) {
                        rp = 0;
                        rph ^= 1;
                    }
                }
                if (P.trace && lane == 0) P.trace[((size_t)blockIdx.x * P.lmax + i) * 16 + 5] = gtimer();
                if (stop) goto drain;
                continue;
            }
        }
        // the instruction's weight or K/V rows into pages (false: stop)
        auto stream = [&](int i, int opc) -> bool {
            if (opc == MK_OP_ATTN && I.step > P.step) {
                // K/V rows appended by an earlier step of this launch: their writer
                // published them with the layer's attention event of that step --
                // acquire it (long since met) before the bulk copies read the rows
                const int pos0 = attn_pos(P, I) - (I.step - P.step);  // first position appended in this launch
                if (F(I, P_T0) + attn_cached_rows(I, attn_pos(P, I)) > pos0) {
                    const int ev = F(I, W_SIG);
                    const uint32_t target = (uint32_t)F(I, P_ATHR) * (uint32_t)I.step;
                    if (!warp_wait_counter(P, S, ev, target, i, opc)) return false;
                    fence_proxy_async_global();
                }
            }
            Seg s0, s1;
            const int nseg = describe<FL>(P, I, s0, s1);
            // MLP-up pages: groups of 8 gate + 8 up rows (bf16), 16 + 16 (FP8 rows, 32 to a page)
            const int upg = FL == FL_W8 && F(I, P_W8) != 0 ? W8_ROWS / 2 : 8;
            if (P.trace && lane == 0) P.trace[((size_t)blockIdx.x * P.lmax + i) * 16 + 4] = gtimer();
            // Rows go to pages in order, as many whole rows per page as fit.  The
            // two segments of an MLP-up tile share pages in groups of up to 8:
            // gate rows 8g .. 8g + 7, then the same up rows (a tile of n <= 8
            // gate rows is one group: its gate rows, then its up rows).  Attention
            // keeps its K rows and its V rows on separate pages.
            const int row_bytes = nseg > 0 ? s0.row_bytes : 0;
            const int rpp = row_bytes > 0 ? PS / row_bytes : 0;
            if (nseg > 0 && (rpp < 1 || (nseg > 1 && s1.row_bytes != row_bytes))) {
                if (lane == 0) raise_error(P, S, MK_ERR_DEVICE_CHECK, i, -1, 0, 0, opc, 0);
                return false;
            }
            // lane 0: copy rows [r, r + n) of a segment to dst
            auto copy_rows = [&](const Seg &sg, int r, int n, uint8_t *dst, uint64_t *bar) {
                const uint8_t *src = sg.src + (long long)r * sg.stride;
                if (sg.stride == sg.row_bytes) {
                    bulk_g2s(dst, src, (uint32_t)n * row_bytes, bar, pol);
                } else {
                    for (int j = 0; j < n; ++j)
                        bulk_g2s(dst + (size_t)j * row_bytes, src + (long long)j * sg.stride, row_bytes, bar, pol);
                }
            };
            const bool packed = opc != MK_OP_ATTN;
            const int n0 = nseg > 0 ? s0.rows : 0, n1 = nseg > 1 ? s1.rows : 0;
            // pages: packed -> over the concatenated rows; attention -> a fixed
            // number per segment (sized for the split's T rows, filled with the
            // rows cached so far)
            const int total = packed ? n0 + n1 : 0;
            const int npg0 = packed ? 0 : attn_pages(F(I, P_T), P.D, PS);
            const int npages = packed ? (total + rpp - 1) / (rpp > 0 ? rpp : 1) : 2 * npg0;
            bool stop = false;
            for (int k = 0; k < npages; ++k) {
                if (!warp_wait_bar(P, S, &S.empty()[rp], rph ^ 1, 0, i, opc)) {
                    stop = true;
                    break;
                }
                if (lane == 0) {
                    uint8_t *dst = S.pages() + (size_t)rp * PS;
                    uint64_t *bar = &S.full()[rp];
                    if (packed) {
                        const int r = k * rpp, nr = min(rpp, total - r);
                        mbar_expect_tx(bar, (uint32_t)nr * row_bytes);
                        if (nseg == 1) {
                            copy_rows(s0, r, nr, dst, bar);
                        } else {
                            const int gs = min(upg, n0);  // group size; n0 is a multiple of it when above it
                            for (int j = r; j < r + nr;) {
                                const int g = j / (2 * gs), w = j % (2 * gs);
                                const bool up = w >= gs;
                                const int run = min(r + nr - j, gs - (up ? w - gs : w));
                                copy_rows(up ? s1 : s0, g * gs + (up ? w - gs : w), run, dst + (size_t)(j - r) * row_bytes, bar);
                                j += run;
                            }
                        }
                    } else {
                        const bool second = k >= npg0;
                        const Seg &sg = second ? s1 : s0;
                        const int r = (second ? k - npg0 : k) * rpp, nr = max(0, min(rpp, sg.rows - r));
                        mbar_expect_tx(bar, (uint32_t)nr * row_bytes);  // an empty page just completes
                        if (nr > 0) copy_rows(sg, r, nr, dst, bar);
                    }
                }
                __syncwarp();
                ++ring;
                if (++rp == (uint32_t)NP) {
                    rp = 0;
                    rph ^= 1;
                }
            }

            if (P.trace && lane == 0) P.trace[((size_t)blockIdx.x * P.lmax + i) * 16 + 5] = gtimer();
            return !stop;
        };
        if (POOLS && opc == MK_OP_ATTN_POOL) {
            // claim the layer's attention tasks one by one (longest first) until none is left
            const int layer = F(I, P_LAYER), n = F(I, P_PT), base = F(I, P_TBASE);
            uint32_t *claim = P.claims + (size_t)I.step * P.L + layer;
            for (;;) {
                int idx = 0;
                if (lane == 0) idx = (int)atomicAdd(claim, 1u);
                idx = __shfl_sync(FULL, idx, 0);
                const int v = idx < n ? idx : -1;
                if (!post_claim(P, S, cseq++, v, i, opc)) goto drain;
                if (v < 0) break;
                I.w = attn_table_word(P, base + v);
                if (!ins_valid<FL>(P, I)) {
                    if (lane == 0) raise_error(P, S, MK_ERR_DEVICE_CHECK, i, -1, 0, 0, MK_OP_ATTN, 0);
                    goto drain;
                }
                if (!stream(i, MK_OP_ATTN)) goto drain;
            }
            continue;
        }
        if (!stream(i, opc)) goto drain;
    }
drain:
    // no bulk copy may still target this CTA's shared memory when it exits
    if (lane == 0) {
        const uint32_t first = ring > (uint32_t)NP ? ring - NP : 0;
        const uint64_t t0 = gtimer();
        for (uint32_t k = first; k < ring; ++k) {
            const uint32_t p = k % NP, use = k / NP;
            while (!mbar_test(&S.full()[p], use & 1)) {
                if (gtimer() - t0 > 2 * P.timeout_ns) break;  // copies of valid memory land in microseconds
            }
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------- activation-loader warp
template <int MAXB, int FL>
DEV void aloader_role(const KParams &P, const Smem S, const int32_t *myq) {
    constexpr bool GLM = fl_glm(FL);
    const int lane = threadIdx.x & 31;
    const bool two_bufs = P.abuf_count > 1;
    long long key0 = -1, key1 = -1;   // what each activation buffer holds: op row << 32 | first column
    bool ab = false;
    Rope<64> rope64;
    Rope<128> rope128;
    int seen_ev = -1;           // last event seen satisfied, and the target it met
    uint32_t seen_target = 0;
    uint32_t hs = 0;            // activation hand-offs so far; hand-off h uses activation slot h % 2
    HandoffChain chain;
    uint32_t xq = 0;            // tensor-core plans: activation stages (GLM: tiles) staged so far
    int cseq = 0;               // attention-pool claims taken so far
    WIns I;
    fetch_init(I, P, myq);
    // the instruction's event waits (acquire), right before its activation is read
    auto wait_events = [&](int i, int opc) {
        const int cnt = F(I, W_CNT);
        for (int w = 0; w < (cnt & 0xff) && !ab; ++w) {
            const uint32_t ew = (uint32_t)F(I, W_WAIT + 2 * w);
            const uint32_t thr = (uint32_t)F(I, W_WAIT + 2 * w + 1);
            const int ev = (int)(ew & ~WAIT_PREV_EPOCH);
            const int epoch = I.step + 1 - ((ew & WAIT_PREV_EPOCH) ? 1 : 0);
            const uint32_t target = thr * (uint32_t)epoch;
            // counters only grow within a launch: a target already met needs no new round trip
            if (target > 0 && !(ev == seen_ev && target <= seen_target)) {
                ab = !warp_wait_counter(P, S, ev, target, i, opc);
                seen_ev = ev;
                seen_target = target;
            }
        }
        if (!ab && lane == 0 && P.trace) P.trace[((size_t)blockIdx.x * P.lmax + i) * 16 + 2] = gtimer();
    };
    for (I.step = P.step; I.step < P.step + P.nsteps; ++I.step)
    for (int i = 0; i < P.lmax; ++i) {
        if (i == 0) {  // a new step: nothing staged so far holds this step's activations
            key0 = key1 = -1;
            chain.valid = false;
        }
        fetch(I, P, myq, i);
        const int opc = F(I, W_OPC);
        if (opc == MK_OP_NOOP) continue;
        if constexpr (FL == FL_TC) {
            if (is_gemv_op(opc)) {  // tensor-core tile: no slot hand-off, the input streams into the activation ring
                if (!ab && !ins_valid<FL>(P, I)) {
                    if (lane == 0) raise_error(P, S, MK_ERR_DEVICE_CHECK, i, -1, 0, 0, opc, 1);
                    ab = true;
                }
                wait_events(i, opc);
                tc_stage_x(P, S, I, i, xq, ab);
                if (lane == 0 && P.trace) P.trace[((size_t)blockIdx.x * P.lmax + i) * 16 + 11] = gtimer();
                continue;
            }
        }
        if constexpr (FL == FL_GLMTC) {
            if (opc == MK_OP_GLM_GEMM) {  // tensor-core tile: no slot hand-off, its input goes to an activation slot
                if (!ab && !ins_valid<FL>(P, I)) {
                    if (lane == 0) raise_error(P, S, MK_ERR_DEVICE_CHECK, i, -1, 0, 0, opc, 1);
                    ab = true;
                }
                wait_events(i, opc);
                gt_stage_x(P, S, I, i, xq, ab);
                if (lane == 0 && P.trace) P.trace[((size_t)blockIdx.x * P.lmax + i) * 16 + 11] = gtimer();
                continue;
            }
        }
        if (fl_pools(FL, MAXB) && opc == MK_OP_ATTN_POOL) {
            // the pool's wait (the layer's QKV), then each claimed task's hand-off, as an attention slot's
            if (!ab && !ins_valid<FL>(P, I)) {
                if (lane == 0) raise_error(P, S, MK_ERR_DEVICE_CHECK, i, -1, 0, 0, opc, 1);
                ab = true;
            }
            wait_events(i, opc);
            const int base = F(I, P_TBASE);
            for (;;) {
                int v = -1;
                if (!ab) ab = !read_claim(P, S, cseq++, 0, v, i, opc);
                if (ab || v < 0) break;
                I.w = attn_table_word(P, base + v);
                const int sl = hs & 1;
                const uint32_t use = hs >> 1;
                if (!ab) ab = !warp_wait_bar(P, S, &S.act_empty()[sl], (use & 1) ^ 1, 1, i, MK_OP_ATTN);
                float *slot = reinterpret_cast<float *>(S.act(sl));
                const bool g4 = P.Hq <= 4 * P.Hkv;
                if (FL == FL_LEAN || FL == FL_W8 || P.D == 64)
                    g4 ? stage_attn<64, 4>(P, I, slot, ab, rope64) : stage_attn<64, 8>(P, I, slot, ab, rope64);
                else g4 ? stage_attn<128, 4>(P, I, slot, ab, rope128) : stage_attn<128, 8>(P, I, slot, ab, rope128);
                key0 = key1 = -1;
                __syncwarp();
                if (lane == 0) {
                    S.ctrl()[1 + sl] = SLOT_FRESH;
                    mbar_arrive(&S.act_full()[sl]);
                }
                ++hs;
            }
            chain.valid = false;
            continue;
        }
        if (!needs_handoff<FL>(P, I, decode(I), chain)) continue;  // same input as the previous slot: nothing to stage
        const int sl = hs & 1;
        const uint32_t use = hs >> 1;
        if (!ab && !ins_valid<FL>(P, I)) {
            if (lane == 0) raise_error(P, S, MK_ERR_DEVICE_CHECK, i, -1, 0, 0, opc, 1);
            ab = true;
        }
        if (!ab) ab = !warp_wait_bar(P, S, &S.act_empty()[sl], (use & 1) ^ 1, 1, i, opc);
        wait_events(i, opc);
        float *slot = reinterpret_cast<float *>(S.act(sl));
        int flags = 0;
        uint32_t tx = 0;  // bytes of bulk copies completing on the slot's full barrier
        if (GLM) {
            if (FL == FL_GLM && opc == MK_OP_GLM_GEMM) {
                // the tile's activation rows by bulk copies, unless the buffer
                // already holds them (key: the input's device address)
                const long long key = (long long)PTR(I, S_GG_XQ);
                if (key != key0) {
                    if (hs > 0 && !ab)
                        ab = !warp_wait_bar(P, S, &S.act_empty()[(hs - 1) & 1], ((hs - 1) >> 1) & 1, 1, i, opc);
                    if (!ab) tx = stage_glm(P, I, reinterpret_cast<uint8_t *>(S.abuf(0)), &S.act_full()[sl]);
                    key0 = ab ? -1 : key;
                }
            }
        } else if (opc == MK_OP_ATTN) {
            const bool g4 = P.Hq <= 4 * P.Hkv;
            if (FL == FL_LEAN || FL == FL_W8 || P.D == 64)
                g4 ? stage_attn<64, 4>(P, I, slot, ab, rope64) : stage_attn<64, 8>(P, I, slot, ab, rope64);
            else g4 ? stage_attn<128, 4>(P, I, slot, ab, rope128) : stage_attn<128, 8>(P, I, slot, ab, rope128);
            flags = SLOT_FRESH;
            key0 = key1 = -1;
        } else if (FL != FL_TC && opc >= MK_OP_QKV && opc <= MK_OP_LM) {
            // two buffers: buffer sl was last read by instruction i - 2, whose
            // slot release was awaited above; one buffer: instruction i - 1
            // may still read it
            const int bi = two_bufs ? sl : 0;
            // batch-1 row-per-warp tiles read x lane-interleaved (rpw_perm4);
            // the layout is part of what a buffer holds
            const Dec dd = decode(I);
            const bool perm8 = FL == FL_W8 && F(I, P_W8) != 0;  // FP8 tiles' order (their instance only)
            const bool perm = !perm8 && MAXB == 1 && (rpw_tile(P, dd) || (FL != FL_LEAN && FL != FL_W8 && rpw_wide_tile(P, dd)));
            const long long key = ((long long)F(I, W_ROW) << 32) | (uint32_t)F(I, P_K0) | ((long long)perm << 62) |
                                  ((long long)perm8 << 61);
            if (key != (bi ? key1 : key0) || F(I, P_SNAP) > 0) {
                if (!two_bufs && hs > 0 && !ab)
                    ab = !warp_wait_bar(P, S, &S.act_empty()[(hs - 1) & 1], ((hs - 1) >> 1) & 1, 1, i, opc);
                // batch 1: the O tile's residual rows load in the same round trip as x
                const float rv = MAXB == 1 && opc == MK_OP_O ? resid_load1(I) : 0.f;
                stage_gemv<MAXB, FL == FL_W8>(P, I, S.abuf(bi), ab, perm, perm8);
                flags = SLOT_FRESH;
                if (opc == MK_OP_O) {
                    if (MAXB == 1) resid_store1(P, slot, rv);
                    else stage_resid(P, I, slot);
                }
            } else if (opc == MK_OP_O) {
                stage_resid(P, I, slot);
            }
            if (bi) key1 = key;
            else key0 = key;
        } else {
            key0 = key1 = -1;
        }
        __syncwarp();
        if (lane == 0 && P.trace) P.trace[((size_t)blockIdx.x * P.lmax + i) * 16 + 11] = gtimer();
        if (lane == 0) {
            S.ctrl()[1 + sl] = flags;
            if (tx == 0) mbar_arrive(&S.act_full()[sl]);  // (else stage_glm's arrive.expect_tx was the arrival)
        }
        ++hs;
    }
}

// ---------------------------------------------------------------- consumer warps
// Publisher warp.  Every consumer warp posts how many queue slots it has
// finished (a CTA-scope release store when it wrote global memory in the
// slot, else a relaxed one).  Lane 0 of the publisher polls the 8 counters
// with two vector loads; their minimum says every instruction below it is
// fully written back.  A CTA-scope fence turns the polls into acquires, and
// the batch's signals are added to the event counters with release adds
// (cumulative over what the publisher acquired) -- so consumers never wait
// for a GPU-scope fence.
DEV int progress_min(const Smem S) {
    int4 a, b;
    const uint32_t p = saddr((const void *)(S.ctrl() + 8));
    asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w) : "r"(p) : "memory");
    asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w) : "r"(p + 16) : "memory");
    return min(min(min(a.x, a.y), min(a.z, a.w)), min(min(b.x, b.y), min(b.z, b.w)));
}

DEV void publisher_role(const KParams &P, const Smem S, const int32_t *myq) {
    const int lane = threadIdx.x & 31;
    const int total = P.lmax * P.nsteps;
    int next = 0, ni = 0;  // first slot not yet published (launch-wide) and its in-step index
    int wc = queue_word(myq, 0, total > 0), wn = queue_word(myq, slot_ahead(P, 0, 1), total > 1);  // slots next, next + 1
    while (next < total) {
        if (__shfl_sync(FULL, wc, W_OPC) == MK_OP_NOOP) {
            // NoOps only pad the tail of a step's queue: go on at the next step's first slot
            next += P.lmax - ni;
            ni = 0;
            wc = queue_word(myq, 0, next < total);
            wn = queue_word(myq, slot_ahead(P, 0, 1), next + 1 < total);
            continue;
        }
        int done = next, ab = 0, stop = 0;
        uint64_t seen_at = 0;
        if (lane == 0) {
            uint64_t t0 = 0;
            for (uint32_t it = 0;; ++it) {
                done = progress_min(S);
                ab = S.ctrl()[0] != 0;
                if (done > next || ab) break;
                if ((it & 63) == 63) {
                    const uint64_t now = gtimer();
                    if (t0 == 0) t0 = now;
                    if (aborted(P, S)) { stop = 1; break; }
                    if (now - t0 > P.timeout_ns) {
                        raise_error(P, S, MK_ERR_TIMEOUT, next, -1, (uint32_t)done, (uint32_t)next + 1, -1, 4);
                        stop = 1;
                        break;
                    }
                }
            }
            // the CTA-scope fence makes the polls acquires of the consumers'
            // releases; the release adds below then carry their writes to GPU
            // scope (release is cumulative)
            if (!stop && !ab) fence_acq_rel_cta();
            seen_at = P.trace ? gtimer() : 0;
        }
        done = __shfl_sync(FULL, done, 0);
        ab = __shfl_sync(FULL, ab, 0);
        if (__shfl_sync(FULL, stop, 0)) break;
        for (; next < done; ++next) {
            const int cnt = __shfl_sync(FULL, wc, W_CNT), ns = (cnt >> 8) & 0xff;
            const int e0 = __shfl_sync(FULL, wc, W_SIG), i0 = __shfl_sync(FULL, wc, W_SIG + 1);
            const int e1 = __shfl_sync(FULL, wc, W_SIG + 2), i1 = __shfl_sync(FULL, wc, W_SIG + 3);
            if (lane == 0 && !ab) {
                if (ns > 0) red_release_add(P.counters + e0, (uint32_t)i0);
                if (ns > 1) red_release_add(P.counters + e1, (uint32_t)i1);
                if (P.trace) {  // (a slot's stamps: its last step's)
                    const size_t e = ((size_t)blockIdx.x * P.lmax + ni) * 16;
                    P.trace[e + 15] = seen_at;   // seen finished
                    P.trace[e + 14] = gtimer();  // published
                }
            }
            wc = wn;
            wn = queue_word(myq, slot_ahead(P, ni, 2), next + 2 < total);
            ni = ni + 1 == P.lmax ? 0 : ni + 1;
        }
    }
}

// A consumer warp records that queue slot i is finished.
DEV void handoff_progress(const Smem S, int i, bool wrote_global) {
    __syncwarp();
    const int warp = (threadIdx.x >> 5) - FIRST_CONSUMER_WARP;
    if ((threadIdx.x & 31) == 0) {
        if (wrote_global) st_release_cta(&S.ctrl()[8 + warp], i + 1);
        else st_relaxed_cta(&S.ctrl()[8 + warp], i + 1);
    }
}

// GEMV variants: K chunks per consumer thread (NCH) x one page or several.
// One-page tiles compute RPP rows unconditionally, RPP the power of two at or
// above the tile's rows, as long as RPP rows fit the page.
template <int MAXB, int NCH>
DEV bool gemv_geom(const KParams &P, const Smem S, const WIns &I, int i, int sl, const float *slot, uint32_t &ring,
                   RingPos &rq, uint32_t &ured, unsigned long long &lm_best, bool &ab) {
    constexpr int RMAX = rows_max<MAXB>();
    const int total = (F(I, W_OPC) == MK_OP_UP ? 2 : 1) * F(I, P_NROWS), row_bytes = 2 * F(I, P_KC);
    if (F(I, P_NPG) == 1) {
        if (total > 8 && RMAX * row_bytes <= P.page_bytes)
            return gemv_tile<MAXB, NCH, RMAX, true>(P, S, I, i, sl, slot, ring, rq, ured, lm_best, ab);
        if (total > 4 && total <= 8 && 8 * row_bytes <= P.page_bytes)
            return gemv_tile<MAXB, NCH, 8, true>(P, S, I, i, sl, slot, ring, rq, ured, lm_best, ab);
        if (total <= 4 && 4 * row_bytes <= P.page_bytes)
            return gemv_tile<MAXB, NCH, 4, true>(P, S, I, i, sl, slot, ring, rq, ured, lm_best, ab);
    }
    return gemv_tile<MAXB, NCH, RMAX, false>(P, S, I, i, sl, slot, ring, rq, ured, lm_best, ab);
}
template <int MAXB>
DEV bool gemv_dispatch(const KParams &P, const Smem S, const WIns &I, int i, int sl, const float *slot, uint32_t &ring,
                       RingPos &rq, uint32_t &ured, unsigned long long &lm_best, bool &ab) {
    if (mma_tile(P, I)) return gemv_mma_tile<MAXB>(P, S, I, i, sl, slot, ring, rq, ured, lm_best, ab);
    const int nch = ((F(I, P_KC) >> 3) + CONSUMERS - 1) / CONSUMERS;
    constexpr int NCHMAX = MAXB >= 8 ? 1 : (MAXB >= 4 ? 2 : 4);
    if (nch <= 1) return gemv_geom<MAXB, 1>(P, S, I, i, sl, slot, ring, rq, ured, lm_best, ab);
    if constexpr (NCHMAX >= 2) {
        if (nch <= 2) return gemv_geom<MAXB, 2>(P, S, I, i, sl, slot, ring, rq, ured, lm_best, ab);
        if constexpr (NCHMAX >= 4) {
            if (nch <= 4) return gemv_geom<MAXB, 4>(P, S, I, i, sl, slot, ring, rq, ured, lm_best, ab);
            if constexpr (NCHMAX >= 8) return gemv_geom<MAXB, 8>(P, S, I, i, sl, slot, ring, rq, ured, lm_best, ab);
        }
    }
    return false;
}

template <int MAXB, int FL>
DEV void consumer_role(const KParams &P, const Smem S, const int32_t *myq) {
    constexpr bool GLM = fl_glm(FL);
    const int ct = threadIdx.x - CONSUMER_BASE, lane = ct & 31;
    uint32_t ring = 0, cph = 0, ured = 0;
    uint32_t hs = 0;  // activation hand-offs so far (the activation loader counts the same ones)
    HandoffChain chain;
    XRow x;           // batch-1 row-per-warp activation, kept across tiles with the same input
    RingPos rq;       // ring position of the next page (kept in step with ring)
    bool ab = false;
    unsigned long long lm_best = 0;
    TcState tc;       // tensor-core plans: tiles and activation stages so far
    int cseq = 0;     // attention-pool claims taken so far
    WIns I;
    fetch_init(I, P, myq);
    for (I.step = P.step; I.step < P.step + P.nsteps; ++I.step)
    for (int i = 0; i < P.lmax; ++i) {
        if (i == 0) {  // a new step: its own argmax, activations and hand-off chain
            lm_best = 0;
            x.key = -1;
            chain.valid = false;
        }
        fetch(I, P, myq, i);
        const Dec d = decode(I);
        const int opc = d.opc;
        if (opc == MK_OP_NOOP) continue;
        uint64_t t_start = 0;
        if (ct == 0 && P.trace) t_start = gtimer();
        if (fl_pools(FL, MAXB) && opc == MK_OP_ATTN_POOL) {
            // every task the loader claimed for this pool, each with its hand-off, as an attention slot
            const int base = F(I, P_TBASE), cw = ct >> 5;
            for (;;) {
                int v = -1;
                const int seq = cseq++;
                if (!ab) ab = !read_claim(P, S, seq, 1 + cw, v, i, opc);
                if (!ab && v < 0) {
                    // the pool is done here only once its waits are met: the activation loader takes
                    // this last claim after them (an empty pool has no hand-off to order it)
                    ab = !warp_wait_smem(P, S, S.claims_taken(), (uint32_t)(seq + 1), i, opc);
                }
                if (ab || v < 0) break;
                I.w = attn_table_word(P, base + v);
                const int sl = hs & 1;
                if (!ab) ab = !warp_wait_bar(P, S, &S.act_full()[sl], (hs >> 1) & 1, 2, i, MK_OP_ATTN);
                const float *slot = reinterpret_cast<const float *>(S.act(sl));
                if (FL == FL_LEAN || FL == FL_W8 || P.D == 64) attn_task<64, FL>(P, S, I, i, sl, slot, ring, cph, ab);
                else attn_task<128, FL>(P, S, I, i, sl, slot, ring, cph, ab);
                rq.set(ring, P.num_pages);
                ++hs;
            }
            chain.valid = false;
            handoff_progress(S, launch_slot(P, I, i), true);
            if (ct == 0 && P.trace) {
                uint64_t *tr = P.trace + ((size_t)blockIdx.x * P.lmax + i) * 16;
                tr[0] = (uint64_t)opc | ((uint64_t)(uint32_t)d.task << 32);
                tr[1] = t_start;
                tr[3] = gtimer();
            }
            continue;
        }
        // tensor-core tiles take no slot hand-off (their input streams into the activation ring)
        const bool handoff =
            (FL == FL_TC && is_gemv_op(opc)) || (FL == FL_GLMTC && opc == MK_OP_GLM_GEMM) ? false
                                                                                         : needs_handoff<FL>(P, I, d, chain);
        const int sl = hs & 1;
        bool wrote = true;  // the warp wrote global memory in this slot
        if (handoff && !ab) ab = !warp_wait_bar(P, S, &S.act_full()[sl], (hs >> 1) & 1, 2, i, opc);
        if (P.trace && ct == 0) P.trace[((size_t)blockIdx.x * P.lmax + i) * 16 + 13] = gtimer();
        const float *slot = reinterpret_cast<const float *>(S.act(sl));
        if constexpr (GLM) {  // GLM-block plans hold only GLM ops and counters
            if (opc == MK_OP_GLM_GEMM) {
                if constexpr (FL == FL_GLMTC) {
                    wrote = glm_tc_tile(P, S, I, i, ring, tc, ab);
                } else {
                    if (d.nrows == 64) glm_gemm_task<64>(P, S, I, i, sl, ring, ured, ab);
                    else glm_gemm_task<16>(P, S, I, i, sl, ring, ured, ab);
                }
                rq.set(ring, P.num_pages);
            } else if (opc == MK_OP_GLM_A0 || opc == MK_OP_GLM_FIN) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.act_empty()[sl]);  // the slot holds nothing for these
                if (opc == MK_OP_GLM_A0) glm_a0_task(P, S, I, i, ured, ab);
                else glm_fin_task<FL == FL_GLMTC>(P, I, ab);
            } else {  // COUNTER: the slot handshake only
                consumer_sync(P, S, cph, ab, i);
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.act_empty()[sl]);
                wrote = false;
            }
        } else if (opc == MK_OP_ATTN) {
            if (FL == FL_LEAN || FL == FL_W8 || P.D == 64) attn_task<64, FL>(P, S, I, i, sl, slot, ring, cph, ab);
            else attn_task<128, FL>(P, S, I, i, sl, slot, ring, cph, ab);
            rq.set(ring, P.num_pages);
        } else if (FL == FL_TC && is_gemv_op(opc)) {
            wrote = tc_tile(P, S, I, d, i, ring, tc, lm_best, ab);
            rq.set(ring, P.num_pages);
        } else if (FL == FL_TC && opc == MK_OP_NORM) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.act_empty()[sl]);  // the slot holds nothing for it
            norm_task(P, S, I, ab);
        } else if (opc == MK_OP_EMBED) {
            consumer_sync(P, S, cph, ab, i);
            embed_task(P, S, I, i, sl, ab);
        } else if (FL == FL_W8 && opc >= MK_OP_QKV && F(I, P_W8) != 0) {
            if constexpr (FL == FL_W8) wrote = gemv_rpw8(P, S, I, d, i, handoff, sl, slot, x, ring, rq, ab);
        } else if (opc >= MK_OP_QKV) {
            if constexpr (FL != FL_TC) {  // (the tensor-core instance took its GEMV tiles above)
                if (MAXB == 1 && rpw_tile(P, d)) {  // (a constant condition for larger batches)
                    const int kg = d.kc >> 8;
                    if (kg <= 1) gemv_rpw<1>(P, S, d, i, handoff, sl, slot, x, ring, rq, lm_best, ab);
                    else if (kg <= 2) gemv_rpw<2>(P, S, d, i, handoff, sl, slot, x, ring, rq, lm_best, ab);
                    else if (kg <= 4) gemv_rpw<4>(P, S, d, i, handoff, sl, slot, x, ring, rq, lm_best, ab);
                    else gemv_rpw<8>(P, S, d, i, handoff, sl, slot, x, ring, rq, lm_best, ab);
                } else if constexpr (FL != FL_LEAN && FL != FL_W8) {
                    bool wide = false;
                    if constexpr (MAXB == 1) {
                        wide = rpw_wide_tile(P, d);
                        if (wide && d.npg <= 1) gemv_rpw_wide<1>(P, S, d, i, sl, slot, ring, rq, lm_best, ab);
                        else if (wide) gemv_rpw_wide<2>(P, S, d, i, sl, slot, ring, rq, lm_best, ab);
                    }
                    if (!wide) wrote = gemv_dispatch<MAXB>(P, S, I, i, sl, slot, ring, rq, ured, lm_best, ab);
                } else {  // the planner picks the lean instance only for plans without such tiles
                    if (lane == 0 && !ab) raise_error(P, S, MK_ERR_DEVICE_CHECK, i, -1, 0, 0, opc, 2);
                    ab = true;
                }
            }
        } else {  // COUNTER: the slot handshake only
            consumer_sync(P, S, cph, ab, i);
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.act_empty()[sl]);
            wrote = false;
        }
        if (handoff) ++hs;
        handoff_progress(S, launch_slot(P, I, i), wrote);
        if (ct == 0 && P.trace) {
            uint64_t *tr = P.trace + ((size_t)blockIdx.x * P.lmax + i) * 16;
            tr[0] = (uint64_t)opc | ((uint64_t)(uint32_t)d.task << 32);
            tr[1] = t_start;
            tr[3] = gtimer();
        }
    }
}

// ---------------------------------------------------------------- kernel
template <int MAXB, int FL>
__global__ void __launch_bounds__(THREADS, 1) mk_interp(const KParams P) {
    Smem S;
    S.o_abuf = 0;
    S.abuf_stride = P.abuf_count > 1 ? P.abuf_bytes : 0;
    S.o_act0 = P.abuf_count * P.abuf_bytes;
    S.act_stride = P.act_bytes;
    S.o_pages = S.o_act0 + 2 * P.act_bytes;
    S.o_aux = S.o_pages + P.num_pages * P.page_bytes;
    S.o_red0 = S.o_aux + P.aux_bytes - NRED * P.red_bytes;
    S.red_stride = P.red_bytes;
    S.o_bars = S.o_aux + P.aux_bytes;
    S.o_ctrl = S.o_bars + MBAR_BYTES;
    S.num_pages = P.num_pages;
    // tensor-core instances: the batched decoder's, the GLM block's with tcgen05 GEMM tiles
    constexpr bool TC = FL == FL_TC || FL == FL_GLMTC;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int p = 0; p < P.num_pages; ++p) {
            mbar_init(&S.full()[p], 1);
            // tensor-core plans: one arrival, the MMA commit of a weight
            // stage or the last of the 8 warps reading an attention page
            mbar_init(&S.empty()[p], TC ? 1 : CONSUMER_WARPS);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.act_full()[s], 1);
            mbar_init(&S.act_empty()[s], CONSUMER_WARPS);
        }
        mbar_init(S.cbar(), CONSUMER_WARPS);
        if (TC) {
            for (int s = 0; s < TC_XSLOTS; ++s) {
                mbar_init(&S.xfull()[s], 1);
                // GLM tiles: the MMA commit and the four epilogue warps (done with the slot's scales)
                mbar_init(&S.xempty()[s], FL == FL_GLMTC ? 1 + TC_EPI_WARPS : 1);
            }
            for (int a = 0; a < GT_NACC; ++a) {
                mbar_init(&S.accfull()[a], 1);
                mbar_init(&S.accempty()[a], TC_EPI_WARPS);
            }
            mbar_init(S.drain(), 1);
        }
        for (int k = 0; k < CTRL_WORDS; ++k)
            if (k != 31) S.ctrl()[k] = 0;  // (word 31 is the TMEM address, written by warp 3 meanwhile)
        if (TC) {
            for (int p = 0; p < P.num_pages; ++p) S.page_users()[p] = 0;
            // the swizzled stage buffers need 1024-byte alignment: refuse to run otherwise
            if ((saddr(mk_smem) & 1023u) != 0) raise_error(P, S, MK_ERR_DEVICE_CHECK, -1, -1, 0, 0, -1, 3);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    static_assert(GT_TMEM_COLS == TC_TMEM_COLS, "one TMEM allocation serves both tensor-core paths");
    if (TC && warp == 3) {  // the idle warp owns the TMEM accumulators
        tmem_alloc(S.tmem_slot(), TC_TMEM_COLS);
        tmem_relinquish();
    }
    if (TC) tc_fence_before();
    __syncthreads();
    if (TC) tc_fence_after();
    const int32_t *myq = P.queue + (size_t)blockIdx.x * P.lmax * W_WORDS;
    if (warp == 0) loader_role<MAXB, FL>(P, S, myq);
    else if (warp == 1) aloader_role<MAXB, FL>(P, S, myq);
    else if (warp == PUBLISHER_WARP) publisher_role(P, S, myq);
    else if (warp >= FIRST_CONSUMER_WARP) consumer_role<MAXB, FL>(P, S, myq);
    if (TC && warp == FIRST_CONSUMER_WARP + TC_MMA_WARP) {
        // every MMA this warp issued has completed before the accumulators are freed
        if ((threadIdx.x & 31) == 0) tc_commit(S.drain());
        __syncwarp();
        const uint64_t t0 = gtimer();
        while (!mbar_test(S.drain(), 0) && gtimer() - t0 < 2 * P.timeout_ns) {
        }
    }
    if (TC) tc_fence_before();
    __syncthreads();
    if (TC && warp == 3) {
        tc_fence_after();
        tmem_dealloc(*S.tmem_slot(), TC_TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side


constexpr int kMaxDevices = 64;

static int cuda_fail(cudaError_t e, const char *what) {
    return set_error(MK_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

int query_device(int *num_sms, int *smem_optin) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SMs)");
    e = cudaDeviceGetAttribute(smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(smem)");
    return MK_OK;
}

using KernelFn = void (*)(const KParams);

static KernelFn pick_kernel(const Plan &p) {
    if (p.kind == PLAN_GLM) return p.tc ? mk_interp<1, FL_GLMTC> : mk_interp<1, FL_GLM>;
    if (p.tc) return mk_interp<TC_MAXB, FL_TC>;
    const int B = p.B;
    if (p.w8) return mk_interp<1, FL_W8>;
    if (B <= 1) return p.lean ? mk_interp<1, FL_LEAN> : mk_interp<1, FL_GEN>;
    if (B <= 2) return mk_interp<2, FL_GEN>;
    if (B <= 4) return mk_interp<4, FL_GEN>;
    return mk_interp<8, FL_GEN>;
}

static int encode_map(CUtensorMap *m, uint64_t base, uint64_t cols, uint64_t rows, uint32_t box_rows,
                      bool bytes1);

// Operand rows of the GLM block plan, in the planner's op order: A0,
// QKV-A, Head-Gate, Indexer-K, FIN, Q-B, Indexer-Q.  Tensor-core plans also
// get the tensor maps: the five e4m3 weight matrices (boxes of 128 rows),
// then A0's and FIN's activation codes (boxes of the 16 token rows).
static int build_glm_table(Plan &p, uint8_t *ws, std::vector<uint64_t> &tab, std::vector<CUtensorMap> &maps) {
    for (int b = MK_BIND_GLM_X; b <= MK_BIND_GLM_INDEX; ++b)
        if (!p.bind[b][0]) {
            char buf[96];
            std::snprintf(buf, sizeof buf, "binding %d (GLM block) is not set", b);
            return set_error(MK_ERR_UNBOUND, buf);
        }
    auto B = [&](int b) { return p.bind[b][0]; };
    auto row = [&](int o) { return &tab[(size_t)o * N_SLOTS]; };
    uint64_t *r = row(0);
    r[S_GA_X] = B(MK_BIND_GLM_X); r[S_GA_RES] = B(MK_BIND_GLM_RES); r[S_GA_NORM] = B(MK_BIND_GLM_NORM);
    r[S_GA_RES_OUT] = B(MK_BIND_GLM_RES_OUT); r[S_GA_QA] = B(MK_BIND_GLM_QA); r[S_GA_SA] = B(MK_BIND_GLM_SA);
    auto gemm = [&](int o, int w, int sw, int xq, int xs, int out) {
        uint64_t *g = row(o);
        g[S_GG_W] = B(w); g[S_GG_SW] = B(sw); g[S_GG_XQ] = B(xq); g[S_GG_XS] = B(xs); g[S_GG_OUT] = B(out);
    };
    gemm(1, MK_BIND_GLM_W_QKVA, MK_BIND_GLM_S_QKVA, MK_BIND_GLM_QA, MK_BIND_GLM_SA, MK_BIND_GLM_QKVA);
    gemm(2, MK_BIND_GLM_W_GATE, MK_BIND_GLM_S_GATE, MK_BIND_GLM_QA, MK_BIND_GLM_SA, MK_BIND_GLM_GATE);
    gemm(3, MK_BIND_GLM_W_IK, MK_BIND_GLM_S_IK, MK_BIND_GLM_QA, MK_BIND_GLM_SA, MK_BIND_GLM_IK);
    r = row(4);
    r[S_GF_QKVA] = B(MK_BIND_GLM_QKVA); r[S_GF_IK] = B(MK_BIND_GLM_IK); r[S_GF_QB] = B(MK_BIND_GLM_QB);
    r[S_GF_SB] = B(MK_BIND_GLM_SB); r[S_GF_LAT] = B(MK_BIND_GLM_LATENT); r[S_GF_IDX] = B(MK_BIND_GLM_INDEX);
    gemm(5, MK_BIND_GLM_W_QB, MK_BIND_GLM_S_QB, MK_BIND_GLM_QB, MK_BIND_GLM_SB, MK_BIND_GLM_Q);
    gemm(6, MK_BIND_GLM_W_IQ, MK_BIND_GLM_S_IQ, MK_BIND_GLM_QB, MK_BIND_GLM_SB, MK_BIND_GLM_IQ);
    const uint64_t W = (uint64_t)(uintptr_t)ws;
    const uint64_t rope = W + p.ws.rope;
    for (int o : {1, 2, 3, 5, 6}) row(o)[S_GG_ROPE] = rope;
    row(4)[S_GF_ROPE] = rope;
    if (!p.tc) return MK_OK;
    const mk_glm_desc &g = p.glm;
    const int H = g.hidden, QL = g.q_lora, NQKVA = g.q_lora + g.kv_lora + g.rope;
    const struct { int op, bind; uint64_t rows, cols; } mats[5] = {
        {1, MK_BIND_GLM_W_QKVA, (uint64_t)NQKVA, (uint64_t)H},
        {2, MK_BIND_GLM_W_GATE, (uint64_t)g.gate_heads, (uint64_t)H},
        {3, MK_BIND_GLM_W_IK, (uint64_t)g.idx_dim, (uint64_t)H},
        {5, MK_BIND_GLM_W_QB, (uint64_t)g.q_heads * g.q_head_dim, (uint64_t)QL},
        {6, MK_BIND_GLM_W_IQ, (uint64_t)g.idx_heads * g.idx_dim, (uint64_t)QL},
    };
    maps.assign(GT_NTMAPS, CUtensorMap{});
    auto tmap = [&](int idx) { return W + p.ws.tmaps + (uint64_t)idx * sizeof(CUtensorMap); };
    for (int k = 0; k < 5; ++k) {
        if (int rc = encode_map(&maps[k], B(mats[k].bind), mats[k].cols, mats[k].rows, GT_M, true)) return rc;
        row(mats[k].op)[S_GG_TW] = tmap(k);
        row(mats[k].op)[S_GG_TX] = tmap(mats[k].op <= 3 ? 5 : 6);
    }
    if (int rc = encode_map(&maps[5], B(MK_BIND_GLM_QA), H, GT_N, GT_N, true)) return rc;
    if (int rc = encode_map(&maps[6], B(MK_BIND_GLM_QB), QL, GT_N, GT_N, true)) return rc;
    for (int k = 0; k < 3; ++k) row(1 + k)[S_GG_FSUM] = W + p.ws.gsum[k];
    // FIN rounds the sums: QKV-A (op 1) and Indexer-K (op 3) into their bf16
    // outputs, Head-Gate (op 2) into its own
    r = row(4);
    r[S_GF_FQKVA] = W + p.ws.gsum[0]; r[S_GF_FGATE] = W + p.ws.gsum[1]; r[S_GF_FIK] = W + p.ws.gsum[2];
    r[S_GF_GATE] = B(MK_BIND_GLM_GATE);
    return MK_OK;
}

// ---- tensor maps of the tensor-core plans --------------------------------
// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
static_assert(sizeof(CUtensorMap) == 128, "tensor maps are 128-byte records");
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A row-major matrix [rows, cols] of bf16 (or, `bytes1`, of 1-byte e4m3
// codes) read in boxes of 128 bytes of a row (64 bf16 / 128 codes) x
// box_rows rows, landing 128-byte swizzled (the tiles' K-major layout).
// Rows past the end read as zeros.
static int encode_map(CUtensorMap *m, uint64_t base, uint64_t cols, uint64_t rows, uint32_t box_rows,
                      bool bytes1 = false) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return set_error(MK_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * (bytes1 ? 1 : 2)};
    const cuuint32_t box[2] = {(cuuint32_t)(bytes1 ? GT_KS : TC_BOX), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, bytes1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                           reinterpret_cast<void *>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[120];
        std::snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for a %llu x %llu matrix", (int)r,
                      (unsigned long long)rows, (unsigned long long)cols);
        return set_error(MK_ERR_CUDA, buf);
    }
    return MK_OK;
}

// Tensor maps, in the workspace's map table order: the three activations
// (normalised x, attention output, MLP activation; 2 np rows each), then per
// layer Wq, Wk, Wv, Wo, Wg, Wu, Wd, then the LM head.
static int build_tc_maps(Plan &p, uint8_t *ws, std::vector<CUtensorMap> &maps) {
    const mk_model_desc &m = p.model;
    const int L = m.layers, H = m.hidden, QD = m.q_heads * m.head_dim, KD = m.kv_heads * m.head_dim, F = m.ffn;
    maps.assign(TC_NTMAPS_FIXED + TC_WMAPS_PER_LAYER * L + 1, CUtensorMap{});
    const uint64_t W = (uint64_t)(uintptr_t)ws;
    const uint32_t xr = 2 * p.np;
    int rc = encode_map(&maps[0], W + p.ws.xn, H, xr, xr);
    if (!rc) rc = encode_map(&maps[1], W + p.ws.xo, QD, xr, xr);
    if (!rc) rc = encode_map(&maps[2], W + p.ws.act16, F, xr, xr);
    for (int l = 0; l < L && !rc; ++l) {
        CUtensorMap *t = &maps[TC_NTMAPS_FIXED + TC_WMAPS_PER_LAYER * l];
        rc = encode_map(t + 0, p.bind[MK_BIND_WQ][l], H, QD, TC_SEG);
        if (!rc) rc = encode_map(t + 1, p.bind[MK_BIND_WK][l], H, KD, TC_SEG);
        if (!rc) rc = encode_map(t + 2, p.bind[MK_BIND_WV][l], H, KD, TC_SEG);
        if (!rc) rc = encode_map(t + 3, p.bind[MK_BIND_WO][l], QD, H, TC_SEG);
        if (!rc) rc = encode_map(t + 4, p.bind[MK_BIND_WG][l], H, F, TC_SEG);
        if (!rc) rc = encode_map(t + 5, p.bind[MK_BIND_WU][l], H, F, TC_SEG);
        if (!rc) rc = encode_map(t + 6, p.bind[MK_BIND_WD][l], F, H, TC_SEG);
    }
    if (!rc) rc = encode_map(&maps.back(), p.bind[MK_BIND_LM_HEAD][0], H, m.vocab, TC_SEG);
    return rc;
}

static int build_table(Plan &p, uint8_t *ws, std::vector<uint64_t> &tab, std::vector<CUtensorMap> &maps) {
    tab.assign((size_t)p.num_ops * N_SLOTS, 0);
    if (p.kind == PLAN_GLM) return build_glm_table(p, ws, tab, maps);
    if (p.kind != PLAN_LLAMA) return MK_OK;
    const mk_model_desc &m = p.model;
    const int L = m.layers, B = p.B, Hkv = m.kv_heads, D = m.head_dim;
    auto need = [&](int bind, int layer) -> int {
        if (!p.bind[bind][layer]) {
            char buf[96];
            std::snprintf(buf, sizeof buf, "binding %d (layer %d) is not set", bind, layer);
            return set_error(MK_ERR_UNBOUND, buf);
        }
        return MK_OK;
    };
    for (int b : {MK_BIND_EMBED, MK_BIND_LM_HEAD, MK_BIND_NORM_FINAL, MK_BIND_KCACHE, MK_BIND_VCACHE, MK_BIND_TOKENS,
                  MK_BIND_LOGITS, MK_BIND_ARGMAX})
        if (int rc = need(b, 0)) return rc;
    if (p.capture)
        if (int rc = need(MK_BIND_HIDDEN, 0)) return rc;
    for (int l = 0; l < L; ++l) {
        for (int b : {MK_BIND_WQ, MK_BIND_WK, MK_BIND_WV, MK_BIND_WO, MK_BIND_WG, MK_BIND_WU, MK_BIND_WD,
                      MK_BIND_NORM_ATTN, MK_BIND_NORM_MLP})
            if (int rc = need(b, l)) return rc;
        if (p.w8)
            for (int b = MK_BIND_SQ; b <= MK_BIND_SD; ++b)
                if (int rc = need(b, l)) return rc;
        if (m.qk_norm)
            for (int b : {MK_BIND_QNORM, MK_BIND_KNORM})
                if (int rc = need(b, l)) return rc;
    }
    const uint64_t W = (uint64_t)(uintptr_t)ws;
    const uint64_t hres = W + p.ws.hres, hmid = W + p.ws.hmid, qkv = W + p.ws.qkv, part = W + p.ws.part,
                   aout = W + p.ws.attn_out, act = W + p.ws.act, arrive = W + p.ws.arrive, seq0 = W + p.ws.seq0;
    const uint64_t layer_cache = (uint64_t)B * Hkv * p.smax * D * 2;
    const uint64_t hist = p.bind[MK_BIND_HIDDEN][0];
    for (int o = 0; o < p.num_ops; ++o) {
        uint64_t *r = &tab[(size_t)o * N_SLOTS];
        const int l = p.op_layer[o];
        switch (p.op_kind[o]) {
        case MK_OP_EMBED:
            r[S_EMB_W] = p.bind[MK_BIND_EMBED][0]; r[S_EMB_H] = hres;
            r[S_EMB_TOK] = p.bind[MK_BIND_TOKENS][0]; r[S_EMB_KEYS] = p.bind[MK_BIND_ARGMAX][0];
            break;
        case MK_OP_QKV:
            r[S_QKV_WQ] = p.bind[MK_BIND_WQ][l]; r[S_QKV_WK] = p.bind[MK_BIND_WK][l]; r[S_QKV_WV] = p.bind[MK_BIND_WV][l];
            r[S_QKV_NORM] = p.bind[MK_BIND_NORM_ATTN][l]; r[S_QKV_H] = hres; r[S_QKV_OUT] = qkv; r[S_QKV_HIST] = hist;
            break;
        case MK_OP_ATTN:
        case MK_OP_ATTN_POOL:  // (its claimed tasks are attention instructions of this operand row)
            r[S_AT_K] = p.bind[MK_BIND_KCACHE][0] + (uint64_t)l * layer_cache;
            r[S_AT_V] = p.bind[MK_BIND_VCACHE][0] + (uint64_t)l * layer_cache;
            r[S_AT_QKV] = qkv;
            r[S_AT_QN] = m.qk_norm ? p.bind[MK_BIND_QNORM][l] : 0;
            r[S_AT_KN] = m.qk_norm ? p.bind[MK_BIND_KNORM][l] : 0;
            r[S_AT_PART] = part; r[S_AT_OUT] = aout; r[S_AT_ARRIVE] = arrive; r[S_AT_SEQ0] = seq0;
            break;
        case MK_OP_O:
            r[S_O_W] = p.bind[MK_BIND_WO][l]; r[S_O_IN] = aout; r[S_O_HRES] = hres; r[S_O_HMID] = hmid;
            break;
        case MK_OP_UP:
            r[S_UP_WG] = p.bind[MK_BIND_WG][l]; r[S_UP_WU] = p.bind[MK_BIND_WU][l];
            r[S_UP_NORM] = p.bind[MK_BIND_NORM_MLP][l]; r[S_UP_H] = hmid; r[S_UP_OUT] = act;
            break;
        case MK_OP_DOWN:
            r[S_DN_W] = p.bind[MK_BIND_WD][l]; r[S_DN_IN] = act; r[S_DN_HRES] = hres;
            break;
        case MK_OP_LM:
            r[S_LM_W] = p.bind[MK_BIND_LM_HEAD][0]; r[S_LM_NORM] = p.bind[MK_BIND_NORM_FINAL][0]; r[S_LM_H] = hres;
            r[S_LM_LOGITS] = p.bind[MK_BIND_LOGITS][0]; r[S_LM_KEYS] = p.bind[MK_BIND_ARGMAX][0];
            r[S_LM_HIST] = hist;
            break;
        default:
            break;
        }
        if (p.w8 && l >= 0) {  // FP8 projections: their block scales
            switch (p.op_kind[o]) {
            case MK_OP_QKV:
                r[S_W8_S0] = p.bind[MK_BIND_SQ][l]; r[S_W8_S1] = p.bind[MK_BIND_SK][l]; r[S_W8_S2] = p.bind[MK_BIND_SV][l];
                break;
            case MK_OP_O: r[S_W8_S0] = p.bind[MK_BIND_SO][l]; break;
            case MK_OP_UP: r[S_W8_S0] = p.bind[MK_BIND_SG][l]; r[S_W8_S1] = p.bind[MK_BIND_SU][l]; break;
            case MK_OP_DOWN: r[S_W8_S0] = p.bind[MK_BIND_SD][l]; break;
            default: break;
            }
        }
        switch (p.op_kind[o]) {
        case MK_OP_QKV: r[S_G_OUT] = r[S_QKV_OUT]; break;
        case MK_OP_O: r[S_G_OUT] = r[S_O_HRES]; r[S_G_OUT2] = r[S_O_HMID]; break;
        case MK_OP_UP: r[S_G_OUT] = r[S_UP_OUT]; break;
        case MK_OP_DOWN: r[S_G_OUT] = r[S_DN_HRES]; break;
        case MK_OP_LM: r[S_G_OUT] = r[S_LM_LOGITS]; r[S_G_OUT2] = r[S_LM_KEYS]; break;
        default: break;
        }
    }
    if (p.tc) {
        // tensor-core plans: the tiles' tensor maps and bf16 activation rows
        if (int rc = build_tc_maps(p, ws, maps)) return rc;
        auto tmap = [&](int idx) { return W + p.ws.tmaps + (uint64_t)idx * sizeof(CUtensorMap); };
        const uint64_t xn = W + p.ws.xn, xo = W + p.ws.xo, a16 = W + p.ws.act16;
        for (int o = 0; o < p.num_ops; ++o) {
            uint64_t *r = &tab[(size_t)o * N_SLOTS];
            const int l = p.op_layer[o];
            const int wl = TC_NTMAPS_FIXED + TC_WMAPS_PER_LAYER * std::max(l, 0);
            switch (p.op_kind[o]) {
            case MK_OP_NORM: {
                const int which = p.op_aux[o];
                r[S_N_H] = hres;
                r[S_N_W] = which == 0   ? p.bind[MK_BIND_NORM_ATTN][l]
                           : which == 1 ? p.bind[MK_BIND_NORM_MLP][l]
                                        : p.bind[MK_BIND_NORM_FINAL][0];
                r[S_N_XN] = xn; r[S_N_QKV] = qkv; r[S_N_HIST] = hist;
                break;
            }
            case MK_OP_QKV:
                r[S_T_W0] = tmap(wl + 0); r[S_T_W1] = tmap(wl + 1); r[S_T_W2] = tmap(wl + 2); r[S_T_X] = tmap(0);
                break;
            case MK_OP_ATTN:
            case MK_OP_ATTN_POOL: r[S_AT_OUT] = xo; break;
            case MK_OP_O: r[S_T_W0] = tmap(wl + 3); r[S_T_X] = tmap(1); r[S_G_OUT] = hres; break;
            case MK_OP_UP:
                r[S_T_W0] = tmap(wl + 4); r[S_T_W1] = tmap(wl + 5); r[S_T_X] = tmap(0); r[S_G_OUT] = a16;
                break;
            case MK_OP_DOWN: r[S_T_W0] = tmap(wl + 6); r[S_T_X] = tmap(2); r[S_G_OUT] = hres; break;
            case MK_OP_LM:
                r[S_T_W0] = tmap(TC_NTMAPS_FIXED + TC_WMAPS_PER_LAYER * p.model.layers); r[S_T_X] = tmap(0);
                break;
            default: break;
            }
        }
    }
    return MK_OK;
}

static KParams base_params(const Plan &p, uint8_t *ws) {
    KParams k{};
    k.optab = reinterpret_cast<const uint64_t *>(ws + p.ws.optab);
    k.counters = reinterpret_cast<uint32_t *>(ws + p.ws.counters);
    k.err = reinterpret_cast<uint32_t *>(ws + p.ws.err);
    k.num_ops = p.num_ops;
    k.num_events = (int)p.thresholds.size();
    k.num_pages = p.num_pages;
    k.page_bytes = p.page_bytes;
    k.act_bytes = p.act_bytes;
    k.abuf_bytes = p.abuf_bytes;
    k.abuf_count = p.abuf_count;
    k.aux_bytes = p.aux_bytes;
    k.red_bytes = p.red_bytes;
    k.smem_bytes = p.smem_bytes;
    const mk_model_desc &m = p.model;
    k.B = p.B;
    k.H = m.hidden; k.Hq = m.q_heads; k.Hkv = m.kv_heads > 0 ? m.kv_heads : 1; k.D = m.head_dim; k.F = m.ffn;
    k.V = m.vocab; k.L = m.layers; k.Smax = p.smax; k.qk_norm = m.qk_norm; k.nsplit_max = p.nsplit_max;
    k.np = p.tc ? p.np : 0;
    k.claims = p.attn_table.empty() ? nullptr : reinterpret_cast<uint32_t *>(ws + p.ws.claims);
    k.attn_table = p.attn_table.empty() ? nullptr : reinterpret_cast<const int32_t *>(ws + p.ws.atab);
    k.eps = m.eps;
    k.theta = m.rope_theta;
    if (p.kind == PLAN_GLM) {
        k.H = p.glm.hidden;
        k.eps = p.glm.eps;
        k.theta = p.glm.rope_theta;
    }
    return k;
}

}  // namespace mk

using namespace mk;

extern "C" {

int mk_run(mk_plan_t plan, void *workspace, size_t workspace_bytes, int first_step, int num_steps, uint32_t flags,
           uint64_t timeout_ns, void *stream_) {
    if (!plan || !workspace) return set_error(MK_ERR_INVALID, "null plan or workspace");
    Plan &p = plan->p;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (workspace_bytes < p.ws.total) return set_error(MK_ERR_INVALID, "workspace too small");
    if ((uintptr_t)workspace % 256) return set_error(MK_ERR_INVALID, "workspace must be 256-byte aligned");
    if (first_step < 0 || num_steps < 0 || (p.kind == PLAN_LLAMA && first_step + num_steps > p.max_steps))
        return set_error(MK_ERR_INVALID, "steps outside the planned range");
    const bool one_launch = (flags & MK_RUN_ONE_LAUNCH) != 0;
    if (one_launch && p.segments.size() != 1)
        return set_error(MK_ERR_INVALID, "MK_RUN_ONE_LAUNCH needs a megakernel plan");
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaError_t e;
    if (p.table_dirty || p.uploaded_ws != workspace) {
        std::vector<uint64_t> tab;
        std::vector<CUtensorMap> maps;
        if (int rc = build_table(p, ws, tab, maps)) return rc;
        e = cudaMemcpyAsync(ws + p.ws.optab, tab.data(), tab.size() * 8, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "upload operand table");
        if (!maps.empty()) {
            e = cudaMemcpyAsync(ws + p.ws.tmaps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice,
                                stream);
            if (e != cudaSuccess) return cuda_fail(e, "upload tensor maps");
        }
        if (p.uploaded_ws != workspace) {
            e = cudaMemcpyAsync(ws + p.ws.queue, p.words.data(), p.words.size() * 4, cudaMemcpyHostToDevice, stream);
            if (e != cudaSuccess) return cuda_fail(e, "upload queue");
            if (!p.seq0.empty()) {
                e = cudaMemcpyAsync(ws + p.ws.seq0, p.seq0.data(), p.seq0.size() * 4, cudaMemcpyHostToDevice, stream);
                if (e != cudaSuccess) return cuda_fail(e, "upload lengths");
            }
            if (!p.attn_table.empty()) {
                e = cudaMemcpyAsync(ws + p.ws.atab, p.attn_table.data(), p.attn_table.size() * 4,
                                    cudaMemcpyHostToDevice, stream);
                if (e != cudaSuccess) return cuda_fail(e, "upload attention task table");
            }
            if (!p.rope_tab.empty()) {
                e = cudaMemcpyAsync(ws + p.ws.rope, p.rope_tab.data(), p.rope_tab.size() * 4, cudaMemcpyHostToDevice,
                                    stream);
                if (e != cudaSuccess) return cuda_fail(e, "upload RoPE table");
            }
        }
        // the host images must stay valid until the copies ran
        e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return cuda_fail(e, "synchronise uploads");
        p.uploaded_ws = workspace;
        p.table_dirty = false;
    }
    if (first_step == 0) {
        e = cudaMemsetAsync(ws + p.ws.err, 0, p.ws.queue - p.ws.err, stream);  // error record, counters, arrivals
        if (e != cudaSuccess) return cuda_fail(e, "clear counters");
        if (p.kind == PLAN_LLAMA) {
            e = cudaMemsetAsync(reinterpret_cast<void *>(p.bind[MK_BIND_ARGMAX][0]), 0,
                                (size_t)p.max_steps * p.B * 8, stream);
            if (e != cudaSuccess) return cuda_fail(e, "clear argmax");
        }
    }
    KernelFn fn = pick_kernel(p);
    // the attribute is per device: remember what each device was given
    static thread_local int configured_smem[kMaxDevices] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(MK_ERR_INVALID, "device ordinal out of range");
    if (configured_smem[dev] < p.smem_bytes) {
        for (KernelFn f : {mk_interp<1, FL_GEN>, mk_interp<2, FL_GEN>, mk_interp<4, FL_GEN>, mk_interp<8, FL_GEN>,
                           mk_interp<1, FL_GLM>, mk_interp<1, FL_GLMTC>, mk_interp<1, FL_LEAN>,
                           mk_interp<1, FL_W8>, mk_interp<TC_MAXB, FL_TC>}) {
            e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        }
        configured_smem[dev] = p.smem_bytes;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, THREADS, p.smem_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    int sms = 0, smem_optin = 0;
    if (int rc = query_device(&sms, &smem_optin)) return rc;
    KParams k = base_params(p, ws);
    k.timeout_ns = timeout_ns ? timeout_ns : 200000000ull;
    k.flags = (int)flags;
    // one launch per step, or one launch for all of them
    const int launches = one_launch ? (num_steps > 0 ? 1 : 0) : num_steps;
    k.nsteps = one_launch ? num_steps : 1;
    for (int s = first_step; s < first_step + launches; ++s) {
        k.step = s;
        for (const Segment &seg : p.segments) {
            if (per_sm < 1 || seg.workers > per_sm * sms)
                return set_error(MK_ERR_RESIDENCY, "worker grid cannot be co-resident");
            k.queue = reinterpret_cast<const int32_t *>(ws + p.ws.queue) + seg.word_offset;
            k.lmax = seg.lmax;
            k.num_workers = seg.workers;
            k.trace = (flags & MK_RUN_TRACE) && p.segments.size() == 1
                          ? reinterpret_cast<uint64_t *>(ws + p.ws.trace)
                          : nullptr;
            void *args[] = {&k};
            e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(fn), dim3(seg.workers), dim3(THREADS), args,
                                            (size_t)p.smem_bytes, stream);
            if (e != cudaSuccess) return cuda_fail(e, "launch");
        }
    }
    return MK_OK;
}

// ---------------------------------------------------------------- launch probe
__global__ void __launch_bounds__(THREADS, 1) mk_empty() {}

int mk_launch_probe(int num_workers, int cooperative, void *stream) {
    if (num_workers <= 0) return set_error(MK_ERR_INVALID, "num_workers must be positive");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (cooperative) {
        void *args[] = {nullptr};
        e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(mk_empty), dim3(num_workers), dim3(THREADS),
                                        args, 0, st);
    } else {
        mk_empty<<<num_workers, THREADS, 0, st>>>();
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? MK_OK : cuda_fail(e, "probe launch");
}

// ---------------------------------------------------------------- allocation-free entry point
// The workspace of mk_run_static(): a fixed device array owned by this
// library.  Host code only ever sees the array's host-side stand-in; the
// device address comes from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) uint8_t g_static_workspace[MK_STATIC_WORKSPACE_BYTES];

namespace {
std::mutex g_static_mu;
void *g_static_addr[kMaxDevices] = {};      // device address of the array, per device
const void *g_static_owner[kMaxDevices] = {};  // plan whose queue the array holds
}  // namespace

int mk_run_static(mk_plan_t plan, int first_step, int num_steps, uint32_t flags, uint64_t timeout_ns, void *stream,
                  uint64_t *workspace_out) {
    if (!plan) return set_error(MK_ERR_INVALID, "null plan");
    if (plan->p.ws.total > MK_STATIC_WORKSPACE_BYTES) {
        char buf[160];
        std::snprintf(buf, sizeof buf, "plan needs %llu workspace bytes; the static workspace holds %u",
                      (unsigned long long)plan->p.ws.total, (unsigned)MK_STATIC_WORKSPACE_BYTES);
        return set_error(MK_ERR_INVALID, buf);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(MK_ERR_INVALID, "device ordinal out of range");
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mu);
        if (!g_static_addr[dev]) {
            void *addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_static_workspace);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static workspace)");
            g_static_addr[dev] = addr;
        }
        ws = g_static_addr[dev];
        // Another plan may have used the array since this plan's last call:
        // its queue must be uploaded again, and the counters there are the
        // other plan's, so this plan can only start over at step 0 (its wait
        // targets are cumulative over steps).
        if (g_static_owner[dev] != plan) {
            if (first_step != 0)
                return set_error(MK_ERR_INVALID,
                                 "the static workspace was used by another plan since this plan's last call: "
                                 "start again at first_step 0");
            plan->p.uploaded_ws = nullptr;
        }
        g_static_owner[dev] = plan;
    }
    if (workspace_out) *workspace_out = (uint64_t)(uintptr_t)ws;
    return mk_run(plan, ws, MK_STATIC_WORKSPACE_BYTES, first_step, num_steps, flags, timeout_ns, stream);
}

int mk_sync_status(mk_plan_t plan, void *workspace, void *stream, mk_error_record *rec) {
    if (!plan || !workspace) return set_error(MK_ERR_INVALID, "null plan or workspace");
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
    uint32_t w[E_WORDS];
    e = cudaMemcpy(w, static_cast<uint8_t *>(workspace) + plan->p.ws.err, sizeof w, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read error record");
    if (rec) {
        rec->code = (int32_t)w[E_CODE];
        rec->worker = (int32_t)w[E_WORKER];
        rec->slot = (int32_t)w[E_SLOT];
        rec->event = (int32_t)w[E_EVENT];
        rec->observed = w[E_OBSERVED];
        rec->needed = w[E_NEEDED];
        rec->opcode = (int32_t)w[E_OPCODE];
        rec->role = (int32_t)w[E_ROLE];
    }
    if (w[E_CODE]) {
        char buf[200];
        std::snprintf(buf, sizeof buf, "device error %u: worker %u slot %u event %d observed %u needed %u role %u",
                      w[E_CODE], w[E_WORKER], w[E_SLOT], (int)w[E_EVENT], w[E_OBSERVED], w[E_NEEDED], w[E_ROLE]);
        return set_error((int)w[E_CODE], buf);
    }
    return MK_OK;
}

int mk_read_counters(mk_plan_t plan, void *workspace, uint32_t *out) {
    if (!plan || !workspace || !out) return set_error(MK_ERR_INVALID, "null argument");
    cudaError_t e = cudaMemcpy(out, static_cast<uint8_t *>(workspace) + plan->p.ws.counters,
                               plan->p.thresholds.size() * 4, cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? MK_OK : cuda_fail(e, "read counters");
}

int mk_read_trace(mk_plan_t plan, void *workspace, uint64_t *out) {
    if (!plan || !workspace || !out) return set_error(MK_ERR_INVALID, "null argument");
    size_t slots = 0;
    for (auto &s : plan->p.segments) slots += (size_t)s.workers * s.lmax;
    cudaError_t e = cudaMemcpy(out, static_cast<uint8_t *>(workspace) + plan->p.ws.trace, slots * 128,
                               cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? MK_OK : cuda_fail(e, "read trace");
}

}  // extern "C"
