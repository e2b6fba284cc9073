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
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <vector>

#include "planner.h"

namespace mk {

#define DEV __device__ __forceinline__
constexpr unsigned FULL = 0xffffffffu;

// ---------------------------------------------------------------- PTX helpers
DEV uint32_t saddr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
DEV uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
DEV uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
DEV uint32_t ld_relaxed(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
DEV void red_release_add(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
DEV uint32_t atom_acqrel_add(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
DEV void mbar_init(uint64_t *b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(n) : "memory");
}
DEV void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
DEV void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}
DEV bool mbar_test(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(saddr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
DEV void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     saddr(dst)),
                 "l"(src), "r"(bytes), "r"(saddr(bar))
                 : "memory");
}
DEV void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

DEV void bf16x8(uint4 w, float f[8]) {
    f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xffff0000u);
    f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xffff0000u);
    f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xffff0000u);
}
DEV float bf16_at(const uint16_t *p, size_t i) { return __uint_as_float((uint32_t)p[i] << 16); }
DEV float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}
DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}
DEV uint64_t argmax_key(float v, int idx) {
    if (v == 0.0f) v = 0.0f;  // -0 and +0 compare equal
    uint32_t u = __float_as_uint(v);
    uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((uint64_t)ord << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)idx);
}

// ---------------------------------------------------------------- shared state
struct Smem {
    uint8_t *act[2];
    uint8_t *pages;
    float *aux;
    uint64_t *full, *empty, *act_full, *act_empty;
    volatile int *ctrl;  // [0] abort, [1..2] slot flags, [3] attention: last split
};

constexpr int SLOT_FRESH = 1;

DEV void raise_error(const KParams &P, const Smem &S, int code, int slot, int event, uint32_t obs, uint32_t need,
                     int opc, int role) {
    if (atomicCAS(&P.err[E_CODE], 0u, (uint32_t)code) == 0u) {
        P.err[E_WORKER] = blockIdx.x;
        P.err[E_SLOT] = (uint32_t)slot;
        P.err[E_EVENT] = (uint32_t)event;
        P.err[E_OBSERVED] = obs;
        P.err[E_NEEDED] = need;
        P.err[E_OPCODE] = (uint32_t)opc;
        P.err[E_ROLE] = (uint32_t)role;
    }
    atomicExch(&P.err[E_ABORT], 1u);
    S.ctrl[0] = 1;
}

DEV bool aborted(const KParams &P, const Smem &S) {
    if (S.ctrl[0]) return true;
    if (ld_relaxed(&P.err[E_ABORT])) {
        S.ctrl[0] = 1;
        return true;
    }
    return false;
}

// Whole-warp bounded wait on an mbarrier phase; uniform result, false = abort.
DEV bool warp_wait_bar(const KParams &P, const Smem &S, uint64_t *bar, uint32_t parity, int role, int slot, int opc) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (__all_sync(FULL, mbar_test(bar, parity))) return true;
        if ((it & 15) == 15) {
            int stop = 0;
            if (lane == 0) {
                uint64_t now = gtimer();
                if (t0 == 0) t0 = now;
                if (aborted(P, S)) stop = 1;
                else if (now - t0 > P.timeout_ns) {
                    raise_error(P, S, MK_ERR_TIMEOUT, slot, -1, 0, parity, opc, role);
                    stop = 1;
                }
            }
            if (__shfl_sync(FULL, stop, 0)) return false;
        }
    }
}

// Single-thread bounded wait (loader lane).
DEV bool thread_wait_bar(const KParams &P, const Smem &S, uint64_t *bar, uint32_t parity, int slot, int opc) {
    if (mbar_test(bar, parity)) return true;
    uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 15) == 0) {
            if (aborted(P, S)) return false;
            if (gtimer() - t0 > P.timeout_ns) {
                raise_error(P, S, MK_ERR_TIMEOUT, slot, -1, 0, parity, opc, 0);
                return false;
            }
        }
    }
}

// Whole-warp bounded wait for counter >= target (acquire on every poll).
DEV bool warp_wait_counter(const KParams &P, const Smem &S, int ev, uint32_t target, int slot, int opc) {
    const int lane = threadIdx.x & 31;
    const uint32_t *c = P.counters + ev;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t v = ld_acquire(c);
        if (__all_sync(FULL, v >= target)) return true;
        if ((it & 15) == 15) {
            int stop = 0;
            if (lane == 0) {
                uint64_t now = gtimer();
                if (t0 == 0) t0 = now;
                if (aborted(P, S)) stop = 1;
                else if (now - t0 > P.timeout_ns) {
                    raise_error(P, S, MK_ERR_TIMEOUT, slot, ev, v, target, opc, 1);
                    stop = 1;
                }
            }
            if (__shfl_sync(FULL, stop, 0)) return false;
        }
    }
}

// ---------------------------------------------------------------- instruction decoding
struct Seg {
    const uint8_t *src;
    int rows;
    int row_bytes;
    long long stride;
};

DEV int ins_word(const int32_t *ins, int k) { return __ldg(ins + k); }

DEV bool ins_valid(const KParams &P, const int32_t *ins) {
    int opc = ins_word(ins, W_OPC);
    if (opc < 0 || opc >= MK_NUM_OPCODES) return false;
    if (opc == MK_OP_NOOP) return true;
    int row = ins_word(ins, W_ROW);
    if (row < 0 || row >= P.num_ops) return false;
    int cnt = ins_word(ins, W_CNT);
    int nw = cnt & 0xff, ns = (cnt >> 8) & 0xff;
    if (nw > MAX_WAITS || ns > MAX_SIGS) return false;
    for (int i = 0; i < nw; ++i)
        if ((int)((uint32_t)ins_word(ins, W_WAIT + 2 * i) & ~WAIT_PREV_EPOCH) >= P.num_events) return false;
    for (int i = 0; i < ns; ++i)
        if ((uint32_t)ins_word(ins, W_SIG + 2 * i) >= (uint32_t)P.num_events) return false;
    if (opc >= MK_OP_QKV && opc != MK_OP_ATTN) {
        int nrows = ins_word(ins, P_NROWS), kc = ins_word(ins, P_KC);
        if (nrows <= 0 || nrows > MAX_TILE_ROWS || (opc == MK_OP_UP && 2 * nrows > MAX_TILE_ROWS)) return false;
        if (kc <= 0 || kc % 8 || 2 * kc > P.page_bytes || kc * P.B * 4 > P.act_bytes) return false;
    }
    if (opc == MK_OP_ATTN) {
        int T = ins_word(ins, P_T);
        if (T <= 0 || T > 256 || ins_word(ins, P_B) >= P.B || ins_word(ins, P_G) >= P.Hkv) return false;
        if (ins_word(ins, P_SPLIT) >= P.nsplit_max) return false;
    }
    return true;
}

// Cached cache rows of an attention task at this step.
DEV int attn_cached_rows(const KParams &P, const int32_t *ins, int pos) {
    int t0 = ins_word(ins, P_T0), T = ins_word(ins, P_T);
    return max(0, min(T, pos - t0));
}

DEV int seq_pos(const KParams &P, const int32_t *ins) {
    const uint64_t *t = P.optab + (size_t)ins_word(ins, W_ROW) * N_SLOTS;
    const int32_t *seq0 = reinterpret_cast<const int32_t *>(t[S_AT_SEQ0]);
    return __ldg(seq0 + ins_word(ins, P_B)) + P.step;
}

// Weight / cache rows streamed by the loader for one instruction.  Loader and
// consumers call this with the same arguments and walk the same page ring.
DEV int describe(const KParams &P, const int32_t *ins, Seg seg[2]) {
    const int opc = ins_word(ins, W_OPC);
    const uint64_t *t = P.optab + (size_t)ins_word(ins, W_ROW) * N_SLOTS;
    if (opc == MK_OP_QKV || opc == MK_OP_O || opc == MK_OP_DOWN || opc == MK_OP_LM || opc == MK_OP_UP) {
        const long long ktot = ins_word(ins, P_KTOT);
        const long long off = ((long long)ins_word(ins, P_ROW0) * ktot + ins_word(ins, P_K0)) * 2;
        int slot = opc == MK_OP_QKV ? S_QKV_WQ + ins_word(ins, P_MAT)
                 : opc == MK_OP_O   ? S_O_W
                 : opc == MK_OP_DOWN ? S_DN_W
                 : opc == MK_OP_LM  ? S_LM_W
                                    : S_UP_WG;
        seg[0].src = reinterpret_cast<const uint8_t *>(t[slot]) + off;
        seg[0].rows = ins_word(ins, P_NROWS);
        seg[0].row_bytes = ins_word(ins, P_KC) * 2;
        seg[0].stride = ktot * 2;
        if (opc != MK_OP_UP) return 1;
        seg[1] = seg[0];
        seg[1].src = reinterpret_cast<const uint8_t *>(t[S_UP_WU]) + off;
        return 2;
    }
    if (opc == MK_OP_ATTN) {
        const int pos = seq_pos(P, ins);
        const int n = attn_cached_rows(P, ins, pos);
        const long long base = (((long long)ins_word(ins, P_B) * P.Hkv + ins_word(ins, P_G)) * P.Smax +
                                ins_word(ins, P_T0)) * P.D * 2;
        seg[0].src = reinterpret_cast<const uint8_t *>(t[S_AT_K]) + base;
        seg[0].rows = n;
        seg[0].row_bytes = P.D * 2;
        seg[0].stride = P.D * 2;
        seg[1] = seg[0];
        seg[1].src = reinterpret_cast<const uint8_t *>(t[S_AT_V]) + base;
        return 2;
    }
    return 0;
}

// ---------------------------------------------------------------- loader role
DEV void loader_role(const KParams &P, const Smem &S, const int32_t *myq) {
    uint32_t ring = 0;
    const int NP = P.num_pages, PS = P.page_bytes;
    for (int i = 0; i < P.lmax; ++i) {
        if (S.ctrl[0]) break;
        const int32_t *ins = myq + (size_t)i * W_WORDS;
        if (!ins_valid(P, ins)) {
            raise_error(P, S, MK_ERR_DEVICE_CHECK, i, -1, 0, 0, ins_word(ins, W_OPC), 0);
            break;
        }
        Seg seg[2];
        const int nseg = describe(P, ins, seg);
        bool stop = false;
        for (int s = 0; s < nseg && !stop; ++s) {
            const int rpp = PS / seg[s].row_bytes;
            for (int r = 0; r < seg[s].rows; r += rpp) {
                const int nr = min(rpp, seg[s].rows - r);
                const uint32_t p = ring % NP, use = ring / NP;
                if (!thread_wait_bar(P, S, &S.empty[p], (use & 1) ^ 1, i, ins_word(ins, W_OPC))) {
                    stop = true;
                    break;
                }
                uint8_t *dst = S.pages + (size_t)p * PS;
                const uint32_t bytes = (uint32_t)nr * seg[s].row_bytes;
                mbar_expect_tx(&S.full[p], bytes);
                const uint8_t *src = seg[s].src + (long long)r * seg[s].stride;
                if (seg[s].stride == seg[s].row_bytes) {
                    bulk_g2s(dst, src, bytes, &S.full[p]);
                } else {
                    for (int j = 0; j < nr; ++j)
                        bulk_g2s(dst + (size_t)j * seg[s].row_bytes, src + (long long)j * seg[s].stride,
                                 seg[s].row_bytes, &S.full[p]);
                }
                ++ring;
            }
        }
        if (stop) break;
    }
    // no bulk copy may still target this CTA's shared memory when it exits
    const uint32_t first = ring > (uint32_t)NP ? ring - NP : 0;
    const uint64_t t0 = gtimer();
    for (uint32_t k = first; k < ring; ++k) {
        const uint32_t p = k % NP, use = k / NP;
        while (!mbar_test(&S.full[p], use & 1)) {
            if (gtimer() - t0 > 2 * P.timeout_ns) break;  // copies of valid memory land in microseconds
        }
    }
}

// ---------------------------------------------------------------- activation loader role
template <int MAXB>
DEV void aloader_gemv(const KParams &P, const Smem &S, const int32_t *ins, float *slot, bool ab) {
    const int lane = threadIdx.x & 31;
    const int opc = ins_word(ins, W_OPC);
    const uint64_t *t = P.optab + (size_t)ins_word(ins, W_ROW) * N_SLOTS;
    const int B = P.B;
    if (opc == MK_OP_QKV || opc == MK_OP_UP || opc == MK_OP_LM) {
        const int H = P.H;
        const float *h = reinterpret_cast<const float *>(
            t[opc == MK_OP_QKV ? S_QKV_H : opc == MK_OP_UP ? S_UP_H : S_LM_H]);
        const uint16_t *w = reinterpret_cast<const uint16_t *>(
            t[opc == MK_OP_QKV ? S_QKV_NORM : opc == MK_OP_UP ? S_UP_NORM : S_LM_NORM]);
        const int snap = ins_word(ins, P_SNAP);
        float *hist = nullptr;
        if (snap > 0 && !ab) hist = reinterpret_cast<float *>(t[opc == MK_OP_QKV ? S_QKV_HIST : S_LM_HIST]);
        for (int b = 0; b < B; ++b) {
            const float4 *src = reinterpret_cast<const float4 *>(h + (size_t)b * H);
            float4 *dst = reinterpret_cast<float4 *>(slot + (size_t)b * H);
            float ss = 0.f;
            for (int k = lane; k < H / 4; k += 32) {
                float4 v = __ldcg(src + k);
                dst[k] = v;
                ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
                if (hist) reinterpret_cast<float4 *>(hist + ((size_t)(snap - 1) * B + b) * H)[k] = v;
            }
            ss = warp_sum(ss);
            const float scale = rsqrtf(ss / (float)H + P.eps);
            __syncwarp();
            for (int k = lane; k < H; k += 32) slot[(size_t)b * H + k] *= scale * bf16_at(w, k);
        }
    } else {
        // O: attention output [B, Hq*D];  DOWN: act[b][k0 .. k0+kc)
        const int kc = ins_word(ins, P_KC);
        const float *src;
        size_t ld;
        if (opc == MK_OP_O) {
            src = reinterpret_cast<const float *>(t[S_O_IN]);
            ld = (size_t)P.Hq * P.D;
        } else {
            src = reinterpret_cast<const float *>(t[S_DN_IN]) + ins_word(ins, P_K0);
            ld = (size_t)P.F;
        }
        for (int b = 0; b < B; ++b) {
            const float4 *s4 = reinterpret_cast<const float4 *>(src + b * ld);
            float4 *d4 = reinterpret_cast<float4 *>(slot + (size_t)b * kc);
            for (int k = lane; k < kc / 4; k += 32) d4[k] = __ldcg(s4 + k);
        }
    }
}

// q (pre-scaled into log2 units), new k and v of one (sequence, kv group):
// q/k RMSNorm (optional), RoPE at the new position, bf16 rounding of the new
// k/v, and the KV-cache append by the split that owns the new position.
DEV void aloader_attn(const KParams &P, const Smem &S, const int32_t *ins, float *slot, bool ab) {
    const int lane = threadIdx.x & 31;
    const uint64_t *t = P.optab + (size_t)ins_word(ins, W_ROW) * N_SLOTS;
    const int D = P.D, G = P.Hq / P.Hkv, b = ins_word(ins, P_B), g = ins_word(ins, P_G);
    const int pos = seq_pos(P, ins);
    const int t0 = ins_word(ins, P_T0), T = ins_word(ins, P_T);
    const float *src = reinterpret_cast<const float *>(t[S_AT_QKV]) + ((size_t)b * P.Hkv + g) * (G + 2) * D;
    const int QS = D / 4 + 4;                 // padded quarter stride of q in the slot
    float *qp = slot;                         // [G][4][QS]
    float *kn = slot + G * 4 * QS;            // [D]
    float *vn = kn + D;                       // [D]
    const int per = D / 32;                   // elements per lane (2 or 4)
    const float qscale = rsqrtf((float)D) * 1.4426950408889634f;
    // rotation of pair i (i in [0, D/2)), computed once per lane: angle in double, reduced mod 2*pi
    float cs[2], sn[2];
    for (int j = 0; j < D / 64; ++j) {
        const int i = lane + 32 * j;
        const double inv_freq = exp2(-(2.0 * i / D) * log2((double)P.theta));
        const double ang = (double)pos * inv_freq;
        const double two_pi = 6.283185307179586476925286766559;
        const double red = ang - rint(ang / two_pi) * two_pi;
        sincosf((float)red, &sn[j], &cs[j]);
    }
    for (int h = 0; h < G + 2; ++h) {
        float x[4];
        for (int e = 0; e < per; ++e) x[e] = __ldcg(src + (size_t)h * D + lane + 32 * e);
        const bool is_q = h < G, is_k = h == G;
        if (P.qk_norm && (is_q || is_k)) {
            const uint16_t *w = reinterpret_cast<const uint16_t *>(t[is_q ? S_AT_QN : S_AT_KN]);
            float ss = 0.f;
            for (int e = 0; e < per; ++e) ss += x[e] * x[e];
            ss = warp_sum(ss);
            const float sc = rsqrtf(ss / (float)D + P.eps);
            for (int e = 0; e < per; ++e) x[e] = x[e] * sc * bf16_at(w, lane + 32 * e);
        }
        if (is_q || is_k) {
            // element lane+32e pairs with lane+32e +/- D/2: e < per/2 is the first half
            for (int e = 0; e < per / 2; ++e) {
                const float a = x[e], c = x[e + per / 2];
                x[e] = a * cs[e] - c * sn[e];
                x[e + per / 2] = a * sn[e] + c * cs[e];
            }
        }
        for (int e = 0; e < per; ++e) {
            const int d = lane + 32 * e;
            if (is_q) qp[(h * 4 + d / (D / 4)) * QS + d % (D / 4)] = x[e] * qscale;
            else if (is_k) kn[d] = round_bf16(x[e]);
            else vn[d] = round_bf16(x[e]);
        }
    }
    if (!ab && pos >= t0 && pos < t0 + T) {
        __syncwarp();
        const size_t c = (((size_t)b * P.Hkv + g) * P.Smax + pos) * D;
        __nv_bfloat16 *kc = reinterpret_cast<__nv_bfloat16 *>(t[S_AT_K]) + c;
        __nv_bfloat16 *vc = reinterpret_cast<__nv_bfloat16 *>(t[S_AT_V]) + c;
        for (int d = lane; d < D; d += 32) {
            kc[d] = __float2bfloat16_rn(kn[d]);
            vc[d] = __float2bfloat16_rn(vn[d]);
        }
    }
}

template <int MAXB>
DEV void aloader_role(const KParams &P, const Smem &S, const int32_t *myq) {
    const int lane = threadIdx.x & 31;
    long long prev_key = -1;
    bool ab = false;
    for (int i = 0; i < P.lmax; ++i) {
        const int32_t *ins = myq + (size_t)i * W_WORDS;
        const int opc = ins_word(ins, W_OPC);
        if (opc == MK_OP_NOOP) continue;
        const int sl = i & 1;
        const uint32_t use = (uint32_t)(i >> 1);
        if (!ab && !ins_valid(P, ins)) {
            if (lane == 0) raise_error(P, S, MK_ERR_DEVICE_CHECK, i, -1, 0, 0, opc, 1);
            ab = true;
        }
        if (!ab) ab = !warp_wait_bar(P, S, &S.act_empty[sl], (use & 1) ^ 1, 1, i, opc);
        const int cnt = ins_word(ins, W_CNT);
        for (int w = 0; w < (cnt & 0xff) && !ab; ++w) {
            const uint32_t ew = (uint32_t)ins_word(ins, W_WAIT + 2 * w);
            const uint32_t thr = (uint32_t)ins_word(ins, W_WAIT + 2 * w + 1);
            const int ev = (int)(ew & ~WAIT_PREV_EPOCH);
            const int epoch = P.step + 1 - ((ew & WAIT_PREV_EPOCH) ? 1 : 0);
            const uint32_t target = thr * (uint32_t)epoch;
            if (target > 0) ab = !warp_wait_counter(P, S, ev, target, i, opc);
        }
        if (!ab && lane == 0 && P.trace) P.trace[((size_t)blockIdx.x * P.lmax + i) * 4 + 2] = gtimer();
        float *slot = reinterpret_cast<float *>(S.act[sl]);
        int flags = 0;
        if (opc == MK_OP_ATTN) {
            aloader_attn(P, S, ins, slot, ab);
            flags = SLOT_FRESH;
            prev_key = -1;
        } else if (opc >= MK_OP_QKV) {
            const long long key = ((long long)ins_word(ins, W_ROW) << 32) | (uint32_t)ins_word(ins, P_K0);
            if (key != prev_key || ins_word(ins, P_SNAP) > 0) {
                aloader_gemv<MAXB>(P, S, ins, slot, ab);
                flags = SLOT_FRESH;
            }
            prev_key = key;
        } else {
            prev_key = -1;
        }
        __syncwarp();
        if (lane == 0) {
            S.ctrl[1 + sl] = flags;
            mbar_arrive(&S.act_full[sl]);
        }
    }
}

// ---------------------------------------------------------------- consumers
__host__ __device__ constexpr int nch_max(int maxb) { return maxb >= 8 ? 1 : (maxb >= 4 ? 2 : 4); }

template <int MAXB>
struct XRegs {
    float v[nch_max(MAXB)][MAXB][8];
};

DEV void publish(const KParams &P, const int32_t *ins, int ct, bool ab) {
    consumer_sync();
    if (ct == 0 && !ab) {
        const int ns = (ins_word(ins, W_CNT) >> 8) & 0xff;
        for (int s = 0; s < ns; ++s)
            red_release_add(P.counters + ins_word(ins, W_SIG + 2 * s), (uint32_t)ins_word(ins, W_SIG + 2 * s + 1));
    }
}

// Walks the instruction's pages: GEMV over rows resident in the page ring.
template <int MAXB>
DEV void consume_gemv(const KParams &P, const Smem &S, const int32_t *ins, int i, const float *slot, bool fresh,
                      XRegs<MAXB> &xr, uint32_t &ring, bool &ab) {
    constexpr int NCH = nch_max(MAXB);
    const int ct = threadIdx.x - 64, warp = ct >> 5, lane = ct & 31;
    const int opc = ins_word(ins, W_OPC);
    const int B = P.B;
    const int kc = ins_word(ins, P_KC), nchunk = kc / 8, row_bytes = kc * 2;
    if (fresh) {
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
            const int c = ct + CONSUMERS * j;
#pragma unroll
            for (int b = 0; b < MAXB; ++b) {
                if (c < nchunk && b < B) {
                    const float4 *s4 = reinterpret_cast<const float4 *>(slot + (size_t)b * kc + c * 8);
                    float4 a = s4[0], bb = s4[1];
                    xr.v[j][b][0] = a.x; xr.v[j][b][1] = a.y; xr.v[j][b][2] = a.z; xr.v[j][b][3] = a.w;
                    xr.v[j][b][4] = bb.x; xr.v[j][b][5] = bb.y; xr.v[j][b][6] = bb.z; xr.v[j][b][7] = bb.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) xr.v[j][b][e] = 0.f;
                }
            }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.act_empty[i & 1]);  // slot no longer needed

    float *red = S.aux;  // [warp][MAX_TILE_ROWS][MAXB]
    Seg seg[2];
    const int nseg = describe(P, ins, seg);
    const int rpp = P.page_bytes / row_bytes;
    int row_out = 0;
    for (int s = 0; s < nseg; ++s) {
        for (int r = 0; r < seg[s].rows; r += rpp) {
            const int nr = min(rpp, seg[s].rows - r);
            const uint32_t p = ring % P.num_pages, use = ring / P.num_pages;
            if (!ab) ab = !warp_wait_bar(P, S, &S.full[p], use & 1, 2, i, opc);
            const uint8_t *page = S.pages + (size_t)p * P.page_bytes;
            for (int rg = 0; rg < nr; rg += 4) {
                float acc[4][MAXB];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                    for (int b = 0; b < MAXB; ++b) acc[rr][b] = 0.f;
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    if (rg + rr < nr) {
                        const uint8_t *wrow = page + (size_t)(rg + rr) * row_bytes;
#pragma unroll
                        for (int j = 0; j < NCH; ++j) {
                            const int c = ct + CONSUMERS * j;
                            if (c < nchunk) {
                                float w8[8];
                                bf16x8(*reinterpret_cast<const uint4 *>(wrow + c * 16), w8);
#pragma unroll
                                for (int b = 0; b < MAXB; ++b)
#pragma unroll
                                    for (int e = 0; e < 8; ++e) acc[rr][b] = fmaf(w8[e], xr.v[j][b][e], acc[rr][b]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                    for (int b = 0; b < MAXB; ++b) {
                        const float v = warp_sum(acc[rr][b]);
                        if (lane == 0 && rg + rr < nr)
                            red[(warp * MAX_TILE_ROWS + row_out + rg + rr) * MAXB + b] = v;
                    }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[p]);
            ++ring;
            row_out += nr;
        }
    }
    consumer_sync();
    // epilogue
    const uint64_t *t = P.optab + (size_t)ins_word(ins, W_ROW) * N_SLOTS;
    const int nrows = ins_word(ins, P_NROWS), out0 = ins_word(ins, P_OUT0);
    auto rowsum = [&](int r, int b) {
        float y = 0.f;
#pragma unroll
        for (int w = 0; w < CONSUMER_WARPS; ++w) y += red[(w * MAX_TILE_ROWS + r) * MAXB + b];
        return y;
    };
    if (ct < nrows * B && !ab) {
        const int r = ct / B, b = ct % B;
        if (opc == MK_OP_QKV) {
            float *out = reinterpret_cast<float *>(t[S_QKV_OUT]);
            const int G = P.Hq / P.Hkv;
            out[(size_t)b * P.Hkv * (G + 2) * P.D + out0 + r] = rowsum(r, b);
        } else if (opc == MK_OP_O) {
            float *hres = reinterpret_cast<float *>(t[S_O_HRES]);
            float *hmid = reinterpret_cast<float *>(t[S_O_HMID]);
            const size_t k = (size_t)b * P.H + out0 + r;
            const float v = __ldcg(hres + k) + rowsum(r, b);
            hres[k] = v;
            hmid[k] = v;
        } else if (opc == MK_OP_UP) {
            float *act = reinterpret_cast<float *>(t[S_UP_OUT]);
            const float g = rowsum(r, b), u = rowsum(nrows + r, b);
            act[(size_t)b * P.F + out0 + r] = g / (1.0f + expf(-g)) * u;
        } else if (opc == MK_OP_DOWN) {
            float *hres = reinterpret_cast<float *>(t[S_DN_HRES]);
            atomicAdd(hres + (size_t)b * P.H + out0 + r, rowsum(r, b));
        } else if (opc == MK_OP_LM) {
            float *logits = reinterpret_cast<float *>(t[S_LM_LOGITS]);
            logits[(size_t)b * P.V + out0 + r] = rowsum(r, b);
        }
        __threadfence();
    }
    if (opc == MK_OP_LM && ct < B && !ab) {
        float best = -INFINITY;
        int bi = 0;
        for (int r = 0; r < nrows; ++r) {
            const float v = rowsum(r, ct);
            if (v > best) { best = v; bi = r; }
        }
        unsigned long long *keys = reinterpret_cast<unsigned long long *>(t[S_LM_KEYS]);
        atomicMax(keys + (size_t)P.step * B + ct, (unsigned long long)argmax_key(best, out0 + bi));
        __threadfence();
    }
}

// Split-KV attention of one (sequence, kv group, split): scores from the
// cached K rows in the page ring plus the new token, softmax partial
// (max, sum) in log2 units, P.V, partial written out; the last split of the
// (sequence, group) to arrive merges all splits ("Lecture 7 notes", section
// 5.1: attention and attention reduction).
DEV void consume_attn(const KParams &P, const Smem &S, const int32_t *ins, int i, const float *slot, uint32_t &ring,
                      bool &ab) {
    const int ct = threadIdx.x - 64, warp = ct >> 5, lane = ct & 31;
    const uint64_t *t = P.optab + (size_t)ins_word(ins, W_ROW) * N_SLOTS;
    const int D = P.D, G = P.Hq / P.Hkv, b = ins_word(ins, P_B), g = ins_word(ins, P_G);
    const int split = ins_word(ins, P_SPLIT), nsplit = ins_word(ins, P_NSPLIT), layer = ins_word(ins, P_LAYER);
    const int pos = seq_pos(P, ins);
    const int t0 = ins_word(ins, P_T0), T = ins_word(ins, P_T);
    const int ncache = attn_cached_rows(P, ins, pos);
    const bool has_new = pos >= t0 && pos < t0 + T;
    const int ntot = ncache + (has_new ? 1 : 0);
    const int QS = D / 4 + 4;
    const float *qp = slot, *kn = slot + G * 4 * QS, *vn = kn + D;
    float *sc = S.aux;                       // [G][T] scores then probabilities
    float *ow = sc + G * T;                  // [warp][G][D]
    float *ml = ow + CONSUMER_WARPS * G * D; // [G] max, [G] sum
    const int rpp = P.page_bytes / (D * 2);
    const int npg = (ncache + rpp - 1) / rpp;
    const int opc = MK_OP_ATTN;
    // K pages
    const uint32_t kring = ring;
    for (int k = 0; k < npg; ++k) {
        const uint32_t p = (ring + k) % P.num_pages, use = (ring + k) / P.num_pages;
        if (!ab) ab = !warp_wait_bar(P, S, &S.full[p], use & 1, 2, i, opc);
    }
    // scores: a warp takes 8 tokens at a time, 4 lanes per token, D/4 dims per lane
    const int qtr = lane & 3;
    for (int tb = warp * 8; tb < ntot; tb += CONSUMER_WARPS * 8) {
        const int tk = tb + (lane >> 2);
        float s[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) s[h] = 0.f;
        if (tk < ntot) {
            const int d0 = qtr * (D / 4);
            for (int dd = 0; dd < D / 4; dd += 8) {
                float k8[8];
                if (tk < ncache) {
                    const uint32_t p = (kring + tk / rpp) % P.num_pages;
                    const uint8_t *row = S.pages + (size_t)p * P.page_bytes + (size_t)(tk % rpp) * D * 2;
                    bf16x8(*reinterpret_cast<const uint4 *>(row + (d0 + dd) * 2), k8);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) k8[e] = kn[d0 + dd + e];
                }
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    if (h < G) {
                        const float *q = qp + (h * 4 + qtr) * QS + dd;
#pragma unroll
                        for (int e = 0; e < 8; ++e) s[h] = fmaf(q[e], k8[e], s[h]);
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            s[h] += __shfl_xor_sync(FULL, s[h], 1);
            s[h] += __shfl_xor_sync(FULL, s[h], 2);
        }
        if (qtr == 0 && tk < ntot)
            for (int h = 0; h < G; ++h) sc[h * T + tk] = s[h];
    }
    __syncwarp();
    if (lane == 0)
        for (int k = 0; k < npg; ++k) mbar_arrive(&S.empty[(kring + k) % P.num_pages]);
    consumer_sync();
    // softmax statistics per head (one warp per head)
    if (warp < G) {
        float m = -INFINITY;
        for (int tk = lane; tk < ntot; tk += 32) m = fmaxf(m, sc[warp * T + tk]);
        m = warp_max(m);
        float l = 0.f;
        for (int tk = lane; tk < ntot; tk += 32) {
            const float e = exp2f(sc[warp * T + tk] - m);
            sc[warp * T + tk] = e;
            l += e;
        }
        l = warp_sum(l);
        if (lane == 0) {
            ml[warp] = m;
            ml[G + warp] = l;
        }
    }
    // V pages
    const uint32_t vring = kring + npg;
    for (int k = 0; k < npg; ++k) {
        const uint32_t p = (vring + k) % P.num_pages, use = (vring + k) / P.num_pages;
        if (!ab) ab = !warp_wait_bar(P, S, &S.full[p], use & 1, 2, i, opc);
    }
    ring = vring + npg;
    consumer_sync();
    // P.V: warp w takes tokens w, w+8, ...; lane holds D/32 dims
    {
        const int per = D / 32;
        float acc[8][4];
#pragma unroll
        for (int h = 0; h < 8; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[h][e] = 0.f;
        for (int tk = warp; tk < ntot; tk += CONSUMER_WARPS) {
            float v[4];
            if (tk < ncache) {
                const uint32_t p = (vring + tk / rpp) % P.num_pages;
                const uint16_t *row = reinterpret_cast<const uint16_t *>(S.pages + (size_t)p * P.page_bytes +
                                                                         (size_t)(tk % rpp) * D * 2);
                for (int e = 0; e < per; ++e) v[e] = __uint_as_float((uint32_t)row[lane * per + e] << 16);
            } else {
                for (int e = 0; e < per; ++e) v[e] = vn[lane * per + e];
            }
#pragma unroll
            for (int h = 0; h < 8; ++h)
                if (h < G) {
                    const float pr = sc[h * T + tk];
                    for (int e = 0; e < per; ++e) acc[h][e] = fmaf(pr, v[e], acc[h][e]);
                }
        }
        for (int h = 0; h < G; ++h)
            for (int e = 0; e < per; ++e) ow[(warp * G + h) * D + lane * per + e] = acc[h][e];
    }
    __syncwarp();
    if (lane == 0) {
        for (int k = 0; k < npg; ++k) mbar_arrive(&S.empty[(vring + k) % P.num_pages]);
        mbar_arrive(&S.act_empty[i & 1]);
    }
    consumer_sync();
    // partial (o unnormalised, m, l) for every head of the group
    float *part = reinterpret_cast<float *>(t[S_AT_PART]);
    auto part_at = [&](int h, int s) {
        return part + (((size_t)b * P.Hq + g * G + h) * P.nsplit_max + s) * (D + 2);
    };
    for (int k = ct; k < G * D && !ab; k += CONSUMERS) {
        const int h = k / D, d = k % D;
        float o = 0.f;
        for (int w = 0; w < CONSUMER_WARPS; ++w) o += ow[(w * G + h) * D + d];
        part_at(h, split)[d] = o;
    }
    if (ct < G && !ab) {
        part_at(ct, split)[D] = ml[ct];
        part_at(ct, split)[D + 1] = ml[G + ct];
    }
    __threadfence();
    consumer_sync();
    if (ct == 0) {
        int last = 0;
        if (!ab) {
            uint32_t *arrive = reinterpret_cast<uint32_t *>(t[S_AT_ARRIVE]) + ((size_t)layer * P.B + b) * P.Hkv + g;
            const uint32_t old = atom_acqrel_add(arrive, 1u);
            last = old == (uint32_t)(P.step + 1) * (uint32_t)nsplit - 1u;
        }
        S.ctrl[3] = last;
    }
    consumer_sync();
    if (S.ctrl[3] && !ab) {
        float *out = reinterpret_cast<float *>(t[S_AT_OUT]);
        for (int k = ct; k < G * D; k += CONSUMERS) {
            const int h = k / D, d = k % D;
            float M = -INFINITY;
            for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldcg(part_at(h, s) + D));
            float L = 0.f, o = 0.f;
            for (int s = 0; s < nsplit; ++s) {
                const float* ps = part_at(h, s);
                const float f = exp2f(__ldcg(ps + D) - M);
                L += f * __ldcg(ps + D + 1);
                o += f * __ldcg(ps + d);
            }
            out[(size_t)b * P.Hq * D + (size_t)(g * G + h) * D + d] = o / L;
        }
        __threadfence();
    }
}

DEV void consume_embed(const KParams &P, const Smem &S, const int32_t *ins, int i, bool ab) {
    const int ct = threadIdx.x - 64, lane = ct & 31;
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.act_empty[i & 1]);
    if (ab) return;
    const uint64_t *t = P.optab + (size_t)ins_word(ins, W_ROW) * N_SLOTS;
    const uint16_t *E = reinterpret_cast<const uint16_t *>(t[S_EMB_W]);
    float *h = reinterpret_cast<float *>(t[S_EMB_H]);
    int32_t *tokens = reinterpret_cast<int32_t *>(t[S_EMB_TOK]);
    const unsigned long long *keys = reinterpret_cast<const unsigned long long *>(t[S_EMB_KEYS]);
    const bool host_tokens = (P.flags & MK_RUN_HOST_TOKENS) || P.step == 0;
    for (int b = 0; b < P.B; ++b) {
        int tok;
        if (host_tokens) tok = __ldcg(tokens + (size_t)P.step * P.B + b);
        else tok = (int)(0xFFFFFFFFu - (uint32_t)(__ldcg(keys + (size_t)(P.step - 1) * P.B + b) & 0xFFFFFFFFull));
        if (tok < 0 || tok >= P.V) tok = 0;  // invalid ids read row 0 (checked on the host side too)
        if (!host_tokens && ct == 0) tokens[(size_t)P.step * P.B + b] = tok;
        for (int k = ct; k < P.H; k += CONSUMERS) h[(size_t)b * P.H + k] = bf16_at(E, (size_t)tok * P.H + k);
    }
    __threadfence();
}

template <int MAXB>
DEV void consumer_role(const KParams &P, const Smem &S, const int32_t *myq) {
    const int ct = threadIdx.x - 64, lane = ct & 31;
    uint32_t ring = 0;
    bool ab = false;
    XRegs<MAXB> xr;
    for (int i = 0; i < P.lmax; ++i) {
        const int32_t *ins = myq + (size_t)i * W_WORDS;
        const int opc = ins_word(ins, W_OPC);
        if (opc == MK_OP_NOOP) continue;
        uint64_t t_start = 0;
        if (ct == 0 && P.trace) t_start = gtimer();
        const int sl = i & 1;
        if (!ab) ab = !warp_wait_bar(P, S, &S.act_full[sl], (uint32_t)(i >> 1) & 1, 2, i, opc);
        const bool fresh = (S.ctrl[1 + sl] & SLOT_FRESH) != 0;
        const float *slot = reinterpret_cast<const float *>(S.act[sl]);
        if (opc == MK_OP_ATTN) consume_attn(P, S, ins, i, slot, ring, ab);
        else if (opc == MK_OP_EMBED) consume_embed(P, S, ins, i, ab);
        else if (opc >= MK_OP_QKV) consume_gemv<MAXB>(P, S, ins, i, slot, fresh, xr, ring, ab);
        else {  // COUNTER: nothing but the handshake
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.act_empty[sl]);
        }
        publish(P, ins, ct, ab);
        if (ct == 0 && P.trace) {
            uint64_t *tr = P.trace + ((size_t)blockIdx.x * P.lmax + i) * 4;
            tr[0] = (uint64_t)opc | ((uint64_t)(uint32_t)ins_word(ins, W_TASK) << 32);
            tr[1] = t_start;
            tr[3] = gtimer();
        }
    }
}

// ---------------------------------------------------------------- kernel
template <int MAXB>
__global__ void __launch_bounds__(THREADS, 1) mk_interp(const KParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Smem S;
    S.act[0] = smem;
    S.act[1] = smem + P.act_bytes;
    S.pages = smem + 2 * P.act_bytes;
    S.aux = reinterpret_cast<float *>(S.pages + (size_t)P.num_pages * P.page_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(S.aux) + P.aux_bytes);
    S.full = bars;
    S.empty = bars + P.num_pages;
    S.act_full = bars + 2 * P.num_pages;
    S.act_empty = bars + 2 * P.num_pages + 2;
    S.ctrl = reinterpret_cast<volatile int *>(reinterpret_cast<uint8_t *>(bars) + MBAR_BYTES);
    if (threadIdx.x == 0) {
        for (int p = 0; p < P.num_pages; ++p) {
            mbar_init(&S.full[p], 1);
            mbar_init(&S.empty[p], CONSUMER_WARPS);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.act_full[s], 1);
            mbar_init(&S.act_empty[s], CONSUMER_WARPS);
        }
        for (int k = 0; k < 4; ++k) S.ctrl[k] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    const int32_t *myq = P.queue + (size_t)blockIdx.x * P.lmax * W_WORDS;
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        if ((threadIdx.x & 31) == 0) loader_role(P, S, myq);
    } else if (warp == 1) {
        aloader_role<MAXB>(P, S, myq);
    } else {
        consumer_role<MAXB>(P, S, myq);
    }
    __syncthreads();
}

// ---------------------------------------------------------------- host side
static thread_local std::string g_cuda_msg;

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

static KernelFn pick_kernel(int B) {
    if (B <= 1) return mk_interp<1>;
    if (B <= 2) return mk_interp<2>;
    if (B <= 4) return mk_interp<4>;
    return mk_interp<8>;
}

static int build_table(Plan &p, uint8_t *ws, std::vector<uint64_t> &tab) {
    tab.assign((size_t)p.num_ops * N_SLOTS, 0);
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
    k.aux_bytes = p.aux_bytes;
    k.smem_bytes = p.smem_bytes;
    const mk_model_desc &m = p.model;
    k.B = p.B;
    k.H = m.hidden; k.Hq = m.q_heads; k.Hkv = m.kv_heads > 0 ? m.kv_heads : 1; k.D = m.head_dim; k.F = m.ffn;
    k.V = m.vocab; k.L = m.layers; k.Smax = p.smax; k.qk_norm = m.qk_norm; k.nsplit_max = p.nsplit_max;
    k.eps = m.eps;
    k.theta = m.rope_theta;
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
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaError_t e;
    if (p.table_dirty || p.uploaded_ws != workspace) {
        std::vector<uint64_t> tab;
        if (int rc = build_table(p, ws, tab)) return rc;
        e = cudaMemcpyAsync(ws + p.ws.optab, tab.data(), tab.size() * 8, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "upload operand table");
        if (p.uploaded_ws != workspace) {
            e = cudaMemcpyAsync(ws + p.ws.queue, p.words.data(), p.words.size() * 4, cudaMemcpyHostToDevice, stream);
            if (e != cudaSuccess) return cuda_fail(e, "upload queue");
            if (!p.seq0.empty()) {
                e = cudaMemcpyAsync(ws + p.ws.seq0, p.seq0.data(), p.seq0.size() * 4, cudaMemcpyHostToDevice, stream);
                if (e != cudaSuccess) return cuda_fail(e, "upload lengths");
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
    KernelFn fn = pick_kernel(p.B);
    static thread_local int configured_smem = -1;
    if (configured_smem < p.smem_bytes) {
        for (KernelFn f : {mk_interp<1>, mk_interp<2>, mk_interp<4>, mk_interp<8>}) {
            e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        }
        configured_smem = p.smem_bytes;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, THREADS, p.smem_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    int sms = 0, smem_optin = 0;
    if (int rc = query_device(&sms, &smem_optin)) return rc;
    KParams k = base_params(p, ws);
    k.timeout_ns = timeout_ns ? timeout_ns : 200000000ull;
    k.flags = (int)flags;
    for (int s = first_step; s < first_step + num_steps; ++s) {
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
    cudaError_t e = cudaMemcpy(out, static_cast<uint8_t *>(workspace) + plan->p.ws.trace, slots * 32,
                               cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? MK_OK : cuda_fail(e, "read trace");
}

}  // extern "C"
