// Device-side building blocks of the interpreter: PTX wrappers (mbarrier,
// bulk TMA copy, acquire/release counters), the shared-memory map, bounded
// waits with the abort protocol, and warp-distributed instruction decoding.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mk_internal.h"

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
DEV void red_max_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
DEV void red_relaxed_add(uint32_t *p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
DEV void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
DEV void fence_acq_rel_cta() { asm volatile("fence.acq_rel.cta;" ::: "memory"); }
DEV void st_relaxed_cta(volatile int *p, int v) {
    asm volatile("st.relaxed.cta.shared.u32 [%0], %1;" ::"r"(saddr((const void *)p)), "r"(v) : "memory");
}
DEV void st_release_cta(volatile int *p, int v) {
    asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(saddr((const void *)p)), "r"(v) : "memory");
}
DEV int ld_acquire_cta(volatile int *p) {
    int v;
    asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr((const void *)p)) : "memory");
    return v;
}
DEV int ld_relaxed_cta(volatile int *p) {
    int v;
    asm volatile("ld.relaxed.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr((const void *)p)) : "memory");
    return v;
}
// Named hardware barrier 1 over the 8 consumer warps (barrier 0 is the
// block-wide __syncthreads); it also orders their shared-memory accesses.
DEV void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS) : "memory"); }
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
// Like mbar_test, but the thread may sleep up to about `ns` nanoseconds for the phase.
DEV bool mbar_wait_hint(uint64_t *b, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(saddr(b)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
// Weight and cache rows are read once per step: evict-first keeps them from
// displacing activations, counters and the queue in L2.
DEV uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
DEV void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            saddr(dst)),
        "l"(src), "r"(bytes), "r"(saddr(bar)), "l"(pol)
        : "memory");
}
DEV void bulk_g2s_plain(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     saddr(dst)),
                 "l"(src), "r"(bytes), "r"(saddr(bar))
                 : "memory");
}
DEV void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p)); }

// Two fp32 fused multiply-adds in one instruction: acc.{lo,hi} += a.{lo,hi} * b.{lo,hi}, each rounded
// to nearest like fmaf.
DEV void fma2(uint64_t &acc, uint64_t a, uint64_t b) { asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b)); }
DEV uint64_t pack2(float lo, float hi) { return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32); }
DEV float sum2(uint64_t v) { return __uint_as_float((uint32_t)v) + __uint_as_float((uint32_t)(v >> 32)); }
// A 32-bit word of two bf16 weights as an fp32 pair (exact).
DEV uint64_t bf16x2_pair(uint32_t w) { return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)); }
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

// Transposed butterfly: V partial sums per lane -> full warp sums.  After the
// call, for V >= 32 lane l holds sums of indices l*(V/32) + j in v[j]; for
// V < 32 it holds the sum of index l / (32/V) in v[0].  V - 1 + (5 - log2 V)
// shuffles instead of 5 V.
template <int N, int OFF>
struct Bfly {
    template <int V>
    DEV static void run(float (&v)[V], int lane) {
        if constexpr (OFF > 0) {
            if constexpr (N >= 2) {
                constexpr int H = N / 2;
                const bool up = (lane & OFF) != 0;
#pragma unroll
                for (int i = 0; i < H; ++i) {
                    const float send = up ? v[i] : v[i + H];
                    const float keep = up ? v[i + H] : v[i];
                    v[i] = keep + __shfl_xor_sync(FULL, send, OFF);
                }
                Bfly<H, OFF / 2>::run(v, lane);
            } else {
                v[0] += __shfl_xor_sync(FULL, v[0], OFF);
                Bfly<1, OFF / 2>::run(v, lane);
            }
        }
    }
};

// ---------------------------------------------------------------- shared state
// The dynamic shared memory of the interpreter, one array; everything below
// addresses it through offsets so that every access compiles to a
// shared-memory instruction (a generic pointer kept in a struct would not).
extern __shared__ __align__(1024) uint8_t mk_smem[];

// Offsets into the dynamic shared memory and accessors for its regions.
struct Smem {
    uint32_t o_abuf;      // GEMV activation [B][K] (RMSNorm-ed where the op fuses it); one per
    uint32_t abuf_stride; // slot when two fit (stride in bytes), else one shared buffer (stride 0)
    uint32_t o_act0;      // slot 0; slot s at o_act0 + s * act_stride
    uint32_t act_stride;
    uint32_t o_pages;     // page ring
    uint32_t o_aux;       // op scratch (attention scores, partial outputs)
    uint32_t o_red0;      // cross-warp reduction buffers, alternating per instruction
    uint32_t red_stride;  // bytes
    uint32_t o_bars;      // full[NP], empty[NP], act_full[2], act_empty[2], consumer barrier
    uint32_t o_ctrl;      // [0] abort, [1..2] slot flags, [3] attention: last split,
                          // [8..15] consumer warp progress (instructions finished + 1)
    int num_pages;
    DEV float *abuf(int s) const { return reinterpret_cast<float *>(mk_smem + o_abuf + s * abuf_stride); }
    DEV uint8_t *act(int s) const { return mk_smem + o_act0 + s * act_stride; }
    DEV uint8_t *pages() const { return mk_smem + o_pages; }
    DEV float *aux() const { return reinterpret_cast<float *>(mk_smem + o_aux); }
    DEV float *red(int k) const { return reinterpret_cast<float *>(mk_smem + o_red0 + k * red_stride); }
    DEV uint64_t *full() const { return reinterpret_cast<uint64_t *>(mk_smem + o_bars); }
    DEV uint64_t *empty() const { return full() + num_pages; }
    DEV uint64_t *act_full() const { return full() + 2 * num_pages; }
    DEV uint64_t *act_empty() const { return full() + 2 * num_pages + 2; }
    DEV uint64_t *cbar() const { return full() + 2 * num_pages + 4; }
    DEV volatile int *ctrl() const { return reinterpret_cast<volatile int *>(mk_smem + o_ctrl); }
    // tensor-core plans: the activation ring (in the activation-buffer region),
    // its barriers, the two accumulators' barriers, the end-of-run drain, the
    // per-page release counters of attention and the TMEM base address
    DEV uint8_t *xslot(int s) const { return mk_smem + o_abuf + s * abuf_stride; }
    DEV uint64_t *xfull() const { return full() + 2 * num_pages + 5; }
    DEV uint64_t *xempty() const { return xfull() + TC_XSLOTS; }
    DEV uint64_t *accfull() const { return xempty() + TC_XSLOTS; }
    DEV uint64_t *accempty() const { return accfull() + GT_NACC; }
    DEV uint64_t *drain() const { return accempty() + GT_NACC; }
    DEV int *page_users() const { return reinterpret_cast<int *>(mk_smem + o_ctrl) + 16; }
    DEV uint32_t *tmem_slot() const { return reinterpret_cast<uint32_t *>(mk_smem + o_ctrl) + 31; }
    // attention pools: the claim ring (the loader posts claimed task indices,
    // -1 when the pool is empty), how many it posted, and how many each
    // reader took (activation loader, then the 8 consumer warps)
    DEV volatile int *claim_ring() const { return reinterpret_cast<volatile int *>(mk_smem + o_ctrl) + 32; }
    DEV volatile int *claims_posted() const { return reinterpret_cast<volatile int *>(mk_smem + o_ctrl) + 48; }
    DEV volatile int *claims_taken() const { return reinterpret_cast<volatile int *>(mk_smem + o_ctrl) + 49; }
};

constexpr int SLOT_FRESH = 1;
constexpr int CTRL_WORDS = 64;

// Error path, kept out of line so that the hot loops stay small.
static __device__ __noinline__ void raise_error_at(uint32_t *err, Smem S, int code, int slot, int event, uint32_t obs,
                                            uint32_t need, int opc, int role) {
    if (atomicCAS(&err[E_CODE], 0u, (uint32_t)code) == 0u) {
        err[E_WORKER] = blockIdx.x;
        err[E_SLOT] = (uint32_t)slot;
        err[E_EVENT] = (uint32_t)event;
        err[E_OBSERVED] = obs;
        err[E_NEEDED] = need;
        err[E_OPCODE] = (uint32_t)opc;
        err[E_ROLE] = (uint32_t)role;
    }
    atomicExch(&err[E_ABORT], 1u);
    S.ctrl()[0] = 1;
}
DEV void raise_error(const KParams &P, const Smem S, int code, int slot, int event, uint32_t obs, uint32_t need,
                     int opc, int role) {
    raise_error_at(P.err, S, code, slot, event, obs, need, opc, role);
}

DEV bool aborted_at(uint32_t *err, const Smem S) {
    if (S.ctrl()[0]) return true;
    if (ld_relaxed(&err[E_ABORT])) {
        S.ctrl()[0] = 1;
        return true;
    }
    return false;
}
DEV bool aborted(const KParams &P, const Smem S) { return aborted_at(P.err, S); }

// Bounded whole-warp waits.  Each has an inline fast path (the condition
// already holds: one test) and an out-of-line polling loop that gives up
// after the launch's timeout or on a grid-wide abort (uniform result,
// false = abort).  Keeping the loops out of line keeps the code of the hot
// paths small enough for the instruction cache.
static __device__ __noinline__ bool wait_bar_slow(uint32_t *err, uint64_t timeout_ns, Smem S, uint64_t *bar,
                                           uint32_t parity, int role, int slot, int opc) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (__all_sync(FULL, mbar_test(bar, parity))) return true;
        if ((it & 15) == 15) {
            int stop = 0;
            if (lane == 0) {
                uint64_t now = gtimer();
                if (t0 == 0) t0 = now;
                if (aborted_at(err, S)) stop = 1;
                else if (now - t0 > timeout_ns) {
                    raise_error_at(err, S, MK_ERR_TIMEOUT, slot, -1, 0, parity, opc, role);
                    stop = 1;
                }
            }
            if (__shfl_sync(FULL, stop, 0)) return false;
        }
    }
}
DEV bool warp_wait_bar(const KParams &P, const Smem S, uint64_t *bar, uint32_t parity, int role, int slot, int opc) {
    if (__all_sync(FULL, mbar_test(bar, parity))) return true;
    return wait_bar_slow(P.err, P.timeout_ns, S, bar, parity, role, slot, opc);
}

// Shared flag word >= target (acquire, CTA scope).
static __device__ __noinline__ bool wait_smem_slow(uint32_t *err, uint64_t timeout_ns, Smem S, volatile int *flag,
                                            uint32_t target, int slot, int opc) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (__all_sync(FULL, (uint32_t)ld_acquire_cta(flag) >= target)) return true;
        if ((it & 15) == 15) {
            int stop = 0;
            if (lane == 0) {
                uint64_t now = gtimer();
                if (t0 == 0) t0 = now;
                if (aborted_at(err, S)) stop = 1;
                else if (now - t0 > timeout_ns) {
                    raise_error_at(err, S, MK_ERR_TIMEOUT, slot, -1, 0, target, opc, 2);
                    stop = 1;
                }
            }
            if (__shfl_sync(FULL, stop, 0)) return false;
        }
    }
}
DEV bool warp_wait_smem(const KParams &P, const Smem S, volatile int *flag, uint32_t target, int slot, int opc) {
    if (__all_sync(FULL, (uint32_t)ld_acquire_cta(flag) >= target)) return true;
    return wait_smem_slow(P.err, P.timeout_ns, S, flag, target, slot, opc);
}

// Event counter >= target.  Polls are relaxed loads: an acquire load also
// invalidates the SM's L1, which costs the other roles their cached queue
// words (measured: a batch-1 step whose waits were all met went from 0.53 to
// 0.85 ms with acquire polls).  Once the target is seen, one acquire load of
// the counter synchronises with the publisher's release.
static __device__ __noinline__ bool wait_counter_slow(uint32_t *err, uint64_t timeout_ns, Smem S, const uint32_t *c,
                                               int ev, uint32_t target, int slot, int opc) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t v = ld_relaxed(c);
        if (__all_sync(FULL, v >= target)) return true;
        if ((it & 15) == 15) {
            int stop = 0;
            if (lane == 0) {
                uint64_t now = gtimer();
                if (t0 == 0) t0 = now;
                if (aborted_at(err, S)) stop = 1;
                else if (now - t0 > timeout_ns) {
                    raise_error_at(err, S, MK_ERR_TIMEOUT, slot, ev, v, target, opc, 1);
                    stop = 1;
                }
            }
            if (__shfl_sync(FULL, stop, 0)) return false;
        }
    }
}
DEV bool warp_wait_counter(const KParams &P, const Smem S, int ev, uint32_t target, int slot, int opc) {
    const uint32_t *c = P.counters + ev;
    bool ok = __all_sync(FULL, ld_relaxed(c) >= target);
    if (!ok) ok = wait_counter_slow(P.err, P.timeout_ns, S, c, ev, target, slot, opc);
    if (ok) (void)ld_acquire(c);  // an acquire read of the value the polls saw (or a later one)
    return ok;
}

// Barrier of the 8 consumer warps on an mbarrier: each warp reconverges,
// lane 0 arrives, the warp waits for the phase with the same bounded wait as
// every other wait (a lost arrival becomes a recorded timeout, not a hang).
// `phase` counts the barrier uses of this warp (uniform across the warp).
DEV void consumer_sync(const KParams &P, const Smem S, uint32_t &phase, bool &ab, int slot) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(S.cbar());
    if (!ab) ab = !warp_wait_bar(P, S, S.cbar(), phase & 1, 3, slot, -1);
    ++phase;
}

// Trace stamp k of slot i: traced runs only, written by consumer thread 0
// (inside ops, for a breakdown of where an instruction's time goes).
DEV void trace_stamp(const KParams &P, int i, int k) {
    if (P.trace && threadIdx.x == CONSUMER_BASE) P.trace[((size_t)blockIdx.x * P.lmax + i) * 16 + k] = gtimer();
}

DEV bool cta_aborting(const Smem S) { return __shfl_sync(FULL, (int)S.ctrl()[0], 0) != 0; }

// ---------------------------------------------------------------- instruction decoding
// A warp holds one instruction: lane k keeps word k; lanes 0..15 keep the 16
// operand-table slots of its op row, cached while consecutive instructions
// share the row.  Fields are read with shuffles (no repeated global loads).
// The queue is read ahead: while slot i runs, the words of slot i + 2 and the
// operand row of slot i + 1 are in flight, so no role waits on a round trip to
// L2 when it moves to its next instruction.
struct WIns {
    int step = 0;           // decode step of the current slot (a launch may run several)
    int w = 0;              // words of the current slot
    uint64_t orow = 0;      // operand row of the current slot
    int row = -1;
    int w1 = 0, w2 = 0;     // words of the next two slots
    uint64_t orow1 = 0;     // operand row of the next slot
    int row1 = -1;
};

DEV int F(const WIns &I, int k) { return __shfl_sync(FULL, I.w, k); }
DEV uint64_t PTR(const WIns &I, int k) {
    const uint32_t lo = __shfl_sync(FULL, (uint32_t)I.orow, k);
    const uint32_t hi = __shfl_sync(FULL, (uint32_t)(I.orow >> 32), k);
    return ((uint64_t)hi << 32) | lo;
}

// The fields the consumers need of a slot, read with independent shuffles
// issued back to back (one round of shuffle latency instead of a chain).
struct Dec {
    int opc, row, cnt, task, k0, kc, nrows, out0, snap, npg, step;
    uint64_t out, out2;  // GEMV outputs
};
DEV Dec decode(const WIns &I) {
    Dec d;
    d.opc = F(I, W_OPC);
    d.row = F(I, W_ROW);
    d.cnt = F(I, W_CNT);
    d.task = F(I, W_TASK);
    d.k0 = F(I, P_K0);
    d.kc = F(I, P_KC);
    d.nrows = F(I, P_NROWS);
    d.out0 = F(I, P_OUT0);
    d.snap = F(I, P_SNAP);
    d.npg = F(I, P_NPG);
    d.step = I.step;
    d.out = PTR(I, S_G_OUT);
    d.out2 = PTR(I, S_G_OUT2);
    return d;
}

// Lane k's word of queue slot i (all zero, i.e. a NoOp, past the queue's end).
// Slots are numbered through the launch: slot v is queue slot v % lmax of
// step v / lmax.  Lane k's word of queue slot i (in-step index), or 0 (a
// NoOp) where the launch has no such slot.
DEV int queue_word(const int32_t *q, int i, bool exists) {
    return exists ? __ldg(q + (size_t)i * W_WORDS + (threadIdx.x & 31)) : 0;
}
// In-step index of the slot `ahead` slots after in-step index i.
DEV int slot_ahead(const KParams &P, int i, int ahead) {
    int j = i + ahead;
    while (j >= P.lmax) j -= P.lmax;
    return j;
}

// Starts loading the operand row of the instruction held in `w` unless `row`
// already is that row.
DEV void load_orow(const KParams &P, int w, int &row, uint64_t &orow) {
    const int lane = threadIdx.x & 31;
    const int opc = __shfl_sync(FULL, w, W_OPC);
    const int r = __shfl_sync(FULL, w, W_ROW);
    if (opc != MK_OP_NOOP && r != row && r >= 0 && r < P.num_ops) {
        orow = lane < N_SLOTS ? __ldg(P.optab + (size_t)r * N_SLOTS + lane) : 0ull;
        row = r;
    }
}

DEV void fetch_init(WIns &I, const KParams &P, const int32_t *q) {
    const int total = P.lmax * P.nsteps;
    I.w1 = queue_word(q, 0, total > 0);
    load_orow(P, I.w1, I.row1, I.orow1);
    I.w2 = queue_word(q, slot_ahead(P, 0, 1), total > 1);
}

// Moves the warp to slot i of step I.step; slots must be visited in order
// (step by step, slot by slot).
DEV void fetch(WIns &I, const KParams &P, const int32_t *q, int i) {
    I.w = I.w1;
    I.orow = I.orow1;
    I.row = I.row1;
    I.w1 = I.w2;
    const int j = i + 2, steps_on = j >= P.lmax ? (j >= 2 * P.lmax ? 2 : 1) : 0;
    I.w2 = queue_word(q, slot_ahead(P, i, 2), I.step + steps_on < P.step + P.nsteps);
    load_orow(P, I.w1, I.row1, I.orow1);
}
// The launch-wide number of slot i of step I.step (progress words count these).
DEV int launch_slot(const KParams &P, const WIns &I, int i) { return (I.step - P.step) * P.lmax + i; }

// ---------------------------------------------------------------- attention pools
// The loader claims a pool's tasks and posts each claim (a task index, or -1
// once the pool is empty) to the worker's other roles through a ring of
// CLAIM_RING entries; claim `seq` goes to entry seq % CLAIM_RING.  The
// loader reuses an entry only after all nine readers (the activation loader,
// reader 0, and the 8 consumer warps, readers 1..8) took the claim before
// it; every wait is bounded.
DEV bool post_claim(const KParams &P, const Smem S, int seq, int value, int slot, int opc) {
    const int lane = threadIdx.x & 31;
    if (seq >= CLAIM_RING)
        for (int r = 0; r < 1 + CONSUMER_WARPS; ++r)
            if (!warp_wait_smem(P, S, S.claims_taken() + r, (uint32_t)(seq - CLAIM_RING + 1), slot, opc)) return false;
    if (lane == 0) {
        S.claim_ring()[seq % CLAIM_RING] = value;
        st_release_cta(S.claims_posted(), seq + 1);
    }
    __syncwarp();
    return true;
}
// Reader `reader` takes claim `seq` (the whole warp; false on abort or timeout).
DEV bool read_claim(const KParams &P, const Smem S, int seq, int reader, int &value, int slot, int opc) {
    const int lane = threadIdx.x & 31;
    if (!warp_wait_smem(P, S, S.claims_posted(), (uint32_t)(seq + 1), slot, opc)) return false;
    value = S.claim_ring()[seq % CLAIM_RING];
    __syncwarp();
    if (lane == 0) st_release_cta(S.claims_taken() + reader, seq + 1);  // (after the read: release)
    return true;
}
// Lane k's word of attention-table row `row` (a claimed task's instruction).
DEV int attn_table_word(const KParams &P, int row) {
    return __ldg(P.attn_table + (size_t)row * W_WORDS + (threadIdx.x & 31));
}

// Warp-uniform sanity checks of one instruction against the launch.
// Kernel instances ("flavours"): FL_GEN runs every Llama-path op; FL_GLM
// only the GLM-block ops (and holds their code), with warp-level MMA tiles,
// FL_GLMTC the same with tcgen05 tiles -- two instances, so that each holds
// only one GEMM path; FL_LEAN is the batch-1 instance for plans whose GEMV
// tiles all take the row-per-warp path and whose head_dim is 64 -- it holds
// no other GEMV or attention variant, which keeps its registers free of
// spills; FL_TC the batched decoder's tcgen05 instance.
// FL_W8 is the batch-1 instance of plans with FP8 projections (their e4m3
// row-per-warp tiles, the bf16 LM head, attention at head_dim 64).
constexpr int FL_GEN = 0, FL_GLM = 1, FL_LEAN = 2, FL_TC = 3, FL_GLMTC = 4, FL_W8 = 5;
MK_HD constexpr bool fl_glm(int fl) { return fl == FL_GLM || fl == FL_GLMTC; }
// Instances that hold the attention pools (device-side dispatch of attention
// tasks, for batches of variable-length sequences): the batched ones.
MK_HD constexpr bool fl_pools(int fl, int maxb) { return fl == FL_TC || (fl == FL_GEN && maxb > 1); }

template <int FL>
DEV bool ins_valid(const KParams &P, const WIns &I) {
    constexpr bool GLM = fl_glm(FL);
    const int opc = F(I, W_OPC);
    if (opc < 0 || opc >= MK_NUM_OPCODES) return false;
    if (opc == MK_OP_NOOP) return true;
    const int row = F(I, W_ROW);
    if (row < 0 || row >= P.num_ops) return false;
    const int cnt = F(I, W_CNT);
    const int nw = cnt & 0xff, ns = (cnt >> 8) & 0xff;
    if (nw > MAX_WAITS || ns > MAX_SIGS) return false;
    for (int i = 0; i < nw; ++i)
        if ((int)((uint32_t)F(I, W_WAIT + 2 * i) & ~WAIT_PREV_EPOCH) >= P.num_events) return false;
    for (int i = 0; i < ns; ++i)
        if ((uint32_t)F(I, W_SIG + 2 * i) >= (uint32_t)P.num_events) return false;
    constexpr bool TC = FL == FL_TC;
    const bool glm_op = opc >= MK_OP_GLM_A0 && opc <= MK_OP_GLM_FIN;
    if (GLM != glm_op && opc != MK_OP_COUNTER) return false;  // each instance runs its own ops
    if (opc == MK_OP_ATTN_POOL)
        return (FL == FL_TC || (FL == FL_GEN && P.B > 1)) && P.claims && P.attn_table && F(I, P_LAYER) >= 0 && F(I, P_LAYER) < P.L &&
               F(I, P_PT) >= 0 && F(I, P_TBASE) >= 0 && (F(I, W_CNT) & 0xff) <= MAX_WAITS;
    if (opc == MK_OP_NORM && !TC) return false;
    if (opc == MK_OP_NORM)
        return F(I, P_NB) >= 0 && F(I, P_NB) < P.B && P.H % 4 == 0 && P.H <= 8192 && P.np >= P.B;
    if (TC && opc >= MK_OP_QKV && opc <= MK_OP_LM && opc != MK_OP_ATTN) {
        // tensor-core tile: whole stages, segment matrices among the op's maps, rows within the tile
        const int kc = F(I, P_KC), k0 = F(I, P_K0), m0 = F(I, P_MAT), m1 = F(I, P_S1_MAT);
        return kc > 0 && kc % TC_KS == 0 && k0 % TC_BOX == 0 && k0 + kc <= F(I, P_KTOT) &&
               F(I, P_NPG) == kc / TC_KS && m0 >= 0 && m0 < 3 && m1 >= 0 && m1 < 3 && F(I, P_NROWS) > 0 &&
               F(I, P_NROWS) <= TC_M && F(I, P_OUT0) >= 0 && F(I, P_ROW0) >= 0 && F(I, P_S1_ROW0) >= 0 &&
               (P.np == 8 || P.np == 16) && P.B <= P.np && P.page_bytes == TC_STAGE_BYTES &&
               (opc != MK_OP_UP || F(I, P_NROWS) == TC_SEG);
    }
    if (glm_op) {
        const int M = F(I, P_GL_M), T = F(I, P_GL_T);
        if (M <= 0 || M > GLM_MAX_M || T <= 0 || T > GLM_MAX_M || F(I, P_GL_POS0) < 0) return false;
        if (opc == MK_OP_GLM_A0) return F(I, P_ROW0) >= 0 && F(I, P_ROW0) < M && P.H % 128 == 0 && P.H <= 8192;
        if (opc == MK_OP_GLM_FIN) {
            const int ql = F(I, P_GF_QLORA), kl = F(I, P_GF_KVLORA), id = F(I, P_GF_IDX), m = F(I, P_ROW0);
            return m >= 0 && m < M && ql > 0 && ql % 128 == 0 && ql <= 16 * 128 && kl >= 0 && kl % 2 == 0 &&
                   kl <= 2 * CONSUMERS && id - GLM_ROPE <= 2 * CONSUMERS && F(I, P_GF_GATE) <= CONSUMERS &&
                   id >= GLM_ROPE && id % 2 == 0 && F(I, P_GL_POS0) + T <= F(I, P_GF_SLOTS) &&
                   F(I, P_GF_QKVA_LD) >= ql + kl + GLM_ROPE && F(I, P_GF_QKVA_LD) % 4 == 0 && id % 4 == 0 &&
                   F(I, P_GF_SUMS) == (FL == FL_GLMTC ? 1 : 0) && (FL != FL_GLMTC || (P.np == GT_N && F(I, P_GF_GATE) > 0));
        }
        const int nr = F(I, P_NROWS), kc = F(I, P_KC), rpp = F(I, P_RPP);
        if ((F(I, P_GL_TCT) != 0) != (FL == FL_GLMTC)) return false;  // each instance runs its own tiles
        if (FL == FL_GLMTC) {
            // tensor-core tile: whole stages of one scale block, 128-row tiles, the plan's slot and page sizes
            const int k0 = F(I, P_K0), K = F(I, P_KTOT), nst = F(I, P_NPG), sum = F(I, P_GL_SUM);
            return P.np == GT_N && M == GT_N && P.page_bytes == GT_STAGE_BYTES && P.abuf_count >= GT_XSLOTS &&
                   P.abuf_bytes >= GT_XSLOT_BYTES && P.aux_bytes >= GT_EX_BYTES + NRED * P.red_bytes && kc > 0 &&
                   kc % GT_KS == 0 && k0 % GT_KS == 0 && K % GT_KS == 0 && k0 + kc <= K && nst == kc / GT_KS &&
                   nst <= GT_MAX_STAGES && K / GT_KS <= GT_MAX_KB && nr > 0 && nr <= GT_M && F(I, P_ROW0) >= 0 && F(I, P_ROW0) % GT_M == 0 &&
                   F(I, P_OUT0) >= 0 && F(I, P_GL_LD) >= F(I, P_OUT0) + nr && (sum == 0 || sum == 1) &&
                   (F(I, P_GL_ROPE) & ~3) == 0 && (sum == 0 || F(I, P_GL_ROPE) == 0);
        }
        if (nr != 16 && nr != 64) return false;
        if (kc <= 0 || kc % 128 || F(I, P_K0) != 0 || F(I, P_KTOT) != kc || rpp != P.page_bytes / kc || rpp < 1 ||
            F(I, P_NPG) != (nr + rpp - 1) / rpp || F(I, P_NPG) > P.num_pages)
            return false;
        if (GLM_MAX_M * (kc + 16) + GLM_MAX_M * (kc / 128) * 4 > P.abuf_bytes || GLM_MAX_M * 64 * 4 > P.red_bytes)
            return false;
        // each warp's K blocks: at most 32 (their weight scales sit one per lane)
        const int ks = CONSUMER_WARPS / (nr / 8);
        if ((kc / 128 + ks - 1) / ks > 32) return false;
        return F(I, P_GL_LD) >= F(I, P_OUT0) + nr && F(I, P_OUT0) >= 0 && (F(I, P_GL_ROPE) == 0 || nr == 64);
    }
    if (FL != FL_W8 && F(I, P_W8) != 0) return false;  // FP8 tiles run in their instance only
    if (FL == FL_W8 && opc >= MK_OP_QKV && opc <= MK_OP_LM && opc != MK_OP_ATTN && F(I, P_W8) != 0) {
        // FP8 tile: pages of 32 rows of K = 2048 (MLP-up 16 gate + 16 up), one page of up to 32 rows
        // (O 16, MLP-up exactly 16 gate rows) or whole pages, rows in one 128-row block
        if (P.B != 1 || opc == MK_OP_LM || F(I, P_W8) != 1) return false;
        const int nrows = F(I, P_NROWS), npg = F(I, P_NPG), row0 = F(I, P_ROW0);
        const bool up = opc == MK_OP_UP;
        const int rows = (up ? 2 : 1) * nrows;
        if (F(I, P_KC) != W8_K || P.page_bytes != W8_ROWS * W8_K || F(I, P_RPP) != W8_ROWS || nrows <= 0 ||
            npg != (rows + W8_ROWS - 1) / W8_ROWS || npg > 64 || row0 < 0 || row0 / 128 != (row0 + nrows - 1) / 128)
            return false;
        if (up) return nrows % 16 == 0;
        if (opc == MK_OP_O) return npg == 1 && nrows <= RESID_ROWS;
        return npg == 1 || nrows > W8_ROWS * (npg - 1);
    }
    if (opc >= MK_OP_QKV && opc <= MK_OP_LM && opc != MK_OP_ATTN) {
        const int nrows = F(I, P_NROWS), kc = F(I, P_KC);
        // batch > 4 holds 8 rows x 8 sequences in registers, except on the
        // tensor-core path (K slices of 64 per warp, tile rows in two pages of 8+)
        const bool mma = kc % (64 * CONSUMER_WARPS) == 0 && F(I, P_NPG) <= 2 && F(I, P_RPP) >= 8;
        const int rmax = P.B > 4 && !mma ? 8 : MAX_TILE_ROWS;
        const int total = opc == MK_OP_UP ? 2 * nrows : nrows;
        // more rows only as 2 or 4 pages of 16 rows on the batch-1 row-per-warp path
        const bool pages16 = P.B == 1 && kc % 256 == 0 && kc <= 2048 && P.page_bytes == 32 * kc;
        if (nrows <= 0) return false;
        if (opc == MK_OP_UP && nrows > 8 && nrows % 8) return false;  // gate / up rows go to pages in groups of 8
        // more rows only as whole 16-row pages (MLP-up: 8 gate + 8 up) on the batch-1 row-per-warp path
        if (total > rmax && !(pages16 && opc != MK_OP_O && F(I, P_NPG) <= 64 &&
                              (opc == MK_OP_UP ? 2 * nrows == 16 * F(I, P_NPG)
                                               : nrows > 16 * (F(I, P_NPG) - 1) && nrows <= 16 * F(I, P_NPG))))
            return false;
        if (kc <= 0 || kc % 8 || 2 * kc > P.page_bytes || kc * P.B * 4 > P.abuf_bytes) return false;
        const int rpp = F(I, P_RPP);
        const int rows = (opc == MK_OP_UP ? 2 : 1) * nrows;
        if (rpp != P.page_bytes / (2 * kc) || F(I, P_NPG) != (rows + rpp - 1) / rpp) return false;
        // x chunks per consumer thread x batch template must fit the kernel's registers
        const int maxb = P.B <= 1 ? 1 : P.B <= 2 ? 2 : P.B <= 4 ? 4 : 8;
        const int nch = (kc / 8 + CONSUMERS - 1) / CONSUMERS;
        if (nch * maxb > 8 || nch > 4) return false;
    }
    if (opc == MK_OP_ATTN) {
        const int T = F(I, P_T);
        if (T <= 0 || T > 512 || F(I, P_B) >= P.B || F(I, P_G) >= P.Hkv || F(I, P_SPLIT) >= P.nsplit_max) return false;
        if (attn_pages(T, P.D, P.page_bytes) > 4) return false;  // a split spans at most 4 pages of K (and of V)
    }
    return true;
}

// Position in the page ring: page index and the parity of its current use.
struct RingPos {
    uint32_t p = 0, ph = 0;
    DEV void next(int num_pages) {
        if (++p == (uint32_t)num_pages) {
            p = 0;
            ph ^= 1;
        }
    }
    DEV void set(uint32_t ring, int num_pages) {
        p = ring % num_pages;
        ph = (ring / num_pages) & 1;
    }
};

struct Seg {
    const uint8_t *src;
    int rows;
    int row_bytes;
    long long stride;
};

DEV int attn_pos(const KParams &P, const WIns &I) {
    const int32_t *seq0 = reinterpret_cast<const int32_t *>(PTR(I, S_AT_SEQ0));
    return __ldg(seq0 + F(I, P_B)) + I.step;
}
DEV int attn_cached_rows(const WIns &I, int pos) { return max(0, min(F(I, P_T), pos - F(I, P_T0))); }

// Weight / cache rows streamed by the loader for one instruction.  Loader and
// consumers derive the same segments and walk the same page ring.
template <int FL>
DEV int describe(const KParams &P, const WIns &I, Seg &s0, Seg &s1) {
    constexpr bool GLM = fl_glm(FL);
    const int opc = F(I, W_OPC);
    if (opc == MK_OP_QKV || opc == MK_OP_O || opc == MK_OP_DOWN || opc == MK_OP_LM || opc == MK_OP_UP) {
        const long long ktot = F(I, P_KTOT);
        const int eb = FL == FL_W8 && F(I, P_W8) != 0 ? 1 : 2;  // bytes per weight: e4m3 or bf16
        const long long off = ((long long)F(I, P_ROW0) * ktot + F(I, P_K0)) * eb;
        const int slot = opc == MK_OP_QKV ? S_QKV_WQ + F(I, P_MAT)
                       : opc == MK_OP_O   ? S_O_W
                       : opc == MK_OP_DOWN ? S_DN_W
                       : opc == MK_OP_LM  ? S_LM_W
                                          : S_UP_WG;
        s0.src = reinterpret_cast<const uint8_t *>(PTR(I, slot)) + off;
        s0.rows = F(I, P_NROWS);
        s0.row_bytes = F(I, P_KC) * eb;
        s0.stride = ktot * eb;
        if (opc != MK_OP_UP) return 1;
        s1 = s0;
        s1.src = reinterpret_cast<const uint8_t *>(PTR(I, S_UP_WU)) + off;
        return 2;
    }
    if (GLM && opc == MK_OP_GLM_GEMM) {
        const long long ktot = F(I, P_KTOT);
        s0.src = reinterpret_cast<const uint8_t *>(PTR(I, S_GG_W)) + (long long)F(I, P_ROW0) * ktot;
        s0.rows = F(I, P_NROWS);
        s0.row_bytes = F(I, P_KC);
        s0.stride = ktot;
        return 1;
    }
    if (opc == MK_OP_ATTN) {
        const int pos = attn_pos(P, I);
        const int n = attn_cached_rows(I, pos);
        const long long base =
            (((long long)F(I, P_B) * P.Hkv + F(I, P_G)) * P.Smax + F(I, P_T0)) * (long long)P.D * 2;
        s0.src = reinterpret_cast<const uint8_t *>(PTR(I, S_AT_K)) + base;
        s0.rows = n;
        s0.row_bytes = P.D * 2;
        s0.stride = P.D * 2;
        s1 = s0;
        s1.src = reinterpret_cast<const uint8_t *>(PTR(I, S_AT_V)) + base;
        return 2;
    }
    return 0;
}

}  // namespace mk
