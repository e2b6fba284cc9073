// Internal definitions shared by the planner (planner.cpp), the host launch
// code and the interpreter kernel (interp.cu).  Not part of the C ABI.
#pragma once
#include <stdint.h>

#include "../../include/mk.h"

namespace mk {

// ---- instruction word layout: 32 x int32 = 128 bytes ---------------------
// (opcode, operand row, wait/signal counts, waits (event, threshold),
//  signals (event, increment), payload with tile coordinates; no absolute
//  addresses -- "MegaRTP megakernel article", section 4, KernelPlan)
enum : int {
    W_OPC = 0,      // opcode
    W_ROW = 1,      // operand-table row
    W_CNT = 2,      // n_waits | n_signals << 8
    W_TASK = 3,     // task id (traces, error records)
    W_WAIT = 4,     // 3 x {event | 0x80000000 if waiting one epoch back, threshold}
    W_SIG = 10,     // 2 x {event, increment}
    W_P = 14,       // payload, 18 words
    W_WORDS = 32,
};
constexpr int MAX_WAITS = 3;
constexpr int MAX_SIGS = 2;
constexpr uint32_t WAIT_PREV_EPOCH = 0x80000000u;

// GEMV payload (QKV, O, UP, DOWN, LM)
enum : int {
    P_ROW0 = W_P + 0,   // first row in the source matrix
    P_NROWS = W_P + 1,  // rows in the tile (UP: gate rows; the tile also holds as many up rows)
    P_K0 = W_P + 2,     // first column of the K chunk
    P_KC = W_P + 3,     // K chunk length
    P_OUT0 = W_P + 4,   // first output index (QKV: row of the group-major qkv buffer)
    P_MAT = W_P + 5,    // QKV: 0 = Wq, 1 = Wk, 2 = Wv
    P_SNAP = W_P + 6,   // 1 + layer whose residual the activation loader snapshots, or 0
    P_KTOT = W_P + 7,   // row length (elements) of the source matrix
    P_RPP = W_P + 8,    // weight rows per page: page bytes / (2 * K chunk)
    P_NPG = W_P + 9,    // pages of the tile: ceil(rows of all segments / P_RPP)
};
// Tensor-core GEMV tiles (batch 8..16): 128 weight rows in two segments of
// 64 (P_ROW0 = first row of segment 0 in matrix P_MAT, P_S1_ROW0 / P_S1_MAT
// of segment 1; matrices index the op's tensor-map slots S_T_W0 + m), K
// range [P_K0, P_K0 + P_KC) of a row of P_KTOT elements, P_NPG = stages of
// 128 K columns, P_OUT0 = first output row, P_NROWS = rows stored (< 128 only
// for a last partial tile).
enum : int {
    P_S1_ROW0 = W_P + 10,
    P_S1_MAT = W_P + 11,
};
// Batch-1 GEMV tiles of FP8 projections: e4m3 rows (K bytes) with one fp32
// scale per 128 x 128 block; the tile's rows lie in one 128-row block
enum : int {
    P_W8 = W_P + 12,    // 1: the tile's weights are e4m3
};
constexpr int W8_K = 2048;          // K of every FP8 projection tile (row bytes)
constexpr int W8_ROWS = 32;         // e4m3 rows of K = 2048 per 64 KB page
// NORM payload (tensor-core plans)
enum : int {
    P_NB = W_P + 0,      // sequence
    P_NZERO = W_P + 1,   // 1: also zero that sequence's qkv row (the QKV tiles split K and add)
    P_NSNAP = W_P + 2,   // 1 + layer whose residual is captured, or 0
};
// ATTN payload
enum : int {
    P_G = W_P + 0, P_B = W_P + 1, P_SPLIT = W_P + 2, P_T0 = W_P + 3, P_T = W_P + 4,
    P_NSPLIT = W_P + 5, P_LAYER = W_P + 6,
    P_ATHR = W_P + 7,   // threshold of the event the layer's attention tasks signal
};
// ATTN_POOL payload (P_LAYER as above): the layer's attention tasks are rows
// P_TBASE .. P_TBASE + P_PT - 1 of the attention task table, each an ATTN
// instruction (no waits or signals of its own: the pool slot carries them)
enum : int {
    P_PT = W_P + 8,
    P_TBASE = W_P + 9,
};
constexpr int CLAIM_RING = 16;   // claimed task indices in flight between a worker's roles

// GLM block payload.  GEMM tiles use the GEMV fields P_ROW0 (first weight
// row), P_NROWS (16 or 64), P_K0 (0), P_KC = P_KTOT (K, bytes = elements of
// e4m3), P_OUT0 (first output column), P_RPP, P_NPG, plus:
enum : int {
    P_GL_LD = W_P + 10,    // output row stride (elements)
    P_GL_ROPE = W_P + 11,  // GEMM: 1 if the tile's 64 columns are a RoPE slice
    P_GL_M = W_P + 12,     // token rows
    P_GL_T = W_P + 13,     // tokens per request
    P_GL_POS0 = W_P + 14,  // position of each request's first new token
    // A0 / FIN: P_ROW0 is the token row; FIN also:
    P_GF_QLORA = W_P + 1, P_GF_KVLORA = W_P + 2, P_GF_IDX = W_P + 3, P_GF_SLOTS = W_P + 4, P_GF_QKVA_LD = W_P + 5,
    P_GF_SUMS = W_P + 6,   // FIN, tensor-core plans: 1 = the first GEMMs left fp32 sums; FIN rounds them
                           // to bf16 (QKV-A, Indexer-K, Head-Gate outputs) and zeroes them
    P_GF_GATE = W_P + 7,   // FIN: Head-Gate width
    // tensor-core GEMM tiles (128 weight rows x the 16 token rows, see
    // dev_glm_tc.cuh): P_ROW0 first weight row, P_NROWS rows stored (<= 128),
    // P_K0 / P_KC the K range (multiples of 128), P_KTOT = K, P_NPG stages
    // of 128 K, P_GL_ROPE bit j = rows 64 j .. 64 j + 63 are a RoPE slice,
    // and:
    P_GL_TCT = W_P + 15,     // 1: a tensor-core tile
    P_GL_SUM = W_P + 16,     // 1: add the tile's fp32 part into the GEMM's sums (K split over tiles;
                             // FIN rounds them), 0: store the bf16 outputs (with RoPE)
};
constexpr int GLM_MAX_M = 16;     // token rows of the GLM block (A fragments of m16n8k32)
constexpr int GLM_ROPE = 64;      // width of a RoPE slice
// GLM tensor-core tiles: tcgen05.mma kind::f8f6f4 (e4m3 x e4m3, fp32
// accumulators in TMEM), M = 128 weight rows, N = 16 token rows, one stage =
// one 128-wide K block of the block scales.
constexpr int GT_M = 128;                        // weight rows per tile
constexpr int GT_N = 16;                         // token rows (the MMA's N)
constexpr int GT_KS = 128;                       // K per stage (e4m3 bytes of a row)
constexpr int GT_STAGE_BYTES = GT_M * GT_KS;     // 16 KB of weights per stage = one page
constexpr int GT_XSTAGE_BYTES = GT_N * GT_KS;    // 2 KB of activation codes per stage
constexpr int GT_KSTEP = 32;                     // K of one kind::f8f6f4 MMA
constexpr int GT_MAX_STAGES = 12;                // stages of one tile (its activation is staged whole)
constexpr int GT_NACC = 4;                       // accumulators in flight (one per stage)
constexpr int GT_ACC_COLS = 16;                  // TMEM columns of one accumulator
constexpr int GT_TMEM_COLS = GT_NACC * GT_ACC_COLS;
constexpr int GT_XSLOTS = 1;                     // activation slots: a worker's tiles are one per GEMM level,
                                                 // and the levels are an event apart
constexpr int GT_MAX_KB = 64;                    // K blocks of a GEMM's activation (hidden <= 8192)
constexpr int GT_XSLOT_BYTES = GT_MAX_STAGES * GT_XSTAGE_BYTES + GT_N * GT_MAX_KB * 4;  // codes, then all scales
constexpr int GT_EX_BYTES = GT_M * GT_N * 4;     // RoPE exchange of the epilogue warps
constexpr int GT_NTMAPS = 7;                     // 5 weight matrices, 2 activations (A0 codes, FIN codes)

// ---- operand table slots (16 x uint64 per op row) ------------------------
enum : int {
    // EMBED
    S_EMB_W = 0, S_EMB_H = 1, S_EMB_TOK = 2, S_EMB_KEYS = 3,
    // QKV
    S_QKV_WQ = 0, S_QKV_WK = 1, S_QKV_WV = 2, S_QKV_NORM = 3, S_QKV_H = 4, S_QKV_OUT = 5, S_QKV_HIST = 6,
    // ATTN
    S_AT_K = 0, S_AT_V = 1, S_AT_QKV = 2, S_AT_QN = 3, S_AT_KN = 4, S_AT_PART = 5, S_AT_OUT = 6,
    S_AT_ARRIVE = 7, S_AT_SEQ0 = 8,
    // O
    S_O_W = 0, S_O_IN = 1, S_O_HRES = 2, S_O_HMID = 3,
    // UP
    S_UP_WG = 0, S_UP_WU = 1, S_UP_NORM = 2, S_UP_H = 3, S_UP_OUT = 4,
    // DOWN
    S_DN_W = 0, S_DN_IN = 1, S_DN_HRES = 2,
    // LM
    S_LM_W = 0, S_LM_NORM = 1, S_LM_H = 2, S_LM_LOGITS = 3, S_LM_KEYS = 4, S_LM_HIST = 5,
    // GLM A0 / GEMM / FIN
    S_GA_X = 0, S_GA_RES = 1, S_GA_NORM = 2, S_GA_RES_OUT = 3, S_GA_QA = 4, S_GA_SA = 5,
    S_GG_W = 0, S_GG_SW = 1, S_GG_XQ = 2, S_GG_XS = 3, S_GG_OUT = 4, S_GG_ROPE = 5,
    // tensor-core GEMM tiles: weight and activation tensor maps, fp32 sums [16][N] of K-split tiles
    S_GG_TW = 6, S_GG_TX = 7, S_GG_FSUM = 8,
    S_GF_QKVA = 0, S_GF_IK = 1, S_GF_QB = 2, S_GF_SB = 3, S_GF_LAT = 4, S_GF_IDX = 5, S_GF_ROPE = 6,
    S_GF_FQKVA = 7, S_GF_FIK = 8, S_GF_FGATE = 9, S_GF_GATE = 10,  // tensor-core plans: the sums, the gate output
    // NORM (tensor-core plans): residual fp32 [B, H], weight, bf16 high/low rows [2 NP, H],
    // qkv to zero, hidden capture
    S_N_H = 0, S_N_W = 1, S_N_XN = 2, S_N_QKV = 3, S_N_HIST = 4,
    // tensor-core GEMV tiles: the weight tensor maps of the op (QKV: Wq, Wk, Wv; UP: Wg, Wu;
    // else the op's matrix) and the input activation's tensor map (bf16 high/low rows)
    S_T_W0 = 7, S_T_W1 = 8, S_T_W2 = 9, S_T_X = 10,
    // FP8 GEMV tiles: block scales of the op's matrices (QKV: q, k, v; UP: gate, up; else the matrix)
    S_W8_S0 = 11, S_W8_S1 = 12, S_W8_S2 = 13,
    // every GEMV op: its output (QKV: qkv, O: residual, UP: activation, DOWN:
    // residual, LM: logits) and second output (O: mid residual, LM: argmax keys)
    S_G_OUT = 14, S_G_OUT2 = 15,
    N_SLOTS = 16,
};

// ---- error record layout in the workspace (uint32 words) -----------------
enum : int {
    E_CODE = 0, E_WORKER = 1, E_SLOT = 2, E_EVENT = 3, E_OBSERVED = 4, E_NEEDED = 5,
    E_OPCODE = 6, E_ROLE = 7, E_ABORT = 8, E_WORDS = 64,
};

// ---- kernel parameters ---------------------------------------------------
struct KParams {
    const int32_t *queue;   // this launch's [num_workers, lmax, 32]
    const uint64_t *optab;  // [num_ops, 16]
    uint32_t *counters;     // [num_events]
    uint32_t *err;          // error record
    uint64_t *trace;        // [num_workers, lmax, 4] or null
    uint64_t timeout_ns;
    int lmax, num_workers, num_ops, num_events;
    int step, flags;        // first step of this launch, MK_RUN_* flags
    int nsteps;             // steps this launch runs (the queue is walked once per step)
    int num_pages, page_bytes, act_bytes, abuf_bytes, abuf_count, aux_bytes, red_bytes, smem_bytes;
    int B, H, Hq, Hkv, D, F, V, L, Smax, qk_norm, nsplit_max;
    uint32_t *claims;       // attn_pool plans: task claim counters [max_steps][L]
    const int32_t *attn_table;  // attn_pool plans: attention task instructions [tasks][32]
    int np;                 // tensor-core plans: the batch padded to 8 or 16 (N = 2 np), else 0;
                            // GLM plans: 16 with tensor-core GEMM tiles, else 0
    float eps, theta;
};

// Warp roles: warpgroup 0 holds the loader (warp 0), the activation loader
// (1), the publisher (2) and one idle warp (3); warpgroups 1 and 2 are the 8
// consumer warps (warp w of them sits on TMEM lane quarter w % 4).
constexpr int CONSUMER_WARPS = 8;
constexpr int CONSUMERS = CONSUMER_WARPS * 32;
constexpr int FIRST_CONSUMER_WARP = 4;
constexpr int CONSUMER_BASE = FIRST_CONSUMER_WARP * 32;  // thread index of consumer thread 0
constexpr int THREADS = CONSUMERS + CONSUMER_BASE;
constexpr int PUBLISHER_WARP = 2;
constexpr int RESID_ROWS = 16;           // residual slice staged per slot for O tiles
constexpr int MAX_TILE_ROWS = 16;
constexpr int NRED = 4;                  // cross-warp reduction buffers, used round robin by GEMV tiles

// Tensor-core GEMV tiles (batch 8..16; see dev_tc.cuh).
constexpr int TC_M = 128;          // weight rows per tile (two segments of 64)
constexpr int TC_SEG = 64;         // rows per segment
constexpr int TC_KS = 128;         // K columns per stage
constexpr int TC_BOX = 64;         // K columns per TMA box (128 bytes of bf16)
constexpr int TC_STAGE_BYTES = TC_M * TC_KS * 2;   // 32 KB of weights per stage = one page
constexpr int TC_KSTEP = 16;       // K of one kind::f16 MMA
constexpr int TC_ACC_COLS = 32;    // TMEM columns of one accumulator (N <= 32)
constexpr int TC_TMEM_COLS = 2 * TC_ACC_COLS;
constexpr int TC_XSLOTS = 4;       // activation ring slots
constexpr int TC_EPI_WARPS = 4;    // consumer warps 0..3 read the accumulator
constexpr int TC_MMA_WARP = 4;     // consumer warp whose lane 0 issues the MMAs
constexpr int TC_MAXB = 16;        // sequences of a tensor-core plan
constexpr int TC_NTMAPS_FIXED = 3; // tensor maps of the three activations (norm out, attention out, MLP act)
constexpr int TC_WMAPS_PER_LAYER = 7;  // Wq, Wk, Wv, Wo, Wg, Wu, Wd

#ifdef __CUDACC__
#define MK_HD __host__ __device__
#else
#define MK_HD
#endif
// Pages of the ring an attention instruction takes: ceil(T / rows per page)
// pages of K rows, then as many of V rows, however many rows are cached yet
// (the others stay empty), so that the count is fixed by the plan.
// Attention partials a split leaves per query head: one per token part of
// the per-head form (head_dim 64), one of the grouped form (head_dim 128).
MK_HD inline int attn_split_pieces(int G, int D) { return D == 64 ? CONSUMER_WARPS / G : 1; }
MK_HD inline int attn_pages(int T, int D, int page_bytes) {
    return (T + page_bytes / (2 * D) - 1) / (page_bytes / (2 * D));
}
// Bytes of one activation stage of a tensor-core tile: 2 np rows (high
// parts, then low parts) of TC_KS bf16 values.
MK_HD inline int tc_xstage_bytes(int np) { return 2 * np * TC_KS * 2; }

}  // namespace mk

namespace mk {
// ---- shared-memory budget (bytes); the kernel lays memory out in this order:
// two activation slots, the page pool, an op scratch area, mbarriers, flags.
inline int round_up(int x, int a) { return (x + a - 1) / a * a; }
inline int red_bytes(int B) { return CONSUMER_WARPS * MAX_TILE_ROWS * B * 4; }
// attention scratch: each consumer warp's scores over its part of a split
inline int attn_aux_bytes(int G, int T, int D) { return (CONSUMER_WARPS * ((T + CONSUMER_WARPS / G - 1) / (CONSUMER_WARPS / G)) + 32 + 0 * D) * 4; }
constexpr int MBAR_BYTES = 512;    // up to 64 mbarriers
constexpr int CTRL_BYTES = 256;   // 64 flag words
constexpr int MAX_PAGES = 26;      // 2 * MAX_PAGES + 5 mbarriers must fit MBAR_BYTES
constexpr int MAX_PAGES_TC = 16;   // tensor-core plans: 2 * pages + 22 mbarriers
}  // namespace mk
