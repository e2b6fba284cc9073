/*
 * mk.h -- C ABI of libmk: planner and persistent decode megakernel for GB300
 * (sm_103a).  Plain C types only; device buffers are passed as 64-bit device
 * addresses (uint64_t) or void*, the CUDA stream as void* (a cudaStream_t).
 *
 * A decode step of a dense Llama-style decoder runs as ONE resident kernel
 * (one worker CTA per SM).  Each worker interprets its slice of a host-built
 * static queue of tile instructions, int32 [num_workers, lmax, 32], padded
 * with NoOp ("MegaRTP megakernel article", sections 3 and 4, KernelPlan).
 * Instructions synchronise through global event counters: a producer adds to
 * a counter after its write-back, a consumer waits for counter >= target
 * right before it reads the activation ("CMU 15-779 Lecture 7 notes",
 * section 4.1; MegaRTP section 3).  Events are derived from producer /
 * consumer grid cuts with MPK's gcd rule and fork/join lcm normalisation
 * ("MPK code walkthrough", fine-grained pipeline).  Counters are never reset
 * between steps: the target at step s is threshold x (s + 1) (monotone
 * epochs, "GEMM + AllToAll fusion post", section 2).
 *
 * Ownership: a plan owns host memory only.  Every device buffer -- weights,
 * KV caches, outputs and the workspace -- belongs to the caller.  No entry
 * point allocates or frees device memory.
 *
 * Errors: every int-returning call returns MK_OK (0) or an MK_ERR_* code;
 * mk_last_error() then describes it (thread-local).  Device-side failures
 * (a wait that timed out, an instruction that failed its checks) are recorded
 * in the workspace and reported by mk_sync_status(); the kernel never traps.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define MK_OK               0
#define MK_ERR_INVALID      1   /* malformed descriptor or argument */
#define MK_ERR_UNSUPPORTED  2   /* shape the kernels do not handle (divisibility, sizes) */
#define MK_ERR_DEADLOCK     3   /* the planner's own queue simulation did not finish */
#define MK_ERR_CUDA         4   /* a CUDA runtime call failed */
#define MK_ERR_RESIDENCY    5   /* the worker grid cannot be co-resident on the GPU */
#define MK_ERR_TIMEOUT      6   /* a device wait ran past its time budget */
#define MK_ERR_DEVICE_CHECK 7   /* an instruction failed its device-side checks */
#define MK_ERR_UNBOUND      8   /* a required binding was not set */

/* ---- opcodes (word 0 of an instruction) ---- */
#define MK_OP_NOOP     0   /* queue padding */
#define MK_OP_COUNTER  1   /* waits and signals only (explicit-graph plans) */
#define MK_OP_EMBED    2   /* h = E[token] */
#define MK_OP_QKV      3   /* RMSNorm + rows of Wq/Wk/Wv */
#define MK_OP_ATTN     4   /* q/k norm, RoPE, KV append, split-KV attention, last split merges */
#define MK_OP_O        5   /* rows of Wo + residual */
#define MK_OP_UP       6   /* RMSNorm + gate/up rows + SiLU(g) * u */
#define MK_OP_DOWN     7   /* K chunk of Wd rows, added into the residual */
#define MK_OP_LM       8   /* final RMSNorm + LM-head rows + argmax */
#define MK_OP_GLM_A0   9   /* GLM block: Add + RMSNorm + per-128 FP8 quantisation of one token row */
#define MK_OP_GLM_GEMM 10  /* GLM block: rows of an FP8 weight x FP8 activations, block scales, bf16 out (+RoPE) */
#define MK_OP_GLM_FIN  11  /* GLM block: one token's q-lora re-quantisation, RoPE and cache writes */
#define MK_OP_NORM     12  /* tensor-core plans: RMSNorm of one sequence's residual into bf16 high/low rows */
#define MK_OP_ATTN_POOL 13 /* attn_pool plans: one per worker and layer; claims the layer's attention tasks
                              (longest first) from a device counter until none is left */
#define MK_NUM_OPCODES 14

/* ---- plan modes ---- */
#define MK_MODE_MEGAKERNEL 0   /* one persistent launch per step */
#define MK_MODE_PER_OP     1   /* baseline: one launch per op, same device code */

/* ---- mk_run flags ---- */
#define MK_RUN_HOST_TOKENS 1u  /* every step reads tokens[s] (teacher forcing) */
#define MK_RUN_TRACE       2u  /* record per-instruction globaltimer stamps */
#define MK_RUN_ONE_LAUNCH  4u  /* run all num_steps steps in one cooperative launch: every worker walks its
                                  queue once per step, the monotone event epochs order the steps (no launch,
                                  ramp-up or drain between steps); megakernel plans only.  With TRACE, the
                                  stamps of a slot are those of its last step */

typedef struct mk_plan_s *mk_plan_t;

/* Dense Llama-style decoder.  Weights use the usual [out, in] row-major bf16
 * layout; norm weights are bf16 vectors. */
typedef struct {
    int layers, hidden, q_heads, kv_heads, head_dim, ffn, vocab;
    int qk_norm;        /* per-head RMSNorm of q and k before RoPE (Qwen3-style) */
    float eps;          /* RMSNorm epsilon */
    float rope_theta;   /* RoPE base, rotate-half pairing (i, i + head_dim/2) */
    int weight_fp8;     /* 1: the seven projections (Wq Wk Wv Wo Wg Wu Wd) are e4m3 codes, same
                           [out, in] layout, with one fp32 scale per 128 x 128 block (MK_BIND_SQ ..
                           MK_BIND_SD; the block-scale convention of the "MegaRTP megakernel article",
                           section 4); the embedding, LM head and norms stay bf16.  Batch 1 with
                           hidden = q_heads x head_dim = 2048, head_dim 64, ffn a multiple of 2048
                           (MK_ERR_UNSUPPORTED otherwise) */
} mk_model_desc;

typedef struct {
    int batch;             /* sequences decoded together, 1..16 (above 8: tensor-core tiles) */
    const int *seq_len0;   /* host [batch]: cached tokens per sequence before step 0 */
    int max_steps;         /* the plan serves steps 0 .. max_steps-1 */
    int cache_slots;       /* S_max of the KV cache tensors; >= seq_len0[b] + max_steps */
    int capture_hidden;    /* 1: write the residual stream after every layer (tests) */
} mk_step_desc;

typedef struct {
    int num_sms;           /* workers; 0 = all SMs of the current device */
    int smem_per_cta;      /* dynamic shared memory per CTA; 0 = device opt-in maximum */
    int mode;              /* MK_MODE_* */
    /* tile knobs, 0 = default */
    int rows_qkv, rows_o, rows_up, rows_down, kchunk_down, rows_lm, attn_split;
    int page_bytes;        /* shared-memory page size; 0 = 16384 */
    int schedule;          /* MK_SCHED_*: how tasks are dealt to workers */
    int tc_tiles;          /* GEMV tiles on tcgen05 tensor cores (128 weight rows x the batch, TMEM
                              accumulators): 0 = for batch >= 8 where the shape allows, 1 = required
                              (MK_ERR_UNSUPPORTED if the shape does not allow), -1 = never (batch <= 8).
                              GLM block plans: 0 = the FP8 GEMMs on tcgen05 tiles where M = 16, 1 =
                              required, -1 = warp-level MMA tiles */
    int attn_pool;         /* 1: device-side dispatch of the attention tasks ("CMU 15-779 Lecture 7
                              notes", section 6, JIT scheduling; "MPK code walkthrough", the
                              scheduler): every worker gets one MK_OP_ATTN_POOL instruction per
                              layer, which claims tasks from the layer's list, longest first, with an
                              atomic counter until the list is exhausted, so whoever is free takes
                              the next task; the layer's attention then waits for its whole QKV op
                              and O for every worker's pool; batch >= 2.  0 = the host deals attention tasks */
} mk_target_desc;

/* Queue assignment.  Either way tasks go to workers in one topological order,
 * so every queue is deadlock-free. */
enum {
    MK_SCHED_DEFAULT = 0,  /* MK_SCHED_TIMED */
    MK_SCHED_BYTES = 1,    /* least-loaded worker by bytes streamed so far (longest-first per range) */
    MK_SCHED_TIMED = 2     /* earliest finish under a time model of one step: a task is ready a hop
                              after the counters it waits on are met, and holds its worker for a fixed
                              cost plus its bytes at the worker's share of HBM bandwidth */
};

typedef struct {
    int num_workers, lmax, num_tasks, num_events, num_ops, num_launches;
    int num_pages, page_bytes, smem_bytes, act_bytes;
    int rows_qkv, rows_o, rows_up, rows_down, kchunk_down, rows_lm, attn_split;
    int total_slots;                 /* instruction slots over all launches of a step */
    uint64_t workspace_bytes;        /* device bytes mk_run needs */
    uint64_t scratch_offset;         /* workspace offset from which every byte is rewritten
                                        within a step before it is read (activations, partials) */
    uint64_t algorithmic_bytes_step; /* weights once + KV read + KV append, at step 0 */
    int tc_tiles;                    /* 1: the GEMV (GLM: FP8 GEMM) tiles run on tcgen05 tensor cores */
    int ksplit_qkv, ksplit_o;        /* tensor-core plans: K splits of the QKV and O tiles */
    int weight_fp8;                  /* 1: the projections stream e4m3 rows */
    int attn_table_rows;             /* attn_pool plans: rows of the attention task table, else 0 */
} mk_plan_info;

/* ---- bindings: caller-owned device buffers ---- */
#define MK_BIND_EMBED       0   /* bf16 [V, H] */
#define MK_BIND_LM_HEAD     1   /* bf16 [V, H] (may be the embedding) */
#define MK_BIND_NORM_FINAL  2   /* bf16 [H] */
#define MK_BIND_WQ          3   /* per layer, bf16 (e4m3 with weight_fp8) [Hq*D, H] */
#define MK_BIND_WK          4   /* per layer, bf16 (e4m3 with weight_fp8) [Hkv*D, H] */
#define MK_BIND_WV          5   /* per layer, bf16 (e4m3 with weight_fp8) [Hkv*D, H] */
#define MK_BIND_WO          6   /* per layer, bf16 (e4m3 with weight_fp8) [H, Hq*D] */
#define MK_BIND_WG          7   /* per layer, bf16 (e4m3 with weight_fp8) [F, H] */
#define MK_BIND_WU          8   /* per layer, bf16 (e4m3 with weight_fp8) [F, H] */
#define MK_BIND_WD          9   /* per layer, bf16 (e4m3 with weight_fp8) [H, F] */
#define MK_BIND_NORM_ATTN  10   /* per layer, bf16 [H] */
#define MK_BIND_NORM_MLP   11   /* per layer, bf16 [H] */
#define MK_BIND_QNORM      12   /* per layer, bf16 [D] (qk_norm only) */
#define MK_BIND_KNORM      13   /* per layer, bf16 [D] (qk_norm only) */
#define MK_BIND_KCACHE     14   /* bf16 [L, B, Hkv, S_max, D]; layer argument ignored */
#define MK_BIND_VCACHE     15   /* bf16 [L, B, Hkv, S_max, D]; layer argument ignored */
#define MK_BIND_TOKENS     16   /* int32 [max_steps + 1, B]: tokens[s] feeds step s */
#define MK_BIND_LOGITS     17   /* fp32 [B, V]: logits of the last step run */
#define MK_BIND_ARGMAX     18   /* uint64 [max_steps, B]: packed argmax of each step */
#define MK_BIND_HIDDEN     19   /* fp32 [L, B, H]: residual after each layer (capture_hidden) */
/* GLM pre-attention block (mk_plan_glm; M = requests * tokens rows, e4m3 = FP8 "fn"
 * bytes, weight scales fp32 [ceil(N/128), K/128] per 128 x 128 block) */
#define MK_BIND_GLM_X       20   /* bf16 [M, hidden]: block input */
#define MK_BIND_GLM_RES     21   /* bf16 [M, hidden]: residual in */
#define MK_BIND_GLM_NORM    22   /* bf16 [hidden]: RMSNorm weight */
#define MK_BIND_GLM_RES_OUT 23   /* bf16 [M, hidden]: out, x + residual */
#define MK_BIND_GLM_QA      24   /* e4m3 [M, hidden]: out, quantised RMSNorm rows */
#define MK_BIND_GLM_SA      25   /* fp32 [M, hidden/128]: out, their scales */
#define MK_BIND_GLM_W_QKVA  26   /* e4m3 [q_lora + kv_lora + rope, hidden] */
#define MK_BIND_GLM_S_QKVA  27
#define MK_BIND_GLM_W_GATE  28   /* e4m3 [gate_heads, hidden] */
#define MK_BIND_GLM_S_GATE  29
#define MK_BIND_GLM_W_IK    30   /* e4m3 [idx_dim, hidden] */
#define MK_BIND_GLM_S_IK    31
#define MK_BIND_GLM_W_QB    32   /* e4m3 [q_heads * q_head_dim, q_lora] */
#define MK_BIND_GLM_S_QB    33
#define MK_BIND_GLM_W_IQ    34   /* e4m3 [idx_heads * idx_dim, q_lora] */
#define MK_BIND_GLM_S_IQ    35
#define MK_BIND_GLM_QKVA    36   /* bf16 [M, q_lora + kv_lora + rope]: out, QKV-A */
#define MK_BIND_GLM_IK      37   /* bf16 [M, idx_dim]: out, Indexer-K before RoPE */
#define MK_BIND_GLM_QB      38   /* e4m3 [M, q_lora]: out, re-quantised q-lora */
#define MK_BIND_GLM_SB      39   /* fp32 [M, q_lora/128]: out, its scales */
#define MK_BIND_GLM_GATE    40   /* bf16 [M, gate_heads]: out, Head-Gate */
#define MK_BIND_GLM_Q       41   /* bf16 [M, q_heads, q_head_dim]: out, Q-B, last `rope` of each head roped */
#define MK_BIND_GLM_IQ      42   /* bf16 [M, idx_heads, idx_dim]: out, Indexer-Q, last `rope` roped */
#define MK_BIND_GLM_LATENT  43   /* bf16 [requests, cache_slots, kv_lora + rope]: latent cache */
#define MK_BIND_GLM_INDEX   44   /* bf16 [requests, cache_slots, idx_dim]: index cache */
/* FP8 projections (weight_fp8): fp32 block scales [ceil(N/128), K/128] of
 * the matrix [N, K] bound at MK_BIND_WQ + k, per layer */
#define MK_BIND_SQ          45
#define MK_BIND_SK          46
#define MK_BIND_SV          47
#define MK_BIND_SO          48
#define MK_BIND_SG          49
#define MK_BIND_SU          50
#define MK_BIND_SD          51
#define MK_BIND_COUNT       52

/* Packed argmax key: (order-preserving bits of the fp32 logit << 32) |
 * (0xFFFFFFFF - index); the largest key is the largest logit, lowest index on
 * ties.  mk_argmax_index() recovers the index. */
/* (The pages print no argmax layout; greedy decoding takes the usual argmax,
 * lowest index on ties, and the packed key lets every LM-head tile fold its
 * best row into one 64-bit max on the device.) */
int32_t mk_argmax_index(uint64_t key);

/* Device-side failure record, read back by mk_sync_status(). */
typedef struct {
    int32_t code;        /* MK_OK or MK_ERR_TIMEOUT / MK_ERR_DEVICE_CHECK */
    int32_t worker;      /* CTA that recorded it */
    int32_t slot;        /* queue slot of the instruction */
    int32_t event;       /* event waited on (-1 if none) */
    uint32_t observed;   /* counter value seen last */
    uint32_t needed;     /* target it waited for */
    int32_t opcode;
    int32_t role;        /* 0 loader, 1 activation loader, 2 consumers */
} mk_error_record;

/* ---- planning (host only, no CUDA calls unless num_sms/smem are 0) ---- */

/* Plan one decode step of a Llama-style decoder.  The op DAG (per layer:
 * qkv -> attention -> o -> mlp-up -> mlp-down; then the LM head; an
 * embedding task first) is expanded into tile tasks, events are derived with
 * the gcd/lcm rule, tasks are linearised so each event's successors are
 * contiguous ("MPK code walkthrough", building the SM-level DAG), placed
 * longest-first within each successor range, and dealt to workers by the
 * target's schedule (MK_SCHED_*: by default the time-model list scheduler;
 * MK_SCHED_BYTES deals by bytes).  Tile sizes follow the kernel paths: the
 * batch-1 row-per-warp GEMV (K <= 2048 with x in registers; K = 4096 in
 * pages of 8 rows with x in shared memory), 16-row tensor-core tiles when
 * every K is a multiple of 512, else split-K tiles.  Unless the target fixes
 * it, the attention split (16384 / (2 D) positions) doubles, up to 512, while
 * its tasks outnumber the workers.  The plan is checked by simulating its
 * queues.  *out receives a plan the
 * caller frees with mk_free().  Returns MK_ERR_INVALID / MK_ERR_UNSUPPORTED
 * / MK_ERR_DEADLOCK on failure (nothing allocated). */
int mk_plan(const mk_model_desc *model, const mk_step_desc *step, const mk_target_desc *target,
            mk_plan_t *out);

/* Explicit task graphs (tests of the event rules and of the device protocol):
 * ops of MK_OP_COUNTER tasks, either with MPK-style edges (gcd/lcm rule) or
 * with MegaRTP-style publications (whole / tile / tile_cover / tile_reduce,
 * "MegaRTP megakernel article", section 4, TaskGraph). */
typedef struct {
    int grid[3];
    int cost;            /* bytes, for queue balancing */
} mk_graph_op;

typedef struct {
    int prod, cons;      /* op indices */
    int out_map[3];      /* tensor dim cut by each producer grid axis, -1 = none */
    int in_map[3];       /* tensor dim cut by each consumer grid axis, -1 = none */
} mk_graph_edge;

#define MK_PAIR_WHOLE       0
#define MK_PAIR_TILE        1
#define MK_PAIR_TILE_COVER  2
#define MK_PAIR_TILE_REDUCE 3

typedef struct {
    int prod;            /* producing op */
    int first_pub;       /* first publishing task of that op (op-local index) */
    int num_pub;         /* publishing tasks: first_pub .. first_pub+num_pub-1 */
    int strategy;        /* MK_PAIR_* */
    int k;               /* producer tasks per event for cover / reduce */
    int num_cons;
    int cons[4];         /* consumer ops; their tasks are spread evenly over the events */
} mk_graph_pub;

typedef struct {
    int num_ops;
    const mk_graph_op *ops;
    int num_edges;                 /* MPK-style edges, or 0 */
    const mk_graph_edge *edges;
    int num_pubs;                  /* MegaRTP-style publications, or 0 */
    const mk_graph_pub *pubs;
    int round_robin;               /* 1: task i -> worker i mod W, in op order */
} mk_graph_desc;

int mk_plan_graph(const mk_graph_desc *graph, const mk_target_desc *target, mk_plan_t *out);

/* Plan the GLM FP8 pre-attention block ("MegaRTP megakernel article": the
 * computation of GLM-5.2-FP8 decode before sparse FlashMLA; sections 1-2 list
 * its kernels and branches).  Per step, for M = requests x tokens rows:
 *   A0   new residual = x + res (bf16); RMSNorm (weight bound, eps); per
 *        (row, 128 columns) e4m3 with scale amax / 448        (M tasks)
 *   B    QKV-A, Head-Gate, Indexer-K: FP8 GEMMs of A0's rows -- warp-level
 *        tiles: 16 weight rows per task, K split over the 8 consumer warps;
 *        tcgen05 tiles (M = 16): 128 weight rows per task, K split over
 *        tasks (fp32 sums; the last part of a row tile rounds them to bf16)
 *   FIN  per row: q-lora (QKV-A columns 0 .. q_lora-1) re-quantised per 128;
 *        kv-lora || RoPE(k_pe) -> latent cache, Indexer-K with RoPE on its
 *        last `rope` columns -> index cache, at slot pos0 + token  (M tasks)
 *   C    Q-B and Indexer-Q: FP8 GEMMs of the re-quantised q-lora, 64 weight
 *        rows per task (tcgen05 tiles: 128), RoPE on the last `rope` columns
 *        of each head
 * Every GEMM output is sum over 128-wide K blocks of a_scale * w_scale *
 * (a . w), rounded to bf16; RoPE is rotate-half with angle
 * pos * rope_theta^(-2i/rope) on those bf16 values.  Events: A0 -> B (whole),
 * QKV-A + Indexer-K -> FIN (whole), FIN -> C (whole); the next step's A0
 * waits for the previous step's last tasks.  Constraints (MK_ERR_UNSUPPORTED
 * otherwise): M <= 16; hidden, q_lora, kv_lora multiples of 128; rope = 64;
 * q_head_dim and idx_dim multiples of 64 with the roped part the last 64;
 * q_lora + kv_lora + rope, gate_heads, idx_dim multiples of 16; kv_lora
 * and idx_dim - rope at most 512, gate_heads at most 256; tcgen05 tiles
 * also M = 16 and q_lora <= 1536. */
typedef struct {
    int requests, tokens;        /* M = requests * tokens rows, token j of request r is row r * tokens + j */
    int hidden;
    int q_lora, kv_lora, rope;
    int q_heads, q_head_dim;
    int gate_heads;
    int idx_heads, idx_dim;
    int cache_slots;             /* slots per request of both caches */
    int pos0;                    /* position and cache slot of each request's first new token */
    int max_steps;
    float eps, rope_theta;
} mk_glm_desc;

int mk_plan_glm(const mk_glm_desc *glm, const mk_target_desc *target, mk_plan_t *out);

/* Sizes of a plan: workers, queue length, events, ops, pages, the workspace
 * and the algorithmic bytes of one step -- the shapes of what the plan
 * expands into: an instruction tensor, event counters and an operand pointer
 * table ("MegaRTP megakernel article", section 4, the chain OpGraph ->
 * TaskGraph -> KernelPlan).  Host only.  MK_ERR_INVALID on a null argument. */
int mk_plan_info_get(mk_plan_t plan, mk_plan_info *info);

/* Copies of the plan for inspection and bit-exact tests (caller-owned host
 * buffers, sized from mk_plan_info).  The queue is the KernelPlan's fixed
 * instruction tensor, every worker's row padded with NoOp to one length
 * ("MegaRTP megakernel article", section 4, KernelPlan: [148, 5, 32] for its
 * GLM plan); the task table is its TaskGraph.  Host only; MK_ERR_INVALID on a
 * null plan.
 *  queue      int32 [total_slots, 32]   raw instruction words; the megakernel
 *             plan's single launch is [num_workers, lmax, 32]; per-op plans
 *             concatenate one [workers_k, lmax_k, 32] block per launch
 *  task_ids   int32 [total_slots]       task id per slot, -1 = NoOp
 *  thresholds int32 [num_events]              per-step increments of each event
 *  tasks      int32 [num_tasks, MK_TASK_FIELDS]
 * Any pointer may be NULL. */
#define MK_TASK_FIELDS 24
/* tasks row: kind(opcode), layer, bx, by, bz, cost, n_waits, 3 x (event,
 * threshold, epoch_offset), n_signals, 2 x (event, increment), 4 reserved */
int mk_plan_export(mk_plan_t plan, int32_t *queue, int32_t *task_ids, int32_t *thresholds, int32_t *tasks);

/* attn_pool plans: the attention task table the pools claim from ("CMU
 * 15-779 Lecture 7 notes", section 6: the tasks a JIT scheduler hands out),
 * int32 [mk_plan_info.attn_table_rows, 32] instruction words -- per layer its
 * tasks, longest first; a pool instruction's P_TBASE / P_PT name its layer's
 * rows.  Host only; caller-owned buffer; MK_ERR_INVALID on a null argument. */
int mk_plan_export_attn_table(mk_plan_t plan, int32_t *rows);

/* Bind a caller-owned device buffer (MK_BIND_*) into the plan's operand
 * pointer table: one [num_ops, 16] uint64 row per op, shared by all of that
 * op's tile instructions, which carry only the row index ("MegaRTP megakernel
 * article", section 4, OperandPtrTable).  New buffers of the same shapes are
 * rebound without replanning; only a change of shape (batch, lengths, model)
 * needs a new plan (same section: when M or the KV length change, only the
 * host plan is regenerated).  `layer` selects the layer of per-layer bindings
 * and is ignored otherwise.  Host-only; the table is uploaded by the next
 * mk_run.  Pointers must be 16-byte aligned.  MK_ERR_INVALID on an unknown
 * binding or layer.  The library never frees a bound buffer. */
int mk_bind(mk_plan_t plan, int binding, int layer, uint64_t device_ptr);

/* Run steps first_step .. first_step+num_steps-1 asynchronously on `stream`
 * (with MK_RUN_ONE_LAUNCH in one launch: "MegaRTP megakernel article",
 * sections 4-5, and "CMU 15-779 Lecture 7 notes", section 3.1, count the
 * fixed cost a launch adds to every step):
 * a fixed grid of persistent worker CTAs, one per SM, each looping over its
 * own queue row ("MegaRTP megakernel article", section 4, Device).  Before
 * the launch the whole grid is checked for co-residency with its real block
 * and shared-memory size, and event counters are monotone epochs that are
 * not reset between steps ("GEMM + AllToAll fusion post", section 2).
 * A workspace belongs to one plan: the queue is uploaded on a plan's first
 * call with a given workspace and not checked again, so two plans must not
 * take turns on one workspace (mk_run_static handles that case for its array).
 * `workspace` is caller-allocated device memory of at least
 * info.workspace_bytes (256-byte aligned, else MK_ERR_INVALID); it holds the queue, operand table,
 * event counters, activations and the error record.  When first_step == 0
 * the counters, the error record and the ARGMAX binding are cleared.
 * One cooperative launch per step (MK_MODE_MEGAKERNEL) or per op
 * (MK_MODE_PER_OP).  Returns MK_ERR_UNBOUND if a required binding is
 * missing, MK_ERR_RESIDENCY if the grid cannot be co-resident, MK_ERR_CUDA on
 * a launch failure.  timeout_ns bounds every device wait (0 = 200 ms). */
int mk_run(mk_plan_t plan, void *workspace, size_t workspace_bytes, int first_step, int num_steps,
           uint32_t flags, uint64_t timeout_ns, void *stream);
/* (MK_RUN_ONE_LAUNCH: MK_ERR_INVALID for per-op plans.) */

/* Synchronise `stream`, read the device error record into *rec (may be
 * NULL) and return its code (MK_OK, MK_ERR_TIMEOUT, MK_ERR_DEVICE_CHECK) or
 * MK_ERR_CUDA.  (No counterpart on the pages, which name debugging tens of
 * thousands of tasks inside one kernel as an open challenge: "CMU 15-779
 * Lecture 7 notes", section 4.3.  Every device wait here is bounded; a wait
 * that runs out records where it was and the kernel drains and returns.) */
int mk_sync_status(mk_plan_t plan, void *workspace, void *stream, mk_error_record *rec);

/* Copy the event counters (uint32 [num_events]) from the workspace to host.
 * After steps 0 .. n-1 each holds n x its per-step increments (monotone
 * epochs, "GEMM + AllToAll fusion post", section 2).  Synchronous;
 * MK_ERR_CUDA on a failed copy. */
int mk_read_counters(mk_plan_t plan, void *workspace, uint32_t *out);

/* Copy the per-instruction trace to host (a per-task timeline, like the
 * profiler MPK ships: "CMU 15-779 Lecture 7 notes", section 8, item 4):
 * uint64 [total_slots, 16]:
 *   [0] opcode | task << 32      [1] consumer start      [2] activation loader: events met
 *   [3] consumer done            [4] loader issue start  [5] loader issue end
 *   [6..10] stamps of consumer thread 0 inside the op (attention: K pages ready, scores,
 *           V pages ready, P.V, partial written and arrived; tensor-core and GLM GEMM tiles:
 *           [7] pages ready, [9] K loop end, [10] reduction barrier passed; GLM A0: [9] loads
 *           and sum of squares, [10] reduction; batch-1 row-per-warp tiles: [6] x in registers,
 *           [7] first page ready, [8] pages done, [9] epilogue done)
 *   [11] activation loader: activation staged
 *   [13] activation handed to the consumers   [14] published   [15] publisher saw the slot done
 * globaltimer ns (the GPU's globaltimer advances in 256 ns steps on GB300); 0 = not stamped.
 * Only filled by runs with MK_RUN_TRACE. */
int mk_read_trace(mk_plan_t plan, void *workspace, uint64_t *out);

/* Allocation-free variant of mk_run (no counterpart on the source pages).
 *
 * For callers that must not allocate device memory themselves: code embedded
 * in a host application whose own allocator owns the whole device (a direct
 * cudaMalloc there would exceed or fragment that allocator's budget), or a
 * latency-critical loop in which cudaMalloc could block or synchronise the
 * device.  Such callers still pass every input and output through mk_bind();
 * only the workspace (queue, operand table, event counters, activations,
 * error record) moves into a fixed array inside this library.
 *
 * The array is a file-scope static device array of MK_STATIC_WORKSPACE_BYTES
 * (64 MiB); every GPU that loads the library holds it until the process exits.
 * Plans whose mk_plan_info.workspace_bytes exceed it are rejected with
 * MK_ERR_INVALID.  The first call on each device (with that device current)
 * looks up the array's device address.  Any call that uploads a queue --
 * a plan's first call, and the first call after another plan used the array
 * -- synchronises `stream` (as mk_run does for its first call on a
 * workspace), so make such calls outside any stream capture.  All calls
 * share the one array and it keeps the previous call's contents: counters
 * and the error record are cleared when first_step is 0, exactly as in
 * mk_run.  After another plan has used the array, this plan's counters are
 * gone: a call with first_step != 0 is then rejected with MK_ERR_INVALID,
 * and the plan starts again at first_step 0.  Calls whose work overlaps on the GPU
 * (other streams, other threads) race on the array -- serialise them.
 * This entry point calls no cudaMalloc, cudaFree or allocating library
 * routine.  *workspace_out (may be NULL) receives the array's device address,
 * to pass to mk_sync_status(), mk_read_counters() and mk_read_trace(). */
#define MK_STATIC_WORKSPACE_BYTES (64u << 20)
int mk_run_static(mk_plan_t plan, int first_step, int num_steps, uint32_t flags, uint64_t timeout_ns, void *stream,
                  uint64_t *workspace_out);

/* Launch probe (no counterpart call on the pages; they quote a fixed launch
 * cost beside their megakernel timings): launches an empty kernel of
 * num_workers CTAs of the interpreter's block size on `stream`, as a
 * cooperative launch when `cooperative` is non-zero (like mk_run) or a plain
 * one otherwise.  Asynchronous; the caller times it with events.  Returns
 * MK_ERR_CUDA if the launch fails. */
int mk_launch_probe(int num_workers, int cooperative, void *stream);

/* Free the plan's host memory.  NULL-safe.  Never touches device memory.
 * A plan is built once per shape and reused for every step ("CMU 15-779
 * Lecture 7 notes", section 5.1: the schedule is prepared ahead of time and
 * reused for hundreds of forward passes). */
void mk_free(mk_plan_t plan);

/* Thread-local description of the last non-zero status (no counterpart on
 * the pages: the error string of this C ABI). */
const char *mk_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
