// Plan data structures shared by planner.cpp, api.cpp and runtime.cu.
#pragma once
#include <stdint.h>

#include <string>
#include <vector>

#include "mk_internal.h"

namespace mk {

enum { PLAN_LLAMA = 0, PLAN_GRAPH = 1, PLAN_GLM = 2 };

struct TaskRec {
    int opcode = MK_OP_COUNTER;
    int op_row = 0;
    int layer = -1;
    int bid[3] = {0, 0, 0};
    int64_t cost = 0;
    int nw = 0, ns = 0;
    int w_ev[MAX_WAITS] = {0, 0, 0}, w_thr[MAX_WAITS] = {0, 0, 0}, w_off[MAX_WAITS] = {0, 0, 0};
    int s_ev[MAX_SIGS] = {0, 0}, s_inc[MAX_SIGS] = {0, 0};
    int32_t payload[W_WORDS - W_P] = {};
};

struct EventRec {
    int ntrig, first, last;
};

struct Segment {
    int workers = 0, lmax = 0;
    int64_t word_offset = 0, slot_offset = 0;
};

struct Plan {
    int kind = PLAN_GRAPH;
    int mode = MK_MODE_MEGAKERNEL;
    mk_model_desc model{};
    mk_glm_desc glm{};           // PLAN_GLM
    std::vector<float> rope_tab;  // PLAN_GLM: (cos, sin) [tokens][32] of each new position
    std::vector<int32_t> attn_table;  // attn_pool plans: the attention task instructions [L * tasks][32]
    int num_workers = 0, B = 1, max_steps = 1, smax = 0;
    bool capture = false;
    std::vector<int> seq0;
    int rows_qkv = 0, rows_o = 0, rows_up = 0, rows_down = 0, kchunk_down = 0, rows_lm = 0, attn_split = 0;
    int schedule = MK_SCHED_BYTES;  // MK_SCHED_BYTES or MK_SCHED_TIMED
    bool lean = false;  // batch 1, head_dim 64, every GEMV tile on the row-per-warp path: the lean kernel instance
    bool tc = false;    // GEMV tiles on tcgen05 tensor cores (the tensor-core kernel instance)
    bool w8 = false;    // FP8 projections (the batch-1 FP8 kernel instance)
    int np = 0;         // tensor-core plans: batch padded to 8 or 16
    int ksplit_qkv = 1, ksplit_o = 1;
    int glm_ksplit = 1;  // GLM tensor-core plans: K parts of the first GEMMs
    int page_bytes = 16384, act_bytes = 128, abuf_bytes = 128, abuf_count = 1, aux_bytes = 256, red_bytes = 128, num_pages = 2, smem_bytes = 0,
        nsplit_max = 1;
    std::vector<TaskRec> tasks;
    std::vector<int32_t> thresholds;
    std::vector<EventRec> events;
    int num_ops = 0;
    std::vector<int> op_kind, op_layer;
    std::vector<int> op_aux;  // NORM ops: 0 attention norm, 1 MLP norm, 2 final norm
    std::vector<Segment> segments;
    std::vector<int32_t> words;      // all segments' instruction words
    std::vector<int32_t> slot_task;  // task id per slot, -1 = NoOp
    int lmax = 0;
    int64_t alg_bytes = 0;
    // bindings: [binding][layer]
    std::vector<std::vector<uint64_t>> bind;
    // workspace layout (byte offsets) and upload state
    struct {
        uint64_t err, counters, arrive, queue, optab, seq0, rope, hres, hmid, qkv, part, attn_out, act, trace, total;
        uint64_t xn, xo, act16, tmaps;  // tensor-core plans: bf16 high/low activations, tensor maps
        uint64_t claims, atab;          // attn_pool plans: claim counters [max_steps][L], the task table
        uint64_t gsum[3];               // GLM tensor-core plans: fp32 sums of the K-split GEMMs
                                        // (QKV-A, Head-Gate, Indexer-K)
    } ws{};
    void *uploaded_ws = nullptr;
    bool table_dirty = true;
};

int set_error(int code, const std::string &msg);
extern thread_local std::string g_last_error;

int plan_llama(const mk_model_desc *m, const mk_step_desc *s, const mk_target_desc *tgt, int num_workers,
               int smem_per_cta, Plan &p);
int plan_graph(const mk_graph_desc *g, const mk_target_desc *tgt, int num_workers, Plan &p);
int plan_glm(const mk_glm_desc *g, const mk_target_desc *tgt, int num_workers, int smem_per_cta, Plan &p);
void layout_workspace(Plan &p);

}  // namespace mk

struct mk_plan_s {
    mk::Plan p;
};
