// Host-side C ABI of libmk: planning, inspection, bindings.  No CUDA calls
// here except through query_device() when the caller leaves num_sms or
// smem_per_cta at 0.
#include <cstring>
#include <new>

#include "planner.h"

namespace mk {
int query_device(int *num_sms, int *smem_optin);  // runtime.cu

static uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

void layout_workspace(Plan &p) {
    uint64_t off = 0;
    auto take = [&](uint64_t bytes) {
        uint64_t o = off;
        off = align_up(off + std::max<uint64_t>(bytes, 1), 256);
        return o;
    };
    const int B = p.B;
    const int H = p.model.hidden, Hq = p.model.q_heads, Hkv = p.kind == PLAN_LLAMA ? p.model.kv_heads : 1;
    const int D = p.model.head_dim, F = p.model.ffn, L = p.model.layers;
    const int G = p.kind == PLAN_LLAMA ? Hq / Hkv : 1;
    size_t total_slots = 0;
    for (auto &s : p.segments) total_slots += (size_t)s.workers * s.lmax;
    p.ws.err = take(E_WORDS * 4);
    p.ws.counters = take(p.thresholds.size() * 4);
    p.ws.arrive = take(p.kind == PLAN_LLAMA ? (uint64_t)L * B * Hq * 4 : 4);
    // tensor-core plans: bf16 high/low activation rows [2 np, K] of the
    // tiles' inputs (RMSNorm output, attention output, MLP activation); they
    // sit in the region cleared at step 0, so the rows of padding sequences
    // stay zero
    if (p.tc) {
        p.ws.xn = take((uint64_t)2 * p.np * H * 2);
        p.ws.xo = take((uint64_t)2 * p.np * Hq * D * 2);
        p.ws.act16 = take((uint64_t)2 * p.np * F * 2);
    } else {
        p.ws.xn = p.ws.xo = p.ws.act16 = 0;
    }
    // GLM tensor-core plans: the fp32 sums of the K-split GEMMs, zero at step
    // 0 (FIN zeroes them again for the next step)
    p.ws.gsum[0] = p.ws.gsum[1] = p.ws.gsum[2] = 0;
    if (p.kind == PLAN_GLM && p.tc) {
        const int M = GT_N;
        p.ws.gsum[0] = take((uint64_t)M * (p.glm.q_lora + p.glm.kv_lora + p.glm.rope) * 4);
        p.ws.gsum[1] = take((uint64_t)M * p.glm.gate_heads * 4);
        p.ws.gsum[2] = take((uint64_t)M * p.glm.idx_dim * 4);
    }
    // attn_pool plans: one claim counter per step and layer, zero at step 0
    p.ws.claims = p.attn_table.empty() ? 0 : take((uint64_t)p.max_steps * std::max(1, L) * 4);
    p.ws.queue = take(p.words.size() * 4);
    p.ws.atab = p.attn_table.empty() ? 0 : take(p.attn_table.size() * 4);
    p.ws.optab = take((uint64_t)p.num_ops * N_SLOTS * 8);
    p.ws.seq0 = take((uint64_t)B * 4);
    p.ws.rope = take(p.rope_tab.size() * 4);
    if (p.kind == PLAN_LLAMA) {
        p.ws.hres = take((uint64_t)B * H * 4);
        p.ws.hmid = take((uint64_t)B * H * 4);
        p.ws.qkv = take((uint64_t)B * Hkv * (G + 2) * D * 4);
        // attention partials: per query head, split and piece of a split
        p.ws.part = take((uint64_t)B * Hq * p.nsplit_max * attn_split_pieces(G, D) * (D + 2) * 4);
        p.ws.attn_out = take((uint64_t)B * Hq * D * 4);
        p.ws.act = take((uint64_t)B * F * 4);
    } else {
        p.ws.hres = p.ws.hmid = p.ws.qkv = p.ws.part = p.ws.attn_out = p.ws.act = 0;
    }
    p.ws.tmaps = !p.tc                   ? 0
                 : p.kind == PLAN_GLM    ? take((uint64_t)GT_NTMAPS * 128)
                                         : take((uint64_t)(TC_NTMAPS_FIXED + TC_WMAPS_PER_LAYER * L + 1) * 128);
    p.ws.trace = take(total_slots * 16 * 8);
    p.ws.total = off;
}

static int finish_new_plan(Plan &p, mk_plan_t *out) {
    layout_workspace(p);
    p.bind.assign(MK_BIND_COUNT, std::vector<uint64_t>(std::max(1, p.model.layers), 0));
    auto *h = new (std::nothrow) mk_plan_s;
    if (!h) return set_error(MK_ERR_INVALID, "out of host memory");
    h->p = std::move(p);
    *out = h;
    return MK_OK;
}

static int resolve_target(const mk_target_desc *tgt, int &workers, int &smem) {
    workers = tgt ? tgt->num_sms : 0;
    smem = tgt ? tgt->smem_per_cta : 0;
    if (workers <= 0 || smem <= 0) {
        int n = 0, s = 0;
        int rc = query_device(&n, &s);
        if (rc) return rc;
        if (workers <= 0) workers = n;
        if (smem <= 0) smem = s;
    }
    if (workers <= 0 || smem <= 0) return set_error(MK_ERR_INVALID, "no workers or shared memory");
    return MK_OK;
}

}  // namespace mk

using namespace mk;

extern "C" {

int mk_plan(const mk_model_desc *model, const mk_step_desc *step, const mk_target_desc *target, mk_plan_t *out) {
    if (!out) return set_error(MK_ERR_INVALID, "out is null");
    *out = nullptr;
    mk_target_desc def{};
    if (!target) target = &def;
    int workers, smem;
    int rc = resolve_target(target, workers, smem);
    if (rc) return rc;
    Plan p;
    try {
        rc = plan_llama(model, step, target, workers, smem, p);
    } catch (const std::bad_alloc &) {
        return set_error(MK_ERR_INVALID, "out of host memory while planning");
    }
    if (rc) return rc;
    return finish_new_plan(p, out);
}

int mk_plan_graph(const mk_graph_desc *graph, const mk_target_desc *target, mk_plan_t *out) {
    if (!out) return set_error(MK_ERR_INVALID, "out is null");
    *out = nullptr;
    mk_target_desc def{};
    if (!target) target = &def;
    int workers, smem;
    int rc = resolve_target(target, workers, smem);
    if (rc) return rc;
    Plan p;
    try {
        rc = plan_graph(graph, target, workers, p);
    } catch (const std::bad_alloc &) {
        return set_error(MK_ERR_INVALID, "out of host memory while planning");
    }
    if (rc) return rc;
    p.num_pages = 2;
    p.page_bytes = 16384;
    p.act_bytes = 128;
    p.abuf_bytes = 128;
    p.red_bytes = 128;
    p.aux_bytes = 256;
    p.smem_bytes = p.abuf_bytes + 2 * p.act_bytes + p.num_pages * p.page_bytes + p.aux_bytes + MBAR_BYTES + CTRL_BYTES;
    return finish_new_plan(p, out);
}

int mk_plan_glm(const mk_glm_desc *glm, const mk_target_desc *target, mk_plan_t *out) {
    if (!out) return set_error(MK_ERR_INVALID, "out is null");
    *out = nullptr;
    mk_target_desc def{};
    if (!target) target = &def;
    int workers, smem;
    int rc = resolve_target(target, workers, smem);
    if (rc) return rc;
    Plan p;
    try {
        rc = plan_glm(glm, target, workers, smem, p);
    } catch (const std::bad_alloc &) {
        return set_error(MK_ERR_INVALID, "out of host memory while planning");
    }
    if (rc) return rc;
    return finish_new_plan(p, out);
}

int mk_plan_info_get(mk_plan_t plan, mk_plan_info *info) {
    if (!plan || !info) return set_error(MK_ERR_INVALID, "null argument");
    const Plan &p = plan->p;
    std::memset(info, 0, sizeof(*info));
    info->num_workers = p.num_workers;
    info->lmax = p.lmax;
    info->num_tasks = (int)p.tasks.size();
    info->num_events = (int)p.thresholds.size();
    info->num_ops = p.num_ops;
    info->num_launches = (int)p.segments.size();
    info->num_pages = p.num_pages;
    info->page_bytes = p.page_bytes;
    info->smem_bytes = p.smem_bytes;
    info->act_bytes = p.act_bytes;
    info->rows_qkv = p.rows_qkv;
    info->rows_o = p.rows_o;
    info->rows_up = p.rows_up;
    info->rows_down = p.rows_down;
    info->kchunk_down = p.kchunk_down;
    info->rows_lm = p.rows_lm;
    info->attn_split = p.attn_split;
    info->total_slots = (int)p.slot_task.size();
    info->workspace_bytes = p.ws.total;
    info->scratch_offset = p.kind == PLAN_LLAMA ? p.ws.hres : p.ws.total;
    info->algorithmic_bytes_step = (uint64_t)p.alg_bytes;
    info->tc_tiles = p.tc ? 1 : 0;
    info->weight_fp8 = p.w8 ? 1 : 0;
    info->attn_table_rows = (int)(p.attn_table.size() / W_WORDS);
    info->ksplit_qkv = p.ksplit_qkv;
    info->ksplit_o = p.ksplit_o;
    return MK_OK;
}

int mk_plan_export_attn_table(mk_plan_t plan, int32_t *rows) {
    if (!plan || !rows) return set_error(MK_ERR_INVALID, "null plan or buffer");
    const Plan &p = plan->p;
    if (!p.attn_table.empty()) std::memcpy(rows, p.attn_table.data(), p.attn_table.size() * 4);
    return MK_OK;
}

int mk_plan_export(mk_plan_t plan, int32_t *queue, int32_t *task_ids, int32_t *thresholds, int32_t *tasks) {
    if (!plan) return set_error(MK_ERR_INVALID, "null plan");
    const Plan &p = plan->p;
    if (queue) std::memcpy(queue, p.words.data(), p.words.size() * 4);
    if (task_ids) std::memcpy(task_ids, p.slot_task.data(), p.slot_task.size() * 4);
    if (thresholds) std::memcpy(thresholds, p.thresholds.data(), p.thresholds.size() * 4);
    if (tasks) {
        for (size_t i = 0; i < p.tasks.size(); ++i) {
            const TaskRec &t = p.tasks[i];
            int32_t *r = tasks + i * MK_TASK_FIELDS;
            std::memset(r, 0, MK_TASK_FIELDS * 4);
            r[0] = t.opcode;
            r[1] = t.layer;
            r[2] = t.bid[0];
            r[3] = t.bid[1];
            r[4] = t.bid[2];
            r[5] = (int32_t)t.cost;
            r[6] = t.nw;
            for (int k = 0; k < t.nw; ++k) {
                r[7 + 3 * k] = t.w_ev[k];
                r[8 + 3 * k] = t.w_thr[k];
                r[9 + 3 * k] = t.w_off[k];
            }
            r[16] = t.ns;
            for (int k = 0; k < t.ns; ++k) {
                r[17 + 2 * k] = t.s_ev[k];
                r[18 + 2 * k] = t.s_inc[k];
            }
            r[21] = t.op_row;
        }
    }
    return MK_OK;
}

int mk_bind(mk_plan_t plan, int binding, int layer, uint64_t ptr) {
    if (!plan) return set_error(MK_ERR_INVALID, "null plan");
    Plan &p = plan->p;
    if (binding < 0 || binding >= MK_BIND_COUNT) return set_error(MK_ERR_INVALID, "unknown binding");
    if (ptr % 16) return set_error(MK_ERR_INVALID, "device pointers must be 16-byte aligned");
    bool per_layer = (binding >= MK_BIND_WQ && binding <= MK_BIND_KNORM) || (binding >= MK_BIND_SQ && binding <= MK_BIND_SD);
    if (per_layer && (layer < 0 || layer >= (int)p.bind[binding].size()))
        return set_error(MK_ERR_INVALID, "layer out of range");
    p.bind[binding][per_layer ? layer : 0] = ptr;
    p.table_dirty = true;
    return MK_OK;
}

int32_t mk_argmax_index(uint64_t key) { return (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFu)); }

void mk_free(mk_plan_t plan) { delete plan; }

const char *mk_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
