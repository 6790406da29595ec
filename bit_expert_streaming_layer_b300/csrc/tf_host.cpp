// Host-side parts of libtf.so that need no GPU: error reporting, the packed
// expert layout, the packer and the per-layer LFU expert-cache metadata.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "tf_internal.h"

namespace tf {

static thread_local std::string g_last_error;

void set_error(const char* fmt, ...) {
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
}

void clear_error() { g_last_error.clear(); }

tf_status fail(tf_status s, const char* fmt, ...) {
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

bool expert_layout(int H, int I, ExpertLayout* L) {
    if (H <= 0 || I <= 0 || H % TF_GROUP || I % TF_GROUP) return false;
    const size_t h = (size_t)H, i = (size_t)I;
    L->H = H;
    L->I = I;
    L->gu_codes = 0;
    L->gu_sb = L->gu_codes + 2 * i * (h / 2);            // 2I rows of H/2 bytes
    L->d_codes = L->gu_sb + 2 * i * (h / TF_GROUP) * 4;  // 2I rows x H/64 groups x {s,b}
    L->d_sb = L->d_codes + h * (i / 2);                  // H rows of I/2 bytes
    L->payload = L->d_sb + h * (i / TF_GROUP) * 4;       // H rows x I/64 groups x {s,b}
    L->slot = align_up(L->payload, 16384);
    return true;
}

}  // namespace tf

using namespace tf;

extern "C" {

const char* tf_last_error(void) { return g_last_error.c_str(); }

const char* tf_status_string(tf_status s) {
    switch (s) {
        case TF_OK: return "TF_OK";
        case TF_ERR_INVALID_ARG: return "TF_ERR_INVALID_ARG";
        case TF_ERR_CUDA: return "TF_ERR_CUDA";
        case TF_ERR_OOM: return "TF_ERR_OOM";
        case TF_ERR_TIMEOUT: return "TF_ERR_TIMEOUT";
        case TF_ERR_NOT_SUPPORTED: return "TF_ERR_NOT_SUPPORTED";
        default: return "TF_ERR_UNKNOWN";
    }
}

const char* tf_version(void) { return "tf-b300 0.1 (sm_103a)"; }

size_t tf_struct_bytes(int which) {
    switch (which) {
        case 0: return sizeof(tf_expert_table);
        case 1: return sizeof(tf_layer_desc);
        case 2: return sizeof(tf_step_stats);
        case 3: return sizeof(tf_cache_event);
        case 4: return sizeof(tf_prefill_stats);
        case 5: return sizeof(tf_attn_desc);
        default: return 0;
    }
}

size_t tf_expert_payload_bytes(int H, int I) {
    ExpertLayout L;
    return expert_layout(H, I, &L) ? L.payload : 0;
}

size_t tf_expert_slot_bytes(int H, int I) {
    ExpertLayout L;
    return expert_layout(H, I, &L) ? L.slot : 0;
}

tf_status tf_expert_offsets(int H, int I, size_t off[4]) {
    ExpertLayout L;
    if (!off) return fail(TF_ERR_INVALID_ARG, "tf_expert_offsets: off is NULL");
    if (!expert_layout(H, I, &L))
        return fail(TF_ERR_INVALID_ARG, "tf_expert_offsets: H=%d I=%d must be positive multiples of 64", H, I);
    off[0] = L.gu_codes;
    off[1] = L.gu_sb;
    off[2] = L.d_codes;
    off[3] = L.d_sb;
    return TF_OK;
}

tf_status tf_pack_expert(const uint8_t* q, const uint16_t* s, const uint16_t* b, int H, int I, void* blob_out) {
    ExpertLayout L;
    if (!q || !s || !b || !blob_out) return fail(TF_ERR_INVALID_ARG, "tf_pack_expert: null pointer");
    if (!expert_layout(H, I, &L))
        return fail(TF_ERR_INVALID_ARG, "tf_pack_expert: H=%d I=%d must be positive multiples of 64", H, I);
    const size_t h = (size_t)H, i = (size_t)I;
    const size_t ncodes = 3 * h * i;
    for (size_t t = 0; t < ncodes; ++t)
        if (q[t] > 15) return fail(TF_ERR_INVALID_ARG, "tf_pack_expert: code %zu is %u (> 15)", t, (unsigned)q[t]);
    uint8_t* blob = static_cast<uint8_t*>(blob_out);
    const uint8_t* qm[3] = {q, q + i * h, q + 2 * i * h};
    const uint16_t* sm[3] = {s, s + i * h / TF_GROUP, s + 2 * i * h / TF_GROUP};
    const uint16_t* bm[3] = {b, b + i * h / TF_GROUP, b + 2 * i * h / TF_GROUP};
    // gate/up: packed row 2j = gate row j, 2j+1 = up row j
    const size_t gu_row = h / 2, gu_groups = h / TF_GROUP;
    for (size_t j = 0; j < i; ++j) {
        for (int m = 0; m < 2; ++m) {
            const uint8_t* src = qm[m] + j * h;
            uint8_t* dst = blob + L.gu_codes + (2 * j + m) * gu_row;
            for (size_t c = 0; c < gu_row; ++c) dst[c] = (uint8_t)(src[2 * c] | (src[2 * c + 1] << 4));
            uint16_t* sb = reinterpret_cast<uint16_t*>(blob + L.gu_sb + (2 * j + m) * gu_groups * 4);
            for (size_t g = 0; g < gu_groups; ++g) {
                sb[2 * g] = sm[m][j * gu_groups + g];
                sb[2 * g + 1] = bm[m][j * gu_groups + g];
            }
        }
    }
    // down: H rows of I/2 bytes
    const size_t d_row = i / 2, d_groups = i / TF_GROUP;
    for (size_t r = 0; r < h; ++r) {
        const uint8_t* src = qm[2] + r * i;
        uint8_t* dst = blob + L.d_codes + r * d_row;
        for (size_t c = 0; c < d_row; ++c) dst[c] = (uint8_t)(src[2 * c] | (src[2 * c + 1] << 4));
        uint16_t* sb = reinterpret_cast<uint16_t*>(blob + L.d_sb + r * d_groups * 4);
        for (size_t g = 0; g < d_groups; ++g) {
            sb[2 * g] = sm[2][r * d_groups + g];
            sb[2 * g + 1] = bm[2][r * d_groups + g];
        }
    }
    return TF_OK;
}

}  // extern "C"

// ------------------------------------------------------------ LFU metadata

extern "C" {

tf_status tf_expert_cache_create(int n_layers, int n_slots, int n_experts, size_t slot_bytes, void* d_slot_pool,
                                 tf_expert_cache** out) {
    if (!out) return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_create: out is NULL");
    *out = nullptr;
    if (n_layers <= 0 || n_slots <= 0 || n_experts <= 0 || n_experts > TF_MAX_E)
        return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_create: bad sizes L=%d S=%d E=%d", n_layers, n_slots,
                    n_experts);
    if (d_slot_pool && (!aligned16(d_slot_pool) || slot_bytes % 16))
        return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_create: slot pool and slot_bytes must be 16-byte aligned");
    tf_expert_cache* c = new (std::nothrow) tf_expert_cache();
    if (!c) return fail(TF_ERR_OOM, "tf_expert_cache_create: out of host memory");
    c->n_layers = n_layers;
    c->n_slots = n_slots;
    c->n_experts = n_experts;
    c->slot_bytes = slot_bytes;
    c->d_slot_pool = d_slot_pool;
    const size_t n = (size_t)n_layers * (size_t)n_slots;
    c->expert.assign(n, -1);
    c->count.assign(n, 0);
    c->last_use.assign(n, 0);
    *out = c;
    return TF_OK;
}

tf_status tf_expert_cache_lookup(tf_expert_cache* c, int layer, int64_t step, const int32_t* ids, int n,
                                 int32_t* slot_or_minus1, uint8_t* hit) {
    if (!c || !ids || !slot_or_minus1 || !hit || n < 0)
        return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_lookup: null pointer or n < 0");
    if (layer < 0 || layer >= c->n_layers) return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_lookup: bad layer %d", layer);
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= c->n_experts)
            return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_lookup: expert id %d out of range", ids[i]);
    const size_t base = (size_t)layer * c->n_slots;
    for (int i = 0; i < n; ++i) {
        int32_t found = -1;
        for (int s = 0; s < c->n_slots; ++s)
            if (c->expert[base + s] == ids[i]) { found = s; break; }
        slot_or_minus1[i] = found;
        hit[i] = found >= 0;
        if (found >= 0) {
            c->count[base + found] += 1;
            c->last_use[base + found] = step;
        }
        c->trace.push_back(tf_cache_event{(int32_t)step, layer, ids[i], found >= 0 ? 1 : 0, found, -1});
    }
    return TF_OK;
}

tf_status tf_expert_cache_admit(tf_expert_cache* c, int layer, int64_t step, int32_t expert, const int32_t* pinned_ids,
                                int n_pinned, int32_t* slot, int32_t* evicted_or_minus1) {
    if (!c || !slot || !evicted_or_minus1 || (n_pinned > 0 && !pinned_ids) || n_pinned < 0)
        return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_admit: null pointer");
    if (layer < 0 || layer >= c->n_layers) return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_admit: bad layer %d", layer);
    if (expert < 0 || expert >= c->n_experts)
        return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_admit: expert id %d out of range", expert);
    const size_t base = (size_t)layer * c->n_slots;
    for (int s = 0; s < c->n_slots; ++s)
        if (c->expert[base + s] == expert)
            return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_admit: expert %d already resident in slot %d", expert, s);
    int victim = -1;
    for (int s = 0; s < c->n_slots && victim < 0; ++s)
        if (c->expert[base + s] < 0) victim = s;
    if (victim < 0) {
        for (int s = 0; s < c->n_slots; ++s) {
            bool pinned = false;
            for (int j = 0; j < n_pinned; ++j)
                if (pinned_ids[j] == c->expert[base + s]) { pinned = true; break; }
            if (pinned) continue;
            if (victim < 0) { victim = s; continue; }
            const int64_t cs = c->count[base + s], cv = c->count[base + victim];
            if (cs < cv || (cs == cv && c->last_use[base + s] < c->last_use[base + victim])) victim = s;
        }
    }
    if (victim < 0) return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_admit: every slot holds a pinned expert");
    *slot = victim;
    *evicted_or_minus1 = c->expert[base + victim];
    c->expert[base + victim] = expert;
    c->count[base + victim] = 1;
    c->last_use[base + victim] = step;
    // complete the pending miss event of this (step, layer, expert), or add one
    for (size_t t = c->trace.size(); t-- > 0;) {
        tf_cache_event& e = c->trace[t];
        if (e.step != (int32_t)step || e.layer != layer) break;
        if (e.expert == expert && !e.hit && e.slot < 0) {
            e.slot = victim;
            e.evicted = *evicted_or_minus1;
            return TF_OK;
        }
    }
    c->trace.push_back(tf_cache_event{(int32_t)step, layer, expert, 0, victim, *evicted_or_minus1});
    return TF_OK;
}

tf_status tf_expert_cache_invalidate(tf_expert_cache* c, int layer, int32_t slot) {
    if (!c || layer < 0 || layer >= c->n_layers || slot < 0 || slot >= c->n_slots)
        return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_invalidate: bad arguments");
    const size_t i = (size_t)layer * c->n_slots + slot;
    c->expert[i] = -1;
    c->count[i] = 0;
    c->last_use[i] = 0;
    return TF_OK;
}

tf_status tf_expert_cache_trace(tf_expert_cache* c, tf_cache_event* buf, size_t cap, size_t* n) {
    if (!c || !n || (cap > 0 && !buf)) return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_trace: null pointer");
    *n = c->trace.size();
    const size_t m = cap < c->trace.size() ? cap : c->trace.size();
    if (m) std::memcpy(buf, c->trace.data(), m * sizeof(tf_cache_event));
    return TF_OK;
}

tf_status tf_expert_cache_state(tf_expert_cache* c, int layer, int32_t* expert, int64_t* count, int64_t* last_use) {
    if (!c || !expert || !count || !last_use || layer < 0 || layer >= c->n_layers)
        return fail(TF_ERR_INVALID_ARG, "tf_expert_cache_state: bad arguments");
    const size_t base = (size_t)layer * c->n_slots;
    for (int s = 0; s < c->n_slots; ++s) {
        expert[s] = c->expert[base + s];
        count[s] = c->count[base + s];
        last_use[s] = c->last_use[base + s];
    }
    return TF_OK;
}

tf_status tf_expert_cache_destroy(tf_expert_cache* c) {
    if (c)
        for (cudaEvent_t ev : c->copy_events) cudaEventDestroy(ev);
    delete c;
    return TF_OK;
}

}  // extern "C"
