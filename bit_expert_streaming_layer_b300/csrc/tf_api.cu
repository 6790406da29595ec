// C-ABI entry points that enqueue device work: routing, the decode FFN, the
// dequant export, layer handles, the (cached) layer step and the decode stack.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "tf_internal.h"

namespace tf {

tf_status cuda_status(int err, const char* what) {
    if (err == 0) return TF_OK;
    return fail(TF_ERR_CUDA, "%s: %s", what, cudaGetErrorString((cudaError_t)err));
}

static int g_copy_countdown = 0;  // failure injection for the miss-fill engine (0 = off)

constexpr unsigned long long DEFAULT_WAIT_LIMIT_NS = 2000000000ull;
static std::atomic<unsigned long long> g_wait_limit_ns{DEFAULT_WAIT_LIMIT_NS};
unsigned long long test_wait_limit_ns() { return g_wait_limit_ns.load(); }

int smem_limit_once(const void* kernel, int bytes) {
    static std::mutex mu;
    static std::vector<std::pair<const void*, int>> done;  // (kernel, device) pairs already raised
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev)) return (int)e;
    std::lock_guard<std::mutex> lock(mu);
    for (const auto& d : done)
        if (d.first == kernel && d.second == dev) return 0;
    if (cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) return (int)e;
    done.emplace_back(kernel, dev);
    return 0;
}

// ------------------------------------------------------------- profiling
struct Prof {
    bool on = false;
    int capacity = 0;
    std::vector<cudaEvent_t> ev[TF_KERNEL_COUNT];  // 2 per timed launch
    int64_t launches[TF_KERNEL_COUNT] = {};
};
static Prof g_prof;

void prof_before(int kind, void* stream) {
    if (!g_prof.on) return;
    const int64_t n = g_prof.launches[kind];
    if (n < g_prof.capacity) cudaEventRecord(g_prof.ev[kind][2 * n], (cudaStream_t)stream);
}

void prof_after(int kind, void* stream) {
    if (!g_prof.on) return;
    const int64_t n = g_prof.launches[kind]++;
    if (n < g_prof.capacity) cudaEventRecord(g_prof.ev[kind][2 * n + 1], (cudaStream_t)stream);
}

static void prof_release() {
    for (auto& v : g_prof.ev) {
        for (cudaEvent_t e : v) cudaEventDestroy(e);
        v.clear();
    }
    g_prof.on = false;
    g_prof.capacity = 0;
}

static bool valid_dims(int H, int I) { return H > 0 && I > 0 && H % TF_GROUP == 0 && I % TF_GROUP == 0; }

static tf_status check_table(const tf_expert_table* t, const char* fn) {
    if (!t || !t->base) return fail(TF_ERR_INVALID_ARG, "%s: expert table or its base is NULL", fn);
    if (!aligned16(t->base) || t->stride % 16)
        return fail(TF_ERR_INVALID_ARG, "%s: expert base and stride must be 16-byte aligned", fn);
    if (t->n_experts < 1) return fail(TF_ERR_INVALID_ARG, "%s: the table's n_experts must be >= 1", fn);
    if (t->slot_of_expert && t->n_slots < 1)
        return fail(TF_ERR_INVALID_ARG, "%s: a table with a slot map needs n_slots >= 1", fn);
    return TF_OK;
}

static ExpertRef table_ref(const tf_expert_table* t, const int32_t* idx) {
    ExpertRef r;
    std::memset(&r, 0, sizeof(r));
    r.base = static_cast<const char*>(t->base);
    r.stride = t->stride;
    r.slot_map = t->slot_of_expert;
    r.idx = idx;
    r.use_ptrs = 0;
    r.n_experts = t->n_experts;
    r.n_slots = t->n_slots;
    return r;
}

struct RouterWs {
    uint32_t* counters;
    float* logits;
};

static size_t router_ws_bytes(int T, int E) {
    return align_up((size_t)T * 4, 256) + align_up((size_t)T * E * 4, 256);
}

static RouterWs carve_router(void* ws, int T) {
    RouterWs r;
    char* p = static_cast<char*>(ws);
    r.counters = reinterpret_cast<uint32_t*>(p);
    r.logits = reinterpret_cast<float*>(p + align_up((size_t)T * 4, 256));
    return r;
}

}  // namespace tf

using namespace tf;

// ------------------------------------------------------------------ handles

namespace {

struct LayerCarve {
    size_t counters, logits, idx, w, rms, h_routed, h_shared, ys, grouped, grouped_bytes, wave_maps, total;
};

int max_waves_of(const tf_layer_desc* d) { return (d->E + d->k - 1) / d->k; }

LayerCarve layer_carve(const tf_layer_desc* d, int T_max) {
    LayerCarve c;
    size_t o = 0;
    c.counters = o; o += align_up((size_t)T_max * 4, 256);
    c.logits = o;   o += align_up((size_t)T_max * d->E * 4, 256);
    c.idx = o;      o += align_up((size_t)T_max * d->k * 4, 256);
    c.w = o;        o += align_up((size_t)T_max * d->k * 4, 256);
    c.rms = o;      o += align_up((size_t)T_max * 4, 256);
    c.h_routed = o; o += align_up((size_t)d->k * d->I * 4, 256);
    c.h_shared = o; o += align_up((size_t)(d->S > 0 ? d->S : 1) * 4, 256);
    c.ys = o;       o += align_up((size_t)d->H * 4, 256);
    // T_max > 1: the grouped path's workspace (permutation, activations, h, y, shared-expert buffers)
    c.grouped = o;
    c.grouped_bytes = T_max > 1 ? grouped_workspace_bytes(T_max, d->H, d->I, d->E, d->k, d->S) : 0;
    o += align_up(c.grouped_bytes, 256);
    c.wave_maps = o;   // chunked prefill through a cache: per wave the experts' mask and slot map
    o += T_max > 1 ? align_up((size_t)max_waves_of(d) * 2 * d->E * 4, 256) : 0;
    c.total = o;
    return c;
}

tf_status check_desc(const tf_layer_desc* d, const char* fn) {
    if (!d) return fail(TF_ERR_INVALID_ARG, "%s: descriptor is NULL", fn);
    if (!valid_dims(d->H, d->I)) return fail(TF_ERR_INVALID_ARG, "%s: H=%d I=%d must be multiples of 64", fn, d->H, d->I);
    if (d->E < 1 || d->E > TF_MAX_E) return fail(TF_ERR_INVALID_ARG, "%s: E=%d out of range", fn, d->E);
    if (d->k < 1 || d->k > TF_MAX_K || d->k > d->E) return fail(TF_ERR_INVALID_ARG, "%s: k=%d out of range", fn, d->k);
    if (d->S < 0 || d->S % TF_GROUP) return fail(TF_ERR_INVALID_ARG, "%s: S=%d must be a multiple of 64", fn, d->S);
    if (!d->W_r || !aligned16(d->W_r)) return fail(TF_ERR_INVALID_ARG, "%s: W_r NULL or misaligned", fn);
    if (d->S > 0 && (!d->W_sg || !d->W_su || !d->W_sd || !aligned16(d->W_sg) || !aligned16(d->W_su) ||
                     !aligned16(d->W_sd)))
        return fail(TF_ERR_INVALID_ARG, "%s: shared-expert weights NULL or misaligned", fn);
    if (!(d->eps >= 0.0f)) return fail(TF_ERR_INVALID_ARG, "%s: eps must be >= 0", fn);
    if (d->experts.n_experts != 0 && d->experts.n_experts != d->E)
        return fail(TF_ERR_INVALID_ARG, "%s: the expert table's n_experts (%d) is not E (%d)", fn,
                    d->experts.n_experts, d->E);
    if (d->experts.slot_of_expert && d->experts.n_slots < 1)
        return fail(TF_ERR_INVALID_ARG, "%s: a table with a slot map needs n_slots >= 1", fn);
    return TF_OK;
}

}  // namespace

namespace tf {
DecodeParams decode_params(const tf_layer* l, const void* x, void* out, float* delta, const ExpertRef& ex,
                           const float* w, const float* rms_in) {
    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = static_cast<const uint16_t*>(x);
    p.out = static_cast<uint16_t*>(out);
    p.delta = delta;
    p.H = l->d.H;
    p.I = l->d.I;
    p.k = l->d.k;
    p.S = l->d.S;
    p.eps = l->d.eps;
    p.rms_in = rms_in;
    p.ex = ex;
    p.w = w;
    p.Wsg = static_cast<const uint16_t*>(l->d.W_sg);
    p.Wsu = static_cast<const uint16_t*>(l->d.W_su);
    p.Wsd = static_cast<const uint16_t*>(l->d.W_sd);
    p.h_routed = l->h_routed;
    p.h_shared = l->h_shared;
    p.off_gu_sb = l->lay.gu_sb;
    p.off_d_codes = l->lay.d_codes;
    p.off_d_sb = l->lay.d_sb;
    return p;
}

void layer_desc_of(const tf_layer* l, tf_layer_desc* out) { *out = l->d; }
}  // namespace tf

extern "C" {

// ------------------------------------------------------------------ routing

size_t tf_router_workspace_bytes(int T, int E) {
    if (T <= 0 || E <= 0) return 0;
    return router_ws_bytes(T, E);
}

tf_status tf_router_topk(const void* x, int T, int H, const void* W_r, int E, const float* logit_bias, int bias_stride,
                         int k, int32_t* idx, float* w, float* logits, float* rms, void* workspace, size_t ws_bytes,
                         void* stream) {
    const char* fn = "tf_router_topk";
    if (!x || !W_r || !idx || !w || !workspace) return fail(TF_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (T <= 0 || H <= 0 || H % TF_GROUP) return fail(TF_ERR_INVALID_ARG, "%s: T=%d H=%d invalid", fn, T, H);
    if (E < 1 || E > TF_MAX_E) return fail(TF_ERR_INVALID_ARG, "%s: E=%d out of range", fn, E);
    if (k < 1 || k > TF_MAX_K || k > E) return fail(TF_ERR_INVALID_ARG, "%s: k=%d out of range", fn, k);
    if (logit_bias && bias_stride != 0 && bias_stride != E)
        return fail(TF_ERR_INVALID_ARG, "%s: bias_stride must be 0 or E", fn);
    if (ws_bytes < router_ws_bytes(T, E)) return fail(TF_ERR_INVALID_ARG, "%s: workspace too small", fn);
    RouterWs r = carve_router(workspace, T);
    clear_error();
    return cuda_status(launch_router_topk(static_cast<const uint16_t*>(x), T, H, static_cast<const uint16_t*>(W_r), E,
                                          logit_bias, bias_stride, k, idx, w, logits ? logits : r.logits, rms,
                                          r.counters, 1e-6f, stream),
                       fn);
}

// ------------------------------------------------------------------ dequant

tf_status tf_dequant_expert(const void* blob, int H, int I, int matrix, int format, void* out, void* stream) {
    ExpertLayout L;
    if (!blob || !out) return fail(TF_ERR_INVALID_ARG, "tf_dequant_expert: null pointer");
    if (!expert_layout(H, I, &L) || matrix < 0 || matrix > 2 || format < 0 || format > 2)
        return fail(TF_ERR_INVALID_ARG, "tf_dequant_expert: bad H/I/matrix/format");
    clear_error();
    const size_t off_sb = matrix < 2 ? L.gu_sb : L.d_sb;
    const size_t off_codes = matrix < 2 ? L.gu_codes : L.d_codes;
    return cuda_status(launch_dequant(static_cast<const char*>(blob), H, I, matrix, format, out, off_sb, off_codes,
                                      stream),
                       "tf_dequant_expert");
}

// --------------------------------------------------------------- decode FFN

size_t tf_moe_decode_workspace_bytes(int H, int I, int k) {
    if (!valid_dims(H, I) || k < 1 || k > TF_MAX_K) return 0;
    return align_up((size_t)k * I * 4, 256);
}

tf_status tf_moe_ffn_decode(const void* x, void* out, const tf_expert_table* table, const int32_t* idx, const float* w,
                            int k, int H, int I, float* delta, void* workspace, size_t ws_bytes, void* stream) {
    const char* fn = "tf_moe_ffn_decode";
    if (!x || !out || !idx || !w || !workspace) return fail(TF_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!valid_dims(H, I)) return fail(TF_ERR_INVALID_ARG, "%s: H=%d I=%d must be multiples of 64", fn, H, I);
    if (k < 1 || k > TF_MAX_K) return fail(TF_ERR_INVALID_ARG, "%s: k=%d out of range", fn, k);
    if (tf_status s = check_table(table, fn)) return s;
    if (ws_bytes < tf_moe_decode_workspace_bytes(H, I, k)) return fail(TF_ERR_INVALID_ARG, "%s: workspace too small", fn);
    ExpertLayout L;
    expert_layout(H, I, &L);
    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = static_cast<const uint16_t*>(x);
    p.out = static_cast<uint16_t*>(out);
    p.delta = delta;
    p.H = H;
    p.I = I;
    p.k = k;
    p.S = 0;
    p.eps = 1e-6f;
    p.rms_in = nullptr;
    p.ex = table_ref(table, idx);
    p.w = w;
    p.h_routed = static_cast<float*>(workspace);
    p.off_gu_sb = L.gu_sb;
    p.off_d_codes = L.d_codes;
    p.off_d_sb = L.d_sb;
    clear_error();
    int e = launch_gateup(p, 0, k * I, stream);
    if (!e) e = launch_down(p, 1, 0, stream);
    return cuda_status(e, fn);
}

}  // extern "C"

// ------------------------------------------- decode FFN without allocation
//
// Scratch for tf_moe_ffn_decode_noalloc: the k x I fp32 gate/up activations
// that the gate/up kernel writes and the down kernel reads. It lives in the
// library image, so every GPU that loads libtf.so holds these bytes until the
// process exits, and every call of that entry point shares them.
namespace {

constexpr size_t NOALLOC_H_FLOATS = TF_NOALLOC_MAX_KI;
__device__ __align__(256) float g_noalloc_h[NOALLOC_H_FLOATS];

constexpr int NOALLOC_MAX_DEVICES = 64;
float* g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};
std::mutex g_noalloc_mu;

// Device address of g_noalloc_h on the current device, looked up once per
// device. In host code the array's name is only a host-side shadow; passing it
// to a kernel would hand the GPU a wrong address.
tf_status noalloc_scratch(float** out, const char* fn) {
    int dev = -1;
    if (cudaError_t e = cudaGetDevice(&dev)) return cuda_status(e, fn);
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return fail(TF_ERR_NOT_SUPPORTED, "%s: device %d out of range", fn, dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_h)) return cuda_status(e, fn);
        g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return TF_OK;
}

}  // namespace

extern "C" {

tf_status tf_moe_ffn_decode_noalloc(const void* x, void* out, const tf_expert_table* table, const int32_t* idx,
                                    const float* w, int k, int H, int I, float* delta, void* stream) {
    const char* fn = "tf_moe_ffn_decode_noalloc";
    if (!x || !out || !idx || !w) return fail(TF_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!valid_dims(H, I)) return fail(TF_ERR_INVALID_ARG, "%s: H=%d I=%d must be multiples of 64", fn, H, I);
    if (k < 1 || k > TF_MAX_K) return fail(TF_ERR_INVALID_ARG, "%s: k=%d out of range", fn, k);
    if ((size_t)k * (size_t)I > NOALLOC_H_FLOATS)
        return fail(TF_ERR_INVALID_ARG, "%s: k*I = %zu exceeds the built-in scratch of %zu floats", fn,
                    (size_t)k * (size_t)I, NOALLOC_H_FLOATS);
    if (tf_status s = check_table(table, fn)) return s;
    float* scratch = nullptr;
    if (tf_status s = noalloc_scratch(&scratch, fn)) return s;
    ExpertLayout L;
    expert_layout(H, I, &L);
    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = static_cast<const uint16_t*>(x);
    p.out = static_cast<uint16_t*>(out);
    p.delta = delta;
    p.H = H;
    p.I = I;
    p.k = k;
    p.S = 0;
    p.eps = 1e-6f;
    p.rms_in = nullptr;
    p.ex = table_ref(table, idx);
    p.w = w;
    p.h_routed = scratch;  // fully written by the gate/up kernel before the down kernel reads it
    p.off_gu_sb = L.gu_sb;
    p.off_d_codes = L.d_codes;
    p.off_d_sb = L.d_sb;
    clear_error();
    int e = launch_gateup(p, 0, k * I, stream);
    if (!e) e = launch_down(p, 1, 0, stream);
    return cuda_status(e, fn);
}

// ------------------------------------------------------------------ layers

size_t tf_layer_workspace_bytes(const tf_layer_desc* d, int T_max) {
    if (check_desc(d, "tf_layer_workspace_bytes") != TF_OK || T_max < 1) return 0;
    return layer_carve(d, T_max).total;
}

tf_status tf_layer_create(const tf_layer_desc* d, int T_max, void* workspace, size_t ws_bytes, tf_layer** out) {
    const char* fn = "tf_layer_create";
    if (!out) return fail(TF_ERR_INVALID_ARG, "%s: out is NULL", fn);
    *out = nullptr;
    if (tf_status s = check_desc(d, fn)) return s;
    if (T_max < 1) return fail(TF_ERR_INVALID_ARG, "%s: T_max=%d", fn, T_max);
    LayerCarve c = layer_carve(d, T_max);
    if (!workspace || ws_bytes < c.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return fail(TF_ERR_INVALID_ARG, "%s: workspace NULL, misaligned or smaller than %zu bytes", fn, c.total);
    tf_layer* l = new (std::nothrow) tf_layer();
    if (!l) return fail(TF_ERR_OOM, "%s: out of host memory", fn);
    l->d = *d;
    if (l->d.experts.n_experts == 0) l->d.experts.n_experts = d->E;  // 0 stands for the descriptor's E
    l->T_max = T_max;
    expert_layout(d->H, d->I, &l->lay);
    l->ws = static_cast<char*>(workspace);
    l->ws_bytes = ws_bytes;
    l->counters = reinterpret_cast<uint32_t*>(l->ws + c.counters);
    l->logits = reinterpret_cast<float*>(l->ws + c.logits);
    l->idx = reinterpret_cast<int32_t*>(l->ws + c.idx);
    l->w = reinterpret_cast<float*>(l->ws + c.w);
    l->rms = reinterpret_cast<float*>(l->ws + c.rms);
    l->h_routed = reinterpret_cast<float*>(l->ws + c.h_routed);
    l->h_shared = reinterpret_cast<float*>(l->ws + c.h_shared);
    l->ys = reinterpret_cast<float*>(l->ws + c.ys);
    l->grouped_ws = c.grouped_bytes ? l->ws + c.grouped : nullptr;
    l->grouped_bytes = c.grouped_bytes;
    cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&l->h_idx), TF_MAX_K * sizeof(int32_t), cudaHostAllocDefault);
    if (e == cudaSuccess && T_max > 1) {
        l->max_waves = max_waves_of(d);
        l->d_wave_maps = reinterpret_cast<int32_t*>(l->ws + c.wave_maps);
        e = cudaHostAlloc(reinterpret_cast<void**>(&l->h_chunk_ids), (size_t)T_max * d->k * sizeof(int32_t),
                          cudaHostAllocDefault);
        if (e == cudaSuccess)
            e = cudaHostAlloc(reinterpret_cast<void**>(&l->h_wave_maps),
                              (size_t)l->max_waves * 2 * d->E * sizeof(int32_t), cudaHostAllocDefault);
    }
    if (e != cudaSuccess) {
        tf_layer_destroy(l);
        return fail(TF_ERR_OOM, "%s: pinned staging: %s", fn, cudaGetErrorString(e));
    }
    cudaEvent_t* evs[] = {&l->ev_idx, &l->ev_copies, &l->ev_t0, &l->ev_shared, &l->ev_c0, &l->ev_wave};
    for (cudaEvent_t* ev : evs) {
        e = cudaEventCreate(ev);
        if (e != cudaSuccess) {
            tf_layer_destroy(l);
            return cuda_status(e, fn);
        }
    }
    *out = l;
    return TF_OK;
}

tf_status tf_layer_destroy(tf_layer* l) {
    if (!l) return TF_OK;
    cudaEvent_t evs[] = {l->ev_idx, l->ev_copies, l->ev_t0, l->ev_shared, l->ev_c0, l->ev_wave};
    for (cudaEvent_t ev : evs)
        if (ev) cudaEventDestroy(ev);
    if (l->h_idx) cudaFreeHost(l->h_idx);
    if (l->h_chunk_ids) cudaFreeHost(l->h_chunk_ids);
    if (l->h_wave_maps) cudaFreeHost(l->h_wave_maps);
    delete l;
    return TF_OK;
}

tf_status tf_layer_routing(tf_layer* l, int32_t** idx, float** w, float** logits, float** rms) {
    if (!l) return fail(TF_ERR_INVALID_ARG, "tf_layer_routing: layer is NULL");
    if (idx) *idx = l->idx;
    if (w) *w = l->w;
    if (logits) *logits = l->logits;
    if (rms) *rms = l->rms;
    return TF_OK;
}

tf_status tf_profile_begin(int capacity) {
    if (capacity < 1) return fail(TF_ERR_INVALID_ARG, "tf_profile_begin: capacity < 1");
    prof_release();
    for (int k = 0; k < TF_KERNEL_COUNT; ++k) {
        g_prof.launches[k] = 0;
        g_prof.ev[k].resize(2 * (size_t)capacity, nullptr);
        for (auto& e : g_prof.ev[k]) {
            if (cudaError_t err = cudaEventCreate(&e)) {
                e = nullptr;
                prof_release();
                return cuda_status(err, "tf_profile_begin");
            }
        }
    }
    g_prof.capacity = capacity;
    g_prof.on = true;
    return TF_OK;
}

tf_status tf_profile_end(double* ms, int64_t* launches) {
    if (!ms || !launches) return fail(TF_ERR_INVALID_ARG, "tf_profile_end: null pointer");
    if (!g_prof.on) return fail(TF_ERR_INVALID_ARG, "tf_profile_end: profiling is not on");
    g_prof.on = false;
    tf_status st = TF_OK;
    for (int k = 0; k < TF_KERNEL_COUNT; ++k) {
        const int64_t n = g_prof.launches[k] < g_prof.capacity ? g_prof.launches[k] : g_prof.capacity;
        double total = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            if (cudaError_t err = cudaEventSynchronize(g_prof.ev[k][2 * i + 1])) {
                st = cuda_status(err, "tf_profile_end");
                break;
            }
            float t = 0.f;
            cudaEventElapsedTime(&t, g_prof.ev[k][2 * i], g_prof.ev[k][2 * i + 1]);
            total += t;
        }
        ms[k] = total;
        launches[k] = g_prof.launches[k];
    }
    prof_release();
    return st;
}

tf_status tf_test_set_wait_limit_ns(uint64_t ns) {
    g_wait_limit_ns = ns ? (unsigned long long)ns : DEFAULT_WAIT_LIMIT_NS;
    return TF_OK;
}

tf_status tf_test_fail_nth_copy(int n) {
    if (n < 0) return fail(TF_ERR_INVALID_ARG, "tf_test_fail_nth_copy: n < 0");
    g_copy_countdown = n;
    return TF_OK;
}

tf_status tf_layer_step(tf_layer* l, tf_expert_cache* cache, int layer, int64_t step, const void* h_expert_store,
                        const void* x, void* out, int T, const float* logit_bias, int bias_stride,
                        void* compute_stream, void* copy_stream, int measure, tf_step_stats* stats) {
    const char* fn = "tf_layer_step";
    if (!l || !x || !out) return fail(TF_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (T < 1 || T > l->T_max) return fail(TF_ERR_INVALID_ARG, "%s: T=%d outside [1, %d]", fn, T, l->T_max);
    if (logit_bias && bias_stride != 0 && bias_stride != l->d.E)
        return fail(TF_ERR_INVALID_ARG, "%s: bias_stride must be 0 or E", fn);
    const tf_layer_desc& d = l->d;
    if (!cache) {
        if (tf_status s = check_table(&d.experts, fn)) return s;
    } else {
        if (T != 1) return fail(TF_ERR_NOT_SUPPORTED, "%s: the cached step runs one token", fn);
        if (!h_expert_store) return fail(TF_ERR_INVALID_ARG, "%s: a cached step needs the pinned expert store", fn);
        if (!copy_stream) return fail(TF_ERR_INVALID_ARG, "%s: a cached step needs a copy stream", fn);
    }
    if (stats) std::memset(stats, 0, sizeof(*stats));
    if (T > 1) {
        // batched tokens: router for all T, then the grouped routed experts and shared expert (tcgen05 GEMMs)
        clear_error();
        cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
        int e = launch_router_topk(static_cast<const uint16_t*>(x), T, d.H, static_cast<const uint16_t*>(d.W_r), d.E,
                                   logit_bias, bias_stride, d.k, l->idx, l->w, l->logits, l->rms, l->counters, d.eps,
                                   cs);
        if (e) return cuda_status(e, fn);
        GroupedArgs a;
        std::memset(&a, 0, sizeof(a));
        a.x = x;
        a.out = out;
        a.T = T;
        a.table = &d.experts;
        a.E = d.E;
        a.k = d.k;
        a.H = d.H;
        a.I = d.I;
        a.idx = l->idx;
        a.w = l->w;
        a.Wsg = d.W_sg;
        a.Wsu = d.W_su;
        a.Wsd = d.W_sd;
        a.S = d.S;
        a.eps = d.eps;
        a.rms_in = l->rms;   // written by the router above for every token
        a.ws = l->grouped_ws;
        a.ws_bytes = l->grouped_bytes;
        return grouped_run(a, cs, fn);
    }
    clear_error();
    cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
    if (measure && stats) {
        if (int e = cudaEventRecord(l->ev_t0, cs)) return cuda_status(e, fn);
    }
    int e = launch_router_topk(static_cast<const uint16_t*>(x), 1, d.H, static_cast<const uint16_t*>(d.W_r), d.E,
                               logit_bias, bias_stride, d.k, l->idx, l->w, l->logits, l->rms, l->counters, d.eps, cs);
    if (e) return cuda_status(e, fn);

    if (!cache) {
        DecodeParams p = decode_params(l, x, out, nullptr, table_ref(&d.experts, l->idx), l->w, l->rms);
        e = launch_gateup(p, 0, d.k * d.I + d.S, cs);
        if (!e) e = launch_down(p, 1, d.S > 0, cs);
        return cuda_status(e, fn);
    }

    // ---- cached step: ids to the host, shared branch, miss fills, routed experts
    tf_expert_cache* c = cache;
    if (layer < 0 || layer >= c->n_layers) return fail(TF_ERR_INVALID_ARG, "%s: bad layer %d", fn, layer);
    if (!c->d_slot_pool || c->n_experts != d.E || c->slot_bytes < l->lay.payload || c->n_slots < d.k)
        return fail(TF_ERR_INVALID_ARG, "%s: cache does not match the layer (pool, E, slot size or slot count)", fn);
    cudaStream_t ps = static_cast<cudaStream_t>(copy_stream);
    const int k = d.k;
    if ((e = cudaMemcpyAsync(l->h_idx, l->idx, (size_t)k * 4, cudaMemcpyDeviceToHost, cs))) return cuda_status(e, fn);
    if ((e = cudaEventRecord(l->ev_idx, cs))) return cuda_status(e, fn);
    ExpertRef none;
    std::memset(&none, 0, sizeof(none));
    DecodeParams p = decode_params(l, x, out, nullptr, none, l->w, l->rms);
    // the shared branch (gate/up, then down into the fp32 buffer ys) runs while the host decides the copies and
    // while they run; the routed down later adds x + ys + its own terms
    p.ys = d.S > 0 ? l->ys : nullptr;
    if (d.S > 0 && (e = launch_gateup(p, k * d.I, k * d.I + d.S, cs))) return cuda_status(e, fn);
    if (d.S > 0 && (e = launch_down(p, 0, 1, cs))) return cuda_status(e, fn);
    if (measure && stats && (e = cudaEventRecord(l->ev_shared, cs))) return cuda_status(e, fn);
    if ((e = cudaEventSynchronize(l->ev_idx))) return cuda_status(e, fn);  // the one host wait: the CPU decides the I/O
    int32_t ids[TF_MAX_K], slot[TF_MAX_K];
    uint8_t hit[TF_MAX_K];
    std::memcpy(ids, l->h_idx, (size_t)k * 4);
    if (tf_status s = tf_expert_cache_lookup(c, layer, step, ids, k, slot, hit)) return s;
    int32_t admitted[TF_MAX_K];
    int na = 0;
    uint64_t bytes = 0;
    // copy streams: the cache's set (the k-th miss on streams[k mod n]) or the call's copy stream
    const int nstr = c->copy_streams.empty() ? 1 : (int)c->copy_streams.size();
    auto copy_stream_of = [&](int m) { return c->copy_streams.empty() ? ps : c->copy_streams[m % nstr]; };
    if (measure && stats && (e = cudaEventRecord(l->ev_c0, copy_stream_of(0)))) return cuda_status(e, fn);
    const char* pool = static_cast<const char*>(c->d_slot_pool);
    const char* store = static_cast<const char*>(h_expert_store);
    for (int i = 0; i < k; ++i) {
        if (hit[i]) continue;
        int32_t s = -1, evicted = -1;
        tf_status st = tf_expert_cache_admit(c, layer, step, ids[i], ids, k, &s, &evicted);
        if (st == TF_OK) {
            slot[i] = s;
            char* dst = const_cast<char*>(pool) + ((size_t)layer * c->n_slots + s) * c->slot_bytes;
            const char* src = store + ((size_t)layer * d.E + ids[i]) * c->slot_bytes;
            if (g_copy_countdown > 0 && --g_copy_countdown == 0)
                e = (int)cudaErrorInvalidValue;  // injected failure: the copy is not enqueued
            else
                e = (int)cudaMemcpyAsync(dst, src, l->lay.payload, cudaMemcpyHostToDevice, copy_stream_of(na));
            admitted[na++] = s;
            if (e) st = cuda_status(e, "tf_layer_step: expert copy");
            bytes += l->lay.payload;
        }
        if (st != TF_OK) {
            for (int j = 0; j < na; ++j) tf_expert_cache_invalidate(c, layer, admitted[j]);
            std::string msg = tf_last_error();
            return fail(st, "%s: miss fill failed, %d admitted slot(s) rolled back: %s", fn, na, msg.c_str());
        }
    }
    if (c->copy_streams.empty()) {
        if ((e = cudaEventRecord(l->ev_copies, ps))) return cuda_status(e, fn);
        if ((e = cudaStreamWaitEvent(cs, l->ev_copies, 0))) return cuda_status(e, fn);
    } else {
        for (int j = 0; j < nstr; ++j) {
            if ((e = cudaEventRecord(c->copy_events[j], c->copy_streams[j]))) return cuda_status(e, fn);
            if ((e = cudaStreamWaitEvent(cs, c->copy_events[j], 0))) return cuda_status(e, fn);
        }
    }
    ExpertRef r;
    std::memset(&r, 0, sizeof(r));
    r.use_ptrs = 1;
    for (int i = 0; i < k; ++i) r.ptr[i] = pool + ((size_t)layer * c->n_slots + slot[i]) * c->slot_bytes;
    p.ex = r;
    e = launch_gateup(p, 0, k * d.I, cs);
    if (!e) e = launch_down(p, 1, 0, cs);  // out = x + ys + routed terms (ys: the shared down, enqueued above)
    if (e) return cuda_status(e, fn);
    if (stats) {
        std::memcpy(stats->ids, ids, (size_t)k * 4);
        stats->misses = na;
        stats->hits = k - na;
        stats->bytes_fetched = bytes;
        if (measure) {
            if ((e = cudaStreamSynchronize(cs))) return cuda_status(e, fn);
            float t_shared = 0.f, t_copies = 0.f, t_copy = 0.f;
            if (d.S > 0) cudaEventElapsedTime(&t_shared, l->ev_t0, l->ev_shared);
            if (c->copy_streams.empty()) {
                cudaEventElapsedTime(&t_copies, l->ev_t0, l->ev_copies);
                cudaEventElapsedTime(&t_copy, l->ev_c0, l->ev_copies);
            } else {
                for (int j = 0; j < nstr; ++j) {  // the last stream to finish ends the fills
                    float a = 0.f, b = 0.f;
                    cudaEventElapsedTime(&a, l->ev_t0, c->copy_events[j]);
                    cudaEventElapsedTime(&b, l->ev_c0, c->copy_events[j]);
                    t_copies = a > t_copies ? a : t_copies;
                    t_copy = b > t_copy ? b : t_copy;
                }
            }
            stats->shared_ms = t_shared;
            stats->copy_ms = t_copy;
            stats->stall_ms = t_copies > t_shared ? t_copies - t_shared : 0.f;
        }
    }
    return TF_OK;
}

tf_status tf_expert_cache_set_copy_streams(tf_expert_cache* c, void* const* streams, int n) {
    const char* fn = "tf_expert_cache_set_copy_streams";
    if (!c || n < 0 || n > TF_MAX_K || (n > 0 && !streams)) return fail(TF_ERR_INVALID_ARG, "%s: bad arguments", fn);
    for (int j = 0; j < n; ++j)
        if (!streams[j]) return fail(TF_ERR_INVALID_ARG, "%s: stream %d is NULL", fn, j);
    while ((int)c->copy_events.size() < n) {
        cudaEvent_t ev = nullptr;
        if (cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDefault)) return cuda_status(e, fn);
        c->copy_events.push_back(ev);
    }
    c->copy_streams.clear();
    for (int j = 0; j < n; ++j) c->copy_streams.push_back(static_cast<cudaStream_t>(streams[j]));
    return TF_OK;
}

namespace {

// One chunk's waves through the host-metadata cache (tf_layer_prefill_cached).
struct PrefillWaves {
    tf_layer* l;
    tf_expert_cache* c;
    int layer;
    int64_t step0;
    const char* store;
    cudaStream_t cs, ps;
    std::vector<std::vector<int32_t>> waves;
    int hits = 0, misses = 0;
    uint64_t bytes = 0;
};

// Before wave w: the copy stream waits until the earlier waves' GEMMs are done with the slots, the wave's
// lookups and admissions (one LFU step, the wave's experts pinned), one copy per miss, the compute stream
// waits for the copies; the wave's mask and slot map go to the pinned staging row w.
int prefill_before_wave(void* ctx, int w, void* stream) {
    PrefillWaves& P = *static_cast<PrefillWaves*>(ctx);
    const char* fn = "tf_layer_prefill_cached";
    tf_layer* l = P.l;
    tf_expert_cache* c = P.c;
    const int E = l->d.E;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaError_t e = cudaEventRecord(l->ev_wave, cs)) return cuda_status(e, fn);
    if (cudaError_t e = cudaStreamWaitEvent(P.ps, l->ev_wave, 0)) return cuda_status(e, fn);
    const std::vector<int32_t>& ids = P.waves[w];
    const int n = (int)ids.size();
    const int64_t step = P.step0 + w;
    std::vector<int32_t> slot((size_t)n);
    std::vector<uint8_t> hit((size_t)n);
    if (tf_status s = tf_expert_cache_lookup(c, P.layer, step, ids.data(), n, slot.data(), hit.data())) return s;
    std::vector<int32_t> admitted;
    char* pool = static_cast<char*>(c->d_slot_pool);
    for (int i = 0; i < n; ++i) {
        if (hit[i]) continue;
        int32_t s = -1, evicted = -1;
        tf_status st = tf_expert_cache_admit(c, P.layer, step, ids[i], ids.data(), n, &s, &evicted);
        int e = 0;
        if (st == TF_OK) {
            slot[i] = s;
            admitted.push_back(s);
            char* dst = pool + ((size_t)P.layer * c->n_slots + s) * c->slot_bytes;
            const char* src = P.store + ((size_t)P.layer * E + ids[i]) * c->slot_bytes;
            if (g_copy_countdown > 0 && --g_copy_countdown == 0)
                e = (int)cudaErrorInvalidValue;  // injected failure: the copy is not enqueued
            else
                e = (int)cudaMemcpyAsync(dst, src, l->lay.payload, cudaMemcpyHostToDevice, P.ps);
            if (e) st = cuda_status(e, "tf_layer_prefill_cached: expert copy");
            P.bytes += l->lay.payload;
            ++P.misses;
        }
        if (st != TF_OK) {
            for (int32_t a : admitted) tf_expert_cache_invalidate(c, P.layer, a);
            std::string msg = tf_last_error();
            return fail(st, "%s: miss fill failed, %zu admitted slot(s) of wave %d rolled back: %s", fn,
                        admitted.size(), w, msg.c_str());
        }
    }
    P.hits += n - (int)admitted.size();
    int32_t* mask = l->h_wave_maps + (size_t)w * 2 * E;
    int32_t* smap = mask + E;
    for (int e2 = 0; e2 < E; ++e2) {
        mask[e2] = 0;
        smap[e2] = -1;
    }
    for (int i = 0; i < n; ++i) {
        mask[ids[i]] = 1;
        smap[ids[i]] = slot[i];
    }
    if (cudaError_t e = cudaEventRecord(l->ev_copies, P.ps)) return cuda_status(e, fn);
    if (cudaError_t e = cudaStreamWaitEvent(cs, l->ev_copies, 0)) return cuda_status(e, fn);
    return TF_OK;
}

}  // namespace

tf_status tf_layer_prefill_cached(tf_layer* l, tf_expert_cache* c, int layer, int64_t step0, const void* h_expert_store,
                                  const void* x, void* out, int T, const float* logit_bias, int bias_stride,
                                  void* compute_stream, void* copy_stream, tf_prefill_stats* stats) {
    const char* fn = "tf_layer_prefill_cached";
    if (!l || !c || !h_expert_store || !x || !out || !copy_stream) return fail(TF_ERR_INVALID_ARG, "%s: null argument", fn);
    const tf_layer_desc& d = l->d;
    if (l->T_max < 2 || !l->h_chunk_ids) return fail(TF_ERR_INVALID_ARG, "%s: the layer handle needs T_max > 1", fn);
    if (T < 1 || T > l->T_max) return fail(TF_ERR_INVALID_ARG, "%s: T=%d outside [1, %d]", fn, T, l->T_max);
    if (layer < 0 || layer >= c->n_layers) return fail(TF_ERR_INVALID_ARG, "%s: bad layer %d", fn, layer);
    if (!c->d_slot_pool || c->n_experts != d.E || c->slot_bytes < l->lay.payload || c->n_slots < d.k ||
        c->slot_bytes % 16)
        return fail(TF_ERR_INVALID_ARG, "%s: cache does not match the layer (pool, E, slot size or slot count)", fn);
    if (logit_bias && bias_stride != 0 && bias_stride != d.E)
        return fail(TF_ERR_INVALID_ARG, "%s: bias_stride must be 0 or E", fn);
    if (stats) std::memset(stats, 0, sizeof(*stats));
    clear_error();
    cudaStream_t cs = static_cast<cudaStream_t>(compute_stream), ps = static_cast<cudaStream_t>(copy_stream);
    const int k = d.k;
    int e = launch_router_topk(static_cast<const uint16_t*>(x), T, d.H, static_cast<const uint16_t*>(d.W_r), d.E,
                               logit_bias, bias_stride, k, l->idx, l->w, l->logits, l->rms, l->counters, d.eps, cs);
    if (!e) e = cudaMemcpyAsync(l->h_chunk_ids, l->idx, (size_t)T * k * 4, cudaMemcpyDeviceToHost, cs);
    if (!e) e = cudaEventRecord(l->ev_idx, cs);
    if (!e) e = cudaEventSynchronize(l->ev_idx);   // the one host wait: the CPU decides the waves and the copies
    if (e) return cuda_status(e, fn);
    // the chunk's distinct experts in order of first use, in waves of n_slots
    PrefillWaves P;
    P.l = l;
    P.c = c;
    P.layer = layer;
    P.step0 = step0;
    P.store = static_cast<const char*>(h_expert_store);
    P.cs = cs;
    P.ps = ps;
    std::vector<char> seen((size_t)d.E, 0);
    std::vector<int32_t> order;
    for (int i = 0; i < T * k; ++i) {
        const int32_t id = l->h_chunk_ids[i];
        if ((unsigned)id >= (unsigned)d.E) return fail(TF_ERR_CUDA, "%s: router id %d out of range", fn, id);
        if (!seen[id]) {
            seen[id] = 1;
            order.push_back(id);
        }
    }
    for (size_t i = 0; i < order.size(); i += (size_t)c->n_slots)
        P.waves.emplace_back(order.begin() + i, order.begin() + std::min(order.size(), i + (size_t)c->n_slots));
    if ((int)P.waves.size() > l->max_waves) return fail(TF_ERR_INVALID_ARG, "%s: too many waves", fn);
    GroupedWaves wv;
    wv.n = (int)P.waves.size();
    wv.pool = static_cast<const char*>(c->d_slot_pool) + (size_t)layer * c->n_slots * c->slot_bytes;
    wv.slot_bytes = c->slot_bytes;
    wv.n_slots = c->n_slots;
    wv.d_maps = l->d_wave_maps;
    wv.h_maps = l->h_wave_maps;
    wv.before_wave = prefill_before_wave;
    wv.ctx = &P;
    GroupedArgs a;
    std::memset(&a, 0, sizeof(a));
    a.x = x;
    a.out = out;
    a.T = T;
    a.table = nullptr;
    a.E = d.E;
    a.k = k;
    a.H = d.H;
    a.I = d.I;
    a.idx = l->idx;
    a.w = l->w;
    a.Wsg = d.W_sg;
    a.Wsu = d.W_su;
    a.Wsd = d.W_sd;
    a.S = d.S;
    a.eps = d.eps;
    a.rms_in = l->rms;   // written by this chunk's router for every token
    a.ws = l->grouped_ws;
    a.ws_bytes = l->grouped_bytes;
    a.waves = &wv;
    tf_status st = grouped_run(a, cs, fn);
    if (stats) {
        stats->waves = wv.n;
        stats->hits = P.hits;
        stats->misses = P.misses;
        stats->bytes_fetched = P.bytes;
    }
    return st;
}

tf_status tf_stack_decode(tf_layer* const* layers, int L, const void* x, void* out, void* scratch,
                          const float* const* logit_bias, void* stream) {
    const char* fn = "tf_stack_decode";
    if (!layers || L < 1 || !x || !out || !scratch) return fail(TF_ERR_INVALID_ARG, "%s: bad arguments", fn);
    if (scratch == x || scratch == out) return fail(TF_ERR_INVALID_ARG, "%s: scratch must not alias x or out", fn);
    for (int i = 0; i < L; ++i)
        if (!layers[i] || layers[i]->d.H != layers[0]->d.H)
            return fail(TF_ERR_INVALID_ARG, "%s: layer %d is NULL or has another H", fn, i);
    const void* cur = x;
    for (int i = 0; i < L; ++i) {
        void* dst = ((L - 1 - i) % 2 == 0) ? out : scratch;
        tf_status s = tf_layer_step(layers[i], nullptr, i, 0, nullptr, cur, dst, 1,
                                    logit_bias ? logit_bias[i] : nullptr, 0, stream, nullptr, 0, nullptr);
        if (s) return s;
        cur = dst;
    }
    return TF_OK;
}

}  // extern "C"
