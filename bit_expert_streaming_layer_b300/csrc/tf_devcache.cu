// Per-layer LFU expert cache with its metadata in device memory, and the cached
// decode step built on it (tf_device_cache_*, tf_layer_step_device_cache).
//
// The pages' runtime checks a 16-slot LFU cache of experts per token and layer
// and reads the missing experts from slower storage while the GPU computes the
// shared-expert branch (page "Como executar um modelo de 26 bilhoes de
// parametros em dois gigabytes de memoria em um Mac comum", section "Qual e o
// principal truque da arquitetura"). There the CPU decides the reads. Here the
// decision moves onto the GPU, so that a step never waits on the host:
//   k_lfu_step : one warp applies the LFU policy to the k ids the router wrote,
//                updates the slots and the expert -> slot map, appends the
//                trace and writes the layer's miss list;
//   k_fetch    : CTAs copy every missing expert from the pinned host store
//                (mapped into the device's address space) into its slot,
//                reading host memory directly over the bus.
// The routed experts then find their weights through the slot map.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <new>

#include "tf_device.cuh"
#include "tf_internal.h"

namespace tf {
namespace devcache {

constexpr int MAX_SLOTS = 1024;
constexpr int FETCH_THREADS = 256;
constexpr int FETCH_UNROLL = 8;                                   // 16-byte loads in flight per thread
constexpr int FETCH_CHUNK = FETCH_THREADS * FETCH_UNROLL * 16;    // 32 KiB per CTA round

// Device state of one layer (inside the caller's d_state).
struct LayerState {
    int32_t* expert;       // [S], -1 = empty
    long long* count;      // [S] uses since admission
    long long* last_use;   // [S] step of the last use
    int32_t* slot_of;      // [E] slot holding the expert, -1 = none
    long long* ctr;        // [0] step (lookups of this layer so far), [1] hits, [2] misses
    int32_t* miss;         // [0] misses of the last lookup, [1] its hits, [2..2+K) experts, [2+K..2+2K) slots
};

struct LfuArgs {
    LayerState st;
    const int32_t* idx;    // device [k]
    int k, S, E, layer;
    tf_cache_event* trace;
    unsigned long long* trace_n;
    unsigned long long trace_cap;
    uint32_t* err;
};

// (count, last use, slot) of a victim candidate, compared lexicographically.
struct Cand {
    long long cnt, lu;
    int s;
};
__device__ __forceinline__ bool cand_less(const Cand& a, const Cand& b) {
    if (a.s < 0) return false;
    if (b.s < 0) return true;
    if (a.cnt != b.cnt) return a.cnt < b.cnt;
    if (a.lu != b.lu) return a.lu < b.lu;
    return a.s < b.s;
}

__global__ void __launch_bounds__(32) k_lfu_step(LfuArgs a) {
    __shared__ int32_t ex[MAX_SLOTS];
    __shared__ long long cnt[MAX_SLOTS], lu[MAX_SLOTS];
    __shared__ int32_t ids[TF_MAX_K], slot[TF_MAX_K], evicted[TF_MAX_K], hit[TF_MAX_K];
    const int lane = threadIdx.x;
    const int S = a.S, k = a.k;
    for (int s = lane; s < S; s += 32) {
        ex[s] = a.st.expert[s];
        cnt[s] = a.st.count[s];
        lu[s] = a.st.last_use[s];
    }
    int bad = 0;
    if (lane < k) {
        ids[lane] = a.idx[lane];
        bad = (unsigned)ids[lane] >= (unsigned)a.E;
    }
    __syncwarp();
    if (__any_sync(dev::FULL, bad)) {
        // an id the router cannot produce: leave the cache untouched, fetch nothing; the routed experts
        // see the same id out of range and make their outputs NaN
        if (lane == 0) {
            a.st.miss[0] = 0;
            a.st.miss[1] = 0;
            atomicOr(a.err, 1u);
        }
        return;
    }
    const long long step = a.st.ctr[0];
    // pass 1: every id already in a slot is a hit (count + 1, last use = this step)
    if (lane < k) {
        int h = -1;
        for (int s = 0; s < S; ++s)
            if (ex[s] == ids[lane]) {
                h = s;
                break;
            }
        hit[lane] = h >= 0;
        slot[lane] = h;
        evicted[lane] = -1;
    }
    __syncwarp();
    if (lane == 0)
        for (int i = 0; i < k; ++i)
            if (hit[i]) {
                cnt[slot[i]] += 1;
                lu[slot[i]] = step;
            }
    __syncwarp();
    // pass 2: the misses in top-k order, each into the lowest empty slot, else the slot not holding any of
    // this step's ids with the smallest count, then the oldest last use, then the lowest index
    int n_miss = 0;
    for (int i = 0; i < k; ++i) {
        if (hit[i]) continue;
        int empty = S;
        for (int s = lane; s < S; s += 32)
            if (ex[s] < 0) {
                empty = s;
                break;
            }
        empty = (int)__reduce_min_sync(dev::FULL, (unsigned)empty);
        int v = empty < S ? empty : -1;
        if (v < 0) {
            Cand best{0, 0, -1};
            for (int s = lane; s < S; s += 32) {
                bool current = false;
                for (int j = 0; j < k; ++j) current |= ex[s] == ids[j];
                const Cand c{cnt[s], lu[s], current ? -1 : s};
                if (cand_less(c, best)) best = c;
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                Cand other;
                other.cnt = __shfl_xor_sync(dev::FULL, best.cnt, o);
                other.lu = __shfl_xor_sync(dev::FULL, best.lu, o);
                other.s = __shfl_xor_sync(dev::FULL, best.s, o);
                if (cand_less(other, best)) best = other;
            }
            v = best.s;
        }
        if (v < 0) {  // more distinct ids than slots: nothing to evict
            if (lane == 0) atomicOr(a.err, 2u);
            continue;
        }
        if (lane == 0) {
            const int old = ex[v];
            evicted[i] = old;
            if (old >= 0 && a.st.slot_of[old] == v) a.st.slot_of[old] = -1;
            ex[v] = ids[i];
            cnt[v] = 1;
            lu[v] = step;
            slot[i] = v;
            a.st.slot_of[ids[i]] = v;
            a.st.miss[2 + n_miss] = ids[i];
            a.st.miss[2 + TF_MAX_K + n_miss] = v;
        }
        ++n_miss;
        __syncwarp();
    }
    __syncwarp();
    for (int s = lane; s < S; s += 32) {
        a.st.expert[s] = ex[s];
        a.st.count[s] = cnt[s];
        a.st.last_use[s] = lu[s];
    }
    const unsigned long long base = *a.trace_n;
    if (lane < k && base + lane < a.trace_cap) {
        tf_cache_event ev;
        ev.step = (int32_t)step;
        ev.layer = a.layer;
        ev.expert = ids[lane];
        ev.hit = hit[lane];
        ev.slot = slot[lane];
        ev.evicted = evicted[lane];
        a.trace[base + lane] = ev;
    }
    if (lane == 0) {
        *a.trace_n = base + (unsigned long long)k;
        a.st.miss[0] = n_miss;
        a.st.miss[1] = k - n_miss;
        a.st.ctr[0] = step + 1;
        a.st.ctr[1] += k - n_miss;
        a.st.ctr[2] += n_miss;
    }
}

// Copy the layer's missing experts from the host store into their slots: chunks of FETCH_CHUNK
// bytes dealt over the CTAs, 16-byte loads straight from (mapped) host memory.
__global__ void __launch_bounds__(FETCH_THREADS) k_fetch(const char* __restrict__ store, char* __restrict__ pool,
                                                         unsigned long long slot_bytes, unsigned long long payload,
                                                         const int32_t* __restrict__ miss, int layer, int E, int S) {
    const int n = miss[0];
    const int cpe = (int)((payload + FETCH_CHUNK - 1) / FETCH_CHUNK);
    for (int c = blockIdx.x; c < n * cpe; c += gridDim.x) {
        const int m = c / cpe;
        const unsigned long long off = (unsigned long long)(c - m * cpe) * FETCH_CHUNK;
        const int e = miss[2 + m], sl = miss[2 + TF_MAX_K + m];
        const uint4* src = reinterpret_cast<const uint4*>(store + ((unsigned long long)layer * E + e) * slot_bytes + off);
        uint4* dst = reinterpret_cast<uint4*>(pool + ((unsigned long long)layer * S + sl) * slot_bytes + off);
        const unsigned long long rem = payload - off;
        const int nvec = (int)((rem < FETCH_CHUNK ? rem : FETCH_CHUNK) / 16);
        uint4 v[FETCH_UNROLL];
#pragma unroll
        for (int u = 0; u < FETCH_UNROLL; ++u) {
            const int i = u * FETCH_THREADS + threadIdx.x;
            if (i < nvec) v[u] = __ldcs(src + i);
        }
#pragma unroll
        for (int u = 0; u < FETCH_UNROLL; ++u) {
            const int i = u * FETCH_THREADS + threadIdx.x;
            if (i < nvec) dst[i] = v[u];
        }
    }
}

struct Carve {
    size_t err, trace_n, layers0, per_layer, trace, total;
    size_t expert, count, last_use, slot_of, ctr, miss;
};

Carve carve(int L, int S, int E, size_t cap) {
    Carve c;
    size_t o = 0;
    c.err = o; o += 128;
    c.trace_n = o; o += 128;
    c.layers0 = o;
    size_t p = 0;
    c.expert = p; p += align_up((size_t)S * 4, 64);
    c.count = p; p += align_up((size_t)S * 8, 64);
    c.last_use = p; p += align_up((size_t)S * 8, 64);
    c.slot_of = p; p += align_up((size_t)E * 4, 64);
    c.ctr = p; p += 64;
    c.miss = p; p += align_up((size_t)(2 + 2 * TF_MAX_K) * 4, 64);
    c.per_layer = align_up(p, 256);
    o += (size_t)L * c.per_layer;
    c.trace = o; o += align_up(cap * sizeof(tf_cache_event), 256);
    c.total = o;
    return c;
}

}  // namespace devcache
}  // namespace tf

using namespace tf;

struct tf_device_cache {
    int n_layers = 0, n_slots = 0, n_experts = 0;
    size_t slot_bytes = 0, trace_cap = 0;
    char* pool = nullptr;
    const char* store = nullptr;     // device address of the mapped host store
    char* state = nullptr;
    devcache::Carve cv;
    int fetch_ctas = 32;
};

namespace {

devcache::LayerState layer_state(const tf_device_cache* c, int l) {
    char* b = c->state + c->cv.layers0 + (size_t)l * c->cv.per_layer;
    devcache::LayerState s;
    s.expert = reinterpret_cast<int32_t*>(b + c->cv.expert);
    s.count = reinterpret_cast<long long*>(b + c->cv.count);
    s.last_use = reinterpret_cast<long long*>(b + c->cv.last_use);
    s.slot_of = reinterpret_cast<int32_t*>(b + c->cv.slot_of);
    s.ctr = reinterpret_cast<long long*>(b + c->cv.ctr);
    s.miss = reinterpret_cast<int32_t*>(b + c->cv.miss);
    return s;
}

}  // namespace

extern "C" {

size_t tf_device_cache_state_bytes(int n_layers, int n_slots, int n_experts, size_t trace_capacity) {
    if (n_layers < 1 || n_slots < 1 || n_slots > devcache::MAX_SLOTS || n_experts < 1 || n_experts > TF_MAX_E)
        return 0;
    return devcache::carve(n_layers, n_slots, n_experts, trace_capacity).total;
}

tf_status tf_device_cache_create(int n_layers, int n_slots, int n_experts, size_t slot_bytes, void* d_slot_pool,
                                 const void* h_expert_store, void* d_state, size_t state_bytes, size_t trace_capacity,
                                 tf_device_cache** out) {
    const char* fn = "tf_device_cache_create";
    if (!out) return fail(TF_ERR_INVALID_ARG, "%s: out is NULL", fn);
    *out = nullptr;
    if (n_layers < 1 || n_slots < 1 || n_slots > devcache::MAX_SLOTS || n_experts < 1 || n_experts > TF_MAX_E)
        return fail(TF_ERR_INVALID_ARG, "%s: n_layers=%d n_slots=%d (1..%d) n_experts=%d out of range", fn, n_layers,
                    n_slots, devcache::MAX_SLOTS, n_experts);
    if (!d_slot_pool || !h_expert_store || !d_state)
        return fail(TF_ERR_INVALID_ARG, "%s: slot pool, host store and state are required", fn);
    if (slot_bytes == 0 || slot_bytes % 16 || !aligned16(d_slot_pool) || !aligned16(h_expert_store))
        return fail(TF_ERR_INVALID_ARG, "%s: slot size, pool and store must be 16-byte aligned", fn);
    const devcache::Carve cv = devcache::carve(n_layers, n_slots, n_experts, trace_capacity);
    if (state_bytes < cv.total || (reinterpret_cast<uintptr_t>(d_state) & 255))
        return fail(TF_ERR_INVALID_ARG, "%s: state misaligned or smaller than %zu bytes", fn, cv.total);
    void* dstore = nullptr;
    if (cudaError_t e = cudaHostGetDevicePointer(&dstore, const_cast<void*>(h_expert_store), 0)) {
        cudaGetLastError();
        return fail(TF_ERR_NOT_SUPPORTED, "%s: the host store is not mapped for device access: %s", fn,
                    cudaGetErrorString(e));
    }
    tf_device_cache* c = new (std::nothrow) tf_device_cache();
    if (!c) return fail(TF_ERR_OOM, "%s: out of host memory", fn);
    c->n_layers = n_layers;
    c->n_slots = n_slots;
    c->n_experts = n_experts;
    c->slot_bytes = slot_bytes;
    c->trace_cap = trace_capacity;
    c->pool = static_cast<char*>(d_slot_pool);
    c->store = static_cast<const char*>(dstore);
    c->state = static_cast<char*>(d_state);
    c->cv = cv;
    // every slot empty, no expert resident, counters and trace at zero
    cudaError_t e = cudaMemset(c->state, 0, cv.total);
    for (int l = 0; l < n_layers && e == cudaSuccess; ++l) {
        const devcache::LayerState s = layer_state(c, l);
        e = cudaMemset(s.expert, 0xff, (size_t)n_slots * 4);
        if (e == cudaSuccess) e = cudaMemset(s.slot_of, 0xff, (size_t)n_experts * 4);
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        delete c;
        return cuda_status(e, fn);
    }
    *out = c;
    return TF_OK;
}

tf_status tf_device_cache_set_fetch_ctas(tf_device_cache* c, int ctas) {
    if (!c || ctas < 1 || ctas > 4096) return fail(TF_ERR_INVALID_ARG, "tf_device_cache_set_fetch_ctas: bad arguments");
    c->fetch_ctas = ctas;
    return TF_OK;
}

tf_status tf_device_cache_counters(tf_device_cache* c, int64_t* hits, int64_t* misses, int64_t* events, void* stream) {
    const char* fn = "tf_device_cache_counters";
    if (!c) return fail(TF_ERR_INVALID_ARG, "%s: NULL", fn);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int64_t h = 0, m = 0;
    for (int l = 0; l < c->n_layers; ++l) {
        long long ctr[3];
        if (cudaError_t e = cudaMemcpyAsync(ctr, layer_state(c, l).ctr, sizeof(ctr), cudaMemcpyDeviceToHost, st))
            return cuda_status(e, fn);
        if (cudaError_t e = cudaStreamSynchronize(st)) return cuda_status(e, fn);
        h += ctr[1];
        m += ctr[2];
    }
    unsigned long long n = 0;
    if (cudaError_t e = cudaMemcpyAsync(&n, c->state + c->cv.trace_n, 8, cudaMemcpyDeviceToHost, st))
        return cuda_status(e, fn);
    if (cudaError_t e = cudaStreamSynchronize(st)) return cuda_status(e, fn);
    if (hits) *hits = h;
    if (misses) *misses = m;
    if (events) *events = (int64_t)n;
    return TF_OK;
}

tf_status tf_device_cache_trace(tf_device_cache* c, tf_cache_event* buf, size_t cap, size_t* n, void* stream) {
    const char* fn = "tf_device_cache_trace";
    if (!c || !n || (cap && !buf)) return fail(TF_ERR_INVALID_ARG, "%s: bad arguments", fn);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned long long total = 0;
    if (cudaError_t e = cudaMemcpyAsync(&total, c->state + c->cv.trace_n, 8, cudaMemcpyDeviceToHost, st))
        return cuda_status(e, fn);
    if (cudaError_t e = cudaStreamSynchronize(st)) return cuda_status(e, fn);
    size_t have = total < c->trace_cap ? (size_t)total : c->trace_cap;
    if (have > cap) have = cap;
    if (have) {
        if (cudaError_t e = cudaMemcpyAsync(buf, c->state + c->cv.trace, have * sizeof(tf_cache_event),
                                            cudaMemcpyDeviceToHost, st))
            return cuda_status(e, fn);
        if (cudaError_t e = cudaStreamSynchronize(st)) return cuda_status(e, fn);
    }
    *n = (size_t)total;
    return TF_OK;
}

tf_status tf_device_cache_state(tf_device_cache* c, int layer, int32_t* expert, int64_t* count, int64_t* last_use,
                                void* stream) {
    const char* fn = "tf_device_cache_state";
    if (!c || layer < 0 || layer >= c->n_layers) return fail(TF_ERR_INVALID_ARG, "%s: bad arguments", fn);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const devcache::LayerState s = layer_state(c, layer);
    const size_t S = (size_t)c->n_slots;
    cudaError_t e = cudaSuccess;
    if (expert) e = cudaMemcpyAsync(expert, s.expert, S * 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && count) e = cudaMemcpyAsync(count, s.count, S * 8, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && last_use) e = cudaMemcpyAsync(last_use, s.last_use, S * 8, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return cuda_status(e, fn);
}

tf_status tf_device_cache_destroy(tf_device_cache* c) {
    delete c;
    return TF_OK;
}

tf_status tf_layer_step_device_cache(tf_layer* l, tf_device_cache* c, int layer, const void* x, void* out,
                                     const float* logit_bias, int bias_stride, void* compute_stream, void* fetch_stream,
                                     int measure, tf_step_stats* stats) {
    const char* fn = "tf_layer_step_device_cache";
    if (!l || !c || !x || !out || !fetch_stream) return fail(TF_ERR_INVALID_ARG, "%s: null argument", fn);
    const tf_layer_desc& d = l->d;
    if (layer < 0 || layer >= c->n_layers) return fail(TF_ERR_INVALID_ARG, "%s: bad layer %d", fn, layer);
    if (c->n_experts != d.E || c->slot_bytes < l->lay.payload || c->n_slots < d.k)
        return fail(TF_ERR_INVALID_ARG, "%s: cache does not match the layer (E, slot size or slot count)", fn);
    if (logit_bias && bias_stride != 0 && bias_stride != d.E)
        return fail(TF_ERR_INVALID_ARG, "%s: bias_stride must be 0 or E", fn);
    if (stats) std::memset(stats, 0, sizeof(*stats));
    clear_error();
    cudaStream_t cs = static_cast<cudaStream_t>(compute_stream), fs = static_cast<cudaStream_t>(fetch_stream);
    int e = 0;
    if (measure && (e = cudaEventRecord(l->ev_t0, cs))) return cuda_status(e, fn);
    e = launch_router_topk(static_cast<const uint16_t*>(x), 1, d.H, static_cast<const uint16_t*>(d.W_r), d.E,
                           logit_bias, bias_stride, d.k, l->idx, l->w, l->logits, l->rms, l->counters, d.eps, cs);
    if (!e) e = cudaEventRecord(l->ev_idx, cs);
    if (e) return cuda_status(e, fn);

    // fetch stream: the LFU decision, then the copies of the misses
    const devcache::LayerState s = layer_state(c, layer);
    if ((e = cudaStreamWaitEvent(fs, l->ev_idx, 0))) return cuda_status(e, fn);
    if (measure && (e = cudaEventRecord(l->ev_c0, fs))) return cuda_status(e, fn);
    devcache::LfuArgs a;
    a.st = s;
    a.idx = l->idx;
    a.k = d.k;
    a.S = c->n_slots;
    a.E = d.E;
    a.layer = layer;
    a.trace = reinterpret_cast<tf_cache_event*>(c->state + c->cv.trace);
    a.trace_n = reinterpret_cast<unsigned long long*>(c->state + c->cv.trace_n);
    a.trace_cap = c->trace_cap;
    a.err = reinterpret_cast<uint32_t*>(c->state + c->cv.err);
    prof_before(TF_KERNEL_OTHER, fs);
    devcache::k_lfu_step<<<1, 32, 0, fs>>>(a);
    devcache::k_fetch<<<c->fetch_ctas, devcache::FETCH_THREADS, 0, fs>>>(c->store, c->pool, c->slot_bytes,
                                                                         l->lay.payload, s.miss, layer, d.E, c->n_slots);
    prof_after(TF_KERNEL_OTHER, fs);
    if ((e = (int)cudaGetLastError())) return cuda_status(e, fn);
    if ((e = cudaEventRecord(l->ev_copies, fs))) return cuda_status(e, fn);

    // compute stream: the shared branch while the copies run, then the routed experts
    ExpertRef none;
    std::memset(&none, 0, sizeof(none));
    DecodeParams p = decode_params(l, x, out, nullptr, none, l->w, l->rms);
    p.ys = d.S > 0 ? l->ys : nullptr;
    if (d.S > 0 && (e = launch_gateup(p, d.k * d.I, d.k * d.I + d.S, cs))) return cuda_status(e, fn);
    if (d.S > 0 && (e = launch_down(p, 0, 1, cs))) return cuda_status(e, fn);
    if (measure && (e = cudaEventRecord(l->ev_shared, cs))) return cuda_status(e, fn);
    if ((e = cudaStreamWaitEvent(cs, l->ev_copies, 0))) return cuda_status(e, fn);
    ExpertRef r;
    std::memset(&r, 0, sizeof(r));
    r.base = c->pool + (size_t)layer * c->n_slots * c->slot_bytes;
    r.stride = c->slot_bytes;
    r.slot_map = s.slot_of;
    r.idx = l->idx;
    r.n_experts = d.E;
    r.n_slots = c->n_slots;
    p.ex = r;
    e = launch_gateup(p, 0, d.k * d.I, cs);
    if (!e) e = launch_down(p, 1, 0, cs);
    if (e) return cuda_status(e, fn);
    if (measure && stats) {
        int32_t hm[2] = {0, 0};
        if ((e = cudaMemcpyAsync(hm, s.miss, sizeof(hm), cudaMemcpyDeviceToHost, cs))) return cuda_status(e, fn);
        if ((e = cudaMemcpyAsync(stats->ids, l->idx, (size_t)d.k * 4, cudaMemcpyDeviceToHost, cs)))
            return cuda_status(e, fn);
        if ((e = cudaStreamSynchronize(cs))) return cuda_status(e, fn);
        stats->misses = hm[0];
        stats->hits = hm[1];
        stats->bytes_fetched = (uint64_t)hm[0] * l->lay.payload;
        float t_shared = 0.f, t_copies = 0.f, t_copy = 0.f;
        if (d.S > 0) cudaEventElapsedTime(&t_shared, l->ev_t0, l->ev_shared);
        cudaEventElapsedTime(&t_copies, l->ev_t0, l->ev_copies);
        cudaEventElapsedTime(&t_copy, l->ev_c0, l->ev_copies);
        stats->shared_ms = t_shared;
        stats->copy_ms = t_copy;
        stats->stall_ms = t_copies > t_shared ? t_copies - t_shared : 0.f;
    }
    return TF_OK;
}

}  // extern "C"
