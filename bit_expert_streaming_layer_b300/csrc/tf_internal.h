// Internal declarations shared by the host code and the CUDA translation units
// of libtf.so. Not part of the ABI (see include/tf.h).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "tf.h"

namespace tf {

// ------------------------------------------------------------------ errors
void set_error(const char* fmt, ...);
void clear_error();
tf_status fail(tf_status s, const char* fmt, ...);
// Maps a cudaError_t (passed as int) to TF_ERR_CUDA with a message, TF_OK if 0.
tf_status cuda_status(int err, const char* what);

// ------------------------------------------------------------------ layout
struct ExpertLayout {
    int H = 0, I = 0;
    size_t gu_codes = 0;   // offset of the gate/up codes (always 0)
    size_t gu_sb = 0;      // offset of the gate/up {s,b} pairs
    size_t d_codes = 0;    // offset of the down codes
    size_t d_sb = 0;       // offset of the down {s,b} pairs
    size_t payload = 0;    // bytes of one packed expert
    size_t slot = 0;       // payload rounded up to 16 KiB
};
bool expert_layout(int H, int I, ExpertLayout* L);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------ kernel args
// Where the k experts of one token live: either explicit device pointers (the
// cached path, resolved on the host) or a table (base/stride/map + device idx).
struct ExpertRef {
    const char* ptr[TF_MAX_K];   // used when use_ptrs != 0
    const char* base;
    size_t stride;
    const int32_t* slot_map;     // nullable
    const int32_t* idx;          // device [k]
    int use_ptrs;
    int n_experts;               // ids valid in [0, n_experts)
    int n_slots;                 // slot_map entries valid in [0, n_slots)
};

struct DecodeParams {
    const uint16_t* x;           // bf16 [H] (layer input)
    uint16_t* out;               // bf16 [H]
    float* delta;                // nullable fp32 [H]
    int H, I, k, S;
    float eps;
    const float* rms_in;         // nullable device [1]: r from the router (else recomputed)
    ExpertRef ex;
    const float* w;              // device [k]
    const uint16_t* Wsg;         // bf16 [S,H] (S > 0)
    const uint16_t* Wsu;
    const uint16_t* Wsd;         // bf16 [H,S]
    float* h_routed;             // fp32 [k, I]
    float* h_shared;             // fp32 [S]
    float* ys;                   // nullable fp32 [H]: the shared down projection, written by a shared-only down
                                 // launch and added by a routed-only one (so the two can run apart)
    size_t off_gu_sb, off_d_codes, off_d_sb;
};

// Descriptor a layer handle was created with (tf_api.cu).
void layer_desc_of(const tf_layer* l, tf_layer_desc* out);
// Decode-kernel parameters of a layer handle for input x and output out (tf_api.cu).
DecodeParams decode_params(const tf_layer* l, const void* x, void* out, float* delta, const ExpertRef& ex,
                           const float* w, const float* rms_in);

// Limit (ns) of a device-side wait on another warp, role or CTA in the persistent
// kernels: 2 s, unless tf_test_set_wait_limit_ns shortened it (tf_api.cu).
unsigned long long test_wait_limit_ns();

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device); thread-safe. Returns a cudaError_t.
int smem_limit_once(const void* kernel, int bytes);

// Event bracketing of launches while profiling is on (tf_api.cu).
void prof_before(int kind, void* stream);
void prof_after(int kind, void* stream);

// Launchers (defined in tf_decode.cu). They return a CUDA error code (0 = ok).
int launch_router_topk(const uint16_t* x, int T, int H, const uint16_t* Wr, int E, const float* bias,
                       int bias_stride, int k, int32_t* idx, float* w, float* logits, float* rms,
                       uint32_t* counters, float eps, void* stream);
// Row-pair units [u0, u1): routed units are [0, k*I), shared units [k*I, k*I + S).
int launch_gateup(const DecodeParams& p, int u0, int u1, void* stream);
// Down projection + combine: with_routed / with_shared select the terms. Without p.ys:
// out = x + the selected terms. With p.ys: a shared-only launch writes ys = the shared
// term (and no output); a routed-only launch writes out = x + (ys + the routed terms).
int launch_down(const DecodeParams& p, int with_routed, int with_shared, void* stream);
int launch_dequant(const char* blob, int H, int I, int matrix, int format, void* out,
                   size_t off_sb, size_t off_codes, void* stream);

// Experts that stream through a cache while a chunk of tokens runs the grouped
// path (tf_layer_prefill_cached): the chunk's experts are taken in waves; before
// wave w the callback enqueues its fills and makes the compute stream wait for
// them, and fills the wave's row of h_maps: [E] 1 for the wave's experts, then
// [E] the slot of each of them in `pool`.
struct GroupedWaves {
    int n;                                 // waves
    const char* pool;                      // this layer's slots: slot s at pool + s * slot_bytes
    size_t slot_bytes;
    int n_slots;
    int32_t* d_maps;                       // device [n][2][E]
    const int32_t* h_maps;                 // pinned host [n][2][E], filled by before_wave
    int (*before_wave)(void* ctx, int w, void* compute_stream);   // a tf_status
    void* ctx;
};

// The grouped (batched / prefill) layer of tf_grouped.cu: routed experts by
// tcgen05 GEMMs over the token x expert permutation and, when S > 0, the bf16
// shared expert by the same GEMM kernel with TMA-loaded weights.
struct GroupedArgs {
    const void* x;                 // bf16 [T, H]
    void* out;                     // bf16 [T, H]
    int T;
    const tf_expert_table* table;  // resident experts
    int E, k, H, I;
    const int32_t* idx;            // device [T, k]
    const float* w;                // device [T, k]
    float* delta;                  // nullable fp32 [T, H]
    int32_t* perm_out;             // nullable [T*k]
    int32_t* counts_out;           // nullable [E]
    const void* Wsg;               // bf16 [S, H]; S = 0: no shared expert
    const void* Wsu;               // bf16 [S, H]
    const void* Wsd;               // bf16 [H, S]
    int S;
    float eps;
    const float* rms_in;           // nullable device [T]: each token's RMS scale as the router computed it
    void* ws;
    size_t ws_bytes;
    const GroupedWaves* waves;     // nullable: the experts stream through a cache (else the table holds them all)
};
size_t grouped_workspace_bytes(int T, int H, int I, int E, int k, int S);
tf_status grouped_run(const GroupedArgs& a, void* stream, const char* fn);

}  // namespace tf

// Per-layer LFU metadata (host). Defined here so the layer step can reach the
// slot pool; the policy itself lives in tf_host.cpp.
struct tf_expert_cache {
    int n_layers = 0, n_slots = 0, n_experts = 0;
    size_t slot_bytes = 0;
    void* d_slot_pool = nullptr;
    std::vector<int32_t> expert;     // [L][S], -1 = empty
    std::vector<int64_t> count;      // uses since admission
    std::vector<int64_t> last_use;   // step of the last use
    std::vector<tf_cache_event> trace;
    std::vector<cudaStream_t> copy_streams;   // set by tf_expert_cache_set_copy_streams (empty: the call's)
    std::vector<cudaEvent_t> copy_events;     // one per copy stream, owned
};

// A layer handle: its descriptor and the buffers carved from its workspace (tf_api.cu).
struct tf_layer {
    tf_layer_desc d;
    int T_max = 0;
    tf::ExpertLayout lay;
    char* ws = nullptr;
    size_t ws_bytes = 0;
    char* grouped_ws = nullptr;      // T_max > 1 only
    size_t grouped_bytes = 0;
    uint32_t* counters = nullptr;
    float* logits = nullptr;
    int32_t* idx = nullptr;
    float* w = nullptr;
    float* rms = nullptr;
    float* h_routed = nullptr;
    float* h_shared = nullptr;
    float* ys = nullptr;             // fp32 [H]: the shared down projection of the cached steps
    int32_t* h_idx = nullptr;        // pinned staging for the cached step
    cudaEvent_t ev_idx = nullptr, ev_copies = nullptr, ev_t0 = nullptr, ev_shared = nullptr, ev_c0 = nullptr;
    // chunked prefill through a cache (T_max > 1): the chunk's ids and the waves' expert masks and slot maps
    int max_waves = 0;               // ceil(E / k): a wave holds at least k experts (n_slots >= k)
    int32_t* h_chunk_ids = nullptr;  // pinned [T_max * k]
    int32_t* h_wave_maps = nullptr;  // pinned [max_waves][2][E]
    int32_t* d_wave_maps = nullptr;  // workspace [max_waves][2][E]
    cudaEvent_t ev_wave = nullptr;
};
