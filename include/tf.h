/*
 * tf.h -- C ABI of the streamed-expert MoE layer for NVIDIA B300 (sm_103a).
 *
 * The operations follow the per-token, per-layer flow described on the page
 * "Como executar um modelo de 26 bilhoes de parametros em dois gigabytes de
 * memoria em um Mac comum" (devtrends.cc), section "Qual e o principal truque
 * da arquitetura": a router picks 8 experts per layer, a 16-slot LFU cache of
 * expert weights is consulted, missing experts are fetched from slower memory
 * while the GPU computes the shared-expert branch, and the expert FFNs run on
 * the 4-bit weights. The same page, section "Sem dependencias do llama.cpp e
 * MLX", lists the kernels (quantisation, GEMV, MoE, RMSNorm); section
 * "Desempenho no mundo real" describes prefill in which one loaded expert
 * serves a group of rows (the grouped entry point).
 *
 * Conventions
 *  - Every call returns tf_status; nothing throws across the ABI.
 *    tf_last_error() gives a thread-local message for the last failure.
 *  - Arguments are checked before any launch. A bad argument returns
 *    TF_ERR_INVALID_ARG and launches nothing.
 *  - The caller owns every device and pinned-host buffer passed in and keeps it
 *    alive until the work enqueued on the given stream(s) has finished. The
 *    library owns only its opaque handles (tf_expert_cache, tf_layer) and what
 *    they allocate at creation (a few pinned staging words and CUDA events),
 *    and frees them in *_destroy.
 *  - Device work is enqueued on the caller's cudaStream_t (passed as void*;
 *    NULL = legacy default stream). Calls return after enqueueing, except the
 *    cached layer step, whose one host wait is documented there.
 *  - No call allocates device memory: scratch comes from a caller-provided
 *    workspace of the size the matching *_workspace_bytes() returns. A
 *    workspace must be zero-filled once before its first use; the kernels
 *    leave it in that state.
 *  - bf16 and fp16 values are passed as their 16-bit patterns (uint16_t) or as
 *    untyped device pointers; fp32 as float.
 *
 * Number formats
 *  - Hidden states x, out: bf16, row-major [T, H].
 *  - Router weights W_r: bf16 [E, H] row-major.
 *  - Shared expert: bf16 gate [S, H], up [S, H], down [H, S], row-major.
 *  - Routed expert: 4-bit affine codes q in 0..15 with one fp16 scale s and one
 *    fp16 bias b per group of 64 consecutive K values of one output row; the
 *    weight is W = s*q + b (fp32, a single rounding since s*q is exact).
 *    Logical shapes: gate [I, H], up [I, H], down [H, I]. H and I are
 *    multiples of 64.
 *
 * Packed expert blob (one contiguous block per expert; offsets from
 * tf_expert_offsets, all 16-byte aligned):
 *    [0] gate/up codes : 2*I rows of H/2 bytes; row 2j = gate row j, row 2j+1 =
 *                        up row j. Byte m of a row holds column 2m in its low
 *                        nibble and column 2m+1 in its high nibble.
 *    [1] gate/up (s,b) : 2*I rows x H/64 groups of {fp16 s, fp16 b} (4 bytes),
 *                        rows interleaved like [0].
 *    [2] down codes    : H rows of I/2 bytes, same nibble order.
 *    [3] down (s,b)    : H rows x I/64 groups of {fp16 s, fp16 b}.
 *  The payload is 3*(I*H/2 + 4*I*H/64) bytes: 3,345,408 B for H = 2816,
 *  I = 704. tf_expert_slot_bytes rounds it up to 16 KiB (3,358,720 B, the
 *  "3.36 MB per expert at 4 bits" of the page "Show HN: mecanismo de codigo
 *  aberto executando Gemma 4 26B em 2 GB de RAM em qualquer Mac com serie M",
 *  section "Abordagem tecnica (MoE + streaming por SSD)"), the stride of a
 *  cache slot and of the resident expert array.
 *
 * Numerics
 *  - RMSNorm: r = 1/sqrt(sum(x^2)/H + eps), unit gain, n = r*x (fp32).
 *  - Router: z_e = r * sum_k W_r[e,k] x_k (+ bias_e). The sum of x^2 and the
 *    router dot products use a fixed order (32 strided partial sums, then a
 *    xor butterfly 16, 8, 4, 2, 1) with IEEE-rounded mul/add/div/sqrt, so the
 *    selected experts are reproducible bit for bit. Top-k: larger logit first,
 *    equal logits -> lower expert index. Routing weights: softmax over the k
 *    selected logits (they sum to 1).
 *  - Expert FFN: g = Wg n, u = Wu n, h = gelu_tanh(g) * u, y = Wd h, fp32.
 *  - Layer: delta = shared(n) + sum_i w_i y_i (i in top-k order, fp32),
 *    out = bf16(x + delta), round to nearest even.
 */
#ifndef TF_H
#define TF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t tf_status;
enum {
    TF_OK = 0,
    TF_ERR_INVALID_ARG = 1,   /* a null pointer, a bad size or alignment; nothing was launched */
    TF_ERR_CUDA = 2,          /* a CUDA runtime call failed; see tf_last_error() */
    TF_ERR_OOM = 3,           /* a pinned or workspace allocation could not be satisfied */
    TF_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out */
    TF_ERR_NOT_SUPPORTED = 5  /* a valid request this build does not implement */
};

#define TF_GROUP 64
#define TF_MAX_K 32
#define TF_MAX_E 1024

/* Thread-local text of the last error, "" if none. Never NULL. */
const char* tf_last_error(void);
/* Static name of a status code. */
const char* tf_status_string(tf_status s);
/* Library version string. */
const char* tf_version(void);

/* ------------------------------------------------------------------ layout */

/* Payload bytes of one packed expert (0 if H or I is not a positive multiple of 64). */
size_t tf_expert_payload_bytes(int H, int I);
/* Payload rounded up to 16 KiB: stride of a cache slot / resident expert. */
size_t tf_expert_slot_bytes(int H, int I);
/* Byte offsets of the four sections of a packed expert (see the header comment). */
tf_status tf_expert_offsets(int H, int I, size_t off[4]);

/*
 * Host-side packer (no GPU). Inputs are the logical matrices, concatenated in
 * the order gate, up, down:
 *   q : uint8 codes 0..15, gate [I*H] then up [I*H] then down [H*I] (row-major)
 *   s : fp16 scales, gate [I*H/64], up [I*H/64], down [H*I/64]
 *   b : fp16 biases, same shapes as s
 * blob_out receives tf_expert_payload_bytes(H, I) bytes. A code above 15 is an
 * INVALID_ARG (nothing is written past the check).
 */
tf_status tf_pack_expert(const uint8_t* q, const uint16_t* s, const uint16_t* b, int H, int I,
                         void* blob_out);

/* --------------------------------------------------------------- routing */

/*
 * Router GEMV, top-k and routing weights for T tokens (RMSNorm folded in).
 * Devtrends page, section "Qual e o principal truque da arquitetura": the
 * router of each layer determines which 8 experts the current token needs.
 *   x          device bf16 [T, H]
 *   W_r        device bf16 [E, H]
 *   logit_bias device fp32, NULL, or [E] (bias_stride = 0) or [T, E] (bias_stride = E)
 *   idx        device int32 [T, k]  out: experts, best first
 *   w          device fp32  [T, k]  out: routing weights, sum 1
 *   logits     device fp32  [T, E]  out, nullable: z
 *   rms        device fp32  [T]     out, nullable: r
 *   workspace  device, >= tf_router_workspace_bytes(T, E) bytes, zeroed once
 * 1 <= k <= min(E, 32), E <= 1024, H a positive multiple of 64.
 */
size_t tf_router_workspace_bytes(int T, int E);
tf_status tf_router_topk(const void* x, int T, int H, const void* W_r, int E, const float* logit_bias,
                         int bias_stride, int k, int32_t* idx, float* w, float* logits, float* rms,
                         void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------- expert table */

/*
 * Where the packed experts live in device memory. Expert e is at
 *   base + (slot_of_expert ? slot_of_expert[e] : e) * stride
 * (slot_of_expert is a device int32 [n_experts] map, NULL for a resident
 * array). base and stride must be 16-byte aligned.
 *   n_experts  expert ids are valid in [0, n_experts). The kernels read the ids
 *              (and the map) on the device; an id outside that range, or a map
 *              entry outside [0, n_slots), is never turned into an address: the
 *              call's outputs become NaN instead (the error is seen in the data,
 *              since the call returns before the kernels run).
 *   n_slots    with slot_of_expert: the number of slots at base (map entries
 *              are valid in [0, n_slots)); ignored without a map.
 * In a tf_layer_desc, n_experts = 0 stands for the descriptor's E.
 */
typedef struct {
    const void* base;
    size_t stride;
    const int32_t* slot_of_expert;
    int32_t n_experts;
    int32_t n_slots;
} tf_expert_table;

/* Dequantise one matrix (0 gate, 1 up, 2 down) of a packed device expert to a
 * dense row-major device array: fp32 (format = 0), bf16 (format = 1) or fp16
 * (format = 2), each the round-to-nearest-even of the fp32 weight s q + b (the
 * grouped GEMMs take fp16 gate/up and bf16 down weights). Parity export. */
tf_status tf_dequant_expert(const void* blob, int H, int I, int matrix, int format, void* out,
                            void* stream);

/* ------------------------------------------------------------- MoE FFN */

/*
 * Routed-expert FFN of one token with the weighted combine into the residual:
 *   out = x + sum_i w[i] * E_idx[i](RMSNorm(x))      (i in top-k order)
 * table->n_experts >= 1 is required; an id outside it makes out (and delta) NaN.
 * HN page "Show HN: ...", section "Abordagem tecnica (MoE + streaming por
 * SSD)": only a small subset of experts is active per token; devtrends page,
 * section "Sem dependencias do llama.cpp e MLX": fused 4-bit GEMV and MoE kernels.
 *   x, out     device bf16 [H]; out may alias x
 *   idx, w     device int32 [k], fp32 [k] (e.g. from tf_router_topk)
 *   delta      device fp32 [H], nullable: the fp32 update out - x before rounding
 *   workspace  >= tf_moe_decode_workspace_bytes(H, I, k), zeroed once
 */
size_t tf_moe_decode_workspace_bytes(int H, int I, int k);
tf_status tf_moe_ffn_decode(const void* x, void* out, const tf_expert_table* table, const int32_t* idx,
                            const float* w, int k, int H, int I, float* delta, void* workspace,
                            size_t ws_bytes, void* stream);

/*
 * tf_moe_ffn_decode for callers that cannot allocate device memory. The pages
 * have no counterpart: this entry point exists for hosts such as a plugin
 * inside another runtime that owns the device heap, code that runs while a
 * stream is being captured, or an embedded loop with a fixed memory budget,
 * where cudaMalloc is unavailable or forbidden and no workspace can be
 * provided.
 *
 * Same operation, arguments and result as tf_moe_ffn_decode, minus the
 * workspace. The k x I fp32 gate/up scratch comes from a fixed array compiled
 * into libtf.so (TF_NOALLOC_MAX_KI floats, 256 KiB), which every GPU that
 * loads the library keeps until the process exits. The call allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *  - k * I > TF_NOALLOC_MAX_KI returns TF_ERR_INVALID_ARG (nothing launched);
 *    the model shape (k = 8, I = 704) uses 5,632 of the 65,536 floats.
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress) and keeps it for later
 *    calls on that device; make that first call before any stream capture.
 *  - Every call, on any stream, uses the same array. Calls whose kernels
 *    overlap on the GPU (other streams, or host threads racing each other)
 *    race on it and produce wrong results: serialise them. The scratch needs
 *    no zeroing: each call overwrites all of it that it reads.
 */
#define TF_NOALLOC_MAX_KI 65536
tf_status tf_moe_ffn_decode_noalloc(const void* x, void* out, const tf_expert_table* table,
                                    const int32_t* idx, const float* w, int k, int H, int I,
                                    float* delta, void* stream);

/*
 * Grouped (batched / prefill) routed-expert FFN for T tokens: tokens are
 * grouped by expert (histogram, exclusive scan, stable permutation by
 * (expert, token, rank)), each expert's rows run as one dequant-to-16-bit
 * tensor-core GEMM with fp32 accumulation (gate/up with the GELU gate fused,
 * then down), and each token sums its k results in top-k order:
 *   out[t] = x[t] + sum_i w[t,i] * E_idx[t,i](RMSNorm(x[t]))
 * Numerics (tcgen05 kind::f16, fp32 accumulation): the gate/up GEMM takes fp16
 * operands, the weights dequantised to fp16 (RN of the fp32 s q + b) and x p,
 * p = 2^e the power of two of the token's RMS scale r = m 2^e (m in [1, 2)), an
 * exact scaling that keeps the operand near unit size; m multiplies the gate
 * and up sums in fp32 (g = m (Wg (x p))), equal in real arithmetic to Wg (r x).
 * The down GEMM takes bf16 operands: the weights dequantised to bf16 and h
 * rounded to bf16. In tf_layer_step with T > 1 the shared expert's GEMMs take
 * its bf16 weights with x itself and h in bf16, r applied after the gate and up
 * sums.
 * Devtrends page, section "Desempenho no mundo real": during prefill one
 * loaded expert is applied to a whole group of rows at once.
 *   x, out     device bf16 [T, H] (out must not alias x)
 *   idx, w     device int32 [T, k], fp32 [T, k]
 *   delta      device fp32 [T, H], nullable
 *   perm_out   device int32 [T*k], nullable: the (expert, token, rank)-sorted pair order
 *   counts_out device int32 [E], nullable: tokens per expert
 */
size_t tf_moe_grouped_workspace_bytes(int T, int H, int I, int E, int k);
tf_status tf_moe_ffn_grouped(const void* x, void* out, int T, const tf_expert_table* table, int E,
                             const int32_t* idx, const float* w, int k, int H, int I, float* delta,
                             int32_t* perm_out, int32_t* counts_out, void* workspace, size_t ws_bytes,
                             void* stream);

/* ---------------------------------------------------------- expert cache */

/*
 * Per-layer LFU cache of expert slots in HBM (metadata on the host).
 * Devtrends page, section "Qual e o principal truque da arquitetura": the
 * runtime checks a local expert cache of 16 slots managed by LFU and loads a
 * missing expert from storage. Policy, per (step, layer):
 *  - lookup: each resident id is a hit (count += 1, last_use = step);
 *  - admit (each miss, in top-k order): the lowest empty slot, else the slot
 *    not holding any of the pinned ids with the smallest count, then the
 *    oldest last_use, then the lowest index; it restarts at count 1,
 *    last_use = step. Counts never decay.
 * d_slot_pool (caller-owned, may be NULL for metadata-only use) holds
 * n_layers * n_slots slots of slot_bytes each: slot s of layer l is at
 * d_slot_pool + (l * n_slots + s) * slot_bytes.
 * Every lookup/admit appends (step, layer, expert, hit, slot, evicted) events
 * to an internal trace, read back with tf_expert_cache_trace.
 */
typedef struct tf_expert_cache tf_expert_cache;

typedef struct {
    int32_t step, layer, expert, hit, slot, evicted;
} tf_cache_event;

tf_status tf_expert_cache_create(int n_layers, int n_slots, int n_experts, size_t slot_bytes,
                                 void* d_slot_pool, tf_expert_cache** out);
/* ids[n] in top-k order -> slot_or_minus1[n], hit[n]; hits are counted. */
tf_status tf_expert_cache_lookup(tf_expert_cache* c, int layer, int64_t step, const int32_t* ids, int n,
                                 int32_t* slot_or_minus1, uint8_t* hit);
/* Pick and claim a slot for a missing expert (metadata only; the copy is the caller's). */
tf_status tf_expert_cache_admit(tf_expert_cache* c, int layer, int64_t step, int32_t expert,
                                const int32_t* pinned_ids, int n_pinned, int32_t* slot,
                                int32_t* evicted_or_minus1);
/* Mark a slot empty again (used to roll back an admit whose copy failed). */
tf_status tf_expert_cache_invalidate(tf_expert_cache* c, int layer, int32_t slot);
/* Copy up to cap trace events into buf (oldest first); *n = number of events recorded in total. */
tf_status tf_expert_cache_trace(tf_expert_cache* c, tf_cache_event* buf, size_t cap, size_t* n);
/* Slot contents of one layer: expert id (-1 empty), count and last_use per slot. */
tf_status tf_expert_cache_state(tf_expert_cache* c, int layer, int32_t* expert, int64_t* count,
                                int64_t* last_use);
tf_status tf_expert_cache_destroy(tf_expert_cache* c);

/*
 * Copy streams for the miss fills of tf_layer_step (the pages' parallel reads
 * of several experts, HN page, section "Abordagem tecnica (MoE + streaming por
 * SSD)": parallel pread instead of mmap). With n >= 1 streams set, the k-th
 * miss of a step is copied on streams[k mod n] (instead of the call's
 * copy_stream) and the compute stream waits for all of them. n = 0 goes back
 * to the call's copy_stream. The streams must outlive their use.
 */
tf_status tf_expert_cache_set_copy_streams(tf_expert_cache* c, void* const* streams, int n);

/* ------------------------------------------------- device-side cache metadata */

/*
 * The same per-layer LFU expert cache, with its metadata in device memory, so
 * that a cached step never waits on the host. Per layer and token:
 *  - a one-warp kernel applies the policy of tf_expert_cache (lookup, then the
 *    misses in top-k order: lowest empty slot, else the smallest count among
 *    the slots not holding one of the step's ids, then the oldest last use,
 *    then the lowest slot) to the k ids the router wrote, updates the slot map
 *    (expert -> slot) and writes the layer's miss list;
 *  - a copy kernel moves every missing expert from the pinned host store into
 *    its slot, its CTAs reading host memory directly over the bus;
 *  - the routed experts then read their weights through the slot map.
 * The step number of each layer is counted on the device (0 for the layer's
 * first lookup, then 1, 2, ...), as last_use and in the trace.
 * The caller owns d_state (tf_device_cache_state_bytes, 256-byte aligned), the
 * slot pool (n_layers * n_slots slots of slot_bytes; slot s of layer l at
 * d_slot_pool + (l * n_slots + s) * slot_bytes) and the host store (pinned and
 * mapped for device access, which cudaHostAlloc and cudaHostRegister memory is
 * on 64-bit systems with unified addressing; expert (l, e) at
 * h_expert_store + (l * n_experts + e) * slot_bytes). tf_device_cache_create
 * initialises d_state synchronously (every slot empty). Up to trace_capacity
 * events (step, layer, expert, hit, slot, evicted) are recorded on the device.
 * 1 <= n_slots <= 1024, n_experts <= TF_MAX_E.
 */
typedef struct tf_device_cache tf_device_cache;
size_t tf_device_cache_state_bytes(int n_layers, int n_slots, int n_experts, size_t trace_capacity);
tf_status tf_device_cache_create(int n_layers, int n_slots, int n_experts, size_t slot_bytes, void* d_slot_pool,
                                 const void* h_expert_store, void* d_state, size_t state_bytes,
                                 size_t trace_capacity, tf_device_cache** out);
/* CTAs of the copy kernel (default 32). */
tf_status tf_device_cache_set_fetch_ctas(tf_device_cache* c, int ctas);
/* Totals since creation: lookups that hit, misses (= experts copied) and events recorded. Synchronises stream. */
tf_status tf_device_cache_counters(tf_device_cache* c, int64_t* hits, int64_t* misses, int64_t* events,
                                   void* stream);
/* Up to cap recorded events, oldest first; *n = events recorded in total. Synchronises stream. */
tf_status tf_device_cache_trace(tf_device_cache* c, tf_cache_event* buf, size_t cap, size_t* n, void* stream);
/* Slot contents of one layer (expert or -1, count, last_use). Synchronises stream. */
tf_status tf_device_cache_state(tf_device_cache* c, int layer, int32_t* expert, int64_t* count, int64_t* last_use,
                                void* stream);
tf_status tf_device_cache_destroy(tf_device_cache* c);

/* ------------------------------------------------------------ layer step */

/*
 * One MoE layer (no attention): router + top-k, optional shared expert,
 * routed experts and the combine. With a cache, missing experts are copied
 * from pinned host memory by the copy engine on copy_stream while the shared
 * expert runs on compute_stream (the pages' overlap of expert reads with the
 * shared-expert branch, devtrends page, section "Qual e o principal truque da
 * arquitetura").
 */
typedef struct {
    int H, I, E, k, S;          /* S = shared-expert width, 0 = no shared expert */
    float eps;                  /* RMSNorm epsilon (1e-6 in the model configuration) */
    const void* W_r;            /* device bf16 [E, H] */
    const void* W_sg;           /* device bf16 [S, H] or NULL when S = 0 */
    const void* W_su;           /* device bf16 [S, H] */
    const void* W_sd;           /* device bf16 [H, S] */
    tf_expert_table experts;    /* resident experts (used when no cache is given) */
} tf_layer_desc;

typedef struct tf_layer tf_layer;

/* Workspace of a layer handle for up to T_max tokens per step. */
size_t tf_layer_workspace_bytes(const tf_layer_desc* d, int T_max);
/* The handle copies the descriptor and binds the caller's zeroed workspace. */
tf_status tf_layer_create(const tf_layer_desc* d, int T_max, void* workspace, size_t ws_bytes,
                          tf_layer** out);
tf_status tf_layer_destroy(tf_layer* l);
/* Device pointers to the routing of the last step: idx [T,k], w [T,k], logits [T,E], rms [T]. */
tf_status tf_layer_routing(tf_layer* l, int32_t** idx, float** w, float** logits, float** rms);

typedef struct {
    int32_t hits, misses;          /* cache lookups of this step (0 without a cache) */
    uint64_t bytes_fetched;        /* host -> device expert bytes enqueued */
    float copy_ms;                 /* copy-stream time of the miss fills (measure = 1 only) */
    float shared_ms;               /* compute-stream time of the shared-expert branch (measure = 1) */
    float stall_ms;                /* max(0, copies end - shared branch end) (measure = 1) */
    int32_t ids[TF_MAX_K];         /* the k selected experts in top-k order (cached step only; the
                                      host reads them anyway to decide the copies) */
} tf_step_stats;

/*
 * Size in bytes of a structure of this ABI, for bindings to check their own
 * layout against the library's: which = 0 tf_expert_table, 1 tf_layer_desc,
 * 2 tf_step_stats, 3 tf_cache_event, 4 tf_prefill_stats, 5 tf_attn_desc; 0 for
 * any other value.
 */
size_t tf_struct_bytes(int which);

/*
 * out = layer(x). T tokens (T = 1 with a cache). logit_bias as in tf_router_topk.
 * Without a cache all work is enqueued on compute_stream and the call returns.
 * T > 1 (at most the handle's T_max; batched decode or prefill): the router for
 * all T tokens, then the grouped path of tf_moe_ffn_grouped (same requirements:
 * H a multiple of 128 up to 2816, I a multiple of 64) with the shared expert
 * (S a multiple of 64) run by the same tcgen05 GEMM kernel on its bf16
 * weights; out = bf16(x + shared + sum_i w_i y_i), with the numerics of
 * tf_moe_ffn_grouped. stats stay zero for T > 1.
 * With a cache (T = 1), the call enqueues the router and the shared branch,
 * waits on the host for the k selected ids (one small device->host copy: the
 * CPU decides the I/O), updates the LFU metadata for layer `layer` at `step`,
 * enqueues one cudaMemcpyAsync per miss from h_expert_store (pinned, expert
 * (layer, e) at h_expert_store + (layer*E + e) * slot_bytes) on copy_stream,
 * makes compute_stream wait for them, enqueues the routed experts and returns.
 * If a copy cannot be enqueued the admitted slots of this step are rolled back
 * to empty and TF_ERR_CUDA is returned. stats (nullable) is filled; with
 * measure = 1 the call also synchronises to time the copy and shared branches.
 */
tf_status tf_layer_step(tf_layer* l, tf_expert_cache* cache, int layer, int64_t step,
                        const void* h_expert_store, const void* x, void* out, int T,
                        const float* logit_bias, int bias_stride, void* compute_stream,
                        void* copy_stream, int measure, tf_step_stats* stats);

/*
 * One token through layer `layer` with a device-metadata cache: on
 * compute_stream the router and the shared-expert branch (gate/up and down,
 * the latter into an fp32 buffer); on fetch_stream, after the router, the LFU
 * kernel and the copy kernel; then compute_stream waits for fetch_stream and
 * runs the routed experts and the combine, out = bf16(x + shared + sum w_i y_i),
 * the same arithmetic as tf_layer_step. Nothing waits on the host: the call
 * only enqueues (its `step` is counted on the device), unless measure = 1,
 * which synchronises to fill stats (hits, misses, bytes of this call; the
 * shared-branch and copy times, and the stall of the routed experts beyond the
 * shared branch). stats may be NULL.
 */
tf_status tf_layer_step_device_cache(tf_layer* l, tf_device_cache* c, int layer, const void* x, void* out,
                                     const float* logit_bias, int bias_stride, void* compute_stream,
                                     void* fetch_stream, int measure, tf_step_stats* stats);

/*
 * Chunked prefill through the streamed-expert cache: T tokens (a chunk, at most
 * the handle's T_max) through layer `layer` whose experts live in the pinned
 * host store behind the LFU cache `c`. Devtrends page, section "Desempenho no
 * mundo real": prefill runs in chunks and one loaded expert serves all of the
 * chunk's rows that need it. Steps:
 *  1. the router for the T tokens on compute_stream; the T x k ids to the host
 *     (the call's one host wait);
 *  2. the chunk's distinct experts in order of first use (token order, then
 *     rank) are cut into waves of n_slots experts; wave w is one LFU step
 *     (step0 + w) of layer `layer`: a lookup of its experts, then an admit of
 *     each miss with the wave's experts pinned, and one cudaMemcpyAsync per
 *     miss on copy_stream (after the previous wave's GEMMs are done with the
 *     slots);
 *  3. per wave, the grouped GEMMs of tf_moe_ffn_grouped on the wave's experts
 *     and their rows, reading the weights from the slots;
 *  4. the shared expert for the T tokens and the combine, as tf_layer_step with
 *     T > 1: out = bf16(x + shared + sum_i w_i y_i), the same values.
 * stats (nullable): waves, hits, misses and bytes copied; the next call on this
 * layer uses step0 + stats->waves. A copy that cannot be enqueued rolls back
 * the slots its wave admitted and returns TF_ERR_CUDA.
 */
typedef struct {
    int32_t waves, hits, misses;
    uint64_t bytes_fetched;
} tf_prefill_stats;
tf_status tf_layer_prefill_cached(tf_layer* l, tf_expert_cache* c, int layer, int64_t step0,
                                  const void* h_expert_store, const void* x, void* out, int T,
                                  const float* logit_bias, int bias_stride, void* compute_stream,
                                  void* copy_stream, tf_prefill_stats* stats);

/*
 * A decode step through L resident layers for one token: x_{l+1} = layer_l(x_l),
 * x_0 = x, out = x_L. Intermediate activations go to `scratch` (device bf16
 * [H], may alias nothing else). logit_bias[l] may be NULL.
 */
tf_status tf_stack_decode(tf_layer* const* layers, int L, const void* x, void* out, void* scratch,
                          const float* const* logit_bias, void* stream);

/* ------------------------------------------------- fused decode stack */

/*
 * The whole stack of resident layers for one decode token in ONE persistent,
 * cooperative kernel (one CTA per SM). Same operations and output as
 * tf_stack_decode (router, top-k, shared expert, routed experts, combine per
 * layer). Every worker warp streams the weight rows of its tasks into its own
 * shared-memory ring (cp.async.bulk) ahead of computing them; optionally the
 * next layer's data-independent weights are prefetched into L2.
 * Values that cross CTAs (router logits, h, layer outputs) are published as
 * tagged words and polled; no device-wide fence or barrier is used. Built for
 * the model shape H = 2816, I = 704, S = 2112, k = 8 and an even E in
 * [8, 256], the same for all layers; other shapes return TF_ERR_NOT_SUPPORTED
 * (use tf_stack_decode).
 *   layers      L layer handles with resident expert tables
 *   logit_bias  host array of L device pointers (fp32 [E]) or NULL; the
 *               pointers are fixed at creation, their contents may change
 *   workspace   device, >= tf_stack_workspace_bytes(L, E), 256-byte aligned;
 *               holds per-layer tagged routing, h and outputs, the launch
 *               epoch and the error word. tf_stack_create initialises it
 *               (synchronously); each launch advances the epoch on the device,
 *               so steps may be enqueued back to back or captured in a graph.
 * Device-side waits are bounded (2 s); when one runs out the kernel records it
 * and returns early. tf_stack_check synchronises the stream, reports that as
 * TF_ERR_TIMEOUT and re-initialises the workspace.
 * Numerics: router logits and the top-k are bit-identical to tf_router_topk;
 * the routed experts' dot products take n and h_routed as 24-bit fixed point
 * with one power-of-two scale per 32 values (integer sums, exact per block),
 * so the outputs differ from tf_stack_decode only by rounding.
 */
/*
 * Attention half of a decoder layer for one decode token: grouped-query
 * self-attention with RoPE and an FP16 KV cache kept in device memory. The
 * devtrends page names hand-written attention and RoPE kernels (section "Sem
 * dependencias do llama.cpp e MLX") and keeps the FP16 KV cache resident
 * (section "Qual e o principal truque da arquitetura"); it gives no shapes or
 * conventions. The operation (the reading this library takes):
 *   r = 1/sqrt(sum(x^2)/H + eps), n = r x            (unit gain, as the MoE layer)
 *   q = Wq n [nq*d], k = Wk n [nkv*d], v = Wv n [nkv*d] (fp32 sums of bf16 products)
 *   RoPE on every head of q and k: for j < d/2 the pair (j, j + d/2) turns by
 *     the angle pos * rope_theta^(-2j/d):  a' = a cos - b sin, b' = b cos + a sin
 *   k_cache[pos] = fp16(k'), v_cache[pos] = fp16(v)   (round to nearest even)
 *   for each q head h, kv head g = h / (nq / nkv):
 *     s_t = (q'_h . k_cache[t]_g) / sqrt(d), t = 0..pos;  a_h = sum_t softmax(s)_t v_cache[t]_g
 *   out = bf16(x + Wo a)
 * A decoder layer is this call followed by the MoE layer (tf_layer_step) on its
 * output. pos is the 0-based position of the token: the call writes the cache
 * rows of pos and reads rows 0..pos, so rows 0..pos-1 must hold the earlier
 * tokens' keys and values (written by earlier calls, or by the caller).
 */
typedef struct {
    int H;                      /* hidden size: a multiple of 8, at most 12000 */
    int n_q_heads, n_kv_heads;  /* n_q_heads a multiple of n_kv_heads */
    int head_dim;               /* 64, 128 or 256; n_q_heads * head_dim at most 12288 */
    int max_seq;                /* rows of each cache */
    float eps;                  /* RMS epsilon, > 0 */
    float rope_theta;           /* RoPE base, > 0 */
    const void* W_q;            /* device bf16 [n_q_heads*head_dim, H], row-major, 16-byte aligned */
    const void* W_k;            /* device bf16 [n_kv_heads*head_dim, H] */
    const void* W_v;            /* device bf16 [n_kv_heads*head_dim, H] */
    const void* W_o;            /* device bf16 [H, n_q_heads*head_dim] */
} tf_attn_desc;

/* Workspace bytes of tf_attn_decode (0 for an invalid descriptor). */
size_t tf_attn_workspace_bytes(const tf_attn_desc* d);
/* Bytes of one cache (K or V): fp16 [max_seq, n_kv_heads, head_dim] (0 for an invalid descriptor). */
size_t tf_attn_cache_bytes(const tf_attn_desc* d);
/*
 * out = attention half of the layer on x (device bf16 [H]; out may not alias x)
 * for the token at position pos, 0 <= pos < max_seq. k_cache, v_cache: device
 * fp16 caches of tf_attn_cache_bytes each, 16-byte aligned, owned by the
 * caller. Four kernels on `stream`, each a programmatic dependent launch of
 * the previous one; the workspace needs no zero-fill.
 */
tf_status tf_attn_decode(const tf_attn_desc* d, const void* x, void* out, int pos, void* k_cache, void* v_cache,
                         void* workspace, size_t ws_bytes, void* stream);

typedef struct tf_stack tf_stack;
size_t tf_stack_workspace_bytes(int L, int E);
tf_status tf_stack_create(tf_layer* const* layers, int L, const float* const* logit_bias, void* workspace,
                          size_t ws_bytes, tf_stack** out);
/* L2 prefetch of the next layer's data-independent weights (router, shared
 * expert) while a layer runs: on (1) or off (0, the default). */
tf_status tf_stack_set_prefetch(tf_stack* s, int on);
/* Phase trace for measurement: with a device buffer of L * 256 * 16 uint64 set,
 * each step writes, for layer l and CTA c, at buffer[(256 l + c) * 16 + slot],
 * the %globaltimer (ns) at which the CTA's control warps 0 held the whole layer
 * input, 1 published x and n, 2 held all router logits, 3 published the top-k,
 * 4 published h_shared, 5 published h_routed; at which 6 the CTA's last worker
 * finished its routed gate/up tasks, 7 its layer work; and at which the CTA's
 * first worker warp had the data of 8 its first item after its shared gate/up
 * items, 9 its first routed gate/up item, 10 its first item after its routed
 * gate/up items, 11 its first routed-down item, 12 its last routed-down item,
 * and 13 finished the layer, 14 finished computing its first routed gate/up
 * item, 15 its last. NULL turns tracing off. */
tf_status tf_stack_set_trace(tf_stack* s, void* buffer, size_t bytes);
/* out = stack(x) for one token; x, out device bf16 [H], 16-byte aligned, out != x. */
tf_status tf_stack_step(tf_stack* s, const void* x, void* out, void* stream);
tf_status tf_stack_check(tf_stack* s, void* stream);
/* Device buffers of one layer of the last step: idx [k], w [k], logits [E], output [H] (bf16;
 * the last layer's output is the call's `out`). */
tf_status tf_stack_layer_buffers(tf_stack* s, int layer, int32_t** idx, float** w, float** logits,
                                 void** act_out);
tf_status tf_stack_destroy(tf_stack* s);

/* ----------------------------------------------------------- measurement */

/*
 * Per-kernel timing for measurement. Between tf_profile_begin and
 * tf_profile_end every launch of the library's kernels is bracketed by two
 * CUDA events recorded on the stream it is launched on (events are created in
 * tf_profile_begin, outside any timed region). tf_profile_end waits for the
 * events and returns, per kernel kind, the summed event time in ms and the
 * number of launches (arrays of TF_KERNEL_COUNT). Launches beyond `capacity`
 * per kind are counted but not timed.
 */
enum {
    TF_KERNEL_ROUTER = 0,      /* RMS scale + router GEMV + top-k */
    TF_KERNEL_GATEUP = 1,      /* fused int4 / bf16 gate-up GEMV with the GELU gate */
    TF_KERNEL_DOWN = 2,        /* down GEMV + weighted combine */
    TF_KERNEL_LAYER = 3,       /* fused persistent decode-layer kernel */
    TF_KERNEL_PERMUTE = 4,     /* token x expert histogram / scan / permute */
    TF_KERNEL_GEMM = 5,        /* grouped dequant-to-16-bit tensor-core GEMM */
    TF_KERNEL_COMBINE = 6,     /* unpermute-combine */
    TF_KERNEL_OTHER = 7,
    TF_KERNEL_COUNT = 8
};
tf_status tf_profile_begin(int capacity);
tf_status tf_profile_end(double* ms, int64_t* launches);

/* ---------------------------------------------------------- test hooks */

/*
 * Failure injection for the miss-fill engine, host side only (no GPU fault):
 * the n-th expert copy enqueued from now on (1-based) is reported as failed
 * instead of being enqueued, as if cudaMemcpyAsync had returned an error.
 * n = 0 disarms. Used to test the roll-back of admitted cache slots.
 */
tf_status tf_test_fail_nth_copy(int n);

/*
 * Limit of the device-side waits on other warps, roles or CTAs in the fused
 * decode kernel (tf_stack_step) and the grouped GEMMs (tf_moe_ffn_grouped, the
 * batched tf_layer_step), for launches enqueued from now on; 0 restores the
 * default of 2 s. A test shortens it to a few ns so that those waits run out
 * without any fault: the kernels record TF_ERR_TIMEOUT (tf_stack_check reports
 * it and resets the stack; the grouped outputs become NaN) and return. Waits of
 * a warp for its own copies and MMAs keep their fixed 2 s bound and ignore the
 * failure, so that no kernel leaves while data is still landing in its shared
 * memory or TMEM.
 */
tf_status tf_test_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* TF_H */
