// Fused persistent decode kernel: a whole stack of MoE layers for one token in
// one cooperative launch (one CTA per SM).
//
// The per-layer flow is the pages' (page "Como executar um modelo de 26 bilhoes
// de parametros em dois gigabytes de memoria em um Mac comum", section "Qual e
// o principal truque da arquitetura"): router -> top-8 -> expert FFNs, with the
// shared-expert branch beside them. What differs is how it is fed on B300.
//
// Work. Ten worker warps per CTA each own a two-stage shared-memory ring,
// filled by cp.async.bulk copies that the warp issues ahead of use, one lane
// per copy (completion on per-stage mbarriers). A layer is cut into tasks, dealt
// round-robin over all worker warps of the grid (continuing from layer to
// layer):
//   router : one row of W_r (bf16), fixed-order dot product -> one logit
//   sgu    : one shared gate/up row pair (bf16, two stages) -> one h_shared
//   rgu    : two gate/up row pairs of one selected expert (int4) -> two h_routed
//   down   : two output rows: shared down (bf16, two stages, needs h_shared)
//            then the eight experts' down rows (int4, one stage, needs
//            h_routed), weighted combine, residual add, bf16 output
// A worker only blocks when its next copy needs the layer's top-8 experts.
// Because the shared-down rows only need h_shared, which is complete long
// before h_routed, they are computed while the routed gate/up work finishes,
// and the routed-down copies are already in flight when h_routed is ready.
//
// Arithmetic. Router and shared rows: fp32 FMA of the bf16 weights. Routed
// rows (int4): integer dot products (dp4a) of the codes against n or h_routed
// held as 24-bit block fixed point (one power-of-two scale per 32 values) in
// byte digits, exact per block, then the group affine in fp32. The control
// warps build the digits: n's while warp 0 selects the top-8, h_routed's in
// place when it is staged.
//
// The layer input is released in two phases: the raw x (enough for the
// router rows, which apply the RMS scale after their dot products), then r
// and n (for the shared gate/up rows). The top-8 is released as soon as the
// selected experts' addresses are known; the softmax weights follow.
//
// Synchronisation. Every value that crosses CTAs is published as a word that
// carries its own tag, and a reader checks the tags of the words it needs:
// router logits as 64-bit (tag, fp32) words, the layer output as 32-bit
// (tag, bf16) words, h as fp32 words whose 4 lowest mantissa bits hold the tag
// (a perturbation of at most 15 ulp). No fence is on the dependency chain:
// GPU-scope fences cost microseconds while the SM's memory pipeline is full of
// weight copies. Relaxed counters (bumped once per CTA per phase, unordered)
// only tell the readers when to look. Four control warps per CTA do the
// looking: they read the whole tagged block (x, logits, h_shared, h_routed)
// with relaxed vector loads, one round trip for the 128 threads (a bulk copy
// would queue behind the weight copies on the SM's copy engine), check the
// tags, write the values to shared memory (reading again while any is stale),
// and publish to the workers with an mbarrier.
// Control warp 0 also computes the CTA's own copy of the top-8. The epoch
// lives in the workspace; CTA 0 advances it once the last layer's output is
// complete, so a launch needs nothing from the host but its pointers.
//
// Optionally each worker prefetches into L2 the data-independent weights
// (router rows, shared expert) of its tasks in the next layer.
#include <cuda_runtime.h>

#include <cstring>
#include <new>
#include <vector>

#include "tf_device.cuh"
#include "tf_internal.h"

namespace tf {
namespace fused {

using namespace dev;

// model shape of the fused kernel
constexpr int H = 2816, I = 704, S = 2112, K = 8;
constexpr int MAX_E = 256;                 // experts per layer supported by the fused kernel
constexpr int NCTRL = 4;                   // control warps per CTA
constexpr int NWORK = 10;                  // worker warps per CTA
constexpr int NT = (NCTRL + NWORK) * 32;
constexpr int NS = 2;                      // ring stages per worker
constexpr int STAGE = 7040;                // bytes per stage
constexpr int HW = H / 8;                  // 352 words (int4) / 16-byte chunks (bf16) per K = H row
constexpr int WPL = HW / 32;               // 11 per lane
constexpr int ROW_BF = H * 2;              // 5632: bf16 row of K = H
constexpr int SROW_BF = S * 2;             // 4224: bf16 row of K = S
constexpr int GU_ROW = H / 2;              // 1408: int4 gate/up row
constexpr int GU_SB = (H / 64) * 4;        // 176: its {s,b} pairs
constexpr int D_ROW = I / 2;               // 352: int4 down row
constexpr int D_SB = (I / 64) * 4;         // 44: its {s,b} pairs
constexpr int N_SGU = S;                   // tasks of one shared row pair
constexpr int N_RGU = K * I / 2;           // tasks of two routed row pairs
constexpr int RGU_PER_EXPERT = I / 2;      // 352
constexpr int N_DN = H / 2;                // tasks of two output rows
constexpr int RGU_BYTES = 4 * GU_ROW + 4 * GU_SB;   // 6336
constexpr int DN_SB_OFF = K * 2 * D_ROW;            // 5632
constexpr int DN_BYTES = DN_SB_OFF + K * 4 * D_SB;  // 7040
constexpr int H_FLOATS = K * I + S;                 // h_routed then h_shared
constexpr unsigned long long OWN_LIMIT_NS = 2000000000ull;  // 2 s: waits for this warp's own copies
constexpr uint32_t HINT_SLEEP_NS = 64;     // pause between two reads of a hint counter
constexpr int CTRL_BAR = 1;                // named barrier of the control warps
static_assert(HW == 32 * WPL, "lane ownership of the K = H words");
static_assert(ROW_BF <= STAGE && RGU_BYTES <= STAGE && DN_BYTES <= STAGE && SROW_BF <= STAGE, "stage size");
static_assert((K * I) % (8 * NCTRL) == 0 && S % (8 * NCTRL) == 0, "control warps check whole 8-float words");

// shared-memory layout
constexpr int OFF_RING = 0;
constexpr int OFF_XS = OFF_RING + NWORK * NS * STAGE;   // bf16 x [H]
constexpr int OFF_N = OFF_XS + H * 2;                    // fp32 n in two halves per word: n[8w..8w+3] at
                                                         // float4 w, n[8w+4..8w+7] at float4 HW + w
constexpr int OFF_SN = OFF_N + H * 4;                    // fp32 word sums of n [HW] (written, no longer read)
constexpr int OFF_H = OFF_SN + HW * 4;                   // tagged fp32 h_routed [K*I], h_shared [S]
constexpr int OFF_Z = OFF_H + H_FLOATS * 4;              // tagged logits [MAX_E] (64-bit words)
constexpr int HG = H / 32;                               // 32-value blocks of n
constexpr int DIG_WORDS = 28;                            // per block: 4 words x 6 digit words, scale, sum, pad
constexpr int OFF_DIG = OFF_Z + MAX_E * 8;               // n as byte digits for the integer dot products [HG]
constexpr int OFF_RT = OFF_DIG + HG * DIG_WORDS * 4;     // routing cache [2 layers]: expert ptrs, weights, ids
constexpr int RT_BYTES = 2 * (K * 8 + K * 4 + K * 4);
constexpr int OFF_BAR = OFF_RT + RT_BYTES;               // mbarriers
enum { B_X = NWORK * NS, B_XS, B_K, B_HS, B_HR, N_BAR };  // B_XS: raw x staged; B_X: r and n too
constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;            // r, epoch, CTA phase counters, stale count
constexpr int MAX_L = 64;                                // layers (tags are epoch * 64 + layer)
constexpr int OFF_DESC = OFF_MISC + 32;                  // copies of the layer descriptors [MAX_L]
constexpr int HB = K * I / 32;                           // 32-value blocks of h_routed (22 per expert)
static_assert(OFF_DIG % 16 == 0 && HG % 8 == 0 && I % 32 == 0, "digit blocks");
static_assert(DIG_WORDS <= 32, "a digit block is no larger than the 32 fp32 values it replaces (in-place staging)");
static_assert(OFF_H % 16 == 0 && OFF_N % 16 == 0 && OFF_RT % 16 == 0 && OFF_BAR % 8 == 0 && OFF_Z % 16 == 0,
              "alignment");

struct LayerDesc {
    const uint16_t* Wr;
    const uint16_t* Wsg;
    const uint16_t* Wsu;
    const uint16_t* Wsd;
    const char* ebase;
    unsigned long long estride;
    const int32_t* slot_map;
    const float* bias;
    unsigned long long* zt;   // tagged logits [E]: (tag << 32) | fp32 bits
    uint32_t* ht;             // tagged h [H_FLOATS]: routed [K*I] then shared [S], tag in the 4 low mantissa bits
    uint32_t* xt;             // tagged output [H]: (tag16 << 16) | bf16
    float* logits;            // plain copies for inspection, written by CTA 0
    int32_t* idx;
    float* w;
    uint16_t* act_out;        // plain bf16 output (the last layer also writes the call's `out`)
    uint32_t* cnt_z;          // router rows scored (pacing hint, += E per launch)
    uint32_t* cnt_hs;         // CTAs whose shared gate/up tasks are done (+= gridDim per launch)
    uint32_t* cnt_hr;         // CTAs whose routed gate/up tasks are done (+= gridDim per launch)
    uint32_t* cnt_out;        // CTAs whose output rows are done (+= gridDim per launch)
    int E;
    float eps;
    int n_slots;              // with slot_map: its entries are valid in [0, n_slots)
    int pad_;
    unsigned long long off_gu_sb, off_d_codes, off_d_sb;
};

constexpr size_t SMEM_BYTES = OFF_DESC + MAX_L * sizeof(LayerDesc);
static_assert(sizeof(LayerDesc) % 8 == 0 && OFF_DESC % 8 == 0, "descriptor copies move 8-byte words");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory with the descriptors");

struct Params {
    const LayerDesc* layers;
    int L;
    const uint16_t* x;
    uint16_t* out;
    uint32_t* err;
    uint32_t* epoch;             // launch epoch (>= 1), advanced by CTA 0 at the end
    int prefetch;                // 1: prefetch the next layer's data-independent weights into L2
    unsigned long long* trace;   // nullable: TRACE_SLOTS %globaltimer stamps per (layer, CTA)
    unsigned long long dep_limit_ns;   // limit of a wait on other warps or CTAs (2 s unless a test shortens it)
};

// Trace slots per (layer, CTA) (ns stamps of %globaltimer), written when
// Params::trace is set: trace[(layer * TRACE_CTAS + cta) * TRACE_SLOTS + slot].
enum {
    TR_X_READY = 0,      // the control warps hold the whole layer input
    TR_X_STAGED = 1,     // ... published x, r, n
    TR_Z_READY = 2,      // ... hold all router logits
    TR_TOPK = 3,         // ... published the top-k
    TR_HS_STAGED = 4,    // ... published h_shared
    TR_HR_STAGED = 5,    // ... published h_routed
    TR_CTA_HR_DONE = 6,  // the CTA's last worker finished its routed gate/up tasks
    TR_CTA_OUT = 7,      // the CTA's last worker finished the layer
    TR_W_SGU_DONE = 8,   // worker 0 had the data of its first item after its shared gate/up items
    TR_W_RGU_READY = 9,  // ... had the data of its first routed gate/up item
    TR_W_RGU_DONE = 10,  // ... had the data of its first item after its routed gate/up items
    TR_W_DS_DONE = 11,   // ... had the data of its first routed-down item (after its shared-down rows)
    TR_W_RD_READY = 12,  // ... had the data of its last routed-down item
    TR_W_DONE = 13,      // ... finished the layer
    TR_W_RGU1_END = 14,  // ... finished computing its first routed gate/up item
    TR_W_RGU_END = 15,   // ... finished computing its last routed gate/up item
    TRACE_SLOTS = 16,
    TRACE_CTAS = 256
};

enum { T_ROUTER = 0, T_SGU = 1, T_RGU = 2, T_DOWN = 3 };

// The CTA's shared-memory copy of layer l's descriptor (made at kernel start).
extern __shared__ __align__(128) unsigned char g_smem[];
__device__ __forceinline__ const LayerDesc& LD(int l) {
    return reinterpret_cast<const LayerDesc*>(g_smem + OFF_DESC)[l];
}
enum { ERR_TIMEOUT = 1, ERR_BAD_ID = 2 };

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking test of a phase (try_wait may suspend the thread for a while).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Weight copies carry no L2 cache-policy operand: with it, issuing the
// copies measured about 1 % slower per decode step.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void trace_at(const Params& P, int l, int slot) {
    if (P.trace) P.trace[((size_t)l * TRACE_CTAS + blockIdx.x) * TRACE_SLOTS + slot] = gtimer();
}
// Tagged words: relaxed accesses at GPU scope; each 32- or 64-bit element is single-copy atomic.
__device__ __forceinline__ uint4 ld_relaxed_v4(const void* p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void ld_relaxed_v2u64(const void* p, unsigned long long& a, unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const void* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(void* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_v2u64(void* p, unsigned long long a, unsigned long long b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1,%2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void st_relaxed_v2u32(void* p, uint32_t a, uint32_t b) {
    asm volatile("st.relaxed.gpu.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_relaxed_add(uint32_t* p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long tag64(uint32_t tag, float v) {
    return ((unsigned long long)tag << 32) | __float_as_uint(v);
}

__device__ __forceinline__ bool err_set(const uint32_t* err) { return *(volatile const uint32_t*)err != 0; }

// Bounded wait (one lane) on an mbarrier phase that other warps complete: false
// (error recorded) after `limit` ns, or as soon as another CTA has failed. The
// waits use try_wait with the hardware's own suspend time: a suspend-time hint
// (1 us or 100 ns) measured about 1.3 % slower per decode step.
__device__ bool wait_mbar(uint32_t bar, uint32_t parity, uint32_t* err, unsigned long long limit) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 7u) == 0) {
            if (err_set(err)) return false;
            if (gtimer() - t0 > limit) {
                atomicOr(err, ERR_TIMEOUT);
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool warp_wait_mbar(uint32_t bar, uint32_t parity, const Params& P, int lane) {
    bool ok = true;
    if (lane == 0) ok = wait_mbar(bar, parity, P.err, P.dep_limit_ns);
    return __shfl_sync(FULL, (int)ok, 0) != 0;
}
// Wait (one lane) for the warp's own bulk copy to land. It ignores other CTAs'
// failures: a warp never leaves while a copy into its shared memory is in flight.
// Bounded all the same (2 s; a copy that does not land is recorded as a timeout).
__device__ bool wait_own(uint32_t bar, uint32_t parity, uint32_t* err) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 7u) == 0 && gtimer() - t0 > OWN_LIMIT_NS) {
            atomicOr(err, ERR_TIMEOUT);
            return false;
        }
    }
}
__device__ __forceinline__ bool warp_wait_own(uint32_t bar, uint32_t parity, uint32_t* err, int lane) {
    bool ok = true;
    if (lane == 0) ok = wait_own(bar, parity, err);
    return __shfl_sync(FULL, (int)ok, 0) != 0;
}


// ------------------------------------------------------------------ task lists

__device__ __forceinline__ int tasks_per_layer(int E) { return E + N_SGU + N_RGU + N_DN; }
__device__ __forceinline__ int task_kind(int t, int E) {
    if (t < E) return T_ROUTER;
    t -= E;
    if (t < N_SGU) return T_SGU;
    t -= N_SGU;
    return t < N_RGU ? T_RGU : T_DOWN;
}
__device__ __forceinline__ int task_items(int kind) { return kind == T_SGU ? 2 : (kind == T_DOWN ? 3 : 1); }
// First task of layer l owned by global worker gw: task t of layer l has the
// global index l * NTL + t and belongs to worker (l * NTL + t) mod NW.
__device__ __forceinline__ int first_task(int gw, int l, int NTL, int NW) {
    return (int)(((long long)gw - (long long)l * NTL % NW + NW) % NW);
}

// Position in a worker's item sequence (layer, task, item of the task).
struct It {
    int l, t, sub, kind;
};

struct Ctx {
    const Params* P;
    int gw, NW, lane;
    int E, NTL;
};

__device__ __forceinline__ void it_begin_layer(It& it, const Ctx& c, int l) {
    it.l = l;
    it.sub = 0;
    it.t = first_task(c.gw, l, c.NTL, c.NW);
    it.kind = task_kind(it.t, c.E);
}
__device__ __forceinline__ void it_next(It& it, const Ctx& c) {
    if (++it.sub < task_items(it.kind)) return;
    it.sub = 0;
    it.t += c.NW;
    if (it.t >= c.NTL) {
        it_begin_layer(it, c, it.l + 1);
        return;
    }
    it.kind = task_kind(it.t, c.E);
}
__device__ __forceinline__ bool it_needs_topk(const It& it) {
    return it.kind == T_RGU || (it.kind == T_DOWN && it.sub == 2);
}

// CTA routing cache, two layers deep (written by control warp 0).
struct Route {
    const char* ep[2][K];
    float w[2][K];
    int32_t id[2][K];
};
static_assert(sizeof(Route) <= RT_BYTES, "routing cache");

// The warp enqueues the copies of one item into a stage: lane 0 announces the
// bytes on the stage's mbarrier, then one lane per copy issues it (an item's
// copies leave in parallel instead of one after another).
__device__ void issue_item(const Ctx& c, const It& it, const Route* rt, uint32_t dst, uint32_t bar, int lane) {
    const LayerDesc& D = LD(it.l);
    if (it.kind == T_DOWN && it.sub == 2) {
        if (lane == 0) mbar_expect_tx(bar, DN_BYTES);
        __syncwarp();
        if (lane < 2 * K) {
            fence_proxy_async();  // the stage's previous contents were read through the generic proxy
            const int j0 = 2 * (it.t - D.E - N_SGU - N_RGU);
            const int i = lane & (K - 1);
            const char* ep = rt->ep[it.l & 1][i];
            if (lane < K)
                bulk_g2s(dst + i * 2 * D_ROW, ep + D.off_d_codes + (size_t)j0 * D_ROW, 2 * D_ROW, bar);
            else
                bulk_g2s(dst + DN_SB_OFF + i * 4 * D_SB, ep + D.off_d_sb + (size_t)(j0 & ~3) * D_SB, 4 * D_SB, bar);
        }
        return;
    }
    if (it.kind == T_RGU) {
        if (lane == 0) mbar_expect_tx(bar, RGU_BYTES);
        __syncwarp();
        if (lane < 2) {
            fence_proxy_async();
            const int u = it.t - D.E - N_SGU;
            const int i = u / RGU_PER_EXPERT, p0 = 2 * (u % RGU_PER_EXPERT);
            const char* ep = rt->ep[it.l & 1][i];
            if (lane == 0)
                bulk_g2s(dst, ep + (size_t)2 * p0 * GU_ROW, 4 * GU_ROW, bar);
            else
                bulk_g2s(dst + 4 * GU_ROW, ep + D.off_gu_sb + (size_t)2 * p0 * GU_SB, 4 * GU_SB, bar);
        }
        return;
    }
    if (lane != 0) return;
    fence_proxy_async();  // the stage's previous contents were read through the generic proxy
    if (it.kind == T_ROUTER) {
        mbar_expect_tx(bar, ROW_BF);
        bulk_g2s(dst, D.Wr + (size_t)it.t * H, ROW_BF, bar);
    } else if (it.kind == T_SGU) {
        const int j = it.t - D.E;
        mbar_expect_tx(bar, ROW_BF);
        bulk_g2s(dst, (it.sub == 0 ? D.Wsg : D.Wsu) + (size_t)j * H, ROW_BF, bar);
    } else {
        const int j0 = 2 * (it.t - D.E - N_SGU - N_RGU);
        mbar_expect_tx(bar, SROW_BF);
        bulk_g2s(dst, D.Wsd + (size_t)(j0 + it.sub) * S, SROW_BF, bar);
    }
}

// L2 prefetch of the data-independent weights of worker gw's tasks in layer l.
__device__ void prefetch_layer(const Ctx& c, int l) {
    const LayerDesc& D = LD(l);
    for (int t = first_task(c.gw, l, c.NTL, c.NW); t < c.NTL; t += c.NW) {
        const int kind = task_kind(t, c.E);
        if (kind == T_ROUTER) {
            prefetch_l2(D.Wr + (size_t)t * H, ROW_BF);
        } else if (kind == T_SGU) {
            const int j = t - c.E;
            prefetch_l2(D.Wsg + (size_t)j * H, ROW_BF);
            prefetch_l2(D.Wsu + (size_t)j * H, ROW_BF);
        } else if (kind == T_DOWN) {
            const int j0 = 2 * (t - c.E - N_SGU - N_RGU);
            prefetch_l2(D.Wsd + (size_t)j0 * S, 2 * SROW_BF);
        }
    }
}

// ------------------------------------------------------------------ compute

// Packed fp32 pairs for the two-wide FMA of sm_100+ (fma.rn.f32x2).
__device__ __forceinline__ unsigned long long pk2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float sum2(unsigned long long v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}
__device__ __forceinline__ void fma2(unsigned long long& acc, unsigned long long a, unsigned long long b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
// acc + sum over 8 bf16 weights (one 16-byte chunk) times n, packed FMA.
__device__ __forceinline__ unsigned long long dot8_bf16_2(uint4 w, float4 a, float4 b, unsigned long long acc) {
    fma2(acc, pk2(bf_lo(w.x), bf_hi(w.x)), pk2(a.x, a.y));
    fma2(acc, pk2(bf_lo(w.y), bf_hi(w.y)), pk2(a.z, a.w));
    fma2(acc, pk2(bf_lo(w.z), bf_hi(w.z)), pk2(b.x, b.y));
    fma2(acc, pk2(bf_lo(w.w), bf_hi(w.w)), pk2(b.z, b.w));
    return acc;
}
// sum_k W[k] n[k] over a bf16 row of K = H (16-byte chunk w covers n[8w..8w+7],
// held in shared memory as the float4s w and HW + w).
__device__ __forceinline__ float row_bf16(const unsigned char* row, const float* n, int lane) {
    const float4* n4 = reinterpret_cast<const float4*>(n);
    unsigned long long acc = 0ull;
#pragma unroll 1
    for (int m = 0; m < WPL; ++m) {
        const int w = lane + 32 * m;
        const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * w);
        acc = dot8_bf16_2(v, n4[w], n4[HW + w], acc);
    }
    return warp_sum(sum2(acc));
}

// Byte dot products: acc + sum_i a.byte_i * b.byte_i, bytes unsigned (uu) or a signed (su).
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// One word of 8 codes against the digits of its 8 values of n: exact integer sums per digit.
__device__ __forceinline__ void word_digits(uint32_t q, uint32_t lo0, uint32_t hi0, uint32_t lo1, uint32_t hi1,
                                            uint32_t lo2, uint32_t hi2, int& s0, int& s1, int& s2) {
    const uint32_t lo = q & 0x0f0f0f0fu, hi = (q >> 4) & 0x0f0f0f0fu;  // codes of columns 0,2,4,6 / 1,3,5,7
    s0 = dp4a_uu(hi0, hi, dp4a_uu(lo0, lo, s0));
    s1 = dp4a_uu(hi1, hi, dp4a_uu(lo1, lo, s1));
    s2 = dp4a_su(hi2, hi, dp4a_su(lo2, lo, s2));
}

// Four int4 rows of K = H at once (the stage holds 4 rows of codes, then 4 rows
// of {s,b}): lane = (row lane & 3, block lane >> 2, + 8 per step). Per 32-value
// block the codes meet the digits of n in integer arithmetic (exact), then
// s * (scale * sum q n_int) + b * sum n in fp32; the four lanes of a block read
// the same digits.
__device__ __forceinline__ float4 rows4_int4(const unsigned char* st, const uint32_t* dig, int lane) {
    const int r = lane & 3, hb = lane >> 2;
    const unsigned char* crow = st + r * GU_ROW;
    const uint32_t* sbrow = reinterpret_cast<const uint32_t*>(st + 4 * GU_ROW) + r * (GU_SB / 4);
    float acc = 0.0f;
#pragma unroll 2
    for (int m = 0; m < HG / 8; ++m) {
        const int hg = hb + 8 * m;
        const uint4 q = *reinterpret_cast<const uint4*>(crow + 16 * hg);
        const uint4* dp = reinterpret_cast<const uint4*>(dig + hg * DIG_WORDS);
        const uint4 d0 = dp[0], d1 = dp[1], d2 = dp[2], d3 = dp[3], d4 = dp[4], d5 = dp[5];
        const float2 meta = *reinterpret_cast<const float2*>(dig + hg * DIG_WORDS + 24);
        int s0 = 0, s1 = 0, s2 = 0;
        word_digits(q.x, d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, s0, s1, s2);
        word_digits(q.y, d1.z, d1.w, d2.x, d2.y, d2.z, d2.w, s0, s1, s2);
        word_digits(q.z, d3.x, d3.y, d3.z, d3.w, d4.x, d4.y, s0, s1, s2);
        word_digits(q.w, d4.z, d4.w, d5.x, d5.y, d5.z, d5.w, s0, s1, s2);
        const float pq = fmaf((float)s2, 65536.0f, fmaf((float)s1, 256.0f, (float)s0)) * meta.x;
        const uint32_t sbw = sbrow[hg >> 1];
        acc = fmaf(h2f(sbw & 0xffffu), pq, fmaf(h2f(sbw >> 16), meta.y, acc));
    }
    acc += __shfl_xor_sync(FULL, acc, 4);
    acc += __shfl_xor_sync(FULL, acc, 8);
    acc += __shfl_xor_sync(FULL, acc, 16);
    return make_float4(__shfl_sync(FULL, acc, 0), __shfl_sync(FULL, acc, 1), __shfl_sync(FULL, acc, 2),
                       __shfl_sync(FULL, acc, 3));
}

// Wait (one warp) until the hint counter reaches target (modular u32 compare).
// The counter only paces the reading of tagged data; it orders nothing.
__device__ bool wait_hint(const uint32_t* cnt, uint32_t target, const Params& P, int lane) {
    uint32_t* err = P.err;
    int st = 0;  // 1 reached, 2 give up
    if (lane == 0) {
        const uint64_t t0 = gtimer();
        for (uint32_t n = 0;; ++n) {
            if ((int32_t)(ld_relaxed_u32(cnt) - target) >= 0) {
                st = 1;
                break;
            }
            __nanosleep(HINT_SLEEP_NS);
            if ((n & 63u) == 63u) {
                if (err_set(err)) {
                    st = 2;
                    break;
                }
                if (gtimer() - t0 > P.dep_limit_ns) {
                    atomicOr(err, ERR_TIMEOUT);
                    st = 2;
                    break;
                }
            }
        }
    }
    return __shfl_sync(FULL, st, 0) == 1;
}

// A worker finished a phase of a layer: count it in the CTA; the CTA's last
// worker bumps the grid-wide hint counter (relaxed, no fence).
__device__ __forceinline__ void signal_phase(const Params& P, int l, int slot, uint32_t* cta_cnt, uint32_t* gcnt,
                                             int lane) {
    __syncwarp();
    if (lane == 0 && (atomicAdd(cta_cnt, 1u) + 1u) % NWORK == 0) {
        red_relaxed_add(gcnt, 1u);
        if (slot >= 0) trace_at(P, l, slot);
    }
    __syncwarp();
}

__device__ __forceinline__ uint32_t tag4_of(uint32_t epoch, int l) { return 1u + (epoch + (uint32_t)l) % 15u; }
__device__ __forceinline__ uint32_t tagged_f(float v, uint32_t tag4) { return (__float_as_uint(v) & ~15u) | tag4; }
__device__ __forceinline__ void ctrl_sync() { asm volatile("bar.sync %0, %1;" ::"n"(CTRL_BAR), "n"(NCTRL * 32) : "memory"); }

// ---- control warps: read a tagged block into shared memory and check it.
// 16-byte chunks c = cw * 32 + lane + 128 i (c < n16) of the block, read with
// relaxed loads issued back to back (at most NMAX per thread), then handed to f(c, v).
template <int NMAX, typename F>
__device__ __forceinline__ void ctrl_read(const uint32_t* src, int n16, int cw, int lane, F f) {
    uint4 v[NMAX];
#pragma unroll
    for (int i = 0; i < NMAX; ++i) {
        const int c = cw * 32 + lane + i * NCTRL * 32;
        if (c < n16) v[i] = ld_relaxed_v4(src + 4 * c);
    }
#pragma unroll
    for (int i = 0; i < NMAX; ++i) {
        const int c = cw * 32 + lane + i * NCTRL * 32;
        if (c < n16) f(c, v[i]);
    }
}
// All four control warps call this with the same arguments: each reads its
// share of the block in `check` (which writes the values to shared memory and
// returns the number of stale words it saw), and the block is read again while
// any word is stale.
template <typename Check>
__device__ bool ctrl_poll(const Params& P, uint32_t* stale, int cw, int lane, Check check) {
    const uint64_t t0 = gtimer();
    for (int round = 0;; ++round) {
        if (cw == 0 && lane == 0) stale[0] = 0u;
        ctrl_sync();  // the count is reset before any warp adds to it
        {
            const uint32_t bad = check();
            const uint32_t wbad = __reduce_add_sync(FULL, bad);
            if (wbad && lane == 0) atomicAdd(&stale[0], wbad);
        }
        // only warp 0 decides a timeout, so that every control warp takes the same path
        if (cw == 0 && lane == 0 && round > 16 && (err_set(P.err) || gtimer() - t0 > P.dep_limit_ns)) {
            atomicOr(&stale[1], 1u);
            atomicOr(P.err, ERR_TIMEOUT);
        }
        ctrl_sync();
        const uint32_t total = stale[0], abort_now = stale[1];
        ctrl_sync();
        if (abort_now) return false;
        if (total == 0) return true;
        if (round > 16) __nanosleep(256);
    }
}

// The layer input: the tagged output of the previous layer (or the call's x)
// -> x (bf16; released to the router rows), then r, n = r x and the word sums
// of n; all four control warps.
__device__ bool stage_x(const Params& P, int l, uint32_t epoch, uint32_t hint_target, unsigned char* smem,
                        uint32_t bar_xs, uint32_t* stale, int cw, int lane) {
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + OFF_XS);
    if (l == 0) {
        const uint4* s4 = reinterpret_cast<const uint4*>(P.x);
        for (int c = cw * 32 + lane; c < H / 8; c += NCTRL * 32) reinterpret_cast<uint4*>(xs)[c] = __ldcg(s4 + c);
    } else {
        if (cw == 0 && !wait_hint(LD(l - 1).cnt_out, hint_target, P, lane) && lane == 0)
            atomicOr(&stale[1], 1u);  // tells the other control warps to stop
        ctrl_sync();
        if (stale[1]) return false;
        const uint32_t tag16 = (epoch * 64u + (uint32_t)(l - 1)) & 0xffffu;
        auto check = [&]() -> uint32_t {
            uint32_t bad = 0;
            ctrl_read<(H / 4 + NCTRL * 32 - 1) / (NCTRL * 32)>(LD(l - 1).xt, H / 4, cw, lane, [&](int c, uint4 v) {
                bad += ((v.x >> 16) != tag16) + ((v.y >> 16) != tag16) + ((v.z >> 16) != tag16) +
                       ((v.w >> 16) != tag16);  // 4 tagged words per chunk
                reinterpret_cast<uint2*>(xs)[c] = make_uint2((v.x & 0xffffu) | (v.y << 16), (v.z & 0xffffu) | (v.w << 16));
            });
            return bad;
        };
        if (!ctrl_poll(P, stale, cw, lane, check)) return false;
        if (cw == 0 && lane == 0) trace_at(P, l, TR_X_READY);
    }
    ctrl_sync();
    if (cw == 0 && lane == 0) mbar_arrive(bar_xs);  // the router rows need only x (r is applied after the dot)
    float* rs = reinterpret_cast<float*>(smem + OFF_MISC);
    if (cw == 0) {
        float p = 0.0f;
#pragma unroll 8
        for (int k = lane; k < H; k += 32) {
            const float v = bf2f(xs[k]);
            p = fmaf(v, v, p);  // exact square: one rounding per term, as in the canonical sum
        }
        p = warp_sum_canonical(p);
        if (lane == 0) rs[0] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(p, (float)H), LD(l).eps)));
    }
    ctrl_sync();
    const float r = rs[0];
    float* n = reinterpret_cast<float*>(smem + OFF_N);
    float* sn = reinterpret_cast<float*>(smem + OFF_SN);
    for (int w = cw * 32 + lane; w < HW; w += NCTRL * 32) {
        const uint4 v = reinterpret_cast<const uint4*>(xs)[w];
        const float4 a = make_float4(__fmul_rn(r, bf_lo(v.x)), __fmul_rn(r, bf_hi(v.x)), __fmul_rn(r, bf_lo(v.y)),
                                     __fmul_rn(r, bf_hi(v.y)));
        const float4 b = make_float4(__fmul_rn(r, bf_lo(v.z)), __fmul_rn(r, bf_hi(v.z)), __fmul_rn(r, bf_lo(v.w)),
                                     __fmul_rn(r, bf_hi(v.w)));
        reinterpret_cast<float4*>(n)[w] = a;
        reinterpret_cast<float4*>(n)[HW + w] = b;
        sn[w] = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
    }
    ctrl_sync();
    return true;
}

// Bytes 0, 1 and 2 of four integers a, b, c, d gathered as (a_k, b_k, c_k, d_k), k = 0, 1, 2.
__device__ __forceinline__ void digit_words(int a, int b, int c, int d, uint32_t& w0, uint32_t& w1, uint32_t& w2) {
    const uint32_t t0 = __byte_perm((uint32_t)a, (uint32_t)b, 0x5140u);  // a0 b0 a1 b1
    const uint32_t t1 = __byte_perm((uint32_t)c, (uint32_t)d, 0x5140u);  // c0 d0 c1 d1
    const uint32_t t2 = __byte_perm((uint32_t)a, (uint32_t)b, 0x7362u);  // a2 b2 a3 b3
    const uint32_t t3 = __byte_perm((uint32_t)c, (uint32_t)d, 0x7362u);  // c2 d2 c3 d3
    w0 = __byte_perm(t0, t1, 0x5410u);
    w1 = __byte_perm(t0, t1, 0x7632u);
    w2 = __byte_perm(t2, t3, 0x5410u);
}

// A block of 32 values (v[8 j + c] = column 8 j + c) for the integer dot
// products: a shared power-of-two scale puts the largest |v| in [2^22, 2^23);
// each value becomes a 24-bit integer, split into three byte digits (two
// unsigned, the top one signed), packed four to a word in the order of the code
// bytes of a word of codes (columns 0,2,4,6 and 1,3,5,7). Written: per word j
// {lo0, hi0, lo1, hi1, lo2, hi2} at d[6 j], then the inverse scale and the sum
// of the block.
__device__ __forceinline__ void block_digits(const float (&v)[32], uint32_t* d) {
    float m = 0.0f, sum = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float ws = 0.0f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            m = fmaxf(m, fabsf(v[8 * j + c]));
            ws += v[8 * j + c];
        }
        sum += ws;
    }
    float up = 0.0f, down = 0.0f;  // a block below 2^-100 counts as zero
    if (m >= 7.8886e-31f) {
        const int e = (int)((__float_as_uint(m) >> 23) & 0xffu) - 127;  // m in [2^e, 2^(e+1))
        up = __uint_as_float((uint32_t)(127 + 22 - e) << 23);
        down = __uint_as_float((uint32_t)(127 + e - 22) << 23);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        int q[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) q[c] = __float2int_rn(v[8 * j + c] * up);  // |q| < 2^23; v * up is exact
        // byte k of the four integers of columns 0,2,4,6 (then 1,3,5,7) gathered into one word: a 4x4
        // byte transpose (digit 2 = byte 2 is the signed top digit in two's complement)
        uint32_t lo0, lo1, lo2, hi0, hi1, hi2;
        digit_words(q[0], q[2], q[4], q[6], lo0, lo1, lo2);
        digit_words(q[1], q[3], q[5], q[7], hi0, hi1, hi2);
        reinterpret_cast<uint2*>(d + 6 * j)[0] = make_uint2(lo0, hi0);
        reinterpret_cast<uint2*>(d + 6 * j)[1] = make_uint2(lo1, hi1);
        reinterpret_cast<uint2*>(d + 6 * j)[2] = make_uint2(lo2, hi2);
    }
    d[24] = __float_as_uint(down);
    d[25] = __float_as_uint(sum);
}

// n as digit blocks for the routed gate/up rows (control warps 1..3 while warp 0 routes).
__device__ void stage_digits(unsigned char* smem, int t, int nt) {
    const float4* n4 = reinterpret_cast<const float4*>(smem + OFF_N);
    uint32_t* dig = reinterpret_cast<uint32_t*>(smem + OFF_DIG);
    for (int hg = t; hg < HG; hg += nt) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 a = n4[4 * hg + j], b = n4[HW + 4 * hg + j];
            v[8 * j + 0] = a.x;
            v[8 * j + 1] = a.y;
            v[8 * j + 2] = a.z;
            v[8 * j + 3] = a.w;
            v[8 * j + 4] = b.x;
            v[8 * j + 5] = b.y;
            v[8 * j + 6] = b.z;
            v[8 * j + 7] = b.w;
        }
        block_digits(v, dig + hg * DIG_WORDS);
    }
}

// h_routed (fp32, in the h area) -> digit blocks in place, all four control
// warps. The digits are those of block_digits; only the work is spread
// differently: eight consecutive lanes hold one block (a float4 each, read
// contiguously, so without bank conflicts), find its largest |v| and its sum
// with three butterfly steps, convert their four values, and swap two with the
// neighbouring lane, so that the even lane holds columns 0,2,4,6 and the odd
// lane columns 1,3,5,7 of their 8-value word. Every thread holds all its values
// in registers before any digit is written (the digits overwrite the fp32 area).
__device__ void digits_in_place(unsigned char* smem, int cw, int lane) {
    const float4* h4 = reinterpret_cast<const float4*>(smem + OFF_H);
    uint32_t* dig = reinterpret_cast<uint32_t*>(smem + OFF_H);
    constexpr int NQ = HB * 8, PER = NQ / (NCTRL * 32);  // float4s of h_routed, per thread
    static_assert(NQ % (NCTRL * 32) == 0, "whole rounds of the control threads");
    const int t = cw * 32 + lane;
    float4 v[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) v[k] = h4[t + NCTRL * 32 * k];
    ctrl_sync();
    const int c = lane & 7;  // float4 of the block: word c >> 1, columns 0-3 (even c) or 4-7 (odd c)
    const bool odd = c & 1;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int b = (t + NCTRL * 32 * k) >> 3;
        const float4 a = v[k];
        float m = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w)));
        float sum = (a.x + a.y) + (a.z + a.w);
        m = fmaxf(m, __shfl_xor_sync(FULL, m, 1));
        m = fmaxf(m, __shfl_xor_sync(FULL, m, 2));
        m = fmaxf(m, __shfl_xor_sync(FULL, m, 4));
        sum += __shfl_xor_sync(FULL, sum, 1);
        sum += __shfl_xor_sync(FULL, sum, 2);
        sum += __shfl_xor_sync(FULL, sum, 4);
        float up = 0.0f, down = 0.0f;  // a block below 2^-100 counts as zero
        if (m >= 7.8886e-31f) {
            const int e = (int)((__float_as_uint(m) >> 23) & 0xffu) - 127;
            up = __uint_as_float((uint32_t)(127 + 22 - e) << 23);
            down = __uint_as_float((uint32_t)(127 + e - 22) << 23);
        }
        const int q0 = __float2int_rn(a.x * up), q1 = __float2int_rn(a.y * up), q2 = __float2int_rn(a.z * up),
                  q3 = __float2int_rn(a.w * up);
        // even lane: columns 0, 2 (own), 4, 6 (neighbour's q0, q2); odd: 1, 3 (neighbour's q1, q3), 5, 7 (own)
        const int ra = __shfl_xor_sync(FULL, odd ? q0 : q1, 1), rb = __shfl_xor_sync(FULL, odd ? q2 : q3, 1);
        uint32_t w0, w1, w2;
        digit_words(odd ? ra : q0, odd ? rb : q2, odd ? q1 : ra, odd ? q3 : rb, w0, w1, w2);
        uint32_t* d = dig + b * DIG_WORDS + 6 * (c >> 1) + (odd ? 1 : 0);
        d[0] = w0;
        d[2] = w1;
        d[4] = w2;
        if (c == 0) *reinterpret_cast<float2*>(dig + b * DIG_WORDS + 24) = make_float2(down, sum);
    }
}

// Control warp 0: the CTA's copy of the layer's top-k from the tagged logits.
__device__ bool route_layer(const Params& P, int l, uint32_t tag, uint32_t epoch_x_e, unsigned char* smem, Route* rt,
                            int lane, int& sel, float& selz) {
    const LayerDesc& D = LD(l);
    if (!wait_hint(D.cnt_z, epoch_x_e, P, lane)) return false;
    unsigned long long* zt = reinterpret_cast<unsigned long long*>(smem + OFF_Z);
    const uint64_t t0 = gtimer();
    for (;;) {
        // the tagged logits, two per lane and load (relaxed, issued back to back)
        constexpr int NZ = MAX_E / 64;
        unsigned long long za[NZ], zb[NZ];
#pragma unroll
        for (int i = 0; i < NZ; ++i) {
            const int j = 2 * (lane + 32 * i);
            if (j + 1 < D.E) ld_relaxed_v2u64(D.zt + j, za[i], zb[i]);
            else if (j < D.E) za[i] = ld_relaxed_u64(D.zt + j);
        }
        int bad = 0;
#pragma unroll
        for (int i = 0; i < NZ; ++i) {
            const int j = 2 * (lane + 32 * i);
            if (j < D.E) {
                zt[j] = za[i];
                bad |= (uint32_t)(za[i] >> 32) != tag;
            }
            if (j + 1 < D.E) {
                zt[j + 1] = zb[i];
                bad |= (uint32_t)(zb[i] >> 32) != tag;
            }
        }
        __syncwarp();
        if (!__any_sync(FULL, bad)) break;
        __nanosleep(128);
        if (err_set(P.err)) return false;
        if (gtimer() - t0 > P.dep_limit_ns) {
            if (lane == 0) atomicOr(P.err, ERR_TIMEOUT);
            return false;
        }
    }
    if (lane == 0) trace_at(P, l, TR_Z_READY);
    // order-preserving keys (larger logit first, -0 == +0, NaN lowest but above
    // "taken" = 0), held in registers (key m of a lane is expert lane + 32 m);
    // every round takes the best remaining key and the lowest index holding it
    // with two warp reductions
    constexpr int KPL = MAX_E / 32;
    uint32_t key[KPL];
#pragma unroll
    for (int m = 0; m < KPL; ++m) {
        const int j = lane + 32 * m;
        key[m] = 0u;
        if (j < D.E) {
            const float v = __uint_as_float((uint32_t)zt[j]) + 0.0f;
            const uint32_t u = __float_as_uint(v);
            key[m] = isnan(v) ? 1u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
        }
    }
    selz = 0.0f;
    sel = -1;
    if (D.E <= 128) {
        // Four keys per lane, sorted (larger key first, then the lower expert);
        // every round the best head over the warp is taken and its lane pops it.
        uint32_t k0 = key[0], k1 = key[1], k2 = key[2], k3 = key[3];
        uint32_t i0 = lane, i1 = lane + 32, i2 = lane + 64, i3 = lane + 96;
        auto order = [](uint32_t& ka, uint32_t& ia, uint32_t& kb, uint32_t& ib) {
            const bool sw = kb > ka || (kb == ka && ib < ia);
            const uint32_t tk = sw ? kb : ka, ti = sw ? ib : ia;
            kb = sw ? ka : kb;
            ib = sw ? ia : ib;
            ka = tk;
            ia = ti;
        };
        order(k0, i0, k1, i1);
        order(k2, i2, k3, i3);
        order(k0, i0, k2, i2);
        order(k1, i1, k3, i3);
        order(k1, i1, k2, i2);
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const uint32_t kmax = __reduce_max_sync(FULL, k0);
            const uint32_t imin = __reduce_min_sync(FULL, k0 == kmax ? i0 : 0x7fffffffu);
            if (lane == (int)(imin & 31u)) {
                k0 = k1;
                i0 = i1;
                k1 = k2;
                i1 = i2;
                k2 = k3;
                i2 = i3;
                k3 = 0u;
                i3 = 0x7fffffffu;
            }
            if (lane == i) {
                sel = (int)imin;
                selz = __uint_as_float((uint32_t)zt[imin]);
            }
        }
    } else
#pragma unroll 1
    for (int i = 0; i < K; ++i) {
        uint32_t bk = key[0];
        int bm = 0;
#pragma unroll
        for (int m = 1; m < KPL; ++m)
            if (key[m] > bk) {  // m increases: equal keys keep the lower index
                bk = key[m];
                bm = m;
            }
        const uint32_t kmax = __reduce_max_sync(FULL, bk);
        const int imin = (int)__reduce_min_sync(FULL, bk == kmax ? (uint32_t)(lane + 32 * bm) : 0x7fffffffu);
#pragma unroll
        for (int m = 0; m < KPL; ++m)  // a select per register (a value test keeps the array out of local memory)
            key[m] = (key[m] == kmax && lane + 32 * m == imin) ? 0u : key[m];
        if (lane == i) {
            sel = imin;
            selz = __uint_as_float((uint32_t)zt[imin]);
        }
    }
    // the selected experts' addresses: all the routed copies need (the weights come later)
    const int s = l & 1;
    int bad = 0;
    if (lane < K) {
        rt->id[s][lane] = sel;
        int e = sel;
        bad = (unsigned)e >= (unsigned)D.E;
        if (bad) e = 0;  // never form an address from an out-of-range id
        if (D.slot_map) {
            e = __ldcg(D.slot_map + e);
            if ((unsigned)e >= (unsigned)D.n_slots) {
                bad = 1;
                e = 0;
            }
        }
        rt->ep[s][lane] = D.ebase + (size_t)e * D.estride;
    }
    if (__any_sync(FULL, bad)) {
        if (lane == 0) atomicOr(P.err, ERR_BAD_ID);
        return false;
    }
    __syncwarp();
    return true;
}

// Control warp 0, after the top-k is released: the routing weights (softmax
// over the selected logits, summed in top-k order), read by the routed-down
// items only after the later h_routed phase; CTA 0 also publishes the routing.
__device__ void route_weights(const Params& P, int l, unsigned char* smem, Route* rt, bool publish, int lane, int sel,
                              float selz) {
    const LayerDesc& D = LD(l);
    const unsigned long long* zt = reinterpret_cast<const unsigned long long*>(smem + OFF_Z);
    float zmax = __shfl_sync(FULL, selz, 0);
    for (int i = 1; i < K; ++i) {
        const float zi = __shfl_sync(FULL, selz, i);
        if (zi > zmax) zmax = zi;
    }
    const float ev = lane < K ? expf(__fsub_rn(selz, zmax)) : 0.0f;
    float esum = 0.0f;
    for (int i = 0; i < K; ++i) esum = __fadd_rn(esum, __shfl_sync(FULL, ev, i));
    if (lane < K) {
        const float wv = __fdiv_rn(ev, esum);
        rt->w[l & 1][lane] = wv;
        if (publish) {
            D.idx[lane] = sel;
            D.w[lane] = wv;
        }
    }
    if (publish)
        for (int j = lane; j < D.E; j += 32) D.logits[j] = __uint_as_float((uint32_t)zt[j]);
    __syncwarp();
}

// h_shared or h_routed (tagged fp32 words) -> shared memory, in place, checked by
// the four control warps; h_routed is then turned into digit blocks in place.
__device__ bool stage_h(const Params& P, int l, uint32_t tag4, const uint32_t* hint, uint32_t hint_target,
                        bool routed, unsigned char* smem, uint32_t* stale, int cw, int lane) {
    const LayerDesc& D = LD(l);
    if (cw == 0 && !wait_hint(hint, hint_target, P, lane) && lane == 0) atomicOr(&stale[1], 1u);
    ctrl_sync();
    if (stale[1]) return false;
    const int w0 = routed ? 0 : K * I, nw = routed ? K * I : S;  // in floats
    uint32_t* h = reinterpret_cast<uint32_t*>(smem + OFF_H) + w0;
    auto check = [&]() -> uint32_t {
        uint32_t bad = 0;
        ctrl_read<(K * I / 4 + NCTRL * 32 - 1) / (NCTRL * 32)>(D.ht + w0, nw / 4, cw, lane, [&](int c, uint4 v) {
            reinterpret_cast<uint4*>(h)[c] = v;
            bad += ((v.x & 15u) != tag4) + ((v.y & 15u) != tag4) + ((v.z & 15u) != tag4) + ((v.w & 15u) != tag4);
        });
        return bad;
    };
    if (!ctrl_poll(P, stale, cw, lane, check)) return false;
    if (routed) digits_in_place(smem, cw, lane);
    ctrl_sync();
    return true;
}

// ------------------------------------------------------------------ the kernel

__global__ void __launch_bounds__(NT, 1) k_fused_stack(Params P) {
    unsigned char* smem = g_smem;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = gridDim.x;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    const uint32_t bar_x = smem_u32(&bars[B_X]);
    const uint32_t bar_xs = smem_u32(&bars[B_XS]);
    const uint32_t bar_k = smem_u32(&bars[B_K]);
    const uint32_t bar_hs = smem_u32(&bars[B_HS]);
    const uint32_t bar_hr = smem_u32(&bars[B_HR]);
    Route* rt = reinterpret_cast<Route*>(smem + OFF_RT);
    uint32_t* s_epoch = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 4);
    uint32_t* cta_cnt = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 8);  // [0] hs, [1] hr, [2] out
    uint32_t* stale = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 20);   // [0] stale words, [1] abort

    if (threadIdx.x == 0) {
        for (int s = 0; s < NWORK * NS; ++s) mbar_init(smem_u32(&bars[s]), 1);
        mbar_init(bar_x, 1);
        mbar_init(bar_xs, 1);
        mbar_init(bar_k, 1);
        mbar_init(bar_hs, 1);
        mbar_init(bar_hr, 1);
        *s_epoch = ld_relaxed_u32(P.epoch);
        cta_cnt[0] = cta_cnt[1] = cta_cnt[2] = 0;
        stale[0] = stale[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    {  // the layer descriptors, copied once
        const unsigned long long* src = reinterpret_cast<const unsigned long long*>(P.layers);
        unsigned long long* dst = reinterpret_cast<unsigned long long*>(smem + OFF_DESC);
        for (int i = threadIdx.x; i < P.L * (int)(sizeof(LayerDesc) / 8); i += blockDim.x) dst[i] = __ldg(src + i);
    }
    __syncthreads();
    const uint32_t epoch = *s_epoch;
    const uint32_t hint_target = epoch * (uint32_t)G;   // every launch adds G to each per-CTA hint counter
    const int E = LD(0).E;

    if (warp < NCTRL) {
        // ================================================= control warps
        const int cw = warp;
        bool ok = true;
        for (int l = 0; l < P.L && ok; ++l) {
            const LayerDesc& D = LD(l);
            const uint32_t tag = epoch * 64u + (uint32_t)l;
            const uint32_t tag4 = tag4_of(epoch, l);
            if (!(ok = stage_x(P, l, epoch, hint_target, smem, bar_xs, stale, cw, lane))) break;
            if (cw == 0 && lane == 0) {
                mbar_arrive(bar_x);
                trace_at(P, l, TR_X_STAGED);
            }
            int rok = 1, sel = -1;
            float selz = 0.0f;
            if (cw == 0) rok = route_layer(P, l, tag, epoch * (uint32_t)E, smem, rt, lane, sel, selz);
            else
                stage_digits(smem, (cw - 1) * 32 + lane, (NCTRL - 1) * 32);
            ctrl_sync();  // the digits are complete before the top-k (which the routed gate/up items wait for)
            if (cw == 0) {
                if (rok && lane == 0) {
                    mbar_arrive(bar_k);
                    trace_at(P, l, TR_TOPK);
                }
                if (!rok && lane == 0) atomicOr(&stale[1], 1u);
                if (rok) route_weights(P, l, smem, rt, blockIdx.x == 0, lane, sel, selz);
            }
            ctrl_sync();
            if (stale[1]) {
                ok = false;
                break;
            }
            if (!(ok = stage_h(P, l, tag4, D.cnt_hs, hint_target, false, smem, stale, cw, lane))) break;
            if (cw == 0 && lane == 0) {
                mbar_arrive(bar_hs);
                trace_at(P, l, TR_HS_STAGED);
            }
            if (!(ok = stage_h(P, l, tag4, D.cnt_hr, hint_target, true, smem, stale, cw, lane))) break;
            if (cw == 0 && lane == 0) {
                mbar_arrive(bar_hr);
                trace_at(P, l, TR_HR_STAGED);
            }
        }
        // CTA 0 advances the epoch once the last layer's output is complete
        if (ok && blockIdx.x == 0 && warp == 0 && wait_hint(LD(P.L - 1).cnt_out, hint_target, P, lane)) {
            const uint32_t* src = LD(P.L - 1).xt;
            const uint32_t tag16 = (epoch * 64u + (uint32_t)(P.L - 1)) & 0xffffu;
            const uint64_t t0 = gtimer();
            for (;;) {
                int bad = 0;
                for (int c = lane; c < H / 4; c += 32) {
                    const uint4 v = ld_relaxed_v4(src + 4 * c);
                    bad |= ((v.x >> 16) != tag16) | ((v.y >> 16) != tag16) | ((v.z >> 16) != tag16) |
                           ((v.w >> 16) != tag16);
                }
                if (!__any_sync(FULL, bad)) {
                    // the epoch counts launches (mod 2^32): hint targets epoch * G stay consistent with the
                    // counters, and a tag epoch * 64 + layer only repeats 2^26 launches later
                    if (lane == 0) st_relaxed_u32(P.epoch, epoch + 1u);
                    break;
                }
                __nanosleep(256);
                if (err_set(P.err)) break;
                if (gtimer() - t0 > P.dep_limit_ns) {
                    if (lane == 0) atomicOr(P.err, ERR_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ===================================================== worker warps
    const int wk = warp - NCTRL;
    Ctx c;
    c.P = &P;
    c.gw = blockIdx.x + G * wk;
    c.NW = G * NWORK;
    c.lane = lane;
    c.E = E;
    c.NTL = tasks_per_layer(E);
    unsigned char* ring = smem + OFF_RING + (size_t)wk * NS * STAGE;
    const uint32_t ring_u32 = smem_u32(ring);
    const uint32_t bar0 = smem_u32(&bars[wk * NS]);
    const bool w0t = P.trace && wk == 0 && lane == 0;

    It iss, con;
    it_begin_layer(iss, c, 0);
    it_begin_layer(con, c, 0);
    int n_iss = 0, n_con = 0;  // items issued / consumed by this warp
    bool ok = true;
    float carry0 = 0.0f, carry1 = 0.0f;  // partial results carried between the items of a task
    const float* n_s = reinterpret_cast<const float*>(smem + OFF_N);
    const uint32_t* dig_s = reinterpret_cast<const uint32_t*>(smem + OFF_DIG);
    float r = 0.0f;

    // Layers whose top-k this warp has seen published. The routing mbarrier is
    // tested one phase at a time, in order: a parity test of a later phase
    // would succeed before the earlier one completed.
    int k_seen = 0;
    auto topk_known = [&](int lt) -> bool {
        while (k_seen <= lt) {
            int rdy = 0;
            if (lane == 0) rdy = mbar_test_wait(bar_k, k_seen & 1);
            if (!__shfl_sync(FULL, rdy, 0)) return false;
            ++k_seen;
        }
        return true;
    };
    // Fill the ring without blocking: stop at an item whose layer's top-k is not published yet.
    auto try_issue = [&]() {
        while (n_iss < n_con + NS && iss.l < P.L) {
            if (it_needs_topk(iss) && !topk_known(iss.l)) break;
            const int slot = n_iss % NS;
            issue_item(c, iss, rt, ring_u32 + slot * STAGE, bar0 + 8 * slot, lane);
            ++n_iss;
            it_next(iss, c);
        }
        __syncwarp();
    };

    if (P.prefetch && lane == 0) prefetch_layer(c, 0);
    for (int l = 0; l < P.L && ok; ++l) {
        const LayerDesc& D = LD(l);
        const uint32_t tag = epoch * 64u + (uint32_t)l;
        const uint32_t tag4 = tag4_of(epoch, l);
        const uint32_t tag16 = tag & 0xffffu;
        if (P.prefetch && lane == 0) prefetch_layer(c, l + 1 < P.L ? l + 1 : 0);
        try_issue();
        if (!(ok = warp_wait_mbar(bar_xs, l & 1, P, lane))) break;
        bool n_ready = false;  // r and n of this layer (the second x phase) observed
        const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem + OFF_XS);
        uint16_t* pout = l == P.L - 1 ? P.out : nullptr;
        bool hs_sig = false, hr_sig = false, hs_ready = false, hr_ready = false;
        bool t_rgu = false, t_sgu = false, t_rg2 = false, t_ds = false, t_rg1 = false;
        while (con.l == l) {
            // phase signals when the consume pointer leaves a kind of task
            if (!hs_sig && con.kind > T_SGU) {
                signal_phase(P, l, -1, &cta_cnt[0], D.cnt_hs, lane);
                hs_sig = true;
            }
            if (!hr_sig && con.kind > T_RGU) {
                signal_phase(P, l, TR_CTA_HR_DONE, &cta_cnt[1], D.cnt_hr, lane);
                hr_sig = true;
            }
            if (con.kind == T_DOWN) {
                if (con.sub < 2 && !hs_ready) {
                    try_issue();
                    if (!(ok = warp_wait_mbar(bar_hs, l & 1, P, lane))) break;
                    hs_ready = true;
                }
                if (con.sub == 2 && !hr_ready) {
                    try_issue();
                    if (!(ok = warp_wait_mbar(bar_hr, l & 1, P, lane))) break;
                    hr_ready = true;
                }
            }
            // make sure the item is in flight, then wait for it
            try_issue();
            if (n_iss == n_con) {  // blocked on this layer's top-k
                if (k_seen < con.l) {  // never the case: earlier layers' phases were observed at their end
                    if (lane == 0) atomicOr(P.err, ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                if (!(ok = warp_wait_mbar(bar_k, con.l & 1, P, lane))) break;
                k_seen = con.l + 1;
                try_issue();
                if (n_iss == n_con) {
                    if (lane == 0) atomicOr(P.err, ERR_TIMEOUT);
                    ok = false;
                    break;
                }
            }
            const int slot = n_con % NS;
            if (!(ok = warp_wait_own(bar0 + 8 * slot, (n_con / NS) & 1, P.err, lane))) break;
            const unsigned char* st = ring + slot * STAGE;
            if (w0t) {
                if (con.kind == T_RGU && !t_rgu) trace_at(P, l, TR_W_RGU_READY);
                if (con.kind == T_DOWN && con.sub == 2) trace_at(P, l, TR_W_RD_READY);
                if (con.kind > T_SGU && !t_sgu) trace_at(P, l, TR_W_SGU_DONE);
                if (con.kind > T_RGU && !t_rg2) trace_at(P, l, TR_W_RGU_DONE);
                if (con.kind == T_DOWN && con.sub == 2 && !t_ds) trace_at(P, l, TR_W_DS_DONE);
            }
            t_rgu |= con.kind == T_RGU;
            t_sgu |= con.kind > T_SGU;
            t_rg2 |= con.kind > T_RGU;
            t_ds |= con.kind == T_DOWN && con.sub == 2;
            if (con.kind == T_ROUTER) {
                const uint16_t* wrow = reinterpret_cast<const uint16_t*>(st);
                float d = 0.0f;
#pragma unroll 8
                for (int k = lane; k < H; k += 32) d = fmaf(bf2f(wrow[k]), bf2f(xs[k]), d);  // exact products
                d = warp_sum_canonical(d);
                if (!n_ready) {
                    if (!(ok = warp_wait_mbar(bar_x, l & 1, P, lane))) break;
                    n_ready = true;
                    r = reinterpret_cast<const float*>(smem + OFF_MISC)[0];
                }
                float z = __fmul_rn(r, d);
                if (D.bias) z = __fadd_rn(z, D.bias[con.t]);
                if (lane == 0) {
                    st_relaxed_u64(D.zt + con.t, tag64(tag, z));
                    red_relaxed_add(D.cnt_z, 1u);
                }
            } else if (con.kind == T_SGU) {
                if (!n_ready) {
                    if (!(ok = warp_wait_mbar(bar_x, l & 1, P, lane))) break;
                    n_ready = true;
                    r = reinterpret_cast<const float*>(smem + OFF_MISC)[0];
                }
                const float v = row_bf16(st, n_s, lane);
                if (con.sub == 0) {
                    carry0 = v;
                } else if (lane == 0) {
                    st_relaxed_u32(D.ht + K * I + (con.t - D.E), tagged_f(gelu_tanh(carry0) * v, tag4));
                }
            } else if (con.kind == T_RGU) {
                const int u = con.t - D.E - N_SGU;
                const int i = u / RGU_PER_EXPERT, p0 = 2 * (u % RGU_PER_EXPERT);
                const float4 gu = rows4_int4(st, dig_s, lane);  // gate p0, up p0, gate p0+1, up p0+1
                if (lane == 0)
                    st_relaxed_v2u32(D.ht + (size_t)i * I + p0, tagged_f(gelu_tanh(gu.x) * gu.y, tag4),
                                     tagged_f(gelu_tanh(gu.z) * gu.w, tag4));
                if (w0t) {
                    if (!t_rg1) trace_at(P, l, TR_W_RGU1_END);
                    trace_at(P, l, TR_W_RGU_END);
                    t_rg1 = true;
                }
            } else {
                const int j0 = 2 * (con.t - D.E - N_SGU - N_RGU);
                const float* hsh = reinterpret_cast<const float*>(smem + OFF_H) + K * I;
                if (con.sub < 2) {
                    // shared down row j0 + sub (bf16, K = S)
                    unsigned long long ac = 0ull;
#pragma unroll 1
                    for (int ch = lane; ch < S / 8; ch += 32) {
                        const uint4 v = *reinterpret_cast<const uint4*>(st + 16 * ch);
                        const float4 h0 = *reinterpret_cast<const float4*>(hsh + 8 * ch);
                        const float4 h1 = *reinterpret_cast<const float4*>(hsh + 8 * ch + 4);
                        ac = dot8_bf16_2(v, h0, h1, ac);
                    }
                    const float acc = warp_sum(sum2(ac));
                    if (con.sub == 0) carry0 = acc;
                    else carry1 = acc;
                } else {
                    // the 8 experts' down rows j0, j0 + 1 (int4, K = I) against the digit blocks of
                    // h_routed: lane = (expert, 32-value block) pair, both rows per pair, so that each
                    // block's digits are read once; the pairs' routing-weighted terms are summed over the warp
                    const uint32_t* dh = reinterpret_cast<const uint32_t*>(smem + OFF_H);
                    constexpr int NB_E = I / 32, NPAIR = K * NB_E;
                    float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll 2
                    for (int pr = lane; pr < NPAIR; pr += 32) {
                        const int i = pr / NB_E, b = pr - i * NB_E;
                        const uint32_t* db = dh + pr * DIG_WORDS;
                        const uint4* dp = reinterpret_cast<const uint4*>(db);
                        const uint4 d0 = dp[0], d1 = dp[1], d2 = dp[2], d3 = dp[3], d4 = dp[4], d5 = dp[5];
                        const float2 meta = *reinterpret_cast<const float2*>(db + 24);
                        const float wi = rt->w[l & 1][i];
                        const uint32_t* sbb = reinterpret_cast<const uint32_t*>(st + DN_SB_OFF + i * 4 * D_SB) +
                                              (j0 & 3) * (D_SB / 4) + (b >> 1);
#pragma unroll
                        for (int jr = 0; jr < 2; ++jr) {
                            const uint4 q = *reinterpret_cast<const uint4*>(st + i * 2 * D_ROW + jr * D_ROW + 16 * b);
                            int s0 = 0, s1 = 0, s2 = 0;
                            word_digits(q.x, d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, s0, s1, s2);
                            word_digits(q.y, d1.z, d1.w, d2.x, d2.y, d2.z, d2.w, s0, s1, s2);
                            word_digits(q.z, d3.x, d3.y, d3.z, d3.w, d4.x, d4.y, s0, s1, s2);
                            word_digits(q.w, d4.z, d4.w, d5.x, d5.y, d5.z, d5.w, s0, s1, s2);
                            const float pq = fmaf((float)s2, 65536.0f, fmaf((float)s1, 256.0f, (float)s0)) * meta.x;
                            const uint32_t sbw = sbb[jr * (D_SB / 4)];
                            const float yb = fmaf(h2f(sbw & 0xffffu), pq, h2f(sbw >> 16) * meta.y);
                            if (jr == 0) acc0 = fmaf(wi, yb, acc0);
                            else acc1 = fmaf(wi, yb, acc1);
                        }
                    }
                    const float y0 = warp_sum(acc0), y1 = warp_sum(acc1);
                    if (lane == 0) {
                        const uint32_t o0 = f2bf(bf2f(xs[j0]) + (carry0 + y0));
                        const uint32_t o1 = f2bf(bf2f(xs[j0 + 1]) + (carry1 + y1));
                        const uint32_t plain = o0 | (o1 << 16);
                        *reinterpret_cast<uint32_t*>(D.act_out + j0) = plain;
                        if (pout) *reinterpret_cast<uint32_t*>(pout + j0) = plain;
                        st_relaxed_u64(D.xt + j0, ((unsigned long long)(o1 | (tag16 << 16)) << 32) |
                                                      (o0 | (tag16 << 16)));
                    }
                }
            }
            __syncwarp();
            ++n_con;
            it_next(con, c);
        }
        if (!ok) break;
        if (!hs_sig) signal_phase(P, l, -1, &cta_cnt[0], D.cnt_hs, lane);
        if (!hr_sig) signal_phase(P, l, TR_CTA_HR_DONE, &cta_cnt[1], D.cnt_hr, lane);
        // observe this layer's routing and h phases even without items that needed
        // them, so that later parity tests never run two phases behind (the next
        // copies go out first only when a phase is still pending: otherwise the
        // layer's output is counted first)
        const bool all_seen = n_ready && hs_ready && hr_ready && k_seen > l;
        if (!all_seen) try_issue();
        if (!n_ready && !(ok = warp_wait_mbar(bar_x, l & 1, P, lane))) break;
        if (!topk_known(l)) {
            if (!(ok = warp_wait_mbar(bar_k, l & 1, P, lane))) break;
            k_seen = l + 1;
        }
        if (!hs_ready && !(ok = warp_wait_mbar(bar_hs, l & 1, P, lane))) break;
        if (!hr_ready && !(ok = warp_wait_mbar(bar_hr, l & 1, P, lane))) break;
        signal_phase(P, l, TR_CTA_OUT, &cta_cnt[2], D.cnt_out, lane);
        if (w0t) trace_at(P, l, TR_W_DONE);
        if (all_seen) try_issue();
    }

    if (!ok && lane == 0) {
        // let this warp's copies in flight land before the CTA's shared memory goes away
        for (int j = n_con; j < n_iss; ++j) {
            const uint64_t t0 = gtimer();
            while (!mbar_try_wait(bar0 + 8 * (j % NS), (j / NS) & 1))
                if (gtimer() - t0 > OWN_LIMIT_NS) break;
        }
    }
}

}  // namespace fused
}  // namespace tf

// ------------------------------------------------------------------ host side

using namespace tf;

struct tf_stack {
    int L = 0, E = 0;
    char* ws = nullptr;
    size_t ws_bytes = 0;
    fused::LayerDesc* d_layers = nullptr;
    uint32_t* err = nullptr;
    uint32_t* epoch = nullptr;
    char* state = nullptr;          // per-layer blocks (everything the kernel writes)
    size_t state_bytes = 0;
    std::vector<fused::LayerDesc> layers;   // host copy (pointers into ws)
    int grid = 0;
    int prefetch = 0;
    unsigned long long* trace = nullptr;
};

namespace {

struct StackCarve {
    size_t err, epoch, descs, layers0, per_layer, total;
    size_t cnt_z, cnt_hs, cnt_hr, cnt_out, zt, ht, xt, logits, idx, w, act;
};

StackCarve stack_carve(int L, int E) {
    StackCarve c;
    size_t o = 0;
    c.err = o; o += 128;
    c.epoch = o; o += 128;
    c.descs = o; o += align_up((size_t)L * sizeof(fused::LayerDesc), 256);
    c.layers0 = o;
    // per-layer block
    size_t p = 0;
    c.cnt_z = p; p += 128;
    c.cnt_hs = p; p += 128;
    c.cnt_hr = p; p += 128;
    c.cnt_out = p; p += 128;
    c.zt = p; p += align_up((size_t)E * 8, 128);
    c.ht = p; p += align_up((size_t)fused::H_FLOATS * 4, 128);
    c.xt = p; p += align_up((size_t)fused::H * 4, 128);
    c.logits = p; p += align_up((size_t)E * 4, 128);
    c.idx = p; p += 128;
    c.w = p; p += 128;
    c.act = p; p += align_up((size_t)fused::H * 2, 128);
    c.per_layer = align_up(p, 256);
    c.total = o + (size_t)L * c.per_layer;
    return c;
}

// Zero the error word and every per-layer block, and start the epoch at 1 (a zeroed
// tagged word carries tag 0, which no launch with epoch >= 1 uses for layer 0).
cudaError_t stack_reset(tf_stack* s, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(s->err, 0, 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(s->state, 0, s->state_bytes, st);
    static const uint32_t one = 1;
    if (e == cudaSuccess) e = cudaMemcpyAsync(s->epoch, &one, 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

}  // namespace

extern "C" {

size_t tf_stack_workspace_bytes(int L, int E) {
    if (L < 1 || L > fused::MAX_L || E < fused::K || E > TF_MAX_E) return 0;
    return stack_carve(L, E).total;
}

tf_status tf_stack_create(tf_layer* const* layers, int L, const float* const* logit_bias, void* workspace,
                          size_t ws_bytes, tf_stack** out) {
    const char* fn = "tf_stack_create";
    if (!out) return fail(TF_ERR_INVALID_ARG, "%s: out is NULL", fn);
    *out = nullptr;
    if (!layers || L < 1) return fail(TF_ERR_INVALID_ARG, "%s: no layers", fn);
    if (L > fused::MAX_L) return fail(TF_ERR_NOT_SUPPORTED, "%s: at most %d layers (L=%d)", fn, fused::MAX_L, L);
    std::vector<tf_layer_desc> ds((size_t)L);
    for (int l = 0; l < L; ++l) {
        if (!layers[l]) return fail(TF_ERR_INVALID_ARG, "%s: layer %d is NULL", fn, l);
        layer_desc_of(layers[l], &ds[l]);
        const tf_layer_desc& d = ds[l];
        if (d.H != fused::H || d.I != fused::I || d.S != fused::S || d.k != fused::K)
            return fail(TF_ERR_NOT_SUPPORTED,
                        "%s: the fused kernel is built for H=2816 I=704 S=2112 k=8 (layer %d has H=%d I=%d S=%d k=%d);"
                        " use tf_stack_decode",
                        fn, l, d.H, d.I, d.S, d.k);
        if (d.E != ds[0].E) return fail(TF_ERR_INVALID_ARG, "%s: all layers need the same E", fn);
        if (!d.experts.base || !aligned16(d.experts.base) || d.experts.stride % 16)
            return fail(TF_ERR_INVALID_ARG, "%s: layer %d needs a resident, 16-byte aligned expert table", fn, l);
    }
    const int E = ds[0].E;
    if (E < fused::K || E > fused::MAX_E || E % 2)
        return fail(TF_ERR_NOT_SUPPORTED, "%s: the fused kernel takes an even E in [8, %d] (E=%d)", fn, fused::MAX_E, E);
    StackCarve sc = stack_carve(L, E);
    if (!workspace || ws_bytes < sc.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return fail(TF_ERR_INVALID_ARG, "%s: workspace NULL, misaligned or smaller than %zu bytes", fn, sc.total);
    int dev = 0, sms = 0, coop = 0, occ = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    cudaError_t e = cudaFuncSetAttribute(fused::k_fused_stack, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)fused::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fused::k_fused_stack, fused::NT, fused::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_status(e, fn);
    if (!coop || occ < 1) return fail(TF_ERR_NOT_SUPPORTED, "%s: cooperative launch unavailable (occupancy %d)", fn, occ);
    tf_stack* s = new (std::nothrow) tf_stack();
    if (!s) return fail(TF_ERR_OOM, "%s: out of host memory", fn);
    s->L = L;
    s->E = E;
    s->ws = static_cast<char*>(workspace);
    s->ws_bytes = ws_bytes;
    s->err = reinterpret_cast<uint32_t*>(s->ws + sc.err);
    s->epoch = reinterpret_cast<uint32_t*>(s->ws + sc.epoch);
    s->d_layers = reinterpret_cast<fused::LayerDesc*>(s->ws + sc.descs);
    s->state = s->ws + sc.layers0;
    s->state_bytes = (size_t)L * sc.per_layer;
    s->grid = sms;
    ExpertLayout lay;
    expert_layout(fused::H, fused::I, &lay);
    s->layers.resize((size_t)L);
    for (int l = 0; l < L; ++l) {
        char* base = s->state + (size_t)l * sc.per_layer;
        fused::LayerDesc& D = s->layers[l];
        std::memset(&D, 0, sizeof(D));
        const tf_layer_desc& d = ds[l];
        D.Wr = static_cast<const uint16_t*>(d.W_r);
        D.Wsg = static_cast<const uint16_t*>(d.W_sg);
        D.Wsu = static_cast<const uint16_t*>(d.W_su);
        D.Wsd = static_cast<const uint16_t*>(d.W_sd);
        D.ebase = static_cast<const char*>(d.experts.base);
        D.estride = d.experts.stride;
        D.slot_map = d.experts.slot_of_expert;
        D.bias = logit_bias ? logit_bias[l] : nullptr;
        D.cnt_z = reinterpret_cast<uint32_t*>(base + sc.cnt_z);
        D.cnt_hs = reinterpret_cast<uint32_t*>(base + sc.cnt_hs);
        D.cnt_hr = reinterpret_cast<uint32_t*>(base + sc.cnt_hr);
        D.cnt_out = reinterpret_cast<uint32_t*>(base + sc.cnt_out);
        D.zt = reinterpret_cast<unsigned long long*>(base + sc.zt);
        D.ht = reinterpret_cast<uint32_t*>(base + sc.ht);
        D.xt = reinterpret_cast<uint32_t*>(base + sc.xt);
        D.logits = reinterpret_cast<float*>(base + sc.logits);
        D.idx = reinterpret_cast<int32_t*>(base + sc.idx);
        D.w = reinterpret_cast<float*>(base + sc.w);
        D.act_out = reinterpret_cast<uint16_t*>(base + sc.act);
        D.E = E;
        D.eps = d.eps;
        D.n_slots = d.experts.n_slots;
        D.off_gu_sb = lay.gu_sb;
        D.off_d_codes = lay.d_codes;
        D.off_d_sb = lay.d_sb;
    }
    e = cudaMemcpy(s->d_layers, s->layers.data(), (size_t)L * sizeof(fused::LayerDesc), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = stack_reset(s, nullptr);
    if (e != cudaSuccess) {
        delete s;
        return cuda_status(e, fn);
    }
    *out = s;
    return TF_OK;
}

tf_status tf_stack_set_prefetch(tf_stack* s, int on) {
    if (!s) return fail(TF_ERR_INVALID_ARG, "tf_stack_set_prefetch: NULL");
    s->prefetch = on ? 1 : 0;
    return TF_OK;
}

tf_status tf_stack_set_trace(tf_stack* s, void* buffer, size_t bytes) {
    if (!s) return fail(TF_ERR_INVALID_ARG, "tf_stack_set_trace: NULL");
    const size_t need = (size_t)s->L * fused::TRACE_CTAS * fused::TRACE_SLOTS * 8;  // L x 256 x 16 stamps
    if (buffer && bytes < need) return fail(TF_ERR_INVALID_ARG, "tf_stack_set_trace: the buffer needs %zu bytes", need);
    if (buffer && s->grid > fused::TRACE_CTAS)
        return fail(TF_ERR_NOT_SUPPORTED, "tf_stack_set_trace: more than %d CTAs", fused::TRACE_CTAS);
    if (buffer && (reinterpret_cast<uintptr_t>(buffer) & 7))
        return fail(TF_ERR_INVALID_ARG, "tf_stack_set_trace: the buffer must be 8-byte aligned");
    s->trace = static_cast<unsigned long long*>(buffer);
    return TF_OK;
}

tf_status tf_stack_step(tf_stack* s, const void* x, void* out, void* stream) {
    const char* fn = "tf_stack_step";
    if (!s || !x || !out) return fail(TF_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned16(x) || !aligned16(out)) return fail(TF_ERR_INVALID_ARG, "%s: x and out must be 16-byte aligned", fn);
    if (x == out) return fail(TF_ERR_INVALID_ARG, "%s: out must not alias x", fn);
    fused::Params P;
    P.layers = s->d_layers;
    P.L = s->L;
    P.x = static_cast<const uint16_t*>(x);
    P.out = static_cast<uint16_t*>(out);
    P.err = s->err;
    P.epoch = s->epoch;
    P.prefetch = s->prefetch;
    P.trace = s->trace;
    P.dep_limit_ns = test_wait_limit_ns();
    void* args[] = {&P};
    clear_error();
    prof_before(TF_KERNEL_LAYER, stream);
    cudaError_t e = cudaLaunchCooperativeKernel((void*)fused::k_fused_stack, dim3(s->grid), dim3(fused::NT), args,
                                                fused::SMEM_BYTES, static_cast<cudaStream_t>(stream));
    prof_after(TF_KERNEL_LAYER, stream);
    return cuda_status(e, fn);
}

tf_status tf_stack_check(tf_stack* s, void* stream) {
    if (!s) return fail(TF_ERR_INVALID_ARG, "tf_stack_check: NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t err = 0;
    cudaError_t e = cudaMemcpyAsync(&err, s->err, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e, "tf_stack_check");
    if (err) {
        // a bounded wait gave up: start again from a zeroed state and epoch 1
        e = stack_reset(s, st);
        if (e != cudaSuccess) return cuda_status(e, "tf_stack_check");
        return fail(TF_ERR_TIMEOUT, "tf_stack_check: a device-side wait timed out (error word 0x%x)", err);
    }
    return TF_OK;
}

tf_status tf_stack_layer_buffers(tf_stack* s, int layer, int32_t** idx, float** w, float** logits, void** act_out) {
    if (!s || layer < 0 || layer >= s->L) return fail(TF_ERR_INVALID_ARG, "tf_stack_layer_buffers: bad arguments");
    const fused::LayerDesc& D = s->layers[layer];
    if (idx) *idx = D.idx;
    if (w) *w = D.w;
    if (logits) *logits = D.logits;
    if (act_out) *act_out = D.act_out;
    return TF_OK;
}

tf_status tf_stack_destroy(tf_stack* s) {
    delete s;
    return TF_OK;
}

}  // extern "C"
