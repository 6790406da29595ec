// Fused persistent decode kernel: a whole stack of MoE layers for one token in
// one cooperative launch (one CTA per SM).
//
// The per-layer flow is the pages' (page "Como executar um modelo de 26 bilhoes
// de parametros em dois gigabytes de memoria em um Mac comum", section "Qual e
// o principal truque da arquitetura"): router -> top-8 -> expert FFNs, with the
// shared-expert branch beside them. What differs is how it is fed on B300.
//
// Work. Ten worker warps per CTA each own a two-stage shared-memory ring,
// filled by cp.async.bulk copies that the warp's lane 0 issues ahead of use
// (completion on per-stage mbarriers). A layer is cut into tasks, dealt
// round-robin over all worker warps of the grid (continuing from layer to
// layer):
//   router : one row of W_r (bf16), fixed-order dot product -> one logit
//   sgu    : one shared gate/up row pair (bf16, two stages) -> one h_shared
//   rgu    : two gate/up row pairs of one selected expert (int4) -> two h_routed
//   down   : two output rows: shared down (bf16, two stages) and the eight
//            experts' down rows (int4, one stage), weighted combine, residual
//            add, bf16 output
// A worker only blocks when its next copy needs the layer's top-8 experts.
//
// Synchronisation. Every value that crosses CTAs (router logits, h, the layer
// output) is published as one 32- or 64-bit word that carries the value and a
// tag (launch epoch x 64 + layer); a reader polls the words it needs until all
// tags are current. No fence is on the dependency chain: GPU-scope fences cost
// microseconds while the SM's memory pipeline is full of weight copies. Two
// relaxed counters per layer (bumped once per CTA, without ordering) only tell
// the readers when polling is worth starting. Four control warps per CTA poll and stage: warp 0 stages the
// layer input (x, r, n = r x) and computes the CTA's own copy of the top-8 from
// the tagged logits, and warps 0..3 stage h for the down projections; each
// stage is published to the workers with an mbarrier. The epoch lives in the
// workspace; CTA 0 advances it once the last layer's output is complete, so a
// launch needs nothing from the host but its pointers.
//
// While a layer runs, each worker prefetches into L2 the data-independent
// weights (router rows, shared expert) of its tasks in the next layer.
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
constexpr int D_WORDS = I / 8;             // 88 words per down row
constexpr int N_SGU = S;                   // tasks of one shared row pair
constexpr int N_RGU = K * I / 2;           // tasks of two routed row pairs
constexpr int RGU_PER_EXPERT = I / 2;      // 352
constexpr int N_DN = H / 2;                // tasks of two output rows
constexpr int RGU_BYTES = 4 * GU_ROW + 4 * GU_SB;   // 6336
constexpr int DN_SB_OFF = K * 2 * D_ROW;            // 5632
constexpr int DN_BYTES = DN_SB_OFF + K * 4 * D_SB;  // 7040
constexpr int H_FLOATS = K * I + S;                 // h_routed then h_shared
constexpr int H_QUARTER = H_FLOATS / NCTRL;         // 1936 words per control warp
constexpr unsigned long long TIMEOUT_NS = 2000000000ull;  // 2 s per wait
constexpr uint32_t SUSPEND_NS = 1000;      // suspend hint of a blocking mbarrier test
constexpr uint32_t HINT_SLEEP_NS = 256;    // pause between two reads of a hint counter
static_assert(HW == 32 * WPL, "lane ownership of the K = H words");
static_assert(ROW_BF <= STAGE && RGU_BYTES <= STAGE && DN_BYTES <= STAGE && SROW_BF <= STAGE, "stage size");
static_assert(H_FLOATS % (8 * NCTRL) == 0 && (K * I) % 8 == 0, "h quarters hold whole 8-float words");
static_assert((H_QUARTER / 2 + 31) / 32 <= 32 && (H / 4) / 32 <= 32, "poll masks fit 32 bits");

// shared-memory layout
constexpr int OFF_RING = 0;
constexpr int OFF_XS = OFF_RING + NWORK * NS * STAGE;   // bf16 x [H]
constexpr int OFF_N = OFF_XS + H * 2;                    // fp32 n [H]
constexpr int OFF_SN = OFF_N + H * 4;                    // fp32 word sums of n [HW]
constexpr int OFF_H = OFF_SN + HW * 4;                   // fp32 h_routed [K*I], h_shared [S]
constexpr int OFF_SH = OFF_H + H_FLOATS * 4;             // fp32 word sums of h_routed [K*I/8]
constexpr int OFF_Z = OFF_SH + (K * I / 8) * 4;          // top-k scratch: fp32 z [MAX_E], taken [MAX_E]
constexpr int OFF_RT = OFF_Z + MAX_E * 5;                // routing cache [2 layers]: expert ptrs, weights, ids
constexpr int RT_BYTES = 2 * (K * 8 + K * 4 + K * 4);
constexpr int OFF_BAR = OFF_RT + RT_BYTES;               // mbarriers
constexpr int N_BAR = NWORK * NS + 4;                    // stages, XREADY, TOPKREADY, HREADY, HHINT
constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;            // r, epoch
constexpr size_t SMEM_BYTES = OFF_MISC + 16;
static_assert(OFF_H % 16 == 0 && OFF_N % 16 == 0 && OFF_RT % 16 == 0 && OFF_BAR % 8 == 0 && OFF_Z % 16 == 0,
              "alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

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
    unsigned long long* ht;   // tagged h [H_FLOATS]: routed [K*I] then shared [S]
    uint32_t* xt;             // tagged output [H]: (tag16 << 16) | bf16
    float* logits;            // plain copies for inspection, written by CTA 0
    int32_t* idx;
    float* w;
    uint16_t* act_out;        // plain bf16 output (the last layer also writes the call's `out`)
    uint32_t* cnt_z;          // router rows of this layer scored (pacing hint, += E per launch)
    uint32_t* cnt_h;          // CTAs whose h tasks of this layer are done (pacing hint, += gridDim per launch)
    uint32_t* cnt_out;        // CTAs whose output rows of this layer are done (same)
    int E;
    float eps;
    unsigned long long off_gu_sb, off_d_codes, off_d_sb;
};

struct Params {
    const LayerDesc* layers;
    int L;
    const uint16_t* x;
    uint16_t* out;
    uint32_t* err;
    uint32_t* epoch;             // launch epoch (>= 1), advanced by CTA 0 at the end
    int prefetch;                // 1: prefetch the next layer's data-independent weights into L2
    unsigned long long* trace;   // nullable: TRACE_SLOTS %globaltimer stamps per (layer, CTA)
};

// Trace slots per (layer, CTA) (ns stamps of %globaltimer), written when
// Params::trace is set: trace[(layer * TRACE_CTAS + cta) * TRACE_SLOTS + slot].
enum {
    TR_X_READY = 0,      // control warp 0 saw the whole layer input
    TR_X_STAGED = 1,     // ... published x, r, n
    TR_Z_READY = 2,      // ... saw all router logits
    TR_TOPK = 3,         // ... published the top-k
    TR_H_HINT = 4,       // ... saw the h hint counter complete
    TR_H_STAGED = 5,     // ... staged its quarter of h
    TR_CTA_H_DONE = 6,   // the CTA's last worker finished its h-producing items
    TR_CTA_OUT = 7,      // the CTA's last worker finished the layer
    TRACE_SLOTS = 8,
    TRACE_CTAS = 256
};

enum { T_ROUTER = 0, T_SGU = 1, T_RGU = 2, T_DOWN = 3 };
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
// Blocking test: the thread sleeps until the phase completes or about ns elapse.
__device__ __forceinline__ bool mbar_wait_hint(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
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

// Bounded wait on an mbarrier phase (one lane); false (error recorded) on timeout or when another CTA failed.
__device__ bool wait_mbar(uint32_t bar, uint32_t parity, uint32_t* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_wait_hint(bar, parity, SUSPEND_NS)) return true;
        if ((n & 7u) == 0) {
            if (err_set(err)) return false;
            if (gtimer() - t0 > TIMEOUT_NS) {
                atomicOr(err, ERR_TIMEOUT);
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool warp_wait_mbar(uint32_t bar, uint32_t parity, uint32_t* err, int lane) {
    bool ok = true;
    if (lane == 0) ok = wait_mbar(bar, parity, err);
    return __shfl_sync(FULL, (int)ok, 0) != 0;
}

// Pacing of a warp polling tagged data; gives up (error recorded) after TIMEOUT_NS.
struct Poll {
    uint64_t t0;
    int rounds;
    __device__ void start() {
        t0 = gtimer();
        rounds = 0;
    }
    // After a round: true = poll again, false = done (nothing pending) or give up.
    __device__ bool again(bool pending_any, uint32_t* err, int lane) {
        if (!pending_any) return false;
        ++rounds;
        int stop = 0;
        if (lane == 0 && (rounds & 15) == 0) {
            if (err_set(err)) {
                stop = 1;
            } else if (gtimer() - t0 > TIMEOUT_NS) {
                atomicOr(err, ERR_TIMEOUT);
                stop = 1;
            }
        }
        __nanosleep(rounds < 8 ? 64 : 256);
        return __shfl_sync(FULL, stop, 0) == 0;
    }
};

// Wait (one warp) until the hint counter reaches target (modular u32 compare).
// The counter only paces the polling of tagged data; it orders nothing.
__device__ bool wait_hint(const uint32_t* cnt, uint32_t target, uint32_t* err, int lane) {
    int st = 0;  // 0 waiting, 1 reached, 2 give up
    if (lane == 0) {
        const uint64_t t0 = gtimer();
        for (uint32_t n = 0;; ++n) {
            if ((int32_t)(ld_relaxed_u32(cnt) - target) >= 0) { st = 1; break; }
            __nanosleep(HINT_SLEEP_NS);
            if ((n & 15u) == 15u) {
                if (err_set(err)) { st = 2; break; }
                if (gtimer() - t0 > TIMEOUT_NS) { atomicOr(err, ERR_TIMEOUT); st = 2; break; }
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
        trace_at(P, l, slot);
    }
    __syncwarp();
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

// Lane 0 enqueues the copies of one item into a stage.
__device__ void issue_item(const Ctx& c, const It& it, const Route* rt, uint32_t dst, uint32_t bar, uint64_t pol) {
    const LayerDesc& D = c.P->layers[it.l];
    fence_proxy_async();  // the stage's previous contents were read through the generic proxy
    if (it.kind == T_ROUTER) {
        mbar_expect_tx(bar, ROW_BF);
        bulk_g2s(dst, D.Wr + (size_t)it.t * H, ROW_BF, bar, pol);
    } else if (it.kind == T_SGU) {
        const int j = it.t - D.E;
        mbar_expect_tx(bar, ROW_BF);
        bulk_g2s(dst, (it.sub == 0 ? D.Wsg : D.Wsu) + (size_t)j * H, ROW_BF, bar, pol);
    } else if (it.kind == T_RGU) {
        const int u = it.t - D.E - N_SGU;
        const int i = u / RGU_PER_EXPERT, p0 = 2 * (u % RGU_PER_EXPERT);
        const char* ep = rt->ep[it.l & 1][i];
        mbar_expect_tx(bar, RGU_BYTES);
        bulk_g2s(dst, ep + (size_t)2 * p0 * GU_ROW, 4 * GU_ROW, bar, pol);
        bulk_g2s(dst + 4 * GU_ROW, ep + D.off_gu_sb + (size_t)2 * p0 * GU_SB, 4 * GU_SB, bar, pol);
    } else {
        const int j0 = 2 * (it.t - D.E - N_SGU - N_RGU);
        if (it.sub < 2) {
            mbar_expect_tx(bar, SROW_BF);
            bulk_g2s(dst, D.Wsd + (size_t)(j0 + it.sub) * S, SROW_BF, bar, pol);
        } else {
            mbar_expect_tx(bar, DN_BYTES);
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const char* ep = rt->ep[it.l & 1][i];
                bulk_g2s(dst + i * 2 * D_ROW, ep + D.off_d_codes + (size_t)j0 * D_ROW, 2 * D_ROW, bar, pol);
                bulk_g2s(dst + DN_SB_OFF + i * 4 * D_SB, ep + D.off_d_sb + (size_t)(j0 & ~3) * D_SB, 4 * D_SB, bar,
                         pol);
            }
        }
    }
}

// L2 prefetch of the data-independent weights of worker gw's tasks in layer l.
__device__ void prefetch_layer(const Ctx& c, int l) {
    const LayerDesc& D = c.P->layers[l];
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
// Byte b of x as the fp32 value 128 + x.byte_b (bytes hold one code 0..15): the
// byte lands in mantissa bits 16..23 under the exponent of 128.0f.
template <int B>
__device__ __forceinline__ float byte128(uint32_t x) {
    return __uint_as_float(__byte_perm(x, 0x43000000u, 0x7054u | (B << 8)));
}
// sum_p (128 + q_p) n_p over the 8 codes of one word (code p in bits 4p..4p+3).
__device__ __forceinline__ float dot8_q128_2(uint32_t q, float4 a, float4 b) {
    const uint32_t lo = q & 0x0f0f0f0fu, hi = (q >> 4) & 0x0f0f0f0fu;  // codes 0,2,4,6 / 1,3,5,7
    unsigned long long acc = 0ull;
    fma2(acc, pk2(byte128<0>(lo), byte128<0>(hi)), pk2(a.x, a.y));
    fma2(acc, pk2(byte128<1>(lo), byte128<1>(hi)), pk2(a.z, a.w));
    fma2(acc, pk2(byte128<2>(lo), byte128<2>(hi)), pk2(b.x, b.y));
    fma2(acc, pk2(byte128<3>(lo), byte128<3>(hi)), pk2(b.z, b.w));
    return sum2(acc);
}
// acc + sum over 8 bf16 weights (one 16-byte chunk) times n, packed FMA.
__device__ __forceinline__ unsigned long long dot8_bf16_2(uint4 w, float4 a, float4 b, unsigned long long acc) {
    fma2(acc, pk2(bf_lo(w.x), bf_hi(w.x)), pk2(a.x, a.y));
    fma2(acc, pk2(bf_lo(w.y), bf_hi(w.y)), pk2(a.z, a.w));
    fma2(acc, pk2(bf_lo(w.z), bf_hi(w.z)), pk2(b.x, b.y));
    fma2(acc, pk2(bf_lo(w.w), bf_hi(w.w)), pk2(b.z, b.w));
    return acc;
}
// acc + sum_p (s q_p + b) v_p = acc + s (P - 128 S) + b S for one word of codes.
__device__ __forceinline__ float word_affine(uint32_t q, uint32_t sbw, float4 a, float4 b, float S, float acc) {
    const float P = dot8_q128_2(q, a, b);
    return fmaf(h2f(sbw & 0xffffu), fmaf(-128.0f, S, P), fmaf(h2f(sbw >> 16), S, acc));
}
__device__ __forceinline__ void warp_sum4(float& a, float& b, float& c, float& d) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        a += __shfl_xor_sync(FULL, a, o);
        b += __shfl_xor_sync(FULL, b, o);
        c += __shfl_xor_sync(FULL, c, o);
        d += __shfl_xor_sync(FULL, d, o);
    }
}

// sum_k W[k] n[k] over a bf16 row of K = H (16-byte chunk w covers n[8w..8w+7]).
__device__ __forceinline__ float row_bf16(const unsigned char* row, const float* n, int lane) {
    const float4* n4 = reinterpret_cast<const float4*>(n);
    unsigned long long acc[2] = {0ull, 0ull};
#pragma unroll
    for (int m = 0; m < WPL; ++m) {
        const int w = lane + 32 * m;
        const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * w);
        acc[m & 1] = dot8_bf16_2(v, n4[2 * w], n4[2 * w + 1], acc[m & 1]);
    }
    return warp_sum(sum2(acc[0]) + sum2(acc[1]));
}

// Four int4 rows of K = H at once (codes: 4 rows of HW words; sb: 4 rows of H/64
// words): lane sums over the words w = lane + 32 m, then four warp reductions.
__device__ __forceinline__ float4 rows4_int4(const uint32_t* codes, const uint32_t* sb, const float* n,
                                             const float* sn, int lane) {
    const float4* n4 = reinterpret_cast<const float4*>(n);
    constexpr int SBW = GU_SB / 4;
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
    for (int m = 0; m < WPL; ++m) {
        const int w = lane + 32 * m, g = w >> 3;
        const float4 na = n4[2 * w], nb = n4[2 * w + 1];
        const float S = sn[w];
        a0 = word_affine(codes[w], sb[g], na, nb, S, a0);
        a1 = word_affine(codes[HW + w], sb[SBW + g], na, nb, S, a1);
        a2 = word_affine(codes[2 * HW + w], sb[2 * SBW + g], na, nb, S, a2);
        a3 = word_affine(codes[3 * HW + w], sb[3 * SBW + g], na, nb, S, a3);
    }
    warp_sum4(a0, a1, a2, a3);
    return make_float4(a0, a1, a2, a3);
}

// ---- control warp 0: the layer input. Wait for every tagged output word of the
// previous layer (or take the call's x), then publish x (bf16), r, n = r x and the
// word sums of n.
__device__ bool stage_x(const Params& P, int l, uint32_t prev_tag16, uint32_t hint_target, unsigned char* smem,
                        int lane) {
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + OFF_XS);
    uint4* x4 = reinterpret_cast<uint4*>(xs);
    constexpr int NCH = H / 4 / 32;   // 22 chunks of 4 tagged words per lane
    if (l == 0) {
        const uint4* s4 = reinterpret_cast<const uint4*>(P.x);
#pragma unroll
        for (int m = 0; m < WPL; ++m) x4[lane + 32 * m] = __ldcg(s4 + lane + 32 * m);
    } else {
        if (!wait_hint(P.layers[l - 1].cnt_out, hint_target, P.err, lane)) return false;
        const uint32_t* src = P.layers[l - 1].xt;
        uint32_t pend = (1u << NCH) - 1u;
        Poll poll;
        poll.start();
        for (;;) {
            // all loads of a round are issued before any is checked (one round trip per round)
            constexpr int BATCH = 8;
#pragma unroll
            for (int m0 = 0; m0 < NCH; m0 += BATCH) {
                const uint32_t pb = pend;
                uint4 v[BATCH];
#pragma unroll
                for (int i = 0; i < BATCH; ++i)
                    if (m0 + i < NCH && (pb >> (m0 + i) & 1u)) v[i] = ld_relaxed_v4(src + 4 * (lane + 32 * (m0 + i)));
#pragma unroll
                for (int i = 0; i < BATCH; ++i) {
                    const int m = m0 + i;
                    if (m < NCH && (pb >> m & 1u) && (v[i].x >> 16) == prev_tag16 && (v[i].y >> 16) == prev_tag16 &&
                        (v[i].z >> 16) == prev_tag16 && (v[i].w >> 16) == prev_tag16) {
                        reinterpret_cast<uint2*>(xs)[lane + 32 * m] = make_uint2(
                            (v[i].x & 0xffffu) | (v[i].y << 16), (v[i].z & 0xffffu) | (v[i].w << 16));
                        pend &= ~(1u << m);
                    }
                }
            }
            if (!poll.again(__any_sync(FULL, pend != 0), P.err, lane)) break;
        }
        if (__any_sync(FULL, pend != 0)) return false;
        if (lane == 0) trace_at(P, l, TR_X_READY);
    }
    __syncwarp();
    const float eps = P.layers[l].eps;
    float p = 0.0f;
#pragma unroll 8
    for (int k = lane; k < H; k += 32) {
        const float v = bf2f(xs[k]);
        p = fmaf(v, v, p);  // exact square: one rounding per term, as in the canonical sum
    }
    p = warp_sum_canonical(p);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(p, (float)H), eps)));
    float* n = reinterpret_cast<float*>(smem + OFF_N);
    float* sn = reinterpret_cast<float*>(smem + OFF_SN);
#pragma unroll
    for (int m = 0; m < WPL; ++m) {
        const int w = lane + 32 * m;
        const uint4 v = x4[w];
        const float4 a = make_float4(__fmul_rn(r, bf_lo(v.x)), __fmul_rn(r, bf_hi(v.x)), __fmul_rn(r, bf_lo(v.y)),
                                     __fmul_rn(r, bf_hi(v.y)));
        const float4 b = make_float4(__fmul_rn(r, bf_lo(v.z)), __fmul_rn(r, bf_hi(v.z)), __fmul_rn(r, bf_lo(v.w)),
                                     __fmul_rn(r, bf_hi(v.w)));
        reinterpret_cast<float4*>(n)[2 * w] = a;
        reinterpret_cast<float4*>(n)[2 * w + 1] = b;
        sn[w] = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
    }
    if (lane == 0) reinterpret_cast<float*>(smem + OFF_MISC)[0] = r;
    __syncwarp();
    return true;
}

// ---- control warp 0: the CTA's copy of the layer's top-k from the tagged logits.
__device__ bool route_layer(const Params& P, int l, uint32_t tag, uint32_t epoch_x_e, unsigned char* smem, Route* rt,
                            bool publish, int lane) {
    const LayerDesc& D = P.layers[l];
    float* zs = reinterpret_cast<float*>(smem + OFF_Z);
    if (!wait_hint(D.cnt_z, epoch_x_e, P.err, lane)) return false;
    constexpr int NCH = MAX_E / 2 / 32;   // <= 4 chunks of 2 tagged logits per lane
    const int nch = D.E / 2;
    uint32_t pend = 0;
#pragma unroll
    for (int m = 0; m < NCH; ++m)
        if (lane + 32 * m < nch) pend |= 1u << m;
    Poll poll;
    poll.start();
    for (;;) {
        const uint32_t pb = pend;
        unsigned long long va[NCH], vb[NCH];
#pragma unroll
        for (int m = 0; m < NCH; ++m)
            if (pb >> m & 1u) ld_relaxed_v2u64(D.zt + 2 * (lane + 32 * m), va[m], vb[m]);
#pragma unroll
        for (int m = 0; m < NCH; ++m) {
            if ((pb >> m & 1u) && (uint32_t)(va[m] >> 32) == tag && (uint32_t)(vb[m] >> 32) == tag) {
                const int ch = lane + 32 * m;
                zs[2 * ch] = __uint_as_float((uint32_t)va[m]);
                zs[2 * ch + 1] = __uint_as_float((uint32_t)vb[m]);
                pend &= ~(1u << m);
            }
        }
        if (!poll.again(__any_sync(FULL, pend != 0), P.err, lane)) break;
    }
    if (__any_sync(FULL, pend != 0)) return false;
    if (lane == 0) trace_at(P, l, TR_Z_READY);
    __syncwarp();
    const int s = l & 1;
    // Top-k by rounds of two warp reductions: the largest remaining logit (as an
    // order-preserving key, -0 == +0, NaN lowest), then the lowest index holding it.
    constexpr int PER = MAX_E / 32;
    uint32_t key[PER];
    float val[PER];
    uint32_t alive = 0;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
        const int j = lane + 32 * m;
        val[m] = j < D.E ? zs[j] : 0.0f;
        const float v = val[m] + 0.0f;  // -0 -> +0
        const uint32_t u = __float_as_uint(v);
        key[m] = isnan(v) ? 0u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
        if (j < D.E) alive |= 1u << m;
    }
    float selz = 0.0f;
    int sel = -1;
    for (int i = 0; i < K; ++i) {
        uint32_t bk = 0u;
        int bi = 0x7fffffff;
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            const int j = lane + 32 * m;
            if ((alive >> m & 1u) && (key[m] > bk || (key[m] == bk && j < bi))) {
                bk = key[m];
                bi = j;
            }
        }
        const uint32_t kmax = __reduce_max_sync(FULL, bk);
        const int imin = (int)__reduce_min_sync(FULL, (uint32_t)(bk == kmax ? bi : 0x7fffffff));
        float vsel = 0.0f;
#pragma unroll
        for (int m = 0; m < PER; ++m)
            if (lane + 32 * m == imin) {
                vsel = val[m];
                alive &= ~(1u << m);
            }
        vsel = __shfl_sync(FULL, vsel, imin & 31);
        if (lane == i) {
            sel = imin;
            selz = vsel;
        }
    }
    // softmax over the selected logits, summed in top-k order
    float zmax = __shfl_sync(FULL, selz, 0);
    for (int i = 1; i < K; ++i) {
        const float zi = __shfl_sync(FULL, selz, i);
        if (zi > zmax) zmax = zi;
    }
    const float ev = lane < K ? expf(__fsub_rn(selz, zmax)) : 0.0f;
    float esum = 0.0f;
    for (int i = 0; i < K; ++i) esum = __fadd_rn(esum, __shfl_sync(FULL, ev, i));
    if (lane < K) {
        rt->id[s][lane] = sel;
        rt->w[s][lane] = __fdiv_rn(ev, esum);
    }
    __syncwarp();
    int bad = 0;
    if (lane < K) {
        int e = rt->id[s][lane];
        bad = (unsigned)e >= (unsigned)D.E;
        if (bad) e = 0;  // never form an address from an out-of-range id
        if (D.slot_map) e = __ldcg(D.slot_map + e);
        rt->ep[s][lane] = D.ebase + (size_t)e * D.estride;
        if (publish) {
            D.idx[lane] = rt->id[s][lane];
            D.w[lane] = rt->w[s][lane];
        }
    }
    if (publish)
        for (int j = lane; j < D.E; j += 32) D.logits[j] = zs[j];
    if (__any_sync(FULL, bad)) {
        if (lane == 0) atomicOr(P.err, ERR_BAD_ID);
        return false;
    }
    __syncwarp();
    return true;
}

// ---- control warps 0..3: quarter q of h (tagged fp32) -> shared memory, plus the
// word sums of its h_routed part.
__device__ bool stage_h(const Params& P, int l, uint32_t tag, uint32_t hint_target, uint32_t bar_hh,
                        unsigned char* smem, int q, int lane) {
    const LayerDesc& D = P.layers[l];
    // control warp 0 reads the hint counter; warps 1..3 sleep on an mbarrier until it is reached
    if (q == 0) {
        if (!wait_hint(D.cnt_h, hint_target, P.err, lane)) return false;
        if (lane == 0) {
            mbar_arrive(bar_hh);
            trace_at(P, l, TR_H_HINT);
        }
    } else if (!warp_wait_mbar(bar_hh, l & 1, P.err, lane)) {
        return false;
    }
    float* h = reinterpret_cast<float*>(smem + OFF_H);
    float* sh = reinterpret_cast<float*>(smem + OFF_SH);
    constexpr int NCHQ = H_QUARTER / 2;              // 968 chunks of 2 tagged words
    constexpr int NCH = (NCHQ + 31) / 32;            // 31 per lane
    const int w0 = q * H_QUARTER;
    uint32_t pend = 0;
#pragma unroll
    for (int m = 0; m < NCH; ++m)
        if (lane + 32 * m < NCHQ) pend |= 1u << m;
    Poll poll;
    poll.start();
    for (;;) {
        // all loads of a batch are issued before any is checked
        constexpr int BATCH = 8;
#pragma unroll
        for (int m0 = 0; m0 < NCH; m0 += BATCH) {
            const uint32_t pb = pend;
            unsigned long long va[BATCH], vb[BATCH];
#pragma unroll
            for (int i = 0; i < BATCH; ++i)
                if (m0 + i < NCH && (pb >> (m0 + i) & 1u))
                    ld_relaxed_v2u64(D.ht + w0 + 2 * (lane + 32 * (m0 + i)), va[i], vb[i]);
#pragma unroll
            for (int i = 0; i < BATCH; ++i) {
                const int m = m0 + i;
                if (m < NCH && (pb >> m & 1u) && (uint32_t)(va[i] >> 32) == tag && (uint32_t)(vb[i] >> 32) == tag) {
                    *reinterpret_cast<float2*>(h + w0 + 2 * (lane + 32 * m)) =
                        make_float2(__uint_as_float((uint32_t)va[i]), __uint_as_float((uint32_t)vb[i]));
                    pend &= ~(1u << m);
                }
            }
        }
        if (!poll.again(__any_sync(FULL, pend != 0), P.err, lane)) break;
    }
    if (__any_sync(FULL, pend != 0)) return false;
    __syncwarp();
    // word sums of h_routed for the 8-float words of this quarter
    for (int w8 = w0 / 8 + lane; w8 < (w0 + H_QUARTER) / 8 && w8 < K * I / 8; w8 += 32) {
        const float4 a = reinterpret_cast<const float4*>(h)[2 * w8];
        const float4 b = reinterpret_cast<const float4*>(h)[2 * w8 + 1];
        sh[w8] = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
    }
    __syncwarp();
    return true;
}

// ------------------------------------------------------------------ the kernel

__global__ void __launch_bounds__(NT, 1) k_fused_stack(Params P) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = gridDim.x;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    const uint32_t bar_x = smem_u32(&bars[NWORK * NS]);
    const uint32_t bar_k = smem_u32(&bars[NWORK * NS + 1]);
    const uint32_t bar_h = smem_u32(&bars[NWORK * NS + 2]);
    const uint32_t bar_hh = smem_u32(&bars[NWORK * NS + 3]);
    Route* rt = reinterpret_cast<Route*>(smem + OFF_RT);
    uint32_t* s_epoch = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 4);
    uint32_t* cta_cnt = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 8);  // [0] h phase, [1] output phase

    if (threadIdx.x == 0) {
        for (int s = 0; s < NWORK * NS; ++s) mbar_init(smem_u32(&bars[s]), 1);
        mbar_init(bar_x, 1);
        mbar_init(bar_k, 1);
        mbar_init(bar_h, NCTRL);
        mbar_init(bar_hh, 1);
        *s_epoch = ld_relaxed_u32(P.epoch);
        cta_cnt[0] = 0;
        cta_cnt[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint32_t epoch = *s_epoch;
    const uint32_t hint_target = epoch * (uint32_t)G;   // every launch adds G to each hint counter
    const int E = P.layers[0].E;

    if (warp < NCTRL) {
        // ================================================= control warps
        bool ok = true;
        for (int l = 0; l < P.L && ok; ++l) {
            const uint32_t tag = epoch * 64u + (uint32_t)l;
            if (warp == 0) {
                ok = stage_x(P, l, (tag - 1u) & 0xffffu, hint_target, smem, lane);
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive(bar_x);
                    trace_at(P, l, TR_X_STAGED);
                }
                ok = route_layer(P, l, tag, epoch * (uint32_t)E, smem, rt, blockIdx.x == 0, lane);
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive(bar_k);
                    trace_at(P, l, TR_TOPK);
                }
            }
            ok = stage_h(P, l, tag, hint_target, bar_hh, smem, warp, lane);
            if (!ok) break;
            if (lane == 0) {
                mbar_arrive(bar_h);
                if (warp == 0) trace_at(P, l, TR_H_STAGED);
            }
        }
        // CTA 0 advances the epoch once the last layer's output is complete
        if (ok && blockIdx.x == 0 && warp == 0 && wait_hint(P.layers[P.L - 1].cnt_out, hint_target, P.err, lane)) {
            const uint32_t* src = P.layers[P.L - 1].xt;
            const uint32_t tag16 = (epoch * 64u + (uint32_t)(P.L - 1)) & 0xffffu;
            constexpr int NCH = H / 4 / 32;
            uint32_t pend = (1u << NCH) - 1u;
            Poll poll;
            poll.start();
            for (;;) {
                constexpr int BATCH = 8;
#pragma unroll
                for (int m0 = 0; m0 < NCH; m0 += BATCH) {
                    const uint32_t pb = pend;
                    uint4 v[BATCH];
#pragma unroll
                    for (int i = 0; i < BATCH; ++i)
                        if (m0 + i < NCH && (pb >> (m0 + i) & 1u)) v[i] = ld_relaxed_v4(src + 4 * (lane + 32 * (m0 + i)));
#pragma unroll
                    for (int i = 0; i < BATCH; ++i)
                        if (m0 + i < NCH && (pb >> (m0 + i) & 1u) && (v[i].x >> 16) == tag16 &&
                            (v[i].y >> 16) == tag16 && (v[i].z >> 16) == tag16 && (v[i].w >> 16) == tag16)
                            pend &= ~(1u << (m0 + i));
                }
                if (!poll.again(__any_sync(FULL, pend != 0), P.err, lane)) break;
            }
            // the epoch counts launches (mod 2^32): hint targets epoch * G stay consistent with the
            // counters, and a tag epoch * 64 + layer only repeats 2^26 launches later
            if (!__any_sync(FULL, pend != 0) && lane == 0) st_relaxed_u32(P.epoch, epoch + 1u);
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
    const uint64_t pol = evict_first_policy();

    It iss, con;
    it_begin_layer(iss, c, 0);
    it_begin_layer(con, c, 0);
    int n_iss = 0, n_con = 0;  // items issued / consumed by this warp
    bool ok = true;
    float carry0 = 0.0f, carry1 = 0.0f;  // partial results carried between the items of a task
    const float* n_s = reinterpret_cast<const float*>(smem + OFF_N);
    const float* sn_s = reinterpret_cast<const float*>(smem + OFF_SN);
    float r = 0.0f;
    int h_seen = 0;  // layers whose staged h this warp has seen (phases are observed in order)

    // Layers whose top-k this warp has seen published. The routing mbarrier is
    // tested one phase at a time, in order: a parity test of a later phase
    // would succeed before the earlier one completed.
    int k_seen = 0;
    auto topk_known = [&](int lt) -> bool {
        while (k_seen <= lt) {
            int rdy = 0;
            if (lane == 0) rdy = mbar_try_wait(bar_k, k_seen & 1);
            if (!__shfl_sync(FULL, rdy, 0)) return false;
            ++k_seen;
        }
        return true;
    };
    // Fill the ring without blocking: stop at an item whose layer's top-k is not published yet.
    auto try_issue = [&]() {
        while (n_iss < n_con + NS && iss.l < P.L) {
            if (it_needs_topk(iss) && !topk_known(iss.l)) break;
            if (lane == 0) {
                const int slot = n_iss % NS;
                issue_item(c, iss, rt, ring_u32 + slot * STAGE, bar0 + 8 * slot, pol);
            }
            ++n_iss;
            it_next(iss, c);
        }
        __syncwarp();
    };

    if (P.prefetch && lane == 0) prefetch_layer(c, 0);
    for (int l = 0; l < P.L && ok; ++l) {
        const LayerDesc& D = P.layers[l];
        const uint32_t tag = epoch * 64u + (uint32_t)l;
        const uint32_t tag16 = tag & 0xffffu;
        if (P.prefetch && lane == 0) prefetch_layer(c, l + 1 < P.L ? l + 1 : 0);
        try_issue();
        if (!(ok = warp_wait_mbar(bar_x, l & 1, P.err, lane))) break;
        r = reinterpret_cast<const float*>(smem + OFF_MISC)[0];
        const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem + OFF_XS);
        uint16_t* pout = l == P.L - 1 ? P.out : nullptr;
        bool h_ready = false, h_signalled = false;
        while (con.l == l) {
            if (con.kind == T_DOWN && !h_ready) {
                signal_phase(P, l, TR_CTA_H_DONE, &cta_cnt[0], D.cnt_h, lane);
                h_signalled = true;
                try_issue();
                if (!(ok = warp_wait_mbar(bar_h, l & 1, P.err, lane))) break;
                h_seen = l + 1;
                h_ready = true;
            }
            // make sure the item is in flight, then wait for it
            try_issue();
            if (n_iss == n_con) {  // blocked on this layer's top-k
                if (k_seen < con.l) {  // never the case: earlier layers' phases were observed at their end
                    if (lane == 0) atomicOr(P.err, ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                if (!(ok = warp_wait_mbar(bar_k, con.l & 1, P.err, lane))) break;
                k_seen = con.l + 1;
                try_issue();
                if (n_iss == n_con) {
                    if (lane == 0) atomicOr(P.err, ERR_TIMEOUT);
                    ok = false;
                    break;
                }
            }
            const int slot = n_con % NS;
            if (!(ok = warp_wait_mbar(bar0 + 8 * slot, (n_con / NS) & 1, P.err, lane))) break;
            const unsigned char* st = ring + slot * STAGE;
            if (con.kind == T_ROUTER) {
                const uint16_t* wrow = reinterpret_cast<const uint16_t*>(st);
                float d = 0.0f;
#pragma unroll 8
                for (int k = lane; k < H; k += 32) d = fmaf(bf2f(wrow[k]), bf2f(xs[k]), d);  // exact products
                d = warp_sum_canonical(d);
                float z = __fmul_rn(r, d);
                if (D.bias) z = __fadd_rn(z, D.bias[con.t]);
                if (lane == 0) {
                    st_relaxed_u64(D.zt + con.t, tag64(tag, z));
                    red_relaxed_add(D.cnt_z, 1u);
                }
            } else if (con.kind == T_SGU) {
                const float v = row_bf16(st, n_s, lane);
                if (con.sub == 0) {
                    carry0 = v;
                } else if (lane == 0) {
                    st_relaxed_u64(D.ht + K * I + (con.t - D.E), tag64(tag, gelu_tanh(carry0) * v));
                }
            } else if (con.kind == T_RGU) {
                const int u = con.t - D.E - N_SGU;
                const int i = u / RGU_PER_EXPERT, p0 = 2 * (u % RGU_PER_EXPERT);
                const uint32_t* codes = reinterpret_cast<const uint32_t*>(st);
                const uint32_t* sb = reinterpret_cast<const uint32_t*>(st + 4 * GU_ROW);
                const float4 gu = rows4_int4(codes, sb, n_s, sn_s, lane);  // gate p0, up p0, gate p0+1, up p0+1
                if (lane == 0)
                    st_relaxed_v2u64(D.ht + (size_t)i * I + p0, tag64(tag, gelu_tanh(gu.x) * gu.y),
                                     tag64(tag, gelu_tanh(gu.z) * gu.w));
            } else {
                const int j0 = 2 * (con.t - D.E - N_SGU - N_RGU);
                const float* hsh = reinterpret_cast<const float*>(smem + OFF_H) + K * I;
                if (con.sub < 2) {
                    // shared down row j0 + sub (bf16, K = S): chunks ch = lane + 32 t, t < 9
                    unsigned long long ac[2] = {0ull, 0ull};
#pragma unroll
                    for (int t = 0; t < (S / 8 + 31) / 32; ++t) {
                        const int ch = lane + 32 * t;
                        if (ch < S / 8) {
                            const uint4 v = *reinterpret_cast<const uint4*>(st + 16 * ch);
                            const float4 h0 = *reinterpret_cast<const float4*>(hsh + 8 * ch);
                            const float4 h1 = *reinterpret_cast<const float4*>(hsh + 8 * ch + 4);
                            ac[t & 1] = dot8_bf16_2(v, h0, h1, ac[t & 1]);
                        }
                    }
                    const float acc = warp_sum(sum2(ac[0]) + sum2(ac[1]));
                    if (con.sub == 0) carry0 = acc;
                    else carry1 = acc;
                } else {
                    // the 8 experts' down rows j0, j0 + 1 (int4, K = I), weighted
                    const float* hr = reinterpret_cast<const float*>(smem + OFF_H);
                    const float* sh = reinterpret_cast<const float*>(smem + OFF_SH);
                    float y0 = 0.0f, y1 = 0.0f, z0 = 0.0f, z1 = 0.0f;
                    const int sbrow = j0 & 3;
#pragma unroll
                    for (int i = 0; i < K; ++i) {
                        const uint32_t* codes = reinterpret_cast<const uint32_t*>(st + i * 2 * D_ROW);
                        const uint32_t* sb = reinterpret_cast<const uint32_t*>(st + DN_SB_OFF + i * 4 * D_SB) +
                                             sbrow * (D_SB / 4);
                        const float* hi = hr + i * I;
                        float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
                        for (int t = 0; t < (D_WORDS + 31) / 32; ++t) {
                            const int w = lane + 32 * t;
                            if (w < D_WORDS) {
                                const float4 ha = *reinterpret_cast<const float4*>(hi + 8 * w);
                                const float4 hb = *reinterpret_cast<const float4*>(hi + 8 * w + 4);
                                const float sw = sh[i * D_WORDS + w];
                                p0 = word_affine(codes[w], sb[w >> 3], ha, hb, sw, p0);
                                p1 = word_affine(codes[D_WORDS + w], sb[D_SB / 4 + (w >> 3)], ha, hb, sw, p1);
                            }
                        }
                        const float wi = rt->w[l & 1][i];
                        if (i & 1) {
                            z0 = fmaf(wi, p0, z0);
                            z1 = fmaf(wi, p1, z1);
                        } else {
                            y0 = fmaf(wi, p0, y0);
                            y1 = fmaf(wi, p1, y1);
                        }
                    }
                    y0 += z0;
                    y1 += z1;
                    float dummy0 = 0.0f, dummy1 = 0.0f;
                    warp_sum4(y0, y1, dummy0, dummy1);
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
        if (!h_signalled) signal_phase(P, l, TR_CTA_H_DONE, &cta_cnt[0], D.cnt_h, lane);
        // observe this layer's routing and h phases even without items that needed them,
        // so that later parity tests never run two phases behind
        try_issue();
        if (!topk_known(l)) {
            if (!(ok = warp_wait_mbar(bar_k, l & 1, P.err, lane))) break;
            k_seen = l + 1;
        }
        if (h_seen <= l) {
            if (!(ok = warp_wait_mbar(bar_h, l & 1, P.err, lane))) break;
            h_seen = l + 1;
        }
        signal_phase(P, l, TR_CTA_OUT, &cta_cnt[1], D.cnt_out, lane);
    }

    if (!ok && lane == 0) {
        // let this warp's copies in flight land before the CTA's shared memory goes away
        for (int j = n_con; j < n_iss; ++j) {
            const uint64_t t0 = gtimer();
            while (!mbar_try_wait(bar0 + 8 * (j % NS), (j / NS) & 1))
                if (gtimer() - t0 > TIMEOUT_NS) break;
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
    size_t cnt_z, cnt_h, cnt_out, zt, ht, xt, logits, idx, w, act;
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
    c.cnt_h = p; p += 128;
    c.cnt_out = p; p += 128;
    c.zt = p; p += align_up((size_t)E * 8, 128);
    c.ht = p; p += align_up((size_t)fused::H_FLOATS * 8, 128);
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
    if (L < 1 || E < fused::K || E > TF_MAX_E) return 0;
    return stack_carve(L, E).total;
}

tf_status tf_stack_create(tf_layer* const* layers, int L, const float* const* logit_bias, void* workspace,
                          size_t ws_bytes, tf_stack** out) {
    const char* fn = "tf_stack_create";
    if (!out) return fail(TF_ERR_INVALID_ARG, "%s: out is NULL", fn);
    *out = nullptr;
    if (!layers || L < 1) return fail(TF_ERR_INVALID_ARG, "%s: no layers", fn);
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
        D.cnt_h = reinterpret_cast<uint32_t*>(base + sc.cnt_h);
        D.cnt_out = reinterpret_cast<uint32_t*>(base + sc.cnt_out);
        D.zt = reinterpret_cast<unsigned long long*>(base + sc.zt);
        D.ht = reinterpret_cast<unsigned long long*>(base + sc.ht);
        D.xt = reinterpret_cast<uint32_t*>(base + sc.xt);
        D.logits = reinterpret_cast<float*>(base + sc.logits);
        D.idx = reinterpret_cast<int32_t*>(base + sc.idx);
        D.w = reinterpret_cast<float*>(base + sc.w);
        D.act_out = reinterpret_cast<uint16_t*>(base + sc.act);
        D.E = E;
        D.eps = d.eps;
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
    const size_t need = (size_t)s->L * fused::TRACE_CTAS * fused::TRACE_SLOTS * 8;
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
