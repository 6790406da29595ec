// Fused persistent decode kernel: a whole stack of MoE layers for one token in
// one cooperative launch (one CTA per SM).
//
// The per-layer flow is the pages' (page "Como executar um modelo de 26 bilhoes
// de parametros em dois gigabytes de memoria em um Mac comum", section "Qual e
// o principal truque da arquitetura"): router -> top-8 -> expert FFNs, with the
// shared-expert branch beside them. What differs is how it is fed on B300: the
// weights of every layer are a fixed byte stream (router rows, shared gate/up,
// the selected experts' gate/up, then all down projections). One producer
// thread per CTA streams its share of that stream into a ring of shared-memory
// stages with cp.async.bulk (L2 evict-first, completion on mbarriers) and only
// ever waits for the top-8 ids of the current layer; eleven consumer warps
// compute from shared memory. Data dependencies between CTAs (routing ready,
// all h ready, layer output ready) are global counters with bounded waits, so
// the HBM stream keeps running while consumers wait.
//
// Work units per layer (static round-robin over CTAs, continuing across layers):
//   router : 4 rows of W_r (bf16), fixed-order dot products; the CTA that
//            completes the last row runs top-8 + softmax and raises the flag
//   sgu    : 2 row pairs of the shared gate/up (bf16) -> h_shared
//   rgu    : 8 row pairs of one selected expert's gate/up (int4) -> h_routed
//   down   : 4 output rows: shared down (bf16) + the 8 experts' down (int4),
//            weighted combine, residual add, bf16 output
#include <cooperative_groups.h>
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
constexpr int NC = 352;                    // consumer threads (11 warps)
constexpr int NT = NC + 32;                // + producer warp
constexpr int HC = H / 32;                 // 88 column chunks of a K = H row
constexpr int NS = 6;                      // ring stages
constexpr int STAGE = 30720;               // bytes per stage
constexpr int ROW_BF = H * 2;              // 5632: bf16 row of K = H
constexpr int SROW_BF = S * 2;             // 4224: bf16 row of K = S
constexpr int GU_CODE_ROW = H / 2;         // 1408
constexpr int GU_SB_ROW = (H / 64) * 4;    // 176
constexpr int D_CODE_ROW = I / 2;          // 352
constexpr int D_SB_ROW = (I / 64) * 4;     // 44
constexpr int N_SGU = S / 2;               // 1056 units of 2 shared row pairs
constexpr int N_RGU = K * I / 8;           // 704 units of 8 routed row pairs
constexpr int N_DN = H / 4;                // 704 units of 4 output rows
constexpr int RGU_PER_EXPERT = I / 8;      // 88
constexpr int RGU_SB_OFF = 16 * GU_CODE_ROW;           // 22528
constexpr int DN_CODE_OFF = 4 * SROW_BF;                // 16896
constexpr int DN_SB_OFF = DN_CODE_OFF + K * 4 * D_CODE_ROW;  // 28160
constexpr int RED_FLOATS = 4 * 88 + 4 * NC;             // 1760
constexpr unsigned long long TIMEOUT_NS = 2000000000ull;  // 2 s per wait
static_assert(NC == H / 8, "x is staged with one 16-byte load per consumer thread");
static_assert(NC == 4 * HC && NC == K * (I / 16) && NC == 4 * (S / 24), "thread roles");
static_assert(DN_SB_OFF + K * 4 * D_SB_ROW <= STAGE && RGU_SB_OFF + 16 * GU_SB_ROW <= STAGE, "stage size");

enum { SYNC_ROUTER = 0, SYNC_TOPK = 1, SYNC_H = 2, SYNC_OUT = 3, SYNC_WORDS = 32 };

struct LayerDesc {
    const uint16_t* Wr;
    const uint16_t* Wsg;
    const uint16_t* Wsu;
    const uint16_t* Wsd;
    const char* ebase;
    unsigned long long estride;
    const int32_t* slot_map;
    const float* bias;
    float* logits;
    int32_t* idx;
    float* w;
    float* h_routed;
    float* h_shared;
    uint16_t* act_out;   // this layer's output (the last layer writes the call's `out`)
    uint32_t* sync;      // SYNC_WORDS words (one 128-byte line)
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
};

enum { U_ROUTER = 0, U_SGU = 1, U_RGU = 2, U_DOWN = 3 };
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
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}
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
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"r"(NC) : "memory"); }

// Consumer barrier that also ANDs a flag over the consumer threads, so that a
// failed bounded wait in any thread makes all of them leave together.
__device__ __forceinline__ bool consumer_all(bool v) {
    int r;
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.s32 p, %1, 0;\n bar.red.and.pred p, 1, %2, p;\n selp.s32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((int)v), "r"(NC)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ bool err_set(const uint32_t* err) { return *(volatile const uint32_t*)err != 0; }

// Bounded wait on an mbarrier phase; false (error recorded) on timeout or when another CTA failed.
__device__ bool wait_mbar(uint32_t bar, uint32_t parity, uint32_t* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 255u) == 0) {
            if (err_set(err)) return false;
            if (gtimer() - t0 > TIMEOUT_NS) {
                atomicOr(err, ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait until *p >= target (acquire).
__device__ bool wait_ge(const uint32_t* p, uint32_t target, uint32_t* err) {
    if (ld_acquire(p) >= target) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t n = 1;; ++n) {
        if (ld_acquire(p) >= target) return true;
        __nanosleep(64);
        if ((n & 63u) == 0) {
            if (err_set(err)) return false;
            if (gtimer() - t0 > TIMEOUT_NS) {
                atomicOr(err, ERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ int units_per_layer(int E) { return (E + 3) / 4 + N_SGU + N_RGU + N_DN; }

// First unit of layer l owned by CTA c: units are dealt round-robin over the
// grid, continuing from layer to layer.
__device__ __forceinline__ int first_unit(int c, int l, int NU, int G) {
    const long long base = ((long long)l * NU) % G;
    return (int)((c - base + G) % G);
}

__device__ __forceinline__ int unit_kind(int g, int NR, int* u) {
    if (g < NR) { *u = g; return U_ROUTER; }
    g -= NR;
    if (g < N_SGU) { *u = g; return U_SGU; }
    g -= N_SGU;
    if (g < N_RGU) { *u = g; return U_RGU; }
    *u = g - N_RGU;
    return U_DOWN;
}

// ------------------------------------------------------------------ producer

__device__ void producer(const Params& P, unsigned char* ring, uint64_t* full, uint64_t* empty) {
    const uint64_t pol = evict_first_policy();
    const int c = blockIdx.x, G = gridDim.x;
    int it = 0;
    for (int l = 0; l < P.L; ++l) {
        const LayerDesc& D = P.layers[l];
        const int E = D.E, NR = (E + 3) / 4, NU = units_per_layer(E);
        const char* eptr[K];
        bool have_idx = false;
        for (int g = first_unit(c, l, NU, G); g < NU; g += G) {
            int u;
            const int kind = unit_kind(g, NR, &u);
            if (kind >= U_RGU && !have_idx) {
                if (!wait_ge(D.sync + SYNC_TOPK, 1, P.err)) goto bail;
                bool bad = false;
#pragma unroll
                for (int i = 0; i < K; ++i) {
                    int e = __ldcg(D.idx + i);
                    bad |= (unsigned)e >= (unsigned)E;
                    e = bad ? 0 : e;
                    if (D.slot_map) e = __ldcg(D.slot_map + e);
                    eptr[i] = D.ebase + (size_t)e * D.estride;
                }
                if (bad) {   // never form an address from an out-of-range id
                    atomicOr(P.err, ERR_BAD_ID);
                    goto bail;
                }
                have_idx = true;
            }
            const int slot = it % NS;
            if (!wait_mbar(smem_u32(&empty[slot]), ((it / NS) & 1) ^ 1, P.err)) goto bail;
            const uint32_t dst = smem_u32(ring + (size_t)slot * STAGE);
            const uint32_t fb = smem_u32(&full[slot]);
            if (kind == U_ROUTER) {
                const int nr = min(4, E - 4 * u);
                mbar_expect_tx(fb, nr * ROW_BF);
                bulk_g2s(dst, D.Wr + (size_t)4 * u * H, nr * ROW_BF, fb, pol);
            } else if (kind == U_SGU) {
                mbar_expect_tx(fb, 4 * ROW_BF);
                bulk_g2s(dst, D.Wsg + (size_t)2 * u * H, 2 * ROW_BF, fb, pol);
                bulk_g2s(dst + 2 * ROW_BF, D.Wsu + (size_t)2 * u * H, 2 * ROW_BF, fb, pol);
            } else if (kind == U_RGU) {
                const int i = u / RGU_PER_EXPERT, p0 = 8 * (u % RGU_PER_EXPERT);
                mbar_expect_tx(fb, 16 * (GU_CODE_ROW + GU_SB_ROW));
                bulk_g2s(dst, eptr[i] + (size_t)2 * p0 * GU_CODE_ROW, 16 * GU_CODE_ROW, fb, pol);
                bulk_g2s(dst + RGU_SB_OFF, eptr[i] + D.off_gu_sb + (size_t)2 * p0 * GU_SB_ROW, 16 * GU_SB_ROW, fb,
                         pol);
            } else {
                const int j0 = 4 * u;
                mbar_expect_tx(fb, 4 * SROW_BF + K * 4 * (D_CODE_ROW + D_SB_ROW));
                bulk_g2s(dst, D.Wsd + (size_t)j0 * S, 4 * SROW_BF, fb, pol);
#pragma unroll
                for (int i = 0; i < K; ++i) {
                    bulk_g2s(dst + DN_CODE_OFF + i * 4 * D_CODE_ROW, eptr[i] + D.off_d_codes + (size_t)j0 * D_CODE_ROW,
                             4 * D_CODE_ROW, fb, pol);
                    bulk_g2s(dst + DN_SB_OFF + i * 4 * D_SB_ROW, eptr[i] + D.off_d_sb + (size_t)j0 * D_SB_ROW,
                             4 * D_SB_ROW, fb, pol);
                }
            }
            ++it;
        }
    }
    return;
bail:
    // let copies already in flight land before the CTA's shared memory goes away
    for (int j = it - NS; j < it; ++j) {
        if (j < 0) continue;
        const uint64_t t0 = gtimer();
        while (!mbar_try_wait(smem_u32(&full[j % NS]), (j / NS) & 1))
            if (gtimer() - t0 > TIMEOUT_NS) break;
    }
}

// ------------------------------------------------------------------ consumers

struct Regs {
    float4 nc[8];   // n at k = 32c .. 32c+31 (int4 gate/up chunks)
    float4 n2[8];   // n at k = 8c + 704q + j, q < 4 (bf16 shared gate/up)
    float Sc;       // sum of nc
    float4 hs[6];   // h_shared at k = 8c + 704q + j, q < 3 (shared down)
    float4 hr[4];   // h_routed[i2] at k = 16c16 .. 16c16+15 (routed down)
    float Sr;       // sum of hr
    float wi;       // routing weight of expert i2
};

__device__ __forceinline__ float sum4(float4 a) { return ((a.x + a.y) + a.z) + a.w; }

__device__ void consumer(const Params& P, unsigned char* ring, uint64_t* full, uint64_t* empty, uint16_t* sx,
                         float* red, float* tot, float* s_r, int* s_flag) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = tid % HC, s4 = tid / HC;          // gate/up and shared-down roles
    const int i2 = tid / (I / 16), c16 = tid % (I / 16);  // routed-down role
    const int cta = blockIdx.x, G = gridDim.x;
    Regs R;
    int it = 0;
    bool ok = true;
    for (int l = 0; l < P.L && ok; ++l) {
        const LayerDesc& D = P.layers[l];
        const int E = D.E, NR = (E + 3) / 4, NU = units_per_layer(E);
        const uint16_t* xin = l == 0 ? P.x : P.layers[l - 1].act_out;
        uint16_t* xout = l == P.L - 1 ? P.out : D.act_out;
        // ---- layer input: wait for every output row of the previous layer
        if (l > 0) {
            if (tid == 0) *s_flag = wait_ge(P.layers[l - 1].sync + SYNC_OUT, N_DN, P.err);
            consumer_sync();
            if (!*s_flag) { ok = false; break; }
        }
        reinterpret_cast<uint4*>(sx)[tid] = __ldcg(reinterpret_cast<const uint4*>(xin) + tid);
        consumer_sync();
        if (warp == 0) {
            float p = 0.0f;
#pragma unroll 8
            for (int kk = lane; kk < H; kk += 32) {
                const float v = bf2f(sx[kk]);
                p = fmaf(v, v, p);
            }
            p = warp_sum_canonical(p);
            if (lane == 0) *s_r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(p, (float)H), D.eps)));
        }
        consumer_sync();
        const float r = *s_r;
        {
            const uint4* xs = reinterpret_cast<const uint4*>(sx);
            float Sc = 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 v = xs[4 * c + q];
                R.nc[2 * q] = make_float4(__fmul_rn(r, bf_lo(v.x)), __fmul_rn(r, bf_hi(v.x)), __fmul_rn(r, bf_lo(v.y)),
                                          __fmul_rn(r, bf_hi(v.y)));
                R.nc[2 * q + 1] = make_float4(__fmul_rn(r, bf_lo(v.z)), __fmul_rn(r, bf_hi(v.z)),
                                              __fmul_rn(r, bf_lo(v.w)), __fmul_rn(r, bf_hi(v.w)));
                Sc += sum4(R.nc[2 * q]) + sum4(R.nc[2 * q + 1]);
                const uint4 v2 = xs[c + 88 * q];
                R.n2[2 * q] = make_float4(__fmul_rn(r, bf_lo(v2.x)), __fmul_rn(r, bf_hi(v2.x)),
                                          __fmul_rn(r, bf_lo(v2.y)), __fmul_rn(r, bf_hi(v2.y)));
                R.n2[2 * q + 1] = make_float4(__fmul_rn(r, bf_lo(v2.z)), __fmul_rn(r, bf_hi(v2.z)),
                                              __fmul_rn(r, bf_lo(v2.w)), __fmul_rn(r, bf_hi(v2.w)));
            }
            R.Sc = Sc;
        }
        bool h_loaded = false;
        for (int g = first_unit(cta, l, NU, G); g < NU; g += G) {
            int u;
            const int kind = unit_kind(g, NR, &u);
            const int slot = it % NS;
            const bool got = wait_mbar(smem_u32(&full[slot]), (it / NS) & 1, P.err);
            if (!consumer_all(got)) { ok = false; break; }
            const unsigned char* st = ring + (size_t)slot * STAGE;
            ++it;
            if (kind == U_ROUTER) {
                const int nr = min(4, E - 4 * u);
                if (warp < nr) {
                    const uint16_t* wrow = reinterpret_cast<const uint16_t*>(st + warp * ROW_BF);
                    float d = 0.0f;
#pragma unroll 8
                    for (int kk = lane; kk < H; kk += 32) d = fmaf(bf2f(wrow[kk]), bf2f(sx[kk]), d);
                    d = warp_sum_canonical(d);
                    const int e = 4 * u + warp;
                    float z = __fmul_rn(r, d);
                    if (D.bias) z = __fadd_rn(z, D.bias[e]);
                    if (lane == 0) {
                        D.logits[e] = z;
                        __threadfence();
                    }
                }
                consumer_sync();
                if (tid == 0) {
                    mbar_arrive(smem_u32(&empty[slot]));
                    const uint32_t ticket = atomicAdd(D.sync + SYNC_ROUTER, (uint32_t)nr);
                    *s_flag = (ticket + (uint32_t)nr == (uint32_t)E);
                }
                consumer_sync();
                if (*s_flag) {  // this CTA scored the last router rows: top-k for the layer
                    __threadfence();
                    float* zs = red;
                    unsigned char* taken = reinterpret_cast<unsigned char*>(red + 1024);
                    for (int j = tid; j < E; j += NC) {
                        zs[j] = __ldcg(D.logits + j);
                        taken[j] = 0;
                    }
                    consumer_sync();
                    if (warp == 0) {
                        warp_topk_softmax(zs, taken, E, K, lane, D.idx, D.w);
                        __threadfence();
                        __syncwarp();
                        if (lane == 0) st_release(D.sync + SYNC_TOPK, 1);
                    }
                    consumer_sync();
                }
            } else if (kind == U_SGU) {
                // stage rows: gate 2u, gate 2u+1, up 2u, up 2u+1
                const unsigned char* row = st + s4 * ROW_BF;
                float acc = 0.0f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v = *reinterpret_cast<const uint4*>(row + 1408 * q + 16 * c);
                    acc = dot8_bf16(v, R.n2[2 * q], R.n2[2 * q + 1], acc);
                }
                consumer_sync();
                if (tid == 0) mbar_arrive(smem_u32(&empty[slot]));
                red[s4 * HC + c] = acc;
                consumer_sync();
                if (warp < 4) {
                    const float* rr = red + warp * HC;
                    float v = rr[lane] + rr[lane + 32] + (lane < HC - 64 ? rr[lane + 64] : 0.0f);
                    v = warp_sum(v);
                    if (lane == 0) tot[warp] = v;
                }
                consumer_sync();
                if (warp == 0) {
                    if (lane < 2) {
                        D.h_shared[2 * u + lane] = gelu_tanh(tot[lane]) * tot[2 + lane];
                        __threadfence();
                    }
                    __syncwarp();
                    if (lane == 0) red_release_add(D.sync + SYNC_H, 1);
                }
            } else if (kind == U_RGU) {
                const int i = u / RGU_PER_EXPERT, p0 = 8 * (u % RGU_PER_EXPERT);
                float part[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int rw = s4 + 4 * t;
                    const uint4 q = *reinterpret_cast<const uint4*>(st + rw * GU_CODE_ROW + 16 * c);
                    const uint32_t sb =
                        *reinterpret_cast<const uint32_t*>(st + RGU_SB_OFF + rw * GU_SB_ROW + 4 * (c >> 1));
                    float P0 = 0.0f, P1 = 0.0f;
                    P0 = dot8_q128(q.x, R.nc[0], R.nc[1], P0);
                    P1 = dot8_q128(q.y, R.nc[2], R.nc[3], P1);
                    P0 = dot8_q128(q.z, R.nc[4], R.nc[5], P0);
                    P1 = dot8_q128(q.w, R.nc[6], R.nc[7], P1);
                    part[t] = chunk_affine(sb, P0 + P1, R.Sc);
                }
                consumer_sync();
                if (tid == 0) mbar_arrive(smem_u32(&empty[slot]));
#pragma unroll
                for (int t = 0; t < 4; ++t) red[(s4 + 4 * t) * HC + c] = part[t];
                consumer_sync();
                for (int rw = warp; rw < 16; rw += NC / 32) {
                    const float* rr = red + rw * HC;
                    float v = rr[lane] + rr[lane + 32] + (lane < HC - 64 ? rr[lane + 64] : 0.0f);
                    v = warp_sum(v);
                    if (lane == 0) tot[rw] = v;
                }
                consumer_sync();
                if (warp == 0) {
                    if (lane < 8) {
                        D.h_routed[(size_t)i * I + p0 + lane] = gelu_tanh(tot[2 * lane]) * tot[2 * lane + 1];
                        __threadfence();
                    }
                    __syncwarp();
                    if (lane == 0) red_release_add(D.sync + SYNC_H, 1);
                }
            } else {
                if (!h_loaded) {
                    if (tid == 0) *s_flag = wait_ge(D.sync + SYNC_H, N_SGU + N_RGU, P.err);
                    consumer_sync();
                    if (!*s_flag) { ok = false; break; }
#pragma unroll
                    for (int q = 0; q < 3; ++q) {
                        const float4* hsrc = reinterpret_cast<const float4*>(D.h_shared + 8 * c + 704 * q);
                        R.hs[2 * q] = __ldcg(hsrc);
                        R.hs[2 * q + 1] = __ldcg(hsrc + 1);
                    }
                    const float4* hrs = reinterpret_cast<const float4*>(D.h_routed + (size_t)i2 * I + 16 * c16);
                    float Sr = 0.0f;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        R.hr[q] = __ldcg(hrs + q);
                        Sr += sum4(R.hr[q]);
                    }
                    R.Sr = Sr;
                    R.wi = __ldcg(D.w + i2);
                    h_loaded = true;
                }
                const int j0 = 4 * u;
                const unsigned char* srow = st + s4 * SROW_BF;
                float acc1 = 0.0f;
#pragma unroll
                for (int q = 0; q < 3; ++q) {
                    const uint4 v = *reinterpret_cast<const uint4*>(srow + 1408 * q + 16 * c);
                    acc1 = dot8_bf16(v, R.hs[2 * q], R.hs[2 * q + 1], acc1);
                }
                float part[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint2 q = *reinterpret_cast<const uint2*>(st + DN_CODE_OFF + i2 * 4 * D_CODE_ROW +
                                                                    t * D_CODE_ROW + 8 * c16);
                    const uint32_t sb = *reinterpret_cast<const uint32_t*>(st + DN_SB_OFF + i2 * 4 * D_SB_ROW +
                                                                           t * D_SB_ROW + 4 * (c16 >> 2));
                    float P0 = 0.0f;
                    P0 = dot8_q128(q.x, R.hr[0], R.hr[1], P0);
                    P0 = dot8_q128(q.y, R.hr[2], R.hr[3], P0);
                    part[t] = R.wi * chunk_affine(sb, P0, R.Sr);
                }
                consumer_sync();
                if (tid == 0) mbar_arrive(smem_u32(&empty[slot]));
                red[s4 * HC + c] = acc1;
#pragma unroll
                for (int t = 0; t < 4; ++t) red[4 * HC + t * NC + tid] = part[t];
                consumer_sync();
                if (warp < 4) {
                    const float* r1 = red + warp * HC;
                    const float* r2 = red + 4 * HC + warp * NC;
                    float v = r1[lane] + r1[lane + 32] + (lane < HC - 64 ? r1[lane + 64] : 0.0f);
#pragma unroll
                    for (int m = 0; m < NC / 32; ++m) v += r2[lane + 32 * m];
                    v = warp_sum(v);
                    if (lane == 0) tot[warp] = v;
                }
                consumer_sync();
                if (warp == 0) {
                    if (lane < 4) {
                        xout[j0 + lane] = f2bf(bf2f(sx[j0 + lane]) + tot[lane]);
                        __threadfence();
                    }
                    __syncwarp();
                    if (lane == 0) red_release_add(D.sync + SYNC_OUT, 1);
                }
            }
        }
    }
    // CTA 0 returns the sync words to zero once the last layer is complete
    if (ok && cta == 0 && tid == 0) {
        if (wait_ge(P.layers[P.L - 1].sync + SYNC_OUT, N_DN, P.err)) {
            for (int l = 0; l < P.L; ++l)
                for (int s = 0; s < 4; ++s) P.layers[l].sync[s] = 0;
            __threadfence();
        }
    }
}

__global__ void __launch_bounds__(NT, 1) k_fused_stack(Params P) {
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * STAGE);
    uint64_t* empty = full + NS;
    uint16_t* sx = reinterpret_cast<uint16_t*>(empty + NS);
    float* red = reinterpret_cast<float*>(sx + H);
    float* tot = red + RED_FLOATS;
    __shared__ float s_r;
    __shared__ int s_flag;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= NC) {
        if (threadIdx.x == NC) producer(P, ring, full, empty);
        return;
    }
    consumer(P, ring, full, empty, sx, red, tot, &s_r, &s_flag);
}

constexpr size_t SMEM_BYTES = (size_t)NS * STAGE + 2 * NS * 8 + H * 2 + (RED_FLOATS + 16) * 4;

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
    std::vector<fused::LayerDesc> layers;   // host copy (pointers into ws)
    size_t sync_off = 0, sync_bytes = 0;
    int grid = 0;
};

namespace {

struct StackCarve {
    size_t err, descs, per_layer, total;
    size_t logits, idx, w, h_routed, h_shared, act, sync;
};

StackCarve stack_carve(int L, int E) {
    StackCarve c;
    size_t o = 0;
    c.err = o; o += 256;
    c.descs = o; o += align_up((size_t)L * sizeof(fused::LayerDesc), 256);
    // per-layer block
    size_t p = 0;
    c.sync = p; p += 128;
    c.logits = p; p += align_up((size_t)E * 4, 128);
    c.idx = p; p += 128;
    c.w = p; p += 128;
    c.h_routed = p; p += align_up((size_t)fused::K * fused::I * 4, 128);
    c.h_shared = p; p += align_up((size_t)fused::S * 4, 128);
    c.act = p; p += align_up((size_t)fused::H * 2, 128);
    c.per_layer = align_up(p, 256);
    c.total = o + (size_t)L * c.per_layer;
    return c;
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
    s->d_layers = reinterpret_cast<fused::LayerDesc*>(s->ws + sc.descs);
    s->grid = sms;
    ExpertLayout lay;
    expert_layout(fused::H, fused::I, &lay);
    s->layers.resize((size_t)L);
    for (int l = 0; l < L; ++l) {
        char* base = s->ws + sc.descs + align_up((size_t)L * sizeof(fused::LayerDesc), 256) + (size_t)l * sc.per_layer;
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
        D.sync = reinterpret_cast<uint32_t*>(base + sc.sync);
        D.logits = reinterpret_cast<float*>(base + sc.logits);
        D.idx = reinterpret_cast<int32_t*>(base + sc.idx);
        D.w = reinterpret_cast<float*>(base + sc.w);
        D.h_routed = reinterpret_cast<float*>(base + sc.h_routed);
        D.h_shared = reinterpret_cast<float*>(base + sc.h_shared);
        D.act_out = reinterpret_cast<uint16_t*>(base + sc.act);
        D.E = E;
        D.eps = d.eps;
        D.off_gu_sb = lay.gu_sb;
        D.off_d_codes = lay.d_codes;
        D.off_d_sb = lay.d_sb;
    }
    e = cudaMemset(s->ws, 0, sc.total);
    if (e == cudaSuccess)
        e = cudaMemcpy(s->d_layers, s->layers.data(), (size_t)L * sizeof(fused::LayerDesc), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        delete s;
        return cuda_status(e, fn);
    }
    *out = s;
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
        // a bounded wait gave up: return the sync words and the error word to zero
        for (int l = 0; l < s->L; ++l) cudaMemsetAsync(s->layers[l].sync, 0, 128, st);
        cudaMemsetAsync(s->err, 0, 4, st);
        cudaStreamSynchronize(st);
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
