// Decode-path kernels of the streamed-expert MoE layer (sm_103a):
//   k_router_topk : RMS scale, router GEMV (one warp per expert row), top-k and
//                   routing weights by the last CTA to finish a token;
//   k_gateup      : fused int4 dequant-GEMV of the gate and up rows of the
//                   selected experts (and the bf16 shared-expert rows) with the
//                   GELU gate applied in registers;
//   k_down        : int4 down projection of the selected experts plus the bf16
//                   shared down projection, weighted combine into the residual.
//
// Page "Como executar um modelo de 26 bilhoes de parametros em dois gigabytes de
// memoria em um Mac comum", sections "Qual e o principal truque da arquitetura"
// (router -> 8 experts, shared branch) and "Sem dependencias do llama.cpp e MLX"
// (hand-written RMSNorm, GEMV, quantisation and MoE kernels).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tf_device.cuh"
#include "tf_internal.h"

namespace tf {

namespace {

using namespace dev;

// ------------------------------------------------------------------- router

constexpr int RT_WARPS = 8;

__global__ void __launch_bounds__(RT_WARPS * 32)
k_router_topk(const uint16_t* __restrict__ x, int H, const uint16_t* __restrict__ Wr, int E,
              const float* __restrict__ bias, int bias_stride, int k, int32_t* __restrict__ idx,
              float* __restrict__ wout, float* __restrict__ logits, float* __restrict__ rms,
              uint32_t* __restrict__ counters, float eps) {
    // shared: x [H] then one W_r row [H] per warp (bf16), staged with 16-byte loads
    extern __shared__ float4 rsm4[];
    uint16_t* sx = reinterpret_cast<uint16_t*>(rsm4);
    const int t = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint16_t* sw = sx + (size_t)(warp + 1) * H;
    const int nvec = H / 8;
    const int e = blockIdx.x * RT_WARPS + warp;
    {
        const uint4* gx = reinterpret_cast<const uint4*>(x + (size_t)t * H);
        uint4* dx = reinterpret_cast<uint4*>(sx);
#pragma unroll 4
        for (int v = threadIdx.x; v < nvec; v += blockDim.x) dx[v] = __ldg(gx + v);
        if (e < E) {
            const char* gw = reinterpret_cast<const char*>(Wr + (size_t)e * H);
            uint4* dw = reinterpret_cast<uint4*>(sw);
#pragma unroll 4
            for (int v = lane; v < nvec; v += 32) dw[v] = ldg_stream(gw + 16 * (size_t)v);
        }
    }
    __syncthreads();
    // r in the canonical order (every warp computes the same value)
    float p = 0.0f;
#pragma unroll 8
    for (int kk = lane; kk < H; kk += 32) {
        const float v = bf2f(sx[kk]);
        p = fmaf(v, v, p);  // exact square, one rounding per term
    }
    p = warp_sum_canonical(p);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(p, (float)H), eps)));
    if (e < E) {
        float d = 0.0f;
#pragma unroll 8
        for (int kk = lane; kk < H; kk += 32) d = fmaf(bf2f(sw[kk]), bf2f(sx[kk]), d);  // exact products
        d = warp_sum_canonical(d);
        float z = __fmul_rn(r, d);
        if (bias) z = __fadd_rn(z, bias[(size_t)t * bias_stride + e]);
        if (lane == 0) {
            logits[(size_t)t * E + e] = z;
            __threadfence();  // publish before this CTA's arrival is counted
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && rms) rms[t] = r;

    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t ticket = atomicAdd(&counters[t], 1u);
        s_last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // Last CTA of token t: top-k over all E logits, then softmax over the k.
    __shared__ float s_z[TF_MAX_E];
    __shared__ unsigned char s_taken[TF_MAX_E];
    for (int j = threadIdx.x; j < E; j += blockDim.x) {
        s_z[j] = __ldcg(logits + (size_t)t * E + j);
        s_taken[j] = 0;
    }
    __syncthreads();
    if (warp == 0) {
        warp_topk_softmax(s_z, s_taken, E, k, lane, idx + (size_t)t * k, wout + (size_t)t * k);
        if (lane == 0) counters[t] = 0;  // leave the workspace zeroed for the next call
    }
}

// ----------------------------------------------------- router for many tokens
//
// The same logits as k_router_topk, computed for a run of tokens against a
// block of EW experts whose rows are held in shared memory as fp32 (converted
// once per CTA, reused by every token of the CTA). The fixed summation order is
// kept exactly: the canonical sum has 32 partials, partial p summing the terms
// k = p, p + 32, p + 64, ... in increasing k, then a xor butterfly 16, 8, 4, 2,
// 1. Here lane p of a warp owns partial p (so a warp reads 32 consecutive
// values of x and of each W_r row per step: coalesced, no bank conflicts) of
// TT tokens x EW experts at a time (each W_r value read from shared memory
// serves TT tokens), and the butterfly runs across the lanes.
// Products of two bf16 values are exact in fp32, so each fused multiply-add
// rounds once, as in the canonical sum; fp32 addition is commutative, so every
// lane ends with the canonical value.

constexpr int RL_THREADS = 256;
constexpr int RL_WARPS = RL_THREADS / 32;
constexpr int RL_SMEM_MAX = 227 * 1024;   // the expert block of W_r as fp32 (EW * H * 4 bytes) fits this
constexpr int RL_WLOADS = 6;              // loads of W_r in flight per thread while the block is filled

__device__ __forceinline__ float lane_butterfly(float v) {
#pragma unroll
    for (int d = 16; d; d >>= 1) v = __fadd_rn(v, __shfl_xor_sync(FULL, v, d));
    return v;
}

template <int EW, int TT, int AHEAD = 8>   // AHEAD: steps of x loaded ahead of their products
__global__ void __launch_bounds__(RL_THREADS)
k_router_lanes(const uint16_t* __restrict__ x, int T, int H, const uint16_t* __restrict__ Wr, int E,
               const float* __restrict__ bias, int bias_stride, float* __restrict__ logits,
               float* __restrict__ rms, float eps, int tokens_per_cta) {
    dev::pdl_wait();
    dev::pdl_trigger();
    extern __shared__ float4 rl4[];
    float* wsm = reinterpret_cast<float*>(rl4);   // [EW][H] fp32
    const int e0 = blockIdx.x * EW;
    const int nv = H / 8;
    // the block's rows, RL_WLOADS 16-byte loads in flight per thread before their conversions
    for (int v0 = threadIdx.x; v0 < EW * nv; v0 += RL_WLOADS * RL_THREADS) {
        uint4 wv[RL_WLOADS];
#pragma unroll
        for (int u = 0; u < RL_WLOADS; ++u) {
            const int v = v0 + u * RL_THREADS, e = v / nv, c = v - e * nv;
            wv[u] = v < EW * nv && e0 + e < E ? __ldg(reinterpret_cast<const uint4*>(Wr + (size_t)(e0 + e) * H) + c)
                                              : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < RL_WLOADS; ++u) {
            const int v = v0 + u * RL_THREADS, e = v / nv, c = v - e * nv;
            if (v < EW * nv) {
                float4* d = reinterpret_cast<float4*>(wsm + (size_t)e * H + 8 * c);
                d[0] = make_float4(bf_lo(wv[u].x), bf_hi(wv[u].x), bf_lo(wv[u].y), bf_hi(wv[u].y));
                d[1] = make_float4(bf_lo(wv[u].z), bf_hi(wv[u].z), bf_lo(wv[u].w), bf_hi(wv[u].w));
            }
        }
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.y * tokens_per_cta;
    const int t1 = min(T, t0 + tokens_per_cta);
    const int nj = H / 32;
    for (int tb = t0 + warp * TT; tb < t1; tb += RL_WARPS * TT) {
        const uint16_t* xr[TT];
#pragma unroll
        for (int i = 0; i < TT; ++i) xr[i] = x + (size_t)(tb + i < t1 ? tb + i : tb) * H + lane;
        float acc[TT][EW], sq[TT];
#pragma unroll
        for (int i = 0; i < TT; ++i) {
            sq[i] = 0.0f;
#pragma unroll
            for (int e = 0; e < EW; ++e) acc[i][e] = 0.0f;
        }
        for (int j0 = 0; j0 < nj; j0 += AHEAD) {
            float xv[AHEAD][TT];
#pragma unroll
            for (int a = 0; a < AHEAD; ++a)
#pragma unroll
                for (int i = 0; i < TT; ++i)
                    xv[a][i] = j0 + a < nj ? __uint_as_float((uint32_t)__ldg(xr[i] + 32 * (j0 + a)) << 16) : 0.0f;
#pragma unroll
            for (int a = 0; a < AHEAD; ++a) {
                if (j0 + a < nj) {   // partial `lane`, term k = 32 (j0 + a) + lane: increasing k
                    const float* wk = wsm + 32 * (j0 + a) + lane;
#pragma unroll
                    for (int i = 0; i < TT; ++i) sq[i] = __fmaf_rn(xv[a][i], xv[a][i], sq[i]);
#pragma unroll
                    for (int e = 0; e < EW; ++e) {
                        const float w = wk[(size_t)e * H];
#pragma unroll
                        for (int i = 0; i < TT; ++i) acc[i][e] = __fmaf_rn(w, xv[a][i], acc[i][e]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < TT; ++i) {
            const int t = tb + i;
            const float ss = lane_butterfly(sq[i]);
            const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), eps)));
            float mine = 0.0f;
#pragma unroll
            for (int e = 0; e < EW; ++e) {
                const float d = lane_butterfly(acc[i][e]);
                if (lane == e) mine = d;
            }
            const int ge = e0 + lane;
            if (t < t1 && lane < EW && ge < E) {
                float z = __fmul_rn(r, mine);
                if (bias) z = __fadd_rn(z, bias[(size_t)t * bias_stride + ge]);
                logits[(size_t)t * E + ge] = z;
            }
            if (t < t1 && lane == 0 && blockIdx.x == 0 && rms) rms[t] = r;
        }
    }
}

// One warp per token: top-k of its logits and the softmax over the selected ones.
__global__ void __launch_bounds__(256) k_topk_rows(const float* __restrict__ logits, int T, int E, int k,
                                                   int32_t* __restrict__ idx, float* __restrict__ wout) {
    dev::pdl_wait();
    dev::pdl_trigger();
    extern __shared__ float tks[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* z = tks + (size_t)warp * E;
    unsigned char* taken = reinterpret_cast<unsigned char*>(tks + (size_t)8 * E) + (size_t)warp * E;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    for (int j = lane; j < E; j += 32) {
        z[j] = logits[(size_t)t * E + j];
        taken[j] = 0;
    }
    __syncwarp();
    warp_topk_softmax(z, taken, E, k, lane, idx + (size_t)t * k, wout + (size_t)t * k);
}

// --------------------------------------------------------------- gate / up

constexpr int GU_WARPS = 8;

// Shared-memory prologue: n = r * x (fp32) and the 32-column chunk sums of n.
__device__ __forceinline__ void load_normalised(const DecodeParams& p, float* n, float* csum) {
    __shared__ float s_r;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        const float r = p.rms_in ? p.rms_in[0] : rms_scale_warp(p.x, p.H, p.eps, lane);
        if (lane == 0) s_r = r;
    }
    __syncthreads();
    const float r = s_r;
    const uint4* gx = reinterpret_cast<const uint4*>(p.x);
#pragma unroll 2
    for (int v = threadIdx.x; v < p.H / 8; v += blockDim.x) {
        const uint4 xv = __ldg(gx + v);
        float4* d = reinterpret_cast<float4*>(n + 8 * v);
        d[0] = make_float4(__fmul_rn(r, bf_lo(xv.x)), __fmul_rn(r, bf_hi(xv.x)), __fmul_rn(r, bf_lo(xv.y)),
                           __fmul_rn(r, bf_hi(xv.y)));
        d[1] = make_float4(__fmul_rn(r, bf_lo(xv.z)), __fmul_rn(r, bf_hi(xv.z)), __fmul_rn(r, bf_lo(xv.w)),
                           __fmul_rn(r, bf_hi(xv.w)));
    }
    __syncthreads();
    for (int c = threadIdx.x; c < p.H / 32; c += blockDim.x) {
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) s += n[32 * c + j];
        csum[c] = s;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(GU_WARPS * 32) k_gateup(DecodeParams p, int u0, int u1) {
    extern __shared__ float4 smem4[];
    float* n = reinterpret_cast<float*>(smem4);
    float* csum = n + p.H;
    load_normalised(p, n, csum);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H, I = p.I;
    const int nchunk = H / 32;     // 16-byte code chunks per row (32 codes)
    const int routed_units = p.k * I;
    const float4* n4 = reinterpret_cast<const float4*>(n);
    for (int u = u0 + blockIdx.x * GU_WARPS + warp; u < u1; u += gridDim.x * GU_WARPS) {
        float ag = 0.0f, au = 0.0f;
        float* dst;
        if (u < routed_units) {
            const int i = u / I, j = u - (u / I) * I;
            const char* blob = expert_ptr(p.ex, i);
            dst = p.h_routed + (size_t)i * I + j;
            if (!blob) {  // out-of-range expert id: no load, the output becomes NaN
                if (lane == 0) *dst = qnan();
                continue;
            }
            const char* gq = blob + (size_t)(2 * j) * (H / 2);
            const char* uq = gq + H / 2;
            const uint32_t* gsb = reinterpret_cast<const uint32_t*>(blob + p.off_gu_sb + (size_t)(2 * j) * (H / 64) * 4);
            const uint32_t* usb = gsb + H / 64;
            for (int c0 = 0; c0 < nchunk; c0 += 96) {   // up to 3 chunks per lane, loads issued first
                uint4 qg[3], qu[3];
                uint32_t sbg[3], sbu[3];
#pragma unroll
                for (int t = 0; t < 3; ++t) {
                    const int c = c0 + lane + 32 * t;
                    if (c < nchunk) {
                        qg[t] = ldg_stream(gq + 16 * c);
                        qu[t] = ldg_stream(uq + 16 * c);
                        sbg[t] = __ldg(gsb + (c >> 1));
                        sbu[t] = __ldg(usb + (c >> 1));
                    }
                }
#pragma unroll
                for (int t = 0; t < 3; ++t) {
                    const int c = c0 + lane + 32 * t;
                    if (c < nchunk) {
                        const float4* nn = n4 + 8 * c;
                        float pg = 0.0f, pu = 0.0f;
                        pg = dot8_q128(qg[t].x, nn[0], nn[1], pg);
                        pu = dot8_q128(qu[t].x, nn[0], nn[1], pu);
                        pg = dot8_q128(qg[t].y, nn[2], nn[3], pg);
                        pu = dot8_q128(qu[t].y, nn[2], nn[3], pu);
                        pg = dot8_q128(qg[t].z, nn[4], nn[5], pg);
                        pu = dot8_q128(qu[t].z, nn[4], nn[5], pu);
                        pg = dot8_q128(qg[t].w, nn[6], nn[7], pg);
                        pu = dot8_q128(qu[t].w, nn[6], nn[7], pu);
                        const float S = csum[c];
                        ag += chunk_affine(sbg[t], pg, S);
                        au += chunk_affine(sbu[t], pu, S);
                    }
                }
            }
        } else {
            const int j = u - routed_units;
            const char* gw = reinterpret_cast<const char*>(p.Wsg + (size_t)j * H);
            const char* uw = reinterpret_cast<const char*>(p.Wsu + (size_t)j * H);
            const int nv = H / 8;
            for (int c0 = 0; c0 < nv; c0 += 128) {     // up to 4 16-byte chunks per lane per batch
                uint4 a[4], b[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int c = c0 + lane + 32 * t;
                    if (c < nv) {
                        a[t] = ldg_stream(gw + 16 * c);
                        b[t] = ldg_stream(uw + 16 * c);
                    }
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int c = c0 + lane + 32 * t;
                    if (c < nv) {
                        const float4 n0 = n4[2 * c], n1 = n4[2 * c + 1];
                        ag = dot8_bf16(a[t], n0, n1, ag);
                        au = dot8_bf16(b[t], n0, n1, au);
                    }
                }
            }
            dst = p.h_shared + j;
        }
        ag = warp_sum(ag);
        au = warp_sum(au);
        if (lane == 0) *dst = gelu_tanh(ag) * au;
    }
}

// ------------------------------------------------------------------- down

constexpr int DN_WARPS = 8;

// float offset of the shared-expert h in the down kernel's shared memory (multiple of 4)
__host__ __device__ __forceinline__ int down_hs_offset(int kr, int I) { return (kr * I + kr * (I / 32) + 3) & ~3; }

__global__ void __launch_bounds__(DN_WARPS * 32) k_down(DecodeParams p, int with_routed, int with_shared) {
    extern __shared__ float4 smem4[];
    const int H = p.H, I = p.I, k = p.k, S = p.S;
    const int kr = with_routed ? k : 0;
    float* hr = reinterpret_cast<float*>(smem4);     // [kr, I]
    float* hcs = hr + kr * I;                        // [kr, I/32] chunk sums of h
    float* hs = hr + down_hs_offset(kr, I);          // [S], 16-byte aligned for float4 reads
    __shared__ float s_w[TF_MAX_K];
    __shared__ const char* s_ptr[TF_MAX_K];
    {
        const float4* g = reinterpret_cast<const float4*>(p.h_routed);
        float4* d = reinterpret_cast<float4*>(hr);
#pragma unroll 4
        for (int t = threadIdx.x; t < kr * I / 4; t += blockDim.x) d[t] = __ldcg(g + t);
        if (with_shared) {
            const float4* gs = reinterpret_cast<const float4*>(p.h_shared);
            float4* ds = reinterpret_cast<float4*>(hs);
#pragma unroll 4
            for (int t = threadIdx.x; t < S / 4; t += blockDim.x) ds[t] = __ldcg(gs + t);
        }
    }
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    if (threadIdx.x < kr) {
        s_w[threadIdx.x] = p.w[threadIdx.x];
        s_ptr[threadIdx.x] = expert_ptr(p.ex, threadIdx.x);
        if (!s_ptr[threadIdx.x]) s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {  // an out-of-range expert id: no load through it; the outputs become NaN
        for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < H; j += gridDim.x * blockDim.x) {
            p.out[j] = 0x7fc0u;
            if (p.delta) p.delta[j] = qnan();
        }
        return;
    }
    for (int c = threadIdx.x; c < kr * (I / 32); c += blockDim.x) {
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) s += hr[32 * c + j];
        hcs[c] = s;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cpr = I / 32;                  // code chunks per down row
    const int ntask = kr * cpr;
    const float4* hr4 = reinterpret_cast<const float4*>(hr);
    const float4* hs4 = reinterpret_cast<const float4*>(hs);
    for (int j = blockIdx.x * DN_WARPS + warp; j < H; j += gridDim.x * DN_WARPS) {
        float acc = 0.0f, accs = 0.0f;
        for (int t0 = 0; t0 < ntask; t0 += 192) {      // up to 6 chunks per lane, loads first
            uint4 q[6];
            uint32_t sb[6];
#pragma unroll
            for (int u = 0; u < 6; ++u) {
                const int t = t0 + lane + 32 * u;
                if (t < ntask) {
                    const int i = t / cpr, c = t - (t / cpr) * cpr;
                    const char* blob = s_ptr[i];
                    q[u] = ldg_stream(blob + p.off_d_codes + (size_t)j * (I / 2) + 16 * c);
                    sb[u] = __ldg(reinterpret_cast<const uint32_t*>(blob + p.off_d_sb + (size_t)j * (I / 64) * 4) +
                                  (c >> 1));
                }
            }
#pragma unroll
            for (int u = 0; u < 6; ++u) {
                const int t = t0 + lane + 32 * u;
                if (t < ntask) {
                    const int i = t / cpr, c = t - (t / cpr) * cpr;
                    const float4* hh = hr4 + (i * I + 32 * c) / 4;
                    float P = 0.0f;
                    P = dot8_q128(q[u].x, hh[0], hh[1], P);
                    P = dot8_q128(q[u].y, hh[2], hh[3], P);
                    P = dot8_q128(q[u].z, hh[4], hh[5], P);
                    P = dot8_q128(q[u].w, hh[6], hh[7], P);
                    acc = fmaf(s_w[i], chunk_affine(sb[u], P, hcs[i * cpr + c]), acc);
                }
            }
        }
        if (with_shared) {
            const char* dw = reinterpret_cast<const char*>(p.Wsd + (size_t)j * S);
            const int nv = S / 8;
            for (int c0 = 0; c0 < nv; c0 += 288) {
                uint4 a[9];
#pragma unroll
                for (int u = 0; u < 9; ++u) {
                    const int c = c0 + lane + 32 * u;
                    if (c < nv) a[u] = ldg_stream(dw + 16 * c);
                }
#pragma unroll
                for (int u = 0; u < 9; ++u) {
                    const int c = c0 + lane + 32 * u;
                    if (c < nv) accs = dot8_bf16(a[u], hs4[2 * c], hs4[2 * c + 1], accs);
                }
            }
        }
        acc = warp_sum(acc);
        accs = warp_sum(accs);
        if (lane == 0) {
            if (p.ys && !with_routed) {
                p.ys[j] = accs;  // the shared term alone; a routed-only launch adds the rest
            } else {
                const float d = (p.ys ? p.ys[j] : accs) + acc;  // same sum as a launch with both terms
                p.out[j] = f2bf(bf2f(p.x[j]) + d);
                if (p.delta) p.delta[j] = d;
            }
        }
    }
}

// ------------------------------------------------------------------ dequant

__global__ void k_dequant(const char* __restrict__ blob, int H, int I, int matrix, int format, void* out,
                          size_t off_sb, size_t off_codes) {
    // matrix 0/1: [I, H] rows at packed rows 2j+matrix; matrix 2: [H, I]
    const int R = matrix < 2 ? I : H, K = matrix < 2 ? H : I;
    const size_t total = (size_t)R * K;
    for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < total; t += (size_t)gridDim.x * blockDim.x) {
        const size_t j = t / K, kk = t % K;
        const size_t prow = matrix < 2 ? 2 * j + matrix : j;
        const uint8_t byte = (uint8_t)blob[off_codes + prow * (K / 2) + kk / 2];
        const uint32_t q = (kk & 1) ? (byte >> 4) : (byte & 15u);
        const uint32_t sb = *reinterpret_cast<const uint32_t*>(blob + off_sb + (prow * (K / 64) + kk / 64) * 4);
        const float w = __fadd_rn(__fmul_rn(h2f(sb & 0xffffu), (float)q), h2f(sb >> 16));
        if (format == 1) static_cast<uint16_t*>(out)[t] = f2bf(w);
        else if (format == 2) static_cast<uint16_t*>(out)[t] = __half_as_ushort(__float2half_rn(w));
        else static_cast<float*>(out)[t] = w;
    }
}

}  // namespace

static int sm_count();

// Many tokens: the token-tiled logits, then one warp per token for the top-k. A wide expert block (8 rows) for
// large T keeps every SM busy with few W_r conversions; a narrow one (2 rows) spreads small batches over more CTAs.
static int launch_router_many(const uint16_t* x, int T, int H, const uint16_t* Wr, int E, const float* bias,
                              int bias_stride, int k, int32_t* idx, float* w, float* logits, float* rms, float eps,
                              cudaStream_t st) {
    // eight experts per CTA where their rows fit shared memory, else two; a warp takes one token at a time
    // for small batches (more CTAs) and four for large ones (four tokens per load of W_r; eight measured slower)
    const bool ew8 = (size_t)8 * H * 4 <= (size_t)RL_SMEM_MAX;
    const int EW = ew8 ? 8 : 2;
    if ((size_t)EW * H * 4 > (size_t)RL_SMEM_MAX) return (int)cudaErrorInvalidValue;   // H beyond one CTA
    const bool wide = T > 256;
    const int TT = wide ? 4 : 1;
    const int gx = (E + EW - 1) / EW;
    const int step = RL_WARPS * TT;                 // tokens of one pass of the CTA's warps
    const int target = 2 * sm_count();
    int gy = (target + gx - 1) / gx;
    int per = (T + gy - 1) / gy;
    per = (per + step - 1) / step * step;
    gy = (T + per - 1) / per;
    const size_t smem = (size_t)EW * H * 4;
    const void* kern = ew8 ? (wide ? (const void*)k_router_lanes<8, 4> : (const void*)k_router_lanes<8, 1>)
                           : (wide ? (const void*)k_router_lanes<2, 4> : (const void*)k_router_lanes<2, 1>);
    // the limit is raised once to the largest size any call may ask for (a smaller one would refuse later calls)
    if (int e = smem_limit_once(kern, RL_SMEM_MAX)) return e;
    const dim3 grid(gx, gy);
    if (ew8 && wide)
        launch_dependent(k_router_lanes<8, 4>, grid, dim3(RL_THREADS), smem, st, x, T, H, Wr, E, bias, bias_stride, logits, rms,
                         eps, per);
    else if (ew8)
        launch_dependent(k_router_lanes<8, 1>, grid, dim3(RL_THREADS), smem, st, x, T, H, Wr, E, bias, bias_stride, logits, rms,
                         eps, per);
    else if (wide)
        launch_dependent(k_router_lanes<2, 4>, grid, dim3(RL_THREADS), smem, st, x, T, H, Wr, E, bias, bias_stride, logits, rms,
                         eps, per);
    else
        launch_dependent(k_router_lanes<2, 1>, grid, dim3(RL_THREADS), smem, st, x, T, H, Wr, E, bias, bias_stride, logits, rms,
                         eps, per);
    const size_t tk_smem = (size_t)8 * E * 5;   // <= 40 KB for E <= 1024: within the default limit
    launch_dependent(k_topk_rows, dim3((T + 7) / 8), dim3(256), tk_smem, st, logits, T, E, k, idx, w);
    return (int)cudaGetLastError();
}

int launch_router_topk(const uint16_t* x, int T, int H, const uint16_t* Wr, int E, const float* bias,
                       int bias_stride, int k, int32_t* idx, float* w, float* logits, float* rms,
                       uint32_t* counters, float eps, void* stream) {
    if (T > 1 && (size_t)2 * H * 4 <= (size_t)RL_SMEM_MAX) {
        prof_before(TF_KERNEL_ROUTER, stream);
        const int e = launch_router_many(x, T, H, Wr, E, bias, bias_stride, k, idx, w, logits, rms, eps,
                                         (cudaStream_t)stream);
        prof_after(TF_KERNEL_ROUTER, stream);
        return e;
    }
    dim3 grid((E + RT_WARPS - 1) / RT_WARPS, T);
    const size_t smem = (size_t)(RT_WARPS + 1) * H * 2;
    if (int e = smem_limit_once((const void*)k_router_topk, 200 * 1024)) return e;
    prof_before(TF_KERNEL_ROUTER, stream);
    k_router_topk<<<grid, RT_WARPS * 32, smem, (cudaStream_t)stream>>>(x, H, Wr, E, bias, bias_stride, k, idx, w,
                                                                    logits, rms, counters, eps);
    prof_after(TF_KERNEL_ROUTER, stream);
    return (int)cudaGetLastError();
}

static int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

int launch_gateup(const DecodeParams& p, int u0, int u1, void* stream) {
    if (u1 <= u0) return 0;
    const size_t smem = (size_t)p.H * 4 + (size_t)(p.H / 32) * 4;
    if (int e = smem_limit_once((const void*)k_gateup, 64 * 1024)) return e;
    const int units = u1 - u0;
    int grid = (units + GU_WARPS - 1) / GU_WARPS;
    const int cap = sm_count() * 4;
    if (grid > cap) grid = cap;
    prof_before(TF_KERNEL_GATEUP, stream);
    k_gateup<<<grid, GU_WARPS * 32, smem, (cudaStream_t)stream>>>(p, u0, u1);
    prof_after(TF_KERNEL_GATEUP, stream);
    return (int)cudaGetLastError();
}

int launch_down(const DecodeParams& p, int with_routed, int with_shared, void* stream) {
    const int kr = with_routed ? p.k : 0;
    const size_t smem = ((size_t)down_hs_offset(kr, p.I) + (with_shared ? (size_t)p.S : 0)) * 4;
    if (int e = smem_limit_once((const void*)k_down, 200 * 1024)) return e;
    int grid = (p.H + DN_WARPS - 1) / DN_WARPS;
    const int cap = sm_count() * 2;
    if (grid > cap) grid = cap;
    prof_before(TF_KERNEL_DOWN, stream);
    k_down<<<grid, DN_WARPS * 32, smem, (cudaStream_t)stream>>>(p, with_routed, with_shared);
    prof_after(TF_KERNEL_DOWN, stream);
    return (int)cudaGetLastError();
}

int launch_dequant(const char* blob, int H, int I, int matrix, int format, void* out, size_t off_sb,
                   size_t off_codes, void* stream) {
    prof_before(TF_KERNEL_OTHER, stream);
    k_dequant<<<sm_count() * 4, 256, 0, (cudaStream_t)stream>>>(blob, H, I, matrix, format, out, off_sb, off_codes);
    prof_after(TF_KERNEL_OTHER, stream);
    return (int)cudaGetLastError();
}

}  // namespace tf
