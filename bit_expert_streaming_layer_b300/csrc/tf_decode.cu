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

#include "tf_internal.h"

namespace tf {

namespace {

constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
__device__ __forceinline__ float h2f(uint32_t h16) { return __half2float(__ushort_as_half((unsigned short)h16)); }

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Code p (0..7) of a 32-bit word of packed nibbles, as the fp32 value 128 + q.
// The nibble is moved to bits 16..19 under the exponent of 128.0f, where one
// mantissa step is exactly 1 (Kim et al. 2022 / Frantar et al. 2024 use the
// same magic-exponent conversion for fp16).
template <int P>
__device__ __forceinline__ float q128(uint32_t w) {
    uint32_t v;
    if constexpr (P == 4) v = w;
    else if constexpr (P < 4) v = w << (16 - 4 * P);
    else v = w >> (4 * P - 16);
    return __uint_as_float((v & 0x000f0000u) | 0x43000000u);
}

// sum_p (128 + q_p) * n[p] over the 8 codes of one word.
__device__ __forceinline__ float dot8_q128(uint32_t w, float4 a, float4 b, float acc) {
    acc = fmaf(q128<0>(w), a.x, acc);
    acc = fmaf(q128<1>(w), a.y, acc);
    acc = fmaf(q128<2>(w), a.z, acc);
    acc = fmaf(q128<3>(w), a.w, acc);
    acc = fmaf(q128<4>(w), b.x, acc);
    acc = fmaf(q128<5>(w), b.y, acc);
    acc = fmaf(q128<6>(w), b.z, acc);
    acc = fmaf(q128<7>(w), b.w, acc);
    return acc;
}

// sum over 8 bf16 weights (one 16-byte chunk) times n.
__device__ __forceinline__ float dot8_bf16(uint4 w, float4 a, float4 b, float acc) {
    acc = fmaf(bf_lo(w.x), a.x, acc);
    acc = fmaf(bf_hi(w.x), a.y, acc);
    acc = fmaf(bf_lo(w.y), a.z, acc);
    acc = fmaf(bf_hi(w.y), a.w, acc);
    acc = fmaf(bf_lo(w.z), b.x, acc);
    acc = fmaf(bf_hi(w.z), b.y, acc);
    acc = fmaf(bf_lo(w.w), b.z, acc);
    acc = fmaf(bf_hi(w.w), b.w, acc);
    return acc;
}

// Contribution of a 32-code chunk: sum_k (s q_k + b) n_k = s (P - 128 S) + b S,
// with P = sum (128 + q_k) n_k and S = sum n_k; sb holds {fp16 s, fp16 b}.
__device__ __forceinline__ float chunk_affine(uint32_t sb, float P, float S) {
    const float s = h2f(sb & 0xffffu), b = h2f(sb >> 16);
    return fmaf(s, fmaf(-128.0f, S, P), b * S);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}

// Fixed-order warp sum: lane l holds the partial over k = l (mod 32); the xor
// butterfly 16, 8, 4, 2, 1 gives every lane the same IEEE-rounded result.
__device__ __forceinline__ float warp_sum_canonical(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(FULL, v, o));
    return v;
}

__device__ __forceinline__ float gelu_tanh(float v) {
    const float c = 0.7978845608028654f, a = 0.044715f;
    const float inner = c * (v + a * v * v * v);
    return 0.5f * v * (1.0f + tanhf(inner));
}

// r = 1/sqrt(sum x^2 / H + eps) in the canonical order; call with a full warp.
__device__ __forceinline__ float rms_scale_warp(const uint16_t* x, int H, float eps, int lane) {
    float p = 0.0f;
    for (int k = lane; k < H; k += 32) {
        const float v = bf2f(x[k]);
        p = fmaf(v, v, p);  // v*v is exact in fp32: one rounding, as in the canonical sum
    }
    p = warp_sum_canonical(p);
    const float ms = __fdiv_rn(p, (float)H);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

// Ranking used by top-k: larger logit first, equal -> lower index, NaN last;
// ib < 0 marks "no candidate yet".
__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib) {
    if (ia < 0) return false;
    if (ib < 0) return true;
    const bool na = isnan(a), nb = isnan(b);
    if (na || nb) return (na == nb) ? (ia < ib) : nb;
    if (a > b) return true;
    if (a < b) return false;
    return ia < ib;
}

__device__ __forceinline__ const char* expert_ptr(const ExpertRef& r, int i) {
    if (r.use_ptrs) return r.ptr[i];
    int e = r.idx[i];
    if (r.slot_map) e = r.slot_map[e];
    return r.base + (size_t)e * r.stride;
}

// ------------------------------------------------------------------- router

constexpr int RT_WARPS = 8;

__global__ void __launch_bounds__(RT_WARPS * 32)
k_router_topk(const uint16_t* __restrict__ x, int H, const uint16_t* __restrict__ Wr, int E,
              const float* __restrict__ bias, int bias_stride, int k, int32_t* __restrict__ idx,
              float* __restrict__ wout, float* __restrict__ logits, float* __restrict__ rms,
              uint32_t* __restrict__ counters, float eps) {
    const int t = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint16_t* xt = x + (size_t)t * H;
    const float r = rms_scale_warp(xt, H, eps, lane);
    const int e = blockIdx.x * RT_WARPS + warp;
    if (e < E) {
        const uint16_t* wr = Wr + (size_t)e * H;
        float d = 0.0f;
#pragma unroll 8
        for (int kk = lane; kk < H; kk += 32) d = fmaf(bf2f(wr[kk]), bf2f(xt[kk]), d);  // exact products
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
    __shared__ float s_selz[TF_MAX_K];
    __shared__ int s_sel[TF_MAX_K];
    for (int j = threadIdx.x; j < E; j += blockDim.x) {
        s_z[j] = __ldcg(logits + (size_t)t * E + j);
        s_taken[j] = 0;
    }
    __syncthreads();
    if (warp == 0) {
        for (int i = 0; i < k; ++i) {
            float best = 0.0f;
            int bi = -1;
            for (int j = lane; j < E; j += 32)
                if (!s_taken[j] && ranks_before(s_z[j], j, best, bi)) { best = s_z[j]; bi = j; }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const float ob = __shfl_xor_sync(FULL, best, o);
                const int oi = __shfl_xor_sync(FULL, bi, o);
                if (ranks_before(ob, oi, best, bi)) { best = ob; bi = oi; }
            }
            if (lane == 0) {
                s_sel[i] = bi;
                s_selz[i] = best;
                s_taken[bi] = 1;
            }
            __syncwarp();
        }
        if (lane == 0) {
            float zmax = s_selz[0];
            for (int i = 1; i < k; ++i)
                if (s_selz[i] > zmax) zmax = s_selz[i];
            float ev[TF_MAX_K];
            float sum = 0.0f;
            for (int i = 0; i < k; ++i) {
                ev[i] = expf(__fsub_rn(s_selz[i], zmax));
                sum = __fadd_rn(sum, ev[i]);
            }
            for (int i = 0; i < k; ++i) {
                idx[(size_t)t * k + i] = s_sel[i];
                wout[(size_t)t * k + i] = __fdiv_rn(ev[i], sum);
            }
            counters[t] = 0;  // leave the workspace zeroed for the next call
        }
    }
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
    for (int kk = threadIdx.x; kk < p.H; kk += blockDim.x) n[kk] = __fmul_rn(r, bf2f(p.x[kk]));
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
            const char* gq = blob + (size_t)(2 * j) * (H / 2);
            const char* uq = gq + H / 2;
            const uint32_t* gsb = reinterpret_cast<const uint32_t*>(blob + p.off_gu_sb + (size_t)(2 * j) * (H / 64) * 4);
            const uint32_t* usb = gsb + H / 64;
            for (int c = lane; c < nchunk; c += 32) {
                const uint4 qg = ldg_stream(gq + 16 * c);
                const uint4 qu = ldg_stream(uq + 16 * c);
                const uint32_t sbg = __ldg(gsb + (c >> 1));
                const uint32_t sbu = __ldg(usb + (c >> 1));
                const float4* nn = n4 + 8 * c;
                float pg = 0.0f, pu = 0.0f;
                pg = dot8_q128(qg.x, nn[0], nn[1], pg);
                pu = dot8_q128(qu.x, nn[0], nn[1], pu);
                pg = dot8_q128(qg.y, nn[2], nn[3], pg);
                pu = dot8_q128(qu.y, nn[2], nn[3], pu);
                pg = dot8_q128(qg.z, nn[4], nn[5], pg);
                pu = dot8_q128(qu.z, nn[4], nn[5], pu);
                pg = dot8_q128(qg.w, nn[6], nn[7], pg);
                pu = dot8_q128(qu.w, nn[6], nn[7], pu);
                const float S = csum[c];
                ag += chunk_affine(sbg, pg, S);
                au += chunk_affine(sbu, pu, S);
            }
            dst = p.h_routed + (size_t)i * I + j;
        } else {
            const int j = u - routed_units;
            const char* gw = reinterpret_cast<const char*>(p.Wsg + (size_t)j * H);
            const char* uw = reinterpret_cast<const char*>(p.Wsu + (size_t)j * H);
            for (int c = lane; c < H / 8; c += 32) {
                const uint4 a = ldg_stream(gw + 16 * c);
                const uint4 b = ldg_stream(uw + 16 * c);
                const float4 n0 = n4[2 * c], n1 = n4[2 * c + 1];
                ag = dot8_bf16(a, n0, n1, ag);
                au = dot8_bf16(b, n0, n1, au);
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
    for (int t = threadIdx.x; t < kr * I; t += blockDim.x) hr[t] = __ldcg(p.h_routed + t);
    if (with_shared)
        for (int t = threadIdx.x; t < S; t += blockDim.x) hs[t] = __ldcg(p.h_shared + t);
    if (threadIdx.x < kr) {
        s_w[threadIdx.x] = p.w[threadIdx.x];
        s_ptr[threadIdx.x] = expert_ptr(p.ex, threadIdx.x);
    }
    __syncthreads();
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
        for (int t = lane; t < ntask; t += 32) {
            const int i = t / cpr, c = t - (t / cpr) * cpr;
            const char* blob = s_ptr[i];
            const uint4 q = ldg_stream(blob + p.off_d_codes + (size_t)j * (I / 2) + 16 * c);
            const uint32_t sb =
                __ldg(reinterpret_cast<const uint32_t*>(blob + p.off_d_sb + (size_t)j * (I / 64) * 4) + (c >> 1));
            const float4* hh = hr4 + (i * I + 32 * c) / 4;
            float P = 0.0f;
            P = dot8_q128(q.x, hh[0], hh[1], P);
            P = dot8_q128(q.y, hh[2], hh[3], P);
            P = dot8_q128(q.z, hh[4], hh[5], P);
            P = dot8_q128(q.w, hh[6], hh[7], P);
            acc = fmaf(s_w[i], chunk_affine(sb, P, hcs[i * cpr + c]), acc);
        }
        if (with_shared) {
            const char* dw = reinterpret_cast<const char*>(p.Wsd + (size_t)j * S);
            for (int c = lane; c < S / 8; c += 32) {
                const uint4 a = ldg_stream(dw + 16 * c);
                accs = dot8_bf16(a, hs4[2 * c], hs4[2 * c + 1], accs);
            }
        }
        acc = warp_sum(acc);
        accs = warp_sum(accs);
        if (lane == 0) {
            const float d = accs + acc;
            p.out[j] = f2bf(bf2f(p.x[j]) + d);
            if (p.delta) p.delta[j] = d;
        }
    }
}

// ------------------------------------------------------------------ dequant

__global__ void k_dequant(const char* __restrict__ blob, int H, int I, int matrix, int as_bf16, void* out,
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
        if (as_bf16) static_cast<uint16_t*>(out)[t] = f2bf(w);
        else static_cast<float*>(out)[t] = w;
    }
}

}  // namespace

int launch_router_topk(const uint16_t* x, int T, int H, const uint16_t* Wr, int E, const float* bias,
                       int bias_stride, int k, int32_t* idx, float* w, float* logits, float* rms,
                       uint32_t* counters, float eps, void* stream) {
    dim3 grid((E + RT_WARPS - 1) / RT_WARPS, T);
    prof_before(TF_KERNEL_ROUTER, stream);
    k_router_topk<<<grid, RT_WARPS * 32, 0, (cudaStream_t)stream>>>(x, H, Wr, E, bias, bias_stride, k, idx, w,
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
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
        attr = true;
    }
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
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_down, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        attr = true;
    }
    int grid = (p.H + DN_WARPS - 1) / DN_WARPS;
    const int cap = sm_count() * 2;
    if (grid > cap) grid = cap;
    prof_before(TF_KERNEL_DOWN, stream);
    k_down<<<grid, DN_WARPS * 32, smem, (cudaStream_t)stream>>>(p, with_routed, with_shared);
    prof_after(TF_KERNEL_DOWN, stream);
    return (int)cudaGetLastError();
}

int launch_dequant(const char* blob, int H, int I, int matrix, int as_bf16, void* out, size_t off_sb,
                   size_t off_codes, void* stream) {
    prof_before(TF_KERNEL_OTHER, stream);
    k_dequant<<<sm_count() * 4, 256, 0, (cudaStream_t)stream>>>(blob, H, I, matrix, as_bf16, out, off_sb, off_codes);
    prof_after(TF_KERNEL_OTHER, stream);
    return (int)cudaGetLastError();
}

}  // namespace tf
