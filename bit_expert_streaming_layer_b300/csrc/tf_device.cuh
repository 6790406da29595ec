// Device helpers shared by the decode kernels (tf_decode.cu) and the fused
// persistent decode kernel (tf_fused.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tf_internal.h"

namespace tf {
namespace dev {

constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
__device__ __forceinline__ float h2f(uint32_t h16) { return __half2float(__ushort_as_half((unsigned short)h16)); }

// Programmatic dependent launch (the kernels of the grouped path and the many-token
// router): pdl_wait returns once the stream's preceding kernel has completed and its
// writes are visible (at once when this kernel was not launched as a dependent);
// pdl_trigger lets the next kernel of the stream start its CTAs, which then wait in
// their own pdl_wait. A kernel calls pdl_wait before it reads anything an earlier
// kernel wrote, so every earlier kernel has completed by then.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

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
    // 0.5 v (1 + tanh(u)) = v / (1 + e^(-2u)), since 1 + tanh(u) = 2 / (1 + e^(-2u)): one fast exponential and
    // one fast division (relative error near 1e-6, far below the 16-bit rounding of the gated product); for a
    // large negative v the denominator overflows to +inf and the quotient is -0, the limit of the function
    const float c = 0.7978845608028654f, a = 0.044715f;
    const float inner = c * (v + a * v * v * v);
    return __fdividef(v, 1.0f + __expf(-2.0f * inner));
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

// Address of the i-th selected expert, or NULL when its id (or its slot) is out
// of range: an invalid id is never turned into an address.
__device__ __forceinline__ const char* expert_ptr(const ExpertRef& r, int i) {
    if (r.use_ptrs) return r.ptr[i];
    int e = r.idx[i];
    if ((unsigned)e >= (unsigned)r.n_experts) return nullptr;
    if (r.slot_map) {
        e = r.slot_map[e];
        if ((unsigned)e >= (unsigned)r.n_slots) return nullptr;
    }
    return r.base + (size_t)e * r.stride;
}

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fc00000); }

// ---------------------------------------------------- top-k of one token
// Warp 0 of a CTA: the k best of z[0..E) (larger first, ties -> lower index,
// NaN last), then softmax over the k selected logits. `z` and `taken` are
// shared-memory scratch of E entries; results go to idx_out / w_out.
__device__ __forceinline__ void warp_topk_softmax(float* z, unsigned char* taken, int E, int k, int lane,
                                                  int32_t* idx_out, float* w_out) {
    int sel = -1;
    float selz = 0.0f;
    for (int i = 0; i < k; ++i) {
        float best = 0.0f;
        int bi = -1;
        for (int j = lane; j < E; j += 32)
            if (!taken[j] && ranks_before(z[j], j, best, bi)) { best = z[j]; bi = j; }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ob = __shfl_xor_sync(FULL, best, o);
            const int oi = __shfl_xor_sync(FULL, bi, o);
            if (ranks_before(ob, oi, best, bi)) { best = ob; bi = oi; }
        }
        if (lane == i) { sel = bi; selz = best; }
        if (lane == 0) taken[bi] = 1;
        __syncwarp();
    }
    // softmax over the selected logits, summed in top-k order by lane 0
    float zmax = __shfl_sync(FULL, selz, 0);
    for (int i = 1; i < k; ++i) {
        const float zi = __shfl_sync(FULL, selz, i);
        if (zi > zmax) zmax = zi;
    }
    const float ev = lane < k ? expf(__fsub_rn(selz, zmax)) : 0.0f;
    float sum = 0.0f;
    for (int i = 0; i < k; ++i) sum = __fadd_rn(sum, __shfl_sync(FULL, ev, i));
    if (lane < k) {
        idx_out[lane] = sel;
        w_out[lane] = __fdiv_rn(ev, sum);
    }
}

}  // namespace dev

// Launch a kernel as a programmatic dependent of the stream's preceding kernel
// (its CTAs may start while that kernel finishes; they wait in dev::pdl_wait).
template <typename... K, typename... A>
inline cudaError_t launch_dependent(void (*kern)(K...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<A&&>(args)...);
}
}  // namespace tf
