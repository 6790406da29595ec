// Attention half of a decoder layer for one decode token: RMS scale, q/k/v
// projections, RoPE, the FP16 KV cache row of the position, attention over the
// cached positions and the output projection with the residual.
//
// The pages name hand-written attention and RoPE kernels (page "Como executar
// um modelo de 26 bilhoes de parametros em dois gigabytes de memoria em um Mac
// comum", section "Sem dependencias do llama.cpp e MLX") and keep the FP16 KV
// cache resident (same page, section "Qual e o principal truque da
// arquitetura"). They give no shapes; the operation is the reading documented
// at tf_attn_decode in tf.h (pre-norm grouped-query attention, RoPE on the
// pairs (j, j + d/2)).
//
// Four launches on the caller's stream, each a programmatic dependent of the
// previous one:
//   k_attn_qkv      one warp per row pair (j, j + d/2) of a q, k or v head:
//                   the two dot products with x, the RMS scale, the rotation
//                   (angle in double precision), then q to the workspace and
//                   k, v as fp16 into the cache rows of the position;
//   k_attn_partial  one CTA per (q head, chunk of 256 positions): scores
//                   (a group of d/8 lanes per cached key row, 16-byte loads),
//                   the chunk's maximum and exponential sum, and the
//                   exponential-weighted sum of its value rows;
//   k_attn_combine  one CTA per q head: the chunks merged under one maximum;
//   k_attn_out      one warp per output row: out = bf16(x + Wo a).
// The memory traffic is the weights once (bf16) plus the cache rows up to the
// position (fp16), each key and value row read by the q heads of its group.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "tf_device.cuh"
#include "tf_internal.h"

namespace tf {
namespace attn {

using namespace dev;

constexpr int WARPS = 8;            // warps per CTA of the projection kernels
constexpr int CH = 256;             // cached positions per partial CTA
constexpr int PT = 256;             // threads of a partial CTA
constexpr int MAX_H = 12000;        // x as fp32 in shared memory (with 33 more floats, within 48 KB)
constexpr int MAX_QD = 12288;       // a as fp32 in shared memory (48 KB)

struct Params {
    const uint16_t* x;              // bf16 [H]
    uint16_t* out;                  // bf16 [H]
    const uint16_t* Wq;             // bf16 [nq*d, H]
    const uint16_t* Wk;             // bf16 [nkv*d, H]
    const uint16_t* Wv;             // bf16 [nkv*d, H]
    const uint16_t* Wo;             // bf16 [H, nq*d]
    __half* kc;                     // fp16 [max_seq, nkv, d]
    __half* vc;                     // fp16 [max_seq, nkv, d]
    float* q;                       // workspace fp32 [nq*d] (rotated)
    float* pm;                      // workspace fp32 [nq, nch]: chunk maxima
    float* pl;                      // workspace fp32 [nq, nch]: chunk exponential sums
    float* pacc;                    // workspace fp32 [nq, nch, d]: chunk weighted value sums
    float* a;                       // workspace fp32 [nq*d]: attention output
    int H, nq, nkv, d, pos, nch;
    float eps;
    double theta;
};

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}

// RMS scale of x and x itself (fp32) in shared memory, by the whole CTA.
__device__ float stage_x(const Params& p, float* xs, float* red) {
    float ss = 0.0f;
    for (int k = threadIdx.x; k < p.H; k += blockDim.x) {
        const float v = bf2f(p.x[k]);
        xs[k] = v;
        ss = fmaf(v, v, ss);
    }
    ss = warp_sum_f(ss);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[w] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
        red[32] = rsqrtf(t / (float)p.H + p.eps);
    }
    __syncthreads();
    return red[32];
}

// Dot product of one bf16 row of length H with x (fp32 in shared memory), whole warp.
__device__ __forceinline__ float row_dot(const uint16_t* row, const float* xs, int H, int lane) {
    const uint4* r8 = reinterpret_cast<const uint4*>(row);
    float acc = 0.0f;
    for (int c = lane; c < H / 8; c += 32) {
        const uint4 w = ldg_stream(r8 + c);
        const float4 a = reinterpret_cast<const float4*>(xs)[2 * c];
        const float4 b = reinterpret_cast<const float4*>(xs)[2 * c + 1];
        acc = fmaf(bf_lo(w.x), a.x, acc);
        acc = fmaf(bf_hi(w.x), a.y, acc);
        acc = fmaf(bf_lo(w.y), a.z, acc);
        acc = fmaf(bf_hi(w.y), a.w, acc);
        acc = fmaf(bf_lo(w.z), b.x, acc);
        acc = fmaf(bf_hi(w.z), b.y, acc);
        acc = fmaf(bf_lo(w.w), b.z, acc);
        acc = fmaf(bf_hi(w.w), b.w, acc);
    }
    return warp_sum_f(acc);
}

// Row pairs: [0, nq*d/2) q, then nkv*d/2 k, then nkv*d/2 v; pair (head, j) covers rows j and j + d/2.
__global__ void __launch_bounds__(WARPS * 32) k_attn_qkv(Params p) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) float smem[];
    float* xs = smem;
    float* red = smem + p.H;  // 33 floats
    const float r = stage_x(p, xs, red);
    const int lane = threadIdx.x & 31;
    const int half = p.d / 2;
    const int nqp = p.nq * half, nkp = p.nkv * half;
    const int pair = blockIdx.x * WARPS + (threadIdx.x >> 5);
    if (pair >= nqp + 2 * nkp) return;
    int kind, hp;
    if (pair < nqp) {
        kind = 0;
        hp = pair;
    } else if (pair < nqp + nkp) {
        kind = 1;
        hp = pair - nqp;
    } else {
        kind = 2;
        hp = pair - nqp - nkp;
    }
    const int head = hp / half, j = hp - head * half;
    const uint16_t* W = kind == 0 ? p.Wq : (kind == 1 ? p.Wk : p.Wv);
    const size_t r0 = (size_t)head * p.d + j;
    const float a = r * row_dot(W + r0 * p.H, xs, p.H, lane);
    const float b = r * row_dot(W + (r0 + half) * p.H, xs, p.H, lane);
    if (lane != 0) return;
    float ra = a, rb = b;
    if (kind < 2) {
        double sn, cs;
        sincos((double)p.pos * pow(p.theta, -2.0 * (double)j / (double)p.d), &sn, &cs);
        ra = (float)((double)a * cs - (double)b * sn);
        rb = (float)((double)b * cs + (double)a * sn);
    }
    if (kind == 0) {
        p.q[r0] = ra;
        p.q[r0 + half] = rb;
    } else {
        __half* c = (kind == 1 ? p.kc : p.vc) + ((size_t)p.pos * p.nkv + head) * p.d;
        c[j] = __float2half_rn(ra);
        c[j + half] = __float2half_rn(rb);
    }
}

// One (q head, chunk) of the cached positions 0..pos.
__global__ void __launch_bounds__(PT) k_attn_partial(Params p) {
    pdl_wait();
    pdl_trigger();
    __shared__ __align__(16) float qs[256];
    __shared__ float sc[CH];
    __shared__ float red[PT / 32 + 2];
    __shared__ __align__(16) float accs[PT];
    const int h = blockIdx.x, ch = blockIdx.y;
    const int g = h / (p.nq / p.nkv);
    const int t0 = ch * CH;
    const int nt = min(CH, p.pos + 1 - t0);
    const int d = p.d, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int j = threadIdx.x; j < d; j += PT) qs[j] = p.q[h * d + j];
    __syncthreads();
    // scores: a group of d/8 lanes per key row (8 fp16 per lane)
    const int gl = d / 8, per_warp = 32 / gl;
    const int sub = lane / gl, e = lane - sub * gl;
    const float scale = rsqrtf((float)d);
    for (int tb = w * per_warp; tb < nt; tb += (PT / 32) * per_warp) {  // tb is the same for the whole warp
        const int t = tb + sub;
        float s = 0.0f;
        if (t < nt) {
            const uint4 kv = *reinterpret_cast<const uint4*>(p.kc + ((size_t)(t0 + t) * p.nkv + g) * d + 8 * e);
            const __half2* k2 = reinterpret_cast<const __half2*>(&kv);
            const float4 qa = reinterpret_cast<const float4*>(qs)[2 * e];
            const float4 qb = reinterpret_cast<const float4*>(qs)[2 * e + 1];
            const float2 f0 = __half22float2(k2[0]), f1 = __half22float2(k2[1]), f2 = __half22float2(k2[2]),
                         f3 = __half22float2(k2[3]);
            s = qa.x * f0.x;
            s = fmaf(qa.y, f0.y, s);
            s = fmaf(qa.z, f1.x, s);
            s = fmaf(qa.w, f1.y, s);
            s = fmaf(qb.x, f2.x, s);
            s = fmaf(qb.y, f2.y, s);
            s = fmaf(qb.z, f3.x, s);
            s = fmaf(qb.w, f3.y, s);
        }
        for (int o = gl / 2; o; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
        if (t < nt && e == 0) sc[t] = s * scale;
    }
    __syncthreads();
    // the chunk's maximum, then exp(s - m) and its sum
    float m = -INFINITY;
    for (int t = threadIdx.x; t < nt; t += PT) m = fmaxf(m, sc[t]);
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
    if (lane == 0) red[w] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = red[0];
        for (int i = 1; i < PT / 32; ++i) mm = fmaxf(mm, red[i]);
        red[PT / 32] = mm;
    }
    __syncthreads();
    m = red[PT / 32];
    float l = 0.0f;
    for (int t = threadIdx.x; t < nt; t += PT) {
        const float v = __expf(sc[t] - m);
        sc[t] = v;
        l += v;
    }
    l = warp_sum_f(l);
    __syncthreads();  // every thread has read red[PT / 32]
    if (lane == 0) red[w] = l;
    __syncthreads();
    // weighted value sum: thread = (dimension j, part of the positions)
    const int parts = PT / d, j = threadIdx.x % d, part = threadIdx.x / d;
    float acc = 0.0f;
    for (int t = part; t < nt; t += parts)
        acc = fmaf(sc[t], __half2float(p.vc[((size_t)(t0 + t) * p.nkv + g) * d + j]), acc);
    accs[threadIdx.x] = acc;
    __syncthreads();
    const size_t o = (size_t)h * p.nch + ch;
    if (threadIdx.x < d) {
        float s = 0.0f;
        for (int i = 0; i < parts; ++i) s += accs[i * d + threadIdx.x];
        p.pacc[o * d + threadIdx.x] = s;
    }
    if (threadIdx.x == 0) {
        float ll = 0.0f;
        for (int i = 0; i < PT / 32; ++i) ll += red[i];
        p.pm[o] = m;
        p.pl[o] = ll;
    }
}

// The chunks of one q head merged: a = sum_c e^(m_c - M) acc_c / sum_c e^(m_c - M) l_c.
__global__ void k_attn_combine(Params p) {
    pdl_wait();
    pdl_trigger();
    const int h = blockIdx.x, j = threadIdx.x;
    const int nc = (p.pos + 1 + CH - 1) / CH;
    const size_t o = (size_t)h * p.nch;
    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, p.pm[o + c]);
    float L = 0.0f, acc = 0.0f;
    for (int c = 0; c < nc; ++c) {
        const float f = __expf(p.pm[o + c] - M);
        L = fmaf(f, p.pl[o + c], L);
        acc = fmaf(f, p.pacc[(o + c) * p.d + j], acc);
    }
    p.a[h * p.d + j] = acc / L;
}

// out = bf16(x + Wo a), one warp per output row.
__global__ void __launch_bounds__(WARPS * 32) k_attn_out(Params p) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) float as[];
    const int QD = p.nq * p.d;
    for (int c = threadIdx.x; c < QD; c += blockDim.x) as[c] = p.a[c];
    __syncthreads();
    const int i = blockIdx.x * WARPS + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (i >= p.H) return;
    const float y = row_dot(p.Wo + (size_t)i * QD, as, QD, lane);
    if (lane == 0) p.out[i] = f2bf(bf2f(p.x[i]) + y);
}

struct Workspace {
    size_t q, pm, pl, pacc, a, total;
};
inline Workspace ws_layout(const tf_attn_desc* d) {
    Workspace w;
    const size_t QD = (size_t)d->n_q_heads * d->head_dim;
    const size_t nch = ((size_t)d->max_seq + CH - 1) / CH;
    w.q = 0;
    w.pm = align_up(w.q + QD * 4, 256);
    w.pl = align_up(w.pm + (size_t)d->n_q_heads * nch * 4, 256);
    w.pacc = align_up(w.pl + (size_t)d->n_q_heads * nch * 4, 256);
    w.a = align_up(w.pacc + (size_t)d->n_q_heads * nch * d->head_dim * 4, 256);
    w.total = align_up(w.a + QD * 4, 256);
    return w;
}

}  // namespace attn
}  // namespace tf

using namespace tf;

static tf_status check_desc(const tf_attn_desc* d, const char* fn) {
    if (!d) return fail(TF_ERR_INVALID_ARG, "%s: NULL descriptor", fn);
    if (d->H < 8 || d->H % 8 || d->H > attn::MAX_H)
        return fail(TF_ERR_INVALID_ARG, "%s: H=%d must be a multiple of 8 in [8, %d]", fn, d->H, attn::MAX_H);
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256)
        return fail(TF_ERR_INVALID_ARG, "%s: head_dim=%d must be 64, 128 or 256", fn, d->head_dim);
    if (d->n_kv_heads < 1 || d->n_q_heads < d->n_kv_heads || d->n_q_heads % d->n_kv_heads)
        return fail(TF_ERR_INVALID_ARG, "%s: n_q_heads=%d must be a positive multiple of n_kv_heads=%d", fn,
                    d->n_q_heads, d->n_kv_heads);
    if ((long long)d->n_q_heads * d->head_dim > attn::MAX_QD)
        return fail(TF_ERR_INVALID_ARG, "%s: n_q_heads * head_dim above %d", fn, attn::MAX_QD);
    if (d->max_seq < 1) return fail(TF_ERR_INVALID_ARG, "%s: max_seq=%d", fn, d->max_seq);
    if (!(d->eps > 0.0f) || !(d->rope_theta > 0.0f)) return fail(TF_ERR_INVALID_ARG, "%s: eps and rope_theta must be > 0", fn);
    if (!d->W_q || !d->W_k || !d->W_v || !d->W_o) return fail(TF_ERR_INVALID_ARG, "%s: NULL weight pointer", fn);
    if (!aligned16(d->W_q) || !aligned16(d->W_k) || !aligned16(d->W_v) || !aligned16(d->W_o))
        return fail(TF_ERR_INVALID_ARG, "%s: weights must be 16-byte aligned", fn);
    return TF_OK;
}

extern "C" size_t tf_attn_workspace_bytes(const tf_attn_desc* d) {
    if (check_desc(d, "tf_attn_workspace_bytes")) return 0;
    return attn::ws_layout(d).total;
}

extern "C" size_t tf_attn_cache_bytes(const tf_attn_desc* d) {
    if (check_desc(d, "tf_attn_cache_bytes")) return 0;
    return (size_t)d->max_seq * d->n_kv_heads * d->head_dim * 2;
}

extern "C" tf_status tf_attn_decode(const tf_attn_desc* d, const void* x, void* out, int pos, void* k_cache,
                                    void* v_cache, void* workspace, size_t ws_bytes, void* stream) {
    const char* fn = "tf_attn_decode";
    if (tf_status s = check_desc(d, fn)) return s;
    if (!x || !out || !k_cache || !v_cache || !workspace) return fail(TF_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (pos < 0 || pos >= d->max_seq) return fail(TF_ERR_INVALID_ARG, "%s: pos=%d outside [0, %d)", fn, pos, d->max_seq);
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace))
        return fail(TF_ERR_INVALID_ARG, "%s: caches and workspace must be 16-byte aligned", fn);
    const attn::Workspace L = attn::ws_layout(d);
    if (ws_bytes < L.total) return fail(TF_ERR_INVALID_ARG, "%s: workspace too small", fn);
    attn::Params p;
    std::memset(&p, 0, sizeof(p));
    char* ws = static_cast<char*>(workspace);
    p.x = static_cast<const uint16_t*>(x);
    p.out = static_cast<uint16_t*>(out);
    p.Wq = static_cast<const uint16_t*>(d->W_q);
    p.Wk = static_cast<const uint16_t*>(d->W_k);
    p.Wv = static_cast<const uint16_t*>(d->W_v);
    p.Wo = static_cast<const uint16_t*>(d->W_o);
    p.kc = static_cast<__half*>(k_cache);
    p.vc = static_cast<__half*>(v_cache);
    p.q = reinterpret_cast<float*>(ws + L.q);
    p.pm = reinterpret_cast<float*>(ws + L.pm);
    p.pl = reinterpret_cast<float*>(ws + L.pl);
    p.pacc = reinterpret_cast<float*>(ws + L.pacc);
    p.a = reinterpret_cast<float*>(ws + L.a);
    p.H = d->H;
    p.nq = d->n_q_heads;
    p.nkv = d->n_kv_heads;
    p.d = d->head_dim;
    p.pos = pos;
    p.nch = (d->max_seq + attn::CH - 1) / attn::CH;
    p.eps = d->eps;
    p.theta = (double)d->rope_theta;
    clear_error();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int pairs = (p.nq + 2 * p.nkv) * p.d / 2;
    const size_t smem_qkv = (size_t)p.H * 4 + 33 * 4;
    const size_t smem_out = (size_t)p.nq * p.d * 4;
    int e = (int)launch_dependent(attn::k_attn_qkv, dim3((pairs + attn::WARPS - 1) / attn::WARPS),
                                  dim3(attn::WARPS * 32), smem_qkv, st, p);
    const int nc = (pos + 1 + attn::CH - 1) / attn::CH;
    if (!e) e = (int)launch_dependent(attn::k_attn_partial, dim3(p.nq, nc), dim3(attn::PT), 0, st, p);
    if (!e) e = (int)launch_dependent(attn::k_attn_combine, dim3(p.nq), dim3(p.d), 0, st, p);
    if (!e)
        e = (int)launch_dependent(attn::k_attn_out, dim3((p.H + attn::WARPS - 1) / attn::WARPS), dim3(attn::WARPS * 32),
                                  smem_out, st, p);
    return cuda_status(e, fn);
}
