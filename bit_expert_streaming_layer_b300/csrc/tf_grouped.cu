// Grouped (batched / prefill) routed-expert FFN on the 5th-generation tensor
// cores: token x expert histogram, exclusive scan, stable permutation, grouped
// dequant-to-16-bit tcgen05 GEMMs with fp32 accumulation in TMEM, and the
// unpermute-combine.
//
// Page "Como executar um modelo de 26 bilhoes de parametros em dois gigabytes de
// memoria em um Mac comum", section "Desempenho no mundo real": during prefill
// one loaded expert is applied to a whole group of rows. Here every expert's
// rows are gathered into one contiguous block (the permutation), each block
// runs as GEMMs against that expert's weights, and every token then sums its k
// results in top-k order.
//
// GEMM orientation (swap-AB): the weights are the M side (128 rows per tile,
// dequantised from int4 to bf16 in shared memory), the tokens are the N side
// (up to 256 per tile, loaded by TMA). D[m, n] = sum_k W[m, k] X[n, k] lives in
// TMEM as 128 lanes x N fp32 columns; two accumulators let the epilogue of one
// tile overlap the MMAs of the next. Warp roles in a 768-thread CTA:
//   warp 0      TMA producer of the weights: int4 codes (3-D tensor map over all
//               experts, 128 bytes of each of 128 rows per copy = 4 K stages,
//               128-byte swizzled) and scales/biases (bulk copy per tile)
//   warp 1      TMEM owner and MMA issuer (one elected lane issues tcgen05.mma
//               and tcgen05.commit; the warp waits as a whole)
//   warp 2      TMA producer of the token rows (2-D tensor map, SW128)
//   warp 3      second MMA issuer for tiles of up to 128 token rows: warps 1
//               and 3 take the stages of even and odd running index into two
//               accumulators, which the epilogue adds
//   warps 4..7  epilogue: tcgen05.ld, GELU-gate (gate/up) or plain (down), store
//   warps 8..23 dequant, two groups of eight warps on alternate K stages:
//               codes -> 16-bit RN(s q + b) into the SW128 A tile; the first
//               warp of a group also waits for the stage's token tile, so that
//               "A full" stands for both operands and an MMA warp waits once
//               per stage.
// Every ring (codes, A, tokens) is sized by the launch's shared-memory plan;
// the weight producer runs ahead of the MMAs by as many code stages as fit. A
// ring that two warps or groups read in turn has an even depth, so that a
// waiter never skips a phase of a barrier it tests by parity.
// Numerics: 16-bit operands, fp32 accumulation in TMEM. The token operand is
// the layer input x itself and the RMS scale r of each token multiplies its
// gate and up sums in the epilogue, as the router applies it after its dot
// products: equal in real arithmetic to feeding r x, without rounding r x to
// 16 bits (which alone cost up to 2.6 % against the fp32 layer in bf16). The
// routed gate/up GEMM runs on fp16 operands: weights dequantised to fp16 (RN of
// the exact s q + b, one fma.rn.f16x2; the same as RN of the fp32 weight
// whenever that is exact, as for every weight whose terms stay below 1 in
// magnitude) and x p, where p = 2^e is the power of two of the token's
// RMS scale r = m 2^e (m in [1, 2)): the scaling is exact and keeps the operand
// near unit size (|x p| < 2 sqrt(H)) however large x grows, and m then
// multiplies the gate and up sums. With the expert weights of the model
// configuration (a mean weight near 0.09 that cancels in tokens with a small
// update), bf16 gate/up weights alone cost up to 0.8 % against the fp32 layer;
// fp16 takes the same kind::f16 instruction at the same rate with three more
// mantissa bits. The routed down GEMM stays on bf16 operands (the dequantised
// weights and h): h reaches about 7e4 in fed-back stacks of these weights,
// beyond fp16. Worst checked token against the fp32 layer: 0.7 %. The shared
// expert's weights are given as bf16, so its GEMMs take bf16 operands (x, its
// weights, h).
//
// The same kernel runs the bf16 shared expert of a batched layer (a_bf16 = 1):
// the producer loads the weight tiles by TMA straight into the SW128 A stages
// and the dequant warps stay idle. For the shared gate/up the tile interleaves
// 8-row boxes of the gate and up matrices (rows 16i..16i+7 gate, 16i+8..16i+15
// up), so a GELU pair sits in lanes m and m ^ 8 of one epilogue warp.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <type_traits>

#include "tf_device.cuh"
#include "tf_internal.h"

namespace tf {
namespace grouped {

using namespace dev;

constexpr int NB = 256;                // tokens per GEMM tile (MMA N <= 256)
constexpr int BM = 128;                // weight rows per GEMM tile (MMA M)
constexpr int BK = 64;                 // K per pipeline stage (one quant group, 128 bytes of 16-bit values)
constexpr int BOX_SMALL = 16;          // token rows per TMA box for tiles of up to 64 rows
constexpr int BOX_BIG = 128;           // ... and for larger tiles (two loads per 256-row stage)
constexpr int NBST_MAX = 8;            // token (B) stages: as many as the plan gives
constexpr int NA_MAX = 12, NCS_MAX = 8;    // weight (A) and code stages: as many as shared memory holds
constexpr int CW = 4;                  // K stages per code stage: 128 contiguous bytes of each weight row per load
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int C_BYTES = BM * BK * CW / 2;        // 16 KB of codes per code stage
constexpr int N_DQ_WARPS = 8;          // warps of one dequant group: a weight row per pair of threads
constexpr int N_DQ = 2 * N_DQ_WARPS;   // dequant warps (8 .. 23): two groups, taking alternate K stages
constexpr int GEMM_THREADS = (8 + N_DQ) * 32;
constexpr unsigned long long OWN_LIMIT_NS = 2000000000ull;   // waits for this thread's own copies and MMAs
enum {
    BAR_CF = 0,                      // codes full [NCS_MAX]
    BAR_CE = BAR_CF + NCS_MAX,       // codes empty [NCS_MAX]
    BAR_AF = BAR_CE + NCS_MAX,       // A full [NA_MAX]
    BAR_AE = BAR_AF + NA_MAX,        // A empty [NA_MAX]
    BAR_BF = BAR_AE + NA_MAX,        // B full [NBST_MAX]
    BAR_BE = BAR_BF + NBST_MAX,      // B empty [NBST_MAX]
    BAR_SF = BAR_BE + NBST_MAX,      // sb full [2]
    BAR_SE = BAR_SF + 2,             // sb empty [2]
    BAR_DF = BAR_SE + 2,             // accumulator full [2]
    BAR_DE = BAR_DF + 2,             // accumulator empty [2]
    N_BARS = BAR_DE + 2
};
constexpr size_t GEMM_SMEM = 227 * 1024;                       // every launch takes a whole SM's shared memory
constexpr int SMEM_USABLE = (int)GEMM_SMEM - 1024 - N_BARS * 8 - 16;   // after aligning the base to 1 KB
static_assert(A_BYTES % 1024 == 0, "SW128 tiles");
static_assert(CW % 2 == 0, "a pipeline stage of one or two K blocks never spans two code stages");

// Shared-memory plan of one launch (offsets from the 1 KB-aligned base). The
// token stages are sized to the largest token tile the launch can see, and the
// rest goes to the streamed operand: code stages (int4 weights, dequantised by
// the CUDA cores) or weight stages (bf16 weights by TMA), so that enough bytes
// are in flight per SM for small tiles too.
struct Layout {
    int na, ncs, nb;    // A stages, code stages (0 for bf16 weights), token (B) stages
    int sb_stage;       // bytes of one tile's {s,b} words (two buffers; 0 for bf16 weights)
    int n_mma;          // MMA warps: 2 (tiles of up to 128 token rows: the stages of even / odd running index into
                        // two accumulators, added by the epilogue) or 1
    int acc_cols;       // TMEM columns of one accumulator (accumulator (item parity, MMA warp) at
                        // column (parity * n_mma + warp) * acc_cols)
    int sw;             // K blocks (of BK) per pipeline stage: 2 for int4 tiles of up to 128 tokens (one wait, one
                        // fence and one arrival per 128 of K), else 1
    int b_stage;        // bytes of one token stage (sw sub-tiles of b_stage / sw bytes, one per K block)
    int box_big;        // 1: tiles over 64 rows load 128-row boxes
    int off_b, off_c, off_sb, off_bar;
};

struct GemmParams {
    const char* ebase;          // resident experts: expert e at ebase + e * estride
    unsigned long long estride;
    unsigned long long off_sb;  // offset of this matrix's {s,b} section in an expert
    int K;                      // reduction length (H for gate/up, I for down)
    int MT;                     // weight-row tiles per expert (2I/128 or H/128)
    int E;
    const int32_t* counts;      // [E] rows per expert
    const int32_t* offsets;     // [E+1] first permuted row of each expert
    const int32_t* tiles;       // [E+1] prefix of tiles (MT * ceil(count / NB)) per expert
    int mode;                   // 0: gate/up -> h bf16 [P, I]; 1: down -> y fp32 [P, H]
    uint16_t* hout;
    float* yout;
    int ldo;                    // row length of the output (I or H)
    uint32_t* err;
    int a_bf16;                 // 1: bf16 weight matrices by TMA (tmA, and tmA2 for the up rows); 0: int4 codes
    int pair_log2;              // gate/up: the up row of tile row m is m ^ (1 << pair_log2)
    int ksplit;                 // K split into ksplit items per tile (> 1: raw fp32 partial sums go to part)
    float* part;                // [ksplit][ntok][mrows] partial sums (ksplit > 1)
    int ntok, mrows;
    const float* col_scale;     // gate/up: the RMS scale of each token row of the B operand (g, u *= it)
    int f16;                    // 1: fp16 operands (dequantised A and B), 0: bf16
    const int32_t* slot_of;     // nullable [E]: expert e's weights are slot slot_of[e] of ebase (the cache's slots)
    Layout lay;
    unsigned long long dep_limit_ns;   // limit of a wait on another role (2 s unless a test shortens it)
};

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
// try_wait with the hardware's own suspend time (no suspend-time hint).
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// tcgen05 (TMEM allocation, MMA, commit, loads, ordering fences)
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_ld8(uint32_t taddr, float* v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzled
// layout (rows of 128 bytes, 8-row atoms of 1 KB): start address >> 4, leading
// byte offset 16 B (unused for this layout), stride byte offset 1024 B between
// 8-row groups, descriptor version 1, layout SWIZZLE_128B (2).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3ffffu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// Instruction descriptor of kind::f16: fp32 accumulator, A and B both bf16
// (format 1) or both fp16 (format 0), both K-major, N (multiple of 16, <= 256)
// and M = 128.
__device__ __forceinline__ uint32_t idesc_f16(int n, int bf16) {
    const uint32_t ab = bf16 ? ((1u << 7) | (1u << 10)) : 0u;
    return (1u << 4) | ab | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// Bounded mbarrier wait of one thread on another role; after `limit` ns it
// raises the CTA's abort flag (and the global error word) and returns false, and
// it returns false as soon as the flag is up.
__device__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, uint32_t* err,
                         unsigned long long limit) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try(bar, parity)) return true;
        if ((n & 7u) == 0) {
            if (*abort_flag) return false;
            if (gtimer() - t0 > limit) {
                *abort_flag = 1u;
                atomicOr(err, 1u);
                return false;
            }
        }
    }
}
// Wait for this thread's own copies or MMAs to complete: it ignores the abort flag
// (nothing may still write to shared memory or TMEM when the CTA releases them) and
// is bounded by a fixed 2 s.
__device__ bool wait_own(uint32_t bar, uint32_t parity, uint32_t* err) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try(bar, parity)) return true;
        if ((n & 7u) == 0 && gtimer() - t0 > OWN_LIMIT_NS) {
            atomicOr(err, 1u);
            return false;
        }
    }
}

// The same wait by every lane of a warp (they read the same barrier state);
// lane 0's verdict is the warp's.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, uint32_t* err,
                                          unsigned long long limit) {
    const int ok = wait_bar(bar, parity, abort_flag, err, limit) ? 1 : 0;
    return __shfl_sync(FULL, ok, 0) != 0;
}
// One lane of a converged warp, chosen by the hardware.
__device__ __forceinline__ bool elect_one() {
    uint32_t e;
    asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n" : "=r"(e));
    return e != 0;
}

// Slot and phase of a ring of n stages, advanced one stage at a time.
struct Ring {
    int i = 0, ph = 0;
    __device__ __forceinline__ void next(int n) {
        if (++i == n) {
            i = 0;
            ph ^= 1;
        }
    }
};

// Work item w -> (expert, token block, weight tile), weight tiles fastest so that
// consecutive items share their token rows in L2.
struct Item {
    int e, row0, nrows, mt, kc;  // kc: which K chunk (split K)
};
__device__ __forceinline__ Item decode_item(const GemmParams& p, int w) {
    int lo = 0, hi = p.E;  // largest e with tiles[e] <= w
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.tiles + mid) <= w) lo = mid;
        else hi = mid;
    }
    Item it;
    it.e = lo;
    const int local0 = w - __ldg(p.tiles + lo);
    it.kc = local0 % p.ksplit;
    const int local = local0 / p.ksplit;
    const int nb = local / p.MT;
    it.mt = local - nb * p.MT;
    it.row0 = __ldg(p.offsets + lo) + nb * NB;
    const int rem = __ldg(p.counts + lo) - nb * NB;
    it.nrows = rem < NB ? rem : NB;
    return it;
}

// 128 + q for byte B of x (bytes hold one code), as fp32.
template <int B>
__device__ __forceinline__ float byte128(uint32_t x) {
    return __uint_as_float(__byte_perm(x, 0x43000000u, 0x7054u | (B << 8)));
}
// Packed fp32 pairs (sm_100+ two-wide add and FMA; each lane is the IEEE operation).
__device__ __forceinline__ unsigned long long pk2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpk2(unsigned long long v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// Eight codes of one word -> eight bf16 weights RN(fl(s q + b)) packed in a uint4, in
// the natural K order: (128 + q) - 128 is exact, s q is exact, so each weight takes
// one fp32 rounding, then one to bf16. Columns 2j and 2j+1 share a packed pair.
__device__ __forceinline__ uint4 dequant8_bf16(uint32_t q, float s, float b) {
    const uint32_t lo = q & 0x0f0f0f0fu, hi = (q >> 4) & 0x0f0f0f0fu;  // codes 0,2,4,6 / 1,3,5,7
    const unsigned long long S2 = pk2(s, s), B2 = pk2(b, b), M2 = pk2(-128.0f, -128.0f);
    const unsigned long long q0 = add2(pk2(byte128<0>(lo), byte128<0>(hi)), M2);
    const unsigned long long q1 = add2(pk2(byte128<1>(lo), byte128<1>(hi)), M2);
    const unsigned long long q2 = add2(pk2(byte128<2>(lo), byte128<2>(hi)), M2);
    const unsigned long long q3 = add2(pk2(byte128<3>(lo), byte128<3>(hi)), M2);
    const unsigned long long w[4] = {fma2(S2, q0, B2), fma2(S2, q1, B2), fma2(S2, q2, B2), fma2(S2, q3, B2)};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float a, c;
        unpk2(w[j], a, c);
        const __nv_bfloat162 v = __floats2bfloat162_rn(a, c);
        o[j] = *reinterpret_cast<const uint32_t*>(&v);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Order of the K columns inside every block of 8 in the fp16 operands of the routed gate/up GEMM:
// position p of a block holds column KPERM[p] = (0, 4, 1, 5, 2, 6, 3, 7)[p] (column c sits at
// position 2 (c & 3) + (c >> 2)). Both operands take the same order, so the products and their
// sum over K are those of the natural order; the order lets one mask pick two codes of a word.
constexpr int kperm_pos(int c) { return ((c & 3) << 1) | (c >> 2); }
static_assert(kperm_pos(0) == 0 && kperm_pos(4) == 1 && kperm_pos(1) == 2 && kperm_pos(5) == 3 && kperm_pos(2) == 4 &&
                  kperm_pos(6) == 5 && kperm_pos(3) == 6 && kperm_pos(7) == 7,
              "K order of the fp16 gate/up operands");

// Eight codes of one word (code 2j in the low nibble of byte j, 2j+1 in the high one) -> eight
// fp16 weights RN(s q + b), one rounding of the exact value (fma.rn.f16x2; s, b and the integer q
// are exact fp16 operands), in the K order above. A nibble at bits 0-3 of a half under the
// exponent of 1024 (0x6400) reads 1024 + q, one at bits 4-7 under that of 64 (0x5400) reads
// 64 + q; the subtraction of 1024 or 64 is exact. s2, b2: (s, s) and (b, b).
__device__ __forceinline__ uint4 dequant8_f16(uint32_t q, uint32_t s2, uint32_t b2) {
    const uint32_t q8 = q >> 8;
    const uint32_t t[4] = {(q & 0x000f000fu) | 0x64006400u,    // codes 0, 4
                           (q & 0x00f000f0u) | 0x54005400u,    // codes 1, 5
                           (q8 & 0x000f000fu) | 0x64006400u,   // codes 2, 6
                           (q8 & 0x00f000f0u) | 0x54005400u};  // codes 3, 7
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t v;
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(v) : "r"(t[j]), "r"((j & 1) ? 0x54005400u : 0x64006400u));
        asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[j]) : "r"(s2), "r"(v), "r"(b2));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_group_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2, GemmParams p) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NA = p.lay.na, NCS = p.lay.ncs, NBST = p.lay.nb, SW = p.lay.sw;
    const int OFF_A = 0, OFF_B = p.lay.off_b, OFF_C = p.lay.off_c, OFF_SB = p.lay.off_sb;
    const int B_BYTES = p.lay.b_stage, B_SUB = B_BYTES / SW, A_STAGE = SW * A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.lay.off_bar);
    const int OFF_MISC = p.lay.off_bar + N_BARS * 8;
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC + 4);
    const int KS = p.K / BK / p.ksplit;  // K blocks (of BK) per item
    const int NST = (KS + SW - 1) / SW;  // pipeline stages per item (the last may hold fewer than SW blocks)
    const int total = __ldg(p.tiles + p.E);
    const int gpr = p.K / 64;  // quant groups per weight row

    if (threadIdx.x == 0) {
        for (int i = 0; i < NCS; ++i) {
            mbar_init(bar(BAR_CF + i), 1);
            mbar_init(bar(BAR_CE + i), N_DQ);
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(bar(BAR_AF + i), p.a_bf16 ? 1 : N_DQ_WARPS);  // TMA bytes, or a dequant group
            mbar_init(bar(BAR_AE + i), 1);
        }
        for (int i = 0; i < NBST; ++i) {
            mbar_init(bar(BAR_BF + i), 1);
            mbar_init(bar(BAR_BE + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(BAR_SF + i), 1);
            mbar_init(bar(BAR_SE + i), N_DQ);
            mbar_init(bar(BAR_DF + i), p.lay.n_mma);
            mbar_init(bar(BAR_DE + i), 4);
        }
        *abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || warp == 2) {
        // ================================================ TMA producers: the weights (warp 0: {s,b} and codes, or
        // bf16 weight tiles) and the token tiles (warp 2) have a warp each, so that the weight stream runs as far
        // ahead as its own ring allows instead of in step with the three token stages. The whole warp walks the
        // loop and waits; one elected lane issues.
        const bool wprod = warp == 0;
        int ci = 0, bi = 0, ai = 0, it_local = 0, si = 0;   // copies issued (for the drains below)
        Ring cr, br, ar;
        bool ok = true;
        for (int w = blockIdx.x; w < total && ok; w += gridDim.x, ++it_local) {
            const Item it = decode_item(p, w);
            const int ks0 = it.kc * KS;
            if (wprod) {
                const int se = p.slot_of ? __ldg(p.slot_of + it.e) : it.e;   // where the expert's weights are
                if (!p.a_bf16) {
                    const int sbi = it_local & 1;
                    if (!(ok = warp_wait(bar(BAR_SE + sbi), ((it_local >> 1) & 1) ^ 1, abort_flag, p.err, p.dep_limit_ns)))
                        break;
                    ++si;
                    if (elect_one()) {
                        const uint32_t sb_bytes = (uint32_t)(BM * gpr * 4);
                        mbar_expect_tx(bar(BAR_SF + sbi), sb_bytes);
                        bulk_g2s(smem_u32(smem + OFF_SB + sbi * p.lay.sb_stage),
                                 p.ebase + (size_t)se * p.estride + p.off_sb + (size_t)it.mt * BM * gpr * 4, sb_bytes,
                                 bar(BAR_SF + sbi));
                    }
                    __syncwarp();
                }
                for (int ks = 0; ks < KS; ++ks) {
                    if (p.a_bf16) {
                        const int as = ar.i;
                        if (!(ok = warp_wait(bar(BAR_AE + as), ar.ph ^ 1, abort_flag, p.err, p.dep_limit_ns))) break;
                        if (elect_one()) {
                            mbar_expect_tx(bar(BAR_AF + as), A_BYTES);
                            const uint32_t dst = smem_u32(smem + OFF_A + as * A_BYTES);
                            if (p.mode == 0) {
                                // 8 gate rows, then the same 8 up rows, per 16-row band (1 KB boxes keep the SW128 atoms)
                                for (int g = 0; g < BM / 16; ++g) {
                                    tma_load_2d(dst + g * 2048, &tmA, (ks0 + ks) * BK, it.mt * (BM / 2) + g * 8,
                                                bar(BAR_AF + as));
                                    tma_load_2d(dst + g * 2048 + 1024, &tmA2, (ks0 + ks) * BK, it.mt * (BM / 2) + g * 8,
                                                bar(BAR_AF + as));
                                }
                            } else {
                                tma_load_2d(dst, &tmA, (ks0 + ks) * BK, it.mt * BM, bar(BAR_AF + as));
                            }
                        }
                        __syncwarp();
                        ++ai;
                        ar.next(NA);
                    } else if (ks % CW == 0) {
                        // codes of the next CW stages: 128 contiguous bytes of each of the tile's 128 rows (past
                        // the end of a row, as for the last stages of the down matrix, the box reads zeros)
                        const int cs = cr.i;
                        if (!(ok = warp_wait(bar(BAR_CE + cs), cr.ph ^ 1, abort_flag, p.err, p.dep_limit_ns))) break;
                        if (elect_one()) {
                            mbar_expect_tx(bar(BAR_CF + cs), C_BYTES);
                            tma_load_3d(smem_u32(smem + OFF_C + cs * C_BYTES), &tmA, (ks0 + ks) * (BK / 2), it.mt * BM,
                                        se, bar(BAR_CF + cs));
                        }
                        __syncwarp();
                        ++ci;
                        cr.next(NCS);
                    }
                }
            } else {
                const bool big = p.lay.box_big && it.nrows > 64;
                const int box = big ? BOX_BIG : BOX_SMALL;
                const int nbox = (it.nrows + box - 1) / box;
                for (int st = 0; st < NST; ++st) {
                    // with dequantised weights the token ring is the A ring (same depth): a token slot is free
                    // when the MMAs of its stage have completed, as the A slot
                    const int bs = br.i, kb0 = st * SW, nk = KS - kb0 < SW ? KS - kb0 : SW;
                    if (!(ok = warp_wait(bar((p.a_bf16 ? BAR_BE : BAR_AE) + bs), br.ph ^ 1, abort_flag, p.err,
                                         p.dep_limit_ns)))
                        break;
                    if (elect_one()) {
                        mbar_expect_tx(bar(BAR_BF + bs), (uint32_t)(nk * nbox * box * BK * 2));
                        for (int t = 0; t < nk; ++t)
                            for (int r = 0; r < nbox; ++r)
                                tma_load_2d(smem_u32(smem + OFF_B + bs * B_BYTES + t * B_SUB + r * box * BK * 2),
                                            big ? &tmB2 : &tmB, (ks0 + kb0 + t) * BK, it.row0 + r * box,
                                            bar(BAR_BF + bs));
                    }
                    __syncwarp();
                    ++bi;
                    br.next(NBST);
                }
            }
        }
        // let every copy this warp issued land before the CTA can exit (also after an abort)
        for (int j = ci - NCS; j < ci; ++j)
            if (j >= 0) wait_own(bar(BAR_CF + j % NCS), (j / NCS) & 1, p.err);
        for (int j = bi - NBST; j < bi; ++j)
            if (j >= 0) wait_own(bar(BAR_BF + j % NBST), (j / NBST) & 1, p.err);
        for (int j = ai - NA; j < ai; ++j)
            if (j >= 0) wait_own(bar(BAR_AF + j % NA), (j / NA) & 1, p.err);
        for (int j = si - 2; j < si; ++j)   // the {s,b} copies of the last two items
            if (j >= 0) wait_own(bar(BAR_SF + (j & 1)), (j >> 1) & 1, p.err);
    } else if (warp == 1 || (warp == 3 && p.lay.n_mma == 2)) {
        // ================================================ MMA issuers: the whole warp waits, one elected lane issues.
        // With two MMA warps, warp 1 takes the stages of even running index and warp 3 those of odd index, each
        // into its own accumulator (their wait -> issue chains, the pipeline's serial part, then overlap); both walk
        // every stage to keep the rings in step. The A ring's depth is a multiple of the MMA warps, so that an A
        // slot is always read by the same warp and its barriers complete in that warp's order.
        // the stage width is a compile-time constant of each copy of the role (one or two K blocks)
        auto mma_role = [&](auto sw_tag) {
            constexpr int TSW = decltype(sw_tag)::value;
            const int NMW = p.lay.n_mma, mw = warp == 1 ? 0 : 1;
            int it_local = 0, issued = 0, j = 0;   // j: running index of the stage
            Ring ar, br, last;   // last: ring position of this warp's latest stage (its MMAs complete before TMEM is freed)
            bool ok = true;
            for (int w = blockIdx.x; w < total && ok; w += gridDim.x, ++it_local) {
                const Item it = decode_item(p, w);
                const int ab = it_local & 1;
                if (!(ok = warp_wait(bar(BAR_DE + ab), ((it_local >> 1) & 1) ^ 1, abort_flag, p.err, p.dep_limit_ns))) break;
                tc_fence_after();
                const int n_mma = ((it.nrows + 15) / 16) * 16;
                const uint32_t idesc = idesc_f16(n_mma, !p.f16);
                const uint32_t d_tmem = tmem + (uint32_t)((ab * NMW + mw) * p.lay.acc_cols);
                bool started = false;   // this warp's accumulator holds a sum of the item
                for (int st = 0; st < NST; ++st, ++j) {
                    if ((j & (NMW - 1)) == mw) {   // NMW is 1 or 2
                        const int as = ar.i, bs = br.i, nk = KS - st * TSW < TSW ? KS - st * TSW : TSW;
                        if (!(ok = warp_wait(bar(BAR_AF + as), ar.ph, abort_flag, p.err, p.dep_limit_ns))) break;
                        if (p.a_bf16 && !(ok = warp_wait(bar(BAR_BF + bs), br.ph, abort_flag, p.err, p.dep_limit_ns)))
                            break;
                        tc_fence_after();
                        if (elect_one()) {   // the same lane each time: the warp is converged and elect.sync picks its first
    #pragma unroll
                            for (int t = 0; t < TSW; ++t) {   // the stage's K blocks (nk of them)
                                if (TSW == 1 || t < nk) {
                                    const uint64_t ad = sw128_desc(smem_u32(smem + OFF_A + as * A_STAGE + t * A_BYTES));
                                    const uint64_t bd = sw128_desc(smem_u32(smem + OFF_B + bs * B_BYTES + t * B_SUB));
    #pragma unroll
                                    for (int k = 0; k < BK / 16; ++k)  // 32 bytes of K per MMA: +2 in the start-address field
                                        tc_mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, started || t > 0 || k > 0);
                                }
                            }
                            tc_commit(bar(BAR_AE + as));
                            if (p.a_bf16) tc_commit(bar(BAR_BE + bs));
                        }
                        __syncwarp();
                        started = true;
                        last = ar;
                        ++issued;
                    }
                    ar.next(NA);
                    br.next(NBST);
                }
                if (!ok) break;
                // the accumulator is complete (a warp with no stage in this item arrives at once)
                if (elect_one()) tc_commit(bar(BAR_DF + ab));   // the lane that issued the MMAs: a commit tracks its own
                __syncwarp();
            }
            // the MMAs this warp issued complete before TMEM is released (also after an abort)
            if (issued > 0) wait_own(bar(BAR_AE + last.i), last.ph, p.err);
        };
        if (SW == 2)
            mma_role(std::integral_constant<int, 2>{});
        else
            mma_role(std::integral_constant<int, 1>{});
    } else if (warp >= 4 && warp < 8) {
        // ================================================ epilogue
        const int q = warp & 3;
        const int m = q * 32 + lane;  // TMEM lane = weight row within the tile
        int it_local = 0;
        for (int w = blockIdx.x; w < total; w += gridDim.x, ++it_local) {
            const Item it = decode_item(p, w);
            const int ab = it_local & 1;
            int okw = 1;
            if (lane == 0) okw = wait_bar(bar(BAR_DF + ab), (it_local >> 1) & 1, abort_flag, p.err, p.dep_limit_ns);
            if (!__shfl_sync(FULL, okw, 0)) break;
            tc_fence_after();
            const int NMW = p.lay.n_mma;
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * NMW * p.lay.acc_cols);
            // with two MMA warps the item's stages start at running index it_local * NST: a one-stage item has a
            // sum in one accumulator only
            const int j0 = it_local * NST;
            const bool use0 = NMW == 1 || NST > 1 || (j0 & 1) == 0, use1 = NMW == 2 && (NST > 1 || (j0 & 1) == 1);
            auto epi = [&](auto two_tag) {
                constexpr bool TWO = decltype(two_tag)::value;   // two MMA warps: two accumulators
                // columns c*8 .. c*8+7 of this row (with two accumulators: the even-stage one plus the odd-stage one)
                auto ld_acc = [&](int c, float* v) {
                    if constexpr (!TWO) {
                        tc_ld8(tbase + (uint32_t)(c * 8), v);
                    } else {
                        if (use0) {
                            tc_ld8(tbase + (uint32_t)(c * 8), v);
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
                        }
                        if (use1) {
                            float v1[8];
                            tc_ld8(tbase + (uint32_t)(p.lay.acc_cols + c * 8), v1);
#pragma unroll
                            for (int i = 0; i < 8; ++i) v[i] = use0 ? __fadd_rn(v[i], v1[i]) : v1[i];
                        }
                    }
                };
                const int nchunks = (it.nrows + 7) / 8;
                if (p.ksplit > 1) {
                    // raw partial sums of this K chunk, token-major so that the warp's rows are contiguous
                    const int row = it.mt * BM + m;
                    for (int c = 0; c < nchunks; ++c) {
                        float v[8];
                        ld_acc(c, v);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int n = c * 8 + i;
                            if (n < it.nrows) p.part[((size_t)it.kc * p.ntok + it.row0 + n) * p.mrows + row] = v[i];
                        }
                    }
                } else if (p.mode == 0) {
                    // h column of this row pair: 2^ps gate rows then their 2^ps up rows, repeated
                    const int ps = p.pair_log2;
                    const int j = it.mt * (BM / 2) + ((m >> (ps + 1)) << ps) + (m & ((1 << ps) - 1));
                    const bool up = (m >> ps) & 1;
                    for (int c = 0; c < nchunks; ++c) {
                        float v[8];
                        ld_acc(c, v);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float other = __shfl_xor_sync(FULL, v[i], 1 << ps);
                            const float g = up ? other : v[i], u = up ? v[i] : other;
                            const int n = c * 8 + i;
                            if ((i & 1) == (int)up && n < it.nrows) {
                                const float sc = __ldg(p.col_scale + it.row0 + n);
                                const float hv = gelu_tanh(__fmul_rn(sc, g)) * __fmul_rn(sc, u);
                                p.hout[(size_t)(it.row0 + n) * p.ldo + j] = f2bf(hv);
                            }
                        }
                    }
                } else {
                    const int jg = it.mt * BM + m;
                    for (int c = 0; c < nchunks; ++c) {
                        float v[8];
                        ld_acc(c, v);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int n = c * 8 + i;
                            if (n < it.nrows) p.yout[(size_t)(it.row0 + n) * p.ldo + jg] = v[i];
                        }
                    }
                }
            };
            if (NMW == 2)
                epi(std::true_type{});
            else
                epi(std::false_type{});
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_DE + ab));
        }
    } else if (warp >= 8 && !p.a_bf16) {
        // ================================================ dequant: two groups of eight warps; group g takes the K
        // stages whose running index is g modulo 2, so that stages are dequantised side by side, and every warp
        // walks every stage to keep the code and A rings in step. A waiter never skips a phase of a barrier it
        // tests by parity: the A ring's depth is even (tiles of up to 128 rows: each slot has one group and one
        // MMA warp), or (three stages, one MMA warp) the in-order completion of the MMAs orders the phases.
        const int t = threadIdx.x - 8 * 32;
        const int grp = t / (N_DQ_WARPS * 32);
        const int r = (t >> 1) & (BM - 1), hf = t & 1;   // weight row in the tile, half of the 64-code group
        auto run = [&](auto f16_tag, auto sw_tag) {
            constexpr bool F16 = decltype(f16_tag)::value;
            constexpr int TSW = decltype(sw_tag)::value;   // K blocks per stage, a compile-time constant
            Ring cr, ar;
            int g = 0, it_local = 0;   // g: the group whose stage is next
            bool ok = true;
            for (int w = blockIdx.x; w < total && ok; w += gridDim.x, ++it_local) {
                const int sbi = it_local & 1;
                if (!(ok = warp_wait(bar(BAR_SF + sbi), (it_local >> 1) & 1, abort_flag, p.err, p.dep_limit_ns))) break;
                const uint32_t* sbrow = reinterpret_cast<const uint32_t*>(smem + OFF_SB + sbi * p.lay.sb_stage) + r * gpr;
                for (int st = 0; st < NST; ++st) {
                    const int kb0 = st * TSW, nk = KS - kb0 < TSW ? KS - kb0 : TSW;   // K blocks of this stage
                    const bool mine = g == grp;
                    // a stage never spans two code stages (SW divides CW)
                    if (kb0 % CW == 0 && !(ok = warp_wait(bar(BAR_CF + cr.i), cr.ph, abort_flag, p.err, p.dep_limit_ns)))
                        break;
                    if (mine && !(ok = warp_wait(bar(BAR_AE + ar.i), ar.ph ^ 1, abort_flag, p.err, p.dep_limit_ns))) break;
                    if (mine) {
#pragma unroll
                        for (int t = 0; t < TSW; ++t) {   // the stage's K blocks (nk of them)
                            if (TSW > 1 && t >= nk) break;
                            const int kb = kb0 + t, sub = kb % CW;
                            // the code box lands 128-byte swizzled: 16-byte chunk j of row r sits at chunk
                            // j ^ (r & 7), so the 16 rows a warp reads spread over all banks
                            const uint4 qv = *reinterpret_cast<const uint4*>(smem + OFF_C + cr.i * C_BYTES +
                                                                             r * (CW * BK / 2) + (((sub * 2 + hf) ^ (r & 7)) << 4));
                            const uint32_t sbw = sbrow[kb];
                            unsigned char* arow =
                                smem + OFF_A + ar.i * A_STAGE + t * A_BYTES + (r >> 3) * 1024 + (r & 7) * 128;
                            const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
                            if constexpr (F16) {
                                const uint32_t s2 = __byte_perm(sbw, 0, 0x1010), b2 = __byte_perm(sbw, 0, 0x3232);
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    const int chunk = hf * 4 + c;  // 16-byte chunk (8 columns) of the 128-byte row
                                    *reinterpret_cast<uint4*>(arow + ((chunk ^ (r & 7)) << 4)) = dequant8_f16(qw[c], s2, b2);
                                }
                            } else {
                                const float s = h2f(sbw & 0xffffu), b = h2f(sbw >> 16);
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    const int chunk = hf * 4 + c;
                                    *reinterpret_cast<uint4*>(arow + ((chunk ^ (r & 7)) << 4)) = dequant8_bf16(qw[c], s, b);
                                }
                            }
                        }
                        fence_proxy_async();  // generic-proxy writes, read next by the tensor core
                        __syncwarp();
                        // the stage's token tile has landed before its A stage is reported full
                        if ((warp & (N_DQ_WARPS - 1)) == 0 &&
                            !(ok = warp_wait(bar(BAR_BF + ar.i), ar.ph, abort_flag, p.err, p.dep_limit_ns)))
                            break;
                        if (lane == 0) mbar_arrive(bar(BAR_AF + ar.i));
                    }
                    if ((kb0 + nk) % CW == 0 || kb0 + nk == KS) {   // the code stage is used up
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(BAR_CE + cr.i));
                        cr.next(NCS);
                    }
                    ar.next(NA);
                    g ^= 1;
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_SE + sbi));
            }
        };
        using W1 = std::integral_constant<int, 1>;
        using W2 = std::integral_constant<int, 2>;
        if (p.f16) {
            if (SW == 2) run(std::true_type{}, W2{}); else run(std::true_type{}, W1{});
        } else {
            if (SW == 2) run(std::false_type{}, W2{}); else run(std::false_type{}, W1{});
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ routing -> permutation

// Exclusive prefix sum of v over the threads of a 1024-thread CTA (thread order);
// wsum is shared scratch of 32 ints.
__device__ __forceinline__ int block_exclusive_scan(int v, int32_t* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int z = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, z, o);
            if (lane >= o) z += y;
        }
        wsum[lane] = z;
    }
    __syncthreads();
    const int r = x - v + (warp > 0 ? wsum[warp - 1] : 0);
    __syncthreads();
    return r;
}

// One CTA: the GEMM tile prefixes of one wave of experts (experts outside the
// wave get no tile; their rows keep their places in the permutation).
__global__ void __launch_bounds__(1024) k_wave_plan(const int32_t* __restrict__ counts, const int32_t* __restrict__ mask,
                                                     int E, int mt_gu, int mt_d, int32_t* tiles_gu, int32_t* tiles_d) {
    pdl_wait();
    pdl_trigger();
    __shared__ int32_t wsum[32];
    const int e = threadIdx.x;
    const int c = e < E && __ldg(mask + e) ? __ldg(counts + e) : 0;
    const int nb = (c + NB - 1) / NB;
    const int excl = block_exclusive_scan(nb, wsum);
    if (e < E) {
        tiles_gu[e] = excl * mt_gu;
        tiles_d[e] = excl * mt_d;
    }
    if (e == E - 1) {
        tiles_gu[E] = (excl + nb) * mt_gu;
        tiles_d[E] = (excl + nb) * mt_d;
    }
}

// One CTA: tokens per expert, exclusive scan, GEMM tile prefixes.
__global__ void __launch_bounds__(1024) k_group_hist(const int32_t* __restrict__ idx, int P, int E, int mt_gu,
                                                      int mt_d, int32_t* counts, int32_t* offsets, int32_t* tiles_gu,
                                                      int32_t* tiles_d, uint32_t* err) {
    pdl_wait();
    pdl_trigger();
    __shared__ int32_t cnt[TF_MAX_E];
    __shared__ int32_t wsum[32];
    if (threadIdx.x == 0) *err = 0u;   // a new call: no GEMM wait has given up yet
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int e = __ldg(idx + p);
        if ((unsigned)e < (unsigned)E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // exclusive scans of counts and of tiles (E <= 1024: one expert per thread)
    const int e = threadIdx.x;
    const int c = e < E ? cnt[e] : 0;
    const int nb = (c + NB - 1) / NB;
    const int excl[2] = {block_exclusive_scan(c, wsum), block_exclusive_scan(nb, wsum)};
    if (e < E) {
        counts[e] = c;
        offsets[e] = excl[0];
        tiles_gu[e] = excl[1] * mt_gu;
        tiles_d[e] = excl[1] * mt_d;
    }
    if (e == E - 1) {
        offsets[E] = excl[0] + c;
        tiles_gu[E] = (excl[1] + nb) * mt_gu;
        tiles_d[E] = (excl[1] + nb) * mt_d;
    }
}

// CTA e: stable positions of the pairs routed to expert e (pairs p = t * k + i in
// increasing p, i.e. sorted by (expert, token, rank)).
__global__ void __launch_bounds__(1024) k_group_pos(const int32_t* __restrict__ idx, int P,
                                                     const int32_t* __restrict__ offsets, int32_t* perm,
                                                     int32_t* inv) {
    pdl_wait();
    pdl_trigger();
    __shared__ int32_t wcnt[32];
    __shared__ int32_t base_s;
    const int e = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) base_s = offsets[e];
    __syncthreads();
    for (int p0 = 0; p0 < P; p0 += blockDim.x) {
        const int p = p0 + threadIdx.x;
        const bool mine = p < P && __ldg(idx + p) == e;
        const unsigned ball = __ballot_sync(FULL, mine);
        if (lane == 0) wcnt[warp] = __popc(ball);
        __syncthreads();
        int before = 0, total = 0;
        for (int w2 = 0; w2 < 32; ++w2) {
            const int v = wcnt[w2];
            before += w2 < warp ? v : 0;
            total += v;
        }
        const int base = base_s;
        if (mine) {
            const int pos = base + before + __popc(ball & ((1u << lane) - 1u));
            perm[pos] = p;
            inv[p] = pos;
        }
        __syncthreads();
        if (threadIdx.x == 0) base_s = base + total;
        __syncthreads();
    }
}

// Pairs whose expert id is out of range get no row: their inverse is -1.
__global__ void k_group_inv_init(const int32_t* __restrict__ idx, int P, int E, int32_t* inv) {
    pdl_wait();
    pdl_trigger();
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p < P && (unsigned)__ldg(idx + p) >= (unsigned)E) inv[p] = -1;
}

// Work plan of the shared expert: one "expert" holding all T tokens in order.
__global__ void k_shared_plan(int T, int mt_gu, int mt_d, int ks_gu, int ks_d, int32_t* counts, int32_t* offsets,
                              int32_t* tiles_gu, int32_t* tiles_d) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) {
        const int nb = (T + NB - 1) / NB;
        counts[0] = T;
        offsets[0] = 0;
        offsets[1] = T;
        tiles_gu[0] = 0;
        tiles_gu[1] = nb * mt_gu * ks_gu;
        tiles_d[0] = 0;
        tiles_d[1] = nb * mt_d * ks_d;
    }
}

// Split-K shared gate/up: h[t][j] = bf16(gelu(r_t g) r_t u), g and u summed over
// the K chunks in order (gate row of column j and its up row 8 rows further, per
// the 8-row interleave of the tiles), r_t the token's RMS scale.
__global__ void k_shared_gu_combine(const float* __restrict__ part, const float* __restrict__ rms, int ks, int T,
                                    int S, uint16_t* hs) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= S) return;
    const int jj = j & 63;
    const int rg = (j >> 6) * BM + (jj >> 3) * 16 + (jj & 7);
    float g = 0.0f, u = 0.0f;
    for (int c = 0; c < ks; ++c) {
        const float* pr = part + ((size_t)c * T + t) * (2 * S);
        g += pr[rg];
        u += pr[rg + 8];
    }
    const float r = rms[t];
    hs[(size_t)t * S + j] = f2bf(gelu_tanh(__fmul_rn(r, g)) * __fmul_rn(r, u));
}

// Split-K shared down: ys[t][i] = sum of the K chunks in order.
__global__ void k_shared_down_combine(const float* __restrict__ part, int ks, int T, int H, float* ys) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= H) return;
    float y = 0.0f;
    for (int c = 0; c < ks; ++c) y += part[((size_t)c * T + t) * H + i];
    ys[(size_t)t * H + i] = y;
}

// r_t = 1/sqrt(mean(x_t^2) + eps) in the canonical order, one warp per token.
__global__ void k_group_rms(const uint16_t* __restrict__ x, int T, int H, float eps, float* rms) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const float r = rms_scale_warp(x + (size_t)t * H, H, eps, lane);
    if (lane == 0) rms[t] = r;
}

// bf16 pair times a power of two p -> fp16 pair (the product is exact; the
// conversion rounds only values in the fp16 subnormal range).
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w, float p) {
    const __half2 h = __floats2half2_rn(bf_lo(w) * p, bf_hi(w) * p);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Row pos of the permuted activations: x_t p_t as fp16 (t = perm[pos] / k, p_t the
// power of two of the RMS scale r_t = m_t p_t, m_t in [1, 2)), its columns in the
// order kperm_pos gives within each block of 8, and m_t, the scale of the row's
// gate and up sums.
__global__ void k_group_gather(const uint16_t* __restrict__ x, const float* __restrict__ rms,
                               const int32_t* __restrict__ perm, int P, int k, int H, uint16_t* xp,
                               float* __restrict__ rp) {
    pdl_wait();
    pdl_trigger();
    const int pos = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (pos >= P) return;
    const int t = __ldg(perm + pos) / k;
    const uint32_t rb = __float_as_uint(__ldg(rms + t));
    const float p = __uint_as_float(rb & 0x7f800000u);                 // 2^e (r > 0 is a normal fp32 value)
    if (lane == 0) rp[pos] = __uint_as_float((rb & 0x007fffffu) | 0x3f800000u);   // m = r / p, exact
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)pos * H);
    for (int v = lane; v < H / 8; v += 32) {
        const uint4 a = __ldg(src + v);
        const uint32_t h01 = bf2_to_h2(a.x, p), h23 = bf2_to_h2(a.y, p), h45 = bf2_to_h2(a.z, p), h67 = bf2_to_h2(a.w, p);
        // columns (0, 4, 1, 5, 2, 6, 3, 7) of the block, the order of the dequantised gate/up weights
        dst[v] = make_uint4(__byte_perm(h01, h45, 0x5410), __byte_perm(h01, h45, 0x7632), __byte_perm(h23, h67, 0x5410),
                            __byte_perm(h23, h67, 0x7632));
    }
}

// out[t] = bf16(x[t] + delta), delta = ys[t] + sum_i w[t,i] y[inv[t k + i]],
// the shared term first (ys NULL: none), then the routed terms in top-k order.
__global__ void k_group_combine(const uint16_t* __restrict__ x, const float* __restrict__ y,
                                const float* __restrict__ ys,
                                const int32_t* __restrict__ inv, const float* __restrict__ w, int k, int H,
                                const uint32_t* err, uint16_t* out, float* delta) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.y;
    const int j = (blockIdx.x * blockDim.x + threadIdx.x) * 4;   // four columns per thread
    if (*err) {  // a GEMM wait timed out: the outputs are NaN, never stale or partial values
        for (int c = j; c < j + 4 && c < H; ++c) {
            out[(size_t)t * H + c] = 0x7fc0u;
            if (delta) delta[(size_t)t * H + c] = __int_as_float(0x7fc00000);
        }
        return;
    }
    __shared__ int32_t rows[TF_MAX_K];
    __shared__ float ws[TF_MAX_K];
    if (threadIdx.x < k) {
        rows[threadIdx.x] = __ldg(inv + (size_t)t * k + threadIdx.x);
        ws[threadIdx.x] = __ldg(w + (size_t)t * k + threadIdx.x);
    }
    __syncthreads();
    if (j < H) {
        float4 acc = ys ? __ldg(reinterpret_cast<const float4*>(ys + (size_t)t * H + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int i = 0; i < k; ++i) {
            if (rows[i] < 0) continue;
            const float4 v = __ldg(reinterpret_cast<const float4*>(y + (size_t)rows[i] * H + j));
            acc.x = fmaf(ws[i], v.x, acc.x);
            acc.y = fmaf(ws[i], v.y, acc.y);
            acc.z = fmaf(ws[i], v.z, acc.z);
            acc.w = fmaf(ws[i], v.w, acc.w);
        }
        const uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (size_t)t * H + j));
        const float o0 = bf_lo(xv.x) + acc.x, o1 = bf_hi(xv.x) + acc.y;
        const float o2 = bf_lo(xv.y) + acc.z, o3 = bf_hi(xv.y) + acc.w;
        *reinterpret_cast<uint2*>(out + (size_t)t * H + j) =
            make_uint2((uint32_t)f2bf(o0) | ((uint32_t)f2bf(o1) << 16), (uint32_t)f2bf(o2) | ((uint32_t)f2bf(o3) << 16));
        if (delta) *reinterpret_cast<float4*>(delta + (size_t)t * H + j) = acc;
    }
}

// ------------------------------------------------------------------ host

struct Carve {
    size_t err, counts, offsets, tiles_gu, tiles_d, perm, inv, rms, rp, xp, hb, y;
    size_t s_plan, hs, ys, spart;  // shared expert (S > 0): plan arrays, h, y, split-K sums
    size_t total;
};

Carve carve(int T, int H, int I, int E, int k, int S) {
    Carve c;
    const size_t P = (size_t)T * k;
    size_t o = 0;
    c.err = o; o += 256;
    c.counts = o; o += align_up((size_t)E * 4, 256);
    c.offsets = o; o += align_up((size_t)(E + 1) * 4, 256);
    c.tiles_gu = o; o += align_up((size_t)(E + 1) * 4, 256);
    c.tiles_d = o; o += align_up((size_t)(E + 1) * 4, 256);
    c.perm = o; o += align_up(P * 4, 256);
    c.inv = o; o += align_up(P * 4, 256);
    c.rms = o; o += align_up((size_t)T * 4, 256);
    c.rp = o; o += align_up(P * 4, 256);
    c.xp = o; o += align_up(P * H * 2, 256);
    c.hb = o; o += align_up(P * I * 2, 256);
    c.y = o; o += align_up(P * H * 4, 256);
    c.s_plan = c.hs = c.ys = c.spart = 0;
    if (S > 0) {
        c.s_plan = o; o += 256;  // counts[1], offsets[2], tiles_gu[2], tiles_d[2]
        c.hs = o; o += align_up((size_t)T * S * 2, 256);
        c.ys = o; o += align_up((size_t)T * H * 4, 256);
        // split-K partial sums, used while the tokens fit one 256-row tile (at most 4 chunks)
        const size_t tk = (size_t)(T < NB ? T : NB);
        const size_t rows = (size_t)(2 * S > H ? 2 * S : H);
        c.spart = o; o += align_up(4 * tk * rows * 4, 256);
    }
    c.total = o;
    return c;
}

// The driver's tensor-map encoder, looked up through the runtime so that the
// library needs no link-time dependency on the driver library.
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encoder();
    if (!fn) return false;
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major 16-bit [rows, cols] (bf16, or fp16 with f16 = true) as a 2-D SW128 map with boxes of 64 columns
// (128 bytes) x box_rows rows.
bool encode_rows(CUtensorMap* m, const void* base, int cols, int rows, int box_rows, bool f16 = false) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t str[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {BK, (cuuint32_t)box_rows};
    return encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, str, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

// Shared-memory plan of one launch for token tiles of up to max_rows rows and a
// reduction of K: bf16 weights by TMA (a_bf16) or int4 codes dequantised into A
// stages. Tiles of up to 128 token rows stream weights: two MMA warps over two
// A / token stages of two K blocks each (bf16 weights: as many one-block stages
// as fit, an even number); the rest goes to code stages. Larger tiles are bound
// by the tensor core: one MMA warp, three A and three token stages of one K
// block, the rest to code stages (bf16 weights: to weight stages). A ring that
// two warps read in turn has an even depth, so that each slot has one reader.
// na = 0 when nothing fits.
Layout plan_layout(int max_rows, bool a_bf16, int K) {
    Layout l;
    std::memset(&l, 0, sizeof(l));
    int rows = max_rows > 64 ? (max_rows + BOX_BIG - 1) / BOX_BIG * BOX_BIG : (max_rows + 15) / 16 * 16;
    if (rows > NB) rows = NB;
    const bool small = max_rows <= 64;
    l.box_big = !small;
    l.sw = !a_bf16 && max_rows <= 128 ? 2 : 1;
    l.b_stage = l.sw * rows * BK * 2;
    l.n_mma = max_rows <= 128 ? 2 : 1;
    l.acc_cols = l.n_mma == 2 ? 128 : NB;
    if (a_bf16) {
        // with two MMA warps both rings have an even depth: a slot is read by one warp only
        if (small) {
            l.na = SMEM_USABLE / (A_BYTES + l.b_stage);
            if (l.na > NBST_MAX) l.na = NBST_MAX;
            l.nb = l.na;
        } else {
            l.nb = l.n_mma == 2 ? 4 : 3;
            l.na = (SMEM_USABLE - l.nb * l.b_stage) / A_BYTES;
            if (l.na > NA_MAX) l.na = NA_MAX;
        }
        if (l.n_mma == 2) {
            l.na &= ~1;
            l.nb &= ~1;
        }
        l.off_b = l.na * A_BYTES;
        l.off_c = l.off_b + l.nb * l.b_stage;
        l.off_sb = l.off_c;
        l.off_bar = l.off_sb;
        if (l.na < 2) l.na = 0;
    } else {
        // up to 128 token rows: two stages of two K blocks (an even depth: each slot has one dequant group and
        // one of the two MMA warps); larger tiles: three stages of one, one MMA warp
        l.na = l.nb = l.sw == 2 ? 2 : 3;
        l.sb_stage = BM * (K / 64) * 4;
        l.off_b = l.na * l.sw * A_BYTES;
        l.off_c = l.off_b + l.nb * l.b_stage;
        l.ncs = (SMEM_USABLE - l.off_c - 2 * l.sb_stage) / C_BYTES;
        if (l.ncs > NCS_MAX) l.ncs = NCS_MAX;
        l.off_sb = l.off_c + l.ncs * C_BYTES;
        l.off_bar = l.off_sb + 2 * l.sb_stage;
        if (l.ncs < 1) l.na = 0;
    }
    return l;
}

}  // namespace grouped

size_t grouped_workspace_bytes(int T, int H, int I, int E, int k, int S) {
    if (T < 1 || H < 64 || I < 64 || E < 1 || E > TF_MAX_E || k < 1 || k > TF_MAX_K || S < 0) return 0;
    return grouped::carve(T, H, I, E, k, S).total;
}

tf_status grouped_run(const GroupedArgs& a, void* stream, const char* fn) {
    using namespace grouped;
    const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k, S = a.S;
    const tf_expert_table* table = a.table;
    if (!a.x || !a.out || (!table && !a.waves) || !a.idx || !a.w || !a.ws)
        return fail(TF_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (a.x == a.out) return fail(TF_ERR_INVALID_ARG, "%s: out must not alias x", fn);
    if (T < 1) return fail(TF_ERR_INVALID_ARG, "%s: T=%d", fn, T);
    if (H % 128 || I % 64 || H > 2816 || H < 128 || I < 64)
        return fail(TF_ERR_INVALID_ARG, "%s: H must be a multiple of 128 (<= 2816) and I a multiple of 64 (H=%d I=%d)",
                    fn, H, I);
    if (E < 1 || E > TF_MAX_E || k < 1 || k > TF_MAX_K || k > E)
        return fail(TF_ERR_INVALID_ARG, "%s: E=%d k=%d out of range", fn, E, k);
    if (S < 0 || S % 64 || (S > 0 && (!a.Wsg || !a.Wsu || !a.Wsd)))
        return fail(TF_ERR_INVALID_ARG, "%s: the shared expert needs S a multiple of 64 and three weights (S=%d)", fn,
                    S);
    if (S > 0 && (!aligned16(a.Wsg) || !aligned16(a.Wsu) || !aligned16(a.Wsd)))
        return fail(TF_ERR_INVALID_ARG, "%s: shared weights must be 16-byte aligned", fn);
    if (a.waves) {
        if (!a.waves->pool || !aligned16(a.waves->pool) || a.waves->slot_bytes % 16 || a.waves->n_slots < 1 ||
            !a.waves->d_maps || !a.waves->h_maps || !a.waves->before_wave || a.waves->n < 0)
            return fail(TF_ERR_INVALID_ARG, "%s: bad cache waves", fn);
    } else {
        if (!table->base || !aligned16(table->base) || table->stride % 16)
            return fail(TF_ERR_INVALID_ARG, "%s: expert table base and stride must be 16-byte aligned", fn);
        if (table->slot_of_expert)
            return fail(TF_ERR_NOT_SUPPORTED, "%s: the grouped path takes a resident expert table (no slot map)", fn);
        if (table->n_experts != 0 && table->n_experts != E)
            return fail(TF_ERR_INVALID_ARG, "%s: the expert table's n_experts (%d) is not E (%d)", fn,
                        table->n_experts, E);
    }
    if (!aligned16(a.x) || !aligned16(a.out) || (a.delta && !aligned16(a.delta)))
        return fail(TF_ERR_INVALID_ARG, "%s: x, out and delta must be 16-byte aligned", fn);
    if ((size_t)T * k > (size_t)INT32_MAX / 4) return fail(TF_ERR_INVALID_ARG, "%s: T*k too large", fn);
    const Carve c = carve(T, H, I, E, k, S);
    if (a.ws_bytes < c.total || (reinterpret_cast<uintptr_t>(a.ws) & 255))
        return fail(TF_ERR_INVALID_ARG, "%s: workspace misaligned or smaller than %zu bytes", fn, c.total);
    ExpertLayout lay;
    expert_layout(H, I, &lay);
    if ((a.waves ? a.waves->slot_bytes : table->stride) < lay.payload)
        return fail(TF_ERR_INVALID_ARG, "%s: expert stride below the payload size", fn);
    // the largest token tile of this call (an expert gets each token at most once) and the GEMMs' plans
    const int max_rows = T < NB ? T : NB;
    const Layout lay_gu = plan_layout(max_rows, false, H), lay_d = plan_layout(max_rows, false, I);
    const Layout lay_sgu = plan_layout(max_rows, true, H), lay_sd = plan_layout(max_rows, true, S > 0 ? S : 64);
    if (!lay_gu.na || !lay_d.na || !lay_sgu.na || !lay_sd.na)
        return fail(TF_ERR_INVALID_ARG, "%s: H=%d I=%d do not fit the GEMM's shared memory", fn, H, I);

    char* ws = static_cast<char*>(a.ws);
    uint32_t* err = reinterpret_cast<uint32_t*>(ws + c.err);
    int32_t* counts = reinterpret_cast<int32_t*>(ws + c.counts);
    int32_t* offsets = reinterpret_cast<int32_t*>(ws + c.offsets);
    int32_t* tiles_gu = reinterpret_cast<int32_t*>(ws + c.tiles_gu);
    int32_t* tiles_d = reinterpret_cast<int32_t*>(ws + c.tiles_d);
    int32_t* perm = reinterpret_cast<int32_t*>(ws + c.perm);
    int32_t* inv = reinterpret_cast<int32_t*>(ws + c.inv);
    float* rms = reinterpret_cast<float*>(ws + c.rms);
    float* rp = reinterpret_cast<float*>(ws + c.rp);
    uint16_t* xp = reinterpret_cast<uint16_t*>(ws + c.xp);
    uint16_t* hb = reinterpret_cast<uint16_t*>(ws + c.hb);
    float* y = reinterpret_cast<float*>(ws + c.y);
    int32_t* s_plan = S > 0 ? reinterpret_cast<int32_t*>(ws + c.s_plan) : nullptr;
    uint16_t* hs = S > 0 ? reinterpret_cast<uint16_t*>(ws + c.hs) : nullptr;
    float* ys = S > 0 ? reinterpret_cast<float*>(ws + c.ys) : nullptr;
    const int P = T * k;

    // tensor maps: codes of every expert (3-D; with waves, of every slot of the layer's cache), permuted
    // activations and h (2-D, SW128)
    CUtensorMap tmA_gu, tmA_d, tmB_gu, tmB_d;
    const char* base = a.waves ? a.waves->pool : static_cast<const char*>(table->base);
    const size_t estride = a.waves ? a.waves->slot_bytes : table->stride;
    const int n_units = a.waves ? a.waves->n_slots : E;    // the 3rd dimension of the code maps
    {
        cuuint64_t dims[3] = {(cuuint64_t)H / 2, (cuuint64_t)2 * I, (cuuint64_t)n_units};
        cuuint64_t str[2] = {(cuuint64_t)H / 2, (cuuint64_t)estride};
        cuuint32_t box[3] = {CW * BK / 2, BM, 1};
        if (!encode(&tmA_gu, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base + lay.gu_codes, dims, str, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return fail(TF_ERR_CUDA, "%s: tensor map of the gate/up codes", fn);
    }
    {
        cuuint64_t dims[3] = {(cuuint64_t)I / 2, (cuuint64_t)H, (cuuint64_t)n_units};
        cuuint64_t str[2] = {(cuuint64_t)I / 2, (cuuint64_t)estride};
        cuuint32_t box[3] = {CW * BK / 2, BM, 1};
        if (!encode(&tmA_d, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base + lay.d_codes, dims, str, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return fail(TF_ERR_CUDA, "%s: tensor map of the down codes", fn);
    }
    CUtensorMap tmB_gu2, tmB_d2;
    if (!encode_rows(&tmB_gu, xp, H, P, BOX_SMALL, true) || !encode_rows(&tmB_gu2, xp, H, P, BOX_BIG, true))
        return fail(TF_ERR_CUDA, "%s: tensor map of the permuted activations", fn);
    if (!encode_rows(&tmB_d, hb, I, P, BOX_SMALL) || !encode_rows(&tmB_d2, hb, I, P, BOX_BIG))
        return fail(TF_ERR_CUDA, "%s: tensor map of h", fn);
    // shared expert: bf16 weights as SW128 row boxes (8 rows for the interleaved gate/up tile, 128 for down)
    CUtensorMap tmS_g, tmS_u, tmS_d, tmS_xn, tmS_h, tmS_xn2, tmS_h2;
    if (S > 0) {
        if (!encode_rows(&tmS_g, a.Wsg, H, S, 8) || !encode_rows(&tmS_u, a.Wsu, H, S, 8) ||
            !encode_rows(&tmS_d, a.Wsd, S, H, BM) || !encode_rows(&tmS_xn, a.x, H, T, BOX_SMALL) ||
            !encode_rows(&tmS_h, hs, S, T, BOX_SMALL) || !encode_rows(&tmS_xn2, a.x, H, T, BOX_BIG) ||
            !encode_rows(&tmS_h2, hs, S, T, BOX_BIG))
            return fail(TF_ERR_CUDA, "%s: tensor maps of the shared expert", fn);
    }
    if (int e = smem_limit_once((const void*)k_group_gemm, (int)GEMM_SMEM)) return cuda_status(e, fn);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    clear_error();

    const int mt_gu = 2 * I / BM, mt_d = H / BM;
    const uint16_t* x16 = static_cast<const uint16_t*>(a.x);
    prof_before(TF_KERNEL_PERMUTE, stream);
    if (a.rms_in)
        rms = const_cast<float*>(a.rms_in);   // the router's scale of every token (the same canonical sum)
    else
        launch_dependent(k_group_rms, dim3((T + 7) / 8), dim3(256), 0, st, x16, T, H, a.eps, rms);
    launch_dependent(k_group_hist, dim3(1), dim3(1024), 0, st, a.idx, P, E, mt_gu, mt_d, counts, offsets, tiles_gu, tiles_d, err);
    launch_dependent(k_group_pos, dim3(E), dim3(1024), 0, st, a.idx, P, offsets, perm, inv);
    launch_dependent(k_group_inv_init, dim3((P + 255) / 256), dim3(256), 0, st, a.idx, P, E, inv);
    launch_dependent(k_group_gather, dim3((P + 7) / 8), dim3(256), 0, st, x16, rms, perm, P, k, H, xp, rp);
    // the shared expert has few weight tiles (2S/128 and H/128); while the tokens fit one tile row, split K
    // so that more SMs stream its weights (chunks of at least 4 stages)
    auto split_of = [](int kstages) {
        for (int c : {4, 3, 2})
            if (kstages % c == 0 && kstages / c >= 4) return c;
        return 1;
    };
    const bool one_block = T <= NB;
    const int ks_gu = (S > 0 && one_block) ? split_of(H / BK) : 1;
    const int ks_d = (S > 0 && one_block) ? split_of(S / BK) : 1;
    float* spart = S > 0 ? reinterpret_cast<float*>(ws + c.spart) : nullptr;
    if (S > 0) {
        launch_dependent(k_shared_plan, dim3(1), dim3(32), 0, st, T, 2 * S / BM, H / BM, ks_gu, ks_d, s_plan, s_plan + 1, s_plan + 3,
                                        s_plan + 5);
    }
    prof_after(TF_KERNEL_PERMUTE, stream);
    if (cudaError_t e = cudaGetLastError()) return cuda_status(e, fn);

    GemmParams gp;
    std::memset(&gp, 0, sizeof(gp));
    gp.ebase = base;
    gp.estride = estride;
    gp.E = E;
    gp.counts = counts;
    gp.offsets = offsets;
    gp.err = err;
    gp.ksplit = 1;
    gp.dep_limit_ns = test_wait_limit_ns();

    auto routed_gemms = [&](const int32_t* slot_of) {
        gp.slot_of = slot_of;
        gp.off_sb = lay.gu_sb;
        gp.K = H;
        gp.MT = mt_gu;
        gp.tiles = tiles_gu;
        gp.mode = 0;
        gp.hout = hb;
        gp.yout = nullptr;
        gp.ldo = I;
        gp.col_scale = rp;
        gp.f16 = 1;
        gp.lay = lay_gu;
        launch_dependent(k_group_gemm, dim3(sms), dim3(GEMM_THREADS), GEMM_SMEM, st, tmA_gu, tmB_gu, tmA_gu, tmB_gu2, gp);
        gp.off_sb = lay.d_sb;
        gp.K = I;
        gp.MT = mt_d;
        gp.tiles = tiles_d;
        gp.mode = 1;
        gp.hout = nullptr;
        gp.yout = y;
        gp.ldo = H;
        gp.f16 = 0;
        gp.lay = lay_d;
        launch_dependent(k_group_gemm, dim3(sms), dim3(GEMM_THREADS), GEMM_SMEM, st, tmA_d, tmB_d, tmA_d, tmB_d2, gp);
    };
    prof_before(TF_KERNEL_GEMM, stream);
    if (!a.waves) {
        routed_gemms(nullptr);
    } else {
        // the chunk's experts in waves: each wave's fills, its slot map, its tile plan, then its GEMMs
        const GroupedWaves& wv = *a.waves;
        for (int w = 0; w < wv.n; ++w) {
            if (int s = wv.before_wave(wv.ctx, w, stream)) return s;
            int32_t* dmap = wv.d_maps + (size_t)w * 2 * E;
            if (cudaError_t e = cudaMemcpyAsync(dmap, wv.h_maps + (size_t)w * 2 * E, (size_t)2 * E * 4,
                                                cudaMemcpyHostToDevice, st))
                return cuda_status(e, fn);
            launch_dependent(k_wave_plan, dim3(1), dim3(1024), 0, st, counts, dmap, E, mt_gu, mt_d, tiles_gu, tiles_d);
            routed_gemms(dmap + E);
        }
    }
    if (S > 0) {
        GemmParams sp;
        std::memset(&sp, 0, sizeof(sp));
        sp.E = 1;
        sp.counts = s_plan;
        sp.offsets = s_plan + 1;
        sp.err = err;
        sp.dep_limit_ns = gp.dep_limit_ns;
        sp.a_bf16 = 1;
        sp.pair_log2 = 3;
        sp.ntok = T;
        sp.part = spart;
        sp.K = H;
        sp.MT = 2 * S / BM;
        sp.tiles = s_plan + 3;
        sp.mode = 0;
        sp.hout = hs;
        sp.ldo = S;
        sp.col_scale = rms;          // the shared expert's token rows are the tokens in order
        sp.ksplit = ks_gu;
        sp.mrows = 2 * S;
        sp.lay = lay_sgu;
        launch_dependent(k_group_gemm, dim3(sms), dim3(GEMM_THREADS), GEMM_SMEM, st, tmS_g, tmS_xn, tmS_u, tmS_xn2, sp);
        if (ks_gu > 1) launch_dependent(k_shared_gu_combine, dim3(dim3((S + 255) / 256, T)), dim3(256), 0, st, spart, rms, ks_gu, T, S, hs);
        sp.K = S;
        sp.MT = H / BM;
        sp.tiles = s_plan + 5;
        sp.mode = 1;
        sp.hout = nullptr;
        sp.yout = ys;
        sp.ldo = H;
        sp.ksplit = ks_d;
        sp.mrows = H;
        sp.lay = lay_sd;
        launch_dependent(k_group_gemm, dim3(sms), dim3(GEMM_THREADS), GEMM_SMEM, st, tmS_d, tmS_h, tmS_d, tmS_h2, sp);
        if (ks_d > 1) launch_dependent(k_shared_down_combine, dim3(dim3((H + 255) / 256, T)), dim3(256), 0, st, spart, ks_d, T, H, ys);
    }
    prof_after(TF_KERNEL_GEMM, stream);
    if (cudaError_t e = cudaGetLastError()) return cuda_status(e, fn);

    prof_before(TF_KERNEL_COMBINE, stream);
    launch_dependent(k_group_combine, dim3(dim3((H / 4 + 127) / 128, T)), dim3(128), 0, st, x16, y, ys, inv, a.w, k, H, err,
                                                                  static_cast<uint16_t*>(a.out), a.delta);
    prof_after(TF_KERNEL_COMBINE, stream);
    if (a.perm_out) cudaMemcpyAsync(a.perm_out, perm, (size_t)P * 4, cudaMemcpyDeviceToDevice, st);
    if (a.counts_out) cudaMemcpyAsync(a.counts_out, counts, (size_t)E * 4, cudaMemcpyDeviceToDevice, st);
    return cuda_status(cudaGetLastError(), fn);
}

}  // namespace tf

extern "C" {

size_t tf_moe_grouped_workspace_bytes(int T, int H, int I, int E, int k) {
    return tf::grouped_workspace_bytes(T, H, I, E, k, 0);
}

tf_status tf_moe_ffn_grouped(const void* x, void* out, int T, const tf_expert_table* table, int E, const int32_t* idx,
                             const float* w, int k, int H, int I, float* delta, int32_t* perm_out, int32_t* counts_out,
                             void* workspace, size_t ws_bytes, void* stream) {
    tf::GroupedArgs a;
    std::memset(&a, 0, sizeof(a));
    a.x = x;
    a.out = out;
    a.T = T;
    a.table = table;
    a.E = E;
    a.k = k;
    a.H = H;
    a.I = I;
    a.idx = idx;
    a.w = w;
    a.delta = delta;
    a.perm_out = perm_out;
    a.counts_out = counts_out;
    a.S = 0;
    a.eps = 1e-6f;
    a.ws = workspace;
    a.ws_bytes = ws_bytes;
    return tf::grouped_run(a, stream, "tf_moe_ffn_grouped");
}

}  // extern "C"
