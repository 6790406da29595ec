"""Seeded synthetic inputs for the streamed-expert MoE layer (shared by the
oracle, the tests and the benchmark).

Nothing here computes any part of the layer: the functions draw SplitMix64
random numbers (counter-based, so every element can be produced on its own)
and encode them in the layer's input formats: bf16 hidden states and dense
weights, 4-bit expert codes with fp16 per-group scale and bias, and Zipf
router-logit biases.

Every draw is keyed by (seed, tensor, layer, expert, matrix); see gen.c for
the exact definitions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libtfgen.so")

# tensor ids absorbed into every stream key
T_X = 1          # hidden states
T_WR = 2         # router weights
T_Q = 3          # expert 4-bit codes
T_S = 4          # expert fp16 scales
T_B = 5          # expert fp16 biases
T_SH = 6         # shared-expert bf16 weights (matrix 0 gate, 1 up, 2 down)
T_ZIPF = 7       # Zipf rank -> expert permutation
T_COIN = 8       # per-(step, layer) coin of the repeat-previous-top-k workload
T_NOISE = 9      # per-(step, layer) router-logit noise of the streaming workload
T_ATTN = 10      # attention weights (matrix 0 q, 1 k, 2 v, 3 o) and synthetic cache contents (matrix 4 k, 5 v)

GATE, UP, DOWN = 0, 1, 2
GROUP = 64

SCALE_LO, SCALE_HI = 0.005, 0.02
BIAS_LO, BIAS_HI = -0.08, 0.08
ROUTER_SIGMA = 0.02
SHARED_SIGMA = 0.02


def build(force: bool = False) -> str:
    """Compile gen.c into libtfgen.so (plain C, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, u16p, u8p, i32p, f32p = (ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint16),
                                       ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_float))
        L.wl_key.restype = u64
        L.wl_key.argtypes = [u64] * 5
        L.wl_u64.restype = u64
        L.wl_u64.argtypes = [u64, u64]
        L.wl_unif53.restype = ctypes.c_double
        L.wl_unif53.argtypes = [u64, u64]
        L.wl_normal_bf16.argtypes = [u64, u64, ctypes.c_double, u16p]
        L.wl_normal_f32.argtypes = [u64, u64, ctypes.c_double, f32p]
        L.wl_uniform_f16.argtypes = [u64, u64, ctypes.c_double, ctypes.c_double, u16p]
        L.wl_codes.argtypes = [u64, u64, u8p]
        L.wl_permutation.argtypes = [u64, ctypes.c_int32, i32p]
        L.wl_zipf_bias.argtypes = [u64, ctypes.c_int32, ctypes.c_double, ctypes.c_double, f32p, i32p]
        L.wl_f32_to_bf16.restype = ctypes.c_uint16
        L.wl_f32_to_bf16.argtypes = [ctypes.c_float]
        L.wl_f32_to_f16.restype = ctypes.c_uint16
        L.wl_f32_to_f16.argtypes = [ctypes.c_float]
        _lib = L
    return _lib


def _p(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def key(seed, tensor, layer=0, expert=0, matrix=0) -> int:
    return lib().wl_key(seed, tensor, layer, expert, matrix)


def normal_bf16(k: int, n: int, sigma: float, out: np.ndarray | None = None) -> np.ndarray:
    out = np.empty(n, np.uint16) if out is None else out
    lib().wl_normal_bf16(k, n, sigma, _p(out, ctypes.c_uint16))
    return out


def uniform_f16(k: int, n: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(n, np.uint16)
    lib().wl_uniform_f16(k, n, lo, hi, _p(out, ctypes.c_uint16))
    return out


def codes(k: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint8)
    lib().wl_codes(k, n, _p(out, ctypes.c_uint8))
    return out


def permutation(k: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    lib().wl_permutation(k, n, _p(out, ctypes.c_int32))
    return out


def zipf_bias(seed: int, layer: int, E: int, s: float, alpha: float = 1.0):
    """Zipf(s) popularity bias over E experts for one layer -> (bias[E] f32, rank->expert perm)."""
    bias = np.empty(E, np.float32)
    perm = np.empty(E, np.int32)
    lib().wl_zipf_bias(key(seed, T_ZIPF, layer), E, s, alpha, _p(bias, ctypes.c_float), _p(perm, ctypes.c_int32))
    return bias, perm


def coin(seed: int, layer: int, step: int) -> bool:
    """Fair coin for (step, layer) of the repeat-previous-top-k workload."""
    return lib().wl_unif53(key(seed, T_COIN, layer), step) < 0.5


def route_noise(seed: int, layer: int, step: int, E: int, sigma: float) -> np.ndarray:
    """N(0, sigma) per expert for (step, layer), as float32 (bf16-rounded values): the token-dependent part of the
    router logits in the streaming workload."""
    bits = normal_bf16(key(seed, T_NOISE, layer, step), E, sigma)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def hidden(seed: int, step: int, T: int, H: int) -> np.ndarray:
    """x ~ N(0,1) as bf16 bits, shape [T, H]."""
    return normal_bf16(key(seed, T_X, step), T * H, 1.0).reshape(T, H)


def router_weights(seed: int, layer: int, E: int, H: int) -> np.ndarray:
    """W_r ~ N(0, 0.02) as bf16 bits, [E, H] row-major."""
    return normal_bf16(key(seed, T_WR, layer), E * H, ROUTER_SIGMA).reshape(E, H)


def shared_weights(seed: int, layer: int, H: int, S: int):
    """Dense shared-expert FFN ~ N(0, 0.02) bf16 bits: gate [S,H], up [S,H], down [H,S]."""
    g = normal_bf16(key(seed, T_SH, layer, 0, GATE), S * H, SHARED_SIGMA).reshape(S, H)
    u = normal_bf16(key(seed, T_SH, layer, 0, UP), S * H, SHARED_SIGMA).reshape(S, H)
    d = normal_bf16(key(seed, T_SH, layer, 0, DOWN), H * S, SHARED_SIGMA).reshape(H, S)
    return g, u, d


def attention_weights(seed: int, layer: int, H: int, nq: int, nkv: int, d: int):
    """Attention projections as bf16 bits: Wq [nq*d, H], Wk, Wv [nkv*d, H] ~ N(0, 1/sqrt(H)),
    Wo [H, nq*d] ~ N(0, 0.5/sqrt(nq*d))."""
    sq, so = float(H) ** -0.5, 0.5 * float(nq * d) ** -0.5
    q = normal_bf16(key(seed, T_ATTN, layer, 0, 0), nq * d * H, sq).reshape(nq * d, H)
    k = normal_bf16(key(seed, T_ATTN, layer, 0, 1), nkv * d * H, sq).reshape(nkv * d, H)
    v = normal_bf16(key(seed, T_ATTN, layer, 0, 2), nkv * d * H, sq).reshape(nkv * d, H)
    o = normal_bf16(key(seed, T_ATTN, layer, 0, 3), H * nq * d, so).reshape(H, nq * d)
    return q, k, v, o


def cache_rows(seed: int, layer: int, rows: int, nkv: int, d: int):
    """Synthetic contents of the first `rows` rows of an fp16 K and V cache, ~ N(0, 1) (k) and N(0, 0.5) (v),
    as fp16 bits [rows, nkv, d] (drawn as bf16 values, which fp16 holds exactly in this range)."""
    out = []
    for m, sigma in ((4, 1.0), (5, 0.5)):
        b = normal_bf16(key(seed, T_ATTN, layer, 0, m), rows * nkv * d, sigma)
        f = np.clip((b.astype(np.uint32) << 16).view(np.float32), -60000.0, 60000.0)
        out.append(f.astype(np.float16).view(np.uint16).reshape(rows, nkv, d))
    return out[0], out[1]


def expert_matrix(seed: int, layer: int, expert: int, matrix: int, R: int, K: int):
    """Logical int4 affine matrix [R, K]: codes q in 0..15 (uint8), fp16 bits of the
    per-(row, 64-column group) scale s ~ U(0.005, 0.02) and bias b ~ U(-0.08, 0.08)."""
    assert K % GROUP == 0
    q = codes(key(seed, T_Q, layer, expert, matrix), R * K).reshape(R, K)
    s = uniform_f16(key(seed, T_S, layer, expert, matrix), R * (K // GROUP), SCALE_LO, SCALE_HI).reshape(R, K // GROUP)
    b = uniform_f16(key(seed, T_B, layer, expert, matrix), R * (K // GROUP), BIAS_LO, BIAS_HI).reshape(R, K // GROUP)
    return q, s, b


def expert(seed: int, layer: int, e: int, H: int, I: int) -> dict:
    """All three matrices of one expert: gate [I,H], up [I,H], down [H,I]."""
    out = {}
    for m, name, (R, K) in ((GATE, "gate", (I, H)), (UP, "up", (I, H)), (DOWN, "down", (H, I))):
        out[name] = expert_matrix(seed, layer, e, m, R, K)
    return out


def experts_parallel(seed: int, layer: int, ids, H: int, I: int, workers: int | None = None):
    """Generate several experts on a thread pool (the C calls release the GIL)."""
    workers = workers or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(workers) as ex:
        return list(ex.map(lambda e: expert(seed, layer, int(e), H, I), ids))


# --- encodings used by tests to read the generated bits back -------------------------------

def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)


def f16_to_f32(a: np.ndarray) -> np.ndarray:
    return a.view(np.float16).astype(np.float32)
