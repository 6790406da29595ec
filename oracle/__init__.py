"""CPU oracle for the streamed-expert MoE layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product (the CUDA library and its
binding) never does, and the oracle shares no code with it: both sides are fed
by the seeded generators in ``workload/`` and nothing else.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, built twice:
fp32 and fp64, and once more as fp32 with OpenMP over its independent output
rows, which gives bit-identical results and is used only to time the oracle on
all host cores); this module only loads it and marshals numpy arrays.

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
closed forms, brute force, hand-written traces and the pages' fixed facts.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
EPS = 1e-6
K_ACTIVE = 8


def _lib_path(bits: int, mt: bool = False) -> str:
    return os.path.join(_HERE, "liboracle%d%s.so" % (bits, "mt" if mt else ""))


def build(force: bool = False) -> None:
    """Compile the fp32 and fp64 oracles (-O2, no FMA contraction, no fast-math, SSE2), and the fp32 oracle
    once more with OpenMP over its independent output rows (bit-identical results, for timing on all cores)."""
    for bits, mt, defs in ((32, False, ["-DREAL=float", "-DREAL_IS_DOUBLE=0"]),
                           (64, False, ["-DREAL=double", "-DREAL_IS_DOUBLE=1"]),
                           (32, True, ["-DREAL=float", "-DREAL_IS_DOUBLE=0", "-fopenmp"])):
        out = _lib_path(bits, mt)
        if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
            tmp = out + ".tmp%d" % os.getpid()
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                                   "-fno-fast-math", "-msse2", "-mfpmath=sse", *defs, "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, out)


class Expert(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p * 3), ("s", ctypes.c_void_p * 3), ("b", ctypes.c_void_p * 3)]


class CacheEvent(ctypes.Structure):
    _fields_ = [("step", ctypes.c_int32), ("layer", ctypes.c_int32), ("expert", ctypes.c_int32),
                ("hit", ctypes.c_int32), ("slot", ctypes.c_int32), ("evicted", ctypes.c_int32)]


_libs: dict = {}


def lib(bits: int = 32, mt: bool = False):
    """The fp32 (bits = 32) or fp64 oracle; mt = True: the fp32 build whose row loops use all cores."""
    key = (bits, mt)
    if key not in _libs:
        build()
        L = ctypes.CDLL(_lib_path(bits, mt))
        R = ctypes.c_float if bits == 32 else ctypes.c_double
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        L.or_half_to_float.restype = ctypes.c_float
        L.or_half_to_float.argtypes = [ctypes.c_uint16]
        L.or_bf16_to_float.restype = ctypes.c_float
        L.or_bf16_to_float.argtypes = [ctypes.c_uint16]
        L.or_float_to_bf16.restype = ctypes.c_uint16
        L.or_float_to_bf16.argtypes = [ctypes.c_float]
        L.or_float_to_half.restype = ctypes.c_uint16
        L.or_float_to_half.argtypes = [ctypes.c_float]
        L.or_rms_scale.restype = R
        L.or_rms_scale.argtypes = [vp, i32, ctypes.c_double]
        L.or_normalise.argtypes = [vp, i32, R, vp]
        L.or_router_logits.argtypes = [vp, i32, vp, i32, vp, R, vp]
        L.or_topk.argtypes = [vp, i32, i32, vp]
        L.or_softmax_selected.argtypes = [vp, vp, i32, vp]
        L.or_dequant.restype = R
        L.or_dequant.argtypes = [ctypes.c_uint8, ctypes.c_uint16, ctypes.c_uint16]
        L.or_dequant_matrix.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        L.or_gelu.restype = R
        L.or_gelu.argtypes = [R]
        L.or_expert_ffn.argtypes = [vp, i32, i32, ctypes.POINTER(Expert), i32, i32, R, vp]
        L.or_shared_ffn.argtypes = [vp, i32, i32, vp, vp, vp, i32, R, vp]
        L.or_route.argtypes = [vp, i32, vp, i32, vp, i32, ctypes.c_double, ctypes.POINTER(R), vp, vp, vp]
        L.or_layer_combine.argtypes = [vp, i32, i32, R, i32, ctypes.POINTER(Expert), vp, i32, vp, vp, vp,
                                       i32, vp, vp]
        L.or_lfu_new.restype = vp
        L.or_lfu_new.argtypes = [i32, i32]
        L.or_lfu_free.argtypes = [vp]
        L.or_lfu_step.restype = i32
        L.or_lfu_step.argtypes = [vp, i32, i32, vp, i32, ctypes.POINTER(CacheEvent)]
        L.or_lfu_state.argtypes = [vp, i32, vp, vp, vp]
        L.or_attn_decode.argtypes = [vp, i32, i32, i32, i32, ctypes.c_double, ctypes.c_double, i32, vp, vp, vp, vp,
                                     vp, vp, vp, vp, vp]
        L.or_real_bytes.restype = i32
        L.or_threads.restype = i32
        _libs[key] = L
    return _libs[key]


def threads(mt: bool = True) -> int:
    """Threads the row loops of the oracle build use (1 for the plain build)."""
    return lib(32, mt).or_threads()


def _dt(bits):
    return np.float32 if bits == 32 else np.float64


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ------------------------------------------------------------------------ scalar pieces

def half_to_float(h: int) -> float:
    return lib().or_half_to_float(h)


def float_to_bf16(f: float) -> int:
    return lib().or_float_to_bf16(f)


def float_to_half(f: float) -> int:
    return lib().or_float_to_half(f)


FMT = {"fp32": 0, "bf16": 1, "fp16": 2}   # operand formats of the FFN readings (rounding before products)


def gelu(v: float, bits: int = 32) -> float:
    return lib(bits).or_gelu(v)


def dequant(q: int, s: int, b: int, bits: int = 32) -> float:
    return lib(bits).or_dequant(q, s, b)


def dequant_matrix(q, s, b, fmt: str = "fp32", bits: int = 32) -> np.ndarray:
    R, K = q.shape
    q, qp = _c(q, np.uint8)
    s, sp = _c(s, np.uint16)
    b, bp = _c(b, np.uint16)
    W = np.empty((R, K), _dt(bits))
    lib(bits).or_dequant_matrix(qp, sp, bp, R, K, FMT[fmt], W.ctypes.data)
    return W


# ----------------------------------------------------------------------------- routing

def rms_scale(x, bits: int = 32, eps: float = EPS) -> float:
    x, xp = _c(x, np.uint16)
    return lib(bits).or_rms_scale(xp, x.shape[-1], eps)


def normalise(x, r, bits: int = 32) -> np.ndarray:
    x, xp = _c(x, np.uint16)
    n = np.empty(x.shape[-1], _dt(bits))
    lib(bits).or_normalise(xp, x.shape[-1], r, n.ctypes.data)
    return n


def router_logits(x, Wr, bias=None, r=None, bits: int = 32) -> np.ndarray:
    x, xp = _c(x, np.uint16)
    Wr, wp = _c(Wr, np.uint16)
    E, H = Wr.shape
    if r is None:
        r = rms_scale(x, bits)
    bp = None
    if bias is not None:
        bias, bp = _c(bias, np.float32)
    z = np.empty(E, _dt(bits))
    lib(bits).or_router_logits(xp, H, wp, E, bp, r, z.ctypes.data)
    return z


def topk(z, k: int = K_ACTIVE, bits: int = 32) -> np.ndarray:
    z, zp = _c(z, _dt(bits))
    idx = np.empty(k, np.int32)
    lib(bits).or_topk(zp, z.shape[0], k, idx.ctypes.data)
    return idx


def softmax_selected(z, idx, bits: int = 32) -> np.ndarray:
    z, zp = _c(z, _dt(bits))
    idx, ip = _c(idx, np.int32)
    w = np.empty(idx.shape[0], _dt(bits))
    lib(bits).or_softmax_selected(zp, ip, idx.shape[0], w.ctypes.data)
    return w


def route(x, Wr, bias=None, k: int = K_ACTIVE, bits: int = 32, eps: float = EPS, mt: bool = False):
    """One token's routing -> (r, z[E], idx[k] best first, w[k])."""
    x, xp = _c(x, np.uint16)
    Wr, wp = _c(Wr, np.uint16)
    E, H = Wr.shape
    bp = None
    if bias is not None:
        bias, bp = _c(bias, np.float32)
    R = ctypes.c_float if bits == 32 else ctypes.c_double
    r = R()
    z = np.empty(E, _dt(bits))
    idx = np.empty(k, np.int32)
    w = np.empty(k, _dt(bits))
    lib(bits, mt).or_route(xp, H, wp, E, bp, k, eps, ctypes.byref(r), z.ctypes.data, idx.ctypes.data,
                           w.ctypes.data)
    return r.value, z, idx, w


# --------------------------------------------------------------------------------- FFN

def _expert_struct(ex: dict, keep: list) -> Expert:
    st = Expert()
    for m, name in enumerate(("gate", "up", "down")):
        q, s, b = ex[name]
        q, qp = _c(q, np.uint8)
        s, sp = _c(s, np.uint16)
        b, bp = _c(b, np.uint16)
        keep += [q, s, b]
        st.q[m], st.s[m], st.b[m] = qp, sp, bp
    return st


def expert_ffn(n, ex: dict, fmt: str = "fp32", bits: int = 32, in_scale: float = 1.0,
               fmt_down: str | None = None) -> np.ndarray:
    """y = Wd (gelu(c Wg n) * (c Wu n)), c = in_scale, for one logical expert (see workload.expert); fmt rounds
    Wg, Wu and n, fmt_down (default: fmt) rounds Wd and h before their products."""
    n, np_ = _c(n, _dt(bits))
    I, H = ex["gate"][0].shape
    keep: list = []
    st = _expert_struct(ex, keep)
    y = np.empty(H, _dt(bits))
    lib(bits).or_expert_ffn(np_, H, I, ctypes.byref(st), FMT[fmt], FMT[fmt_down or fmt], in_scale, y.ctypes.data)
    return y


def shared_ffn(n, Wg, Wu, Wd, fmt: str = "fp32", bits: int = 32, in_scale: float = 1.0) -> np.ndarray:
    n, np_ = _c(n, _dt(bits))
    S, H = Wg.shape
    Wg, gp = _c(Wg, np.uint16)
    Wu, up = _c(Wu, np.uint16)
    Wd, dp = _c(Wd, np.uint16)
    y = np.empty(H, _dt(bits))
    lib(bits).or_shared_ffn(np_, H, S, gp, up, dp, FMT[fmt], in_scale, y.ctypes.data)
    return y


def layer_combine(x, r, experts: list, w, shared=None, tc: bool = False, bits: int = 32, mt: bool = False):
    """out = bf16(x + delta), delta = shared + sum_i w_i y_i (experts given in top-k order). tc = True is the
    tensor-core reading (x fed as it is, r applied after the gate/up dot products; fp16 operands for the routed
    experts' gate/up with x scaled by the power of two of r, bf16 for their down and for the shared expert).

    Returns (out bf16 bits [H], delta [H])."""
    x, xp = _c(x, np.uint16)
    H = x.shape[0]
    k = len(experts)
    I = experts[0]["gate"][0].shape[0] if k else 0
    keep: list = []
    arr = (Expert * max(k, 1))()
    for i, ex in enumerate(experts):
        arr[i] = _expert_struct(ex, keep)
    w, wp = _c(w, _dt(bits))
    S, gp, up, dp = 0, None, None, None
    if shared is not None:
        Wg, Wu, Wd = shared
        S = Wg.shape[0]
        Wg, gp = _c(Wg, np.uint16)
        Wu, up = _c(Wu, np.uint16)
        Wd, dp = _c(Wd, np.uint16)
    out = np.empty(H, np.uint16)
    delta = np.empty(H, _dt(bits))
    lib(bits, mt).or_layer_combine(xp, H, I, r, k, arr, wp, S, gp, up, dp, int(tc), out.ctypes.data,
                                   delta.ctypes.data)
    return out, delta


# --------------------------------------------------------------------------------- LFU

class LFU:
    """Per-layer LFU expert-cache simulator (events are (step, layer, expert, hit, slot, evicted))."""

    def __init__(self, n_layers: int, n_slots: int):
        self._L = lib()
        self._h = self._L.or_lfu_new(n_layers, n_slots)
        self.n_slots = n_slots

    def step(self, step: int, layer: int, ids) -> list:
        ids, ip = _c(ids, np.int32)
        ev = (CacheEvent * max(1, ids.shape[0]))()
        rc = self._L.or_lfu_step(self._h, step, layer, ip, ids.shape[0], ev)
        if rc < 0:
            raise ValueError("no evictable slot")
        return [(e.step, e.layer, e.expert, e.hit, e.slot, e.evicted) for e in ev[:ids.shape[0]]]

    def state(self, layer: int):
        S = self.n_slots
        ex = np.empty(S, np.int32)
        cnt = np.empty(S, np.int64)
        lu = np.empty(S, np.int64)
        self._L.or_lfu_state(self._h, layer, ex.ctypes.data, cnt.ctypes.data, lu.ctypes.data)
        return ex, cnt, lu

    def __del__(self):
        try:
            self._L.or_lfu_free(self._h)
        except Exception:
            pass


# ------------------------------------------------------------------------ attention

def attn_decode(x, pos: int, Wq, Wk, Wv, Wo, k_cache, v_cache, nq: int, nkv: int, d: int,
                theta: float = 10000.0, eps: float = EPS, bits: int = 64):
    """Attention half of a decoder layer for one token at position pos (see or_attn_decode).

    x: bf16 bits [H]; W*: bf16 bits, Wq [nq*d, H], Wk/Wv [nkv*d, H], Wo [H, nq*d]; k_cache, v_cache: fp16
    bits [max_seq, nkv, d] (uint16 arrays, updated in place at row pos). Returns (out bf16 bits [H],
    scores of q head 0 [pos + 1], attention output a [nq*d])."""
    H = int(np.asarray(x).size)
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
    assert k_cache.size >= (pos + 1) * nkv * d and v_cache.size >= (pos + 1) * nkv * d
    xa, xp = _c(x, np.uint16)
    ws = [_c(w, np.uint16) for w in (Wq, Wk, Wv, Wo)]
    assert ws[0][0].size == nq * d * H and ws[1][0].size == nkv * d * H and ws[2][0].size == nkv * d * H
    assert ws[3][0].size == H * nq * d
    dt = _dt(bits)
    out = np.zeros(H, dtype=np.uint16)
    sc = np.zeros(pos + 1, dtype=dt)
    a = np.zeros(nq * d, dtype=dt)
    lib(bits).or_attn_decode(xp, H, nq, nkv, d, float(eps), float(theta), int(pos), ws[0][1], ws[1][1], ws[2][1],
                             ws[3][1], k_cache.ctypes.data, v_cache.ctypes.data, out.ctypes.data, sc.ctypes.data,
                             a.ctypes.data)
    return out, sc, a
