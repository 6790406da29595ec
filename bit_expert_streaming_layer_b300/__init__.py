"""Python binding of libtf.so, the B300 (sm_103a) streamed-expert MoE layer.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. PyTorch supplies device / pinned memory and streams. The functions
keep the C names (``tf_*``); tensors are passed by ``data_ptr()``, streams as
``torch.cuda.Stream`` (default: the current stream). A non-OK status raises
``TFError`` carrying the library's message.

There is no fallback: if libtf.so is missing the import fails.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtf.so")

TF_OK, TF_ERR_INVALID_ARG, TF_ERR_CUDA, TF_ERR_OOM, TF_ERR_TIMEOUT, TF_ERR_NOT_SUPPORTED = range(6)
TF_GROUP, TF_MAX_K, TF_MAX_E = 64, 32, 1024


class TFError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__("%s -> %s: %s" % (fn, _STATUS.get(status, status), msg))
        self.status = status


_STATUS = {0: "TF_OK", 1: "TF_ERR_INVALID_ARG", 2: "TF_ERR_CUDA", 3: "TF_ERR_OOM", 4: "TF_ERR_TIMEOUT",
           5: "TF_ERR_NOT_SUPPORTED"}


class ExpertTable(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("stride", ctypes.c_size_t), ("slot_of_expert", ctypes.c_void_p),
                ("n_experts", ctypes.c_int32), ("n_slots", ctypes.c_int32)]


class CacheEvent(ctypes.Structure):
    _fields_ = [("step", ctypes.c_int32), ("layer", ctypes.c_int32), ("expert", ctypes.c_int32),
                ("hit", ctypes.c_int32), ("slot", ctypes.c_int32), ("evicted", ctypes.c_int32)]


class LayerDesc(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("S", ctypes.c_int), ("eps", ctypes.c_float), ("W_r", ctypes.c_void_p), ("W_sg", ctypes.c_void_p),
                ("W_su", ctypes.c_void_p), ("W_sd", ctypes.c_void_p), ("experts", ExpertTable)]


class StepStats(ctypes.Structure):
    _fields_ = [("hits", ctypes.c_int32), ("misses", ctypes.c_int32), ("bytes_fetched", ctypes.c_uint64),
                ("copy_ms", ctypes.c_float), ("shared_ms", ctypes.c_float), ("stall_ms", ctypes.c_float),
                ("ids", ctypes.c_int32 * TF_MAX_K)]


class PrefillStats(ctypes.Structure):
    _fields_ = [("waves", ctypes.c_int32), ("hits", ctypes.c_int32), ("misses", ctypes.c_int32),
                ("bytes_fetched", ctypes.c_uint64)]


class AttnDesc(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("max_seq", ctypes.c_int), ("eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("W_q", ctypes.c_void_p), ("W_k", ctypes.c_void_p),
                ("W_v", ctypes.c_void_p), ("W_o", ctypes.c_void_p)]


# exported symbols and their C signatures (restype, argtypes)
_vp, _i32, _i64, _sz, _f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_S = ctypes.c_int32
SIGNATURES = {
    "tf_last_error": (ctypes.c_char_p, []),
    "tf_status_string": (ctypes.c_char_p, [_S]),
    "tf_version": (ctypes.c_char_p, []),
    "tf_struct_bytes": (_sz, [_i32]),
    "tf_expert_payload_bytes": (_sz, [_i32, _i32]),
    "tf_expert_slot_bytes": (_sz, [_i32, _i32]),
    "tf_expert_offsets": (_S, [_i32, _i32, _vp]),
    "tf_pack_expert": (_S, [_vp, _vp, _vp, _i32, _i32, _vp]),
    "tf_router_workspace_bytes": (_sz, [_i32, _i32]),
    "tf_router_topk": (_S, [_vp, _i32, _i32, _vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "tf_dequant_expert": (_S, [_vp, _i32, _i32, _i32, _i32, _vp, _vp]),
    "tf_moe_decode_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "tf_moe_ffn_decode": (_S, [_vp, _vp, ctypes.POINTER(ExpertTable), _vp, _vp, _i32, _i32, _i32, _vp, _vp, _sz,
                               _vp]),
    "tf_moe_ffn_decode_noalloc": (_S, [_vp, _vp, ctypes.POINTER(ExpertTable), _vp, _vp, _i32, _i32, _i32, _vp, _vp]),
    "tf_moe_grouped_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "tf_moe_ffn_grouped": (_S, [_vp, _vp, _i32, ctypes.POINTER(ExpertTable), _i32, _vp, _vp, _i32, _i32, _i32, _vp,
                                _vp, _vp, _vp, _sz, _vp]),
    "tf_expert_cache_create": (_S, [_i32, _i32, _i32, _sz, _vp, ctypes.POINTER(_vp)]),
    "tf_expert_cache_lookup": (_S, [_vp, _i32, _i64, _vp, _i32, _vp, _vp]),
    "tf_expert_cache_admit": (_S, [_vp, _i32, _i64, ctypes.c_int32, _vp, _i32, _vp, _vp]),
    "tf_expert_cache_invalidate": (_S, [_vp, _i32, ctypes.c_int32]),
    "tf_expert_cache_trace": (_S, [_vp, _vp, _sz, ctypes.POINTER(_sz)]),
    "tf_expert_cache_state": (_S, [_vp, _i32, _vp, _vp, _vp]),
    "tf_expert_cache_destroy": (_S, [_vp]),
    "tf_expert_cache_set_copy_streams": (_S, [_vp, ctypes.POINTER(_vp), _i32]),
    "tf_device_cache_state_bytes": (_sz, [_i32, _i32, _i32, _sz]),
    "tf_device_cache_create": (_S, [_i32, _i32, _i32, _sz, _vp, _vp, _vp, _sz, _sz, ctypes.POINTER(_vp)]),
    "tf_device_cache_set_fetch_ctas": (_S, [_vp, _i32]),
    "tf_device_cache_counters": (_S, [_vp, ctypes.POINTER(_i64), ctypes.POINTER(_i64), ctypes.POINTER(_i64), _vp]),
    "tf_device_cache_trace": (_S, [_vp, _vp, _sz, ctypes.POINTER(_sz), _vp]),
    "tf_device_cache_state": (_S, [_vp, _i32, _vp, _vp, _vp, _vp]),
    "tf_device_cache_destroy": (_S, [_vp]),
    "tf_layer_step_device_cache": (_S, [_vp, _vp, _i32, _vp, _vp, _vp, _i32, _vp, _vp, _i32,
                                        ctypes.POINTER(StepStats)]),
    "tf_layer_workspace_bytes": (_sz, [ctypes.POINTER(LayerDesc), _i32]),
    "tf_layer_create": (_S, [ctypes.POINTER(LayerDesc), _i32, _vp, _sz, ctypes.POINTER(_vp)]),
    "tf_layer_destroy": (_S, [_vp]),
    "tf_layer_routing": (_S, [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                              ctypes.POINTER(_vp)]),
    "tf_layer_step": (_S, [_vp, _vp, _i32, _i64, _vp, _vp, _vp, _i32, _vp, _i32, _vp, _vp, _i32,
                           ctypes.POINTER(StepStats)]),
    "tf_layer_prefill_cached": (_S, [_vp, _vp, _i32, _i64, _vp, _vp, _vp, _i32, _vp, _i32, _vp, _vp,
                                     ctypes.POINTER(PrefillStats)]),
    "tf_stack_decode": (_S, [ctypes.POINTER(_vp), _i32, _vp, _vp, _vp, ctypes.POINTER(_vp), _vp]),
    "tf_stack_workspace_bytes": (_sz, [_i32, _i32]),
    "tf_attn_workspace_bytes": (_sz, [ctypes.POINTER(AttnDesc)]),
    "tf_attn_cache_bytes": (_sz, [ctypes.POINTER(AttnDesc)]),
    "tf_attn_decode": (_S, [ctypes.POINTER(AttnDesc), _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp]),
    "tf_stack_create": (_S, [ctypes.POINTER(_vp), _i32, ctypes.POINTER(_vp), _vp, _sz, ctypes.POINTER(_vp)]),
    "tf_stack_set_prefetch": (_S, [_vp, _i32]),
    "tf_stack_set_trace": (_S, [_vp, _vp, _sz]),
    "tf_stack_step": (_S, [_vp, _vp, _vp, _vp]),
    "tf_stack_check": (_S, [_vp, _vp]),
    "tf_stack_layer_buffers": (_S, [_vp, _i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                    ctypes.POINTER(_vp)]),
    "tf_stack_destroy": (_S, [_vp]),
    "tf_profile_begin": (_S, [_i32]),
    "tf_profile_end": (_S, [_vp, _vp]),
    "tf_test_fail_nth_copy": (_S, [_i32]),
    "tf_test_set_wait_limit_ns": (_S, [ctypes.c_uint64]),
}

KERNEL_NAMES = ["router", "gateup", "down", "layer", "permute", "gemm", "combine", "other"]

_lib = None


def lib():
    """The loaded libtf.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libtf.so not found at %s; build it with "
                              "`python -m bit_expert_streaming_layer_b300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def last_error() -> str:
    return lib().tf_last_error().decode()


def _check(status: int, fn: str):
    if status != TF_OK:
        raise TFError(status, fn, last_error())


# ----------------------------------------------------------------- helpers

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


class _CudaArray:
    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def device_view(ptr: int, shape, typestr: str):
    """A torch tensor viewing device memory the library owns or carved (no copy)."""
    import torch
    return torch.as_tensor(_CudaArray(ptr, shape, typestr), device="cuda")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- layout

def tf_expert_payload_bytes(H: int, I: int) -> int:
    return lib().tf_expert_payload_bytes(H, I)


def tf_expert_slot_bytes(H: int, I: int) -> int:
    return lib().tf_expert_slot_bytes(H, I)


def tf_expert_offsets(H: int, I: int):
    off = (ctypes.c_size_t * 4)()
    _check(lib().tf_expert_offsets(H, I, off), "tf_expert_offsets")
    return list(off)


def tf_pack_expert(q, s, b, H: int, I: int, blob_out) -> None:
    """Pack logical codes/scales/biases (host numpy arrays or CPU tensors, concatenated gate, up, down)
    into blob_out (host memory: numpy array, CPU tensor or raw address)."""
    def hp(a):
        if isinstance(a, int):
            return a
        if hasattr(a, "ctypes"):
            return a.ctypes.data
        return a.data_ptr()
    _check(lib().tf_pack_expert(hp(q), hp(s), hp(b), H, I, hp(blob_out)), "tf_pack_expert")


# ----------------------------------------------------------------- routing

def tf_router_workspace_bytes(T: int, E: int) -> int:
    return lib().tf_router_workspace_bytes(T, E)


def tf_router_topk(x, T, H, W_r, E, logit_bias, bias_stride, k, idx, w, logits, rms, workspace, ws_bytes,
                   stream=None) -> None:
    _check(lib().tf_router_topk(_ptr(x), T, H, _ptr(W_r), E, _ptr(logit_bias), bias_stride, k, _ptr(idx), _ptr(w),
                                _ptr(logits), _ptr(rms), _ptr(workspace), ws_bytes, _stream(stream)),
           "tf_router_topk")


def tf_dequant_expert(blob, H, I, matrix, as_bf16, out, stream=None) -> None:
    _check(lib().tf_dequant_expert(_ptr(blob), H, I, matrix, as_bf16, _ptr(out), _stream(stream)),
           "tf_dequant_expert")


def expert_table(base, stride: int, slot_of_expert=None, n_experts: int = 0, n_slots: int = 0) -> ExpertTable:
    """Expert e at base + (slot_of_expert[e] if a map is given else e) * stride; ids valid in [0, n_experts)
    (0: the layer's E where a layer descriptor carries the table), map entries in [0, n_slots)."""
    return ExpertTable(_ptr(base), stride, _ptr(slot_of_expert), n_experts, n_slots)


# ----------------------------------------------------------------- MoE FFN

def tf_moe_decode_workspace_bytes(H: int, I: int, k: int) -> int:
    return lib().tf_moe_decode_workspace_bytes(H, I, k)


def tf_moe_ffn_decode(x, out, table: ExpertTable, idx, w, k, H, I, delta, workspace, ws_bytes, stream=None) -> None:
    _check(lib().tf_moe_ffn_decode(_ptr(x), _ptr(out), ctypes.byref(table), _ptr(idx), _ptr(w), k, H, I, _ptr(delta),
                                   _ptr(workspace), ws_bytes, _stream(stream)), "tf_moe_ffn_decode")


TF_NOALLOC_MAX_KI = 65536


def tf_moe_ffn_decode_noalloc(x, out, table: ExpertTable, idx, w, k, H, I, delta, stream=None) -> None:
    """tf_moe_ffn_decode without a workspace: the scratch is a fixed array inside libtf.so
    (for callers that cannot allocate device memory). Calls that overlap on the GPU share
    that array and race; the first call on a device should come before any stream capture."""
    _check(lib().tf_moe_ffn_decode_noalloc(_ptr(x), _ptr(out), ctypes.byref(table), _ptr(idx), _ptr(w), k, H, I,
                                           _ptr(delta), _stream(stream)), "tf_moe_ffn_decode_noalloc")


def tf_moe_grouped_workspace_bytes(T, H, I, E, k) -> int:
    return lib().tf_moe_grouped_workspace_bytes(T, H, I, E, k)


def tf_moe_ffn_grouped(x, out, T, table: ExpertTable, E, idx, w, k, H, I, delta, perm_out, counts_out, workspace,
                       ws_bytes, stream=None) -> None:
    _check(lib().tf_moe_ffn_grouped(_ptr(x), _ptr(out), T, ctypes.byref(table), E, _ptr(idx), _ptr(w), k, H, I,
                                    _ptr(delta), _ptr(perm_out), _ptr(counts_out), _ptr(workspace), ws_bytes,
                                    _stream(stream)), "tf_moe_ffn_grouped")


# ----------------------------------------------------------------- cache

class ExpertCache:
    """Owner of a tf_expert_cache handle (per-layer LFU metadata)."""

    def __init__(self, n_layers: int, n_slots: int, n_experts: int, slot_bytes: int, d_slot_pool=None):
        h = ctypes.c_void_p()
        _check(lib().tf_expert_cache_create(n_layers, n_slots, n_experts, slot_bytes, _ptr(d_slot_pool),
                                            ctypes.byref(h)), "tf_expert_cache_create")
        self.handle = h.value
        self.n_slots = n_slots

    def lookup(self, layer: int, step: int, ids):
        import numpy as np
        ids = np.ascontiguousarray(ids, np.int32)
        slot = np.empty(ids.shape[0], np.int32)
        hit = np.empty(ids.shape[0], np.uint8)
        _check(lib().tf_expert_cache_lookup(self.handle, layer, step, ids.ctypes.data, ids.shape[0], slot.ctypes.data,
                                            hit.ctypes.data), "tf_expert_cache_lookup")
        return slot, hit

    def admit(self, layer: int, step: int, expert: int, pinned_ids):
        import numpy as np
        pinned = np.ascontiguousarray(pinned_ids, np.int32)
        slot, ev = ctypes.c_int32(), ctypes.c_int32()
        _check(lib().tf_expert_cache_admit(self.handle, layer, step, expert, pinned.ctypes.data, pinned.shape[0],
                                           ctypes.byref(slot), ctypes.byref(ev)), "tf_expert_cache_admit")
        return slot.value, ev.value

    def invalidate(self, layer: int, slot: int):
        _check(lib().tf_expert_cache_invalidate(self.handle, layer, slot), "tf_expert_cache_invalidate")

    def trace(self):
        n = ctypes.c_size_t()
        _check(lib().tf_expert_cache_trace(self.handle, None, 0, ctypes.byref(n)), "tf_expert_cache_trace")
        buf = (CacheEvent * max(1, n.value))()
        _check(lib().tf_expert_cache_trace(self.handle, buf, n.value, ctypes.byref(n)), "tf_expert_cache_trace")
        return [(e.step, e.layer, e.expert, e.hit, e.slot, e.evicted) for e in buf[:n.value]]

    def state(self, layer: int):
        import numpy as np
        ex = np.empty(self.n_slots, np.int32)
        cnt = np.empty(self.n_slots, np.int64)
        lu = np.empty(self.n_slots, np.int64)
        _check(lib().tf_expert_cache_state(self.handle, layer, ex.ctypes.data, cnt.ctypes.data, lu.ctypes.data),
               "tf_expert_cache_state")
        return ex, cnt, lu

    def set_copy_streams(self, streams) -> None:
        """Stripe the miss fills over these streams (empty list: back to the call's copy stream)."""
        self._streams = list(streams)
        arr = (ctypes.c_void_p * max(1, len(self._streams)))(*[_stream(s) for s in self._streams])
        _check(lib().tf_expert_cache_set_copy_streams(self.handle, arr, len(self._streams)),
               "tf_expert_cache_set_copy_streams")

    def close(self):
        if self.handle:
            lib().tf_expert_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tf_device_cache_state_bytes(n_layers: int, n_slots: int, n_experts: int, trace_capacity: int) -> int:
    return lib().tf_device_cache_state_bytes(n_layers, n_slots, n_experts, trace_capacity)


class DeviceCache:
    """Owner of a tf_device_cache handle: the per-layer LFU cache with its metadata in device memory.
    `state` must be a device tensor of tf_device_cache_state_bytes(...) bytes kept alive by the caller; the
    pool and the pinned host store likewise."""

    def __init__(self, n_layers: int, n_slots: int, n_experts: int, slot_bytes: int, d_slot_pool, h_expert_store,
                 state, trace_capacity: int = 0):
        h = ctypes.c_void_p()
        self.state_buf, self.pool, self.store = state, d_slot_pool, h_expert_store
        _check(lib().tf_device_cache_create(n_layers, n_slots, n_experts, slot_bytes, _ptr(d_slot_pool),
                                            _ptr(h_expert_store), _ptr(state), state.numel() * state.element_size(),
                                            trace_capacity, ctypes.byref(h)), "tf_device_cache_create")
        self.handle = h.value
        self.n_slots = n_slots

    def set_fetch_ctas(self, ctas: int) -> None:
        _check(lib().tf_device_cache_set_fetch_ctas(self.handle, ctas), "tf_device_cache_set_fetch_ctas")

    def counters(self, stream=None):
        """(hits, misses, events recorded) since creation."""
        h, m, n = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib().tf_device_cache_counters(self.handle, ctypes.byref(h), ctypes.byref(m), ctypes.byref(n),
                                              _stream(stream)), "tf_device_cache_counters")
        return h.value, m.value, n.value

    def trace(self, stream=None):
        n = ctypes.c_size_t()
        _check(lib().tf_device_cache_trace(self.handle, None, 0, ctypes.byref(n), _stream(stream)),
               "tf_device_cache_trace")
        buf = (CacheEvent * max(1, n.value))()
        _check(lib().tf_device_cache_trace(self.handle, buf, n.value, ctypes.byref(n), _stream(stream)),
               "tf_device_cache_trace")
        return [(e.step, e.layer, e.expert, e.hit, e.slot, e.evicted) for e in buf[:n.value]]

    def state(self, layer: int, stream=None):
        import numpy as np
        ex = np.empty(self.n_slots, np.int32)
        cnt = np.empty(self.n_slots, np.int64)
        lu = np.empty(self.n_slots, np.int64)
        _check(lib().tf_device_cache_state(self.handle, layer, ex.ctypes.data, cnt.ctypes.data, lu.ctypes.data,
                                           _stream(stream)), "tf_device_cache_state")
        return ex, cnt, lu

    def close(self):
        if self.handle:
            lib().tf_device_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ----------------------------------------------------------------- layers

def layer_desc(H, I, E, k, S, W_r, W_sg=None, W_su=None, W_sd=None, experts: ExpertTable | None = None,
               eps: float = 1e-6) -> LayerDesc:
    return LayerDesc(H, I, E, k, S, eps, _ptr(W_r), _ptr(W_sg), _ptr(W_su), _ptr(W_sd),
                     experts if experts is not None else ExpertTable(None, 0, None, 0, 0))


def tf_layer_workspace_bytes(desc: LayerDesc, T_max: int) -> int:
    return lib().tf_layer_workspace_bytes(ctypes.byref(desc), T_max)


class Layer:
    """Owner of a tf_layer handle; `workspace` must be a zeroed device tensor kept alive by the caller."""

    def __init__(self, desc: LayerDesc, T_max: int, workspace):
        h = ctypes.c_void_p()
        self.desc = desc
        self.workspace = workspace
        _check(lib().tf_layer_create(ctypes.byref(desc), T_max, _ptr(workspace), workspace.numel() *
                                     workspace.element_size(), ctypes.byref(h)), "tf_layer_create")
        self.handle = h.value

    def routing(self):
        """Device addresses of the last step's routing: idx, w, logits, rms."""
        p = [ctypes.c_void_p() for _ in range(4)]
        _check(lib().tf_layer_routing(self.handle, *[ctypes.byref(v) for v in p]), "tf_layer_routing")
        return [v.value for v in p]

    def routing_tensors(self, T: int = 1):
        """The last step's routing as torch views: idx [T,k] int32, w [T,k], logits [T,E], rms [T]."""
        d = self.desc
        pi, pw, pl, pr = self.routing()
        return (device_view(pi, (T, d.k), "<i4"), device_view(pw, (T, d.k), "<f4"),
                device_view(pl, (T, d.E), "<f4"), device_view(pr, (T,), "<f4"))

    def close(self):
        if self.handle:
            lib().tf_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tf_layer_step(layer: Layer, cache: ExpertCache | None, layer_index: int, step: int, h_expert_store, x, out, T,
                  logit_bias=None, bias_stride: int = 0, compute_stream=None, copy_stream=None, measure: int = 0):
    stats = StepStats()
    _check(lib().tf_layer_step(layer.handle, cache.handle if cache else None, layer_index, step, _ptr(h_expert_store),
                               _ptr(x), _ptr(out), T, _ptr(logit_bias), bias_stride, _stream(compute_stream),
                               _stream(copy_stream) if copy_stream is not None else None, measure,
                               ctypes.byref(stats)), "tf_layer_step")
    return stats


def tf_layer_step_device_cache(layer: Layer, cache: DeviceCache, layer_index: int, x, out, logit_bias=None,
                               bias_stride: int = 0, compute_stream=None, fetch_stream=None, measure: int = 0):
    stats = StepStats()
    _check(lib().tf_layer_step_device_cache(layer.handle, cache.handle, layer_index, _ptr(x), _ptr(out),
                                            _ptr(logit_bias), bias_stride, _stream(compute_stream),
                                            _stream(fetch_stream), measure, ctypes.byref(stats)),
           "tf_layer_step_device_cache")
    return stats


def tf_layer_prefill_cached(layer: Layer, cache: ExpertCache, layer_index: int, step0: int, h_expert_store, x, out,
                            T: int, logit_bias=None, bias_stride: int = 0, compute_stream=None, copy_stream=None):
    """A chunk of T tokens through one layer with its experts streamed through the LFU cache, in waves of the
    cache's slot count; returns PrefillStats (waves, hits, misses, bytes_fetched)."""
    stats = PrefillStats()
    _check(lib().tf_layer_prefill_cached(layer.handle, cache.handle, layer_index, step0, _ptr(h_expert_store), _ptr(x),
                                         _ptr(out), T, _ptr(logit_bias), bias_stride, _stream(compute_stream),
                                         _stream(copy_stream), ctypes.byref(stats)), "tf_layer_prefill_cached")
    return stats


def tf_stack_decode(layers, x, out, scratch, logit_bias=None, stream=None) -> None:
    L = len(layers)
    arr = (ctypes.c_void_p * L)(*[l.handle for l in layers])
    bias = None
    if logit_bias is not None:
        bias = (ctypes.c_void_p * L)(*[_ptr(b) for b in logit_bias])
    _check(lib().tf_stack_decode(arr, L, _ptr(x), _ptr(out), _ptr(scratch), bias, _stream(stream)),
           "tf_stack_decode")


class Stack:
    """Owner of a tf_stack handle (fused persistent decode kernel over resident layers).
    `workspace` must be a device tensor of tf_stack_workspace_bytes(L, E) bytes kept alive by the caller."""

    def __init__(self, layers, workspace, logit_bias=None):
        L = len(layers)
        arr = (ctypes.c_void_p * L)(*[l.handle for l in layers])
        bias = None
        if logit_bias is not None:
            bias = (ctypes.c_void_p * L)(*[_ptr(b) for b in logit_bias])
        h = ctypes.c_void_p()
        self.layers, self.workspace, self.L = layers, workspace, L
        _check(lib().tf_stack_create(arr, L, bias, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     ctypes.byref(h)), "tf_stack_create")
        self.handle = h.value

    def set_prefetch(self, on: bool) -> None:
        _check(lib().tf_stack_set_prefetch(self.handle, 1 if on else 0), "tf_stack_set_prefetch")

    def set_trace(self, buf) -> None:
        """buf: device tensor of >= L * 16 int64 (or None to stop tracing)."""
        nbytes = 0 if buf is None else buf.numel() * buf.element_size()
        _check(lib().tf_stack_set_trace(self.handle, _ptr(buf), nbytes), "tf_stack_set_trace")

    def layer_buffers(self, layer: int):
        p = [ctypes.c_void_p() for _ in range(4)]
        _check(lib().tf_stack_layer_buffers(self.handle, layer, *[ctypes.byref(v) for v in p]),
               "tf_stack_layer_buffers")
        return [v.value for v in p]

    def close(self):
        if self.handle:
            lib().tf_stack_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tf_stack_workspace_bytes(L: int, E: int) -> int:
    return lib().tf_stack_workspace_bytes(L, E)


def tf_stack_step(stack: Stack, x, out, stream=None) -> None:
    _check(lib().tf_stack_step(stack.handle, _ptr(x), _ptr(out), _stream(stream)), "tf_stack_step")


def tf_stack_check(stack: Stack, stream=None) -> None:
    _check(lib().tf_stack_check(stack.handle, _stream(stream)), "tf_stack_check")


def tf_profile_begin(capacity: int) -> None:
    _check(lib().tf_profile_begin(capacity), "tf_profile_begin")


def tf_profile_end() -> dict:
    """{kernel name: (summed event ms, launches)} since tf_profile_begin."""
    ms = (ctypes.c_double * len(KERNEL_NAMES))()
    n = (ctypes.c_int64 * len(KERNEL_NAMES))()
    _check(lib().tf_profile_end(ms, n), "tf_profile_end")
    return {name: (ms[i], n[i]) for i, name in enumerate(KERNEL_NAMES)}


def tf_test_fail_nth_copy(n: int) -> None:
    _check(lib().tf_test_fail_nth_copy(n), "tf_test_fail_nth_copy")


def tf_test_set_wait_limit_ns(ns: int) -> None:
    """Limit of the kernels' waits on other warps / CTAs for later launches (0: the default 2 s)."""
    _check(lib().tf_test_set_wait_limit_ns(ns), "tf_test_set_wait_limit_ns")


# ----------------------------------------------------------------- attention

def attn_desc(H: int, n_q_heads: int, n_kv_heads: int, head_dim: int, max_seq: int, W_q, W_k, W_v, W_o,
              eps: float = 1e-6, rope_theta: float = 10000.0) -> AttnDesc:
    """Descriptor of the attention half of a decoder layer (W_*: device bf16 tensors or pointers)."""
    return AttnDesc(H, n_q_heads, n_kv_heads, head_dim, max_seq, eps, rope_theta, _ptr(W_q), _ptr(W_k), _ptr(W_v),
                    _ptr(W_o))


def tf_attn_workspace_bytes(d: AttnDesc) -> int:
    return lib().tf_attn_workspace_bytes(ctypes.byref(d))


def tf_attn_cache_bytes(d: AttnDesc) -> int:
    return lib().tf_attn_cache_bytes(ctypes.byref(d))


def tf_attn_decode(d: AttnDesc, x, out, pos: int, k_cache, v_cache, workspace, ws_bytes: int, stream=None) -> None:
    _check(lib().tf_attn_decode(ctypes.byref(d), _ptr(x), _ptr(out), pos, _ptr(k_cache), _ptr(v_cache),
                                _ptr(workspace), ws_bytes, _stream(stream)), "tf_attn_decode")
