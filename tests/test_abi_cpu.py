"""C-ABI library checks that need no GPU: it loads, exports every symbol the
header declares, rejects bad arguments before touching the device, packs
experts in the documented layout, and its LFU metadata reproduces the oracle's
cache traces bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest

import bit_expert_streaming_layer_b300 as B
import oracle as O
import workload as W
from golden_io import load_lfu_trace, lfu_trace_names

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "tf.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tf_[a-z0-9_]+)\s*\(", text)))


def test_library_loads_and_exports_every_declared_symbol():
    L = B.lib()
    names = header_functions()
    assert len(names) >= 25
    for n in names:
        assert hasattr(L, n), n
        assert n in B.SIGNATURES, "binding lacks " + n
    assert set(B.SIGNATURES) == set(names)


def test_binding_structures_match_the_library_layout():
    L = B.lib()
    for which, cls in enumerate([B.ExpertTable, B.LayerDesc, B.StepStats, B.CacheEvent, B.PrefillStats,
                                 B.AttnDesc]):
        assert L.tf_struct_bytes(which) == ctypes.sizeof(cls), cls.__name__
    assert L.tf_struct_bytes(6) == 0


def test_version_and_status_strings():
    assert b"sm_103a" in B.lib().tf_version()
    assert B.lib().tf_status_string(1) == b"TF_ERR_INVALID_ARG"


def test_layout_sizes_match_the_pages_expert_size():
    assert B.tf_expert_payload_bytes(2816, 704) == 3_345_408
    assert B.tf_expert_slot_bytes(2816, 704) == 3_358_720
    off = B.tf_expert_offsets(2816, 704)
    assert off == [0, 2 * 704 * 1408, 2 * 704 * 1408 + 2 * 704 * 44 * 4,
                   2 * 704 * 1408 + 2 * 704 * 44 * 4 + 2816 * 352]
    assert all(o % 16 == 0 for o in off)
    assert B.tf_expert_payload_bytes(2816, 700) == 0
    with pytest.raises(B.TFError) as e:
        B.tf_expert_offsets(100, 64)
    assert e.value.status == B.TF_ERR_INVALID_ARG


def _unpack_blob(blob, H, I):
    """Independent reader of the documented blob layout -> logical (q, s, b) per matrix."""
    off = B.tf_expert_offsets(H, I)
    out = {}
    gu = blob[off[0]:off[1]].reshape(2 * I, H // 2)
    gq = np.empty((2 * I, H), np.uint8)
    gq[:, 0::2] = gu & 15
    gq[:, 1::2] = gu >> 4
    gsb = blob[off[1]:off[2]].view(np.uint16).reshape(2 * I, H // 64, 2)
    dq_b = blob[off[2]:off[3]].reshape(H, I // 2)
    dq = np.empty((H, I), np.uint8)
    dq[:, 0::2] = dq_b & 15
    dq[:, 1::2] = dq_b >> 4
    dsb = blob[off[3]:off[3] + H * (I // 64) * 4].view(np.uint16).reshape(H, I // 64, 2)
    out["gate"] = (gq[0::2], gsb[0::2, :, 0], gsb[0::2, :, 1])
    out["up"] = (gq[1::2], gsb[1::2, :, 0], gsb[1::2, :, 1])
    out["down"] = (dq, dsb[:, :, 0], dsb[:, :, 1])
    return out


@pytest.mark.parametrize("H,I", [(2816, 704), (320, 192), (64, 64)])
def test_pack_expert_layout(H, I):
    ex = W.expert(5, 1, 3, H, I)
    q = np.concatenate([ex[m][0].ravel() for m in ("gate", "up", "down")])
    s = np.concatenate([ex[m][1].ravel() for m in ("gate", "up", "down")])
    b = np.concatenate([ex[m][2].ravel() for m in ("gate", "up", "down")])
    blob = np.zeros(B.tf_expert_payload_bytes(H, I), np.uint8)
    B.tf_pack_expert(q, s, b, H, I, blob)
    back = _unpack_blob(blob, H, I)
    for m in ("gate", "up", "down"):
        for a, r in zip(back[m], ex[m]):
            assert np.array_equal(a, r), m


def test_pack_rejects_bad_codes_and_shapes():
    H, I = 64, 64
    q = np.zeros(3 * H * I, np.uint8)
    s = np.zeros(3 * H * I // 64, np.uint16)
    b = np.zeros_like(s)
    blob = np.zeros(B.tf_expert_payload_bytes(H, I), np.uint8)
    q[17] = 16
    with pytest.raises(B.TFError) as e:
        B.tf_pack_expert(q, s, b, H, I, blob)
    assert e.value.status == B.TF_ERR_INVALID_ARG and "16" in str(e.value)
    with pytest.raises(B.TFError):
        B.tf_pack_expert(q, s, b, 100, I, blob)


def test_device_entry_points_reject_bad_arguments_before_launch():
    L = B.lib()
    # null pointers and bad sizes are caught on the host: no CUDA call is made
    assert L.tf_router_topk(None, 1, 2816, None, 128, None, 0, 8, None, None, None, None, None, 0, None) == 1
    assert L.tf_router_topk(8, 1, 2816, 8, 128, None, 0, 33, 8, 8, None, None, 8, 1 << 20, None) == 1
    assert L.tf_router_topk(8, 1, 2816, 8, 2000, None, 0, 8, 8, 8, None, None, 8, 1 << 20, None) == 1
    assert L.tf_router_topk(8, 1, 100, 8, 128, None, 0, 8, 8, 8, None, None, 8, 1 << 20, None) == 1
    t = B.ExpertTable(8, 3, None)     # stride not a multiple of 16
    assert L.tf_moe_ffn_decode(8, 8, ctypes.byref(t), 8, 8, 8, 2816, 704, None, 8, 1 << 20, None) == 1
    t = B.ExpertTable(16, 16, None, 128)
    assert L.tf_moe_ffn_decode(8, 8, ctypes.byref(t), 8, 8, 8, 2816, 704, None, 8, 16, None) == 1  # small ws
    assert b"workspace" in L.tf_last_error()
    # the id range must be given: the kernels check every id against it before forming an address
    t = B.ExpertTable(16, 16, None, 0)
    assert L.tf_moe_ffn_decode(8, 8, ctypes.byref(t), 8, 8, 8, 2816, 704, None, 8, 1 << 20, None) == 1
    assert b"n_experts" in L.tf_last_error()
    assert L.tf_moe_ffn_decode_noalloc(8, 8, ctypes.byref(t), 8, 8, 8, 2816, 704, None, None) == 1
    t = B.ExpertTable(16, 16, 256, 128, 0)   # a slot map without its slot count
    assert L.tf_moe_ffn_decode(8, 8, ctypes.byref(t), 8, 8, 8, 2816, 704, None, 8, 1 << 20, None) == 1
    assert b"n_slots" in L.tf_last_error()
    d = B.layer_desc(2816, 704, 128, 8, 2112, 16, 16, 16, 16, B.ExpertTable(16, 16, None, 64))
    assert B.tf_layer_workspace_bytes(d, 1) == 0          # the table's id range is not the layer's E
    d = B.layer_desc(2816, 704, 128, 8, 2112, 16)   # shared weights missing
    assert B.tf_layer_workspace_bytes(d, 1) == 0
    h = ctypes.c_void_p()
    assert L.tf_layer_create(ctypes.byref(d), 1, 256, 1 << 30, ctypes.byref(h)) == 1
    assert b"shared" in L.tf_last_error()
    assert L.tf_layer_step(None, None, 0, 0, None, None, None, 1, None, 0, None, None, 0, None) == 1
    # grouped path: shapes, aliasing, alignment and table kind are checked before any launch
    t = B.ExpertTable(256, 3358720, None)
    ws = B.tf_moe_grouped_workspace_bytes(4, 2816, 704, 128, 8)
    grouped = L.tf_moe_ffn_grouped
    assert grouped(256, 256, 4, ctypes.byref(t), 128, 256, 256, 8, 2816, 704, None, None, None, 256, ws, None) == 1
    assert b"alias" in L.tf_last_error()
    assert grouped(256, 512, 4, ctypes.byref(t), 128, 256, 256, 8, 2880, 704, None, None, None, 256, ws, None) == 1
    assert grouped(256, 512, 4, ctypes.byref(t), 128, 256, 256, 33, 2816, 704, None, None, None, 256, ws, None) == 1
    assert grouped(256, 512, 4, ctypes.byref(t), 128, 256, 256, 8, 2816, 704, None, None, None, 256, ws - 1,
                   None) == 1
    assert grouped(256, 512, 4, ctypes.byref(t), 128, 256, 256, 8, 2816, 704, None, None, None, 128, ws, None) == 1
    tm = B.ExpertTable(256, 3358720, 512)   # a slot map: the grouped path takes resident experts only
    assert grouped(256, 512, 4, ctypes.byref(tm), 128, 256, 256, 8, 2816, 704, None, None, None, 256, ws,
                   None) == 5
    te = B.ExpertTable(256, 3358720, None, 64)   # the table's id range is not E
    assert grouped(256, 512, 4, ctypes.byref(te), 128, 256, 256, 8, 2816, 704, None, None, None, 256, ws,
                   None) == 1
    assert b"n_experts" in L.tf_last_error()


def test_workspace_sizes():
    assert B.tf_router_workspace_bytes(1, 128) == 256 + 512
    # grouped: error word, routing tables, permuted activations, h and y for T*k rows
    T, k, H, I, E = 4096, 8, 2816, 704, 128
    P = T * k
    assert B.tf_moe_grouped_workspace_bytes(T, H, I, E, k) >= P * H * 2 + P * I * 2 + P * H * 4
    assert B.tf_moe_grouped_workspace_bytes(T, H, I, 2000, k) == 0
    assert B.tf_moe_decode_workspace_bytes(2816, 704, 8) == 8 * 704 * 4
    d = B.layer_desc(2816, 704, 128, 8, 2112, 16, 16, 16, 16, B.ExpertTable(16, 16, None))
    assert B.tf_layer_workspace_bytes(d, 1) > 8 * 704 * 4 + 2112 * 4
    # a handle for batched steps also holds the grouped path's buffers and the shared expert's n, h and y
    T = 64
    w64 = B.tf_layer_workspace_bytes(d, T)
    assert w64 >= B.tf_layer_workspace_bytes(d, 1) + B.tf_moe_grouped_workspace_bytes(T, H, I, E, k) + \
        T * H * 2 + T * 2112 * 2 + T * H * 4


# ------------------------------------------------------------- LFU metadata

def _run_product_lfu(cache, step, layer, ids):
    slot, hit = cache.lookup(layer, step, ids)
    for i, e in enumerate(ids):
        if not hit[i]:
            s, ev = cache.admit(layer, step, int(e), ids)
            slot[i] = s


@pytest.mark.parametrize("name", lfu_trace_names())
def test_product_lfu_matches_golden_traces(name):
    slots, layers, inputs, events = load_lfu_trace(name)
    c = B.ExpertCache(layers, slots, 64, 16)
    for step, layer, ids in inputs:
        _run_product_lfu(c, step, layer, np.array(ids, np.int32))
    assert c.trace() == events


def test_product_lfu_matches_oracle_on_long_skewed_run():
    rng = np.random.default_rng(3)
    Ls, S, E, k = 4, 16, 128, 8
    bias = [W.zipf_bias(7, l, E, 1.1)[0] for l in range(Ls)]
    prod = B.ExpertCache(Ls, S, E, 16)
    ora = O.LFU(Ls, S)
    want = []
    prev = [None] * Ls
    for step in range(400):
        for l in range(Ls):
            z = bias[l] + rng.standard_normal(E).astype(np.float32)
            if prev[l] is not None and rng.random() < 0.5:
                z[prev[l]] += 30
            ids = O.topk(z, k)
            prev[l] = ids
            want += ora.step(step, l, ids)
            _run_product_lfu(prod, step, l, ids)
    got = prod.trace()
    assert got == want
    hits = sum(e[3] for e in got) / len(got)
    assert 0.3 < hits < 0.95
    for l in range(Ls):
        ex_p, cnt_p, lu_p = prod.state(l)
        ex_o, cnt_o, lu_o = ora.state(l)
        assert np.array_equal(ex_p, ex_o) and np.array_equal(cnt_p, cnt_o) and np.array_equal(lu_p, lu_o)


def test_product_lfu_rejects_misuse_and_rolls_back():
    c = B.ExpertCache(1, 2, 8, 16)
    c.lookup(0, 0, np.array([1, 2], np.int32))
    c.admit(0, 0, 1, [1, 2])
    c.admit(0, 0, 2, [1, 2])
    with pytest.raises(B.TFError):          # both slots pinned by the current ids
        c.admit(0, 0, 3, [1, 2])
    with pytest.raises(B.TFError):          # already resident
        c.admit(0, 1, 1, [1])
    with pytest.raises(B.TFError):
        c.lookup(0, 1, np.array([9], np.int32))
    c.invalidate(0, 1)
    ex, cnt, lu = c.state(0)
    assert ex.tolist() == [1, -1] and cnt.tolist() == [1, 0]


def test_attention_descriptor_checks_and_sizes():
    """The attention entry points check their descriptor on the host (no launch, no device needed)."""
    good = B.attn_desc(2816, 16, 8, 128, 4096, 16, 16, 16, 16)
    assert B.tf_attn_cache_bytes(good) == 4096 * 8 * 128 * 2
    assert B.tf_attn_workspace_bytes(good) >= (2 * 2048 + 16 * 16 * (128 + 2)) * 4
    for bad in (B.attn_desc(2816, 16, 8, 96, 4096, 16, 16, 16, 16),       # head_dim not 64/128/256
                B.attn_desc(2816, 12, 8, 128, 4096, 16, 16, 16, 16),      # n_q_heads not a multiple of n_kv_heads
                B.attn_desc(2820, 16, 8, 128, 4096, 16, 16, 16, 16),      # H not a multiple of 8
                B.attn_desc(2816, 16, 8, 128, 0, 16, 16, 16, 16),         # no cache rows
                B.attn_desc(2816, 16, 8, 128, 4096, 16, 16, 16, 8),       # unaligned W_o
                B.attn_desc(2816, 16, 8, 128, 4096, 16, 16, 16, 0)):      # NULL W_o
        assert B.tf_attn_workspace_bytes(bad) == 0
        assert B.tf_attn_cache_bytes(bad) == 0
        with pytest.raises(B.TFError) as e:
            B.tf_attn_decode(bad, 16, 32, 0, 64, 64, 128, 1 << 20, stream=0)
        assert e.value.status == B.TF_ERR_INVALID_ARG
    for pos in (-1, 4096):
        with pytest.raises(B.TFError) as e:
            B.tf_attn_decode(good, 16, 32, pos, 64, 64, 128, 1 << 20, stream=0)
        assert e.value.status == B.TF_ERR_INVALID_ARG
    with pytest.raises(B.TFError) as e:   # workspace too small
        B.tf_attn_decode(good, 16, 32, 0, 64, 64, 128, 64, stream=0)
    assert e.value.status == B.TF_ERR_INVALID_ARG
