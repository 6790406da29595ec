"""GPU parity of the decode path (router, dequant, expert FFN, layer step,
decode stack, cached step) against the CPU oracle, through the C ABI.

Bit-exact: RMS scale, router logits, top-k ids, dequantised weights, cache
traces. Within tolerance (tests/parity.py): routing weights and layer outputs.
Every output buffer is filled with NaN before the call, and the test checks
that no NaN survives (full coverage of the writes).
"""
import numpy as np
import pytest
import torch

import bit_expert_streaming_layer_b300 as B
import oracle as O
import workload as W
from parity import CONTRACT_TOL, bf16_to_f64, delta_rel_err, elem_rel_err, max_rel_err
from workload.model import SyntheticStack, bf16_bits, expert_logical_concat, hidden_tensor, _u16_to_bf16_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda"

SMALL = dict(H=320, I=192, E=13, k=4, S=128)
MEDIUM = dict(H=1024, I=256, E=40, k=8, S=256)
FULL = dict(H=2816, I=704, E=128, k=8, S=2112)


def nan_f32(*shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device=DEV)


def nan_bf16(*shape):
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device=DEV)


def f32_bits(t):
    return t.detach().cpu().numpy().view(np.uint32)


# ------------------------------------------------------------------- router

def _router_case(T, H, E, k, bias_mode, seed=11):
    x = hidden_tensor(seed, 0, T, H)
    Wr_bits = W.router_weights(seed, 0, E, H)
    if bias_mode == "ties":
        # identical rows -> identical logits; lower index must win and come first
        for dup in (5, 9, E - 1):
            Wr_bits[dup] = Wr_bits[2]
    Wr = _u16_to_bf16_tensor(Wr_bits).to(DEV)
    bias, stride = None, 0
    if bias_mode == "shared":
        bias = torch.from_numpy(W.zipf_bias(seed, 0, E, 1.1)[0]).to(DEV)
    elif bias_mode == "per_token":
        bias = torch.randn(T, E, generator=torch.Generator().manual_seed(seed)).float().to(DEV)
        stride = E
    elif bias_mode == "ties":
        b = np.zeros(E, np.float32)
        b[[2, 5, 9, E - 1]] = 50.0      # far above every other logit: the tied group is the top 4
        bias = torch.from_numpy(b).to(DEV)
    ws = torch.zeros(B.tf_router_workspace_bytes(T, E), dtype=torch.uint8, device=DEV)
    idx = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    w, logits, rms = nan_f32(T, k), nan_f32(T, E), nan_f32(T)
    B.tf_router_topk(x, T, H, Wr, E, bias, stride, k, idx, w, logits, rms, ws, ws.numel())
    torch.cuda.synchronize()
    xb = bf16_bits(x)
    bias_np = None if bias is None else bias.cpu().numpy()
    for t in range(T):
        bt = None if bias_np is None else (bias_np[t] if stride else bias_np)
        r, z, i_o, w_o = O.route(xb[t], Wr_bits, bt, k)
        assert f32_bits(rms[t:t + 1])[0] == np.float32(r).view(np.uint32)
        assert np.array_equal(f32_bits(logits[t]), z.view(np.uint32))
        assert idx[t].cpu().numpy().tolist() == i_o.tolist()
        assert np.max(np.abs(w[t].cpu().numpy() - w_o)) <= 4e-7
    return idx.cpu().numpy(), ws


@pytest.mark.parametrize("T,H,E,k,bias_mode", [
    (1, 2816, 128, 8, "none"), (1, 2816, 128, 8, "shared"), (5, 320, 13, 4, "shared"),
    (7, 1024, 40, 8, "per_token"), (3, 2816, 128, 8, "ties"), (2, 64, 16, 16, "none"),
    (64, 2816, 128, 8, "none")])
def test_router_topk_bitexact(T, H, E, k, bias_mode):
    idx, ws = _router_case(T, H, E, k, bias_mode)
    if bias_mode == "ties":
        for t in range(T):
            assert idx[t][:4].tolist() == [2, 5, 9, E - 1]
    # the kernel leaves its workspace zeroed
    assert int(ws.sum()) == 0 or int(ws[:256].sum()) == 0


# ------------------------------------------------------------------- dequant

@pytest.mark.parametrize("H,I", [(2816, 704), (320, 192)])
def test_dequant_expert_bitexact(H, I):
    q, s, b = expert_logical_concat(3, 0, 1, H, I)
    blob = np.zeros(B.tf_expert_payload_bytes(H, I), np.uint8)
    B.tf_pack_expert(q, s, b, H, I, blob)
    d_blob = torch.from_numpy(blob).to(DEV)
    ex = W.expert(3, 0, 1, H, I)
    for m, name in enumerate(("gate", "up", "down")):
        R, K = ex[name][0].shape
        want = O.dequant_matrix(*ex[name])
        want_bf = O.dequant_matrix(*ex[name], fmt="bf16")
        out = nan_f32(R, K)
        B.tf_dequant_expert(d_blob, H, I, m, 0, out)
        out_bf = nan_bf16(R, K)
        B.tf_dequant_expert(d_blob, H, I, m, 1, out_bf)
        torch.cuda.synchronize()
        assert np.array_equal(f32_bits(out), want.view(np.uint32)), name
        got_bf = bf16_to_f64(bf16_bits(out_bf)).astype(np.float32)
        assert np.array_equal(got_bf.view(np.uint32), want_bf.astype(np.float32).view(np.uint32)), name
        # fp16: the operand of the grouped tensor-core GEMMs
        want_h = O.dequant_matrix(*ex[name], fmt="fp16")
        out_h = torch.full((R, K), float("nan"), dtype=torch.float16, device=DEV)
        B.tf_dequant_expert(d_blob, H, I, m, 2, out_h)
        torch.cuda.synchronize()
        got_h = out_h.cpu().numpy().astype(np.float32)
        assert np.array_equal(got_h.view(np.uint32), want_h.astype(np.float32).view(np.uint32)), name


# --------------------------------------------------------------- decode FFN

def _device_experts(seed, layer, ids, E, H, I):
    slot = B.tf_expert_slot_bytes(H, I)
    host = torch.zeros(E * slot, dtype=torch.uint8, pin_memory=True)
    for e in ids:
        q, s, b = expert_logical_concat(seed, layer, int(e), H, I)
        B.tf_pack_expert(q, s, b, H, I, host.data_ptr() + int(e) * slot)
    return host.to(DEV), slot


@pytest.mark.parametrize("cfg", [SMALL, MEDIUM, FULL], ids=["small", "medium", "full"])
def test_moe_ffn_decode_parity(cfg):
    H, I, E, k = cfg["H"], cfg["I"], cfg["E"], cfg["k"]
    seed = 21
    x = hidden_tensor(seed, 0, 1, H)[0]
    xb = bf16_bits(x)
    Wr = W.router_weights(seed, 0, E, H)
    r, z, idx, w = O.route(xb, Wr, None, k)
    d_exp, slot = _device_experts(seed, 0, idx, E, H, I)
    table = B.expert_table(d_exp, slot, n_experts=E)
    d_idx = torch.from_numpy(idx).to(DEV)
    d_w = torch.from_numpy(w.astype(np.float32)).to(DEV)
    ws = torch.zeros(B.tf_moe_decode_workspace_bytes(H, I, k), dtype=torch.uint8, device=DEV)
    out, delta = nan_bf16(H), nan_f32(H)
    B.tf_moe_ffn_decode(x, out, table, d_idx, d_w, k, H, I, delta, ws, ws.numel())
    torch.cuda.synchronize()
    experts = [W.expert(seed, 0, int(e), H, I) for e in idx]
    out_o, delta_o = O.layer_combine(xb, r, experts, w)
    got_d = delta.cpu().numpy()
    got_o = bf16_to_f64(bf16_bits(out))
    assert not np.isnan(got_d).any() and not np.isnan(got_o).any()
    assert max_rel_err(got_o, bf16_to_f64(out_o)) <= CONTRACT_TOL
    assert max_rel_err(got_d, delta_o) <= CONTRACT_TOL
    # the fp32 path is far inside the contract: 100x tighter normwise, and elementwise
    # with a 1e-2 rms floor (near-zero entries carry the absolute rounding of the sums)
    assert max_rel_err(got_d, delta_o) <= 1e-4
    assert elem_rel_err(got_d, delta_o, floor=1e-2) <= 1e-2
    # out may alias x
    x2 = x.clone()
    B.tf_moe_ffn_decode(x2, x2, table, d_idx, d_w, k, H, I, None, ws, ws.numel())
    torch.cuda.synchronize()
    assert torch.equal(x2.view(torch.int16), out.view(torch.int16))


def test_moe_ffn_decode_out_of_range_ids_give_nan_without_a_read():
    """An id outside the table's range (or a slot-map entry outside its slots) is never turned into an
    address: the output and the update become NaN. The ids are checked on the device before any load."""
    H, I, E, k = 512, 256, 8, 4
    seed = 23
    d_exp, slot = _device_experts(seed, 0, np.arange(E), E, H, I)
    x = hidden_tensor(seed, 0, 1, H)[0]
    ws = torch.zeros(B.tf_moe_decode_workspace_bytes(H, I, k), dtype=torch.uint8, device=DEV)
    d_w = torch.full((k,), 0.25, dtype=torch.float32, device=DEV)
    smap = torch.tensor([0, 1, 2, 3, 4, 5, 6, 99], dtype=torch.int32, device=DEV)   # expert 7 -> slot 99
    cases = [(B.expert_table(d_exp, slot, n_experts=E), [0, 1, E, 2]),
             (B.expert_table(d_exp, slot, n_experts=E), [0, -1, 1, 2]),
             (B.expert_table(d_exp, slot, smap, n_experts=E, n_slots=E), [0, 1, 7, 2])]
    for table, ids in cases:
        d_idx = torch.tensor(ids, dtype=torch.int32, device=DEV)
        out, delta = nan_bf16(H), nan_f32(H)
        out.zero_()
        delta.zero_()
        B.tf_moe_ffn_decode(x, out, table, d_idx, d_w, k, H, I, delta, ws, ws.numel())
        torch.cuda.synchronize()
        assert torch.isnan(out.float()).all() and torch.isnan(delta).all(), ids
    # the same ids in range give finite outputs
    d_idx = torch.tensor([0, 1, 6, 2], dtype=torch.int32, device=DEV)
    out, delta = nan_bf16(H), nan_f32(H)
    B.tf_moe_ffn_decode(x, out, cases[2][0], d_idx, d_w, k, H, I, delta, ws, ws.numel())
    torch.cuda.synchronize()
    assert not torch.isnan(out.float()).any() and not torch.isnan(delta).any()


# ------------------------------------------------------------- layer step

def _check_layer(stack, l, x_bits, out_bits, layer_idx=None, bias=None):
    """Oracle check of one layer on the GPU's own input (teacher forcing)."""
    H, I, E, k, S = stack.H, stack.I, stack.E, stack.k, stack.S
    Wr = W.router_weights(stack.seed, l, E, H)
    r, z, idx, w = O.route(x_bits, Wr, bias, k)
    if layer_idx is not None:
        assert layer_idx.tolist() == idx.tolist()
    experts = W.experts_parallel(stack.seed, l, idx, H, I)
    shared = W.shared_weights(stack.seed, l, H, S) if S else None
    out_o, delta_o = O.layer_combine(x_bits, r, experts, w, shared)
    got = bf16_to_f64(out_bits)
    assert not np.isnan(got).any()
    assert max_rel_err(got, bf16_to_f64(out_o)) <= CONTRACT_TOL
    assert delta_rel_err(out_bits, x_bits, delta_o) <= CONTRACT_TOL
    return idx


@pytest.mark.parametrize("cfg", [SMALL, MEDIUM, FULL], ids=["small", "medium", "full"])
def test_layer_step_resident_parity(cfg):
    stack = SyntheticStack(31, 1, **cfg)
    x = hidden_tensor(31, 0, 1, cfg["H"])[0]
    out = nan_bf16(cfg["H"])
    B.tf_layer_step(stack.layers[0], None, 0, 0, None, x, out, 1)
    torch.cuda.synchronize()
    idx, w, logits, rms = stack.layers[0].routing_tensors()
    _check_layer(stack, 0, bf16_bits(x), bf16_bits(out), layer_idx=idx[0].cpu().numpy())
    stack.close()


@pytest.mark.parametrize("cfg,L,steps", [(SMALL, 5, 3), (MEDIUM, 4, 2)], ids=["small", "medium"])
def test_stack_decode_teacher_forced(cfg, L, steps):
    stack = SyntheticStack(41, L, **cfg)
    H = cfg["H"]
    x0 = hidden_tensor(41, 0, 1, H)[0]
    cur = x0.clone()
    for step in range(steps):
        inputs = []
        for l in range(L):
            out = nan_bf16(H)
            B.tf_layer_step(stack.layers[l], None, l, step, None, cur, out, 1)
            torch.cuda.synchronize()
            inputs.append(bf16_bits(cur))
            _check_layer(stack, l, inputs[-1], bf16_bits(out))
            cur = out
        # the fused entry point reproduces the chained layer steps bit for bit
        stacked = nan_bf16(H)
        scratch = nan_bf16(H)
        start = _u16_to_bf16_tensor(inputs[0]).to(DEV)
        B.tf_stack_decode(stack.layers, start, stacked, scratch)
        torch.cuda.synchronize()
        assert torch.equal(stacked.view(torch.int16), cur.view(torch.int16))
    stack.close()


def test_stack_decode_full_size_sampled_layers():
    """30 full-size layers, output fed back for 3 steps; oracle on sampled (step, layer) points."""
    L, H = 30, FULL["H"]
    stack = SyntheticStack(1, L, **FULL)
    cur = hidden_tensor(1, 0, 1, H)[0]
    sample = {(0, 0), (0, 17), (1, 29), (2, 5)}
    for step in range(3):
        for l in range(L):
            out = nan_bf16(H)
            B.tf_layer_step(stack.layers[l], None, l, step, None, cur, out, 1)
            if (step, l) in sample:
                torch.cuda.synchronize()
                _check_layer(stack, l, bf16_bits(cur), bf16_bits(out))
            cur = out
    torch.cuda.synchronize()
    assert not torch.isnan(cur.float()).any()
    stack.close()


# ------------------------------------------------------------- cached step

def _biased_logits(seed, l, E, s, alpha, prev_ids, step):
    bias = W.zipf_bias(seed, l, E, s, alpha)[0].copy()
    if prev_ids is not None and W.coin(seed, l, step):
        bias[prev_ids] += 30.0
    return bias


@pytest.mark.parametrize("cfg,L,slots,steps", [
    (dict(H=320, I=192, E=24, k=4, S=128), 3, 6, 25),
    (FULL, 3, 16, 12)], ids=["small", "full"])
def test_cached_step_traces_and_outputs(cfg, L, slots, steps):
    H, E, k = cfg["H"], cfg["E"], cfg["k"]
    cached = SyntheticStack(51, L, resident=False, n_slots=slots, **cfg)
    resident = SyntheticStack(51, L, resident=True, **cfg)
    copy_stream = torch.cuda.Stream()
    lfu = O.LFU(L, slots)
    want = []
    prev = [None] * L
    cur_c = hidden_tensor(51, 0, 1, H)[0]
    cur_r = cur_c.clone()
    bias_d = torch.empty(E, dtype=torch.float32, device=DEV)
    for step in range(steps):
        for l in range(L):
            bias_d.copy_(torch.from_numpy(_biased_logits(51, l, E, 1.1, 1.0, prev[l], step)))
            out_c, out_r = nan_bf16(H), nan_bf16(H)
            st = B.tf_layer_step(cached.layers[l], cached.cache, l, step, cached.store, cur_c, out_c, 1, bias_d, 0,
                                 None, copy_stream, measure=1)
            B.tf_layer_step(resident.layers[l], None, l, step, None, cur_r, out_r, 1, bias_d, 0)
            torch.cuda.synchronize()
            ids = cached.layers[l].routing_tensors()[0][0].cpu().numpy()
            prev[l] = ids
            ev = lfu.step(step, l, ids)
            want += ev
            assert st.hits + st.misses == k and st.misses == sum(1 for e in ev if not e[3])
            assert list(st.ids[:k]) == ids.tolist()
            assert st.bytes_fetched == st.misses * cached.payload
            # the cached path computes the same bits as the resident one
            assert torch.equal(out_c.view(torch.int16), out_r.view(torch.int16))
            cur_c, cur_r = out_c, out_r
    assert cached.cache.trace() == want
    cached.close()
    resident.close()


def test_cached_step_copy_failure_rolls_back():
    cfg = dict(H=320, I=192, E=24, k=4, S=128)
    st = SyntheticStack(61, 1, resident=False, n_slots=6, **cfg)
    cs = torch.cuda.Stream()
    x = hidden_tensor(61, 0, 1, cfg["H"])[0]
    out = nan_bf16(cfg["H"])
    B.tf_test_fail_nth_copy(3)           # cold cache: 4 misses; the third copy fails
    with pytest.raises(B.TFError) as e:
        B.tf_layer_step(st.layers[0], st.cache, 0, 0, st.store, x, out, 1, None, 0, None, cs)
    B.tf_test_fail_nth_copy(0)
    assert e.value.status == B.TF_ERR_CUDA and "rolled back" in str(e.value)
    torch.cuda.synchronize()
    ex, cnt, lu = st.cache.state(0)
    assert (ex >= 0).sum() == 0           # every slot admitted in the failed step is empty again
    # the next attempt succeeds and fills the cache
    B.tf_layer_step(st.layers[0], st.cache, 0, 1, st.store, x, out, 1, None, 0, None, cs)
    torch.cuda.synchronize()
    ex, cnt, lu = st.cache.state(0)
    assert (ex >= 0).sum() == cfg["k"]
    assert not torch.isnan(out.float()).any()
    st.close()
