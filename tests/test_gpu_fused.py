"""GPU parity of the fused persistent decode kernel (tf_stack_*) against the
CPU oracle, through the C ABI, at the model's full layer shape.

Each layer is checked on the GPU's own input (teacher forcing): router logits
and top-8 ids bit for bit, routing weights to a few ulp, the layer output
within the contract tolerance. The kernel is also checked for determinism and
against the per-layer-kernel path.
"""
import numpy as np
import pytest
import torch

import bit_expert_streaming_layer_b300 as B
import oracle as O
import workload as W
from parity import CONTRACT_TOL, bf16_to_f64, delta_rel_err, max_rel_err
from workload.model import SyntheticStack, bf16_bits, hidden_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda"
FULL = dict(H=2816, I=704, E=128, k=8, S=2112)


def _view(ptr, shape, typestr):
    return B.device_view(ptr, shape, typestr)


def _check_layer(seed, l, x_bits, out_bits, idx_g, w_g, logits_g, bias=None, E=None):
    H, I, k, S = FULL["H"], FULL["I"], FULL["k"], FULL["S"]
    E = FULL["E"] if E is None else E
    r, z, idx, w = O.route(x_bits, W.router_weights(seed, l, E, H), bias, k)
    assert np.array_equal(logits_g.view(np.uint32), z.view(np.uint32)), "router logits differ"
    assert idx_g.tolist() == idx.tolist()
    assert np.max(np.abs(w_g - w)) <= 4e-7
    experts = W.experts_parallel(seed, l, idx, H, I)
    out_o, delta_o = O.layer_combine(x_bits, r, experts, w, W.shared_weights(seed, l, H, S))
    got = bf16_to_f64(out_bits)
    assert not np.isnan(got).any()
    assert max_rel_err(got, bf16_to_f64(out_o)) <= CONTRACT_TOL
    err = delta_rel_err(out_bits, x_bits, delta_o)
    assert err <= CONTRACT_TOL
    return err


def _make(seed, L, bias=None):
    st = SyntheticStack(seed, L, **FULL)
    ws = torch.zeros(B.tf_stack_workspace_bytes(L, FULL["E"]), dtype=torch.uint8, device=DEV)
    fs = B.Stack(st.layers, ws, bias)
    return st, fs, ws


@pytest.mark.parametrize("with_bias", [False, True], ids=["plain", "zipf_bias"])
def test_fused_stack_teacher_forced(with_bias):
    seed, L, steps, H = 3, 4, 3, FULL["H"]
    bias_t = None
    if with_bias:
        bias_t = [torch.from_numpy(W.zipf_bias(seed, l, FULL["E"], 1.2)[0]).to(DEV) for l in range(L)]
    st, fs, ws = _make(seed, L, bias_t)
    x = hidden_tensor(seed, 0, 1, H)[0]
    errs = []
    for step in range(steps):
        out = torch.full((H,), float("nan"), dtype=torch.bfloat16, device=DEV)
        B.tf_stack_step(fs, x, out)
        B.tf_stack_check(fs)
        xin = bf16_bits(x)
        for l in range(L):
            pi, pw, pl, pa = fs.layer_buffers(l)
            y = out if l == L - 1 else _view(pa, (H,), "<i2").view(torch.bfloat16)
            yb = bf16_bits(y)
            idx_g = _view(pi, (FULL["k"],), "<i4").cpu().numpy()
            w_g = _view(pw, (FULL["k"],), "<f4").cpu().numpy()
            lg = _view(pl, (FULL["E"],), "<f4").cpu().numpy()
            b = None if bias_t is None else bias_t[l].cpu().numpy()
            errs.append(_check_layer(seed, l, xin, yb, idx_g, w_g, lg, b))
            xin = yb
        x = out
    assert max(errs) < 1e-4      # fp32 accumulation: far inside the contract
    fs.close()
    st.close()


def test_fused_stack_deterministic_and_matches_layer_path():
    seed, L, H = 5, 6, FULL["H"]
    st, fs, ws = _make(seed, L)
    x = hidden_tensor(seed, 0, 1, H)[0]
    a = torch.empty(H, dtype=torch.bfloat16, device=DEV)
    b = torch.empty(H, dtype=torch.bfloat16, device=DEV)
    B.tf_stack_step(fs, x, a)
    B.tf_stack_step(fs, x, b)
    B.tf_stack_check(fs)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # the per-layer-kernel path computes the same layers (different fp32 summation order)
    ref = torch.empty(H, dtype=torch.bfloat16, device=DEV)
    scratch = torch.empty(H, dtype=torch.bfloat16, device=DEV)
    B.tf_stack_decode(st.layers, x, ref, scratch)
    torch.cuda.synchronize()
    assert max_rel_err(bf16_to_f64(bf16_bits(a)), bf16_to_f64(bf16_bits(ref))) <= CONTRACT_TOL
    # many back-to-back launches reuse the self-resetting sync words
    cur = x.clone()
    for _ in range(20):
        nxt = torch.empty_like(cur)
        B.tf_stack_step(fs, cur, nxt)
        cur = nxt
    B.tf_stack_check(fs)
    assert not torch.isnan(cur.float()).any()
    fs.close()
    st.close()


def test_fused_stack_rejects_other_shapes():
    st = SyntheticStack(9, 1, H=320, I=192, E=16, k=4, S=128)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    with pytest.raises(B.TFError) as e:
        B.Stack(st.layers, ws)
    assert e.value.status == B.TF_ERR_NOT_SUPPORTED
    st.close()


@pytest.mark.parametrize("E", [256, 8], ids=["E256_max", "E8_min"])
def test_fused_stack_expert_count_limits(E):
    """The largest expert count the fused kernel takes (8 top-k keys per lane) and
    the smallest (the top-8 is every expert), teacher-forced over two steps."""
    seed, L, H = 13, 2, FULL["H"]
    cfg = dict(FULL, E=E)
    st = SyntheticStack(seed, L, **cfg)
    ws = torch.zeros(B.tf_stack_workspace_bytes(L, E), dtype=torch.uint8, device=DEV)
    fs = B.Stack(st.layers, ws)
    x = hidden_tensor(seed, 0, 1, H)[0]
    for step in range(2):
        out = torch.full((H,), float("nan"), dtype=torch.bfloat16, device=DEV)
        B.tf_stack_step(fs, x, out)
        B.tf_stack_check(fs)
        xin = bf16_bits(x)
        for l in range(L):
            pi, pw, pl, pa = fs.layer_buffers(l)
            y = out if l == L - 1 else _view(pa, (H,), "<i2").view(torch.bfloat16)
            yb = bf16_bits(y)
            idx_g = _view(pi, (FULL["k"],), "<i4").cpu().numpy()
            w_g = _view(pw, (FULL["k"],), "<f4").cpu().numpy()
            lg = _view(pl, (E,), "<f4").cpu().numpy()
            _check_layer(seed, l, xin, yb, idx_g, w_g, lg, None, E=E)
            xin = yb
        x = out
    fs.close()
    st.close()
