"""Bounded device-side waits, driven until they run out (no fault, no hang).

The fused decode kernel and the grouped GEMM kernel bound every wait on another
warp, role or CTA (2 s by default) and report a wait that ran out as
TF_ERR_TIMEOUT: tf_stack_check returns it and resets the stack; the grouped
outputs become NaN. tf_test_set_wait_limit_ns shortens that limit to 1 ns for
the launches of a test, so that those waits run out on an ordinary input; waits
of a warp for its own copies and MMAs keep their own bound, so every kernel
still drains what it started before it returns. After the limit is restored the
next launch must compute the right result again (checked against the oracle).
"""
import numpy as np
import pytest
import torch

import bit_expert_streaming_layer_b300 as B
import oracle as O
import workload as W
from parity import CONTRACT_TOL, bf16_to_f64, max_rel_err
from workload.model import SyntheticStack, bf16_bits, hidden_tensor, pack_layer_experts

pytestmark = pytest.mark.gpu
DEV = "cuda"
FULL = dict(H=2816, I=704, E=128, k=8, S=2112)


def _short_waits(run, attempts=3):
    """Run `run()` with the wait limit at 1 ns until it reports a timeout (True), the limit restored after."""
    B.tf_test_set_wait_limit_ns(1)
    try:
        for _ in range(attempts):
            if run():
                return True
        return False
    finally:
        B.tf_test_set_wait_limit_ns(0)


def test_fused_stack_wait_timeout_is_reported_and_recovers():
    st = SyntheticStack(9, 2, **FULL)
    ws = torch.zeros(B.tf_stack_workspace_bytes(2, FULL["E"]), dtype=torch.uint8, device=DEV)
    fs = B.Stack(st.layers, ws)
    x = hidden_tensor(9, 0, 1, FULL["H"])[0]

    def run():
        out = torch.empty_like(x)
        B.tf_stack_step(fs, x, out)
        try:
            B.tf_stack_check(fs)
        except B.TFError as e:
            assert e.status == B.TF_ERR_TIMEOUT and "timed out" in str(e)
            return True
        return False

    assert _short_waits(run)
    # limit restored: the next steps run to completion and layer 0 matches the oracle
    for _ in range(2):
        out = torch.full_like(x, float("nan"))
        B.tf_stack_step(fs, x, out)
        B.tf_stack_check(fs)
    assert not torch.isnan(out.float()).any()
    pi, pw, pl, pa = fs.layer_buffers(0)
    y0 = bf16_bits(B.device_view(pa, (FULL["H"],), "<i2").view(torch.bfloat16))
    idx0 = B.device_view(pi, (FULL["k"],), "<i4").cpu().numpy()
    xb = bf16_bits(x)
    r, _, ridx, rw = O.route(xb, W.router_weights(9, 0, FULL["E"], FULL["H"]), None, FULL["k"])
    assert idx0.tolist() == ridx.tolist()
    ex = W.experts_parallel(9, 0, ridx, FULL["H"], FULL["I"])
    o, _ = O.layer_combine(xb, r, ex, rw, W.shared_weights(9, 0, FULL["H"], FULL["S"]))
    assert max_rel_err(bf16_to_f64(y0), bf16_to_f64(o)) <= CONTRACT_TOL
    fs.close()
    st.close()


def test_grouped_gemm_wait_timeout_poisons_outputs_and_recovers():
    H, I, E, k, T, seed = FULL["H"], FULL["I"], FULL["E"], FULL["k"], 128, 43
    slot = B.tf_expert_slot_bytes(H, I)
    host = torch.empty(E * slot, dtype=torch.uint8, pin_memory=True)
    pack_layer_experts(seed, 0, E, H, I, host)
    d_exp = host.to(DEV)
    table = B.expert_table(d_exp, slot)
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)) + 0.05
    w = (w / w.sum(1, keepdims=True)).astype(np.float32)
    d_idx, d_w = torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV)
    x = hidden_tensor(seed, 0, T, H)
    ws = torch.zeros(B.tf_moe_grouped_workspace_bytes(T, H, I, E, k), dtype=torch.uint8, device=DEV)

    def call():
        out = torch.zeros(T, H, dtype=torch.bfloat16, device=DEV)
        delta = torch.zeros(T, H, dtype=torch.float32, device=DEV)
        B.tf_moe_ffn_grouped(x, out, T, table, E, d_idx, d_w, k, H, I, delta, None, None, ws, ws.numel())
        torch.cuda.synchronize()
        return out, delta

    def run():
        out, delta = call()
        nan_o, nan_d = torch.isnan(out.float()), torch.isnan(delta)
        if nan_o.any():
            # a wait that ran out poisons every output, never a partial or stale result
            assert nan_o.all() and nan_d.all()
            return True
        assert not nan_d.any()
        return False

    assert _short_waits(run)
    out, delta = call()
    assert not torch.isnan(out.float()).any() and not torch.isnan(delta).any()
    xb, dl = bf16_bits(x), delta.cpu().numpy()
    for t in (0, 77, T - 1):
        ex = [W.expert(seed, 0, int(e), H, I) for e in idx[t]]
        _, d_o = O.layer_combine(xb[t], O.rms_scale(xb[t]), ex, w[t], None, tc=True)
        assert max_rel_err(dl[t], d_o) <= CONTRACT_TOL, t
