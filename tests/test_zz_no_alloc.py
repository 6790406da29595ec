"""The allocation-free decode FFN, tf_moe_ffn_decode_noalloc, through the C ABI.

Some callers cannot call cudaMalloc at all (a plugin inside a runtime that owns
the device heap, code running while a stream is captured, a loop with a fixed
memory budget), so they cannot hand the library a workspace. This entry point
takes its scratch from an array built into libtf.so instead. These tests check
that it gives the same result as tf_moe_ffn_decode with a caller workspace, bit
for bit (both launch the same kernels with the same arguments but the scratch
address), on two calls in a row (the second call finds the first call's data in
the shared array); that its first call agrees with the CPU oracle within the
contract tolerance; and that it refuses sizes beyond the array.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import bit_expert_streaming_layer_b300 as B
import oracle as O
import workload as W
from parity import CONTRACT_TOL, bf16_to_f64, max_rel_err
from workload.model import bf16_bits, expert_logical_concat, hidden_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda"
H, I, E, K = 2816, 704, 24, 8


def _experts(seed):
    slot = B.tf_expert_slot_bytes(H, I)
    host = torch.zeros(E * slot, dtype=torch.uint8, pin_memory=True)
    for e in range(E):
        q, s, b = expert_logical_concat(seed, 0, e, H, I)
        B.tf_pack_expert(q, s, b, H, I, host.data_ptr() + e * slot)
    return host.to(DEV), slot


def _case(seed, step):
    rng = np.random.default_rng(seed * 100 + step)
    idx = torch.from_numpy(rng.choice(E, K, replace=False).astype(np.int32)).to(DEV)
    wv = rng.random(K).astype(np.float32)
    w = torch.from_numpy(wv / wv.sum()).to(DEV)
    x = hidden_tensor(seed, step, 1, H)[0]
    return x, idx, w


def test_noalloc_matches_workspace_path_on_two_calls_in_a_row():
    seed = 5
    d_exp, slot = _experts(seed)
    table = B.expert_table(d_exp, slot, n_experts=E)
    ws = torch.zeros(B.tf_moe_decode_workspace_bytes(H, I, K), dtype=torch.uint8, device=DEV)
    for step in range(2):
        x, idx, w = _case(seed, step)
        ref_out = torch.full((H,), float("nan"), dtype=torch.bfloat16, device=DEV)
        ref_delta = torch.full((H,), float("nan"), dtype=torch.float32, device=DEV)
        B.tf_moe_ffn_decode(x, ref_out, table, idx, w, K, H, I, ref_delta, ws, ws.numel())
        out = torch.full((H,), float("nan"), dtype=torch.bfloat16, device=DEV)
        delta = torch.full((H,), float("nan"), dtype=torch.float32, device=DEV)
        B.tf_moe_ffn_decode_noalloc(x, out, table, idx, w, K, H, I, delta)
        torch.cuda.synchronize()
        got_o, want_o = bf16_bits(out), bf16_bits(ref_out)
        got_d, want_d = delta.cpu().numpy(), ref_delta.cpu().numpy()
        assert not np.isnan(bf16_to_f64(got_o)).any() and not np.isnan(got_d).any()
        assert np.array_equal(got_o, want_o), step
        assert np.array_equal(got_d.view(np.uint32), want_d.view(np.uint32)), step
        if step == 0:
            # the oracle: out = bf16(x + sum_i w_i E_i(RMSNorm(x))), fp32
            xb = bf16_bits(x)
            ids = idx.cpu().numpy()
            out_o, delta_o = O.layer_combine(xb, O.rms_scale(xb), [W.expert(seed, 0, int(e), H, I) for e in ids],
                                             w.cpu().numpy(), None)
            assert max_rel_err(bf16_to_f64(got_o), bf16_to_f64(out_o)) <= CONTRACT_TOL
            assert max_rel_err(got_d, delta_o) <= CONTRACT_TOL
        # out may alias x, as for the workspace entry point
        x2 = x.clone()
        B.tf_moe_ffn_decode_noalloc(x2, x2, table, idx, w, K, H, I, None)
        torch.cuda.synchronize()
        assert np.array_equal(bf16_bits(x2), want_o), step


def test_noalloc_rejects_sizes_beyond_its_scratch():
    d_exp = torch.zeros(16, dtype=torch.uint8, device=DEV)
    table = B.expert_table(d_exp, 16, n_experts=E)
    x = torch.zeros(H, dtype=torch.bfloat16, device=DEV)
    idx = torch.zeros(32, dtype=torch.int32, device=DEV)
    w = torch.zeros(32, dtype=torch.float32, device=DEV)
    I_big = (B.TF_NOALLOC_MAX_KI // 32 // 64 + 1) * 64      # k * I just above the array
    with pytest.raises(B.TFError) as e:
        B.tf_moe_ffn_decode_noalloc(x, x, table, idx, w, 32, H, I_big, None)
    assert e.value.status == B.TF_ERR_INVALID_ARG
    assert "scratch" in str(e.value)
    torch.cuda.synchronize()
