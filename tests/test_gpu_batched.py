"""GPU parity of the batched layer step (tf_layer_step with T > 1) against the
CPU oracle, through the C ABI.

T tokens go through the router, the grouped routed experts and the bf16 shared
expert, both on the tcgen05 GEMM kernel. The oracle is the per-token decode
layer with the shared expert, in its tensor-core reading (x fed as it is with
the RMS scale applied after the gate/up sums; fp16 weights and h for the routed
experts, bf16 h for the shared expert; fp32 accumulation) and in its plain fp32
reading (the contract). Checked per token: the RMS scale, the router logits and top-k ids
bit for bit, the weights to a few ulp, and the output and its update within
the contract tolerance against both readings. The layer step exposes no fp32
update, so the update is out - x, allowed the bf16 output's own rounding
(1.5 ulp of out, see parity.delta_rel_err). Small shapes check every
token; the model's shape with 64 tokens (the batched-decode workload) checks
sampled tokens.
"""
import numpy as np
import pytest
import torch

import bit_expert_streaming_layer_b300 as B
import oracle as O
import workload as W
from parity import CONTRACT_TOL, bf16_to_f64, delta_rel_err, max_rel_err, out_rel_err
from workload.model import SyntheticStack, bf16_bits, hidden_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(seed, T, cfg, steps=1):
    st = SyntheticStack(seed, 1, T_max=T, **cfg)
    lay = st.layers[0]
    outs, xs, routes = [], [], []
    x = hidden_tensor(seed, 0, T, cfg["H"])
    for step in range(steps):
        out = torch.full_like(x, float("nan"))
        B.tf_layer_step(lay, None, 0, step, None, x, out, T)
        torch.cuda.synchronize()
        idx, w, logits, rms = (t.cpu().numpy().copy() for t in lay.routing_tensors(T))
        outs.append(bf16_bits(out))
        xs.append(bf16_bits(x))
        routes.append((idx, w, logits, rms))
        x = out
    return st, outs, xs, routes


def _check(seed, cfg, st, x_bits, out_bits, route, tokens):
    H, I, E, k, S = cfg["H"], cfg["I"], cfg["E"], cfg["k"], cfg["S"]
    idx_g, w_g, lg_g, rms_g = route
    Wr = W.router_weights(seed, 0, E, H)
    shared = W.shared_weights(seed, 0, H, S)
    cache = {}
    worst = 0.0
    for t in tokens:
        r, z, idx, w = O.route(x_bits[t], Wr, None, k)
        assert np.float32(rms_g[t]).view(np.uint32) == np.float32(r).view(np.uint32), t
        assert np.array_equal(lg_g[t].view(np.uint32), z.view(np.uint32)), t
        assert idx_g[t].tolist() == idx.tolist(), t
        assert np.max(np.abs(w_g[t] - w)) <= 4e-7
        for e in idx:
            if int(e) not in cache:
                cache[int(e)] = W.expert(seed, 0, int(e), H, I)
        ex = [cache[int(e)] for e in idx]
        out_o, delta_o = O.layer_combine(x_bits[t], r, ex, w, shared, tc=True)
        got = bf16_to_f64(out_bits[t])
        assert not np.isnan(got).any(), t
        assert max_rel_err(got, bf16_to_f64(out_o)) <= CONTRACT_TOL, t
        err = delta_rel_err(out_bits[t], x_bits[t], delta_o)
        assert err <= CONTRACT_TOL, (t, err)
        worst = max(worst, err)
        # the contract as written: the bf16 tensor-core path against the plain fp32 oracle (the bf16 output
        # against the oracle's exact x + delta, allowing the output's own rounding to bf16)
        _, delta_f = O.layer_combine(x_bits[t], r, ex, w, shared, tc=False)
        err_fo = out_rel_err(out_bits[t], x_bits[t], delta_f)
        assert err_fo <= CONTRACT_TOL, (t, err_fo)
        err_f = delta_rel_err(out_bits[t], x_bits[t], delta_f)
        assert err_f <= CONTRACT_TOL, (t, err_f)
    return worst


@pytest.mark.parametrize("cfg,T", [
    (dict(H=512, I=256, E=16, k=4, S=192), 37),      # ragged token tile, several shared tiles
    (dict(H=256, I=128, E=8, k=2, S=64), 300),      # more than one 256-token tile for the shared expert
    (dict(H=512, I=256, E=16, k=4, S=192), 2),
], ids=["small", "two_tiles", "two_tokens"])
def test_batched_step_small_all_tokens(cfg, T):
    seed = 71
    st, outs, xs, routes = _run(seed, T, cfg, steps=2)
    worst = 0.0
    for s in range(2):
        worst = max(worst, _check(seed, cfg, st, xs[s], outs[s], routes[s], range(T)))
    assert worst < 5e-3
    st.close()


def test_batched_step_model_shape_64_tokens():
    """H = 2816, I = 704, E = 128, k = 8, S = 2112: the batched-decode layer, 64 tokens."""
    cfg = dict(H=2816, I=704, E=128, k=8, S=2112)
    seed, T = 73, 64
    st, outs, xs, routes = _run(seed, T, cfg)
    tokens = sorted(set(np.random.default_rng(seed).choice(T, 6, replace=False).tolist()) | {0, T - 1})
    _check(seed, cfg, st, xs[0], outs[0], routes[0], tokens)
    assert not np.isnan(bf16_to_f64(outs[0])).any()
    st.close()


def test_batched_step_is_deterministic_and_order_equivariant():
    cfg = dict(H=512, I=256, E=16, k=4, S=192)
    seed, T = 79, 48
    st = SyntheticStack(seed, 1, T_max=T, **cfg)
    lay = st.layers[0]
    x = hidden_tensor(seed, 0, T, cfg["H"])
    a, b = torch.empty_like(x), torch.empty_like(x)
    B.tf_layer_step(lay, None, 0, 0, None, x, a, T)
    B.tf_layer_step(lay, None, 0, 0, None, x, b, T)
    order = torch.from_numpy(np.random.default_rng(seed).permutation(T)).to(DEV)
    c = torch.empty_like(x)
    B.tf_layer_step(lay, None, 0, 0, None, x[order].contiguous(), c, T)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(c.view(torch.int16), a[order].view(torch.int16))
    st.close()
