"""GPU parity of the grouped (batched / prefill) routed-expert path,
tf_moe_ffn_grouped, against the CPU oracle, through the C ABI.

The oracle is the per-token decode layer, looped over tokens, in two readings:
its tensor-core reading (x fed as it is, the RMS scale applied after the
gate/up sums, every dequantised weight and h rounded to fp16, fp32
accumulation; the kernel's own roundings) and its plain fp32 reading (the
contract: the tensor-core path within 1e-2 of the fp32 oracle). Checked:
  - the permutation and the per-expert counts exactly (a stable sort by expert
    of the (token, rank) pairs, and the histogram of the ids);
  - every token's output and update within the contract tolerance, on all
    tokens of the small cases and on sampled tokens (always including tokens
    of the most loaded expert) at the model's full shape;
  - full coverage (outputs start as NaN) and shapes with ragged tails: experts
    with no tokens, experts with more than one 256-token GEMM tile, T = 1.
"""
import numpy as np
import pytest
import torch

import bit_expert_streaming_layer_b300 as B
import oracle as O
import workload as W
from parity import CONTRACT_TOL, bf16_to_f64, max_rel_err, out_rel_err
from workload.model import bf16_bits, hidden_tensor, pack_layer_experts

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _experts_device(seed, E, H, I):
    slot = B.tf_expert_slot_bytes(H, I)
    host = torch.empty(E * slot, dtype=torch.uint8, pin_memory=True)
    pack_layer_experts(seed, 0, E, H, I, host)
    return host.to(DEV), slot


def _routing(seed, T, E, k, zipf_s, skip=()):
    """Seeded top-k ids (distinct per token, Zipf(zipf_s) popularity over a random
    rank -> expert map; experts in `skip` never chosen) and positive weights summing to 1."""
    rng = np.random.default_rng(seed)
    allowed = np.array([e for e in range(E) if e not in skip])
    p = np.arange(1, len(allowed) + 1, dtype=np.float64) ** -zipf_s
    p /= p.sum()
    ranked = rng.permutation(allowed)
    idx = np.stack([ranked[rng.choice(len(allowed), k, replace=False, p=p)] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)) + 0.05
    w = (w / w.sum(1, keepdims=True)).astype(np.float32)
    return idx, w


def _run(x, idx, w, d_exp, slot, E, k, H, I):
    T = x.shape[0]
    ws = torch.zeros(B.tf_moe_grouped_workspace_bytes(T, H, I, E, k), dtype=torch.uint8, device=DEV)
    out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    delta = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    perm = torch.full((T * k,), -1, dtype=torch.int32, device=DEV)
    counts = torch.full((E,), -1, dtype=torch.int32, device=DEV)
    d_idx = torch.from_numpy(idx).to(DEV)
    d_w = torch.from_numpy(w).to(DEV)
    B.tf_moe_ffn_grouped(x, out, T, B.expert_table(d_exp, slot), E, d_idx, d_w, k, H, I, delta, perm, counts, ws,
                         ws.numel())
    torch.cuda.synchronize()
    return bf16_bits(out), delta.cpu().numpy(), perm.cpu().numpy(), counts.cpu().numpy()


def _check_permutation(idx, perm, counts, E):
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert np.array_equal(perm, np.argsort(idx.ravel(), kind="stable").astype(np.int32))


def _check_tokens(seed, x_bits, idx, w, out_bits, delta, tokens, H, I, worst_fp32=None):
    """Per token: output and update within the contract against the oracle's tensor-core reading and
    against its plain fp32 reading; returns the worst update error of the former (worst_fp32[0] gets the
    worst of the latter)."""
    worst_fp32 = worst_fp32 if worst_fp32 is not None else [0.0]
    cache = {}
    worst = 0.0
    for t in tokens:
        for e in idx[t]:
            if int(e) not in cache:
                cache[int(e)] = W.expert(seed, 0, int(e), H, I)
        r = O.rms_scale(x_bits[t])
        ex = [cache[int(e)] for e in idx[t]]
        got_o = bf16_to_f64(out_bits[t])
        assert not np.isnan(got_o).any() and not np.isnan(delta[t]).any(), t
        # the tensor-core reading (the kernel's own roundings): tight
        out_o, delta_o = O.layer_combine(x_bits[t], r, ex, w[t], None, tc=True)
        e_out = max_rel_err(got_o, bf16_to_f64(out_o))
        e_delta = max_rel_err(delta[t], delta_o)
        assert e_out <= CONTRACT_TOL, (t, e_out)
        assert e_delta <= CONTRACT_TOL, (t, e_delta)
        worst = max(worst, e_delta)
        # the contract as written: the bf16 tensor-core path against the plain fp32 oracle (the bf16 output
        # against the oracle's exact x + delta, allowing the output's own rounding to bf16)
        _, delta_f = O.layer_combine(x_bits[t], r, ex, w[t], None, tc=False)
        e_f = max_rel_err(delta[t], delta_f)
        assert e_f <= CONTRACT_TOL, (t, e_f)
        e_fo = out_rel_err(out_bits[t], x_bits[t], delta_f)
        assert e_fo <= CONTRACT_TOL, (t, e_fo)
        worst_fp32[0] = max(worst_fp32[0], e_f)
    return worst


@pytest.mark.parametrize("H,I,E,k,T,zipf_s,skip", [
    (512, 256, 16, 4, 37, 0.0, (5,)),        # one tile per expert, an expert with no tokens
    (512, 256, 8, 2, 700, 1.2, ()),          # skewed: the top experts span several 256-token tiles
    (512, 256, 16, 4, 1, 0.0, ()),           # a single token
], ids=["small", "multi_tile", "one_token"])
def test_grouped_small_all_tokens(H, I, E, k, T, zipf_s, skip):
    seed = 31
    d_exp, slot = _experts_device(seed, E, H, I)
    x = hidden_tensor(seed, 0, T, H)
    x_bits = bf16_bits(x)
    idx, w = _routing(seed, T, E, k, zipf_s, skip)
    out, delta, perm, counts = _run(x, idx, w, d_exp, slot, E, k, H, I)
    _check_permutation(idx, perm, counts, E)
    for e in skip:
        assert counts[e] == 0
    worst_fp32 = [0.0]
    worst = _check_tokens(seed, x_bits, idx, w, out, delta, range(T), H, I, worst_fp32)
    assert worst < 5e-3
    assert worst_fp32[0] < CONTRACT_TOL


def _sampled_tokens(idx, counts, n, seed):
    rng = np.random.default_rng(seed)
    top = int(np.argmax(counts))
    with_top = np.nonzero((idx == top).any(1))[0]
    pick = set(rng.choice(idx.shape[0], n, replace=False).tolist())
    pick.update(with_top[:2].tolist())
    pick.update([0, idx.shape[0] - 1])
    return sorted(pick)


@pytest.mark.parametrize("T,zipf_s", [(512, 1.2), (4096, 1.2)], ids=["full_512", "prefill_4096"])
def test_grouped_full_shape_sampled(T, zipf_s):
    """The model's shape (H = 2816, I = 704, E = 128, k = 8); T = 4096 with a
    Zipf(1.2) skew is the prefill-shaped layer."""
    H, I, E, k, seed = 2816, 704, 128, 8, 41
    d_exp, slot = _experts_device(seed, E, H, I)
    x = hidden_tensor(seed, 1, T, H)
    x_bits = bf16_bits(x)
    idx, w = _routing(seed, T, E, k, zipf_s)
    out, delta, perm, counts = _run(x, idx, w, d_exp, slot, E, k, H, I)
    _check_permutation(idx, perm, counts, E)
    assert counts.max() > 256  # several token tiles for the most loaded expert
    assert not np.isnan(bf16_to_f64(out)).any() and not np.isnan(delta).any()
    _check_tokens(seed, x_bits, idx, w, out, delta, _sampled_tokens(idx, counts, 8, seed), H, I)


def test_grouped_is_deterministic_and_token_order_equivariant():
    """Permuting the tokens permutes the outputs bit for bit (each token's sum
    runs in its own top-k order, whatever the rows' positions)."""
    H, I, E, k, T, seed = 512, 256, 16, 4, 96, 53
    d_exp, slot = _experts_device(seed, E, H, I)
    x = hidden_tensor(seed, 2, T, H)
    idx, w = _routing(seed, T, E, k, 1.0)
    out1, d1, _, _ = _run(x, idx, w, d_exp, slot, E, k, H, I)
    out2, d2, _, _ = _run(x, idx, w, d_exp, slot, E, k, H, I)
    assert np.array_equal(out1, out2) and np.array_equal(d1.view(np.uint32), d2.view(np.uint32))
    order = np.random.default_rng(seed).permutation(T)
    out3, d3, _, _ = _run(x[torch.from_numpy(order).to(DEV)].contiguous(), idx[order], w[order], d_exp, slot, E, k, H,
                          I)
    assert np.max(np.abs(bf16_to_f64(out3) - bf16_to_f64(out1[order]))) == 0.0


def test_grouped_inputs_beyond_fp16_range():
    """Hidden states far beyond the fp16 range (x scaled by 2^16, up to about 3e5): the fp16 operand is x times
    the power of two of its RMS scale, so the outputs stay finite and within the contract of both readings."""
    H, I, E, k, T, seed = 512, 256, 16, 4, 24, 37
    d_exp, slot = _experts_device(seed, E, H, I)
    x = hidden_tensor(seed, 0, T, H) * 65536.0
    x_bits = bf16_bits(x)
    assert np.max(np.abs(bf16_to_f64(x_bits))) > 65504.0
    idx, w = _routing(seed, T, E, k, 0.0)
    out, delta, perm, counts = _run(x, idx, w, d_exp, slot, E, k, H, I)
    _check_permutation(idx, perm, counts, E)
    worst_fp32 = [0.0]
    worst = _check_tokens(seed, x_bits, idx, w, out, delta, range(T), H, I, worst_fp32)
    assert worst < 5e-3 and worst_fp32[0] < CONTRACT_TOL
