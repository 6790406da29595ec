"""GPU parity of the attention half of a decoder layer (tf_attn_decode) against the CPU oracle.

The oracle (oracle.attn_decode, fp64) and the CUDA path get the same seeded bf16
weights, hidden states and fp16 cache rows. Checked per decode step: the
layer update out - x against the oracle's Wo a (contract 1e-2, and a tighter
1e-3 that the fp32 arithmetic meets), and the cache rows the step writes (the
rotated keys and the values as fp16, within one fp16 step or 1e-5 of the row's
largest value: both sides round their own fp32 / fp64 sums).
"""
import numpy as np
import pytest
import torch

import bit_expert_streaming_layer_b300 as B
import oracle as O
import workload as W
from parity import CONTRACT_TOL, bf16_to_f64, delta_rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV)


def _h(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def _f16_close(got, want):
    """Within one fp16 step of the oracle's row, or 1e-5 of the row's largest value: both sides round their own
    sums (fp32 here, fp64 there) to fp16, and a value that is small against the row's terms keeps the fp32
    sum's absolute error, which can be several fp16 steps of that small value."""
    g, w = _h(got), _h(want)
    step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(w), 2.0 ** -14))) - 10)
    return bool(np.all(np.abs(g - w) <= np.maximum(1.01 * step, 1e-5 * np.max(np.abs(w)))))


class _Case:
    def __init__(self, seed, H, nq, nkv, d, max_seq):
        self.H, self.nq, self.nkv, self.d, self.max_seq = H, nq, nkv, d, max_seq
        self.w = W.attention_weights(seed, 0, H, nq, nkv, d)
        self.dw = [_dev(m) for m in self.w]
        self.desc = B.attn_desc(H, nq, nkv, d, max_seq, *self.dw)
        cb = B.tf_attn_cache_bytes(self.desc)
        assert cb == max_seq * nkv * d * 2
        self.kc = torch.zeros(cb // 2, dtype=torch.int16, device=DEV)
        self.vc = torch.zeros(cb // 2, dtype=torch.int16, device=DEV)
        self.ws_bytes = B.tf_attn_workspace_bytes(self.desc)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=DEV)
        self.K = np.zeros((max_seq, nkv, d), np.uint16)
        self.V = np.zeros((max_seq, nkv, d), np.uint16)

    def prefill(self, seed, rows):
        k, v = W.cache_rows(seed, 0, rows, self.nkv, self.d)
        self.K[:rows], self.V[:rows] = k, v
        n = rows * self.nkv * self.d
        self.kc[:n] = torch.from_numpy(k.reshape(-1).view(np.int16)).to(DEV)
        self.vc[:n] = torch.from_numpy(v.reshape(-1).view(np.int16)).to(DEV)

    def step(self, x_bits, pos):
        x = _dev(x_bits)
        out = torch.full((self.H,), -1, dtype=torch.int16, device=DEV)
        B.tf_attn_decode(self.desc, x, out, pos, self.kc, self.vc, self.ws, self.ws_bytes)
        torch.cuda.synchronize()
        ref_out, _, a = O.attn_decode(x_bits, pos, *self.w, self.K, self.V, self.nq, self.nkv, self.d)
        delta = (bf16_to_f64(self.w[3]).reshape(self.H, -1) @ a)
        got = out.cpu().numpy().view(np.uint16)
        return got, ref_out, delta

    def cache_row(self, pos):
        n = self.nkv * self.d
        k = self.kc[pos * n:(pos + 1) * n].cpu().numpy().view(np.uint16)
        v = self.vc[pos * n:(pos + 1) * n].cpu().numpy().view(np.uint16)
        return k, v


def test_attention_decode_steps_match_the_oracle():
    """Six decode steps from position 0 at the model's hidden size (16 q heads, 8 kv heads, d = 128)."""
    c = _Case(21, 2816, 16, 8, 128, 64)
    for pos in range(6):
        x = W.hidden(21, pos, 1, 2816)[0]
        got, ref, delta = c.step(x, pos)
        assert delta_rel_err(got, x, delta) <= 1e-3
        assert delta_rel_err(got, x, delta) <= CONTRACT_TOL
        k, v = c.cache_row(pos)
        assert _f16_close(k, c.K[pos].reshape(-1)) and _f16_close(v, c.V[pos].reshape(-1))
        # the oracle continues from its own cache; keep the GPU's rows equal to it for the next step
        c.kc[pos * 1024:(pos + 1) * 1024] = torch.from_numpy(c.K[pos].reshape(-1).view(np.int16)).to(DEV)
        c.vc[pos * 1024:(pos + 1) * 1024] = torch.from_numpy(c.V[pos].reshape(-1).view(np.int16)).to(DEV)


@pytest.mark.parametrize("H,nq,nkv,d,pos", [(2816, 16, 8, 128, 700), (1024, 8, 2, 64, 300),
                                            (1024, 4, 4, 256, 513), (512, 4, 1, 64, 255), (512, 2, 2, 128, 256)],
                         ids=["d128_3chunks", "d64_gqa4", "d256_mha", "d64_one_kv_head_full_chunk",
                              "d128_chunk_edge"])
def test_attention_decode_over_a_filled_cache(H, nq, nkv, d, pos):
    """One step at position pos over cache rows 0..pos-1 filled with seeded values: several chunks of 256
    positions, a ragged last chunk, and the lane groups of each head size."""
    c = _Case(31 + pos, H, nq, nkv, d, pos + 8)
    c.prefill(32 + pos, pos)
    x = W.hidden(33, pos, 1, H)[0]
    got, ref, delta = c.step(x, pos)
    assert delta_rel_err(got, x, delta) <= 1e-3
    k, v = c.cache_row(pos)
    assert _f16_close(k, c.K[pos].reshape(-1)) and _f16_close(v, c.V[pos].reshape(-1))
    # rows before pos are left as they were
    n = pos * nkv * d
    assert np.array_equal(c.kc[:n].cpu().numpy().view(np.uint16), c.K[:pos].reshape(-1))
    assert np.array_equal(c.vc[:n].cpu().numpy().view(np.uint16), c.V[:pos].reshape(-1))


def test_attention_then_moe_is_one_decoder_layer():
    """The decoder layer is the attention half followed by the MoE layer on its output: the attention output
    feeds tf_layer_step unchanged, and the chained result matches the two oracles chained."""
    from workload.model import SyntheticStack
    from test_gpu_decode import _check_layer, FULL
    H = FULL["H"]
    c = _Case(41, H, 16, 8, 128, 8)
    st = SyntheticStack(42, 1, **FULL)
    x = W.hidden(43, 0, 1, H)[0]
    got_attn, _, delta = c.step(x, 0)
    assert delta_rel_err(got_attn, x, delta) <= 1e-3
    mid = _dev(got_attn)
    out = torch.empty_like(mid)
    B.tf_layer_step(st.layers[0], None, 0, 0, None, mid, out, 1)
    torch.cuda.synchronize()
    _check_layer(st, 0, got_attn, out.cpu().numpy().view(np.uint16))
    st.close()
