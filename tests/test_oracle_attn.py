"""Pins of the oracle's attention half of a decoder layer (CPU only).

The pages name hand-written attention and RoPE kernels and a resident FP16 KV
cache (page "Como executar um modelo de 26 bilhoes de parametros em dois
gigabytes de memoria em um Mac comum", sections "Sem dependencias do llama.cpp
e MLX" and "Qual e o principal truque da arquitetura") but give no shapes or
conventions. The oracle's reading (pre-norm grouped-query attention, RoPE on
the pairs (j, j + d/2), the cache rows rounded to fp16) is checked here against
what fixes it independently of its own code: exact special cases, numpy's
matrix product and float16 conversion, and the geometry of a rotation.
"""
import numpy as np
import pytest

import oracle as O

H, NQ, NKV, D, S = 128, 4, 2, 32, 16


def _bf16(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _f(bits16):
    return (np.asarray(bits16, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _h(bits16):
    return np.asarray(bits16, dtype=np.uint16).view(np.float16).astype(np.float64)


def _weights(seed, scale=0.2):
    rng = np.random.default_rng(seed)
    Wq = _bf16(rng.standard_normal((NQ * D, H)) * scale)
    Wk = _bf16(rng.standard_normal((NKV * D, H)) * scale)
    Wv = _bf16(rng.standard_normal((NKV * D, H)) * scale)
    Wo = _bf16(rng.standard_normal((H, NQ * D)) * scale)
    return Wq, Wk, Wv, Wo


def _x(seed):
    return _bf16(np.random.default_rng(seed).standard_normal(H))


def _cache():
    return np.zeros((S, NKV, D), np.uint16), np.zeros((S, NKV, D), np.uint16)


def _n(x):
    xf = _f(x)
    return xf / np.sqrt(np.mean(xf * xf) + O.EPS)


def test_single_position_returns_the_value_row():
    """With one cached position the softmax weight is 1: every head's output is its kv head's V row."""
    Wq, Wk, Wv, Wo = _weights(1)
    K, V = _cache()
    x = _x(2)
    _, sc, a = O.attn_decode(x, 0, Wq, Wk, Wv, Wo, K, V, NQ, NKV, D)
    a = a.reshape(NQ, D)
    for h in range(NQ):
        assert np.array_equal(a[h], _h(V[0, h // (NQ // NKV)]))
    assert sc.shape == (1,)


def test_cache_rows_at_position_zero_are_fp16_of_the_projections():
    """At position 0 RoPE turns by angle 0: K[0] and V[0] are the fp16 roundings of Wk n and Wv n."""
    Wq, Wk, Wv, Wo = _weights(3)
    K, V = _cache()
    x = _x(4)
    O.attn_decode(x, 0, Wq, Wk, Wv, Wo, K, V, NQ, NKV, D)
    n = _n(x)
    for W, C in ((Wk, K), (Wv, V)):
        ref = (_f(W) @ n).astype(np.float16).view(np.uint16)
        got = C[0].reshape(-1)
        ulps = np.abs(got.astype(np.int32) - ref.astype(np.int32))
        assert ulps.max() <= 1                 # fp64 -> fp32 -> fp16 against numpy's fp64 -> fp16
        assert np.mean(ulps == 0) > 0.98


def test_rope_turns_each_pair_by_its_angle():
    """Key pair (j, j + d/2) at position p is the position-0 pair turned by p * theta^(-2j/d):
    same length, angle difference p * theta^(-2j/d) (mod 2 pi), up to the fp16 rounding of the cache."""
    Wq, Wk, Wv, Wo = _weights(5)
    K, V = _cache()
    x = _x(6)
    for pos in range(6):
        O.attn_decode(x, pos, Wq, Wk, Wv, Wo, K, V, NQ, NKV, D)
    k0 = _h(K[0])
    for pos in (1, 5):
        kp = _h(K[pos])
        for g in range(NKV):
            for j in (0, 1, D // 2 - 1):
                a0, b0 = k0[g, j], k0[g, j + D // 2]
                ap, bp = kp[g, j], kp[g, j + D // 2]
                r0 = np.hypot(a0, b0)
                assert abs(np.hypot(ap, bp) - r0) <= 2e-3 * r0 + 1e-4
                turn = np.angle(complex(ap, bp) / complex(a0, b0))
                want = pos * 10000.0 ** (-2.0 * j / D)
                diff = (turn - want + np.pi) % (2 * np.pi) - np.pi
                assert abs(diff) < 3e-3


def test_scores_depend_on_the_relative_position_only():
    """With the same input at every position, s(pos, t) = s(pos + c, t + c) up to the fp16 cache rounding."""
    Wq, Wk, Wv, Wo = _weights(7)
    K, V = _cache()
    x = _x(8)
    sc = {}
    for pos in range(10):
        _, s, _ = O.attn_decode(x, pos, Wq, Wk, Wv, Wo, K, V, NQ, NKV, D)
        sc[pos] = s
    for c in (1, 3):
        for t in range(0, 6):
            assert abs(sc[6][t] - sc[6 + c][t + c]) <= 5e-3 * (1 + abs(sc[6][t]))


def test_zero_query_averages_the_values():
    """Wq = 0 gives equal scores, so each head's output is the mean of its kv head's cached V rows."""
    Wq, Wk, Wv, Wo = _weights(9)
    Wq = np.zeros_like(Wq)
    K, V = _cache()
    for pos in range(5):
        _, s, a = O.attn_decode(_x(100 + pos), pos, Wq, Wk, Wv, Wo, K, V, NQ, NKV, D)
    assert np.all(s == 0.0)
    a = a.reshape(NQ, D)
    for h in range(NQ):
        want = _h(V[:5, h // (NQ // NKV)]).mean(axis=0)
        assert np.allclose(a[h], want, rtol=1e-12, atol=1e-12)


def test_zero_output_projection_returns_the_input():
    Wq, Wk, Wv, Wo = _weights(11)
    K, V = _cache()
    x = _x(12)
    out, _, _ = O.attn_decode(x, 0, Wq, Wk, Wv, np.zeros_like(Wo), K, V, NQ, NKV, D)
    assert np.array_equal(out, x)


def test_grouped_query_heads_share_their_kv_head():
    """Only kv head 1 carries values: q heads 2 and 3 (nq / nkv = 2 per kv head) see them, heads 0 and 1 see zeros."""
    Wq, Wk, Wv, Wo = _weights(13)
    Wv = Wv.copy()
    Wv[:D] = 0
    K, V = _cache()
    _, _, a = O.attn_decode(_x(14), 0, Wq, Wk, Wv, Wo, K, V, NQ, NKV, D)
    a = a.reshape(NQ, D)
    assert np.all(a[0] == 0) and np.all(a[1] == 0)
    assert np.any(a[2] != 0) and np.array_equal(a[2], a[3])


@pytest.mark.parametrize("bits", [32, 64])
def test_output_is_the_residual_plus_the_projection(bits):
    """out = bf16(x + Wo a), checked with numpy's product on the oracle's own a."""
    Wq, Wk, Wv, Wo = _weights(15)
    K, V = _cache()
    x = _x(16)
    for pos in range(3):
        out, _, a = O.attn_decode(x, pos, Wq, Wk, Wv, Wo, K, V, NQ, NKV, D, bits=bits)
    want = _f(x) + _f(Wo) @ a.astype(np.float64)
    got = _f(out)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-6)


def test_scores_and_softmax_against_numpy():
    """Head 0 at position 0: s = q . K[0] / sqrt(d) with q = Wq n (no turn at position 0); at a later
    position the output of head 0 is numpy's softmax of the oracle's scores applied to the cached V rows."""
    Wq, Wk, Wv, Wo = _weights(17)
    K, V = _cache()
    x = _x(18)
    _, s0, _ = O.attn_decode(x, 0, Wq, Wk, Wv, Wo, K, V, NQ, NKV, D)
    q = _f(Wq) @ _n(x)
    want = q[:D] @ _h(K[0, 0]) / np.sqrt(D)
    assert abs(s0[0] - want) <= 1e-9 * (1 + abs(want))
    for pos in range(1, 7):
        _, s, a = O.attn_decode(_x(200 + pos), pos, Wq, Wk, Wv, Wo, K, V, NQ, NKV, D)
    p = np.exp(s - s.max())
    p /= p.sum()
    want_a = p @ _h(V[:7, 0])
    assert np.allclose(a[:D], want_a, rtol=1e-12, atol=1e-12)
