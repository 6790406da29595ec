"""Pins of the CPU oracle against things other than itself (CPU only).

Each test ties one oracle function to a fixed fact of the pages, a closed form,
a brute-force enumeration, an independent library routine or a hand-worked
trace, so that a dropped term, a wrong sign or index or a transposed operand in
the oracle fails somewhere here.

Pages cited (by title):
  [HN]  "Show HN: mecanismo de codigo aberto executando Gemma 4 26B em 2 GB de RAM em
         qualquer Mac com serie M" (hndistilled.com), section "Abordagem tecnica (MoE +
         streaming por SSD)".
  [DT]  "Como executar um modelo de 26 bilhoes de parametros em dois gigabytes de memoria
         em um Mac comum" (devtrends.cc), section "Qual e o principal truque da arquitetura".
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
import workload as W
from golden_io import load_lfu_trace, lfu_trace_names

H, I, E, K_ACT, SLOTS, LAYERS = 2816, 704, 128, 8, 16, 30


# ----------------------------------------------------------------------- fixed facts

def expert_payload_bytes(H, I, group=64):
    """Bytes of one expert at 4 bits: codes (half a byte each) + fp16 scale and bias per group."""
    per_matrix = I * H // 2 + 2 * (I * H // group) * 2
    return 3 * per_matrix


def test_fact_expert_size_3_36_MB():
    # [HN]: one expert is 3.36 MB at 4 bits.
    payload = expert_payload_bytes(H, I)
    assert payload == 3_345_408
    stride = -(-payload // 16384) * 16384
    assert stride == 3_358_720
    assert f"{stride / 1e6:.2f}" == "3.36"
    assert f"{payload / 1e6:.2f}" == "3.35"


def test_fact_bytes_per_token_band():
    # [HN]: 60-70% hit rate and 250-320 MB read per token, 30 layers x 8 experts.
    per_expert = 3_358_720
    lo = LAYERS * K_ACT * per_expert * (1 - 0.70) / 1e6
    hi = LAYERS * K_ACT * per_expert * (1 - 0.60) / 1e6
    assert 240 < lo < 250 and 320 < hi < 325      # overlaps the quoted 250-320 MB
    # [DT]: ~14.3 GB of 4-bit weights with a 1.35 GB resident core.
    total = LAYERS * E * expert_payload_bytes(H, I) / 1e9 + 1.35
    assert abs(total - 14.3) < 0.15


def test_fact_eight_active_experts_distinct():
    # [DT]: the router of each layer picks 8 experts for the token.
    x = W.hidden(0, 0, 1, H)[0]
    Wr = W.router_weights(0, 0, E, H)
    r, z, idx, w = O.route(x, Wr)
    assert idx.shape == (8,) and len(set(idx.tolist())) == 8
    assert np.all((idx >= 0) & (idx < E))


def test_fact_sixteen_slots_lfu_resident():
    # [DT]: 16 slots with LFU; after each step all 8 current experts are resident.
    rng = np.random.default_rng(0)
    lfu = O.LFU(1, SLOTS)
    for step in range(200):
        ids = rng.choice(E, 8, replace=False).astype(np.int32)
        lfu.step(step, 0, ids)
        ex, cnt, lu = lfu.state(0)
        assert set(ids.tolist()) <= set(ex.tolist())
        assert (ex >= 0).sum() <= SLOTS


# ------------------------------------------------------------------------- encodings

def test_half_to_float_all_codes():
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float32)
    got = np.array([O.half_to_float(int(c)) for c in codes], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _nearest_bf16_bruteforce(f32):
    """Round an fp32 to bf16 by comparing the two neighbouring bf16 values exactly."""
    u = int(np.float32(f32).view(np.uint32))
    lo = u >> 16
    cand = [lo, lo + 1]
    vals = [Fraction(float(np.uint32((c & 0xFFFF) << 16).view(np.float32))) for c in cand]
    x = Fraction(float(f32))
    d = [abs(v - x) for v in vals]
    if d[0] < d[1]:
        return cand[0] & 0xFFFF
    if d[1] < d[0]:
        return cand[1] & 0xFFFF
    return cand[0] & 0xFFFF if cand[0] % 2 == 0 else cand[1] & 0xFFFF


def test_float_to_bf16_round_nearest_even():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, 4000, dtype=np.uint64).astype(np.uint32)
    bits = bits[((bits >> 23) & 0xFF) < 0xFE]         # finite, away from overflow
    ties = (rng.integers(0, 2**15, 400).astype(np.uint32) << 16) | 0x8000   # exact halfway cases
    ties = ties[((ties >> 23) & 0xFF) < 0xFE]
    for b in np.concatenate([bits, ties.astype(np.uint32)]):
        f = np.uint32(b).view(np.float32)
        assert O.float_to_bf16(float(f)) == _nearest_bf16_bruteforce(f), hex(int(b))


# -------------------------------------------------------------------------- dequant

def test_dequant_zero_code_is_bias_exactly():
    s = W.uniform_f16(W.key(9, W.T_S), 500, W.SCALE_LO, W.SCALE_HI)
    b = W.uniform_f16(W.key(9, W.T_B), 500, W.BIAS_LO, W.BIAS_HI)
    for si, bi in zip(s, b):
        assert O.dequant(0, int(si), int(bi)) == np.float16(np.uint16(bi).view(np.float16)).astype(np.float32)


def test_dequant_single_rounding_of_exact_value():
    # s*q + b computed exactly (Fraction), then rounded once to fp32 (numpy, RN-even).
    s = W.uniform_f16(W.key(10, W.T_S), 300, W.SCALE_LO, W.SCALE_HI)
    b = W.uniform_f16(W.key(10, W.T_B), 300, W.BIAS_LO, W.BIAS_HI)
    for si, bi in zip(s, b):
        sv = Fraction(float(np.uint16(si).view(np.float16)))
        bv = Fraction(float(np.uint16(bi).view(np.float16)))
        for q in range(16):
            exact = sv * q + bv
            want = np.float32(float(exact))   # float(exact) is exact here (<= 53 bits); one fp32 rounding
            assert O.dequant(q, int(si), int(bi)) == want


def test_dequant_power_of_two_exact_and_requant_roundtrip():
    for sexp in (-8, -7, -6):
        s16 = int(np.float16(2.0 ** sexp).view(np.uint16))
        for b in (-0.0625, 0.0, 0.03125):
            b16 = int(np.float16(b).view(np.uint16))
            for q in range(16):
                assert O.dequant(q, s16, b16) == q * 2.0 ** sexp + b
    s = W.uniform_f16(W.key(11, W.T_S), 400, W.SCALE_LO, W.SCALE_HI)
    b = W.uniform_f16(W.key(11, W.T_B), 400, W.BIAS_LO, W.BIAS_HI)
    for si, bi in zip(s, b):
        sv = float(np.uint16(si).view(np.float16))
        bv = float(np.uint16(bi).view(np.float16))
        for q in range(16):
            w = O.dequant(q, int(si), int(bi))
            assert round((w - bv) / sv) == q


def test_dequant_matrix_layout_and_bf16_variant():
    R, K = 5, 192
    q, s, b = W.expert_matrix(3, 0, 0, 0, R, K)
    Wm = O.dequant_matrix(q, s, b)
    Wb = O.dequant_matrix(q, s, b, fmt="bf16")
    Wh = O.dequant_matrix(q, s, b, fmt="fp16")
    # fp16 weights: numpy's own round-to-nearest-even conversion of the fp32 weight
    assert np.array_equal(Wh, Wm.astype(np.float16).astype(np.float32))
    sf, bf = W.f16_to_f32(s), W.f16_to_f32(b)
    for j in range(R):
        for k in range(K):
            g = k // 64
            assert Wm[j, k] == np.float32(float(Fraction(float(sf[j, g])) * int(q[j, k]) + Fraction(float(bf[j, g]))))
            assert O.float_to_bf16(float(Wm[j, k])) == _nearest_bf16_bruteforce(Wm[j, k])
            assert Wb[j, k] == W.bf16_to_f32(np.array([_nearest_bf16_bruteforce(Wm[j, k])], np.uint16))[0]


# --------------------------------------------------------------------------- RMSNorm, router

def test_rms_scale_matches_fp64_closed_form():
    for seed in range(5):
        x = W.hidden(seed, 0, 1, H)[0]
        xf = W.bf16_to_f32(x).astype(np.float64)
        ref = 1.0 / math.sqrt(float(np.mean(xf * xf)) + 1e-6)
        r = O.rms_scale(x)
        assert abs(r - ref) <= 4 * np.spacing(np.float32(ref))


def test_router_logits_within_fp32_bound_of_exact():
    x = W.hidden(2, 0, 1, H)[0]
    Wr = W.router_weights(2, 0, E, H)
    bias, _ = W.zipf_bias(2, 0, E, 1.1)
    r = O.rms_scale(x)
    z = O.router_logits(x, Wr, bias, r)
    xf = W.bf16_to_f32(x).astype(np.float64)
    Wf = W.bf16_to_f32(Wr).astype(np.float64)
    exact = r * (Wf @ xf) + bias.astype(np.float64)
    bound = (H * 2.0 ** -24 * (np.abs(Wf) @ np.abs(xf)) * r + np.abs(exact) * 2.0 ** -22)
    assert np.all(np.abs(z - exact) <= bound)


def _rank_key(z, e):
    return (-(z if not math.isnan(z) else -math.inf), e)


def test_topk_bruteforce_small_with_ties():
    rng = np.random.default_rng(5)
    for trial in range(60):
        En = int(rng.integers(8, 13))
        k = int(rng.integers(1, min(8, En) + 1))
        z = rng.integers(-3, 4, En).astype(np.float32)       # many deliberate ties
        if trial % 5 == 0:
            z[rng.integers(0, En)] = -0.0
        best = None
        for subset in itertools.combinations(range(En), k):
            inside = set(subset)
            ok = all(_rank_key(float(z[a]), a) < _rank_key(float(z[b]), b)
                     for a in inside for b in range(En) if b not in inside)
            if ok:
                assert best is None
                best = subset
        want = sorted(best, key=lambda e: _rank_key(float(z[e]), e))
        assert O.topk(z, k).tolist() == want


def test_topk_full_sort_E128():
    rng = np.random.default_rng(6)
    for _ in range(50):
        z = (rng.standard_normal(E) * 2).astype(np.float32)
        z[rng.integers(0, E, 10)] = z[rng.integers(0, E)]       # ties
        order = np.lexsort((np.arange(E), -z.astype(np.float64)))
        assert O.topk(z, 8).tolist() == order[:8].tolist()


def test_routing_weights_sum_to_one_and_descend():
    for seed in range(20):
        x = W.hidden(seed, 0, 1, H)[0]
        Wr = W.router_weights(seed, 0, E, H)
        r, z, idx, w = O.route(x, Wr)
        s = np.float32(0)
        for v in w:
            s = np.float32(s + v)
        assert abs(float(s) - 1.0) <= 8 * 2.0 ** -24
        assert np.all(np.diff(w) <= 0)
        # softmax over the selected 8 == full softmax restricted and renormalised (fp64)
        zz = z.astype(np.float64)
        p = np.exp(zz - zz.max())
        p = p / p.sum()
        ref = p[idx] / p[idx].sum()
        assert np.allclose(w, ref, rtol=1e-6, atol=0)


# ----------------------------------------------------------------------------- GELU

def test_gelu_special_values_and_identity():
    assert O.gelu(0.0) == 0.0
    for v in (10.0, 20.0, 50.0):
        assert O.gelu(v) == np.float32(v)
    assert abs(O.gelu(-20.0)) < 1e-30
    for v in np.linspace(-8, 8, 161):
        v = float(np.float32(v))
        # gelu(v) - gelu(-v) = v for the tanh form (odd part of 0.5 v (1 + tanh(.)))
        assert abs((O.gelu(v, 64) - O.gelu(-v, 64)) - v) < 1e-12 * max(1.0, abs(v))


def test_gelu_close_to_exact_gaussian_cdf_form():
    # The tanh form approximates v * Phi(v) within ~1e-3 (Hendrycks & Gimpel 2016);
    # dropping the cubic term or mis-scaling the constant exceeds this bound.
    for v in np.linspace(-6, 6, 241):
        exact = v * 0.5 * (1 + math.erf(v / math.sqrt(2)))
        assert abs(O.gelu(float(v), 64) - exact) < 1.1e-3


def test_gelu_fp32_within_bound_of_fp64():
    # relative 2e-6, plus the cancellation in 1 + tanh(.) for negative v: |v|/2 * ulp(1)
    for v in np.linspace(-12, 12, 481):
        v32 = float(np.float32(v))
        a, b = O.gelu(v32, 32), O.gelu(v32, 64)
        assert abs(a - b) <= 2e-6 * abs(b) + 4e-8 * abs(v32)


# ---------------------------------------------------------------------- expert FFN

def _const_f16(v, shape):
    return np.full(shape, np.float16(v).view(np.uint16), np.uint16)


def test_expert_ffn_permutation_closed_form():
    """Gate = permutation, up = all-ones rows, down = another permutation (s = 1, b = 0):
    y_j = gelu(n_{pi(sigma(j))}) * sum(n). Pins nibble/row/column indexing of all three
    matrices, the GELU gate and the down projection; a transposed operand fails."""
    Hs, Is = 256, 128
    rng = np.random.default_rng(7)
    pi = rng.permutation(Hs)[:Is]          # gate row j picks column pi[j]
    sigma = rng.integers(0, Is, Hs)        # down row j picks column sigma[j]
    qg = np.zeros((Is, Hs), np.uint8)
    qg[np.arange(Is), pi] = 1
    qu = np.zeros((Is, Hs), np.uint8)
    qd = np.zeros((Hs, Is), np.uint8)
    qd[np.arange(Hs), sigma] = 1
    one, zero = _const_f16(1.0, (Is, Hs // 64)), _const_f16(0.0, (Is, Hs // 64))
    ex = {"gate": (qg, one, zero),
          "up": (qu, _const_f16(0.5, (Is, Hs // 64)), one),     # q = 0 -> every weight is b = 1
          "down": (qd, _const_f16(1.0, (Hs, Is // 64)), _const_f16(0.0, (Hs, Is // 64)))}
    n = rng.standard_normal(Hs).astype(np.float64)
    y = O.expert_ffn(n, ex, bits=64)
    S = n.sum()
    gel = lambda v: 0.5 * v * (1 + math.tanh(math.sqrt(2 / math.pi) * (v + 0.044715 * v ** 3)))
    want = np.array([gel(n[pi[sigma[j]]]) * S for j in range(Hs)])
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)


def test_expert_ffn_group_constant_code():
    """A constant code c in one group of a row gives (s c + b) * sum_{k in group} n_k."""
    Hs, Is = 320, 64
    rng = np.random.default_rng(8)
    n = rng.standard_normal(Hs)
    for g in range(Hs // 64):
        q = np.zeros((Is, Hs), np.uint8)
        c = int(rng.integers(1, 16))
        q[:, 64 * g:64 * g + 64] = c
        s = _const_f16(0.0, (Is, Hs // 64))
        b = _const_f16(0.0, (Is, Hs // 64))
        s[:, g] = np.float16(0.125).view(np.uint16)
        b[:, g] = np.float16(-0.25).view(np.uint16)
        Wm = O.dequant_matrix(q, s, b, bits=64)
        assert np.allclose(Wm @ n, (0.125 * c - 0.25) * n[64 * g:64 * g + 64].sum(), rtol=1e-12)


def test_shared_ffn_closed_form():
    Hs, Ss = 192, 96
    rng = np.random.default_rng(9)
    pi = rng.permutation(Hs)[:Ss]
    sigma = rng.integers(0, Ss, Hs)
    one = np.float32(1.0).view(np.uint32) >> 16
    two = np.float32(2.0).view(np.uint32) >> 16
    Wg = np.zeros((Ss, Hs), np.uint16)
    Wg[np.arange(Ss), pi] = one
    Wu = np.full((Ss, Hs), two, np.uint16)
    Wd = np.zeros((Hs, Ss), np.uint16)
    Wd[np.arange(Hs), sigma] = one
    n = rng.standard_normal(Hs)
    y = O.shared_ffn(n, Wg, Wu, Wd, bits=64)
    gel = lambda v: 0.5 * v * (1 + math.tanh(math.sqrt(2 / math.pi) * (v + 0.044715 * v ** 3)))
    want = np.array([gel(n[pi[sigma[j]]]) * 2 * n.sum() for j in range(Hs)])
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)


def _rn_bf16(v) -> np.float64:
    """fp32(v) rounded to the nearest bf16 (ties to even), by exhaustive comparison of the two neighbours."""
    f = np.float32(v)
    return np.float64(W.bf16_to_f32(np.array([_nearest_bf16_bruteforce(f)], np.uint16))[0])


def _rn_f16(v) -> np.float64:
    """fp32(v) rounded to the nearest fp16 (ties to even), by numpy's conversion."""
    return np.float64(np.float16(np.float32(v)))


def test_float_to_half_round_nearest_even():
    rng = np.random.default_rng(3)
    vals = rng.standard_normal(20000).astype(np.float32) * (np.float32(10.0) ** rng.integers(-9, 5, 20000))
    ties = (np.arange(1, 2048, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -24)   # subnormal ties
    ties2 = (np.arange(1024, 2048, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -3)  # normal ties
    edge = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -70000.0, 2.0 ** -25, 2.0 ** -24, 6.1e-5],
                    np.float32)
    with np.errstate(over="ignore"):
        for v in np.concatenate([vals.astype(np.float32), ties, ties2, edge]):
            assert O.float_to_half(float(v)) == int(np.float32(v).astype(np.float16).view(np.uint16)), v


def _gelu64(v):
    return 0.5 * v * (1 + math.tanh(math.sqrt(2 / math.pi) * (v + 0.044715 * v ** 3)))


def _spread_input(rng, n):
    """Values of magnitude in [1/8, 4) whose fp32 form is almost never a bf16 value: rounding them to bf16
    changes them, and every bf16 value of this range is a multiple of 2^-10, so sums of up to 2^10 of them
    are exact in fp64 (and in fp32)."""
    mag = 2.0 ** rng.uniform(-3, 2, n)
    return np.where(rng.random(n) < 0.5, -mag, mag).astype(np.float32).astype(np.float64)


def _bf16_branch_variants(n, pi, sigma, wg=1.0, wu=1.0, c=1.0, rnd=_rn_bf16):
    """Closed forms of y = Wd (gelu(c Wg n) * (c Wu n)) for gate rows e_pi(j) * wg, up rows all wu, down rows
    e_sigma(j) (exact weights), in a rounded-operand reading (rnd: bf16 or fp16) and in the readings a slip
    would produce."""
    _rn_bf16 = rnd
    nb = np.array([_rn_bf16(v) for v in n])
    out = {}
    for name, nn, round_h, round_gu in (("bf16 n and h", nb, True, False), ("fp32 n", n, True, False),
                                        ("no h rounding", nb, False, False), ("g, u rounded", nb, False, True)):
        U = c * (wu * nn.sum())
        h = []
        for j in range(len(pi)):
            g = c * (wg * nn[pi[j]])
            u = U
            if round_gu:
                g, u = _rn_bf16(g), _rn_bf16(u)
            v = _gelu64(g) * u
            h.append(_rn_bf16(v) if round_h else v)
        out[name] = np.array([h[sigma[j]] for j in range(len(sigma))])
    return out


def _assert_only_reading(y, variants, want="bf16 n and h"):
    assert np.array_equal(y, variants[want])
    for name, v in variants.items():
        if name != want:
            assert not np.allclose(y, v, rtol=1e-6, atol=0), name   # the pin tells the readings apart


def test_expert_ffn_bf16_operands_closed_form():
    """The bf16 reading of an expert (fmt = "bf16"): n, every dequantised weight and h
    are rounded to bf16 before their products. Gate = permutation, up = all-ones rows, down = another
    permutation (weights exact in bf16), n not representable in bf16:
        y_j = bf16(gelu(bf16(n_a)) * sum_k bf16(n_k)),   a = pi(sigma(j)).
    Keeping n in fp32, dropping the rounding of h, or rounding g and u instead of h all fail."""
    Hs, Is = 256, 128
    rng = np.random.default_rng(17)
    pi = rng.permutation(Hs)[:Is]
    sigma = rng.integers(0, Is, Hs)
    qg = np.zeros((Is, Hs), np.uint8)
    qg[np.arange(Is), pi] = 1
    qd = np.zeros((Hs, Is), np.uint8)
    qd[np.arange(Hs), sigma] = 1
    one, zero = _const_f16(1.0, (Is, Hs // 64)), _const_f16(0.0, (Is, Hs // 64))
    ex = {"gate": (qg, one, zero),
          "up": (np.zeros((Is, Hs), np.uint8), _const_f16(0.5, (Is, Hs // 64)), one),
          "down": (qd, _const_f16(1.0, (Hs, Is // 64)), _const_f16(0.0, (Hs, Is // 64)))}
    n = _spread_input(rng, Hs)
    y = O.expert_ffn(n, ex, fmt="bf16", bits=64)
    _assert_only_reading(y, _bf16_branch_variants(n, pi, sigma))
    # the fp32 reading of the same expert keeps every operand as it is
    assert np.allclose(O.expert_ffn(n, ex, fmt="fp32", bits=64),
                       [_gelu64(n[pi[sigma[j]]]) * n.sum() for j in range(Hs)], rtol=1e-12, atol=0)


def test_expert_ffn_bf16_scale_after_the_dot_products():
    """The bf16 reading of a layer feeds the raw bf16 input x and applies the RMS scale c = r to g and u after
    their dot products (before GELU): y_j = bf16(gelu(c bf16(v_a)) * c sum_k bf16(v_k)). A scale left out, or
    applied to h instead of g and u, fails."""
    Hs, Is = 256, 128
    rng = np.random.default_rng(21)
    pi = rng.permutation(Hs)[:Is]
    sigma = rng.integers(0, Is, Hs)
    qg = np.zeros((Is, Hs), np.uint8)
    qg[np.arange(Is), pi] = 1
    qd = (np.arange(Is)[None, :] == sigma[:, None]).astype(np.uint8)
    one, zero = _const_f16(1.0, (Is, Hs // 64)), _const_f16(0.0, (Is, Hs // 64))
    ex = {"gate": (qg, one, zero),
          "up": (np.zeros((Is, Hs), np.uint8), _const_f16(0.5, (Is, Hs // 64)), one),
          "down": (qd, _const_f16(1.0, (Hs, Is // 64)), _const_f16(0.0, (Hs, Is // 64)))}
    v = _spread_input(rng, Hs)
    c = 0.7317
    y = O.expert_ffn(v, ex, fmt="bf16", bits=64, in_scale=c)
    want = _bf16_branch_variants(v, pi, sigma, c=c)["bf16 n and h"]
    assert np.array_equal(y, want)
    assert not np.allclose(y, _bf16_branch_variants(v, pi, sigma)["bf16 n and h"], rtol=1e-6, atol=0)
    h_scaled = np.array([_rn_bf16(c * c * _gelu64(_rn_bf16(v[pi[sigma[j]]])) * np.sum([_rn_bf16(t) for t in v]))
                         for j in range(Hs)])
    assert not np.allclose(y, h_scaled, rtol=1e-6, atol=0)


def test_expert_ffn_fp16_operands_closed_form():
    """The fp16 reading of a routed expert (the tensor-core reading of the routed GEMMs): v, every dequantised
    weight and h rounded to fp16, the scale c after the dot products:
        y_j = fp16(gelu(c fp16(v_a)) * c sum_k fp16(v_k)).
    The bf16 rounding, or none, fails."""
    Hs, Is = 256, 128
    rng = np.random.default_rng(22)
    pi = rng.permutation(Hs)[:Is]
    sigma = rng.integers(0, Is, Hs)
    qg = np.zeros((Is, Hs), np.uint8)
    qg[np.arange(Is), pi] = 3
    qd = (np.arange(Is)[None, :] == sigma[:, None]).astype(np.uint8)
    s16 = np.float16(0.0131)
    w_g = np.float64(np.float32(s16)) * 3
    ex = {"gate": (qg, _const_f16(float(s16), (Is, Hs // 64)), _const_f16(0.0, (Is, Hs // 64))),
          "up": (np.zeros((Is, Hs), np.uint8), _const_f16(0.5, (Is, Hs // 64)), _const_f16(1.0, (Is, Hs // 64))),
          "down": (qd, _const_f16(1.0, (Hs, Is // 64)), _const_f16(0.0, (Hs, Is // 64)))}
    v = _spread_input(rng, Hs) * 37.0          # values fp16 does not hold exactly either
    c = 0.0613
    y = O.expert_ffn(v, ex, fmt="fp16", bits=64, in_scale=c)
    want = _bf16_branch_variants(v, pi, sigma, wg=_rn_f16(w_g), c=c, rnd=_rn_f16)
    assert np.array_equal(y, want["bf16 n and h"])
    for name in ("fp32 n", "no h rounding", "g, u rounded"):
        assert not np.allclose(y, want[name], rtol=1e-7, atol=0), name
    assert not np.allclose(y, _bf16_branch_variants(v, pi, sigma, wg=_rn_bf16(w_g), c=c)["bf16 n and h"],
                           rtol=1e-6, atol=0)


def test_layer_combine_tensor_core_reading_feeds_x_and_r():
    """layer_combine's tensor-core reading is the shared FFN (bf16 operands, input x, scale r after the gate/up
    dot products) and the routed FFNs (fp16 operands, input x p, scale r / p, p the power of two of r); its fp32
    reading feeds n = r x with scale 1."""
    Hs, Is, Ss, k = 192, 64, 128, 3
    x = W.hidden(6, 0, 1, Hs)[0]
    r = O.rms_scale(x, 64)
    xf = W.bf16_to_f32(x).astype(np.float64)
    experts = [W.expert(30 + i, 0, 0, Hs, Is) for i in range(k)]
    Wg, Wu, Wd = W.shared_weights(6, 0, Hs, Ss)
    w = np.array([0.5, 0.3, 0.2])
    _, delta = O.layer_combine(x, r, experts, w, (Wg, Wu, Wd), tc=True, bits=64)
    p = 2.0 ** math.floor(math.log2(r))
    assert 1.0 <= r / p < 2.0
    want = O.shared_ffn(xf, Wg, Wu, Wd, fmt="bf16", bits=64, in_scale=r)
    for i in range(k):
        want = want + w[i] * O.expert_ffn(xf * p, experts[i], fmt="fp16", fmt_down="bf16", bits=64, in_scale=r / p)
    assert np.array_equal(delta, want)
    alt = O.shared_ffn(xf, Wg, Wu, Wd, fmt="bf16", bits=64, in_scale=r)
    for i in range(k):   # fp16 for the down products too: a different reading, which the pin tells apart
        alt = alt + w[i] * O.expert_ffn(xf * p, experts[i], fmt="fp16", bits=64, in_scale=r / p)
    assert not np.array_equal(delta, alt)
    # the same layer with x scaled by 2^20: the fp16 operand x p is the same, the update scales with x
    xb = (W.bf16_to_f32(x) * np.float32(2.0 ** 20)).view(np.uint32) >> 16
    xb = xb.astype(np.uint16)
    r2 = O.rms_scale(xb, 64)
    _, d2 = O.layer_combine(xb, r2, experts, w, None, tc=True, bits=64)
    _, d1 = O.layer_combine(x, r, experts, w, None, tc=True, bits=64)
    assert np.all(np.isfinite(d2)) and np.allclose(d2, d1, rtol=1e-6, atol=0)
    n = O.normalise(x, r, 64)
    for fs, fe, xin, c in (("bf16", "fp16", n, 1.0), ("bf16", "bf16", xf, r), ("fp16", "fp16", xf, r)):
        wrong = O.shared_ffn(xin, Wg, Wu, Wd, fmt=fs, bits=64, in_scale=c)
        for i in range(k):
            wrong = wrong + w[i] * O.expert_ffn(xin, experts[i], fmt=fe, bits=64, in_scale=c)
        assert not np.array_equal(delta, wrong), (fs, fe)
    _, delta32 = O.layer_combine(x, r, experts, w, (Wg, Wu, Wd), tc=False, bits=64)
    want32 = O.shared_ffn(n, Wg, Wu, Wd, bits=64)
    for i in range(k):
        want32 = want32 + w[i] * O.expert_ffn(n, experts[i], bits=64)
    assert np.array_equal(delta32, want32)


def test_expert_ffn_bf16_rounds_the_dequantised_weights():
    """The gate weight s q (code 3, bias 0) is not a bf16 value. In the bf16 reading the gate row holds
    bf16(s q) at its permuted column, so g_j = bf16(s q) bf16(n_a); keeping the fp32 weight gives s q."""
    Hs, Is = 192, 64
    rng = np.random.default_rng(18)
    pi = rng.permutation(Hs)[:Is]
    sigma = rng.integers(0, Is, Hs)
    s16 = np.float16(0.0131)
    w_exact = np.float64(np.float32(s16)) * 3                  # s q is exact in fp32
    w_bf16 = _rn_bf16(w_exact)
    assert w_bf16 != w_exact
    qg = np.zeros((Is, Hs), np.uint8)
    qg[np.arange(Is), pi] = 3
    qd = (np.arange(Is)[None, :] == sigma[:, None]).astype(np.uint8)
    ex = {"gate": (qg, _const_f16(float(s16), (Is, Hs // 64)), _const_f16(0.0, (Is, Hs // 64))),
          "up": (np.zeros((Is, Hs), np.uint8), _const_f16(0.5, (Is, Hs // 64)), _const_f16(1.0, (Is, Hs // 64))),
          "down": (qd, _const_f16(1.0, (Hs, Is // 64)), _const_f16(0.0, (Hs, Is // 64)))}
    n = _spread_input(rng, Hs)
    y = O.expert_ffn(n, ex, fmt="bf16", bits=64)
    assert np.array_equal(y, _bf16_branch_variants(n, pi, sigma, wg=w_bf16)["bf16 n and h"])
    assert not np.allclose(y, _bf16_branch_variants(n, pi, sigma, wg=w_exact)["bf16 n and h"], rtol=1e-6, atol=0)


def test_shared_ffn_bf16_operands_closed_form():
    """The bf16 reading of the shared expert (weights already bf16): n and h rounded to bf16.
    Gate = permutation, up = all-twos rows, down = permutation:
        y_j = bf16(gelu(bf16(n_a)) * 2 sum_k bf16(n_k))."""
    Hs, Ss = 192, 96
    rng = np.random.default_rng(19)
    pi = rng.permutation(Hs)[:Ss]
    sigma = rng.integers(0, Ss, Hs)
    one = np.float32(1.0).view(np.uint32) >> 16
    two = np.float32(2.0).view(np.uint32) >> 16
    Wg = np.zeros((Ss, Hs), np.uint16)
    Wg[np.arange(Ss), pi] = one
    Wu = np.full((Ss, Hs), two, np.uint16)
    Wd = np.zeros((Hs, Ss), np.uint16)
    Wd[np.arange(Hs), sigma] = one
    n = _spread_input(rng, Hs)
    y = O.shared_ffn(n, Wg, Wu, Wd, fmt="bf16", bits=64)
    _assert_only_reading(y, _bf16_branch_variants(n, pi, sigma, wu=2.0))


def test_layer_combine_weighted_sum_closed_form():
    """delta = shared + sum_i w_i y_i with per-expert closed forms, out = bf16(x + delta)."""
    Hs, Is, Ss, k = 128, 64, 64, 3
    rng = np.random.default_rng(10)
    x = W.hidden(4, 0, 1, Hs)[0]
    r = O.rms_scale(x, 64)
    n = O.normalise(x, r, 64)
    experts, ys = [], []
    for i in range(k):
        ex = W.expert(20 + i, 0, 0, Hs, Is)
        experts.append(ex)
        ys.append(O.expert_ffn(n, ex, bits=64))
    Wg, Wu, Wd = W.shared_weights(4, 0, Hs, Ss)
    ysh = O.shared_ffn(n, Wg, Wu, Wd, bits=64)
    w = np.array([0.5, 0.3, 0.2])
    out, delta = O.layer_combine(x, r, experts, w, (Wg, Wu, Wd), bits=64)
    want = ysh + sum(w[i] * ys[i] for i in range(k))
    assert np.allclose(delta, want, rtol=1e-13, atol=1e-13)
    xf = W.bf16_to_f32(x).astype(np.float64)
    for j in range(Hs):
        assert out[j] == _nearest_bf16_bruteforce(np.float32(xf[j] + delta[j]))


def test_fp32_oracle_bounded_by_fp64_oracle_full_layer():
    """Whole layer at full shapes (H=2816, I=704, E=128, shared 2112): fp32 vs fp64 oracle."""
    S = 2112
    x = W.hidden(0, 0, 1, H)[0]
    Wr = W.router_weights(0, 0, E, H)
    r32, z32, idx, w32 = O.route(x, Wr, bits=32)
    r64, z64, idx64, w64 = O.route(x, Wr, bits=64)
    assert idx.tolist() == idx64.tolist()
    assert abs(r32 - r64) <= 2 * np.spacing(np.float32(r64))
    experts = W.experts_parallel(0, 0, idx, H, I)
    shared = W.shared_weights(0, 0, H, S)
    out32, d32 = O.layer_combine(x, r32, experts, w32, shared, bits=32)
    out64, d64 = O.layer_combine(x, r64, experts, w64, shared, bits=64)
    rel = np.max(np.abs(d32 - d64)) / np.max(np.abs(d64))
    assert rel < 1e-5
    # bf16 outputs agree except for rare rounding-boundary flips of one bf16 ulp
    diff = np.abs(W.bf16_to_f32(out32) - W.bf16_to_f32(out64))
    assert np.all(diff <= np.abs(W.bf16_to_f32(out64)) * 2.0 ** -7 + 1e-30)


def test_all_cores_build_is_bit_identical():
    """The OpenMP build only spreads independent rows over threads: its routing and layer output equal the
    single-threaded oracle's bit for bit (full shapes, with the shared expert)."""
    S = 2112
    x = W.hidden(2, 0, 1, H)[0]
    Wr = W.router_weights(2, 0, E, H)
    r1, z1, i1, w1 = O.route(x, Wr)
    r2, z2, i2, w2 = O.route(x, Wr, mt=True)
    assert np.float32(r1).view(np.uint32) == np.float32(r2).view(np.uint32)
    assert np.array_equal(z1.view(np.uint32), z2.view(np.uint32)) and np.array_equal(i1, i2)
    assert np.array_equal(w1.view(np.uint32), w2.view(np.uint32))
    experts = W.experts_parallel(2, 0, i1, H, I)
    shared = W.shared_weights(2, 0, H, S)
    o1, d1 = O.layer_combine(x, r1, experts, w1, shared)
    o2, d2 = O.layer_combine(x, r1, experts, w1, shared, mt=True)
    assert np.array_equal(o1, o2) and np.array_equal(d1.view(np.uint32), d2.view(np.uint32))
    assert O.threads(False) == 1 and O.threads(True) >= 1


def test_oracle_precisions():
    assert O.lib(32).or_real_bytes() == 4
    assert O.lib(64).or_real_bytes() == 8


# ------------------------------------------------------------------------------ LFU

@pytest.mark.parametrize("name", lfu_trace_names())
def test_lfu_golden_traces(name):
    slots, layers, inputs, events = load_lfu_trace(name)
    lfu = O.LFU(layers, slots)
    got = []
    for step, layer, ids in inputs:
        got += lfu.step(step, layer, np.array(ids, np.int32))
    assert got == events


def test_lfu_invariants_random_long_run():
    rng = np.random.default_rng(11)
    Ls, S, En, k = 3, 16, 128, 8
    lfu = O.LFU(Ls, S)
    cold = [0] * Ls
    for step in range(300):
        for layer in range(Ls):
            hot = rng.choice(24, 5, replace=False)
            ids = np.unique(np.concatenate([hot, rng.choice(En, 8, replace=False)]))[:k]
            rng.shuffle(ids)
            before_ex, before_cnt, before_lu = lfu.state(layer)
            ev = lfu.step(step, layer, ids.astype(np.int32))
            ex, cnt, lu = lfu.state(layer)
            hits = sum(e[3] for e in ev)
            misses = len(ev) - hits
            assert hits + misses == len(ids)
            assert set(ids.tolist()) <= set(ex.tolist()) and (ex >= 0).sum() <= S
            evictions = sum(1 for e in ev if e[5] >= 0)
            cold_fills = sum(1 for e in ev if e[3] == 0 and e[5] < 0)
            cold[layer] += cold_fills
            assert evictions == misses - cold_fills
            for e in ev:
                assert e[5] not in ids.tolist()
                if e[3]:
                    assert before_ex[e[4]] == e[2]
                elif e[5] >= 0:
                    # the victim had the minimum count among the slots it could have taken
                    cand = [s for s in range(S) if before_ex[s] not in ids.tolist()]
                    assert before_cnt[e[4]] == min(before_cnt[s] for s in cand) or e[4] in [
                        x[4] for x in ev if x[3] == 0]
    assert all(c <= S for c in cold)
