"""Error metrics used by the parity tests.

Contract (the layer outputs): the max relative error of a vector against the
oracle, read as max_i |a_i - r_i| / max_i |r_i| (per token), must be <= 1e-2.
It is checked on the bf16 layer output and on the fp32 update delta = out - x
(before rounding), since after the first layers the residual dominates out.

Outputs are bf16 by the layer's format. Where a bf16 output is compared with
the plain fp32 oracle across different arithmetic (the bf16 tensor-core path),
it is compared with the oracle's exact x + delta, allowing the output's own
rounding to bf16 (out_rel_err); where no fp32 update is exposed, out - x is
compared with the oracle's delta allowing 1.5 ulp of out (delta_rel_err).

The fp32 decode path is also held to a much tighter elementwise bound,
max_i |a_i - r_i| / max(|r_i|, 1e-3 * rms(r)), which catches a wrong term that
the normwise bound would hide.
"""
import numpy as np

CONTRACT_TOL = 1e-2


def max_rel_err(a, r) -> float:
    a = np.asarray(a, np.float64)
    r = np.asarray(r, np.float64)
    return float(np.max(np.abs(a - r)) / max(np.max(np.abs(r)), 1e-30))


def elem_rel_err(a, r, floor: float = 1e-3) -> float:
    a = np.asarray(a, np.float64)
    r = np.asarray(r, np.float64)
    rms = np.sqrt(np.mean(r * r))
    den = np.maximum(np.abs(r), floor * rms)
    return float(np.max(np.abs(a - r) / den))


def bf16_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (v as float64)."""
    v = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def delta_rel_err(out_bits, x_bits, delta_ref) -> float:
    """Error of the layer update recovered from a bf16 output, out - x, against the
    reference fp32 update, after allowing the output's own rounding: out is the
    bf16 of x + delta, so out - x can differ from delta by half an ulp of out, and
    a rounding-boundary flip adds one more ulp (1.5 ulp of out in all)."""
    o = bf16_to_f64(out_bits)
    x = bf16_to_f64(x_bits)
    d = np.asarray(delta_ref, np.float64)
    excess = np.maximum(np.abs((o - x) - d) - 1.5 * bf16_ulp(o), 0.0)
    return float(np.max(excess) / max(np.max(np.abs(d)), 1e-30))


def out_rel_err(out_bits, x_bits, delta_ref) -> float:
    """Error of a bf16 layer output against the reference's exact output x + delta (before any rounding to
    bf16), after allowing the output's own rounding to bf16 (half an ulp of out). Comparing two independently
    rounded bf16 outputs instead would charge up to two ulps of quantisation (up to 1.6 % relative) to the
    arithmetic being checked."""
    o = bf16_to_f64(out_bits)
    ref = bf16_to_f64(x_bits) + np.asarray(delta_ref, np.float64)
    excess = np.maximum(np.abs(o - ref) - 0.5 * bf16_ulp(o), 0.0)
    return float(np.max(excess) / max(np.max(np.abs(ref)), 1e-30))

