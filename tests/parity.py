"""Error metrics used by the parity tests.

Contract (the layer outputs): the max relative error of a vector against the
oracle, read as max_i |a_i - r_i| / max_i |r_i| (per token), must be <= 1e-2.
It is checked on the bf16 layer output and on the fp32 update delta = out - x
(before rounding), since after the first layers the residual dominates out.

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
