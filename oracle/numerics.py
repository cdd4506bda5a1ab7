"""IEEE-754 storage rounding and bit decoding, written from the format definitions.

TEST INFRASTRUCTURE. This package is the fp64 CPU oracle of the PowerSGD step. Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline`` / reference
leg may import or execute it. The CUDA library never calls into it and shares no code
with it.

Formats (binary16, bfloat16, binary32) are described by their significand precision p
(hidden bit included), the minimum normal exponent emin and the maximum exponent emax.
The bit widths are the ones "AIGC 基本功|混合精度与数值稳定性", §3.1 states: FP16 is
1/5/10 (sign/exponent/fraction), BF16 1/8/7, FP32 1/8/23.
"""
from __future__ import annotations

import numpy as np

# name -> (p, emin, emax, exponent bits, fraction bits)
FORMATS = {
    "f16": (11, -14, 15, 5, 10),
    "bf16": (8, -126, 127, 8, 7),
    "f32": (24, -126, 127, 8, 23),
    "f64": (53, -1022, 1023, 11, 52),
}


def max_finite(fmt: str) -> float:
    p, _, emax, _, _ = FORMATS[fmt]
    return (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax


def min_normal(fmt: str) -> float:
    return 2.0 ** FORMATS[fmt][1]


def min_subnormal(fmt: str) -> float:
    p, emin, _, _, _ = FORMATS[fmt]
    return 2.0 ** (emin - (p - 1))


def round_to_format(x, fmt: str) -> np.ndarray:
    """Round fp64 values to the nearest value of ``fmt``, ties to even (IEEE-754 RNE).

    The result is returned as fp64 holding exactly representable values of ``fmt``.
    Let e = floor(log2 |x|), clamped below at emin so that subnormals share the
    quantum of the smallest binade. The quantum is then 2^(e - p + 1), and x is
    rounded to an integer multiple of it with ties to even. A rounded magnitude above
    the largest finite value becomes an infinity of x's sign. NaN and +-Inf pass
    through. This is the rounding that "AIGC 基本功|混合精度与数值稳定性", §04 applies
    when it writes values back to FP16/BF16.
    """
    if fmt == "f64":
        return np.array(x, dtype=np.float64, copy=True)
    x = np.asarray(x, dtype=np.float64)
    shape = x.shape
    x = x.reshape(-1)
    p, emin, _, _, _ = FORMATS[fmt]
    with np.errstate(invalid="ignore", over="ignore"):
        _, ex = np.frexp(x)  # x = f * 2**ex with 0.5 <= |f| < 1 (ex = 0 for 0, inf, nan)
        np.subtract(ex, p, out=ex)  # quantum exponent e - (p - 1) with e = ex - 1
        np.maximum(ex, emin - (p - 1), out=ex)  # subnormals share the smallest binade
        q = np.ldexp(1.0, ex)
        y = np.divide(x, q)  # exact: q is a power of two
        np.rint(y, out=y)  # ties to even
        np.multiply(y, q, out=y)
        big = np.abs(y) > max_finite(fmt)
        y[big] = np.copysign(np.inf, x[big])
        nf = ~np.isfinite(x)
        y[nf] = x[nf]
    return y.reshape(shape)


def decode_bits(bits, fmt: str) -> np.ndarray:
    """Value of each bit pattern of ``fmt`` (uint array), from sign, exponent and fraction.

    Normal: (-1)^s * (1 + f / 2^F) * 2^(E - bias). Subnormal (E = 0):
    (-1)^s * (f / 2^F) * 2^(1 - bias). E all ones: Inf when f = 0, NaN otherwise.
    """
    p, emin, emax, ebits, fbits = FORMATS[fmt]
    bits = np.asarray(bits, dtype=np.uint64)
    sign = (bits >> np.uint64(ebits + fbits)) & np.uint64(1)
    expf = ((bits >> np.uint64(fbits)) & np.uint64((1 << ebits) - 1)).astype(np.int64)
    frac = (bits & np.uint64((1 << fbits) - 1)).astype(np.float64)
    bias = emax
    val = np.where(
        expf == 0,
        frac / 2.0 ** fbits * 2.0 ** (1 - bias),
        (1.0 + frac / 2.0 ** fbits) * np.exp2((expf - bias).astype(np.float64)),
    )
    top = expf == (1 << ebits) - 1
    val = np.where(top & (frac == 0), np.inf, val)
    val = np.where(top & (frac != 0), np.nan, val)
    return np.where(sign == 1, -val, val)


def is_representable(x, fmt: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    r = round_to_format(x, fmt)
    return (r == x) | (np.isnan(x) & np.isnan(r))
