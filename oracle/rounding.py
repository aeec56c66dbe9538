"""Round float64 values to fp16 / bf16 (round to nearest, ties to even).

TEST INFRASTRUCTURE ONLY (see the package docstring).

fp16 uses numpy's float64 -> float16 cast, which rounds once, directly from
double, to nearest-even.  bf16 has no numpy dtype, so `round_bf16` rounds by
the definition of a binary floating-point format with 8 significant bits and
the float32 exponent range: the quantum of a value v is 2**(floor(log2|v|) - 7)
for normal results and 2**-133 below 2**-126; the value is divided by its
quantum, rounded to an integer with ties to even (numpy.rint), and scaled back;
magnitudes that round above the largest finite bf16 become infinities.
"""
from __future__ import annotations

import numpy as np

_BF16_MAX = float.fromhex("0x1.fep127")      # (2 - 2**-7) * 2**127
_BF16_EMIN = -126                             # smallest normal exponent
_BF16_P = 8                                   # significant bits


def round_fp16(v: np.ndarray) -> np.ndarray:
    """float64 array of the fp16-nearest values (ties to even); magnitudes past
    the fp16 range become infinities, as IEEE rounding gives."""
    with np.errstate(over="ignore"):
        return np.asarray(v, dtype=np.float64).astype(np.float16).astype(np.float64)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """float64 array of the bf16-nearest values (ties to even)."""
    v = np.asarray(v, dtype=np.float64)
    out = np.array(v, copy=True)
    finite = np.isfinite(v) & (v != 0.0)
    a = v[finite]
    # frexp: a = m * 2**e with 0.5 <= |m| < 1, so floor(log2|a|) = e - 1.
    _, e = np.frexp(a)
    expo = np.maximum(e - 1, _BF16_EMIN)
    q = np.ldexp(1.0, expo - (_BF16_P - 1))
    r = np.rint(a / q) * q
    r = np.where(np.abs(r) > _BF16_MAX, np.copysign(np.inf, r), r)
    out[finite] = r
    return out


def round_to(v: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "fp16":
        return round_fp16(v)
    if dtype == "bf16":
        return round_bf16(v)
    raise ValueError(f"unknown output dtype {dtype!r}")
