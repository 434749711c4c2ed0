"""Round-to-nearest-even to bfloat16, emulated on float64 / float32 arrays.

bfloat16 keeps float32's 8-bit exponent and 7 stored mantissa bits.  The pages
run the trunk in bf16 with branches computed at higher precision and rounded
back ("Llama 3.1 70B", Residual add: the add happens in the trunk dtype; RMSNorm
reference implementation: ``type_as`` after the fp32 scale).  The oracle applies
this rounding at exactly the points the block defines, directly from the
float64 value (a single rounding, no detour through float32).

Pinned in tests against torch's float32 -> bfloat16 conversion (a library
routine), including ties, subnormals and overflow.
"""
from __future__ import annotations

import numpy as np

BF16_MAX = float.fromhex("0x1.fe00000000000p+127")   # largest finite bf16
_MIN_NORMAL = 2.0 ** -126
_SUB_STEP = 2.0 ** -133                               # bf16 subnormal spacing


def round_bf16(a):
    """Return ``a`` rounded to the nearest bfloat16 (ties to even), same dtype as input
    (float64 or float32).  NaN stays NaN, +-inf stays, overflow goes to +-inf."""
    a = np.asarray(a)
    if a.dtype == np.float64:
        shift, ubits = 45, np.uint64          # 52 mantissa bits -> keep 7
    elif a.dtype == np.float32:
        shift, ubits = 16, np.uint32          # 23 mantissa bits -> keep 7
    else:
        raise TypeError(f"round_bf16 expects float64/float32, got {a.dtype}")
    src = np.ascontiguousarray(a)
    bits = src.view(ubits).copy()
    lsb = (bits >> ubits(shift)) & ubits(1)
    bits += ubits((1 << (shift - 1)) - 1) + lsb
    bits &= ~ubits((1 << shift) - 1)
    out = bits.view(src.dtype)
    with np.errstate(invalid="ignore", over="ignore"):
        mag = np.abs(src)
        # values below the bf16 normal range round on the fixed subnormal grid
        tiny = mag < _MIN_NORMAL
        if np.any(tiny):
            out = np.where(tiny, np.round(src / _SUB_STEP) * _SUB_STEP, out).astype(src.dtype)
        # anything that rounds above the largest finite bf16 overflows
        big = np.abs(out) > BF16_MAX
        if np.any(big):
            out = np.where(big, np.copysign(np.inf, src), out).astype(src.dtype)
        out = np.where(np.isfinite(src), out, src)
    return out.reshape(a.shape)


def identity(a):
    """No rounding: the fp32 workload keeps every intermediate unrounded."""
    return a
