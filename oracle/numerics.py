"""Rounding and widening helpers of the oracle (test infrastructure).

The numeric contract the oracle follows (the pages fix no precision beyond
SWIFT's FP16 experiments, so this is the plainest reading for a bf16 model):
weights are bf16; every GEMM input (the RMS-normalised hidden state, the
attention output, the SwiGLU product) and every stored K/V value is rounded
to bf16; everything else is kept at full precision (fp64 here).
"""

from __future__ import annotations

import numpy as np


def bf16_round(x):
    """Round to the nearest bfloat16 value (8 significant bits), ties to even.

    Written from the definition: write x = m * 2**e with 0.5 <= |m| < 1, keep
    8 significant bits of m with round-half-even, clamp the quantum at the
    bfloat16 subnormal spacing 2**-133.  Returns fp64 values.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    q = np.maximum(e - 8, -133)          # exponent of one unit in the last place
    r = np.rint(np.ldexp(m, e - q))      # numpy rint rounds half to even
    out = np.ldexp(r, q)
    big = np.abs(out) > 3.3895313892515355e38   # largest finite bfloat16
    if np.any(big):
        out = np.where(big, np.copysign(np.inf, x), out)
    return out


def widen(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) or fp32 values -> fp64."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)
