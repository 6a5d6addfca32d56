"""Philox4x32-10 and the samplers built on it (test infrastructure).

Philox4x32-10 is the counter-based generator of Salmon, Moraes, Dror and
Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): ten rounds of
two 32x32->64-bit multiplies (multipliers 0xD2511F53 and 0xCD9E8D57) on a
128-bit counter, with a 64-bit key bumped by the Weyl constants 0x9E3779B9
and 0xBB67AE85 between rounds.

The pages draw random numbers with an unspecified random() / sample()
(LayerSkip blog §3.3).  The reading taken here: every draw is a function of
(seed, absolute token position, decoding round, stream), with counter words
(c0 = vocab block v // 4, c1 = position, c2 = round, c3 = stream) and key
(seed low 32 bits, seed high 32 bits).  Streams: 0 = draft sample,
1 = acceptance uniform, 2 = residual / bonus sample.  A uniform is
u = ((r >> 9) + 0.5) * 2**-23, which is exact in fp32 and lies in (0, 1).
Sampling from weights w is Gumbel-max: argmax_v (log w_v - log(-log u_v)),
lowest index on ties.
"""

from __future__ import annotations

import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)

STREAM_DRAFT = 0
STREAM_ACCEPT = 1
STREAM_RESAMPLE = 2


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds.  ``ctr``: 4 uint32 arrays (broadcastable);
    ``key``: (k0, k1).  Returns 4 uint64 arrays holding 32-bit words."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _MASK32 for c in ctr)
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    for _ in range(10):
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1,
                          hi0 ^ c3 ^ np.uint64(k1), lo0)
        k0 = (k0 + _W0) & 0xFFFFFFFF
        k1 = (k1 + _W1) & 0xFFFFFFFF
    return c0, c1, c2, c3


def _key(seed: int):
    return (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)


def uniforms_table(seed: int, pos, rnd, stream: int, n: int) -> np.ndarray:
    """u_v for v = 0..n-1 at every (position, round) of the broadcast arrays
    ``pos`` and ``rnd``: shape [*broadcast shape, n] (fp64 holding values
    exact in fp32).  Word w of vocabulary block b is u_{4b + w}."""
    pos, rnd = np.broadcast_arrays(np.asarray(pos, dtype=np.uint64),
                                   np.asarray(rnd, dtype=np.uint64))
    blocks = np.arange((n + 3) // 4, dtype=np.uint64)
    words = philox4x32_10((blocks, pos[..., None], rnd[..., None], stream), _key(seed))
    r = np.stack(words, axis=-1).reshape(*pos.shape, -1)[..., :n]
    return ((r >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def uniforms(seed: int, pos: int, rnd: int, stream: int, n: int) -> np.ndarray:
    """u_v for v = 0..n-1 (fp64 holding values exact in fp32)."""
    return uniforms_table(seed, pos, rnd, stream, n)


def uniform(seed: int, pos: int, rnd: int, stream: int) -> float:
    return float(uniforms(seed, pos, rnd, stream, 1)[0])


def gumbel_argmax_u(logw: np.ndarray, u: np.ndarray) -> int:
    """Gumbel-max with given uniforms: argmax_v (logw_v - log(-log u_v)),
    lowest index on ties."""
    return int(np.argmax(logw - np.log(-np.log(u))))


def gumbel_argmax(logw: np.ndarray, seed: int, pos: int, rnd: int, stream: int) -> int:
    """Sample v with probability proportional to exp(logw_v) by Gumbel-max."""
    return gumbel_argmax_u(logw, uniforms(seed, pos, rnd, stream, logw.shape[0]))
