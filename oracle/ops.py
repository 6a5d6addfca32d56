"""Per-kernel references for the parity tests (test infrastructure).

Each function restates one step of the decoder forward (oracle.model) or of
the acceptance rule (oracle.speculative) on explicit inputs, so that one
CUDA kernel can be compared with it in isolation.  All arithmetic is fp64;
the bf16 rounding points follow the numeric contract of oracle.numerics.
"""

from __future__ import annotations

from types import SimpleNamespace
from typing import List

import numpy as np

from .model import OracleModel, KVCache, logsumexp, softmax, top2
from .numerics import bf16_round, widen
from .philox import gumbel_argmax, uniform
from .speculative import accept_stochastic as _accept


def linear(W_bits: np.ndarray, act: np.ndarray) -> np.ndarray:
    """y[m] = W act[m] (W as bf16 bits, act as values)."""
    W = widen(W_bits)
    return np.stack([W @ a for a in act])


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    return x * (1.0 / np.sqrt(np.mean(x * x) + eps)) * g


def rmsnorm_linear(W_bits, x, g, eps) -> np.ndarray:
    W = widen(W_bits)
    return np.stack([W @ bf16_round(rmsnorm(r, g, eps)) for r in x])


def swiglu(Wg_bits, Wu_bits, x, g, eps) -> np.ndarray:
    Wg, Wu = widen(Wg_bits), widen(Wu_bits)
    out = []
    for r in x:
        h = bf16_round(rmsnorm(r, g, eps))
        gate, up = Wg @ h, Wu @ h
        out.append(bf16_round(gate / (1.0 + np.exp(-gate)) * up))
    return np.stack(out)


def silu_product(Wg_bits, Wu_bits, act) -> np.ndarray:
    """u[m] = bf16(silu(Wg act[m]) * (Wu act[m])): the SwiGLU activation of
    already-normalised bf16 rows."""
    Wg, Wu = widen(Wg_bits), widen(Wu_bits)
    out = []
    for a in act:
        gate, up = Wg @ a, Wu @ a
        out.append(bf16_round(gate / (1.0 + np.exp(-gate)) * up))
    return np.stack(out)


def score_attention(q: np.ndarray, cand, N: int, split: int, K: np.ndarray, V: np.ndarray,
                    WK: np.ndarray, WV: np.ndarray, H: int, Hkv: int) -> np.ndarray:
    """Attention of candidate-mask scoring windows (SWIFT §4.1.2 parallel
    prediction): query row (candidate cand[j], window row i) sits at position
    split + i and sees the shared cache's keys 0..split-1 (K, V: [Hkv,
    max_seq, dh]) followed by its own candidate's window keys 0..i (WK, WV:
    [rows, Hkv, dh], row k N + w).  q: [len(cand) N, H, dh] after RoPE.
    Returns bf16-rounded outputs [len(cand) N, H dh]."""
    dh = q.shape[2]
    group = H // Hkv
    out = np.zeros((len(cand) * N, H * dh))
    for j, k in enumerate(cand):
        for i in range(N):
            t = j * N + i
            for h in range(H):
                kvh = h // group
                keys = np.concatenate([K[kvh, :split], WK[k * N: k * N + i + 1, kvh]])
                vals = np.concatenate([V[kvh, :split], WV[k * N: k * N + i + 1, kvh]])
                sc = keys @ q[t, h] / np.sqrt(dh)
                e = np.exp(sc - np.max(sc))
                out[t, h * dh:(h + 1) * dh] = (e @ vals) / np.sum(e)
    return bf16_round(out)


def _shape(H, Hkv, dh, theta):
    return SimpleNamespace(n_heads=H, n_kv_heads=Hkv, head_dim=dh, rope_theta=theta,
                           norm_eps=1e-5)


def attention(qkv: np.ndarray, pos0: int, K: np.ndarray, V: np.ndarray, H: int, Hkv: int,
              dh: int, theta: float):
    """RoPE + bf16 K/V append + causal attention for rows at pos0..pos0+M-1.

    K, V: [Hkv, max_seq, dh] (values; updated copies are returned).
    Returns (out [M, H dh] bf16-rounded, K, V).
    """
    m = OracleModel.__new__(OracleModel)
    m.s = _shape(H, Hkv, dh, theta)
    i = np.arange(dh // 2, dtype=np.float64)
    m.inv_freq = theta ** (-2.0 * i / dh)
    kv = KVCache.__new__(KVCache)
    kv.K, kv.V = [K.copy()], [V.copy()]
    qs = []
    for r, row in enumerate(qkv):
        pos = pos0 + r
        q = m.rope(row[: H * dh].reshape(H, dh), pos)
        k = m.rope(row[H * dh:(H + Hkv) * dh].reshape(Hkv, dh), pos)
        v = row[(H + Hkv) * dh:].reshape(Hkv, dh)
        kv.K[0][:, pos] = bf16_round(k)
        kv.V[0][:, pos] = bf16_round(v)
        qs.append(q)
    out = np.stack([bf16_round(m.attention_row(q, kv, 0, pos0 + r)) for r, q in enumerate(qs)])
    return out, kv.K[0], kv.V[0]


def row_summary(z: np.ndarray, T: float = 0.0, seed: int = 0, pos: int = 0, rnd: int = 0,
                stream: int = 0) -> dict:
    """The LM-head row summary of logits z: top-2, lse, confidence, sample."""
    t = top2(z)
    lse = logsumexp(z)
    out = {"top1": t[0], "z1": t[1], "top2": t[2], "z2": t[3], "lse": lse,
           "conf": float(np.exp(t[1] - lse)), "gap": t[1] - t[3]}
    if T > 0.0:
        out["lse_t"] = logsumexp(z / T)
        out["sample"] = gumbel_argmax(z / T, seed, pos, rnd, stream)
    return out


def lm_head(W_bits, x, g, eps) -> np.ndarray:
    return rmsnorm_linear(W_bits, x, g, eps)


def accept_stochastic(P: np.ndarray, Q: np.ndarray, drafts: List[int], T: float, seed: int,
                      rnd: int, n: int):
    """The min(1, p/q) rule with the library's counter layout."""
    return _accept(P, list(Q), list(drafts), T,
                   draw_u=lambda j: uniform(seed, n + j, rnd, 1),
                   draw_tok=lambda j, logw: gumbel_argmax(logw, seed, n + j, rnd, 2))


def accept_margins(P: np.ndarray, Q: np.ndarray, drafts: List[int], T: float, seed: int,
                   rnd: int, n: int) -> List[float]:
    """|log u_j - log(p_j(y_j)/q_j(y_j))| for each draft (distance to the decision boundary)."""
    out = []
    for j, y in enumerate(drafts):
        p = softmax(P[j] / T)
        q = softmax(Q[j] / T)
        u = uniform(seed, n + j, rnd, 1)
        out.append(abs(np.log(u) - np.log(p[y] / q[y])))
    return out


def resample_gap(P: np.ndarray, Q: np.ndarray, a: int, T: float, seed: int, rnd: int,
                 n: int) -> float:
    """Gap between the two best Gumbel-perturbed scores of the token sampled
    after the accepted prefix (residual at a < d, bonus at a == d)."""
    from .philox import uniforms
    d = Q.shape[0]
    if a < d:
        p, q = softmax(P[a] / T), softmax(Q[a] / T)
        w = np.maximum(p - q, 0.0)
        with np.errstate(divide="ignore"):
            logw = np.log(w) if np.any(w > 0) else np.log(p)
    else:
        logw = P[d] / T
    g = -np.log(-np.log(uniforms(seed, n + a, rnd, 2, P.shape[1])))
    s = np.sort(logw + g)
    return float(s[-1] - s[-2])
