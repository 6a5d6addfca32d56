"""The oracle's Llama-style decoder (test infrastructure).

What the target model computes is the plain definition of a Llama-2 decoder,
the model all three pages build on (SWIFT digest §2 and §5.1; LayerSkip blog
§3.1-3.2, where ``model.layers[l]`` and the shared ``model.lm_head`` are the
two building blocks of drafting and verification):

    x   = E[token]
    per layer l:
      h   = rmsnorm(x) * g_attn                (bf16-rounded)
      q,k,v = Wqkv h;  q,k = rope(q,k, pos)     (k, v stored bf16-rounded)
      a   = softmax(q K^T / sqrt(dh), causal) V (bf16-rounded)
      x  += Wo a
      h2  = rmsnorm(x) * g_mlp                 (bf16-rounded)
      u   = silu(Wg h2) * (Wu h2)              (bf16-rounded)
      x  += Wd u
    z   = Wlm (rmsnorm(x) * g_final)           (normed input bf16-rounded)

RoPE is the rotate-half form: dimensions i and i + dh/2 form a pair rotated
by pos * theta**(-2i/dh).  Attention heads share K/V heads in groups of
H / Hkv (grouped-query attention; H == Hkv is plain multi-head).

Every row is computed on its own, one matrix-vector product at a time, so a
row's result never depends on how many rows are processed together.  That is
what makes the oracle's own self-speculative output bit-identical to its
autoregressive output.  In "fp32" mode (the tiny fp32 workload) nothing is
rounded; all arithmetic is fp64 in both modes.
"""

from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

from .numerics import bf16_round, widen


class KVCache:
    """Per-layer K and V, [L][Hkv, max_seq, dh] fp64 (holding bf16 values in bf16 mode)."""

    def __init__(self, n_layers: int, n_kv_heads: int, max_seq: int, head_dim: int):
        self.K = [np.zeros((n_kv_heads, max_seq, head_dim)) for _ in range(n_layers)]
        self.V = [np.zeros((n_kv_heads, max_seq, head_dim)) for _ in range(n_layers)]
        self.max_seq = max_seq

    def fork(self) -> "KVCache":
        c = KVCache.__new__(KVCache)
        c.K = [k.copy() for k in self.K]
        c.V = [v.copy() for v in self.V]
        c.max_seq = self.max_seq
        return c


class OracleModel:
    def __init__(self, shape, weights: Dict, cache_limit_bytes: int = 2 << 30):
        self.s = shape
        self.w = weights
        self.bf16 = weights["dtype"] == "bf16"
        self._cache: Dict = {}
        self._cache_bytes = 0
        self._limit = cache_limit_bytes
        dh = shape.head_dim
        i = np.arange(dh // 2, dtype=np.float64)
        self.inv_freq = shape.rope_theta ** (-2.0 * i / dh)

    # ---- weights -------------------------------------------------------
    def mat(self, layer: Optional[int], name: str) -> np.ndarray:
        key = (layer, name)
        if key in self._cache:
            return self._cache[key]
        src = self.w[name] if layer is None else self.w["layers"][layer][name]
        m = widen(src)
        if self._cache_bytes + m.nbytes <= self._limit:
            self._cache[key] = m
            self._cache_bytes += m.nbytes
        return m

    def rnd(self, x: np.ndarray) -> np.ndarray:
        return bf16_round(x) if self.bf16 else x

    # ---- building blocks ------------------------------------------------
    def rmsnorm(self, x: np.ndarray, g: np.ndarray) -> np.ndarray:
        return x * (1.0 / np.sqrt(np.mean(x * x) + self.s.norm_eps)) * g

    def rope(self, v: np.ndarray, pos: int) -> np.ndarray:
        """v: [heads, dh]; rotate pairs (i, i + dh/2) by pos * inv_freq[i]."""
        half = self.s.head_dim // 2
        ang = pos * self.inv_freq
        c, s = np.cos(ang), np.sin(ang)
        a, b = v[:, :half], v[:, half:]
        return np.concatenate([a * c - b * s, a * s + b * c], axis=1)

    def embed(self, tok: int) -> np.ndarray:
        return widen(self.w["tok_embed"][int(tok)])

    def attention_row(self, q: np.ndarray, kv: KVCache, layer: int, pos: int) -> np.ndarray:
        """q: [H, dh] (after RoPE).  Keys/values at positions 0..pos of ``layer``."""
        s = self.s
        group = s.n_heads // s.n_kv_heads
        out = np.empty((s.n_heads, s.head_dim))
        scale = 1.0 / np.sqrt(s.head_dim)
        for h in range(s.n_heads):
            kvh = h // group
            K = kv.K[layer][kvh, : pos + 1]
            V = kv.V[layer][kvh, : pos + 1]
            sc = (K @ q[h]) * scale
            m = np.max(sc)
            e = np.exp(sc - m)
            out[h] = (e @ V) / np.sum(e)
        return out.reshape(-1)

    def layer(self, l: int, X: np.ndarray, positions: Sequence[int], kv: KVCache,
              attn: bool = True, mlp: bool = True) -> np.ndarray:
        """Run rows X ([M, D], consecutive positions) through layer l; writes K/V.
        ``attn`` / ``mlp`` False leave that sublayer's residual branch out (an
        attention sublayer that does not run writes no K/V)."""
        X = X.copy()
        if attn:
            X = self._attention_sublayer(l, X, positions, kv)
        if mlp:
            X = self._mlp_sublayer(l, X)
        return X

    def _attention_sublayer(self, l: int, X: np.ndarray, positions: Sequence[int],
                            kv: KVCache) -> np.ndarray:
        s = self.s
        H, Hkv, dh = s.n_heads, s.n_kv_heads, s.head_dim
        g1 = self.mat(l, "attn_norm")
        Wqkv = self.mat(l, "wqkv")
        qs = []
        for m, pos in enumerate(positions):
            h = self.rnd(self.rmsnorm(X[m], g1))
            qkv = Wqkv @ h
            q = self.rope(qkv[: H * dh].reshape(H, dh), pos)
            k = self.rope(qkv[H * dh:(H + Hkv) * dh].reshape(Hkv, dh), pos)
            v = qkv[(H + Hkv) * dh:].reshape(Hkv, dh)
            kv.K[l][:, pos] = self.rnd(k)
            kv.V[l][:, pos] = self.rnd(v)
            qs.append(q)
        Wo = self.mat(l, "wo")
        for m, pos in enumerate(positions):
            a = self.rnd(self.attention_row(qs[m], kv, l, pos))
            X[m] = X[m] + Wo @ a
        return X

    def _mlp_sublayer(self, l: int, X: np.ndarray) -> np.ndarray:
        g2 = self.mat(l, "mlp_norm")
        Wg, Wu, Wd = self.mat(l, "w_gate"), self.mat(l, "w_up"), self.mat(l, "w_down")
        for m in range(X.shape[0]):
            h2 = self.rnd(self.rmsnorm(X[m], g2))
            gate = Wg @ h2
            up = Wu @ h2
            u = self.rnd(gate / (1.0 + np.exp(-gate)) * up)
            X[m] = X[m] + Wd @ u
        return X

    def lm_head(self, X: np.ndarray) -> np.ndarray:
        """Final RMSNorm + LM head; returns logits [M, V] (fp64)."""
        g = self.mat(None, "final_norm")
        W = self.mat(None, "lm_head")
        return np.stack([W @ self.rnd(self.rmsnorm(x, g)) for x in X])

    def run_layers(self, X: np.ndarray, positions: Sequence[int], kv: KVCache,
                   layers: Sequence[int], parts=None) -> np.ndarray:
        """``parts`` (optional): layer -> (attention runs, MLP runs)."""
        for l in layers:
            a, m = parts(l) if parts is not None else (True, True)
            X = self.layer(l, X, positions, kv, attn=a, mlp=m)
        return X

    def new_cache(self, max_seq: int) -> KVCache:
        s = self.s
        return KVCache(s.n_layers, s.n_kv_heads, max_seq, s.head_dim)

    def embed_rows(self, toks: Sequence[int]) -> np.ndarray:
        return np.stack([self.embed(t) for t in toks])


def softmax(z: np.ndarray) -> np.ndarray:
    m = np.max(z)
    e = np.exp(z - m)
    return e / np.sum(e)


def logsumexp(z: np.ndarray) -> float:
    m = np.max(z)
    return float(m + np.log(np.sum(np.exp(z - m))))


def top2(z: np.ndarray) -> List:
    """(top1 id, top1 value, top2 id, top2 value); lowest id wins ties."""
    i1 = int(np.argmax(z))
    z2 = z.copy()
    z2[i1] = -np.inf
    i2 = int(np.argmax(z2))
    return [i1, float(z[i1]), i2, float(z[i2])]
