"""Lossy early-exit decoding and per-layer exit features (test infrastructure).

LayerSkip blog §3 (inference, mode one): the model can also simply stop at
an early layer and read the next token from the shared LM head there; that
is faster but not lossless, since nothing verifies the token.  Here the
"early" model is the draft layer set of the policy: layers 0..E in exit
mode, the layers outside the skip set (and their kept sublayers) in skip
mode.  Each step feeds the pending token through those layers only, writes
their K/V, and picks the next token from the shared final RMSNorm + LM head
exactly as an autoregressive step picks it (greedy, or a Gumbel-max sample
drawn at the same counters).

AdaInfer (the EE-structure page, steps 1-2): after every decoder layer l the
last token's hidden state goes through the LM head; the softmax p of those
logits gives the two features gap = p1 - p2 and top prob = p1, and the label
is 1 when that layer's top-1 token equals the final layer's.  Reading taken
here: the hidden state passes through the shared final RMSNorm before the
LM head (the early-exit head of the other two pages), and the features are
taken for the pending token of one autoregressive step, which commits the
final layer's token as that step would.  The classifiers trained on these
pairs (SVM, CRF) need training data and are not part of this restatement.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List

import numpy as np

from .model import OracleModel, logsumexp
from .philox import STREAM_RESAMPLE
from .speculative import SSDState, _pick


def lossy_step(model: OracleModel, st: SSDState, policy) -> np.ndarray:
    """One early-exit step: the pending token through the draft layers only."""
    L = model.s.n_layers
    st.round += 1
    n = st.n
    X = model.embed_rows([st.tokens[-1]])
    X = model.run_layers(X, [n - 1], st.kv, policy.draft_layers(L),
                         parts=policy.sublayers if policy.mode == "skip" else None)
    z = model.lm_head(X)[0]
    st.tokens.append(_pick(z, policy.temperature, policy.seed, n, st.round, STREAM_RESAMPLE))
    return z


def lossy_generate(model: OracleModel, st: SSDState, policy, n_new: int) -> List[np.ndarray]:
    return [lossy_step(model, st, policy) for _ in range(n_new)]


@dataclass
class LayerFeatures:
    top1: List[int]        # per layer (from min_layer on): argmax of the exit-head logits
    top_prob: List[float]  # p1
    gap: List[float]       # p1 - p2
    label: List[int]       # 1 where top1 equals the final layer's top1
    min_layer: int


def exit_features(z: np.ndarray):
    """(top1, p1, p1 - p2) of softmax(z); lowest id wins ties."""
    lse = logsumexp(z)
    i1 = int(np.argmax(z))
    z2 = z.copy()
    z2[i1] = -np.inf
    i2 = int(np.argmax(z2))
    p1, p2 = float(np.exp(z[i1] - lse)), float(np.exp(z[i2] - lse))
    return i1, p1, p1 - p2


def layer_features(model: OracleModel, st: SSDState, policy, min_layer: int = 0) -> LayerFeatures:
    """One autoregressive step of the pending token with the exit head
    applied after every layer l >= min_layer; commits the final token."""
    L = model.s.n_layers
    st.round += 1
    n = st.n
    X = model.embed_rows([st.tokens[-1]])
    f = LayerFeatures([], [], [], [], min_layer)
    z = None
    for l in range(L):
        X = model.layer(l, X, [n - 1], st.kv)
        if l >= min_layer:
            z = model.lm_head(X)[0]
            t, p1, gap = exit_features(z)
            f.top1.append(t)
            f.top_prob.append(p1)
            f.gap.append(gap)
    final = f.top1[-1]
    f.label = [int(t == final) for t in f.top1]
    st.tokens.append(_pick(z, policy.temperature, policy.seed, n, st.round, STREAM_RESAMPLE))
    return f
