"""Matchness scoring of candidate skip sets (test infrastructure).

SWIFT §4.1 and §4.1.2: a candidate layer set is validated against tokens the
LLM already generated, by one parallel forward of the layer-skipped model
over a window of the context; its matchness is the fraction of window tokens
it predicts (top-1) correctly, and the best-scoring candidate is kept.  SWIFT
D.2 fixes the window at gamma = 32.

Reading taken here: with committed tokens t[0..n-1], the window inputs are
t[n-N-1 .. n-2] at their own positions and the ground truth is t[n-N .. n-1].
Each candidate model attends to the full-model K/V of the prefix
[0, n-N-1) and to its own K/V for the window positions (computed causally in
the same pass).  Skipped layers are the identity.  Ties in the best score go
to the lowest candidate index.
"""

from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

from .model import OracleModel


def score_masks(model: OracleModel, tokens: Sequence[int], kv, masks: Sequence[Sequence[int]],
                N: int) -> Tuple[np.ndarray, int, List[np.ndarray]]:
    """Returns (matchness [K], best index, per-mask logits [N, V])."""
    n = len(tokens)
    L = model.s.n_layers
    inputs = list(tokens[n - N - 1: n - 1])
    targets = np.asarray(tokens[n - N: n])
    positions = range(n - N - 1, n - 1)
    scores = np.zeros(len(masks))
    logits = []
    for k, skip in enumerate(masks):
        own = kv.fork()
        skip = set(skip)
        X = model.embed_rows(inputs)
        X = model.run_layers(X, positions, own, [l for l in range(L) if l not in skip])
        Z = model.lm_head(X)
        logits.append(Z)
        scores[k] = np.sum(np.argmax(Z, axis=1) == targets) / N
    best = int(np.argmax(scores))
    return scores, best, logits


def score_masks_bruteforce(model: OracleModel, tokens: Sequence[int], kv,
                           masks: Sequence[Sequence[int]], N: int) -> np.ndarray:
    """The same count, one window token at a time (sequential single-row drafts)."""
    n = len(tokens)
    L = model.s.n_layers
    counts = np.zeros(len(masks), dtype=np.int64)
    for k, skip in enumerate(masks):
        own = kv.fork()
        keep = [l for l in range(L) if l not in set(skip)]
        for i in range(N):
            pos = n - N - 1 + i
            X = model.embed_rows([tokens[pos]])
            X = model.run_layers(X, [pos], own, keep)
            pred = int(np.argmax(model.lm_head(X)[0]))
            counts[k] += int(pred == tokens[pos + 1])
    return counts
