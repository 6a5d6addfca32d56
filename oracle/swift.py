"""SWIFT on-the-fly layer-set optimisation, step by step (test infrastructure).

Follows SWIFT §4 (the method alternates context-based layer-set optimisation
with confidence-aware acceleration), §4.1.1 (uniform layer skipping
accelerates generation until the context window is filled), §4.1.2
(candidate layer sets proposed by random search are scored by a parallel
prediction of the prior context tokens; the best matchness guides the
selection; the phase ends at its step limit or when the best candidate stays
unchanged) and §B.2 (up to 1000 steps, early stop after 300 steps without
improvement or once matchness exceeds 0.95).

Readings where the pages are silent (each is listed in the design notes):

* Every candidate skips the same number of layers (the skip ratio), drawn
  from the layers lo_layer..L-1.  The uniform set spaces them evenly:
  layer lo + floor((2i + 1)(L - lo) / (2 count)) for i < count.
* Context accumulation: decoding rounds with the incumbent set; once the
  committed context holds `window` + 1 generated tokens, every round is
  followed by one optimisation step (the window slides with the context).
* One optimisation step scores K candidates in one parallel pass: the
  incumbent first, then K - 1 random proposals (a partial Fisher-Yates
  shuffle of the allowed layers driven by one SplitMix64 stream seeded once,
  numbers drawn in proposal order).  The best is the highest matchness,
  lowest index on ties, so the incumbent survives ties; "unchanged" means
  the incumbent won.
* The optimisation stops (for the rest of the generation) after the step
  whose best matchness exceeds `target`, after `max_steps` steps, or after
  `patience` consecutive unchanged steps.  Periodic Bayesian optimisation
  (SWIFT §4.1.2, every 25 steps in §B.2) is not part of this restatement.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Callable, List, Optional, Sequence, Tuple

from .scoring import score_masks
from .speculative import ssd_round

_M64 = (1 << 64) - 1


class SplitMix64:
    """Steele, Lea and Flood's SplitMix64 (OOPSLA 2014): a Weyl sequence with
    increment 0x9E3779B97F4A7C15, each state passed through a 64-bit
    finaliser."""

    def __init__(self, seed: int):
        self.state = seed & _M64

    def next(self) -> int:
        self.state = (self.state + 0x9E3779B97F4A7C15) & _M64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
        return z ^ (z >> 31)


def uniform_set(lo: int, n_layers: int, count: int) -> Tuple[int, ...]:
    span = n_layers - lo
    return tuple(lo + (2 * i + 1) * span // (2 * count) for i in range(count))


def propose(rng: SplitMix64, lo: int, n_layers: int, count: int) -> Tuple[int, ...]:
    pool = list(range(lo, n_layers))
    for i in range(count):
        j = i + rng.next() % (len(pool) - i)
        pool[i], pool[j] = pool[j], pool[i]
    return tuple(sorted(pool[:count]))


@dataclass(frozen=True)
class SwiftParams:
    skip_count: int
    lo_layer: int = 0
    window: int = 32
    candidates: int = 16
    max_steps: int = 1000
    patience: int = 300
    target: float = 0.95
    seed: int = 0


STOP_NONE, STOP_TARGET, STOP_MAX_STEPS, STOP_PATIENCE = 0, 1, 2, 3


@dataclass
class SwiftStep:
    candidates: List[Tuple[int, ...]]
    scores: List[float]
    best: int
    n_context: int          # committed length the step scored against


@dataclass
class SwiftTrace:
    steps: List[SwiftStep] = field(default_factory=list)
    stopped_by: int = STOP_NONE
    final: Tuple[int, ...] = ()
    rounds: int = 0


def swift_generate(model, st, policy, params: SwiftParams, n_tokens: int,
                   scorer: Optional[Callable] = None) -> SwiftTrace:
    """Generates n_tokens with SWIFT; st (an SSDState after prefill) is
    advanced in place.  ``scorer(tokens, kv, masks, N) -> matchness list``
    defaults to the oracle's parallel-prediction scoring."""
    L = model.s.n_layers
    if scorer is None:
        def scorer(tokens, kv, masks, N):
            return score_masks(model, tokens, kv, masks, N)[0]
    rng = SplitMix64(params.seed)
    inc = uniform_set(params.lo_layer, L, params.skip_count)
    trace = SwiftTrace()
    n_start = st.n
    optimizing = True
    unchanged = 0
    while st.n - n_start < n_tokens:
        ssd_round(model, st, replace(policy, skip=inc, skip_attn=(), skip_mlp=()))
        trace.rounds += 1
        if not optimizing or st.n - n_start < params.window + 1 or st.n - n_start >= n_tokens:
            continue
        cands = [inc] + [propose(rng, params.lo_layer, L, params.skip_count)
                         for _ in range(params.candidates - 1)]
        scores = [float(x) for x in scorer(st.tokens, st.kv, cands, params.window)]
        best = max(range(len(cands)), key=lambda k: (scores[k], -k))
        trace.steps.append(SwiftStep(cands, scores, best, st.n))
        if best == 0:
            unchanged += 1
        else:
            unchanged = 0
            inc = cands[best]
        if scores[best] > params.target:
            optimizing, trace.stopped_by = False, STOP_TARGET
        elif len(trace.steps) >= params.max_steps:
            optimizing, trace.stopped_by = False, STOP_MAX_STEPS
        elif unchanged >= params.patience:
            optimizing, trace.stopped_by = False, STOP_PATIENCE
    # the generation ends exactly n_tokens after the start
    del st.tokens[n_start + n_tokens:]
    trace.final = inc
    return trace
