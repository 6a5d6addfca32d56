"""Pins for the oracle's SWIFT layer-set optimisation loop (SWIFT §4.1,
§4.1.1, §4.1.2, §B.2).

* SplitMix64 reproduces published outputs (tests/golden/splitmix64.json).
* Proposals are sets of `count` distinct layers from lo..L-1; the uniform
  set is evenly spaced.
* The stopping rules fire at the right step: matchness above the target,
  the step limit, `patience` unchanged steps (driven by a scripted scorer).
* The incumbent is candidate 0 and keeps its place on ties.
* Greedy SWIFT output equals greedy autoregressive output (lossless),
  whatever the candidates score.
"""

import json
import os

import numpy as np
import pytest

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt
from synthetic.configs import Policy
from oracle import OracleModel, prefill, ar_generate
from oracle.swift import (SplitMix64, SwiftParams, swift_generate, uniform_set, propose,
                          STOP_TARGET, STOP_MAX_STEPS, STOP_PATIENCE, STOP_NONE)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64.json")


def test_splitmix64_known_answers():
    g = json.load(open(GOLDEN))
    r = SplitMix64(1234567)
    assert [r.next() for _ in range(5)] == [int(x) for x in g["seed_1234567_first5"]]
    assert SplitMix64(0).next() == int(g["seed_0_first"])


def test_proposals_and_uniform_set():
    rng = SplitMix64(5)
    seen = set()
    for _ in range(200):
        c = propose(rng, 4, 40, 16)
        assert len(c) == 16 and len(set(c)) == 16 and all(4 <= l < 40 for l in c)
        assert list(c) == sorted(c)
        seen.add(c)
    assert len(seen) == 200                      # no repeats at C(36, 16)
    assert uniform_set(4, 40, 16) == (5, 7, 9, 11, 14, 16, 18, 20, 23, 25, 27, 29, 32, 34, 36, 38)
    assert uniform_set(0, 4, 2) == (1, 3)
    # layers are covered uniformly by the proposals
    counts = np.zeros(40)
    rng = SplitMix64(9)
    for _ in range(3000):
        for l in propose(rng, 4, 40, 16):
            counts[l] += 1
    exp = 3000 * 16 / 36
    assert np.all(np.abs(counts[4:] - exp) < 6 * np.sqrt(exp))


def _model():
    return OracleModel(TINY.shape, weights_to_numpy(
        make_weights(TINY, dtype="fp32", lm_head_scale=10.0, random_gains=True)))


POL = Policy(mode="skip", d_max=3, tau=None)


def _run(scores_by_step, params, n_tokens=60):
    """Runs the loop with a scripted scorer; returns the trace."""
    m = _model()
    st = prefill(m, make_prompt(TINY), POL, 256)
    calls = []

    def scorer(tokens, kv, masks, N):
        assert N == params.window and len(masks) == params.candidates
        assert len(tokens) - N - 1 >= 0
        s = scores_by_step(len(calls), masks)
        calls.append((list(masks), s))
        return s

    return swift_generate(m, st, POL, params, n_tokens, scorer), calls


def test_stop_on_target():
    p = SwiftParams(skip_count=1, lo_layer=1, window=8, candidates=3, max_steps=50, patience=50)
    tr, calls = _run(lambda t, masks: [0.2, 0.5, 0.1] if t < 2 else [0.5, 0.97, 0.1], p)
    assert tr.stopped_by == STOP_TARGET and len(tr.steps) == 3
    assert tr.steps[0].best == 1 and tr.steps[2].best == 1
    assert tr.final == calls[2][0][1]


def test_stop_on_step_limit_and_incumbent_wins_ties():
    p = SwiftParams(skip_count=1, lo_layer=1, window=8, candidates=3, max_steps=4, patience=50)
    tr, calls = _run(lambda t, masks: [0.3, 0.3, 0.3], p)
    assert tr.stopped_by == STOP_MAX_STEPS and len(tr.steps) == 4
    assert all(s.best == 0 for s in tr.steps)
    assert tr.final == uniform_set(1, 4, 1)
    # the incumbent is candidate 0 of every step
    assert all(c[0][0] == tr.final for c in calls)


def test_stop_on_patience():
    p = SwiftParams(skip_count=2, lo_layer=0, window=8, candidates=4, max_steps=50, patience=3)
    seq = [[0.1, 0.4, 0.2, 0.3], [0.4, 0.1, 0.6, 0.2]] + [[0.5, 0.2, 0.1, 0.0]] * 10
    tr, calls = _run(lambda t, masks: seq[t], p)
    assert [s.best for s in tr.steps] == [1, 2, 0, 0, 0]
    assert tr.stopped_by == STOP_PATIENCE
    assert tr.final == calls[1][0][2]


def test_no_stop_within_budget():
    p = SwiftParams(skip_count=1, lo_layer=1, window=8, candidates=2, max_steps=1000, patience=1000)
    tr, _ = _run(lambda t, masks: [0.0, 0.5], p, n_tokens=30)
    assert tr.stopped_by == STOP_NONE and len(tr.steps) >= 1


@pytest.mark.parametrize("seed", [0, 3])
def test_greedy_swift_is_lossless(seed):
    m = _model()
    prompt = make_prompt(TINY)
    st_ar = prefill(m, prompt, POL, 256)
    ar_generate(m, st_ar, POL, 50)
    st = prefill(m, prompt, POL, 256)
    p = SwiftParams(skip_count=1, lo_layer=1, window=8, candidates=3, max_steps=20, patience=5,
                    seed=seed)
    tr = swift_generate(m, st, POL, p, 50)
    assert st.tokens == st_ar.tokens
    assert len(tr.steps) >= 1
