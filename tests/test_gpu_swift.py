"""GPU SWIFT layer-set optimisation (ssd_swift_generate) against the oracle.

* Greedy SWIFT output is bit-identical to the library's own autoregressive
  output, whatever layer sets the optimisation picks.
* Lockstep replay: the oracle runs the same loop and, at every step,
  - proposes exactly the GPU's candidates (each side implements SplitMix64
    and the Fisher-Yates proposal on its own),
  - scores them on the same committed context; match counts agree except at
    window rows where the oracle's top-1/top-2 gap is <= 0.1,
  - then follows the GPU's scores, so that both take the same decisions;
  the winners, the stop reason, the final set and the tokens agree.
"""

from types import SimpleNamespace

import numpy as np
import pytest

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt
from synthetic.configs import Policy, ModelShape, Workload
from tests.gpu_util import to_device_weights

pytestmark = pytest.mark.gpu

SMALL = Workload(name="small-swift", shape=ModelShape(
    n_layers=6, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=704, vocab=1024),
    scaled_layers=(2, 4), scale=0.1)


@pytest.fixture(scope="module")
def ssd():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as m
    return m


def _params(**kw):
    base = dict(skip_count=2, lo_layer=1, window=8, candidates=4, max_steps=12, patience=4,
                target=0.95, seed=11)
    base.update(kw)
    return SimpleNamespace(**base)


@pytest.mark.parametrize("w,kw", [(SMALL, {}), (SMALL, {"seed": 5, "candidates": 6}),
                                  (TINY, {"skip_count": 1, "candidates": 3})])
def test_swift_is_lossless(ssd, w, kw):
    wts = make_weights(w, dtype="bf16", lm_head_scale=10.0, random_gains=True)
    p = _params(**kw)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=256,
                         max_score_rows=p.candidates * p.window)
    ctx.set_policy(Policy(mode="skip", d_max=4, tau=None))
    prompt = make_prompt(w, 16)
    f1 = ctx.prefill(prompt)
    ar, _ = ctx.decode_ar(48)
    f2 = ctx.prefill(prompt)
    toks, rep, trace = ctx.swift_generate(p, 48, trace_cap=64)
    assert f1 == f2 and toks == ar
    assert rep["steps"] >= 1 and rep["rounds"] >= 1
    assert len(trace[0]) == min(rep["steps"], 64)
    assert ctx.tokens()[len(prompt) + 1:] == ar
    ctx.close()


def _near_tie(z, thr=0.1):
    s = np.sort(z)
    return s[-1] - s[-2] <= thr


def test_swift_lockstep_with_oracle(ssd):
    from oracle import OracleModel, prefill, score_masks
    from oracle.swift import SwiftParams, swift_generate
    w = SMALL
    wts = make_weights(w, dtype="bf16", lm_head_scale=10.0, random_gains=True)
    p = _params(max_steps=8, patience=3)
    pol = Policy(mode="skip", d_max=4, tau=None)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=256,
                         max_score_rows=p.candidates * p.window)
    ctx.set_policy(pol)
    prompt = make_prompt(w, 16)
    ctx.prefill(prompt)
    toks, rep, (g_masks, g_scores, g_best) = ctx.swift_generate(p, 40, trace_cap=64)

    m = OracleModel(w.shape, weights_to_numpy(wts))
    st = prefill(m, prompt, pol, 256)
    step = [0]

    def scorer(tokens, kv, masks, N):
        s = step[0]
        assert s < len(g_masks), "the oracle ran more optimisation steps than the GPU"
        assert [tuple(c) for c in masks] == [tuple(c) for c in g_masks[s]]
        ref, _, logits = score_masks(m, tokens, kv, masks, N)
        for k in range(len(masks)):
            ties = sum(_near_tie(z) for z in logits[k])
            assert abs(round(g_scores[s][k] * N) - round(ref[k] * N)) <= ties, (s, k)
        step[0] += 1
        return g_scores[s]

    op = SwiftParams(skip_count=p.skip_count, lo_layer=p.lo_layer, window=p.window,
                     candidates=p.candidates, max_steps=p.max_steps, patience=p.patience,
                     target=p.target, seed=p.seed)
    tr = swift_generate(m, st, pol, op, 40, scorer)
    assert step[0] == rep["steps"]
    assert [s.best for s in tr.steps] == g_best
    assert tr.stopped_by == rep["stopped_by"]
    assert tuple(tr.final) == rep["final"]
    # greedy tokens (SWIFT is lossless: the model's greedy tokens) agree with
    # the oracle's autoregressive tokens until the oracle's first near-tie
    from oracle import ar_step
    ost = prefill(m, prompt, pol, 256)
    gpu = ctx.tokens()[len(prompt):]
    assert ost.tokens[-1] == gpu[0] or _near_tie(ost.last_logits)
    for i in range(1, min(20, len(gpu))):
        if ost.tokens[-1] != gpu[i - 1]:
            break
        z = ar_step(m, ost, pol)
        if _near_tie(z):
            break
        assert ost.tokens[-1] == gpu[i], i
    ctx.close()


def test_swift_argument_errors(ssd):
    from self_speculative_decoding_gb300 import SSDError
    w = TINY
    wts = make_weights(w, dtype="bf16")
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=128, max_score_rows=16)
    ctx.set_policy(Policy(mode="skip", d_max=2))
    ctx.prefill(make_prompt(w, 10))
    with pytest.raises(SSDError, match="CAPACITY"):
        ctx.swift_generate(_params(skip_count=1, window=8, candidates=3), 10)   # 24 rows > 16
    with pytest.raises(SSDError, match="INVALID_ARG"):
        ctx.swift_generate(_params(skip_count=4, lo_layer=1, candidates=2), 10)  # 4 > 3 layers
    ctx.set_policy(Policy(mode="exit", exit_layer=1, d_max=2))
    with pytest.raises(SSDError, match="STATE"):
        ctx.swift_generate(_params(skip_count=1, candidates=2), 10)
    ctx.close()
