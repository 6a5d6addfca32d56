"""Pins for the oracle's lossy early-exit decoding (LayerSkip blog §3, mode
one) and the AdaInfer per-layer exit features (EE-structure page, steps 1-2).

* exit_features is the softmax's top-2 written out: checked on logits whose
  probabilities are known in closed form.
* Lossy decoding with the whole stack as the "early" model (exit at the last
  layer, or an empty skip set) is plain autoregressive decoding, token for
  token and logit for logit.
* A lossy step computes what the first draft step of a self-speculative
  round computes (the pinned drafting path): same logits, same token.
* With an early exit that drops layers, lossy decoding departs from the
  lossless output (it is not silently running the full model).
* Features: at layer l they equal the features of the exit-at-l draft
  logits; at the last layer they are the committed step's own distribution;
  0 <= gap <= top prob <= 1; the last label is 1.
"""

import math
from dataclasses import replace

import numpy as np
import pytest

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt
from synthetic.configs import Policy
from oracle import OracleModel, prefill, ar_generate, ar_step, ssd_round
from oracle.adaptive import lossy_generate, lossy_step, layer_features, exit_features
from oracle.model import logsumexp
from oracle.speculative import SSDState


def _model(dtype="fp32"):
    return OracleModel(TINY.shape, weights_to_numpy(
        make_weights(TINY, dtype=dtype, lm_head_scale=10.0, random_gains=True)))


def _copy(st):
    return SSDState(tokens=list(st.tokens), kv=st.kv.fork(), round=st.round)


def test_exit_features_closed_form():
    z = np.log(np.array([0.5, 0.25, 0.125, 0.125]))
    t, p1, gap = exit_features(z)
    assert t == 0 and math.isclose(p1, 0.5, rel_tol=1e-12) and math.isclose(gap, 0.25, rel_tol=1e-12)
    z = np.log(np.array([0.1, 0.4, 0.4, 0.1]))          # tie: lowest id first, gap 0
    t, p1, gap = exit_features(z + 3.0)                  # shift-invariant
    assert t == 1 and math.isclose(p1, 0.4, rel_tol=1e-12) and abs(gap) < 1e-15


@pytest.mark.parametrize("pol", [
    Policy(mode="exit", exit_layer=TINY.shape.n_layers - 1, d_max=3),
    Policy(mode="skip", skip=(), d_max=3),
])
def test_lossy_with_the_whole_stack_is_autoregressive(pol):
    m = _model()
    prompt = make_prompt(TINY)
    a = prefill(m, prompt, pol, 128)
    b = prefill(m, prompt, pol, 128)
    za = ar_generate(m, a, pol, 20)
    zb = lossy_generate(m, b, pol, 20)
    assert a.tokens == b.tokens
    assert all(np.array_equal(x, y) for x, y in zip(za, zb))


@pytest.mark.parametrize("pol", [
    Policy(mode="exit", exit_layer=1, d_max=3, tau=None),
    Policy(mode="skip", skip=(2,), d_max=3, tau=None),
    Policy(mode="skip", skip_mlp=(1,), skip_attn=(3,), d_max=3, tau=None),
])
def test_lossy_step_equals_first_draft_step(pol):
    m = _model()
    st = prefill(m, make_prompt(TINY), pol, 128)
    ar_generate(m, st, pol, 5)
    a, b = _copy(st), _copy(st)
    z = lossy_step(m, a, pol)
    rec = ssd_round(m, b, pol)
    assert np.array_equal(z, rec.draft_logits[0])
    assert a.tokens[-1] == rec.draft[0]


def test_early_exit_is_lossy():
    m = _model()
    pol = Policy(mode="exit", exit_layer=0, d_max=3)
    prompt = make_prompt(TINY)
    a = prefill(m, prompt, pol, 128)
    b = prefill(m, prompt, pol, 128)
    ar_generate(m, a, pol, 30)
    lossy_generate(m, b, pol, 30)
    assert a.tokens != b.tokens


@pytest.mark.parametrize("min_layer", [0, 2])
def test_layer_features(min_layer):
    m = _model()
    L = TINY.shape.n_layers
    pol = Policy(mode="skip", skip=(), d_max=3)
    st = prefill(m, make_prompt(TINY), pol, 128)
    ar_generate(m, st, pol, 4)
    ref = _copy(st)
    f = layer_features(m, st, pol, min_layer)
    assert len(f.top1) == L - min_layer
    # the step commits what an autoregressive step commits
    z_final = ar_step(m, ref, pol)
    assert st.tokens == ref.tokens
    assert f.top1[-1] == st.tokens[-1] and f.label[-1] == 1
    assert math.isclose(f.top_prob[-1], float(np.exp(np.max(z_final) - logsumexp(z_final))),
                        rel_tol=1e-12)
    for i, l in enumerate(range(min_layer, L)):
        # features at layer l = those of the exit-at-l draft logits
        b = _copy(ref)
        b.tokens.pop()
        b.round -= 1
        rec = ssd_round(m, b, Policy(mode="exit", exit_layer=l, d_max=1, tau=None))
        t, p1, gap = exit_features(rec.draft_logits[0])
        assert (t, p1, gap) == (f.top1[i], f.top_prob[i], f.gap[i])
        assert 0.0 <= f.gap[i] <= f.top_prob[i] <= 1.0
        assert f.top_prob[i] >= 1.0 / TINY.shape.vocab
        assert f.label[i] == int(f.top1[i] == f.top1[-1])
