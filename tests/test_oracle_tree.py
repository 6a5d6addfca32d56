"""Pins for the oracle's dynamic verification (SWIFT §4.2: the draft's
confidence also sets how many candidates go to the verify; §3.2.1: top-k
drafts raise the accepted length).

What the pages and the mathematics fix, and these tests check:
* greedy decoding stays lossless: with sibling candidates the output equals
  greedy autoregressive decoding token for token;
* a taken sibling's verify row is the full model's prediction after the
  accepted prefix and the sibling: equal (fp64 rounding) to a from-scratch
  forward of the whole sequence, with no cache reuse;
* per round, the emitted tokens start with what the chain rule emits from the
  same verify logits, and there is exactly one more token iff a sibling was
  taken;
* the sibling rule: the draft's second choice for kept drafts whose
  confidence is below tree_tau, at most tree_max, in depth order;
* planted slips (a sibling one position late, a sibling that writes into the
  shared cache instead of a fork) are caught.
"""

import numpy as np
import pytest

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt
from synthetic.configs import Policy
from oracle import OracleModel, prefill, ar_generate, ssd_generate
from oracle import speculative as spec_mod
from oracle.model import top2

TREE_POLICIES = [
    Policy(mode="skip", skip=(2,), d_max=4, tau=None, tree_tau=1.0, tree_max=4),
    Policy(mode="skip", skip=(1, 2), d_max=3, tau=0.05, tree_tau=0.9, tree_max=3),
    Policy(mode="skip", skip=(2,), d_max=5, tau=0.2, tree_tau=0.7, tree_max=2),
    Policy(mode="exit", exit_layer=0, d_max=6, tau=None, tree_tau=1.0, tree_max=6),
]


def _model(head=10.0):
    return OracleModel(TINY.shape, weights_to_numpy(
        make_weights(TINY, dtype="fp32", lm_head_scale=head, random_gains=True)))


def _run(m, pol, n_new=40, prompt_len=12):
    st = prefill(m, make_prompt(TINY, prompt_len), pol, 128)
    g = ssd_generate(m, st, pol, n_new)
    return st, g


def _ar(m, pol, n_new=40, prompt_len=12):
    st = prefill(m, make_prompt(TINY, prompt_len), pol, 128)
    ar_generate(m, st, pol, n_new)
    return st.tokens


@pytest.mark.parametrize("pi", range(len(TREE_POLICIES)))
def test_tree_greedy_equals_ar(pi):
    m = _model()
    pol = TREE_POLICIES[pi]
    st, g = _run(m, pol)
    assert st.tokens == _ar(m, pol)
    assert g.side_rows == sum(len(r.siblings) for r in g.records)


def test_siblings_are_taken():
    # the mechanism is exercised: siblings are verified and some are taken
    m = _model()
    _, g = _run(m, TREE_POLICIES[0])
    assert g.side_rows > 0 and g.side_accepted > 0
    _, g = _run(m, TREE_POLICIES[1])
    assert g.side_accepted > 0


@pytest.mark.parametrize("pi", [0, 1])
def test_taken_sibling_row_equals_fresh_forward(pi):
    m = _model()
    pol = TREE_POLICIES[pi]
    st, g = _run(m, pol)
    L = m.s.n_layers
    checked = 0
    for r in g.records:
        if r.sibling_taken is None:
            continue
        j, s_tok = r.siblings[r.sibling_taken]
        seq = st.tokens[: r.n_before + j] + [s_tok]
        kv = m.new_cache(128)
        X = m.run_layers(m.embed_rows(seq), range(len(seq)), kv, range(L))
        z = m.lm_head(X[-1:])[0]
        np.testing.assert_allclose(r.sibling_logits[r.sibling_taken], z, rtol=0, atol=1e-9)
        checked += 1
    assert checked > 0


@pytest.mark.parametrize("pi", range(len(TREE_POLICIES)))
def test_round_adds_one_token_exactly_when_a_sibling_is_taken(pi):
    m = _model()
    _, g = _run(m, TREE_POLICIES[pi])
    for r in g.records:
        a = 0
        while a < r.d and r.draft[a] == int(np.argmax(r.verify_logits[a])):
            a += 1
        chain = r.draft[:a] + [int(np.argmax(r.verify_logits[a]))]
        assert r.accepted == a
        assert r.emitted[: a + 1] == chain
        assert len(r.emitted) == a + 1 + (r.sibling_taken is not None)
        if r.sibling_taken is not None:
            j, s_tok = r.siblings[r.sibling_taken]
            assert j == a < r.d and s_tok == chain[-1]
            assert r.emitted[-1] == int(np.argmax(r.sibling_logits[r.sibling_taken]))


@pytest.mark.parametrize("pi", range(len(TREE_POLICIES)))
def test_sibling_rule(pi):
    m = _model()
    pol = TREE_POLICIES[pi]
    _, g = _run(m, pol)
    for r in g.records:
        want = [(j, top2(r.draft_logits[j])[2]) for j in range(r.d)
                if r.conf[j] < pol.tree_tau][: pol.tree_max]
        assert r.siblings == want


def test_tree_off_has_no_siblings_and_same_rounds():
    m = _model()
    base = Policy(mode="skip", skip=(2,), d_max=4, tau=None)
    _, g0 = _run(m, base)
    _, g1 = _run(m, Policy(mode="skip", skip=(2,), d_max=4, tau=None, tree_tau=None, tree_max=4))
    assert g1.side_rows == 0
    assert [r.emitted for r in g0.records] == [r.emitted for r in g1.records]


def test_sibling_one_position_late_is_caught(monkeypatch):
    orig = spec_mod.sibling_step
    monkeypatch.setattr(spec_mod, "sibling_step",
                        lambda model, kv, pos, tok: orig(model, kv, pos + 1, tok))
    m = _model()
    st, g = _run(m, TREE_POLICIES[0])
    assert g.side_accepted > 0
    assert st.tokens != _ar(m, TREE_POLICIES[0])


def test_sibling_without_fork_is_caught(monkeypatch):
    def shared(model, kv, pos, tok):
        X = model.run_layers(model.embed_rows([tok]), [pos], kv, range(model.s.n_layers))
        return model.lm_head(X)[0], kv
    monkeypatch.setattr(spec_mod, "sibling_step", shared)
    m = _model()
    pol = TREE_POLICIES[0]
    st, g = _run(m, pol)
    assert st.tokens != _ar(m, pol)
