"""GPU dynamic verification (SWIFT §4.2 / §3.2.1: siblings from the draft's
second choice verified with the chain) through the context C-ABI.

* Greedy output with siblings is bit-identical to the library's own
  autoregressive greedy output, up to 16 verify rows (the wide verify graph
  included).
* Round by round the emitted tokens (a taken sibling's extra token included)
  equal the oracle's until the oracle reports a near decision: a top-1/top-2
  logit gap <= 0.1 (draft, verify or sibling row), a second/third draft
  choice gap <= 0.1 where a sibling is drawn, or a confidence within the
  confidence tolerance of tau or tree_tau.
* Sibling counts (verified, taken) equal the oracle's over a whole
  generation when no near decision occurs in it.
* Policy checks: temperature > 0, tree_max outside 1..8 and more than 16
  verify rows are refused.
"""

import numpy as np
import pytest

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt
from synthetic.configs import Policy, ModelShape, Workload
from tests.gpu_util import to_device_weights, oracle_prompt

pytestmark = pytest.mark.gpu

SMALL_GQA = Workload(name="small-gqa", shape=ModelShape(
    n_layers=6, d_model=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=1408, vocab=2048),
    scaled_layers=(2, 3), scale=0.1)
MID = Workload(name="mid-dh128", shape=ModelShape(
    n_layers=4, d_model=1024, n_heads=8, n_kv_heads=8, head_dim=128, ffn_dim=2816, vocab=4096),
    scaled_layers=(1, 2), scale=0.1)
WIDE = Workload(name="wide-d4096", shape=ModelShape(
    n_layers=3, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn_dim=2048, vocab=4096),
    scaled_layers=(1,), scale=0.1)

CASES = [
    (TINY, Policy(mode="skip", skip=(2,), d_max=4, tau=None, tree_tau=1.0, tree_max=4)),
    (TINY, Policy(mode="skip", skip=(1, 2), d_max=3, tau=0.05, tree_tau=0.9, tree_max=3)),
    (TINY, Policy(mode="exit", exit_layer=1, d_max=6, tau=None, tree_tau=1.0, tree_max=6)),
    (TINY, Policy(mode="skip", skip_attn=(1,), skip_mlp=(2,), d_max=5, tau=None,
                  tree_tau=0.8, tree_max=2)),
    (SMALL_GQA, Policy(mode="skip", skip=(2, 3), d_max=8, tau=None, tree_tau=0.8, tree_max=7)),
    (MID, Policy(mode="skip", skip=(1, 2), d_max=8, tau=0.1, tree_tau=0.9, tree_max=7)),
    (WIDE, Policy(mode="skip", skip=(1,), d_max=8, tau=None, tree_tau=1.0, tree_max=7)),
    (WIDE, Policy(mode="exit", exit_layer=0, d_max=7, tau=None, tree_tau=1.0, tree_max=8)),
]


@pytest.fixture(scope="module")
def ssd():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as m
    return m


def _ctx(ssd, w, head=10.0, max_seq=256):
    wts = make_weights(w, dtype="bf16", lm_head_scale=head, random_gains=True)
    return ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=max_seq), wts


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_tree_greedy_is_bit_identical_to_ar(ssd, ci):
    w, pol = CASES[ci]
    ctx, _ = _ctx(ssd, w)
    ctx.set_policy(pol)
    prompt = make_prompt(w, 20)
    ctx.prefill(prompt)
    ar, _ = ctx.decode_ar(60)
    ctx.prefill(prompt)
    toks, stats = ctx.generate(60)
    assert toks == ar
    if pol.tree_tau >= 1.0:
        assert stats["side_rows"] > 0
    assert stats["side_accepted"] <= stats["rounds"]
    ctx.close()


def _near_tie(z, thr=0.1):
    s = np.sort(z)
    return s[-1] - s[-2] <= thr


def _near_second(z, thr=0.1):
    s = np.sort(z)
    return s[-2] - s[-3] <= thr


def _near_decision(rec, pol, conf_tol):
    """Does the oracle's round hold a decision the GPU may take the other way?
    The stop (tau) and sibling (tree_tau) thresholds, the draft's top-1 at
    every kept step, its top-2 at the steps that drew a sibling, the verify
    rows up to the first rejection, and a taken sibling's own row."""
    for c in rec.conf + ([rec.stop_conf] if rec.stop_conf is not None else []):
        if pol.tau is not None and abs(c - pol.tau) <= conf_tol:
            return True
    if any(abs(c - pol.tree_tau) <= conf_tol for c in rec.conf):
        return True
    if any(_near_tie(z) for z in rec.draft_logits):
        return True
    if any(_near_second(rec.draft_logits[j]) for j, _ in rec.siblings):
        return True
    if any(_near_tie(z) for z in rec.verify_logits[: rec.accepted + 1]):
        return True
    return rec.sibling_taken is not None and _near_tie(rec.sibling_logits[rec.sibling_taken])


@pytest.mark.parametrize("ci,head", [(0, 1.0), (0, 10.0), (1, 10.0), (2, 10.0), (4, 1.0)])
def test_tree_rounds_match_oracle_in_lockstep(ssd, ci, head):
    from oracle import OracleModel, prefill, ssd_round
    w, pol = CASES[ci]
    ctx, wts = _ctx(ssd, w, head)
    ctx.set_policy(pol)
    m = OracleModel(w.shape, weights_to_numpy(wts))
    prompt = oracle_prompt(m, w, pol, lambda p, st: not _near_tie(st.last_logits))
    first = ctx.prefill(prompt)
    st = prefill(m, prompt, pol, 256)
    assert first == st.tokens[-1]
    conf_tol = 1e-3 * head
    rounds = taken = 0
    for _ in range(16):
        drafts, _ = ctx.draft()
        ctx.verify(want_logits=False)
        emitted = ctx.accept()
        rec = ssd_round(m, st, pol)
        if drafts != rec.draft or emitted != rec.emitted:
            assert _near_decision(rec, pol, conf_tol), \
                f"round {rounds}: GPU {drafts} -> {emitted}, oracle {rec.draft} -> {rec.emitted}"
            break
        taken += rec.sibling_taken is not None
        rounds += 1
    assert rounds >= 3, rounds
    ctx.close()


@pytest.mark.parametrize("ci,head", [(0, 10.0), (2, 10.0), (1, 10.0)])
def test_tree_counts_match_oracle(ssd, ci, head):
    # Rounds run in lockstep with the oracle up to the first round whose
    # drafts or emitted tokens differ (or whose confidence lies within the
    # tolerance of tree_tau); generate() then replays exactly those rounds'
    # tokens and must report the same rounds and sibling counts.
    from oracle import OracleModel, prefill, ssd_round
    w, pol = CASES[ci]
    ctx, wts = _ctx(ssd, w, head)
    ctx.set_policy(pol)
    prompt = make_prompt(w)
    m = OracleModel(w.shape, weights_to_numpy(wts))
    st = prefill(m, prompt, pol, 256)
    ctx.prefill(prompt)
    recs = []
    for _ in range(24):
        drafts, _ = ctx.draft()
        ctx.verify(want_logits=False)
        emitted = ctx.accept()
        rec = ssd_round(m, st, pol)
        if drafts != rec.draft or emitted != rec.emitted or \
                any(abs(c - pol.tree_tau) <= 1e-3 * head for c in rec.conf):
            break
        recs.append(rec)
    assert len(recs) >= 3 and sum(len(r.siblings) for r in recs) > 0, len(recs)
    n = sum(len(r.emitted) for r in recs)
    ctx.prefill(prompt)
    toks, stats = ctx.generate(n)
    assert toks == [t for r in recs for t in r.emitted]
    assert (stats["rounds"], stats["side_rows"], stats["side_accepted"]) == \
        (len(recs), sum(len(r.siblings) for r in recs),
         sum(r.sibling_taken is not None for r in recs))
    ctx.close()


def test_tree_off_equals_chain(ssd):
    w = TINY
    base = Policy(mode="skip", skip=(2,), d_max=4, tau=None)
    ctx, _ = _ctx(ssd, w)
    prompt = make_prompt(w, 20)
    ctx.set_policy(base)
    ctx.prefill(prompt)
    a, sa = ctx.generate(50)
    ctx.set_policy(Policy(mode="skip", skip=(2,), d_max=4, tau=None, tree_tau=0.0, tree_max=4))
    ctx.prefill(prompt)
    b, sb = ctx.generate(50)
    assert a == b and sa["rounds"] == sb["rounds"] and sb["side_rows"] == 0
    ctx.close()


def test_tree_policy_checks(ssd):
    from self_speculative_decoding_gb300 import SSDError
    ctx, _ = _ctx(ssd, TINY)
    for pol in (Policy(mode="skip", skip=(2,), d_max=4, temperature=0.7, tree_tau=0.9, tree_max=2),
                Policy(mode="skip", skip=(2,), d_max=4, tree_tau=0.9, tree_max=0),
                Policy(mode="skip", skip=(2,), d_max=4, tree_tau=0.9, tree_max=9),
                Policy(mode="skip", skip=(2,), d_max=12, tree_tau=0.9, tree_max=4)):
        with pytest.raises(SSDError, match="INVALID_ARG"):
            ctx.set_policy(pol)
    ctx.set_policy(Policy(mode="skip", skip=(2,), d_max=11, tree_tau=0.9, tree_max=4))
    ctx.close()
