"""fp32 models on the GPU (SSD_DTYPE_FP32): the tiny fp32 workload at its own
precision -- fp32 weights, activations, K/V and logits, no rounding.

* Greedy self-speculative output is bit-identical to the library's own
  autoregressive output (skip and exit policies, with and without the
  confidence stop).
* Against the oracle's fp32 mode (fp64 arithmetic, no rounding): the first
  token and autoregressive tokens agree, and draft / verify rounds agree in
  lockstep, with every draft and verify logit within rtol 1e-4 (plus 1e-5
  absolute) and every confidence within 1e-5, until the oracle's first near
  tie (top-1/top-2 gap <= 1e-3, where fp32 rounding may decide either way).
* Entry points for bf16 models only refuse an fp32 context.
"""

import numpy as np
import pytest
import torch

from synthetic import TINY, make_weights, weights_to_numpy
from synthetic.configs import Policy
from tests.gpu_util import oracle_prompt, top_gap

pytestmark = pytest.mark.gpu

TIE = 1e-3


@pytest.fixture(scope="module")
def ssd():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as m
    return m


def _ctx(ssd, lm_head_scale=1.0, max_seq=256):
    wts = make_weights(TINY, dtype="fp32", lm_head_scale=lm_head_scale, random_gains=True)
    assert wts["dtype"] == "fp32"
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in wts.items()
           if k != "layers"}
    dev["layers"] = [{k: v.cuda() for k, v in lw.items()} for lw in wts["layers"]]
    ctx = ssd.SSDContext(TINY.shape, dev, max_seq=max_seq)
    assert ctx.fp32
    return ctx, wts


POLICIES = [
    TINY.policy,                                                     # skip {2}, d_max 4, tau 0.5
    Policy(mode="skip", skip=(2,), d_max=4, tau=None),
    Policy(mode="skip", skip=(1, 2), d_max=7, tau=0.2),
    Policy(mode="exit", exit_layer=1, d_max=12, tau=None),
    Policy(mode="skip", skip_attn=(2,), skip_mlp=(1,), d_max=5, tau=None),
]


@pytest.mark.parametrize("pi", range(len(POLICIES)))
def test_fp32_greedy_ssd_is_bit_identical_to_ar(ssd, pi):
    from synthetic import make_prompt
    pol = POLICIES[pi]
    ctx, _ = _ctx(ssd, lm_head_scale=10.0)
    ctx.set_policy(pol)
    prompt = make_prompt(TINY, 20)
    f1 = ctx.prefill(prompt)
    ar, _ = ctx.decode_ar(60)
    f2 = ctx.prefill(prompt)
    toks, stats = ctx.generate(60)
    assert f1 == f2 and toks == ar
    if pol.tau is None:
        assert stats["drafted"] > 0
    ctx.close()


def test_fp32_ar_matches_oracle(ssd):
    from oracle import OracleModel, prefill, ar_generate
    pol = Policy(mode="skip", skip=(2,), d_max=4, tau=None)
    ctx, wts = _ctx(ssd, lm_head_scale=10.0)
    ctx.set_policy(pol)
    m = OracleModel(TINY.shape, weights_to_numpy(wts))
    prompt = oracle_prompt(m, TINY, pol, lambda p, st: top_gap(st.last_logits) > TIE)
    first = ctx.prefill(prompt)
    toks, _ = ctx.decode_ar(40)
    st = prefill(m, prompt, pol, 128)
    zs = [st.last_logits] + ar_generate(m, st, pol, 40)
    got = [first] + toks
    ref = st.tokens[len(prompt):]
    compared = 0
    for a, b, z in zip(got, ref, zs):
        if a != b:
            assert top_gap(z) <= TIE, f"token {compared} differs without a near tie"
            break
        compared += 1
    assert compared >= 20, compared
    ctx.close()


@pytest.mark.parametrize("pol", [
    Policy(mode="skip", skip=(2,), d_max=4, tau=None),
    Policy(mode="exit", exit_layer=1, d_max=6, tau=None),
    Policy(mode="skip", skip=(1, 2), d_max=5, tau=0.15),
], ids=["skip", "exit", "skip-tau"])
def test_fp32_rounds_match_oracle_in_lockstep(ssd, pol):
    from oracle import OracleModel, prefill, ssd_round
    ctx, wts = _ctx(ssd, lm_head_scale=10.0)
    ctx.set_policy(pol)
    m = OracleModel(TINY.shape, weights_to_numpy(wts))
    prompt = oracle_prompt(m, TINY, pol, lambda p, st: top_gap(st.last_logits) > TIE)
    first = ctx.prefill(prompt)
    st = prefill(m, prompt, pol, 256)
    assert first == st.tokens[-1]
    rounds = 0
    for _ in range(12):
        drafts, confs = ctx.draft()
        vlog = ctx.verify(d=len(drafts))
        emitted = ctx.accept()
        rec = ssd_round(m, st, pol)
        ref_conf = rec.conf + ([rec.stop_conf] if rec.stop_conf is not None else [])
        j = next(i for i in range(min(len(drafts), len(rec.draft)) + 1)
                 if i >= len(drafts) or i >= len(rec.draft) or drafts[i] != rec.draft[i])
        for a, b in list(zip(confs, ref_conf))[: j + 1]:
            assert abs(a - b) <= 1e-5
        if drafts != rec.draft:
            tie = (j < len(rec.draft_logits) and top_gap(rec.draft_logits[j]) <= TIE) or (
                pol.tau is not None and j < len(ref_conf) and abs(ref_conf[j] - pol.tau) <= 1e-5)
            assert tie, f"drafts diverge at step {j} without a near tie"
            break
        np.testing.assert_allclose(vlog, rec.verify_logits, rtol=1e-4, atol=1e-5)
        if emitted != rec.emitted:
            k = next(i for i in range(len(emitted) + 1)
                     if i >= len(emitted) or i >= len(rec.emitted) or emitted[i] != rec.emitted[i])
            assert top_gap(rec.verify_logits[min(k, len(rec.verify_logits) - 1)]) <= TIE
            break
        rounds += 1
    assert rounds >= 3, rounds
    ctx.close()


def test_fp32_refuses_bf16_only_features(ssd):
    from self_speculative_decoding_gb300 import SSDError
    ctx, _ = _ctx(ssd)
    with pytest.raises(SSDError, match="INVALID_ARG"):
        ctx.set_policy(Policy(mode="skip", skip=(2,), d_max=4, tree_tau=0.9, tree_max=2))
    ctx.set_policy(Policy(mode="skip", skip=(2,), d_max=4))
    ctx.prefill(list(range(10)))
    with pytest.raises(SSDError, match="INVALID_ARG"):
        ctx.score_masks([(1,), (2,)], 4)
    ctx.close()
