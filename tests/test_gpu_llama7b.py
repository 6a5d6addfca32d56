"""GPU against the oracle on the Llama-2-7B shape (L 32, d_model 4096, 32
heads x 128, FFN 11008, vocab 32000), with the workloads' own bf16 weights
(no sharpening) and a 16-token prompt:

* the SWIFT skip set of the skip workload (odd layers 9..31) with the
  confidence stop off, so that drafts of 8 tokens and 9-row verify passes
  run;
* the LayerSkip exit workload (exit layer 8, d = 12, T = 0.6, Philox seed
  1234): 13-row verify passes from the reused layer 0..8 K/V, sampled drafts,
  min(1, p/q) acceptance.

Rounds run in lockstep until the first decision within the tolerance of its
boundary: every compared confidence within 1e-3 and every compared logit
within LOGIT_TOL.  Tolerance at this depth: both sides round to bf16 at the
same points (the normalised inputs, the attention output, the SwiGLU
product, the stored K/V), but an element whose fp32 (GPU) and fp64 (oracle)
values lie on opposite sides of a bf16 rounding boundary is rounded one
ulp apart; each such difference perturbs the next layer's inputs, so the
rounding differences compound through the 32 layers.  On the 4-6 layer
parity models the logits agree within 0.003-0.006 (the stated 5e-2 holds
there, test_gpu_model.py); on this 32-layer shape the measured deviation
is about 0.1, so logits are compared within LOGIT_TOL = 0.25 and a token
decision counts as near its boundary within the same 0.25 (a top-1/top-2
gap, a Gumbel-score gap) or 0.05 in log(p/q).  The prompt is the first seeded prompt
whose first token is not a near decision on the oracle's side.  Random
weights put many decisions near their boundary at this vocabulary, so the
comparison covers the first round or more; the run asserts at least one
compared draft step and reports the rounds compared.

The fp64 oracle keeps the widened weights (about 53 GB of host memory) and
takes a few seconds per round on the host cores.
"""

from dataclasses import replace

import numpy as np
import pytest
import torch

from synthetic import LLAMA7B_SWIFT, LLAMA7B_LAYERSKIP, make_weights, weights_to_numpy
from tests.gpu_util import oracle_prompt

pytestmark = pytest.mark.gpu

LOGIT_TOL = 0.25


@pytest.fixture(scope="module")
def ssd():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as m
    return m


def _setup(ssd, w, pol):
    from oracle import OracleModel
    wts = make_weights(w, device="cuda", dtype="bf16")
    m = OracleModel(w.shape, weights_to_numpy(wts), cache_limit_bytes=64 << 30)
    packed = ssd.pack_weights(wts, release=True)
    del wts
    ctx = ssd.SSDContext(w.shape, packed, max_seq=128, max_draft=max(pol.d_max, 1))
    ctx.set_policy(pol)
    return ctx, m, packed


def test_llama7b_skip_rounds_match_oracle(ssd):
    from oracle import prefill
    from tests.test_gpu_model import _lockstep, _near_tie
    w = LLAMA7B_SWIFT
    pol = replace(w.policy, tau=None)
    ctx, m, packed = _setup(ssd, w, pol)
    prompt = oracle_prompt(m, w, pol, lambda p, st: not _near_tie(st.last_logits, LOGIT_TOL),
                           length=16, max_seq=128)
    first = ctx.prefill(prompt)
    st = prefill(m, prompt, pol, 128)
    assert first == st.tokens[-1]
    dev = []
    rounds = _lockstep(ctx, m, st, pol, 1.0, min_rounds=0, max_rounds=3, logit_tol=LOGIT_TOL,
                       tie=LOGIT_TOL, dev=dev)
    print(f"7B skip: {rounds} rounds compared, verify-logit deviations {dev}")
    ctx.close()
    del packed, m
    torch.cuda.empty_cache()


def test_llama7b_exit_sampled_rounds_match_oracle(ssd):
    from oracle import prefill
    from tests.test_gpu_model import _sampled_lockstep, _gumbel_gap
    w = LLAMA7B_LAYERSKIP
    pol = w.policy
    assert pol.mode == "exit" and pol.exit_layer == 8 and pol.temperature == 0.6
    ctx, m, packed = _setup(ssd, w, pol)
    T, seed = pol.temperature, pol.seed
    prompt = oracle_prompt(
        m, w, pol, lambda p, st: _gumbel_gap(st.last_logits, T, seed, len(p), 0, 2) > LOGIT_TOL,
        length=16, max_seq=128)
    first = ctx.prefill(prompt)
    st = prefill(m, prompt, pol, 128)
    assert first == st.tokens[-1]
    dev = []
    rounds = _sampled_lockstep(ctx, m, st, pol, 1.0, max_rounds=3, logit_tol=LOGIT_TOL,
                               tie=LOGIT_TOL, dev=dev)
    print(f"7B exit T=0.6: {rounds} rounds compared, verify-logit deviations {dev}")
    ctx.close()
    del packed, m
    torch.cuda.empty_cache()
