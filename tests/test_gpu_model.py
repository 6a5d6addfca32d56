"""End-to-end GPU tests through the context C-ABI.

* The library's greedy self-speculative output is bit-identical to its own
  autoregressive greedy output (no exclusions), for skip and exit policies,
  MHA and GQA shapes, with and without the confidence stop.
* GPU and oracle run the same seeded inputs independently and are compared
  token by token and round by round until the oracle reports a near-tie
  (top-1/top-2 logit gap <= 0.1, or a confidence within 1e-3 of tau), where
  the two may legitimately diverge.  Logits must agree within 5e-2 and
  confidences within 1e-3 on every compared row.
"""

from dataclasses import replace

import numpy as np
import pytest
import torch

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt, shrink
from synthetic.configs import Policy, ModelShape, Workload
from tests.gpu_util import to_device_weights, top_gap, oracle_prompt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssd():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as m
    return m


SMALL_GQA = Workload(name="small-gqa", shape=ModelShape(
    n_layers=6, d_model=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=1408, vocab=2048),
    scaled_layers=(2, 3), scale=0.1)
MID = Workload(name="mid-dh128", shape=ModelShape(
    n_layers=4, d_model=1024, n_heads=8, n_kv_heads=8, head_dim=128, ffn_dim=2816, vocab=4096),
    scaled_layers=(1, 2), scale=0.1)

# wide enough that a verify pass of more than 5 rows does not fit the GEMV's
# 44 KB activation stage: the norm pre-pass and the windowed activation layout run
WIDE = Workload(name="wide-d4096", shape=ModelShape(
    n_layers=3, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn_dim=2048, vocab=4096),
    scaled_layers=(1,), scale=0.1)

CASES = [
    (TINY, Policy(mode="skip", skip=(2,), d_max=4, tau=None)),
    (TINY, Policy(mode="skip", skip=(2,), d_max=4, tau=0.5)),
    (TINY, Policy(mode="skip", skip=(1, 2), d_max=7, tau=0.2)),
    (TINY, Policy(mode="exit", exit_layer=1, d_max=12, tau=None)),
    (TINY, Policy(mode="exit", exit_layer=3, d_max=3, tau=None)),
    (TINY, Policy(mode="skip", skip=(), d_max=15, tau=None)),
    (TINY, Policy(mode="skip", skip=(0,), d_max=1, tau=None)),
    (SMALL_GQA, Policy(mode="skip", skip=(2, 3), d_max=8, tau=None)),
    (SMALL_GQA, Policy(mode="exit", exit_layer=2, d_max=12, tau=None)),
    (MID, Policy(mode="skip", skip=(1, 2), d_max=8, tau=0.1)),
    (MID, Policy(mode="exit", exit_layer=0, d_max=6, tau=None)),
    # sub-layer drops (SWIFT Fig. 10): attention-only, MLP-only and mixed
    (TINY, Policy(mode="skip", skip_attn=(2,), d_max=4, tau=None)),
    (TINY, Policy(mode="skip", skip_mlp=(1, 3), d_max=5, tau=0.2)),
    (SMALL_GQA, Policy(mode="skip", skip=(4,), skip_attn=(2,), skip_mlp=(3,), d_max=6, tau=None)),
    (MID, Policy(mode="skip", skip_attn=(1,), skip_mlp=(2,), d_max=8, tau=None)),
    (WIDE, Policy(mode="skip", skip=(1,), d_max=8, tau=None)),
    (WIDE, Policy(mode="exit", exit_layer=0, d_max=12, tau=None)),
]


def _ctx(ssd, w, lm_head_scale=10.0, max_seq=256, seed_gains=True):
    wts = make_weights(w, dtype="bf16", lm_head_scale=lm_head_scale, random_gains=seed_gains)
    dev = to_device_weights(wts)
    return ssd.SSDContext(w.shape, dev, max_seq=max_seq), wts


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_greedy_ssd_is_bit_identical_to_ar(ssd, ci):
    w, pol = CASES[ci]
    ctx, _ = _ctx(ssd, w)
    ctx.set_policy(pol)
    prompt = make_prompt(w, 20)
    f1 = ctx.prefill(prompt)
    ar, _ = ctx.decode_ar(60)
    f2 = ctx.prefill(prompt)
    toks, stats = ctx.generate(60)
    assert f1 == f2
    assert toks == ar
    assert stats["emitted"] >= 60 and stats["rounds"] >= 60 // (pol.d_max + 1)
    assert ctx.tokens() == [int(t) for t in prompt] + [f1] + ar
    ctx.close()


def test_generation_continues_across_calls_and_rewind(ssd):
    w, pol = CASES[0]
    ctx, _ = _ctx(ssd, w)
    ctx.set_policy(pol)
    prompt = make_prompt(w, 20)
    ctx.prefill(prompt)
    full, _ = ctx.generate(40)
    ctx.prefill(prompt)
    a, _ = ctx.generate(13)
    b, _ = ctx.generate(27)
    assert a + b == full
    n = len(ctx.tokens())
    ctx.rewind(n - 10)
    c, _ = ctx.generate(10)
    assert c == full[-10:]
    ctx.close()


def _near_tie(z, thr=0.1):
    s = np.sort(z)
    return s[-1] - s[-2] <= thr


def test_ar_greedy_matches_oracle(ssd):
    from oracle import OracleModel, prefill, ar_generate
    w = TINY
    pol = Policy(mode="skip", skip=(2,), d_max=4, tau=None)
    ctx, wts = _ctx(ssd, w, lm_head_scale=40.0)
    ctx.set_policy(pol)
    prompt = make_prompt(w)
    first = ctx.prefill(prompt)
    toks, _ = ctx.decode_ar(40)
    m = OracleModel(w.shape, weights_to_numpy(wts))
    st = prefill(m, prompt, pol, 128)
    zs = [st.last_logits] + ar_generate(m, st, pol, 40)
    ref = st.tokens[len(prompt):]
    got = [first] + toks
    compared = 0
    for a, b, z in zip(got, ref, zs):
        if a != b:
            assert _near_tie(z), f"token {compared} differs without a near-tie"
            break
        compared += 1
    assert compared >= 8, compared
    ctx.close()


@pytest.mark.parametrize("w,pol,head", [
    (TINY, Policy(mode="skip", skip=(2,), d_max=4, tau=None), 1.0),
    (TINY, Policy(mode="skip", skip=(2,), d_max=4, tau=None), 10.0),
    (TINY, Policy(mode="skip", skip=(1, 2), d_max=5, tau=0.15), 10.0),
    (SMALL_GQA, Policy(mode="exit", exit_layer=1, d_max=6, tau=None), 1.0),
    (SMALL_GQA, Policy(mode="exit", exit_layer=1, d_max=6, tau=None), 10.0),
    (TINY, Policy(mode="skip", skip_attn=(1,), skip_mlp=(2,), d_max=5, tau=None), 10.0),
    (SMALL_GQA, Policy(mode="skip", skip_mlp=(2, 3), d_max=6, tau=None), 10.0),
    (WIDE, Policy(mode="exit", exit_layer=0, d_max=10, tau=None), 1.0),
])
def test_rounds_match_oracle_in_lockstep(ssd, w, pol, head):
    # Tolerances: logits within 5e-2 and confidences within 1e-3 with the
    # workloads' own LM head (head = 1).  GPU and oracle differ where a
    # bf16-rounded activation lands on the other side of a rounding boundary;
    # an LM head sharpened by `head` multiplies that logit deviation by
    # `head` (measured: 0.003-0.006 at head 1, 0.03-0.06 at head 10), and
    # conf = exp(z1 - lse) moves by at most 2 conf max|dz|, so both
    # tolerances are multiplied by `head` for the sharpened parity models.
    from oracle import OracleModel, prefill, ssd_round
    ctx, wts = _ctx(ssd, w, lm_head_scale=head)
    ctx.set_policy(pol)
    m = OracleModel(w.shape, weights_to_numpy(wts))
    prompt = oracle_prompt(m, w, pol, lambda p, st: not _near_tie(st.last_logits))
    first = ctx.prefill(prompt)
    st = prefill(m, prompt, pol, 256)
    assert first == st.tokens[-1]
    _lockstep(ctx, m, st, pol, head, min_rounds=1 if head == 1.0 else 3)
    ctx.close()


# Model with the workloads' own LM head (no sharpening) whose small vocabulary
# and d_model 1024 give top-1/top-2 logit gaps well above the GPU-oracle
# deviation (0.003-0.006 at this head), so that rounds can be compared at the
# stated tolerances themselves.
MID_V64 = Workload(name="mid-v64", shape=ModelShape(
    n_layers=4, d_model=1024, n_heads=8, n_kv_heads=4, head_dim=128, ffn_dim=2816, vocab=64),
    scaled_layers=(1, 2), scale=0.1)


@pytest.mark.parametrize("pol", [
    Policy(mode="skip", skip=(1, 2), d_max=3, tau=None),
    Policy(mode="exit", exit_layer=0, d_max=4, tau=None),
    Policy(mode="skip", skip=(2,), d_max=3, tau=0.05),
], ids=["skip", "exit", "skip-tau"])
def test_rounds_match_oracle_at_stated_tolerances(ssd, pol):
    # logits within 5e-2 and confidences within 1e-3 (no sharpening factor)
    # over at least three rounds.  The prompt is the first seeded prompt whose
    # oracle rounds 1-3 decide every token with a top-1/top-2 gap above 0.02
    # and every confidence stop more than 2e-3 from tau: chosen on the
    # oracle's values alone.
    from oracle import OracleModel, prefill, ssd_round
    w = MID_V64
    ctx, wts = _ctx(ssd, w, lm_head_scale=1.0)
    ctx.set_policy(pol)
    m = OracleModel(w.shape, weights_to_numpy(wts))

    def clean(prompt, st):
        if top_gap(st.last_logits) <= 0.02:
            return False
        for _ in range(3):
            rec = ssd_round(m, st, pol)
            confs = rec.conf + ([rec.stop_conf] if rec.stop_conf is not None else [])
            if any(top_gap(z) <= 0.02 for z in rec.draft_logits):
                return False
            if any(top_gap(z) <= 0.02 for z in rec.verify_logits[: rec.accepted + 1]):
                return False
            if pol.tau is not None and any(abs(c - pol.tau) <= 2e-3 for c in confs):
                return False
        return True

    prompt = oracle_prompt(m, w, pol, clean)
    first = ctx.prefill(prompt)
    st = prefill(m, prompt, pol, 256)
    assert first == st.tokens[-1]
    _lockstep(ctx, m, st, pol, 1.0, min_rounds=3)
    ctx.close()


def _lockstep(ctx, m, st, pol, head, min_rounds, max_rounds=12, logit_tol=5e-2, tie=0.1,
              dev=None):
    """Greedy rounds in lockstep with the oracle until the first divergence
    at a near tie (top-1/top-2 gap <= tie, or a tau crossing); returns the
    rounds compared.  dev (list, optional) collects each compared round's
    largest verify-logit deviation."""
    from oracle import ssd_round
    conf_tol = 1e-3 * head

    def _near(z):
        return _near_tie(z, tie)

    rounds = 0
    checked = 0
    for _ in range(max_rounds):
        drafts, confs = ctx.draft()
        vlog = ctx.verify(d=len(drafts))
        emitted = ctx.accept()
        rec = ssd_round(m, st, pol)
        # confidences of every draft step run (the stopping one included),
        # up to the first step whose draft token differs (later steps see
        # different inputs)
        ref_conf = rec.conf + ([rec.stop_conf] if rec.stop_conf is not None else [])
        j = next(i for i in range(min(len(drafts), len(rec.draft)) + 1)
                 if i >= len(drafts) or i >= len(rec.draft) or drafts[i] != rec.draft[i])
        for a, b in list(zip(confs, ref_conf))[: j + 1]:
            assert abs(a - b) <= conf_tol
            checked += 1
        if drafts != rec.draft:
            # a divergence is only allowed at a near-tie or a tau crossing
            justified = (j < len(rec.draft_logits) and _near(rec.draft_logits[j])) or (
                pol.tau is not None and j < len(ref_conf) and abs(ref_conf[j] - pol.tau) <= conf_tol)
            assert justified, f"drafts diverge at step {j} without a near-tie"
            break
        dz = float(np.max(np.abs(vlog - rec.verify_logits)))
        if dev is not None:
            dev.append(dz)
        assert dz <= logit_tol * head
        if emitted != rec.emitted:
            j = next(i for i in range(len(emitted) + 1)
                     if i >= len(emitted) or i >= len(rec.emitted) or emitted[i] != rec.emitted[i])
            assert _near(rec.verify_logits[min(j, len(rec.verify_logits) - 1)]), \
                f"emitted tokens diverge at {j} without a near-tie"
            break
        rounds += 1
    assert checked >= 1
    assert rounds >= min_rounds, rounds
    return rounds


@pytest.mark.parametrize("w,pol,head", [
    (SMALL_GQA, Policy(mode="exit", exit_layer=1, d_max=6, temperature=0.6, seed=1234), 4.0),
    (TINY, Policy(mode="skip", skip=(1, 2), d_max=4, temperature=0.6, seed=99), 4.0),
])
def test_sampled_rounds_match_oracle_in_lockstep(ssd, w, pol, head):
    # T > 0: both sides draw the same Philox numbers, so drafts, acceptance
    # decisions and emitted tokens agree wherever the decision is not within
    # the tolerance of its boundary (Gumbel score gap > 0.1, |log u - log(p/q)|
    # > 0.05); the first legitimate divergence ends the comparison.
    from oracle import OracleModel, prefill
    ctx, wts = _ctx(ssd, w, lm_head_scale=head)
    ctx.set_policy(pol)
    m = OracleModel(w.shape, weights_to_numpy(wts))
    T, seed = pol.temperature, pol.seed

    # the prefill's token is drawn like an AR step: round 0, stream 2, position P
    prompt = oracle_prompt(
        m, w, pol, lambda p, st: _gumbel_gap(st.last_logits, T, seed, len(p), 0, 2) > 0.1)
    first = ctx.prefill(prompt)
    st = prefill(m, prompt, pol, 256)
    assert first == st.tokens[-1]

    assert _sampled_lockstep(ctx, m, st, pol, head, max_rounds=16) >= 2
    ctx.close()


def _gumbel_gap(z, T, seed, pos, rnd, stream):
    from oracle.philox import uniforms
    sc = np.sort(z / T - np.log(-np.log(uniforms(seed, pos, rnd, stream, z.shape[0]))))
    return sc[-1] - sc[-2]


def _sampled_lockstep(ctx, m, st, pol, head, max_rounds, logit_tol=5e-2, tie=0.1,
                      margin=0.05, dev=None):
    """Rounds at T > 0 in lockstep with the oracle until the first decision
    within the tolerance of its boundary (Gumbel-score gap <= tie,
    |log u - log(p/q)| <= margin); returns the rounds compared."""
    from oracle import ssd_round
    from oracle import ops as O
    T, seed = pol.temperature, pol.seed
    V = m.s.vocab
    rounds = 0
    for _ in range(max_rounds):
        n, rnd = st.n, st.round + 1
        drafts, _ = ctx.draft()
        vlog = ctx.verify(d=len(drafts))
        emitted = ctx.accept()
        rec = ssd_round(m, st, pol)
        if drafts != rec.draft:
            j = next(i for i in range(len(rec.draft)) if drafts[i] != rec.draft[i])
            assert _gumbel_gap(rec.draft_logits[j], T, seed, n + j, rnd, 0) <= tie, \
                "draft sample differs"
            break
        dz = float(np.max(np.abs(vlog - rec.verify_logits)))
        if dev is not None:
            dev.append(dz)
        assert dz <= logit_tol * head
        Q = np.stack(rec.draft_logits) if rec.draft else np.zeros((0, V))
        margins = O.accept_margins(rec.verify_logits, Q, rec.draft, T, seed, rnd, n)
        k = 0
        while k < min(len(margins), rec.accepted + 1) and margins[k] > margin:
            k += 1
        if k <= rec.accepted and k < len(margins):
            break        # a decision within tolerance of its boundary
        if O.resample_gap(rec.verify_logits, Q, rec.accepted, T, seed, rnd, n) <= tie:
            break
        assert emitted == rec.emitted
        rounds += 1
    return rounds


def test_sublayer_masks_are_validated(ssd):
    from self_speculative_decoding_gb300 import SSDError
    ctx, _ = _ctx(ssd, TINY)
    with pytest.raises(SSDError, match="INVALID_ARG"):
        ctx.set_policy(Policy(mode="skip", skip_mlp=(7,), d_max=2))       # layer >= n_layers
    with pytest.raises(SSDError, match="INVALID_ARG"):
        ctx.set_policy(Policy(mode="exit", exit_layer=1, skip_attn=(0,), d_max=2))
    ctx.close()


def test_state_and_capacity_errors(ssd):
    from self_speculative_decoding_gb300 import SSDError
    w = TINY
    ctx, _ = _ctx(ssd, w, max_seq=64)
    with pytest.raises(SSDError, match="STATE"):
        ctx.prefill([1, 2, 3])                      # no policy yet
    with pytest.raises(SSDError, match="CAPACITY"):
        ctx.set_policy(Policy(mode="skip", skip=(2,), d_max=16))
    with pytest.raises(SSDError, match="INVALID_ARG"):
        ctx.set_policy(Policy(mode="exit", exit_layer=9, d_max=4))
    ctx.set_policy(Policy(mode="skip", skip=(2,), d_max=4))
    with pytest.raises(SSDError, match="CAPACITY"):
        ctx.prefill(list(range(64)))
    with pytest.raises(SSDError, match="INVALID_ARG"):
        ctx.prefill([5000])
    ctx.prefill(list(range(10)))
    with pytest.raises(SSDError, match="STATE"):
        ctx.verify()
    with pytest.raises(SSDError, match="STATE"):
        ctx.accept()
    ctx.draft()
    with pytest.raises(SSDError, match="STATE"):
        ctx.draft()
    ctx.verify(want_logits=False)
    ctx.accept()
    with pytest.raises(SSDError, match="CAPACITY"):
        ctx.generate(60)
    ctx.close()


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_sampled_generation_follows_target_distribution(ssd, T):
    # exit-mode drafting at temperature T on a tiny vocabulary: the first
    # emitted token of a round follows the full model's softmax(z / T)
    # (chi-square).
    from scipy.stats import chisquare
    from oracle import OracleModel, prefill
    from oracle.model import softmax
    w = Workload(name="tiny-v16", shape=ModelShape(n_layers=2, d_model=64, n_heads=1,
                 n_kv_heads=1, head_dim=64, ffn_dim=128, vocab=16))
    wts = make_weights(w, dtype="bf16", lm_head_scale=4.0, random_gains=True)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=64)
    prompt = make_prompt(w, 6)
    m = OracleModel(w.shape, weights_to_numpy(wts))
    p = softmax(prefill(m, prompt, Policy(), 64).last_logits / T)   # target after the prompt
    ctx.set_policy(Policy(mode="exit", exit_layer=0, d_max=3, temperature=T, seed=7))
    ctx.prefill(prompt)
    counts = np.zeros(16)
    n = 3000
    for _ in range(n):
        ctx.rewind(len(prompt))        # prompt[-1] pending again; the round counter moves on
        ctx.draft()
        ctx.verify(want_logits=False)
        counts[ctx.accept()[0]] += 1
    keep = p * n >= 5
    assert keep.sum() >= 4                  # a spread target distribution
    exp = np.append(p[keep] * n, p[~keep].sum() * n)
    obs = np.append(counts[keep], counts[~keep].sum())
    if exp[-1] == 0.0:
        exp, obs = exp[:-1], obs[:-1]
    assert chisquare(obs, exp).pvalue > 1e-3
    ctx.close()


@pytest.mark.parametrize("literal_tau", [False, True])
def test_llama7b_shape_ssd_equals_ar(ssd, literal_tau):
    # the bench workload's shape and skip set, shortened: bit-identity at full size
    from synthetic import LLAMA7B_SWIFT
    w = LLAMA7B_SWIFT
    pol = w.policy if literal_tau else replace(w.policy, tau=None)
    wts = ssd.pack_weights(make_weights(w, device="cuda"), release=True)
    ctx = ssd.SSDContext(w.shape, wts, max_seq=512)
    ctx.set_policy(pol)
    prompt = make_prompt(w, 128)
    f1 = ctx.prefill(prompt)
    ar, _ = ctx.decode_ar(48)
    f2 = ctx.prefill(prompt)
    toks, stats = ctx.generate(48)
    assert f1 == f2 and toks == ar
    if not literal_tau:
        assert stats["drafted"] > 0
    # a second generation from the same prompt repeats the first
    assert ctx.prefill(prompt) == f1
    toks2, _ = ctx.generate(48)
    assert toks2 == toks
    ctx.close()
    del wts
    torch.cuda.empty_cache()
