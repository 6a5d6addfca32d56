"""Draft / verify / accept, step by step (test infrastructure).

Follows the pages' loop: the LayerSkip blog §3.1 (draft_phase: token by
token through the draft layers, shared LM head on the last hidden state),
§3.2 (verify_phase: the full model over d+1 positions, reusing the draft's
KV for the layers it shares with the full model), §3.3 (layerskip_ssd:
accept with min(1, p/q), resample from norm(max(0, p - q)) on the first
rejection, sample a bonus token when every draft is accepted; each verify
yields between 1 and d+1 tokens), and SWIFT §4.2 (drafting halts when the
top-1 confidence falls below a threshold).

Readings where the pages are silent or garbled (each one is listed with its
reason in the design notes):

* State: ``tokens`` t[0..n-1] are committed; the last one, x = t[n-1], is
  pending (not yet run through the full model); K/V at positions < n-1 hold
  full-model values in every layer.  The pseudocode's rebuilt-from-scratch
  KV (draft_phase resets its cache each step) is read as the incremental
  cache its own comment describes.
* Draft step j feeds x (j = 0) or y_{j-1} at position n-1+j through the
  layers below s0 (the first layer the verify recomputes: min of the skip
  set, or E+1), saves that hidden state as the step's boundary state, runs
  the remaining draft layers, and applies the final norm + LM head.
  conf_j = max softmax(z_j) at temperature 1.  If conf_j < tau, y_j is not
  kept and drafting stops.  At temperature 0, y_j = argmax z_j; at T > 0,
  y_j is sampled from q_j = softmax(z_j / T) (an argmax draft with the
  min(1, p/q) rule, as the blog's pseudocode writes it, would not preserve
  the target distribution).
* In skip mode the draft's kept layers above s0 write their (draft) K/V for
  the draft positions; the verify overwrites every position it runs in every
  layer >= s0.  Skipped layers write nothing.  A policy may also drop only the
  attention or only the MLP sublayer of a layer (SWIFT Fig. 10 treats them
  separately): the dropped sublayer's residual branch is left out, and a
  layer whose attention does not run writes no K/V; s0 is then the first
  layer with any dropped sublayer.
* Verify: when the draft filled d_max without feeding y_{d-1}, that token is
  first run through layers 0..s0-1 at position n-1+d.  Then the d+1 boundary
  states (positions n-1..n-1+d) run through layers s0..L-1 and the LM head.
  (The blog takes "the hidden state of layer E" from its KV dictionary; the
  hidden state per position is what the verify needs.)
* Accept: greedy keeps the longest prefix with y_j == argmax p_j and emits
  argmax p_a after it.  Stochastic acceptance uses p = softmax(z_full / T)
  and q = softmax(z_draft / T).  The context grows by the emitted tokens and
  the committed length becomes n + a + 1 (the blog's context update line is
  garbled); K/V beyond the new pending position is stale and is overwritten
  before it is read, which is the rollback.
* Dynamic verification (SWIFT §4.2 and §3.2.1: the draft's confidence also
  sets how many candidates go to the verify; top-k drafts raise the accepted
  length).  Read for greedy decoding as one-level siblings off the drafted
  chain: a kept draft y_j whose confidence is below ``tree_tau`` also sends
  the draft's second choice s_j (at most ``tree_max`` per round, in depth
  order).  The verify computes, besides the chain rows, the full model's
  logits for each sibling at its position n + j given the accepted-so-far
  prefix (tokens before n + j) -- one full-model step on a fork of the
  cache.  Acceptance walks the chain; at the first rejected depth a, when a
  sibling at depth a is the full model's token there, the sibling is taken
  and the full model's token after it is emitted as well, and the cache
  becomes that sibling's fork.  The emitted sequence stays the greedy one.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, List, Optional, Tuple

import numpy as np

from .model import OracleModel, KVCache, softmax, logsumexp, top2
from .philox import (gumbel_argmax, uniform, STREAM_DRAFT, STREAM_ACCEPT,
                     STREAM_RESAMPLE)


@dataclass
class SSDState:
    tokens: List[int]
    kv: KVCache
    round: int = 0

    @property
    def n(self) -> int:
        return len(self.tokens)


@dataclass
class RoundRecord:
    n_before: int
    draft: List[int]
    conf: List[float]
    stop_conf: Optional[float]
    draft_logits: List[np.ndarray]
    verify_logits: np.ndarray
    accepted: int
    emitted: List[int]
    extra_pass: bool = False
    siblings: List[Tuple[int, int]] = field(default_factory=list)   # (depth j, token)
    sibling_logits: List[np.ndarray] = field(default_factory=list)
    sibling_taken: Optional[int] = None

    @property
    def d(self) -> int:
        return len(self.draft)


def _pick(z: np.ndarray, T: float, seed: int, pos: int, rnd: int, stream: int) -> int:
    if T == 0.0:
        return int(np.argmax(z))
    return gumbel_argmax(z / T, seed, pos, rnd, stream)


def prefill(model: OracleModel, prompt, policy, max_seq: int) -> SSDState:
    """Run the prompt through the full model; the first new token is committed
    and pending.  (Decoding round 0 is the prefill's.)"""
    kv = model.new_cache(max_seq)
    P = len(prompt)
    X = model.embed_rows(prompt)
    X = model.run_layers(X, range(P), kv, range(model.s.n_layers))
    z = model.lm_head(X[-1:])[0]
    first = _pick(z, policy.temperature, policy.seed, P, 0, STREAM_RESAMPLE)
    st = SSDState(tokens=[int(t) for t in prompt] + [first], kv=kv, round=0)
    st.last_logits = z
    return st


def ar_step(model: OracleModel, st: SSDState, policy) -> np.ndarray:
    """One autoregressive step: the pending token through every layer."""
    st.round += 1
    n = st.n
    X = model.embed_rows([st.tokens[-1]])
    X = model.run_layers(X, [n - 1], st.kv, range(model.s.n_layers))
    z = model.lm_head(X)[0]
    st.tokens.append(_pick(z, policy.temperature, policy.seed, n, st.round, STREAM_RESAMPLE))
    return z


def ar_generate(model: OracleModel, st: SSDState, policy, n_new: int) -> List[np.ndarray]:
    return [ar_step(model, st, policy) for _ in range(n_new)]


def acceptance_ratio(p: np.ndarray, q: np.ndarray, y: int) -> float:
    """min(1, p(y) / q(y)) (LayerSkip blog §3.3)."""
    return min(1.0, p[y] / q[y])


def residual_distribution(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """norm(max(0, p - q)); if p <= q everywhere the residual is empty and p is used."""
    w = np.maximum(p - q, 0.0)
    s = np.sum(w)
    return p.copy() if s == 0.0 else w / s


def accept_stochastic(P: np.ndarray, Q: List[np.ndarray], ys: List[int], T: float,
                      draw_u: Callable[[int], float],
                      draw_tok: Callable[[int, np.ndarray], int]):
    """The min(1, p/q) rule over the drafts in order (LayerSkip blog §3.3).

    ``P``: verify logits [d+1, V]; ``Q``: draft logits per draft token.
    ``draw_u(j)`` gives the uniform for draft j; ``draw_tok(j, logw)`` samples
    from weights exp(logw).  Returns (accepted count a, emitted tokens).
    """
    d = len(ys)
    for j in range(d):
        p = softmax(P[j] / T)
        q = softmax(Q[j] / T)
        y = ys[j]
        if draw_u(j) < p[y] / q[y]:
            continue
        w = np.maximum(p - q, 0.0)
        with np.errstate(divide="ignore"):
            logw = np.log(w) if np.any(w > 0.0) else np.log(p)
        return j, list(ys[:j]) + [draw_tok(j, logw)]
    return d, list(ys) + [draw_tok(d, P[d] / T)]


def sibling_step(model: OracleModel, kv: KVCache, pos: int, tok: int):
    """A sibling candidate's verify row: one full-model step of ``tok`` at
    ``pos`` on a fork of ``kv`` (which holds the full-model K/V of the
    tokens before ``pos``).  Returns (logits, fork)."""
    kv_s = kv.fork()
    X = model.run_layers(model.embed_rows([tok]), [pos], kv_s, range(model.s.n_layers))
    return model.lm_head(X)[0], kv_s


def ssd_round(model: OracleModel, st: SSDState, policy) -> RoundRecord:
    s = model.s
    L = s.n_layers
    T, seed = policy.temperature, policy.seed
    st.round += 1
    rnd = st.round
    n = st.n
    x = st.tokens[-1]
    s0 = policy.first_recomputed(L)
    post = [l for l in policy.draft_layers(L) if l >= s0]

    tree_tau = getattr(policy, "tree_tau", None)
    tree = tree_tau is not None and tree_tau > 0.0 and T == 0.0 and policy.tree_max > 0
    sibs: List[Tuple[int, int]] = []
    ys: List[int] = []
    confs: List[float] = []
    zs: List[np.ndarray] = []
    bnd: List[np.ndarray] = []
    stop_conf = None
    for j in range(policy.d_max):
        tok = x if j == 0 else ys[-1]
        pos = n - 1 + j
        X = model.embed_rows([tok])
        X = model.run_layers(X, [pos], st.kv, range(s0))
        bnd.append(X[0].copy())
        X = model.run_layers(X, [pos], st.kv, post,
                             parts=policy.sublayers if policy.mode == "skip" else None)
        z = model.lm_head(X)[0]
        conf = float(np.exp(np.max(z) - logsumexp(z)))
        y = _pick(z, T, seed, pos + 1, rnd, STREAM_DRAFT)
        if policy.tau is not None and conf < policy.tau:
            stop_conf = conf
            break
        ys.append(y)
        confs.append(conf)
        zs.append(z)
        if tree and conf < tree_tau and len(sibs) < policy.tree_max:
            sibs.append((j, top2(z)[2]))
    d = len(ys)
    extra = False
    if len(bnd) == d:
        # the last kept draft token was never fed: run it below s0
        tok = ys[-1] if d > 0 else x
        X = model.embed_rows([tok])
        X = model.run_layers(X, [n - 1 + d], st.kv, range(s0))
        bnd.append(X[0].copy())
        extra = True

    Xv = model.run_layers(np.stack(bnd), range(n - 1, n + d), st.kv, range(s0, L))
    P = model.lm_head(Xv)
    forks, sib_logits = [], []
    for j, s_tok in sibs:
        z_s, kv_s = sibling_step(model, st.kv, n + j, s_tok)
        forks.append(kv_s)
        sib_logits.append(z_s)
    taken = None

    if T == 0.0:
        a = 0
        while a < d and ys[a] == int(np.argmax(P[a])):
            a += 1
        t = int(np.argmax(P[a]))
        emitted = ys[:a] + [t]
        for i, (j, s_tok) in enumerate(sibs):
            if a < d and j == a and s_tok == t:
                taken = i
        if taken is not None:
            emitted.append(int(np.argmax(sib_logits[taken])))
            st.kv = forks[taken]
    else:
        a, emitted = accept_stochastic(
            P, zs, ys, T,
            draw_u=lambda j: uniform(seed, n + j, rnd, STREAM_ACCEPT),
            draw_tok=lambda j, logw: gumbel_argmax(logw, seed, n + j, rnd, STREAM_RESAMPLE))
    st.tokens.extend(int(t) for t in emitted)
    return RoundRecord(n_before=n, draft=ys, conf=confs, stop_conf=stop_conf,
                       draft_logits=zs, verify_logits=P, accepted=a, emitted=emitted,
                       extra_pass=extra, siblings=sibs, sibling_logits=sib_logits,
                       sibling_taken=taken)


@dataclass
class GenStats:
    rounds: int = 0
    drafted: int = 0
    accepted: int = 0
    emitted: int = 0
    side_rows: int = 0       # dynamic verification: siblings verified
    side_accepted: int = 0   # rounds that took a sibling
    records: List[RoundRecord] = field(default_factory=list)

    @property
    def mean_accepted_length(self) -> float:
        """M: tokens the full model emits per verify (SWIFT B.3)."""
        return self.emitted / max(self.rounds, 1)

    @property
    def alpha(self) -> float:
        """alpha: fraction of draft tokens accepted (SWIFT B.3)."""
        return self.accepted / max(self.drafted, 1)


def ssd_generate(model: OracleModel, st: SSDState, policy, n_new: int) -> GenStats:
    """Rounds until n_new tokens are emitted; extra tokens of the last round are dropped."""
    target = st.n + n_new
    stats = GenStats()
    while st.n < target:
        r = ssd_round(model, st, policy)
        stats.rounds += 1
        stats.drafted += r.d
        stats.accepted += r.accepted
        stats.emitted += len(r.emitted)
        stats.side_rows += len(r.siblings)
        stats.side_accepted += r.sibling_taken is not None
        stats.records.append(r)
    del st.tokens[target:]
    return stats
