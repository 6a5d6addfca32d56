// Device bodies of the pass set-up and draft-control steps, run by their
// single-CTA kernels (control.cu).  Data written by the preceding kernels (row
// summaries, the residual stream) is read through L2 (ld.global.cg).
#pragma once

#include "kernels.cuh"

namespace ssd {
namespace ctl {

// Embedding (or boundary copy) of the pass's rows, with the sum-of-squares
// partials of every 16-column group (the same order the projection
// epilogues use: ascending columns from zero).  Threads tid < nthr of one
// CTA; s_M (two ints) / s_tok are shared scratch; sync() is their barrier.
template <class Sync>
SSD_DI void begin(const BeginArgs& a, int tid, int nthr, int* s_M, int* s_tok, Sync sync) {
  DevState* st = a.st;
  if (tid == 0) {
    int M = 1, pos0 = 0, slot = 0, ns = 0, side0 = 0;
    switch (a.mode) {
      case BEGIN_TOKENS:
        M = a.M;
        pos0 = a.pos0;
        for (int m = 0; m < M; ++m) s_tok[m] = a.toks_in[m];
        if (a.reset_round) {
          st->round = 0;
          st->j = st->d = st->stop = 0;
          st->n_sib = 0;
        }
        break;
      case BEGIN_AR:
        st->round += 1;
        pos0 = st->n - 1;
        s_tok[0] = a.tokens[st->n - 1];
        break;
      case BEGIN_DRAFT:
      case BEGIN_EXTRA: {
        // draft step j feeds y_{j-1} (the pending token at j = 0); the extra
        // pass feeds y_{d-1}.  A sibling recorded for that draft rides along
        // as a side row at the same position.
        int fed;
        if (a.mode == BEGIN_DRAFT) {
          if (st->j == 0) {
            st->round += 1;
            st->n_sib = 0;
          }
          fed = st->j - 1;
          slot = st->j;
        } else {
          fed = st->d - 1;
        }
        pos0 = st->n + fed;
        s_tok[0] = fed < 0 ? a.tokens[st->n - 1] : st->draft_tok[fed];
        const int k = st->n_sib - 1;
        if (fed >= 0 && k >= 0 && st->sib_depth[k] == fed) {
          M = 2;
          ns = 1;
          side0 = k;
          s_tok[1] = st->sib_tok[k];
          st->side_pos[0] = pos0;
        }
        break;
      }
      case BEGIN_VERIFY:
        // chain rows n-1 .. n-1+d, then every sibling at its own position
        ns = st->n_sib;
        M = st->d + 1 + ns;
        pos0 = st->n - 1;
        for (int i = 0; i < ns; ++i) st->side_pos[i] = st->n + st->sib_depth[i];
        break;
    }
    if (!SSD_CHECK(st, M >= 1 && M <= kMaxRows, DBG_ROWS, M)) M = 1;
    if (!SSD_CHECK(st, pos0 >= 0 && pos0 + M <= st->max_seq, DBG_POS, pos0 + M)) pos0 = 0;
    for (int m = 0; m < M && a.mode != BEGIN_VERIFY; ++m)
      if (!SSD_CHECK(st, s_tok[m] >= 0 && s_tok[m] < st->vocab, DBG_TOKEN, s_tok[m])) s_tok[m] = 0;
    st->M = M;
    st->pos0 = pos0;
    st->slot = slot;
    st->ns = ns;
    st->side0 = side0;
    if (a.mode != BEGIN_VERIFY)
      for (int m = 0; m < M; ++m) st->in_tok[m] = s_tok[m];
    s_M[0] = M;
    s_M[1] = ns;
  }
  sync();
  const int M = s_M[0], D = a.D, NP = D / kSsGroup;
  if (a.mode == BEGIN_VERIFY) {
    const int mc = M - s_M[1];
    for (int e = tid; e < mc * D; e += nthr) a.x[e] = __ldcg(a.bx + e);
    for (int e = tid; e < mc * NP; e += nthr) a.ss[e] = __ldcg(a.bss + e);
    for (int e = tid; e < (M - mc) * D; e += nthr) a.x[mc * D + e] = __ldcg(a.bxs + e);
    for (int e = tid; e < (M - mc) * NP; e += nthr) a.ss[mc * NP + e] = __ldcg(a.bsss + e);
    return;
  }
  for (int e = tid; e < M * NP; e += nthr) {
    const int m = e / NP, grp = e % NP;
    const size_t off = (size_t)s_tok[m] * D + grp * kSsGroup;
    float* dst = a.x + (size_t)m * D + grp * kSsGroup;
    float s = 0.f;
    for (int i = 0; i < kSsGroup; ++i) {
      const float v = a.embed32 ? a.embed32[off + i] : __bfloat162float(a.embed[off + i]);
      dst[i] = v;
      s += v * v;
    }
    a.ss[(size_t)m * NP + grp] = s;
  }
}

// Copy row 0 of the residual (and its partials) into boundary slot j (draft
// step) or d (extra pass), and a side row into the siblings' boundary slot
// of its sibling index; the rest of the pass runs the chain row alone.
template <class Sync>
SSD_DI void save_boundary(const SaveArgs& a, int tid, int nthr, Sync sync) {
  DevState* st = a.st;
  const int slot = a.use_d ? __ldcg(&st->d) : __ldcg(&st->j);
  const int ns = __ldcg(&st->ns), side0 = __ldcg(&st->side0);
  const int D = a.D, NP = D / kSsGroup;
  for (int e = tid; e < D; e += nthr) a.bx[(size_t)slot * D + e] = __ldcg(a.x + e);
  for (int e = tid; e < NP; e += nthr) a.bss[(size_t)slot * NP + e] = __ldcg(a.ss + e);
  if (ns > 0) {
    for (int e = tid; e < D; e += nthr) a.bxs[(size_t)side0 * D + e] = __ldcg(a.x + D + e);
    for (int e = tid; e < NP; e += nthr) a.bsss[(size_t)side0 * NP + e] = __ldcg(a.ss + NP + e);
  }
  sync();  // every thread has read ns before it is cleared
  if (tid == 0 && ns > 0) {
    st->M = 1;
    st->ns = 0;
  }
}

SSD_DI RowStats load_stats(const RowStats* p) {
  const int4 a = __ldcg(reinterpret_cast<const int4*>(p));
  const float4 b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
  const float4 c = __ldcg(reinterpret_cast<const float4*>(p) + 2);
  RowStats r;
  r.top1 = a.x; r.top2 = a.y; r.sample = a.z; r.pad = a.w;
  r.z1 = b.x; r.z2 = b.y; r.lse = b.z; r.conf = b.w;
  r.lse_t = c.x; r.pad2[0] = c.y; r.pad2[1] = c.z; r.pad2[2] = c.w;
  return r;
}

// SWIFT §4.2 confidence-aware stop: the draft token of step j is kept only
// if its top-1 probability reaches tau.  Dynamic verification (greedy): a
// kept draft whose top-1 probability is below tree_tau also gets the
// draft's second choice as a sibling candidate, up to tree_max per round.
// One thread.
SSD_DI void draft_end(const DraftEndArgs& a) {
  DevState* st = a.st;
  const int j = st->j;
  const RowStats rs = load_stats(a.dstats + j);
  st->draft_conf[j] = rs.conf;
  if (rs.conf < a.tau) {
    st->stop = 1;
  } else {
    st->draft_tok[j] = a.temperature > 0.f ? rs.sample : rs.top1;
    st->d = j + 1;
    const int k = st->n_sib;
    if (rs.conf < a.tree_tau && k < a.tree_max) {
      st->sib_depth[k] = j;
      st->sib_tok[k] = rs.top2;
      st->n_sib = k + 1;
    }
  }
  st->j = j + 1;
}

// Commit the token the full model produced for the last row of the pass.
// One thread.
SSD_DI void ar_end(DevState* st, int32_t* tokens, const RowStats* vstats, int row_from_M, float T,
                   int reset) {
  const int row = row_from_M ? st->M - 1 : 0;
  const RowStats rs = load_stats(vstats + row);
  int tok = T > 0.f ? rs.sample : rs.top1;
  const int n = reset ? st->pos0 + st->M : st->n;
  if (!SSD_CHECK(st, tok >= 0 && tok < st->vocab, DBG_TOKEN, tok)) tok = 0;
  if (!SSD_CHECK(st, n >= 0 && n < st->max_seq, DBG_COMMIT, n)) return;
  tokens[n] = tok;
  st->n = n + 1;
  st->emitted[0] = tok;
  st->n_emitted = 1;
  if (reset) st->j = st->d = st->stop = 0;
}

}  // namespace ctl
}  // namespace ssd
