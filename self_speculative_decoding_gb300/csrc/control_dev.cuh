// Device bodies of the pass set-up and draft-control steps, shared by their
// single-CTA kernels (control.cu) and by the persistent pass kernel
// (pass.cu).  Data written by other CTAs earlier in the same kernel (row
// summaries, the residual stream) is read through L2 (ld.global.cg).
#pragma once

#include "kernels.cuh"

namespace ssd {
namespace ctl {

// Embedding (or boundary copy) of the pass's rows, with the sum-of-squares
// partials of every 16-column group (the same order the projection
// epilogues use: ascending columns from zero).  Threads tid < nthr of one
// CTA; s_M / s_tok are shared scratch; sync() is their barrier.
template <class Sync>
SSD_DI void begin(const BeginArgs& a, int tid, int nthr, int* s_M, int* s_tok, Sync sync) {
  DevState* st = a.st;
  if (tid == 0) {
    int M = 1, pos0 = 0, slot = 0;
    switch (a.mode) {
      case BEGIN_TOKENS:
        M = a.M;
        pos0 = a.pos0;
        for (int m = 0; m < M; ++m) s_tok[m] = a.toks_in[m];
        if (a.reset_round) {
          st->round = 0;
          st->j = st->d = st->stop = 0;
        }
        break;
      case BEGIN_AR:
        st->round += 1;
        pos0 = st->n - 1;
        s_tok[0] = a.tokens[st->n - 1];
        break;
      case BEGIN_DRAFT:
        if (st->j == 0) st->round += 1;
        pos0 = st->n - 1 + st->j;
        s_tok[0] = st->j == 0 ? a.tokens[st->n - 1] : st->draft_tok[st->j - 1];
        slot = st->j;
        break;
      case BEGIN_EXTRA:
        pos0 = st->n - 1 + st->d;
        s_tok[0] = st->d > 0 ? st->draft_tok[st->d - 1] : a.tokens[st->n - 1];
        break;
      case BEGIN_VERIFY:
        M = st->d + 1;
        pos0 = st->n - 1;
        break;
    }
    st->M = M;
    st->pos0 = pos0;
    st->slot = slot;
    if (a.mode != BEGIN_VERIFY)
      for (int m = 0; m < M; ++m) st->in_tok[m] = s_tok[m];
    *s_M = M;
  }
  sync();
  const int M = *s_M, D = a.D, NP = D / kSsGroup;
  if (a.mode == BEGIN_VERIFY) {
    for (int e = tid; e < M * D; e += nthr) a.x[e] = __ldcg(a.bx + e);
    for (int e = tid; e < M * NP; e += nthr) a.ss[e] = __ldcg(a.bss + e);
    return;
  }
  for (int e = tid; e < M * NP; e += nthr) {
    const int m = e / NP, grp = e % NP;
    const bf16* src = a.embed + (size_t)s_tok[m] * D + grp * kSsGroup;
    float* dst = a.x + (size_t)m * D + grp * kSsGroup;
    float s = 0.f;
    for (int i = 0; i < kSsGroup; ++i) {
      const float v = __bfloat162float(src[i]);
      dst[i] = v;
      s += v * v;
    }
    a.ss[(size_t)m * NP + grp] = s;
  }
}

// Copy row 0 of the residual (and its partials) into boundary slot j
// (draft step) or d (extra pass).
SSD_DI void save_boundary(DevState* st, int use_d, const float* x, const float* ss, float* bx,
                          float* bss, int D, int tid, int nthr) {
  const int slot = use_d ? st->d : st->j;
  const int NP = D / kSsGroup;
  for (int e = tid; e < D; e += nthr) bx[(size_t)slot * D + e] = __ldcg(x + e);
  for (int e = tid; e < NP; e += nthr) bss[(size_t)slot * NP + e] = __ldcg(ss + e);
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
// if its top-1 probability reaches tau.  One thread.
SSD_DI void draft_end(DevState* st, const RowStats* dstats, float tau, float T) {
  const int j = st->j;
  const RowStats rs = load_stats(dstats + j);
  st->draft_conf[j] = rs.conf;
  if (rs.conf < tau) {
    st->stop = 1;
  } else {
    st->draft_tok[j] = T > 0.f ? rs.sample : rs.top1;
    st->d = j + 1;
  }
  st->j = j + 1;
}

// Commit the token the full model produced for the last row of the pass.
// One thread.
SSD_DI void ar_end(DevState* st, int32_t* tokens, const RowStats* vstats, int row_from_M, float T,
                   int reset) {
  const int row = row_from_M ? st->M - 1 : 0;
  const RowStats rs = load_stats(vstats + row);
  const int tok = T > 0.f ? rs.sample : rs.top1;
  const int n = reset ? st->pos0 + st->M : st->n;
  tokens[n] = tok;
  st->n = n + 1;
  st->emitted[0] = tok;
  st->n_emitted = 1;
  if (reset) st->j = st->d = st->stop = 0;
}

}  // namespace ctl
}  // namespace ssd
