// Pass set-up, draft control and acceptance kernels (sm_103a).
//
// These kernels keep the decoding state in device memory (DevState) so
// that a captured CUDA graph of a draft step, a verify pass or an
// autoregressive step can be replayed for every step without host-side
// argument changes.
#include <algorithm>

#include "control_dev.cuh"

namespace ssd {

namespace {

constexpr int kBeginThreads = 512;
constexpr int kAcceptThreads = 1024;

__global__ void __launch_bounds__(kBeginThreads) begin_kernel(BeginArgs a) {
  __shared__ int s_M[2], s_tok[kMaxRows];
  pdl_wait();
  pdl_trigger();
  ctl::begin(a, threadIdx.x, kBeginThreads, s_M, s_tok, [] { __syncthreads(); });
}

__global__ void save_boundary_kernel(SaveArgs a) {
  pdl_wait();
  pdl_trigger();
  ctl::save_boundary(a, threadIdx.x, blockDim.x, [] { __syncthreads(); });
}

__global__ void draft_end_kernel(DraftEndArgs a) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) ctl::draft_end(a);
}

__global__ void ar_end_kernel(DevState* st, int32_t* tokens, const RowStats* vstats,
                              int row_from_M, float T, int reset) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) ctl::ar_end(st, tokens, vstats, row_from_M, T, reset);
}

// Greedy acceptance: the longest prefix of drafts matching the full
// model's argmax, then the full model's token after it.  Dynamic
// verification (SWIFT §4.2): when draft y_a is rejected and a sibling
// candidate at depth a is the full model's token there, the sibling is
// taken and the full model's token after it (its own verify row) is
// emitted as well.
__global__ void accept_greedy_kernel(DevState* st, int32_t* tokens, const RowStats* vstats) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x != 0) return;
  const int d = st->d, n = st->n, ns = st->n_sib;
  int a = 0;
  while (a < d && st->draft_tok[a] == vstats[a].top1) ++a;
  for (int i = 0; i < a; ++i) st->emitted[i] = st->draft_tok[i];
  const int t = vstats[a].top1;
  st->emitted[a] = t;
  int sib = -1;
  if (a < d)
    for (int i = 0; i < ns; ++i)
      if (st->sib_depth[i] == a && st->sib_tok[i] == t) sib = i;
  int ne = a + 1;
  if (sib >= 0) st->emitted[ne++] = vstats[d + 1 + sib].top1;
  for (int i = 0; i < ne; ++i)
    if (!SSD_CHECK(st, st->emitted[i] >= 0 && st->emitted[i] < st->vocab, DBG_TOKEN, st->emitted[i]))
      st->emitted[i] = 0;
  if (!SSD_CHECK(st, n + ne <= st->max_seq, DBG_COMMIT, n + ne)) return;
  for (int i = 0; i < ne; ++i) tokens[n + i] = st->emitted[i];
  st->n = n + ne;
  st->n_emitted = ne;
  st->accepted = a;
  st->sib_acc = sib;
  st->sib_pos = n + a;
  st->last_d = d;
  st->j = st->d = st->stop = 0;
}

// Device-side generation loop: sets a graph conditional from the decoding
// state (see LoopCond) and keeps the loop's running counts.  One thread.
__global__ void loop_cond_kernel(DevState* st, cudaGraphConditionalHandle h, int what, int arg,
                                 int limit) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x != 0) return;
  unsigned v = 0;
  switch (what) {
    case LOOP_DRAFT_FIRST:  // arg = d_max
      v = arg > 0;
      break;
    case LOOP_DRAFT_NEXT:   // after a draft step; arg = d_max
      st->acc_steps += 1;
      v = !st->stop && st->j < arg;
      break;
    case LOOP_EXTRA:
      v = !st->stop;
      st->acc_extra += v;
      break;
    case LOOP_NOP:          // leaves the condition as it is
      return;
    case LOOP_WIDE:         // arg = rows of the narrow verify graph
      v = st->d + 1 + st->n_sib > arg;
      break;
    case LOOP_ROUND:        // after the acceptance; arg = 1: siblings counted
      st->acc_rounds += 1;
      st->acc_drafted += st->last_d;
      st->acc_accepted += st->accepted;
      st->acc_emitted += st->n_emitted;
      if (arg) {
        st->acc_side_rows += st->n_sib;
        st->acc_side_acc += st->sib_acc >= 0;
      }
      // limit = max_seq - (d_max + 1): another round never writes past the cache
      v = st->n < st->target_n && st->n <= limit && st->err == 0;
      break;
  }
  cudaGraphSetConditional(h, v);
}

// The taken sibling's K/V rows (every layer and KV head) into the cache at
// its position; 16-byte pieces, grid-stride.
__global__ void side_commit_kernel(const DevState* st, bf16* kc, bf16* vc, const bf16* ks,
                                   const bf16* vs, int L, int Hkv, int max_seq, int dh) {
  pdl_wait();
  pdl_trigger();
  const int sib = __ldcg(&st->sib_acc);
  if (sib < 0) return;
  const int pos = __ldcg(&st->sib_pos);
  const int per_row = dh / 8;                       // 16-byte pieces per row
  const int total = 2 * L * Hkv * per_row;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
    const int q = e % per_row, r = e / per_row;     // r = (kv, l, h)
    const int lh = r % (L * Hkv), kv = r / (L * Hkv);
    const bf16* src = (kv ? vs : ks) + ((size_t)lh * kMaxSide + sib) * dh + 8 * q;
    bf16* dst = (kv ? vc : kc) + ((size_t)lh * max_seq + pos) * dh + 8 * q;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

// ---- stochastic acceptance (LayerSkip blog §3.3) ---------------------------

SSD_DI float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, red[w]);
  return r;
}

SSD_DI float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r += red[w];
  return r;
}

SSD_DI void block_argmax(float& v, int& i, float* redv, int* redi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) { redv[warp] = v; redi[warp] = i; }
  __syncthreads();
  v = redv[0];
  i = redi[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
    if (better(redv[w], redi[w], v, i)) { v = redv[w]; i = redi[w]; }
}

// log sum exp (z / T) over one row, fixed order.
SSD_DI float row_lse_t(const float* z, int V, float T, float* red) {
  float mx = -INFINITY;
  for (int v = threadIdx.x; v < V; v += blockDim.x) mx = fmaxf(mx, z[v] / T);
  mx = block_max(mx, red);
  float s = 0.f;
  for (int v = threadIdx.x; v < V; v += blockDim.x) s += expf(z[v] / T - mx);
  s = block_sum(s, red);
  return mx + logf(s);
}

__global__ void __launch_bounds__(kAcceptThreads) accept_stoch_kernel(AcceptArgs a) {
  __shared__ float red[32];
  __shared__ float redv[32];
  __shared__ int redi[32];
  __shared__ int s_dec;
  pdl_wait();
  pdl_trigger();
  DevState* st = a.st;
  const int d = st ? st->d : a.d_static;
  const int n = st ? st->n : a.n_static;
  const int round = st ? st->round : a.round_static;
  const int32_t* drafts = st ? st->draft_tok : a.drafts;
  const int V = a.V;
  const float T = a.temperature;

  int acc = 0;
  float lseP = 0.f, lseQ = 0.f;
  for (; acc < d; ++acc) {
    const float* P = a.P + (size_t)acc * V;
    const float* Q = a.Q + (size_t)acc * V;
    lseP = a.pstats ? a.pstats[acc].lse_t : row_lse_t(P, V, T, red);
    lseQ = a.qstats ? a.qstats[acc].lse_t : row_lse_t(Q, V, T, red);
    if (threadIdx.x == 0) {
      const int y = drafts[acc];
      const float p = expf(P[y] / T - lseP);
      const float q = expf(Q[y] / T - lseQ);
      const uint4 r = philox4x32_10(make_uint4(0u, (uint32_t)(n + acc), (uint32_t)round, 1u),
                                    (uint32_t)a.seed, (uint32_t)(a.seed >> 32));
      s_dec = u01(r.x) < p / q;
    }
    __syncthreads();
    const int ok = s_dec;
    __syncthreads();
    if (!ok) break;
  }
  // sample the token after the accepted prefix
  float bv = -INFINITY, pv = -INFINITY;
  int bi = 0x7fffffff, pi = 0x7fffffff;
  const int row = acc;
  const int pos = n + row;
  const float* P = a.P + (size_t)row * V;
  if (row < d) {
    // residual norm(max(0, p - q)); p itself if the residual is empty
    const float* Q = a.Q + (size_t)row * V;
    // four consecutive entries per thread and Philox call (the argmax does
    // not depend on which thread visits an entry)
    for (int v4 = threadIdx.x * 4; v4 < V; v4 += blockDim.x * 4) {
      float gg[4];
      gumbel4(a.seed, v4 >> 2, pos, round, 2, gg);
#pragma unroll
      for (int w4 = 0; w4 < 4; ++w4) {
        const int v = v4 + w4;
        if (v >= V) break;
        const float lp = P[v] / T - lseP;
        const float w = expf(lp) - expf(Q[v] / T - lseQ);
        const float g = gg[w4];
        if (w > 0.f) {
          const float sc = logf(w) + g;
          if (better(sc, v, bv, bi)) { bv = sc; bi = v; }
        }
        const float sp = lp + g;
        if (better(sp, v, pv, pi)) { pv = sp; pi = v; }
      }
    }
    block_argmax(bv, bi, redv, redi);
    block_argmax(pv, pi, redv, redi);
    if (bv == -INFINITY) bi = pi;
  } else {
    for (int v4 = threadIdx.x * 4; v4 < V; v4 += blockDim.x * 4) {
      float gg[4];
      gumbel4(a.seed, v4 >> 2, pos, round, 2, gg);
#pragma unroll
      for (int w4 = 0; w4 < 4; ++w4) {
        if (v4 + w4 >= V) break;
        const float sc = P[v4 + w4] / T + gg[w4];
        if (better(sc, v4 + w4, bv, bi)) { bv = sc; bi = v4 + w4; }
      }
    }
    block_argmax(bv, bi, redv, redi);
  }
  if (threadIdx.x == 0) {
    if (st) {
      for (int i = 0; i < acc; ++i) st->emitted[i] = drafts[i];
      st->emitted[acc] = bi;
      for (int i = 0; i <= acc; ++i)
        if (!SSD_CHECK(st, st->emitted[i] >= 0 && st->emitted[i] < a.V, DBG_TOKEN, st->emitted[i]))
          st->emitted[i] = 0;
      if (!SSD_CHECK(st, n + acc + 1 <= st->max_seq, DBG_COMMIT, n + acc + 1)) return;
      for (int i = 0; i <= acc; ++i) a.tokens[n + i] = st->emitted[i];
      st->n = n + acc + 1;
      st->n_emitted = acc + 1;
      st->accepted = acc;
      st->last_d = d;
      st->j = st->d = st->stop = 0;
    } else {
      for (int i = 0; i < acc; ++i) a.emitted[i] = drafts[i];
      a.emitted[acc] = bi;
      *a.n_emitted = acc + 1;
    }
  }
}

__global__ void philox_kernel(const uint32_t* ctr, int count, uint64_t key, uint32_t* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count) return;
  const uint4 c = reinterpret_cast<const uint4*>(ctr)[i];
  reinterpret_cast<uint4*>(out)[i] = philox4x32_10(c, (uint32_t)key, (uint32_t)(key >> 32));
}

__global__ void ss_partials_kernel(const float* x, int M, int D, float* ss) {
  const int NP = D / kSsGroup;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= M * NP) return;
  const int m = e / NP, grp = e % NP;
  const float* src = x + (size_t)m * D + grp * kSsGroup;
  float s = 0.f;
  for (int i = 0; i < kSsGroup; ++i) s += src[i] * src[i];
  ss[e] = s;
}

__global__ void rope_table_kernel(float2* tab, int n_pos, int half, double theta) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n_pos * half) return;
  const int pos = e / half, i = e % half;
  const double inv = pow(theta, -2.0 * (double)i / (double)(2 * half));
  const double ang = (double)pos * inv;
  tab[e] = make_float2((float)cos(ang), (float)sin(ang));
}

// Device-side bounded waits, made to run out: an mbarrier nothing arrives on
// and a counter nothing increments.  Each wait must give up after `polls`
// polls and the kernel records which did (bit 0: mbarrier, bit 1: counter).
__global__ void wait_selftest_kernel(const unsigned* never, int polls, int32_t* code) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  int c = 0;
  if (!mbar_wait_n(&bar, 0u, polls)) c |= 1;
  if (!wait_count_n(never, 1u, polls)) c |= 2;
  *code = c;
}

cudaLaunchConfig_t make_cfg(int grid, int block, cudaStream_t s, bool pdl,
                            cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(block);
  lc.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return lc;
}

}  // namespace

cudaError_t launch_begin(const BeginArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t lc = make_cfg(1, kBeginThreads, s, pdl, attr);
  return cudaLaunchKernelEx(&lc, begin_kernel, a);
}

cudaError_t launch_save_boundary(const SaveArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t lc = make_cfg(1, 512, s, pdl, attr);
  return cudaLaunchKernelEx(&lc, save_boundary_kernel, a);
}

cudaError_t launch_draft_end(const DraftEndArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t lc = make_cfg(1, 32, s, pdl, attr);
  return cudaLaunchKernelEx(&lc, draft_end_kernel, a);
}

cudaError_t launch_loop_cond(DevState* st, cudaGraphConditionalHandle h, int what, int arg,
                             int limit, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t lc = make_cfg(1, 32, s, pdl, attr);
  return cudaLaunchKernelEx(&lc, loop_cond_kernel, st, h, what, arg, limit);
}

cudaError_t launch_side_commit(const DevState* st, bf16* kc, bf16* vc, const bf16* ks,
                               const bf16* vs, int L, int Hkv, int max_seq, int dh,
                               cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  const int total = 2 * L * Hkv * (dh / 8);
  const int grid = std::min(152, std::max(1, (total + 255) / 256));
  cudaLaunchConfig_t lc = make_cfg(grid, 256, s, pdl, attr);
  return cudaLaunchKernelEx(&lc, side_commit_kernel, st, kc, vc, ks, vs, L, Hkv, max_seq, dh);
}

cudaError_t launch_ar_end(DevState* st, int32_t* tokens, const RowStats* vstats, int row_from_M,
                          float temperature, int reset, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t lc = make_cfg(1, 32, s, pdl, attr);
  return cudaLaunchKernelEx(&lc, ar_end_kernel, st, tokens, vstats, row_from_M, temperature,
                            reset);
}

cudaError_t launch_accept_greedy(DevState* st, int32_t* tokens, const RowStats* vstats,
                                 cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t lc = make_cfg(1, 32, s, pdl, attr);
  return cudaLaunchKernelEx(&lc, accept_greedy_kernel, st, tokens, vstats);
}

cudaError_t launch_accept_stochastic(const AcceptArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t lc = make_cfg(1, kAcceptThreads, s, pdl, attr);
  return cudaLaunchKernelEx(&lc, accept_stoch_kernel, a);
}

// AdaInfer exit features of n exit-head summaries: out[0][l] = top1 (int
// bits), out[1][l] = p1 = exp(z1 - lse), out[2][l] = p1 - p2 with
// p2 = exp(z2 - lse).
__global__ void exit_features_kernel(const RowStats* st, int n, float* out) {
  const int l = blockIdx.x * blockDim.x + threadIdx.x;
  if (l >= n) return;
  const RowStats r = st[l];
  const float p1 = expf(r.z1 - r.lse), p2 = expf(r.z2 - r.lse);
  out[l] = __int_as_float(r.top1);
  out[n + l] = p1;
  out[2 * n + l] = p1 - p2;
}

cudaError_t launch_exit_features(const RowStats* st, int n, float* out, cudaStream_t s) {
  exit_features_kernel<<<(n + 127) / 128, 128, 0, s>>>(st, n, out);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(const unsigned* never, int polls, int32_t* code, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(never, polls, code);
  return cudaGetLastError();
}

cudaError_t launch_philox(const uint32_t* ctr, int count, uint64_t key, uint32_t* out,
                          cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  philox_kernel<<<(count + 255) / 256, 256, 0, s>>>(ctr, count, key, out);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float2* tab, int n_pos, int half, double theta, cudaStream_t s) {
  const int n = n_pos * half;
  rope_table_kernel<<<(n + 255) / 256, 256, 0, s>>>(tab, n_pos, half, theta);
  return cudaGetLastError();
}

cudaError_t launch_ss_partials(const float* x, int M, int D, float* ss, cudaStream_t s) {
  const int n = M * (D / kSsGroup);
  ss_partials_kernel<<<(n + 255) / 256, 256, 0, s>>>(x, M, D, ss);
  return cudaGetLastError();
}

}  // namespace ssd
