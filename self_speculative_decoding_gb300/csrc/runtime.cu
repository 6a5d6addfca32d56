// libssd context runtime: KV cache, workspaces, CUDA graphs and the
// draft / verify / accept loop (the C-ABI of ssd.h).
//
// One context drives one model on one GPU.  Every step's dynamic values
// (rows, positions, tokens) live in a device-side DevState, so each kind of
// pass is captured once as a CUDA graph and replayed:
//   draft step  : begin(draft) -> layers < s0 -> save boundary -> kept layers
//                 >= s0 -> LM head (+summary) -> draft end (confidence stop)
//   extra pass  : begin(extra) -> layers < s0 -> save boundary
//   verify pass : begin(verify) -> layers s0..L-1 over d+1 rows -> LM head
//   accept      : greedy prefix or min(1, p/q) acceptance, commit, rollback
//   AR step     : begin(ar) -> all layers -> LM head -> commit
// The host reads back a few bytes per draft step (the confidence stop) and
// per round (the emitted tokens).
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/ssd.h"
#include "kernels.cuh"

using namespace ssd;

namespace {

enum Phase { PH_NONE = 0, PH_IDLE = 1, PH_DRAFTED = 2, PH_VERIFIED = 3 };

// Debug builds: the canary after every context workspace.
constexpr size_t kCanaryBytes = 256;
constexpr int kCanaryByte = 0xA5;

struct Graph {
  cudaGraphExec_t exec = nullptr;
  int nodes = 0;
  void reset() {
    if (exec) cudaGraphExecDestroy(exec);
    exec = nullptr;
    nodes = 0;
  }
};

}  // namespace

struct ssd_ctx {
  ssd_config cfg{};
  std::vector<ssd_layer_weights> layers;
  const bf16* embed = nullptr;
  const float* final_norm = nullptr;
  const bf16* lm_head = nullptr;
  cudaStream_t stream = nullptr;
  cudaStream_t cap = nullptr;
  cudaStream_t cap2 = nullptr;  // captures the bodies of the loop graph's conditional nodes
  cudaEvent_t ev = nullptr;
  cudaEvent_t t0 = nullptr, t1 = nullptr;  // pass timing for ssd_stats
  int timeout_ms = 120000;
  bool pdl = true;

  ssd_policy pol{};
  bool has_policy = false;
  int s0 = 0;
  std::vector<int> pre, post, verify_layers;
  std::vector<int> post_parts;  // per post layer: 1 attention runs, 2 MLP runs

  // device buffers
  bf16* kc = nullptr;
  bf16* vc = nullptr;
  float* x = nullptr;
  float* ss = nullptr;
  float* bx = nullptr;
  float* bss = nullptr;
  // dynamic verification: the siblings' boundary states [kMaxSide][D] and
  // side K/V slots [L][Hkv][kMaxSide][dh]
  float* bxs = nullptr;
  float* bsss = nullptr;
  bf16* ks = nullptr;
  bf16* vs = nullptr;
  float* qkv = nullptr;
  bf16* attn = nullptr;
  bf16* u = nullptr;
  bf16* xn = nullptr;           // normalised bf16 rows for passes too wide for the GEMV stage
  float2* rope = nullptr;
  float* attn_part = nullptr;
  unsigned* attn_cnt = nullptr;
  float* g_part = nullptr;      // GEMV split-row-group partials (shared by all GEMVs)
  unsigned* g_cnt = nullptr;
  float* g_rec = nullptr;
  RowStats* dstats = nullptr;
  RowStats* vstats = nullptr;
  float* dlogits = nullptr;
  float* vlogits = nullptr;
  int32_t* tokens = nullptr;
  int32_t* toks_in = nullptr;
  // candidate-mask scoring: rows (candidate-major, up to max_score_rows) of
  // the batched forward, per-layer candidate lists and compact row maps
  float* sc_x = nullptr;          // [rows][D] residual stream
  bf16* sc_xn = nullptr;          // [rows][D] normalised activations (packed units)
  float* sc_qkv = nullptr;        // [rows][(H + 2 Hkv) dh]
  bf16* sc_q = nullptr;           // [rows][H dh] after RoPE
  bf16* sc_sk = nullptr;          // [rows][Hkv dh] window keys (RoPE applied)
  bf16* sc_sv = nullptr;          // [rows][Hkv dh] window values
  bf16* sc_attn = nullptr;        // [rows][H dh] (packed units)
  bf16* sc_u = nullptr;           // [rows][FFN] (packed units)
  unsigned long long* sc_best = nullptr;  // [rows] argmax keys
  int32_t* sc_cand = nullptr;     // [L][256]
  int32_t* sc_map = nullptr;      // [L][rows]
  int32_t* h_sc_cand = nullptr;   // pinned mirrors
  int32_t* h_sc_map = nullptr;
  int32_t* sc_counts = nullptr;
  int32_t* h_counts = nullptr;
  std::vector<int> sc_owner;      // per candidate of the last call: the row block it shares
  int pf_chunk = 0;               // prompt rows per batched prefill chunk
  DevState* st = nullptr;
  DevState* h_st = nullptr;  // pinned mirror
  int32_t* h_tok = nullptr;  // pinned staging [max_seq]

  Graph g_draft, g_extra, g_verify, g_accept, g_ar;
  // device-side generation loop: a whole ssd_generate in one graph launch
  // (rounds, draft steps, the extra pass and the verify width decided on the
  // device by conditional nodes); nodes of its bodies per iteration
  Graph g_loop;
  bool use_loop = true;
  std::string loop_err;  // why the loop graph could not be built (empty: built)
  int loop_nodes_draft = 0, loop_nodes_extra = 0, loop_nodes_round = 0;
  // lossy early-exit step: the AR step over the draft layer set only
  Graph g_lossy;
  // first position whose K/V a lossy step left incomplete (-1: none); the
  // lossless entry points refuse to run until it is rewound or re-prefilled
  int lossy_from = -1;
  // per-layer exit-head summaries and features (ssd_layer_features)
  RowStats* fstats = nullptr;
  float* ffeat = nullptr;         // [3][L]: top1 (as int bits), p1, p1 - p2
  float* h_ffeat = nullptr;
  // verify pass for rounds whose d + 1 rows do not fit the GEMV activation
  // stage (norm pre-pass + bf16 projections); g_verify covers the others
  Graph g_verify_wide;
  // static row bound of the passes being enqueued (0: up to 16 rows)
  int mmax = 0;
  // fp32 model (SSD_DTYPE_FP32): the K/V cache, attention output, SwiGLU
  // product and logits scratch hold fp32 (kc, vc, attn, u allocated at 4
  // bytes an element), weights are row-major fp32, fp32.cu runs the steps
  bool fp32 = false;
  std::vector<unsigned char*> canaries;  // debug builds: the workspaces' canaries
  const float* embed32 = nullptr;
  const float* lm_head32 = nullptr;
  float* lg32 = nullptr;          // logits rows of passes that keep none [16][V]

  Phase phase = PH_NONE;
  // profiling: events recorded around every eager launch
  bool profiling = false;
  int prof_class = 6;
  int prof_graph_cls = 0;   // kernel class captured by b_prof_class
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> prof_events;
  int64_t launches = 0;
  int capturing_nodes = 0;
  bool capturing = false;
  std::string err;
};

namespace {

thread_local char g_static_err[256];

ssd_status fail(ssd_ctx* c, ssd_status s, const std::string& msg) {
  if (c) c->err = msg;
  return s;
}

// NVTX range over the host enqueue of a pass (the device work of graph
// replays is attributed by the profiler's correlation).
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
};

thread_local int g_fail_alloc = -1;

constexpr int kPrefillChunk = 512;  // prompt rows per batched prefill chunk  // fault injection: fail the n-th allocation

#define CK(call)                                                                          \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess)                                                                \
      return fail(c, SSD_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_));  \
  } while (0)

size_t kv_elems(const ssd_config& g) {
  return (size_t)g.n_layers * g.n_kv_heads * g.max_seq * g.head_dim;
}
size_t kv_layer_elems(const ssd_config& g) {
  return (size_t)g.n_kv_heads * g.max_seq * g.head_dim;
}
int qkv_rows(const ssd_config& g) { return (g.n_heads + 2 * g.n_kv_heads) * g.head_dim; }

bool bit(const uint64_t* m, int l) { return (m[l >> 6] >> (l & 63)) & 1ull; }
bool skipped(const ssd_policy& p, int l) { return bit(p.skip_mask, l); }
// Sublayers of layer l the draft runs (skip mode): 1 attention, 2 MLP.
int draft_parts(const ssd_policy& p, int l) {
  if (skipped(p, l)) return 0;
  return (bit(p.skip_attn_mask, l) ? 0 : 1) | (bit(p.skip_mlp_mask, l) ? 0 : 2);
}

// Bounded host wait on the context stream.
ssd_status wait_stream(ssd_ctx* c) {
  CK(cudaEventRecord(c->ev, c->stream));
  const auto t0 = std::chrono::steady_clock::now();
  int spins = 0;
  for (;;) {
    const cudaError_t e = cudaEventQuery(c->ev);
    if (e == cudaSuccess) return SSD_OK;
    if (e != cudaErrorNotReady)
      return fail(c, SSD_ERR_CUDA, std::string("stream: ") + cudaGetErrorString(e));
    if (++spins > 2000) {
      const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                          std::chrono::steady_clock::now() - t0)
                          .count();
      if (ms > c->timeout_ms) return fail(c, SSD_ERR_TIMEOUT, "timed out waiting for the GPU");
      std::this_thread::sleep_for(std::chrono::microseconds(20));
    }
  }
}

ssd_status read_state(ssd_ctx* c) {
  CK(cudaMemcpyAsync(c->h_st, c->st, sizeof(DevState), cudaMemcpyDeviceToHost, c->stream));
  const ssd_status r = wait_stream(c);
  if (r != SSD_OK) return r;
  if (c->h_st->err >= kDbgCodeBase)
    return fail(c, SSD_ERR_STATE,
                "a device bounds check failed (code " + std::to_string(c->h_st->err) + ", value " +
                    std::to_string(c->h_st->err_val) + "); the context must be destroyed");
  if (c->h_st->err != 0)
    return fail(c, SSD_ERR_TIMEOUT,
                "a device-side wait gave up (code " + std::to_string(c->h_st->err) +
                    "); the context must be destroyed");
  return SSD_OK;
}

// ---------------------------------------------------------------------------
// enqueue helpers (eager stream or capture stream)

ssd_status note(ssd_ctx* c, cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(c, SSD_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  if (c->capturing) c->capturing_nodes++;
  else c->launches++;
  if (c->profiling) {
    // close the event pair opened by prof_begin
    cudaEventRecord(c->prof_events.back().second.second, c->stream);
  }
  return SSD_OK;
}

// Opens an event pair before an eager launch of kernel class `cls`.
void prof_begin(ssd_ctx* c, int cls) {
  if (!c->profiling) return;
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  cudaEventRecord(a, c->stream);
  c->prof_events.push_back({cls, {a, b}});
}

void gemv_scratch_args(ssd_ctx* c, LinearArgs& a) {
  a.part = c->g_part;
  a.counter = c->g_cnt;
  a.rec = c->g_rec;
  a.err = &c->st->err;
  a.err_val = &c->st->err_val;
  a.wide = (c->mmax ? c->mmax : kMaxRows) > gemv_stage_rows(a.K) ? 1 : 0;
  a.m_max = c->mmax ? c->mmax : kMaxRows;
}

// Arguments of layer l's five steps (shared by the eager and the captured
// launches).
LinearArgs qkv_args(ssd_ctx* c, int l) {
  const ssd_config& g = c->cfg;
  const ssd_layer_weights& w = c->layers[l];
  LinearArgs a;
  a.W0 = (const bf16*)w.wqkv;
  a.R = qkv_rows(g);
  a.K = g.d_model;
  a.x = c->x;
  a.ss = c->ss;
  a.gain = (const float*)w.attn_norm;
  a.eps = g.norm_eps;
  a.M_dev = &c->st->M;
  a.y = c->qkv;
  gemv_scratch_args(c, a);
  return a;
}

AttnArgs attn_args(ssd_ctx* c, int l) {
  const ssd_config& g = c->cfg;
  AttnArgs a;
  a.qkv = c->qkv;
  a.ld_qkv = qkv_rows(g);
  a.M_dev = &c->st->M;
  a.pos0_dev = &c->st->pos0;
  a.kc = c->kc + (size_t)l * kv_layer_elems(g);
  a.vc = c->vc + (size_t)l * kv_layer_elems(g);
  a.max_seq = g.max_seq;
  a.H = g.n_heads;
  a.Hkv = g.n_kv_heads;
  a.dh = g.head_dim;
  a.rope = c->rope;
  a.out = c->attn;
  a.part = c->attn_part;
  a.counters = c->attn_cnt;
  a.err = &c->st->err;
  a.err_val = &c->st->err_val;
  a.scale = (float)(1.0 / std::sqrt((double)g.head_dim));
  a.ns_dev = &c->st->ns;
  a.side_pos = c->st->side_pos;
  a.side0 = &c->st->side0;
  a.ks = c->ks + (size_t)l * g.n_kv_heads * kMaxSide * g.head_dim;
  a.vs = c->vs + (size_t)l * g.n_kv_heads * kMaxSide * g.head_dim;
  return a;
}

LinearArgs oproj_args(ssd_ctx* c, int l) {
  const ssd_config& g = c->cfg;
  LinearArgs a;
  a.W0 = (const bf16*)c->layers[l].wo;
  a.R = g.d_model;
  a.K = g.n_heads * g.head_dim;
  a.act = c->attn;
  a.M_dev = &c->st->M;
  a.xres = c->x;
  a.ss_out = c->ss;
  gemv_scratch_args(c, a);
  return a;
}

LinearArgs gateup_args(ssd_ctx* c, int l) {
  const ssd_config& g = c->cfg;
  const ssd_layer_weights& w = c->layers[l];
  LinearArgs a;
  a.W0 = (const bf16*)w.w_gate;
  a.W1 = (const bf16*)w.w_up;
  a.R = g.ffn_dim;
  a.K = g.d_model;
  a.x = c->x;
  a.ss = c->ss;
  a.gain = (const float*)w.mlp_norm;
  a.eps = g.norm_eps;
  a.M_dev = &c->st->M;
  a.u = c->u;
  gemv_scratch_args(c, a);
  return a;
}

LinearArgs down_args(ssd_ctx* c, int l) {
  const ssd_config& g = c->cfg;
  LinearArgs a;
  a.W0 = (const bf16*)c->layers[l].w_down;
  a.R = g.d_model;
  a.K = g.ffn_dim;
  a.act = c->u;
  a.M_dev = &c->st->M;
  a.xres = c->x;
  a.ss_out = c->ss;
  gemv_scratch_args(c, a);
  return a;
}

// LM head over the pass's rows; every pass reports lse(z / T), only draft,
// AR and prefill passes draw (sample_stream >= 0).
LinearArgs lm_args(ssd_ctx* c, RowStats* stats, float* logits, const int32_t* slot_dev,
                   int sample_stream) {
  const ssd_config& g = c->cfg;
  LinearArgs a;
  a.W0 = c->lm_head;
  a.R = g.vocab;
  a.K = g.d_model;
  a.x = c->x;
  a.ss = c->ss;
  a.gain = c->final_norm;
  a.eps = g.norm_eps;
  a.M_dev = &c->st->M;
  a.logits = logits;
  a.stats = stats;
  a.slot_dev = slot_dev;
  gemv_scratch_args(c, a);
  a.temperature = c->pol.temperature;
  a.sample = sample_stream >= 0 ? 1 : 0;
  a.seed = c->pol.seed;
  a.round_dev = &c->st->round;
  a.sample_stream = sample_stream < 0 ? 0 : sample_stream;
  a.pos0_dev = &c->st->pos0;
  return a;
}

BeginArgs begin_args(ssd_ctx* c, int mode, int M, int pos0, const int32_t* toks_in, int reset) {
  BeginArgs b;
  b.mode = mode;
  b.st = c->st;
  b.tokens = c->tokens;
  b.toks_in = toks_in;
  b.M = M;
  b.pos0 = pos0;
  b.reset_round = reset;
  b.embed = c->embed;
  b.embed32 = c->embed32;
  b.D = c->cfg.d_model;
  b.x = c->x;
  b.ss = c->ss;
  b.bx = c->bx;
  b.bss = c->bss;
  b.bxs = c->bxs;
  b.bsss = c->bsss;
  return b;
}

// Dynamic verification is on: siblings ride in the draft / extra passes.
bool tree_on(const ssd_ctx* c) { return c->pol.tree_tau > 0.f && c->pol.tree_max > 0; }

SaveArgs save_args(ssd_ctx* c, int use_d) {
  SaveArgs a;
  a.st = c->st;
  a.use_d = use_d;
  a.x = c->x;
  a.ss = c->ss;
  a.bx = c->bx;
  a.bss = c->bss;
  a.bxs = c->bxs;
  a.bsss = c->bsss;
  a.D = c->cfg.d_model;
  return a;
}

DraftEndArgs draft_end_args(ssd_ctx* c) {
  DraftEndArgs a;
  a.st = c->st;
  a.dstats = c->dstats;
  a.tau = c->pol.tau;
  a.temperature = c->pol.temperature;
  a.tree_tau = tree_on(c) ? c->pol.tree_tau : 0.f;
  a.tree_max = tree_on(c) ? c->pol.tree_max : 0;
  return a;
}

// A norm-fused projection of a pass whose rows may not fit the GEMV's
// activation stage runs as a RMSNorm pre-pass into bf16 rows plus a bf16-input
// projection (same bits, bounded shared memory).
ssd_status enq_norm_gemv(ssd_ctx* c, int epi, const LinearArgs& a, cudaStream_t s,
                         const char* what) {
  const int mm = c->mmax ? c->mmax : kMaxRows;
  if (mm <= gemv_stage_rows(a.K)) return note(c, launch_gemv(IN_NORM, epi, a, s, c->pdl), what);
  ssd_status r = note(c, launch_norm_rows(a.x, a.ss, a.gain, a.eps, a.M_static, a.M_dev, a.K, c->xn,
                                          s, c->pdl),
                      "rmsnorm");
  if (r != SSD_OK) return r;
  if (c->profiling) prof_begin(c, 6);
  LinearArgs b = a;
  b.act = c->xn;
  b.x = nullptr;
  b.ss = nullptr;
  b.gain = nullptr;
  return note(c, launch_gemv(IN_BF16, epi, b, s, c->pdl), what);
}

// fp32 models: layer l's steps and the LM head (fp32.cu).
LinearArgs32 lin32(ssd_ctx* c, const void* W, int R, int K) {
  LinearArgs32 a;
  a.W0 = (const float*)W;
  a.R = R;
  a.K = K;
  a.M_dev = &c->st->M;
  a.eps = c->cfg.norm_eps;
  return a;
}

ssd_status enq_layer32(ssd_ctx* c, int l, cudaStream_t s, int parts) {
  const ssd_config& g = c->cfg;
  const ssd_layer_weights& w = c->layers[l];
  const int D = g.d_model, HD = g.n_heads * g.head_dim;
  float* attn = reinterpret_cast<float*>(c->attn);
  float* u = reinterpret_cast<float*>(c->u);
  ssd_status r;
  if (parts & 1) {
    prof_begin(c, 0);
    LinearArgs32 q = lin32(c, w.wqkv, qkv_rows(g), D);
    q.x = c->x;
    q.gain = (const float*)w.attn_norm;
    q.y = c->qkv;
    if ((r = note(c, launch_gemv32(IN_NORM, EPI_STORE, q, s, c->pdl), "qkv")) != SSD_OK) return r;
    prof_begin(c, 1);
    AttnArgs32 at;
    at.qkv = c->qkv;
    at.ld_qkv = qkv_rows(g);
    at.M_dev = &c->st->M;
    at.pos0_dev = &c->st->pos0;
    at.kc = reinterpret_cast<float*>(c->kc) + (size_t)l * kv_layer_elems(g);
    at.vc = reinterpret_cast<float*>(c->vc) + (size_t)l * kv_layer_elems(g);
    at.max_seq = g.max_seq;
    at.H = g.n_heads;
    at.Hkv = g.n_kv_heads;
    at.dh = g.head_dim;
    at.rope = c->rope;
    at.out = attn;
    at.scale = (float)(1.0 / std::sqrt((double)g.head_dim));
    if ((r = note(c, launch_attention32(at, s, c->pdl), "attention")) != SSD_OK) return r;
    prof_begin(c, 2);
    LinearArgs32 o = lin32(c, w.wo, D, HD);
    o.act = attn;
    o.xres = c->x;
    if ((r = note(c, launch_gemv32(IN_BF16, EPI_RESID, o, s, c->pdl), "o_proj")) != SSD_OK) return r;
  }
  if (!(parts & 2)) return SSD_OK;
  prof_begin(c, 3);
  LinearArgs32 gu = lin32(c, w.w_gate, g.ffn_dim, D);
  gu.W1 = (const float*)w.w_up;
  gu.x = c->x;
  gu.gain = (const float*)w.mlp_norm;
  gu.u = u;
  if ((r = note(c, launch_gemv32(IN_NORM, EPI_SWIGLU, gu, s, c->pdl), "gate_up")) != SSD_OK) return r;
  prof_begin(c, 4);
  LinearArgs32 dn = lin32(c, w.w_down, D, g.ffn_dim);
  dn.act = u;
  dn.xres = c->x;
  return note(c, launch_gemv32(IN_BF16, EPI_RESID, dn, s, c->pdl), "down");
}

// fp32 LM head: logits rows [slot + m] (the logits buffer, or the scratch
// rows when the pass keeps none), then their row summaries.
ssd_status enq_lmhead32(ssd_ctx* c, RowStats* stats, float* logits, const int32_t* slot_dev,
                        int sample_stream, cudaStream_t s) {
  const ssd_config& g = c->cfg;
  LinearArgs32 a = lin32(c, c->lm_head32, g.vocab, g.d_model);
  a.x = c->x;
  a.gain = c->final_norm;
  a.y = logits ? logits : c->lg32;
  a.row0_dev = logits ? slot_dev : nullptr;
  ssd_status r = note(c, launch_gemv32(IN_NORM, EPI_STORE, a, s, c->pdl), "lm_head");
  if (r != SSD_OK) return r;
  LmSummaryArgs32 m;
  m.logits = a.y;
  m.V = g.vocab;
  m.M_dev = &c->st->M;
  m.slot_dev = slot_dev;
  m.stats = stats;
  m.temperature = c->pol.temperature;
  m.sample = sample_stream >= 0 ? 1 : 0;
  m.seed = c->pol.seed;
  m.round_dev = &c->st->round;
  m.stream = sample_stream < 0 ? 0 : sample_stream;
  m.pos0_dev = &c->st->pos0;
  // scratch rows are written from row 0 on; a pass that keeps its logits
  // reads them at its slot
  if (!logits) m.slot_dev = nullptr;
  return note(c, launch_lm_summary32(m, s, c->pdl), "lm_summary");
}

ssd_status enq_layer(ssd_ctx* c, int l, cudaStream_t s, int parts = 3) {
  if (c->fp32) return enq_layer32(c, l, s, parts);
  ssd_status r;
  if (!(parts & 1)) goto mlp;
  prof_begin(c, 0);
  if ((r = enq_norm_gemv(c, EPI_STORE, qkv_args(c, l), s, "qkv")) != SSD_OK) return r;
  prof_begin(c, 1);
  if ((r = note(c, launch_attention(attn_args(c, l), s, c->pdl), "attention")) != SSD_OK) return r;
  prof_begin(c, 2);
  if ((r = note(c, launch_gemv(IN_BF16, EPI_RESID, oproj_args(c, l), s, c->pdl), "o_proj")) !=
      SSD_OK)
    return r;
mlp:
  if (!(parts & 2)) return SSD_OK;
  prof_begin(c, 3);
  if ((r = enq_norm_gemv(c, EPI_SWIGLU, gateup_args(c, l), s, "gate_up")) != SSD_OK) return r;
  prof_begin(c, 4);
  return note(c, launch_gemv(IN_BF16, EPI_RESID, down_args(c, l), s, c->pdl), "down");
}

ssd_status enq_layers(ssd_ctx* c, const std::vector<int>& ls, cudaStream_t s,
                      const std::vector<int>* parts = nullptr) {
  for (size_t i = 0; i < ls.size(); ++i) {
    const ssd_status r = enq_layer(c, ls[i], s, parts ? (*parts)[i] : 3);
    if (r != SSD_OK) return r;
  }
  return SSD_OK;
}

ssd_status enq_lmhead(ssd_ctx* c, RowStats* stats, float* logits, const int32_t* slot_dev,
                      int sample_stream, cudaStream_t s) {
  prof_begin(c, 5);
  if (c->fp32) return enq_lmhead32(c, stats, logits, slot_dev, sample_stream, s);
  return enq_norm_gemv(c, EPI_LMHEAD, lm_args(c, stats, logits, slot_dev, sample_stream), s,
                       "lm_head");
}

ssd_status enq_begin(ssd_ctx* c, int mode, cudaStream_t s, int M = 1, int pos0 = 0,
                     const int32_t* toks_in = nullptr, int reset = 0) {
  prof_begin(c, 6);
  return note(c, launch_begin(begin_args(c, mode, M, pos0, toks_in, reset), s, c->pdl), "begin");
}


// ---------------------------------------------------------------------------
// graphs

typedef ssd_status (*Builder)(ssd_ctx*, cudaStream_t);

ssd_status build_graph(ssd_ctx* c, Graph& g, Builder fn) {
  g.reset();
  CK(cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal));
  c->capturing = true;
  c->capturing_nodes = 0;
  ssd_status r = fn(c, c->cap);
  c->capturing = false;
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(c->cap, &graph);
  if (r != SSD_OK) {
    if (graph) cudaGraphDestroy(graph);
    return r;
  }
  if (e != cudaSuccess) return fail(c, SSD_ERR_CUDA, std::string("capture: ") + cudaGetErrorString(e));
  const cudaError_t e2 = cudaGraphInstantiate(&g.exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e2 != cudaSuccess)
    return fail(c, SSD_ERR_CUDA, std::string("instantiate: ") + cudaGetErrorString(e2));
  g.nodes = c->capturing_nodes;
  return SSD_OK;
}

ssd_status b_draft_body(ssd_ctx* c, cudaStream_t s);
ssd_status b_draft(ssd_ctx* c, cudaStream_t s) {
  c->mmax = tree_on(c) ? 2 : 1;
  const ssd_status r = b_draft_body(c, s);
  c->mmax = 0;
  return r;
}
ssd_status b_draft_body(ssd_ctx* c, cudaStream_t s) {
  ssd_status r;
  if ((r = enq_begin(c, BEGIN_DRAFT, s)) != SSD_OK) return r;
  if ((r = enq_layers(c, c->pre, s)) != SSD_OK) return r;
  if ((r = note(c, launch_save_boundary(save_args(c, 0), s, c->pdl), "save_boundary")) != SSD_OK)
    return r;
  if ((r = enq_layers(c, c->post, s, &c->post_parts)) != SSD_OK) return r;
  if ((r = enq_lmhead(c, c->dstats, c->dlogits, &c->st->slot, 0, s)) != SSD_OK) return r;
  return note(c, launch_draft_end(draft_end_args(c), s, c->pdl), "draft_end");
}

ssd_status b_extra_body(ssd_ctx* c, cudaStream_t s);
ssd_status b_extra(ssd_ctx* c, cudaStream_t s) {
  c->mmax = tree_on(c) ? 2 : 1;
  const ssd_status r = b_extra_body(c, s);
  c->mmax = 0;
  return r;
}
ssd_status b_extra_body(ssd_ctx* c, cudaStream_t s) {
  ssd_status r;
  if ((r = enq_begin(c, BEGIN_EXTRA, s)) != SSD_OK) return r;
  if ((r = enq_layers(c, c->pre, s)) != SSD_OK) return r;
  return note(c, launch_save_boundary(save_args(c, 1), s, c->pdl), "save_boundary");
}

ssd_status b_verify_body(ssd_ctx* c, cudaStream_t s);
// Rows the verify graphs are built for: the narrow one up to what the stage
// holds at d_model, the wide one up to d_max + 1 chain rows plus the
// siblings of dynamic verification.
int verify_max_rows(const ssd_ctx* c) {
  return c->pol.d_max + 1 + (tree_on(c) ? c->pol.tree_max : 0);
}
int verify_narrow_rows(const ssd_ctx* c) {
  return std::min(verify_max_rows(c), std::max(1, gemv_stage_rows(c->cfg.d_model)));
}
ssd_status b_verify(ssd_ctx* c, cudaStream_t s) {
  c->mmax = verify_narrow_rows(c);
  const ssd_status r = b_verify_body(c, s);
  c->mmax = 0;
  return r;
}
ssd_status b_verify_wide(ssd_ctx* c, cudaStream_t s) {
  c->mmax = verify_max_rows(c);
  const ssd_status r = b_verify_body(c, s);
  c->mmax = 0;
  return r;
}
ssd_status b_verify_body(ssd_ctx* c, cudaStream_t s) {
  ssd_status r;
  if ((r = enq_begin(c, BEGIN_VERIFY, s)) != SSD_OK) return r;
  if ((r = enq_layers(c, c->verify_layers, s)) != SSD_OK) return r;
  return enq_lmhead(c, c->vstats, c->vlogits, nullptr, -1, s);
}

ssd_status b_accept(ssd_ctx* c, cudaStream_t s) {
  if (c->pol.temperature > 0.f) {
    AcceptArgs a;
    a.P = c->vlogits;
    a.Q = c->dlogits;
    a.pstats = c->vstats;
    a.qstats = c->dstats;
    a.V = c->cfg.vocab;
    a.temperature = c->pol.temperature;
    a.seed = c->pol.seed;
    a.st = c->st;
    a.tokens = c->tokens;
    return note(c, launch_accept_stochastic(a, s, c->pdl), "accept");
  }
  ssd_status r = note(c, launch_accept_greedy(c->st, c->tokens, c->vstats, s, c->pdl), "accept");
  if (r != SSD_OK || !tree_on(c)) return r;
  const ssd_config& g = c->cfg;
  return note(c, launch_side_commit(c->st, c->kc, c->vc, c->ks, c->vs, g.n_layers, g.n_kv_heads,
                                    g.max_seq, g.head_dim, s, c->pdl),
              "side_commit");
}

ssd_status b_ar_body(ssd_ctx* c, cudaStream_t s);
ssd_status b_ar(ssd_ctx* c, cudaStream_t s) {
  c->mmax = 1;
  const ssd_status r = b_ar_body(c, s);
  c->mmax = 0;
  return r;
}
ssd_status b_ar_body(ssd_ctx* c, cudaStream_t s) {
  ssd_status r;
  if ((r = enq_begin(c, BEGIN_AR, s)) != SSD_OK) return r;
  std::vector<int> all(c->cfg.n_layers);
  for (int l = 0; l < c->cfg.n_layers; ++l) all[l] = l;
  if ((r = enq_layers(c, all, s)) != SSD_OK) return r;
  if ((r = enq_lmhead(c, c->vstats, nullptr, nullptr, 2, s)) != SSD_OK) return r;
  prof_begin(c, 6);
  return note(c, launch_ar_end(c->st, c->tokens, c->vstats, 0, c->pol.temperature, 0, s, c->pdl),
              "ar_end");
}

// LayerSkip blog §3, inference mode one: the pending token through the draft
// layer set only, the shared head, and the AR step's commit.
ssd_status b_lossy(ssd_ctx* c, cudaStream_t s) {
  c->mmax = 1;
  ssd_status r;
  if ((r = enq_begin(c, BEGIN_AR, s)) == SSD_OK && (r = enq_layers(c, c->pre, s)) == SSD_OK &&
      (r = enq_layers(c, c->post, s, &c->post_parts)) == SSD_OK &&
      (r = enq_lmhead(c, c->vstats, nullptr, nullptr, 2, s)) == SSD_OK)
    r = note(c, launch_ar_end(c->st, c->tokens, c->vstats, 0, c->pol.temperature, 0, s, c->pdl),
             "ar_end");
  c->mmax = 0;
  return r;
}

ssd_status build_graphs_once(ssd_ctx* c) {
  ssd_status r;
  if ((r = build_graph(c, c->g_draft, b_draft)) != SSD_OK) return r;
  if ((r = build_graph(c, c->g_extra, b_extra)) != SSD_OK) return r;
  if ((r = build_graph(c, c->g_verify, b_verify)) != SSD_OK) return r;
  c->g_verify_wide.reset();
  if (verify_narrow_rows(c) < verify_max_rows(c) &&
      (r = build_graph(c, c->g_verify_wide, b_verify_wide)) != SSD_OK)
    return r;
  if ((r = build_graph(c, c->g_accept, b_accept)) != SSD_OK) return r;
  if ((r = build_graph(c, c->g_lossy, b_lossy)) != SSD_OK) return r;
  return build_graph(c, c->g_ar, b_ar);
}

// ---------------------------------------------------------------------------
// device-side generation loop

// During a capture on `s`: appends a conditional node after the captured
// work so far; returns its body graphs (owned by the node).
cudaGraph_t* add_conditional(cudaStream_t s, cudaGraphConditionalHandle h,
                             cudaGraphConditionalNodeType type, unsigned size, cudaError_t* err) {
  cudaStreamCaptureStatus status;
  cudaGraph_t g = nullptr;
  const cudaGraphNode_t* deps = nullptr;
  const cudaGraphEdgeData* edges = nullptr;
  size_t nd = 0;
  *err = cudaStreamGetCaptureInfo(s, &status, nullptr, &g, &deps, &edges, &nd);
  if (*err != cudaSuccess) return nullptr;
  cudaGraphNodeParams p = {};
  p.type = cudaGraphNodeTypeConditional;
  p.conditional.handle = h;
  p.conditional.type = type;
  p.conditional.size = size;
  cudaGraphNode_t node = nullptr;
  *err = cudaGraphAddNode(&node, g, deps, edges, nd, &p);
  if (*err != cudaSuccess) return nullptr;
  *err = cudaStreamUpdateCaptureDependencies(s, &node, nullptr, 1, cudaStreamSetCaptureDependencies);
  return *err == cudaSuccess ? p.conditional.phGraph_out : nullptr;
}

// Captures builder `fn` (and optionally one condition kernel after it) into
// body graph `g` on the second capture stream; returns the nodes captured.
// Highest committed length from which another round stays inside the cache.
int loop_limit(const ssd_ctx* c) { return c->cfg.max_seq - (c->pol.d_max + 1); }

ssd_status capture_body(ssd_ctx* c, cudaGraph_t g, Builder fn, cudaGraphConditionalHandle h,
                        int what, int arg, int* nodes) {
  CK(cudaStreamBeginCaptureToGraph(c->cap2, g, nullptr, nullptr, 0,
                                   cudaStreamCaptureModeThreadLocal));
  const int n0 = c->capturing_nodes;
  ssd_status r = fn ? fn(c, c->cap2) : SSD_OK;
  if (r == SSD_OK && what >= 0)
    r = note(c, launch_loop_cond(c->st, h, what, arg, loop_limit(c), c->cap2, false), "loop_cond");
  cudaGraph_t out = nullptr;
  const cudaError_t e = cudaStreamEndCapture(c->cap2, &out);
  if (r != SSD_OK) return r;
  if (e != cudaSuccess) return fail(c, SSD_ERR_CUDA, std::string("capture: ") + cudaGetErrorString(e));
  if (nodes) *nodes = c->capturing_nodes - n0;
  return SSD_OK;
}

// The loop graph (one launch runs rounds until n reaches DevState::target_n):
//   while (hR) {                       hR: default 1 at every launch
//     hD = d_max > 0; while (hD) { draft step; hD = !stop && j < d_max }
//     hE = !stop;     if (hE) { extra pass }
//     hW = rows > narrow; if (hW) { wide verify } else { verify }
//     accept; hR = n < target_n
//   }
ssd_status build_loop_graph(ssd_ctx* c) {
  c->g_loop.reset();
  cudaGraph_t G = nullptr;
  CK(cudaGraphCreate(&G, 0));
  cudaGraphConditionalHandle hR, hD, hE, hW;
  cudaError_t e = cudaGraphConditionalHandleCreate(&hR, G, 1, cudaGraphCondAssignDefault);
  ssd_status r = SSD_OK;
  cudaGraph_t body = nullptr;
  if (e == cudaSuccess) {
    cudaGraphNodeParams p = {};
    p.type = cudaGraphNodeTypeConditional;
    p.conditional.handle = hR;
    p.conditional.type = cudaGraphCondTypeWhile;
    p.conditional.size = 1;
    cudaGraphNode_t node = nullptr;
    e = cudaGraphAddNode(&node, G, nullptr, nullptr, 0, &p);
    if (e == cudaSuccess) body = p.conditional.phGraph_out[0];
  }
  if (e == cudaSuccess) e = cudaGraphConditionalHandleCreate(&hD, body, 0, 0);
  if (e == cudaSuccess) e = cudaGraphConditionalHandleCreate(&hE, body, 0, 0);
  if (e == cudaSuccess) e = cudaGraphConditionalHandleCreate(&hW, body, 0, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(G);
    return fail(c, SSD_ERR_CUDA, std::string("loop graph: ") + cudaGetErrorString(e));
  }
  const bool wide = c->g_verify_wide.exec != nullptr;
  int n_draft = 0, n_extra = 0, n_v = 0, n_vw = 0;
  c->capturing = true;
  c->capturing_nodes = 0;
  e = cudaStreamBeginCaptureToGraph(c->cap, body, nullptr, nullptr, 0,
                                    cudaStreamCaptureModeThreadLocal);
  bool open = e == cudaSuccess;
  if (open)
    r = note(c, launch_loop_cond(c->st, hD, LOOP_DRAFT_FIRST, c->pol.d_max, loop_limit(c), c->cap,
                                 false),
             "loop_cond");
  cudaGraph_t* bd = nullptr;
  if (open && r == SSD_OK) bd = add_conditional(c->cap, hD, cudaGraphCondTypeWhile, 1, &e);
  if (bd) r = capture_body(c, bd[0], b_draft, hD, LOOP_DRAFT_NEXT, c->pol.d_max, &n_draft);
  if (bd && r == SSD_OK)
    r = note(c, launch_loop_cond(c->st, hE, LOOP_EXTRA, 0, loop_limit(c), c->cap, false), "loop_cond");
  cudaGraph_t* be = nullptr;
  if (bd && r == SSD_OK) be = add_conditional(c->cap, hE, cudaGraphCondTypeIf, 1, &e);
  if (be) r = capture_body(c, be[0], b_extra, hE, -1, 0, &n_extra);
  // the verify runs in the body of an IF node in both cases (without a wide
  // graph its condition, rows > 0, always holds), so that every conditional
  // node is followed by a plain-launched condition kernel or another
  // conditional node and no programmatic launch depends on one directly
  bool verified = false;
  if (be && r == SSD_OK) {
    r = note(c, launch_loop_cond(c->st, hW, LOOP_WIDE, wide ? verify_narrow_rows(c) : 0,
                                 loop_limit(c), c->cap, false),
             "loop_cond");
    cudaGraph_t* bw =
        r == SSD_OK ? add_conditional(c->cap, hW, cudaGraphCondTypeIf, wide ? 2 : 1, &e) : nullptr;
    if (bw) r = capture_body(c, bw[0], wide ? b_verify_wide : b_verify, hW, -1, 0, &n_vw);
    if (bw && wide && r == SSD_OK) r = capture_body(c, bw[1], b_verify, hW, -1, 0, &n_v);
    verified = bw != nullptr && r == SSD_OK;
  }
  int n_acc = 0;
  if (verified) {
    const int n0 = c->capturing_nodes;
    // a plain launch after the verify's IF node (see above)
    r = note(c, launch_loop_cond(c->st, hE, LOOP_NOP, 0, loop_limit(c), c->cap, false),
             "loop_cond");
    if (r == SSD_OK) r = b_accept(c, c->cap);
    if (r == SSD_OK)
      r = note(c, launch_loop_cond(c->st, hR, LOOP_ROUND, tree_on(c) ? 1 : 0, loop_limit(c),
                                   c->cap, false),
               "loop_cond");
    n_acc = c->capturing_nodes - n0;
  }
  cudaGraph_t out = nullptr;
  if (open) {
    const cudaError_t e2 = cudaStreamEndCapture(c->cap, &out);
    if (e == cudaSuccess) e = e2;
  }
  c->capturing = false;
  if (r == SSD_OK && (e != cudaSuccess || !verified)) {
    r = fail(c, SSD_ERR_CUDA, std::string("loop graph capture: ") + cudaGetErrorString(e));
  }
  if (r == SSD_OK) {
    e = cudaGraphInstantiate(&c->g_loop.exec, G, 0);
    if (e != cudaSuccess) {
      c->g_loop.exec = nullptr;
      r = fail(c, SSD_ERR_CUDA, std::string("loop graph instantiate: ") + cudaGetErrorString(e));
    }
  }
  cudaGraphDestroy(G);
  c->loop_nodes_draft = n_draft;
  c->loop_nodes_extra = n_extra;
  c->loop_nodes_round = std::max(n_v, n_vw) + n_acc + 3;
  return r;
}

// Builds the per-pass graphs, then the device-side generation loop over them.
ssd_status build_graphs(ssd_ctx* c) {
  const ssd_status r = build_graphs_once(c);
  if (r != SSD_OK) return r;
  // the loop graph is an optimisation: without it generation runs the same
  // graphs from the host
  const std::string keep = c->err;
  c->loop_err.clear();
  if (build_loop_graph(c) != SSD_OK) {
    c->g_loop.reset();
    cudaGetLastError();
    c->loop_err = c->err;
    c->err = keep;
  }
  return SSD_OK;
}

ssd_status replay(ssd_ctx* c, Graph& g) {
  CK(cudaGraphLaunch(g.exec, c->stream));
  c->launches += g.nodes;
  return SSD_OK;
}

// algorithmic bytes of one pass: weights of the layers run (+ LM head), K/V
// read for positions [0, pos0 + M) and written for M positions per layer.
double pass_bytes(const ssd_ctx* c, int n_layers_run, bool lm, int pos0, int M) {
  const ssd_config& g = c->cfg;
  const double el = c->fp32 ? 4.0 : 2.0;
  const double layer_w = el * ((double)qkv_rows(g) * g.d_model +
                               (double)g.d_model * g.n_heads * g.head_dim +
                               3.0 * g.d_model * g.ffn_dim);
  const double kv_pos = 2.0 * el * g.n_kv_heads * g.head_dim;
  double b = n_layers_run * (layer_w + kv_pos * (pos0 + M) + kv_pos * M);
  if (lm) b += el * (double)g.vocab * g.d_model;
  return b;
}

// algorithmic bytes of one draft step at position pos: the layers below s0,
// the sublayers the draft runs above it, and the LM head
double draft_bytes(const ssd_ctx* c, int pos) {
  const ssd_config& g = c->cfg;
  const double el = c->fp32 ? 4.0 : 2.0;
  const double attn_w = el * ((double)qkv_rows(g) * g.d_model + (double)g.d_model * g.n_heads * g.head_dim);
  const double mlp_w = el * 3.0 * g.d_model * g.ffn_dim;
  const double kv = 2.0 * el * g.n_kv_heads * g.head_dim * (double)(pos + 2);
  double b = c->pre.size() * (attn_w + kv + mlp_w);
  for (int pt : c->post_parts) b += ((pt & 1) ? attn_w + kv : 0.0) + ((pt & 2) ? mlp_w : 0.0);
  return b + el * (double)g.vocab * g.d_model;
}

ssd_status check_capacity(ssd_ctx* c, int extra) {
  if (c->h_st->n + extra > c->cfg.max_seq)
    return fail(c, SSD_ERR_CAPACITY, "KV cache capacity (max_seq) exceeded");
  return SSD_OK;
}

// Draft loop (host side of the confidence stop).  Returns with h_st read.
ssd_status run_draft(ssd_ctx* c, ssd_stats* stats) {
  ssd_status r;
  const int n = c->h_st->n;
  for (int j = 0; j < c->pol.d_max; ++j) {
    Range nv("ssd draft step");
    if (stats) CK(cudaEventRecord(c->t0, c->stream));
    if ((r = replay(c, c->g_draft)) != SSD_OK) return r;
    if (stats) CK(cudaEventRecord(c->t1, c->stream));
    if ((r = read_state(c)) != SSD_OK) return r;
    if (stats) {
      float ms = 0.f;
      cudaEventElapsedTime(&ms, c->t0, c->t1);
      stats->draft_ms += ms;
      stats->draft_steps++;
      stats->bytes_streamed += draft_bytes(c, n - 1 + j);
    }
    if (c->h_st->stop) break;
  }
  c->phase = PH_DRAFTED;
  return SSD_OK;
}

ssd_status run_verify(ssd_ctx* c, ssd_stats* stats) {
  Range nv("ssd verify");
  ssd_status r;
  const int n = c->h_st->n, d = c->h_st->d, nsib = c->h_st->n_sib;
  if (stats) CK(cudaEventRecord(c->t0, c->stream));
  const bool extra = !c->h_st->stop;
  if (extra) {
    if ((r = replay(c, c->g_extra)) != SSD_OK) return r;
    if (stats) stats->bytes_streamed += pass_bytes(c, (int)c->pre.size(), false, n - 1 + d, 1);
  }
  const bool wide = d + 1 + nsib > verify_narrow_rows(c) && c->g_verify_wide.exec;
  if ((r = replay(c, wide ? c->g_verify_wide : c->g_verify)) != SSD_OK) return r;
  if (stats)
    stats->bytes_streamed += pass_bytes(c, (int)c->verify_layers.size(), true, n - 1, d + 1 + nsib);
  c->phase = PH_VERIFIED;
  return SSD_OK;
}

ssd_status ensure_policy(ssd_ctx* c, bool lossless = true) {
  if (!c->has_policy) return fail(c, SSD_ERR_STATE, "no policy set (ssd_set_policy)");
  if (c->phase == PH_NONE) return fail(c, SSD_ERR_STATE, "no prefill");
  if (lossless && c->lossy_from >= 0)
    return fail(c, SSD_ERR_STATE,
                "positions from " + std::to_string(c->lossy_from) +
                    " were decoded lossily (skipped layers' K/V missing); rewind to <= " +
                    std::to_string(c->lossy_from + 1) + " or prefill again");
  return SSD_OK;
}

// One layer of the batched forward over T compact rows of the scoring
// buffers (compact row t = row map[t] of sc_x, map nullable = identity):
// RMSNorm, QKV projection, RoPE with the window K/V (and, with kv_write, the
// cache at positions split + p % N), attention of the n_active candidates'
// window rows (cand, device), o_proj + residual, RMSNorm, SwiGLU, down +
// residual.
ssd_status enq_rows_layer(ssd_ctx* c, int l, int T, const int32_t* map, const int32_t* cand,
                          int n_active, int N, int split, bool kv_write) {
  const ssd_config& g = c->cfg;
  const int D = g.d_model, HD = g.n_heads * g.head_dim;
  cudaStream_t s = c->stream;
  ssd_status r;
  bf16* at_kc = c->kc + (size_t)l * kv_layer_elems(g);
  bf16* at_vc = c->vc + (size_t)l * kv_layer_elems(g);
  const ssd_layer_weights& w = c->layers[l];
  if ((r = note(c, launch_score_norm(c->sc_x, map, (const float*)w.attn_norm, g.norm_eps, T, D,
                                     c->sc_xn, s),
                "score_norm")) != SSD_OK)
    return r;
  GemmArgs q;
  q.W0 = (const bf16*)w.wqkv;
  q.R = qkv_rows(g);
  q.K = D;
  q.T = T;
  q.act = c->sc_xn;
  q.epi = GEMM_STORE;
  q.err = &c->st->err;
  q.y = c->sc_qkv;
  if ((r = note(c, launch_gemm_rows(q, s), "score_qkv")) != SSD_OK) return r;
  if ((r = note(c, launch_score_rope(c->sc_qkv, T, map, N, split, g.n_heads, g.n_kv_heads,
                                     g.head_dim, c->rope, c->sc_q, c->sc_sk, c->sc_sv,
                                     kv_write ? at_kc : nullptr, kv_write ? at_vc : nullptr,
                                     g.max_seq, s),
                "score_rope")) != SSD_OK)
    return r;
  ScoreAttnArgs at;
  at.q = c->sc_q;
  at.kc = at_kc;
  at.vc = at_vc;
  at.sk = c->sc_sk;
  at.sv = c->sc_sv;
  at.cand = cand;
  at.N = N;
  at.split = split;
  at.max_seq = g.max_seq;
  at.H = g.n_heads;
  at.Hkv = g.n_kv_heads;
  at.dh = g.head_dim;
  at.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)g.head_dim));
  at.out = c->sc_attn;
  at.out_packed = 1;
  at.w_rows = std::max(g.max_score_rows, c->pf_chunk);  // rows of sc_sk / sc_sv
  at.err = &c->st->err;
  if ((r = note(c, launch_score_attn(at, n_active, s), "score_attn")) != SSD_OK) return r;
  GemmArgs o;
  o.W0 = (const bf16*)w.wo;
  o.R = D;
  o.K = HD;
  o.T = T;
  o.act = c->sc_attn;
  o.epi = GEMM_RESID;
  o.err = &c->st->err;
  o.x = c->sc_x;
  o.rowmap = map;
  if ((r = note(c, launch_gemm_rows(o, s), "score_oproj")) != SSD_OK) return r;
  if ((r = note(c, launch_score_norm(c->sc_x, map, (const float*)w.mlp_norm, g.norm_eps, T, D,
                                     c->sc_xn, s),
                "score_norm")) != SSD_OK)
    return r;
  GemmArgs gu;
  gu.W0 = (const bf16*)w.w_gate;
  gu.W1 = (const bf16*)w.w_up;
  gu.R = g.ffn_dim;
  gu.K = D;
  gu.T = T;
  gu.act = c->sc_xn;
  gu.epi = GEMM_SWIGLU;
  gu.err = &c->st->err;
  gu.u = c->sc_u;
  gu.u_packed = 1;
  gu.fast_silu = kv_write ? 0 : 1;  // the prefill's cache keeps the full-precision SiLU
  if ((r = note(c, launch_gemm_rows(gu, s), "score_gate_up")) != SSD_OK) return r;
  GemmArgs dn;
  dn.W0 = (const bf16*)w.w_down;
  dn.R = D;
  dn.K = g.ffn_dim;
  dn.T = T;
  dn.act = c->sc_u;
  dn.epi = GEMM_RESID;
  dn.err = &c->st->err;
  dn.x = c->sc_x;
  dn.rowmap = map;
  if ((r = note(c, launch_gemm_rows(dn, s), "score_down")) != SSD_OK) return r;
    return SSD_OK;
}

// SWIFT §4.1.2: the K candidate layer sets predict the committed tokens
// t[split+1 .. split+N] from t[split .. split+N-1] in one batched forward.
// Row p = k N + i is candidate k's window position split + i; a layer runs
// the rows of the candidates that keep it (compact row t -> p through the
// layer's row map), attending to the shared cache's positions below split
// and to the candidate's own window K/V.  Leaves the match counts in
// sc_counts; the shared cache is only read.
ssd_status enq_score(ssd_ctx* c, const uint64_t* masks, int K, int N, int split) {
  const ssd_config& g = c->cfg;
  const int L = g.n_layers, D = g.d_model, rows = K * N, R = g.max_score_rows;
  // Candidates whose skip decisions agree on every layer so far hold the same
  // rows (all steps of the forward are row-count invariant), so each group
  // computes one block of rows, held by its owner (a member).  At the first
  // layer a group's members disagree on, the subset without the owner takes
  // a copy of the owner's rows before the layer runs.  Scores are identical
  // to computing every candidate on its own.
  auto skips = [&](int k, int l) { return ((masks[4 * k + (l >> 6)] >> (l & 63)) & 1ull) != 0; };
  std::vector<int> owner(K, 0), nact(L, 0);
  std::vector<std::vector<std::pair<int, int>>> copies(L);  // per layer: (from, to) owners
  for (int l = 0; l < L; ++l) {
    int32_t* cand = c->h_sc_cand + (size_t)l * 256;
    int32_t* map = c->h_sc_map + (size_t)l * R;
    std::vector<int> next = owner;
    for (int o = 0; o < K; ++o) {
      if (owner[o] != o) continue;  // o is not an owner
      std::vector<int> keep, skip;
      for (int k = o; k < K; ++k)
        if (owner[k] == o) (skips(k, l) ? skip : keep).push_back(k);
      if (keep.empty()) continue;
      int run = o;
      if (!skip.empty()) {
        const bool o_keeps = !skips(o, l);
        const std::vector<int>& moved = o_keeps ? skip : keep;
        copies[l].push_back({o, moved[0]});
        for (int k : moved) next[k] = moved[0];
        if (!o_keeps) run = moved[0];
      }
      for (int i = 0; i < N; ++i) map[nact[l] * N + i] = run * N + i;
      cand[nact[l]++] = run;
    }
    owner = next;
  }
  // final owners: the LM head and the match count run on their rows
  int nfin = 0;
  {
    int32_t* map = c->h_sc_map + (size_t)L * R;
    for (int o = 0; o < K; ++o)
      if (owner[o] == o) {
        for (int i = 0; i < N; ++i) map[nfin * N + i] = o * N + i;
        ++nfin;
      }
  }
  c->sc_owner.assign(owner.begin(), owner.end());
  CK(cudaMemcpyAsync(c->sc_cand, c->h_sc_cand, (size_t)L * 256 * 4, cudaMemcpyHostToDevice,
                     c->stream));
  CK(cudaMemcpyAsync(c->sc_map, c->h_sc_map, (size_t)(L + 1) * R * 4, cudaMemcpyHostToDevice,
                     c->stream));
  CK(cudaMemsetAsync(c->sc_counts, 0, (size_t)K * sizeof(int32_t), c->stream));
  CK(cudaMemsetAsync(c->sc_best, 0, (size_t)rows * 8, c->stream));
  ssd_status r;
  cudaStream_t s = c->stream;
  if ((r = note(c, launch_score_embed(c->embed, c->tokens, split, N, rows, D, c->sc_x, s),
                "score_embed")) != SSD_OK)
    return r;
  for (int l = 0; l < L; ++l) {
    for (const auto& cp : copies[l])
      CK(cudaMemcpyAsync(c->sc_x + (size_t)cp.second * N * D, c->sc_x + (size_t)cp.first * N * D,
                         (size_t)N * D * sizeof(float), cudaMemcpyDeviceToDevice, s));
    const int T = nact[l] * N;
    if (T == 0) continue;
    if ((r = enq_rows_layer(c, l, T, c->sc_map + (size_t)l * R, c->sc_cand + (size_t)l * 256,
                            nact[l], N, split, false)) != SSD_OK)
      return r;
  }
  const int32_t* fmap = c->sc_map + (size_t)L * R;
  if ((r = note(c, launch_score_norm(c->sc_x, fmap, c->final_norm, g.norm_eps, nfin * N, D,
                                     c->sc_xn, s),
                "score_norm")) != SSD_OK)
    return r;
  GemmArgs lm;
  lm.W0 = c->lm_head;
  lm.R = g.vocab;
  lm.K = D;
  lm.T = nfin * N;
  lm.act = c->sc_xn;
  lm.epi = GEMM_ARGMAX;
  lm.err = &c->st->err;
  lm.best = c->sc_best;
  if ((r = note(c, launch_gemm_rows(lm, s), "score_lm_head")) != SSD_OK) return r;
  return note(c, launch_score_match(c->sc_best, fmap, c->tokens, split, N, nfin * N,
                                    c->sc_counts, s),
              "score_match");
}

}  // namespace

// ===========================================================================
// C-ABI

extern "C" {

ssd_status ssd_create(const ssd_config* cfg, const ssd_weights* w, void* stream, ssd_ctx** out) {
  ssd_ctx* c = nullptr;
  if (!cfg || !w || !out || !w->layers || !w->tok_embed || !w->lm_head || !w->final_norm)
    return SSD_ERR_INVALID_ARG;
  *out = nullptr;
  const ssd_config& g = *cfg;
  if (g.n_layers <= 0 || g.n_layers > 256 || g.d_model <= 0 || g.d_model % 64 ||
      g.n_heads <= 0 || g.n_kv_heads <= 0 || g.n_heads % g.n_kv_heads ||
      (g.head_dim != 64 && g.head_dim != 128) || g.ffn_dim <= 0 || g.ffn_dim % 32 ||
      g.vocab <= 0 || g.vocab % 16 || g.max_seq <= 0 || g.max_seq % kAttnChunk ||
      g.max_draft < 1 || g.max_draft > kMaxRows - 1 || g.max_score_rows < 0 ||
      (g.n_heads * g.head_dim) % 32 || g.n_heads / g.n_kv_heads > 8 || !(g.norm_eps > 0.f) ||
      !(g.rope_theta > 0.f) || (g.dtype != SSD_DTYPE_BF16 && g.dtype != SSD_DTYPE_FP32) ||
      (g.dtype == SSD_DTYPE_FP32 && g.max_score_rows > 0))
    return SSD_ERR_INVALID_ARG;
  // every weight is read with 16-byte vector loads and bulk copies
  auto al16 = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
  if (!al16(w->tok_embed) || !al16(w->final_norm) || !al16(w->lm_head)) return SSD_ERR_INVALID_ARG;
  for (int l = 0; l < g.n_layers; ++l) {
    const ssd_layer_weights& L = w->layers[l];
    if (!L.attn_norm || !L.wqkv || !L.wo || !L.mlp_norm || !L.w_gate || !L.w_up || !L.w_down)
      return SSD_ERR_INVALID_ARG;
    if (!al16(L.attn_norm) || !al16(L.wqkv) || !al16(L.wo) || !al16(L.mlp_norm) ||
        !al16(L.w_gate) || !al16(L.w_up) || !al16(L.w_down))
      return SSD_ERR_INVALID_ARG;
  }
  c = new ssd_ctx();
  c->cfg = g;
  c->layers.assign(w->layers, w->layers + g.n_layers);
  c->fp32 = g.dtype == SSD_DTYPE_FP32;
  c->embed = (const bf16*)w->tok_embed;
  c->final_norm = (const float*)w->final_norm;
  c->lm_head = (const bf16*)w->lm_head;
  if (c->fp32) {
    c->embed32 = (const float*)w->tok_embed;
    c->lm_head32 = (const float*)w->lm_head;
  }
  c->stream = (cudaStream_t)stream;

  auto alloc = [&](void** p, size_t bytes) -> bool {
    if (g_fail_alloc >= 0 && g_fail_alloc-- == 0) {  // injected failure (ssd_debug_fail_alloc)
      g_fail_alloc = -1;
      return false;
    }
#ifdef SSD_DEBUG_CHECKS
    // debug builds: every workspace is followed by a canary of kCanaryBytes
    // bytes of kCanaryByte, checked by ssd_debug_canaries
    const size_t body = (bytes + 255) & ~(size_t)255;
    if (cudaMalloc(p, body + kCanaryBytes) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    unsigned char* guard = static_cast<unsigned char*>(*p) + body;
    cudaMemsetAsync(guard, kCanaryByte, kCanaryBytes, c->stream);
    c->canaries.push_back(guard);
#else
    if (cudaMalloc(p, bytes) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
#endif
    return true;
  };
  const int D = g.d_model, F = g.ffn_dim, V = g.vocab;
  const int nr = kMaxRows;
  const size_t act_el = c->fp32 ? 4 : 2;  // K/V, attention output, SwiGLU product
  // one scratch area serves every GEMV of the context (they run in stream order)
  GemvScratch gs{0, 0, 0};
  {
    const GemvScratch all[5] = {gemv_scratch(qkv_rows(g), D, EPI_STORE),
                                gemv_scratch(D, g.n_heads * g.head_dim, EPI_RESID),
                                gemv_scratch(F, D, EPI_SWIGLU), gemv_scratch(D, F, EPI_RESID),
                                gemv_scratch(V, D, EPI_LMHEAD)};
    for (const GemvScratch& x : all) {
      gs.part_floats = std::max(gs.part_floats, x.part_floats);
      gs.counters = std::max(gs.counters, x.counters);
      gs.rec_floats = std::max(gs.rec_floats, x.rec_floats);
    }
  }
  bool ok = alloc((void**)&c->kc, kv_elems(g) * act_el) &&
            alloc((void**)&c->vc, kv_elems(g) * act_el) &&
            alloc((void**)&c->x, (size_t)nr * D * 4) &&
            alloc((void**)&c->ss, (size_t)nr * (D / kSsGroup) * 4) &&
            alloc((void**)&c->bx, (size_t)nr * D * 4) &&
            alloc((void**)&c->bss, (size_t)nr * (D / kSsGroup) * 4) &&
            alloc((void**)&c->bxs, (size_t)kMaxSide * D * 4) &&
            alloc((void**)&c->bsss, (size_t)kMaxSide * (D / kSsGroup) * 4) &&
            alloc((void**)&c->ks, (size_t)g.n_layers * g.n_kv_heads * kMaxSide * g.head_dim * 2) &&
            alloc((void**)&c->vs, (size_t)g.n_layers * g.n_kv_heads * kMaxSide * g.head_dim * 2) &&
            alloc((void**)&c->qkv, (size_t)nr * qkv_rows(g) * 4) &&
            alloc((void**)&c->attn, (size_t)nr * g.n_heads * g.head_dim * act_el) &&
            alloc((void**)&c->u, (size_t)nr * F * act_el) &&
            (!c->fp32 || alloc((void**)&c->lg32, (size_t)nr * V * 4)) &&
            alloc((void**)&c->xn, (size_t)nr * D * 2) &&
            alloc((void**)&c->rope, (size_t)g.max_seq * (g.head_dim / 2) * sizeof(float2)) &&
            alloc((void**)&c->attn_part,
                  attn_part_floats(g.n_kv_heads, g.n_heads, g.head_dim, g.max_seq) * 4) &&
            alloc((void**)&c->attn_cnt, (size_t)g.n_kv_heads * 4) &&
            alloc((void**)&c->g_part, gs.part_floats * 4) &&
            alloc((void**)&c->g_cnt, gs.counters * 4) &&
            alloc((void**)&c->g_rec, gs.rec_floats * 4) &&
            alloc((void**)&c->dstats, (size_t)nr * sizeof(RowStats)) &&
            alloc((void**)&c->vstats, (size_t)nr * sizeof(RowStats)) &&
            alloc((void**)&c->dlogits, (size_t)nr * V * 4) &&
            alloc((void**)&c->vlogits, (size_t)nr * V * 4) &&
            alloc((void**)&c->tokens, (size_t)g.max_seq * 4) &&
            alloc((void**)&c->toks_in, (size_t)g.max_seq * 4) &&
            alloc((void**)&c->st, sizeof(DevState)) &&
            alloc((void**)&c->fstats, (size_t)g.n_layers * sizeof(RowStats)) &&
            alloc((void**)&c->ffeat, (size_t)3 * g.n_layers * 4);
  if (ok) {
    // the batched forward's rows: candidate-mask scoring (max_score_rows) and
    // the prefill chunks share them; rows of the projections' packed bf16
    // inputs are padded to 16
    c->pf_chunk = g.max_seq < kPrefillChunk ? g.max_seq : kPrefillChunk;
    const size_t r = (size_t)std::max(g.max_score_rows, c->pf_chunk), D = g.d_model,
                 HD = (size_t)g.n_heads * g.head_dim;
    const size_t rp = (r + 15) / 16 * 16;
    const size_t KV = (size_t)g.n_kv_heads * g.head_dim;
    ok = alloc((void**)&c->sc_x, r * D * 4) && alloc((void**)&c->sc_xn, rp * D * 2) &&
         alloc((void**)&c->sc_qkv, r * qkv_rows(g) * 4) && alloc((void**)&c->sc_q, r * HD * 2) &&
         alloc((void**)&c->sc_sk, r * KV * 2) && alloc((void**)&c->sc_sv, r * KV * 2) &&
         alloc((void**)&c->sc_attn, rp * HD * 2) && alloc((void**)&c->sc_u, rp * g.ffn_dim * 2) &&
         alloc((void**)&c->sc_best, r * 8) &&
         alloc((void**)&c->sc_cand, (size_t)g.n_layers * 256 * 4) &&
         alloc((void**)&c->sc_map, (size_t)(g.n_layers + 1) * r * 4) &&
         alloc((void**)&c->sc_counts, 256 * sizeof(int32_t)) &&
         cudaMallocHost((void**)&c->h_counts, 256 * sizeof(int32_t)) == cudaSuccess &&
         cudaMallocHost((void**)&c->h_sc_cand, (size_t)g.n_layers * 256 * 4) == cudaSuccess &&
         cudaMallocHost((void**)&c->h_sc_map, (size_t)(g.n_layers + 1) * r * 4) == cudaSuccess;
    if (ok) cudaMemsetAsync(c->sc_best, 0, r * 8, c->stream);
  }
  if (!ok) {
    ssd_destroy(c);
    return SSD_ERR_OOM;
  }
  if (cudaMallocHost((void**)&c->h_st, sizeof(DevState)) != cudaSuccess ||
      cudaMallocHost((void**)&c->h_ffeat, (size_t)3 * g.n_layers * 4) != cudaSuccess ||
      cudaMallocHost((void**)&c->h_tok, (size_t)g.max_seq * 4) != cudaSuccess ||
      cudaStreamCreateWithFlags(&c->cap, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&c->cap2, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->ev, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreate(&c->t0) != cudaSuccess || cudaEventCreate(&c->t1) != cudaSuccess) {
    cudaGetLastError();
    ssd_destroy(c);
    return SSD_ERR_OOM;
  }
  memset(c->h_st, 0, sizeof(DevState));
  c->h_st->vocab = g.vocab;      // bounds of the debug builds' device checks
  c->h_st->max_seq = g.max_seq;
  cudaMemcpyAsync(c->st, c->h_st, sizeof(DevState), cudaMemcpyHostToDevice, c->stream);
  cudaMemsetAsync(c->attn_cnt, 0, (size_t)g.n_kv_heads * 4, c->stream);
  cudaMemsetAsync(c->g_cnt, 0, gs.counters * 4, c->stream);
  cudaMemsetAsync(c->tokens, 0, (size_t)g.max_seq * 4, c->stream);
  const int half = g.head_dim / 2;
  launch_rope_table(c->rope, g.max_seq, half, (double)g.rope_theta, c->stream);
  {
    AttnArgs probe;
    probe.H = g.n_heads;
    probe.Hkv = g.n_kv_heads;
    probe.dh = g.head_dim;
    probe.max_seq = g.max_seq;
    if ((c->fp32 ? attn32_prepare(g.head_dim, g.max_seq) : attn_prepare(probe)) != cudaSuccess) {
      cudaGetLastError();
      ssd_destroy(c);
      return SSD_ERR_INVALID_ARG;
    }
  }
  const cudaError_t e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) {
    ssd_destroy(c);
    return SSD_ERR_CUDA;
  }
  *out = c;
  return SSD_OK;
}

ssd_status ssd_destroy(ssd_ctx* c) {
  if (!c) return SSD_OK;
  cudaStreamSynchronize(c->stream);
  c->g_draft.reset();
  c->g_extra.reset();
  c->g_verify.reset();
  c->g_verify_wide.reset();
  c->g_accept.reset();
  c->g_ar.reset();
  c->g_lossy.reset();
  c->g_loop.reset();
  void* bufs[] = {c->kc, c->vc, c->x, c->ss, c->bx, c->bss, c->qkv, c->attn, c->u, c->xn, c->rope,
                  c->attn_part, c->attn_cnt, c->lg32, c->g_part, c->g_cnt, c->g_rec, c->dstats, c->vstats,
                  c->dlogits, c->vlogits, c->tokens, c->toks_in, c->st, c->fstats, c->ffeat,
                  c->bxs, c->bsss, c->ks, c->vs};
  for (void* p : bufs)
    if (p) cudaFree(p);
  void* sc[] = {c->sc_x,    c->sc_xn,   c->sc_qkv,  c->sc_q,   c->sc_sk,  c->sc_sv,
                c->sc_attn, c->sc_u,    c->sc_best, c->sc_cand, c->sc_map, c->sc_counts};
  for (void* p : sc)
    if (p) cudaFree(p);
  if (c->h_counts) cudaFreeHost(c->h_counts);
  if (c->h_sc_cand) cudaFreeHost(c->h_sc_cand);
  if (c->h_sc_map) cudaFreeHost(c->h_sc_map);
  if (c->h_st) cudaFreeHost(c->h_st);
  if (c->h_ffeat) cudaFreeHost(c->h_ffeat);
  if (c->h_tok) cudaFreeHost(c->h_tok);
  if (c->cap) cudaStreamDestroy(c->cap);
  if (c->cap2) cudaStreamDestroy(c->cap2);
  if (c->ev) cudaEventDestroy(c->ev);
  if (c->t0) cudaEventDestroy(c->t0);
  if (c->t1) cudaEventDestroy(c->t1);
  cudaGetLastError();
  delete c;
  return SSD_OK;
}

ssd_status ssd_set_policy(ssd_ctx* c, const ssd_policy* p) {
  if (!c || !p) return SSD_ERR_INVALID_ARG;
  const int L = c->cfg.n_layers;
  if (p->mode != SSD_MODE_SKIP && p->mode != SSD_MODE_EXIT)
    return fail(c, SSD_ERR_INVALID_ARG, "policy mode");
  if (p->mode == SSD_MODE_EXIT && (p->exit_layer < 0 || p->exit_layer >= L))
    return fail(c, SSD_ERR_INVALID_ARG, "exit_layer out of range");
  if (p->d_max < 0) return fail(c, SSD_ERR_INVALID_ARG, "d_max < 0");
  if (p->d_max > c->cfg.max_draft) return fail(c, SSD_ERR_CAPACITY, "d_max > max_draft");
  if (!(p->temperature >= 0.f) || !std::isfinite(p->temperature))
    return fail(c, SSD_ERR_INVALID_ARG, "temperature");
  if (c->phase == PH_DRAFTED || c->phase == PH_VERIFIED)
    return fail(c, SSD_ERR_STATE, "a round is in flight");
  for (int l = L; l < 256; ++l)
    if (bit(p->skip_mask, l) || bit(p->skip_attn_mask, l) || bit(p->skip_mlp_mask, l))
      return fail(c, SSD_ERR_INVALID_ARG, "skip masks name layers >= n_layers");
  if (p->mode == SSD_MODE_EXIT)
    for (int w = 0; w < 4; ++w)
      if (p->skip_attn_mask[w] || p->skip_mlp_mask[w])
        return fail(c, SSD_ERR_INVALID_ARG, "sublayer masks need skip mode");
  if (!std::isfinite(p->tree_tau)) return fail(c, SSD_ERR_INVALID_ARG, "tree_tau");
  if (p->tree_tau > 0.f && c->fp32)
    return fail(c, SSD_ERR_INVALID_ARG, "dynamic verification needs a bf16 model");
  if (p->tree_tau > 0.f) {
    if (p->temperature != 0.f)
      return fail(c, SSD_ERR_INVALID_ARG, "dynamic verification (tree_tau > 0) needs temperature 0");
    if (p->tree_max < 1 || p->tree_max > kMaxSide)
      return fail(c, SSD_ERR_INVALID_ARG, "tree_max must be 1..8 when tree_tau > 0");
    if (p->d_max + 1 + p->tree_max > kMaxRows)
      return fail(c, SSD_ERR_INVALID_ARG, "d_max + 1 + tree_max exceeds 16 verify rows");
  }
  c->pol = *p;
  c->pre.clear();
  c->post.clear();
  c->post_parts.clear();
  c->verify_layers.clear();
  if (p->mode == SSD_MODE_SKIP) {
    c->s0 = L;
    for (int l = 0; l < L; ++l)
      if (draft_parts(*p, l) != 3) { c->s0 = l; break; }
    for (int l = 0; l < L; ++l) {
      const int pt = draft_parts(*p, l);
      if (l < c->s0) {
        c->pre.push_back(l);
      } else if (pt) {
        c->post.push_back(l);
        c->post_parts.push_back(pt);
      }
    }
  } else {
    c->s0 = p->exit_layer + 1;
    for (int l = 0; l < c->s0; ++l) c->pre.push_back(l);
  }
  for (int l = c->s0; l < L; ++l) c->verify_layers.push_back(l);
  c->has_policy = true;
  const ssd_status r = build_graphs(c);
  if (r != SSD_OK) c->has_policy = false;
  return r;
}

ssd_status ssd_prefill(ssd_ctx* c, const int32_t* tokens, int32_t n, int32_t* first) {
  if (!c || !tokens || n < 1) return c ? fail(c, SSD_ERR_INVALID_ARG, "prefill args") : SSD_ERR_INVALID_ARG;
  Range nv("ssd prefill");
  if (!c->has_policy) return fail(c, SSD_ERR_STATE, "no policy set (ssd_set_policy)");
  if (n + 1 > c->cfg.max_seq) return fail(c, SSD_ERR_CAPACITY, "prompt longer than max_seq - 1");
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= c->cfg.vocab) return fail(c, SSD_ERR_INVALID_ARG, "token id out of range");
  memcpy(c->h_tok, tokens, (size_t)n * 4);
  CK(cudaMemcpyAsync(c->toks_in, c->h_tok, (size_t)n * 4, cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(c->tokens, c->h_tok, (size_t)n * 4, cudaMemcpyHostToDevice, c->stream));
  // The prompt in chunks of up to pf_chunk rows through the batched forward
  // (tensor-core projections; each chunk attends causally to itself and to
  // the cache of the chunks before it, and writes its K/V into the cache).
  const int D = c->cfg.d_model;
  cudaStream_t s = c->stream;
  ssd_status r;
  if (c->fp32) {
    // fp32 models: the prompt in passes of up to 16 rows through the decode
    // kernels, then the last position's state through the LM head
    int last = 0;
    for (int c0 = 0; c0 < n; c0 += kMaxRows) {
      const int m = std::min(kMaxRows, n - c0);
      if ((r = enq_begin(c, BEGIN_TOKENS, s, m, c0, c->toks_in + c0, 1)) != SSD_OK) return r;
      std::vector<int> all(c->cfg.n_layers);
      for (int l = 0; l < c->cfg.n_layers; ++l) all[l] = l;
      if ((r = enq_layers(c, all, s)) != SSD_OK) return r;
      last = m;
    }
    CK(cudaMemcpyAsync(c->bx, c->x + (size_t)(last - 1) * D, (size_t)D * sizeof(float),
                       cudaMemcpyDeviceToDevice, s));
    if ((r = enq_begin(c, BEGIN_TOKENS, s, 1, n - 1, c->toks_in + n - 1, 1)) != SSD_OK) return r;
    CK(cudaMemcpyAsync(c->x, c->bx, (size_t)D * sizeof(float), cudaMemcpyDeviceToDevice, s));
    if ((r = enq_lmhead(c, c->vstats, nullptr, nullptr, 2, s)) != SSD_OK) return r;
    if ((r = note(c, launch_ar_end(c->st, c->tokens, c->vstats, 1, c->pol.temperature, 1, s,
                                   c->pdl), "prefill_end")) != SSD_OK)
      return r;
    if ((r = read_state(c)) != SSD_OK) return r;
    if (first) *first = c->h_st->emitted[0];
    c->phase = PH_IDLE;
    c->lossy_from = -1;
    return SSD_OK;
  }
  CK(cudaMemsetAsync(c->sc_cand, 0, sizeof(int32_t), s));  // the one "candidate"
  int last = 0;
  for (int c0 = 0; c0 < n; c0 += c->pf_chunk) {
    const int m = std::min(c->pf_chunk, n - c0);
    if ((r = note(c, launch_score_embed(c->embed, c->toks_in, c0, m, m, D, c->sc_x, s),
                  "prefill_embed")) != SSD_OK)
      return r;
    for (int l = 0; l < c->cfg.n_layers; ++l)
      if ((r = enq_rows_layer(c, l, m, nullptr, c->sc_cand, 1, m, c0, true)) != SSD_OK) return r;
    last = m;
  }
  // the last prompt position's state through the decode path's final norm and
  // LM head (row summary; the first token committed as an AR step commits it)
  if ((r = enq_begin(c, BEGIN_TOKENS, s, 1, n - 1, c->toks_in + n - 1, 1)) != SSD_OK) return r;
  CK(cudaMemcpyAsync(c->x, c->sc_x + (size_t)(last - 1) * D, (size_t)D * sizeof(float),
                     cudaMemcpyDeviceToDevice, s));
  if ((r = note(c, launch_ss_partials(c->x, 1, D, c->ss, s), "prefill_ss")) != SSD_OK) return r;
  if ((r = enq_lmhead(c, c->vstats, nullptr, nullptr, 2, s)) != SSD_OK) return r;
  if ((r = note(c, launch_ar_end(c->st, c->tokens, c->vstats, 1, c->pol.temperature, 1, s,
                                 c->pdl), "prefill_end")) != SSD_OK)
    return r;
  if ((r = read_state(c)) != SSD_OK) return r;
  if (first) *first = c->h_st->emitted[0];
  c->phase = PH_IDLE;
  c->lossy_from = -1;
  return SSD_OK;
}

ssd_status ssd_draft(ssd_ctx* c, int32_t* draft_out, float* conf_out, int32_t* d_out) {
  if (!c) return SSD_ERR_INVALID_ARG;
  ssd_status r = ensure_policy(c);
  if (r != SSD_OK) return r;
  if (c->phase != PH_IDLE) return fail(c, SSD_ERR_STATE, "a draft is already pending");
  if ((r = check_capacity(c, c->pol.d_max + 1)) != SSD_OK) return r;
  if ((r = run_draft(c, nullptr)) != SSD_OK) return r;
  const int d = c->h_st->d;
  if (draft_out)
    for (int i = 0; i < d; ++i) draft_out[i] = c->h_st->draft_tok[i];
  if (conf_out)
    for (int i = 0; i < c->h_st->j; ++i) conf_out[i] = c->h_st->draft_conf[i];
  if (d_out) *d_out = d;
  return SSD_OK;
}

ssd_status ssd_verify(ssd_ctx* c, float* logits_out) {
  if (!c) return SSD_ERR_INVALID_ARG;
  if (c->phase != PH_DRAFTED) return fail(c, SSD_ERR_STATE, "verify without a pending draft");
  ssd_status r = run_verify(c, nullptr);
  if (r != SSD_OK) return r;
  if (logits_out) {
    const int d = c->h_st->d;
    CK(cudaMemcpyAsync(logits_out, c->vlogits, (size_t)(d + 1) * c->cfg.vocab * 4,
                       cudaMemcpyDeviceToHost, c->stream));
  }
  return wait_stream(c);
}

ssd_status ssd_accept(ssd_ctx* c, int32_t* emitted_out, int32_t* n_out) {
  if (!c) return SSD_ERR_INVALID_ARG;
  if (c->phase != PH_VERIFIED) return fail(c, SSD_ERR_STATE, "accept without a verify");
  ssd_status r = replay(c, c->g_accept);
  if (r != SSD_OK) return r;
  if ((r = read_state(c)) != SSD_OK) return r;
  c->phase = PH_IDLE;
  const int ne = c->h_st->n_emitted;
  if (emitted_out)
    for (int i = 0; i < ne; ++i) emitted_out[i] = c->h_st->emitted[i];
  if (n_out) *n_out = ne;
  return SSD_OK;
}

// ssd_generate on the device-side loop graph: one launch and one read-back
// per kLoopTokens generated tokens.
constexpr int kLoopTokens = 512;
ssd_status generate_loop(ssd_ctx* c, int32_t n_tokens, int32_t* out, ssd_stats* stats,
                         int n_start) {
  Range nv("ssd generate (device loop)");
  DevState* h = c->h_st;
  h->target_n = n_start + n_tokens;
  h->last_d = 0;
  h->acc_rounds = h->acc_drafted = h->acc_accepted = h->acc_emitted = 0;
  h->acc_steps = h->acc_extra = h->acc_side_rows = h->acc_side_acc = 0;
  const size_t off = offsetof(DevState, target_n);
  const size_t len = offsetof(DevState, pad2) - off;
  CK(cudaMemcpyAsync(reinterpret_cast<char*>(c->st) + off, reinterpret_cast<char*>(h) + off, len,
                     cudaMemcpyHostToDevice, c->stream));
  // one launch per kLoopTokens tokens, so that every bounded host wait covers
  // a bounded amount of work; the rounds continue across launches unchanged
  const int final_n = n_start + n_tokens;
  ssd_status r = SSD_OK;
  for (int n_cur = n_start; n_cur < final_n;) {
    const int32_t target = std::min(final_n, n_cur + kLoopTokens);
    if (target != h->target_n || n_cur != n_start) {
      h->target_n = target;
      CK(cudaMemcpyAsync(&c->st->target_n, &h->target_n, sizeof(int32_t),
                         cudaMemcpyHostToDevice, c->stream));
    }
    CK(cudaGraphLaunch(c->g_loop.exec, c->stream));
    if ((r = read_state(c)) != SSD_OK) break;
    if (h->n <= n_cur) {
      r = fail(c, SSD_ERR_CUDA, "device loop made no progress");
      break;
    }
    n_cur = h->n;
  }
  c->phase = PH_IDLE;
  if (r != SSD_OK) return r;
  const int64_t launches = (int64_t)h->acc_steps * c->loop_nodes_draft +
                           (int64_t)h->acc_extra * c->loop_nodes_extra +
                           (int64_t)h->acc_rounds * c->loop_nodes_round;
  c->launches += launches;
  if (stats) {
    stats->rounds = h->acc_rounds;
    stats->drafted = h->acc_drafted;
    stats->accepted = h->acc_accepted;
    stats->emitted = h->acc_emitted;
    stats->draft_steps = h->acc_steps;
    stats->side_rows = h->acc_side_rows;
    stats->side_accepted = h->acc_side_acc;
    stats->kernel_launches = launches;
    // K/V bytes at the generation's middle position
    const int mid = n_start + n_tokens / 2;
    const double rows = (double)h->acc_drafted + h->acc_rounds + h->acc_side_rows;
    stats->bytes_streamed = h->acc_steps * draft_bytes(c, mid) +
                            h->acc_extra * pass_bytes(c, (int)c->pre.size(), false, mid, 1) +
                            h->acc_rounds * pass_bytes(c, (int)c->verify_layers.size(), true, mid, 0) +
                            rows * (c->verify_layers.size() * 2.0 * 2.0 * 2.0 * c->cfg.n_kv_heads *
                                    c->cfg.head_dim);
  }
  if (out && n_tokens > 0) {
    CK(cudaMemcpyAsync(c->h_tok, c->tokens + n_start, (size_t)n_tokens * 4, cudaMemcpyDeviceToHost,
                       c->stream));
    if ((r = wait_stream(c)) != SSD_OK) return r;
    memcpy(out, c->h_tok, (size_t)n_tokens * 4);
  }
  if (h->n != n_start + n_tokens) {
    const int32_t nn = n_start + n_tokens;
    CK(cudaMemcpyAsync(&c->st->n, &nn, 4, cudaMemcpyHostToDevice, c->stream));
    if ((r = read_state(c)) != SSD_OK) return r;
  }
  return SSD_OK;
}

ssd_status ssd_generate(ssd_ctx* c, int32_t n_tokens, int32_t* out, ssd_stats* stats) {
  if (!c || n_tokens < 0) return SSD_ERR_INVALID_ARG;
  ssd_status r = ensure_policy(c);
  if (r != SSD_OK) return r;
  if (c->phase != PH_IDLE) return fail(c, SSD_ERR_STATE, "a round is in flight");
  if (stats) memset(stats, 0, sizeof(*stats));
  const int64_t l0 = c->launches;
  if ((r = read_state(c)) != SSD_OK) return r;
  const int n_start = c->h_st->n;
  if (n_start + n_tokens + c->pol.d_max + 1 > c->cfg.max_seq)
    return fail(c, SSD_ERR_CAPACITY, "n_tokens + d_max + 1 exceeds the KV capacity");
  if (c->use_loop && c->g_loop.exec && n_tokens > 0)
    return generate_loop(c, n_tokens, out, stats, n_start);
  int got = 0;
  while (got < n_tokens) {
    if ((r = run_draft(c, stats)) != SSD_OK) return r;
    const int d = c->pol.d_max == 0 ? 0 : c->h_st->d;
    if ((r = run_verify(c, stats)) != SSD_OK) return r;
    if ((r = replay(c, c->g_accept)) != SSD_OK) return r;
    if (stats) CK(cudaEventRecord(c->t1, c->stream));
    if ((r = read_state(c)) != SSD_OK) return r;
    if (stats) {
      float ms = 0.f;
      cudaEventElapsedTime(&ms, c->t0, c->t1);
      stats->verify_ms += ms;
    }
    c->phase = PH_IDLE;
    const int ne = c->h_st->n_emitted;
    for (int i = 0; i < ne && got < n_tokens; ++i, ++got)
      if (out) out[got] = c->h_st->emitted[i];
    if (stats) {
      stats->rounds++;
      stats->drafted += d;
      stats->accepted += c->h_st->accepted;
      stats->emitted += ne;
      if (tree_on(c)) {
        stats->side_rows += c->h_st->n_sib;
        stats->side_accepted += c->h_st->sib_acc >= 0 ? 1 : 0;
      }
    }
  }
  if (c->h_st->n != n_start + n_tokens) {
    const int32_t nn = n_start + n_tokens;
    CK(cudaMemcpyAsync(&c->st->n, &nn, 4, cudaMemcpyHostToDevice, c->stream));
    if ((r = read_state(c)) != SSD_OK) return r;
  }
  if (stats) stats->kernel_launches = c->launches - l0;
  return SSD_OK;
}

ssd_status ssd_decode_ar(ssd_ctx* c, int32_t n_tokens, int32_t* out, ssd_stats* stats) {
  if (!c || n_tokens < 0) return SSD_ERR_INVALID_ARG;
  ssd_status r = ensure_policy(c);
  if (r != SSD_OK) return r;
  if (c->phase != PH_IDLE) return fail(c, SSD_ERR_STATE, "a round is in flight");
  if (stats) memset(stats, 0, sizeof(*stats));
  if ((r = read_state(c)) != SSD_OK) return r;
  const int n0 = c->h_st->n;
  if (n0 + n_tokens > c->cfg.max_seq) return fail(c, SSD_ERR_CAPACITY, "max_seq exceeded");
  const int64_t l0 = c->launches;
  Range nv("ssd decode_ar");
  if (stats) CK(cudaEventRecord(c->t0, c->stream));
  for (int i = 0; i < n_tokens; ++i) {
    if ((r = replay(c, c->g_ar)) != SSD_OK) return r;
    if (stats) stats->bytes_streamed += pass_bytes(c, c->cfg.n_layers, true, n0 - 1 + i, 1);
  }
  if (stats) CK(cudaEventRecord(c->t1, c->stream));
  if (out && n_tokens > 0) {
    CK(cudaMemcpyAsync(c->h_tok, c->tokens + n0, (size_t)n_tokens * 4, cudaMemcpyDeviceToHost,
                       c->stream));
  }
  if ((r = read_state(c)) != SSD_OK) return r;
  if (out && n_tokens > 0) memcpy(out, c->h_tok, (size_t)n_tokens * 4);
  if (stats) {
    stats->rounds = n_tokens;
    stats->emitted = n_tokens;
    stats->kernel_launches = c->launches - l0;
    float ms = 0.f;
    if (n_tokens > 0) cudaEventElapsedTime(&ms, c->t0, c->t1);
    stats->ar_ms = ms;
  }
  return SSD_OK;
}

ssd_status ssd_decode_lossy(ssd_ctx* c, int32_t n_tokens, int32_t* out, ssd_stats* stats) {
  if (!c || n_tokens < 0) return SSD_ERR_INVALID_ARG;
  ssd_status r = ensure_policy(c, false);
  if (r != SSD_OK) return r;
  if (c->phase != PH_IDLE) return fail(c, SSD_ERR_STATE, "a round is in flight");
  if (stats) memset(stats, 0, sizeof(*stats));
  if ((r = read_state(c)) != SSD_OK) return r;
  const int n0 = c->h_st->n;
  if (n0 + n_tokens > c->cfg.max_seq) return fail(c, SSD_ERR_CAPACITY, "max_seq exceeded");
  const int64_t l0 = c->launches;
  Range nv("ssd decode_lossy");
  if (stats) CK(cudaEventRecord(c->t0, c->stream));
  for (int i = 0; i < n_tokens; ++i) {
    if ((r = replay(c, c->g_lossy)) != SSD_OK) return r;
    if (stats) stats->bytes_streamed += pass_bytes(c, (int)(c->pre.size() + c->post.size()), true,
                                                   n0 - 1 + i, 1);
  }
  if (stats) CK(cudaEventRecord(c->t1, c->stream));
  // a draft set that drops any sublayer leaves those layers' K/V unwritten
  if (n_tokens > 0 && c->s0 < c->cfg.n_layers && c->lossy_from < 0) c->lossy_from = n0 - 1;
  if (out && n_tokens > 0)
    CK(cudaMemcpyAsync(c->h_tok, c->tokens + n0, (size_t)n_tokens * 4, cudaMemcpyDeviceToHost,
                       c->stream));
  if ((r = read_state(c)) != SSD_OK) return r;
  if (out && n_tokens > 0) memcpy(out, c->h_tok, (size_t)n_tokens * 4);
  if (stats) {
    stats->rounds = n_tokens;
    stats->emitted = n_tokens;
    stats->kernel_launches = c->launches - l0;
    float ms = 0.f;
    if (n_tokens > 0) cudaEventElapsedTime(&ms, c->t0, c->t1);
    stats->draft_ms = ms;
  }
  return SSD_OK;
}

ssd_status ssd_layer_features(ssd_ctx* c, int32_t min_layer, int32_t* top1, float* top_prob,
                              float* gap) {
  if (!c) return SSD_ERR_INVALID_ARG;
  const int L = c->cfg.n_layers;
  if (min_layer < 0 || min_layer >= L || !top1 || !top_prob || !gap)
    return fail(c, SSD_ERR_INVALID_ARG, "layer_features arguments");
  ssd_status r = ensure_policy(c);
  if (r != SSD_OK) return r;
  if (c->phase != PH_IDLE) return fail(c, SSD_ERR_STATE, "a round is in flight");
  if ((r = read_state(c)) != SSD_OK) return r;
  if (c->h_st->n + 1 > c->cfg.max_seq) return fail(c, SSD_ERR_CAPACITY, "max_seq exceeded");
  Range nv("ssd layer_features");
  cudaStream_t s = c->stream;
  // one autoregressive step with the exit head after every layer >= min_layer
  c->mmax = 1;
  if ((r = enq_begin(c, BEGIN_AR, s)) != SSD_OK) { c->mmax = 0; return r; }
  for (int l = 0; l < L && r == SSD_OK; ++l) {
    r = enq_layer(c, l, s);
    if (r == SSD_OK && l >= min_layer && l < L - 1)
      r = enq_lmhead(c, c->fstats + l, nullptr, nullptr, -1, s);
  }
  if (r == SSD_OK) r = enq_lmhead(c, c->vstats, nullptr, nullptr, 2, s);
  if (r == SSD_OK)
    r = note(c, launch_ar_end(c->st, c->tokens, c->vstats, 0, c->pol.temperature, 0, s, c->pdl),
             "ar_end");
  c->mmax = 0;
  if (r != SSD_OK) return r;
  const int nl = L - min_layer;
  CK(cudaMemcpyAsync(c->fstats + (L - 1), c->vstats, sizeof(RowStats), cudaMemcpyDeviceToDevice,
                     s));
  if ((r = note(c, launch_exit_features(c->fstats + min_layer, nl, c->ffeat, s),
                "exit_features")) != SSD_OK)
    return r;
  CK(cudaMemcpyAsync(c->h_ffeat, c->ffeat, (size_t)3 * nl * 4, cudaMemcpyDeviceToHost, s));
  if ((r = read_state(c)) != SSD_OK) return r;
  for (int i = 0; i < nl; ++i) {
    memcpy(&top1[i], &c->h_ffeat[i], 4);
    top_prob[i] = c->h_ffeat[nl + i];
    gap[i] = c->h_ffeat[2 * nl + i];
  }
  return SSD_OK;
}

ssd_status ssd_rewind(ssd_ctx* c, int32_t n) {
  if (!c) return SSD_ERR_INVALID_ARG;
  if (c->phase == PH_NONE) return fail(c, SSD_ERR_STATE, "no prefill");
  ssd_status r = read_state(c);
  if (r != SSD_OK) return r;
  if (n < 2 || n > c->h_st->n) return fail(c, SSD_ERR_INVALID_ARG, "rewind target out of range");
  DevState* hs = c->h_st;
  hs->n = n;
  hs->j = hs->d = hs->stop = 0;
  // the next pass writes position n - 1 and on: incomplete K/V before it stay
  if (c->lossy_from >= 0 && n - 1 <= c->lossy_from) c->lossy_from = -1;
  CK(cudaMemcpyAsync(c->st, hs, sizeof(DevState), cudaMemcpyHostToDevice, c->stream));
  c->phase = PH_IDLE;
  return wait_stream(c);
}

ssd_status ssd_get_tokens(ssd_ctx* c, int32_t* out, int32_t cap, int32_t* n_out) {
  if (!c || !n_out) return SSD_ERR_INVALID_ARG;
  ssd_status r = read_state(c);
  if (r != SSD_OK) return r;
  const int n = c->phase == PH_NONE ? 0 : c->h_st->n;
  *n_out = n;
  if (out && cap > 0 && n > 0) {
    const int k = n < cap ? n : cap;
    CK(cudaMemcpyAsync(c->h_tok, c->tokens, (size_t)k * 4, cudaMemcpyDeviceToHost, c->stream));
    if ((r = wait_stream(c)) != SSD_OK) return r;
    memcpy(out, c->h_tok, (size_t)k * 4);
  }
  return SSD_OK;
}

ssd_status ssd_profile_decode(ssd_ctx* c, int32_t n_steps, ssd_kernel_times* out) {
  if (!c || !out || n_steps <= 0) return SSD_ERR_INVALID_ARG;
  ssd_status r = ensure_policy(c);
  if (r != SSD_OK) return r;
  if (c->phase != PH_IDLE) return fail(c, SSD_ERR_STATE, "a round is in flight");
  if ((r = read_state(c)) != SSD_OK) return r;
  const int n0 = c->h_st->n;
  if (n0 + n_steps > c->cfg.max_seq) return fail(c, SSD_ERR_CAPACITY, "max_seq exceeded");
  memset(out, 0, sizeof(*out));
  DevState saved = *c->h_st;
  c->profiling = true;
  c->prof_events.clear();
  const ssd_config& g = c->cfg;
  std::vector<double> kv_bytes;
  for (int i = 0; i < n_steps; ++i) {
    r = b_ar(c, c->stream);
    if (r != SSD_OK) break;
    // attention reads K/V of positions [0, pos] and writes one position per layer
    kv_bytes.push_back(2.0 * 2.0 * g.n_kv_heads * g.head_dim * (double)(n0 + i + 1));
  }
  c->profiling = false;
  if (r == SSD_OK) r = wait_stream(c);
  const double w_qkv = 2.0 * qkv_rows(g) * g.d_model;
  const double w_o = 2.0 * g.d_model * g.n_heads * g.head_dim;
  const double w_gu = 2.0 * 2.0 * g.ffn_dim * g.d_model;
  const double w_dn = 2.0 * g.d_model * g.ffn_dim;
  const double w_lm = 2.0 * g.vocab * g.d_model;
  int step = -1, layer_in_step = 0;
  for (auto& pe : c->prof_events) {
    const int cls = pe.first;
    float ms = 0.f;
    if (r == SSD_OK) cudaEventElapsedTime(&ms, pe.second.first, pe.second.second);
    if (cls == 6 && layer_in_step == 0) step++;
    out->ms[cls] += ms;
    out->launches[cls]++;
    double b = 0.0;
    switch (cls) {
      case 0: b = w_qkv; break;
      case 1: b = step >= 0 && step < (int)kv_bytes.size() ? kv_bytes[step] : 0.0; break;
      case 2: b = w_o; break;
      case 3: b = w_gu; break;
      case 4: b = w_dn; break;
      case 5: b = w_lm; break;
      default: b = 0.0;
    }
    out->bytes[cls] += b;
    layer_in_step = (cls == 6) ? (layer_in_step ? 0 : 1) : layer_in_step;
    cudaEventDestroy(pe.second.first);
    cudaEventDestroy(pe.second.second);
  }
  c->prof_events.clear();
  for (int k = 0; k < 8; ++k)
    if (out->launches[k]) {
      out->ms[k] /= (double)out->launches[k];
      out->bytes[k] /= (double)out->launches[k];
    }
  if (r != SSD_OK) return r;
  // restore the committed state
  saved.j = saved.d = saved.stop = 0;
  *c->h_st = saved;
  CK(cudaMemcpyAsync(c->st, c->h_st, sizeof(DevState), cudaMemcpyHostToDevice, c->stream));
  return wait_stream(c);
}

namespace {

// ssd_profile_kernels: the launches of one kernel class over every layer of
// an autoregressive step (the LM head: n_layers launches of it), enqueued as
// the step's graph enqueues them, so that consecutive launches overlap
// through programmatic dependent launch as they do in the step.
ssd_status b_prof_class(ssd_ctx* c, cudaStream_t s) {
  c->mmax = 1;
  ssd_status r = SSD_OK;
  const int cls = c->prof_graph_cls;
  for (int l = 0; l < c->cfg.n_layers && r == SSD_OK; ++l) {
    switch (cls) {
      case 0: r = enq_norm_gemv(c, EPI_STORE, qkv_args(c, l), s, "qkv"); break;
      case 1: r = note(c, launch_attention(attn_args(c, l), s, c->pdl), "attention"); break;
      case 2: r = note(c, launch_gemv(IN_BF16, EPI_RESID, oproj_args(c, l), s, c->pdl), "o_proj"); break;
      case 3: r = enq_norm_gemv(c, EPI_SWIGLU, gateup_args(c, l), s, "gate_up"); break;
      case 4: r = note(c, launch_gemv(IN_BF16, EPI_RESID, down_args(c, l), s, c->pdl), "down"); break;
      case 5: r = enq_lmhead(c, c->vstats, nullptr, nullptr, 2, s); break;
      default:   // attention and the o_proj that consumes its output, as the step pairs them
        r = note(c, launch_attention(attn_args(c, l), s, c->pdl), "attention");
        if (r == SSD_OK)
          r = note(c, launch_gemv(IN_BF16, EPI_RESID, oproj_args(c, l), s, c->pdl), "o_proj");
        break;
    }
  }
  c->mmax = 0;
  return r;
}

}  // namespace

ssd_status ssd_profile_kernels(ssd_ctx* c, int32_t reps, ssd_kernel_times* out) {
  if (!c || !out || reps <= 0) return SSD_ERR_INVALID_ARG;
  if (c->fp32) return fail(c, SSD_ERR_INVALID_ARG, "kernel profile of bf16 models only");
  ssd_status r = ensure_policy(c);
  if (r != SSD_OK) return r;
  if (c->phase != PH_IDLE) return fail(c, SSD_ERR_STATE, "a round is in flight");
  if ((r = read_state(c)) != SSD_OK) return r;
  const int n0 = c->h_st->n;
  if (n0 + 1 > c->cfg.max_seq) return fail(c, SSD_ERR_CAPACITY, "max_seq exceeded");
  memset(out, 0, sizeof(*out));
  const DevState saved = *c->h_st;
  const ssd_config& g = c->cfg;
  const int L = g.n_layers;
  const double bytes[8] = {2.0 * qkv_rows(g) * g.d_model,
                           2.0 * 2.0 * g.n_kv_heads * g.head_dim * (double)n0,
                           2.0 * g.d_model * g.n_heads * g.head_dim,
                           2.0 * 2.0 * g.ffn_dim * g.d_model,
                           2.0 * g.d_model * g.ffn_dim,
                           2.0 * g.vocab * g.d_model,
                           0.0,
                           2.0 * 2.0 * g.n_kv_heads * g.head_dim * (double)n0 +
                               2.0 * g.d_model * g.n_heads * g.head_dim};
  // the pass shape of an autoregressive step: one row at position n - 1
  if ((r = enq_begin(c, BEGIN_AR, c->stream)) != SSD_OK) return r;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  for (int cls = 0; cls < 8 && r == SSD_OK; ++cls) {
    if (cls == 6) continue;   // the control kernels are timed by ssd_profile_decode only
    Graph G;
    c->prof_graph_cls = cls;
    if ((r = build_graph(c, G, b_prof_class)) != SSD_OK) break;
    cudaError_t e = cudaGraphLaunch(G.exec, c->stream);   // warm-up
    if (e == cudaSuccess) e = cudaEventRecord(e0, c->stream);
    for (int i = 0; i < reps && e == cudaSuccess; ++i) e = cudaGraphLaunch(G.exec, c->stream);
    if (e == cudaSuccess) e = cudaEventRecord(e1, c->stream);
    if (e != cudaSuccess) {
      r = fail(c, SSD_ERR_CUDA, std::string("profile: ") + cudaGetErrorString(e));
      break;
    }
    if ((r = wait_stream(c)) != SSD_OK) break;
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    out->ms[cls] = ms / ((double)reps * L);
    out->bytes[cls] = bytes[cls];
    out->launches[cls] = cls == 5 ? 1 : cls == 7 ? 0 : L;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (r != SSD_OK) return r;
  // restore the committed state (the profile wrote only scratch buffers and
  // the cache row of the pending position, which the next pass rewrites)
  *c->h_st = saved;
  CK(cudaMemcpyAsync(c->st, c->h_st, sizeof(DevState), cudaMemcpyHostToDevice, c->stream));
  return wait_stream(c);
}

ssd_status ssd_swift_generate(ssd_ctx* c, const ssd_swift_params* pp, int32_t n_tokens,
                              int32_t* out, uint64_t* trace_masks, float* trace_scores,
                              int32_t* trace_best, int32_t trace_cap, ssd_swift_report* rep) {
  if (!c) return SSD_ERR_INVALID_ARG;
  if (c->fp32) return fail(c, SSD_ERR_INVALID_ARG, "SWIFT optimisation needs a bf16 model");
  if (!pp || n_tokens < 0 || trace_cap < 0) return fail(c, SSD_ERR_INVALID_ARG, "swift arguments");
  const ssd_swift_params P = *pp;
  const int L = c->cfg.n_layers;
  if (P.lo_layer < 0 || P.lo_layer >= L || P.skip_count < 1 || P.skip_count > L - P.lo_layer ||
      P.window < 1 || P.candidates < 1 || P.candidates > 256 || P.max_steps < 0 || P.patience < 1)
    return fail(c, SSD_ERR_INVALID_ARG, "swift parameters out of range");
  ssd_status r = ensure_policy(c);
  if (r != SSD_OK) return r;
  if (c->pol.mode != SSD_MODE_SKIP) return fail(c, SSD_ERR_STATE, "swift needs a skip-mode policy");
  if (c->phase != PH_IDLE) return fail(c, SSD_ERR_STATE, "a round is in flight");
  if ((int64_t)P.candidates * P.window > c->cfg.max_score_rows)
    return fail(c, SSD_ERR_CAPACITY, "candidates * window exceeds max_score_rows");
  if ((r = read_state(c)) != SSD_OK) return r;
  const int n_start = c->h_st->n;
  if (n_start + n_tokens + c->pol.d_max + 1 > c->cfg.max_seq)
    return fail(c, SSD_ERR_CAPACITY, "n_tokens + d_max + 1 exceeds the KV capacity");
  if (rep) memset(rep, 0, sizeof(*rep));
  const auto t_begin = std::chrono::steady_clock::now();

  // SplitMix64 (Steele, Lea, Flood, OOPSLA 2014)
  uint64_t rng = P.seed;
  auto next = [&rng]() {
    rng += 0x9E3779B97F4A7C15ull;
    uint64_t z = rng;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  };
  const int span = L - P.lo_layer;
  auto propose = [&]() {
    std::vector<int> pool(span);
    for (int i = 0; i < span; ++i) pool[i] = P.lo_layer + i;
    for (int i = 0; i < P.skip_count; ++i) {
      const int j = i + (int)(next() % (uint64_t)(span - i));
      std::swap(pool[i], pool[j]);
    }
    pool.resize(P.skip_count);
    std::sort(pool.begin(), pool.end());
    return pool;
  };
  std::vector<int> inc(P.skip_count);
  for (int i = 0; i < P.skip_count; ++i) inc[i] = P.lo_layer + (2 * i + 1) * span / (2 * P.skip_count);
  ssd_policy pol = c->pol;
  auto apply = [&](const std::vector<int>& set) {
    memset(pol.skip_mask, 0, sizeof(pol.skip_mask));
    memset(pol.skip_attn_mask, 0, sizeof(pol.skip_attn_mask));
    memset(pol.skip_mlp_mask, 0, sizeof(pol.skip_mlp_mask));
    for (int l : set) pol.skip_mask[l >> 6] |= 1ull << (l & 63);
    return ssd_set_policy(c, &pol);
  };
  if ((r = apply(inc)) != SSD_OK) return r;

  const int K = P.candidates;
  std::vector<uint64_t> masks((size_t)K * 4);
  std::vector<float> scores(K);
  std::vector<std::vector<int>> cands(K);
  bool optimizing = true;
  int steps = 0, unchanged = 0, stopped_by = 0, got = 0;
  double opt_seconds = 0.0;
  ssd_stats st{};
  while (got < n_tokens) {
    if ((r = run_draft(c, &st)) != SSD_OK) return r;
    const int d = c->pol.d_max == 0 ? 0 : c->h_st->d;
    if ((r = run_verify(c, &st)) != SSD_OK) return r;
    if ((r = replay(c, c->g_accept)) != SSD_OK) return r;
    CK(cudaEventRecord(c->t1, c->stream));
    if ((r = read_state(c)) != SSD_OK) return r;
    {
      float ms = 0.f;
      cudaEventElapsedTime(&ms, c->t0, c->t1);
      st.verify_ms += ms;
    }
    c->phase = PH_IDLE;
    const int ne = c->h_st->n_emitted;
    for (int i = 0; i < ne && got < n_tokens; ++i, ++got)
      if (out) out[got] = c->h_st->emitted[i];
    st.rounds++;
    st.drafted += d;
    st.accepted += c->h_st->accepted;
    st.emitted += ne;
    if (tree_on(c)) {
      st.side_rows += c->h_st->n_sib;
      st.side_accepted += c->h_st->sib_acc >= 0 ? 1 : 0;
    }
    const int generated = c->h_st->n - n_start;
    if (!optimizing || generated < P.window + 1 || generated >= n_tokens) continue;
    // one optimisation step: the incumbent, then K-1 proposals
    const auto t0 = std::chrono::steady_clock::now();
    cands[0] = inc;
    for (int k = 1; k < K; ++k) cands[k] = propose();
    std::fill(masks.begin(), masks.end(), 0ull);
    for (int k = 0; k < K; ++k)
      for (int l : cands[k]) masks[(size_t)k * 4 + (l >> 6)] |= 1ull << (l & 63);
    if ((r = ssd_score_masks(c, masks.data(), K, P.window, scores.data(), nullptr)) != SSD_OK)
      return r;
    int best = 0;
    for (int k = 1; k < K; ++k)
      if (scores[k] > scores[best]) best = k;
    if (steps < trace_cap) {
      if (trace_masks) memcpy(trace_masks + (size_t)steps * K * 4, masks.data(), masks.size() * 8);
      if (trace_scores) memcpy(trace_scores + (size_t)steps * K, scores.data(), (size_t)K * 4);
      if (trace_best) trace_best[steps] = best;
    }
    ++steps;
    if (best == 0) {
      ++unchanged;
    } else {
      unchanged = 0;
      inc = cands[best];
      if ((r = apply(inc)) != SSD_OK) return r;
    }
    if (scores[best] > P.target) stopped_by = 1;
    else if (steps >= P.max_steps) stopped_by = 2;
    else if (unchanged >= P.patience) stopped_by = 3;
    if (stopped_by) optimizing = false;
    opt_seconds += std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  }
  if (c->h_st->n != n_start + n_tokens) {   // the last round may emit past the budget
    const int32_t nn = n_start + n_tokens;
    CK(cudaMemcpyAsync(&c->st->n, &nn, 4, cudaMemcpyHostToDevice, c->stream));
    if ((r = read_state(c)) != SSD_OK) return r;
  }
  if (rep) {
    rep->steps = steps;
    rep->stopped_by = stopped_by;
    for (int l : inc) rep->final_mask[l >> 6] |= 1ull << (l & 63);
    rep->rounds = st.rounds;
    rep->drafted = st.drafted;
    rep->accepted = st.accepted;
    rep->emitted = st.emitted;
    rep->opt_seconds = opt_seconds;
    rep->total_seconds =
        std::chrono::duration<double>(std::chrono::steady_clock::now() - t_begin).count();
  }
  return SSD_OK;
}

ssd_status ssd_debug_canaries(ssd_ctx* c, int32_t* checked_out, int32_t* bad_out) {
  if (!c || !checked_out || !bad_out) return SSD_ERR_INVALID_ARG;
  *checked_out = (int32_t)c->canaries.size();
  *bad_out = 0;
  std::vector<unsigned char> h(kCanaryBytes);
  for (unsigned char* g : c->canaries) {
    CK(cudaMemcpyAsync(h.data(), g, kCanaryBytes, cudaMemcpyDeviceToHost, c->stream));
    const ssd_status r = wait_stream(c);
    if (r != SSD_OK) return r;
    for (unsigned char b : h) *bad_out += b != kCanaryByte;
  }
  return SSD_OK;
}

ssd_status ssd_debug_fail_alloc(int32_t n) {
  g_fail_alloc = n < 0 ? -1 : n;
  return SSD_OK;
}

ssd_status ssd_set_device_loop(ssd_ctx* c, int32_t enable, int32_t* active_out) {
  if (!c) return SSD_ERR_INVALID_ARG;
  c->use_loop = enable != 0;
  if (active_out) *active_out = c->use_loop && c->g_loop.exec ? 1 : 0;
  // the reason the loop is unavailable, for ssd_last_error
  if (c->use_loop && !c->g_loop.exec) c->err = "device loop unavailable: " + c->loop_err;
  return SSD_OK;
}

ssd_status ssd_set_timeout_ms(ssd_ctx* c, int32_t ms) {
  if (!c || ms <= 0) return SSD_ERR_INVALID_ARG;
  c->timeout_ms = ms;
  return SSD_OK;
}

const char* ssd_last_error(const ssd_ctx* c) {
  if (!c) {
    snprintf(g_static_err, sizeof(g_static_err), "null context");
    return g_static_err;
  }
  return c->err.c_str();
}

ssd_status ssd_score_masks(ssd_ctx* c, const uint64_t* masks, int32_t K, int32_t N,
                           float* matchness_out, int32_t* best_out) {
  if (!c) return SSD_ERR_INVALID_ARG;
  if (c->fp32) return fail(c, SSD_ERR_INVALID_ARG, "mask scoring needs a bf16 model");
  if (!masks || K < 1 || K > 256 || N < 1 || !matchness_out)
    return fail(c, SSD_ERR_INVALID_ARG, "score_masks arguments");
  ssd_status r = ensure_policy(c);
  if (r != SSD_OK) return r;
  if (c->phase != PH_IDLE) return fail(c, SSD_ERR_STATE, "a round is in flight");
  if ((int64_t)K * N > c->cfg.max_score_rows)
    return fail(c, SSD_ERR_CAPACITY, "K*N exceeds max_score_rows");
  if ((r = read_state(c)) != SSD_OK) return r;
  const int n = c->h_st->n;
  if (N + 2 > n) return fail(c, SSD_ERR_CAPACITY, "window longer than the committed context");
  Range nv("ssd score_masks");
  if ((r = enq_score(c, masks, K, N, n - N - 1)) != SSD_OK) return r;
  CK(cudaMemcpyAsync(c->h_counts, c->sc_counts, (size_t)K * sizeof(int32_t), cudaMemcpyDeviceToHost,
                     c->stream));
  if ((r = read_state(c)) != SSD_OK) return r;
  int best = 0;
  for (int k = 0; k < K; ++k) {
    const int cnt = c->h_counts[c->sc_owner[k]];
    matchness_out[k] = (float)cnt / (float)N;
    if (cnt > c->h_counts[c->sc_owner[best]]) best = k;
  }
  if (best_out) *best_out = best;
  return SSD_OK;
}

}  // extern "C"
