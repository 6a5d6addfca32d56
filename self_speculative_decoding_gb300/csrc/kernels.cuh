// Kernel launch interfaces shared by the context runtime and the op entry points.
#pragma once

#include "common.cuh"

namespace ssd {

enum InMode { IN_BF16 = 0, IN_NORM = 1 };
enum EpiMode { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_LMHEAD = 3 };

// Arguments of the small-M GEMV family: y = W act over M <= 16 rows.
struct LinearArgs {
  const bf16* W0 = nullptr;   // [R][K] row-major
  const bf16* W1 = nullptr;   // second matrix of the SwiGLU pair (up), [R][K]
  int R = 0, K = 0;
  // input
  const bf16* act = nullptr;  // IN_BF16: [M][K]
  const float* x = nullptr;   // IN_NORM: fp32 residual [M][K]
  const float* ss = nullptr;  // IN_NORM: sum-of-squares partials [M][K/16]
  const float* gain = nullptr;
  float eps = 1e-5f;
  int m_max = 0;           // most rows any launch of this GEMV carries (0: M_static, or 16 with M_dev)
  int M_static = 1;
  const int32_t* M_dev = nullptr;
  // 1: the pass's rows may not fit the per-CTA activation stage.  A bf16-input
  // projection whose CTAs own whole row groups then streams each CTA's groups
  // in batches, K window by K window, and loads each activation window once
  // per batch (the same sums in the same order as the staged layout).  Set by
  // the caller from the pass's static row bound; launch_gemv sets it for a
  // static M that does not fit.
  int wide = 0;
  // outputs
  float* y = nullptr;         // EPI_STORE [M][R]
  float* xres = nullptr;      // EPI_RESID [M][R], read and written
  float* ss_out = nullptr;    // EPI_RESID [M][R/16]
  bf16* u = nullptr;          // EPI_SWIGLU [M][R]
  // split-row-group combine scratch (see gemv_scratch); counters start at
  // zero and are returned to zero by the kernel
  float* part = nullptr;
  unsigned* counter = nullptr;
  float* rec = nullptr;       // EPI_LMHEAD summary records
  int* err = nullptr;         // set non-zero if a bulk copy never completed
  int* err_val = nullptr;     // debug builds: the value a failed bounds check saw
  // EPI_LMHEAD
  float* logits = nullptr;    // [slot + M][R] (nullable)
  RowStats* stats = nullptr;  // [slot + M]
  const int32_t* slot_dev = nullptr;
  float temperature = 0.f;    // > 0: the summary includes lse of z / T
  int sample = 0;             // 1: also draw a Gumbel-max sample of softmax(z / T)
  uint64_t seed = 0;
  int round_static = 0;
  const int32_t* round_dev = nullptr;
  int sample_stream = 0;
  int pos0_static = 0;
  const int32_t* pos0_dev = nullptr;
};

// Scratch one launch needs for a matrix of R rows and depth K (floats of
// partial sums, counters, LM-head records).  Consecutive launches on one
// stream may share the same scratch.
struct GemvScratch {
  size_t part_floats, counters, rec_floats;
};
GemvScratch gemv_scratch(int R, int K, int epi);

// W0 / W1 must be in the packed unit layout written by launch_pack.
cudaError_t launch_gemv(int in_mode, int epi, const LinearArgs& a, cudaStream_t st, bool pdl);

// Rows whose activations (K columns) fit the per-CTA stage at once.
int gemv_stage_rows(int K);

// out[m][k] = bf16(rmsnorm(x_m)[k] * gain[k]) for the pass's rows, computed
// exactly as the norm-fused GEMV input computes it (for passes whose rows do
// not fit the stage: the projection then reads bf16 activations).
cudaError_t launch_norm_rows(const float* x, const float* ss, const float* gain, float eps,
                             int M_static, const int32_t* M_dev, int K, bf16* out, cudaStream_t st,
                             bool pdl);

// Row-major W [R][K] -> packed 16x32 units in tensor-core fragment order.
cudaError_t launch_pack(const bf16* src, bf16* dst, int R, int K, cudaStream_t st);

// Attention over the KV cache for the rows of a pass (see ssd_op_attention).
struct AttnArgs {
  const float* qkv = nullptr;  // [M][ld_qkv]
  int ld_qkv = 0;
  int M_static = 1;
  const int32_t* M_dev = nullptr;
  int pos0_static = 0;
  const int32_t* pos0_dev = nullptr;
  bf16* kc = nullptr;          // [Hkv][max_seq][dh]
  bf16* vc = nullptr;
  int max_seq = 0;
  int H = 0, Hkv = 0, dh = 0;
  const float2* rope = nullptr;  // [max_seq][dh/2] (cos, sin)
  bf16* out = nullptr;         // [M][H dh]
  float* part = nullptr;       // [Hkv][max_seq/kAttnChunk][G*16][dh+2]
  unsigned* counters = nullptr;  // [Hkv]
  int* err = nullptr;          // set to 1 if a bulk copy never completed
  int* err_val = nullptr;      // debug builds: the value a failed bounds check saw
  float scale = 1.f;
  // Side rows (dynamic verification): the pass's last *ns_dev rows are
  // sibling candidates at positions side_pos[i] (not pos0 + m).  A side row
  // attends to the cache and chain keys before its position plus its own
  // key; its K/V go to side slot side0 + i of this layer instead of the
  // cache.  ns_dev NULL: no side rows.
  const int32_t* ns_dev = nullptr;
  const int32_t* side_pos = nullptr;  // [kMaxSide]
  const int32_t* side0 = nullptr;
  bf16* ks = nullptr;                 // [Hkv][kMaxSide][dh]
  bf16* vs = nullptr;
};

int attn_grid(const AttnArgs& a);
size_t attn_smem(const AttnArgs& a);
size_t attn_part_floats(int Hkv, int H, int dh, int max_seq);
// Sets the kernel's dynamic shared-memory limit for this head geometry
// (call once before launching or capturing).
cudaError_t attn_prepare(const AttnArgs& a);
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st, bool pdl);

// RoPE (cos, sin) table [n_pos][half], angles pos * theta^(-2i/dh) evaluated
// in double precision and rounded to fp32.
cudaError_t launch_rope_table(float2* tab, int n_pos, int half, double theta, cudaStream_t s);

// ---------------------------------------------------------------------------
// fp32 models (SSD_DTYPE_FP32): the same steps with fp32 weights (row-major,
// not packed), fp32 activations, K/V and logits, and no rounding (fp32.cu).

struct LinearArgs32 {
  const float* W0 = nullptr;  // [R][K] row-major
  const float* W1 = nullptr;  // EPI_SWIGLU: the up matrix
  int R = 0, K = 0;
  const float* act = nullptr; // IN_BF16 (plain input) [M][K]
  const float* x = nullptr;   // IN_NORM [M][K]
  const float* gain = nullptr;
  float eps = 1e-5f;
  int M_static = 1;
  const int32_t* M_dev = nullptr;
  float* y = nullptr;         // EPI_STORE [row0 + M][R]
  const int32_t* row0_dev = nullptr;
  float* xres = nullptr;      // EPI_RESID [M][R]
  float* u = nullptr;         // EPI_SWIGLU [M][R]
};
cudaError_t launch_gemv32(int in_mode, int epi, const LinearArgs32& a, cudaStream_t st, bool pdl);

// Row summaries (RowStats) of logits rows [slot + m], m < M.
struct LmSummaryArgs32 {
  const float* logits = nullptr;
  int V = 0;
  int M_static = 1;
  const int32_t* M_dev = nullptr;
  const int32_t* slot_dev = nullptr;
  RowStats* stats = nullptr;
  float temperature = 0.f;
  int sample = 0;
  uint64_t seed = 0;
  int round_static = 0;
  const int32_t* round_dev = nullptr;
  int stream = 0;
  int pos0_static = 0;
  const int32_t* pos0_dev = nullptr;
};
cudaError_t launch_lm_summary32(const LmSummaryArgs32& a, cudaStream_t st, bool pdl);

struct AttnArgs32 {
  const float* qkv = nullptr;  // [M][ld_qkv]
  int ld_qkv = 0;
  int M_static = 1;
  const int32_t* M_dev = nullptr;
  int pos0_static = 0;
  const int32_t* pos0_dev = nullptr;
  float* kc = nullptr;         // [Hkv][max_seq][dh]
  float* vc = nullptr;
  int max_seq = 0;
  int H = 0, Hkv = 0, dh = 0;
  const float2* rope = nullptr;
  float* out = nullptr;        // [M][H dh]
  float scale = 1.f;
};
size_t attn32_smem(int dh, int max_seq);
cudaError_t attn32_prepare(int dh, int max_seq);
cudaError_t launch_attention32(const AttnArgs32& a, cudaStream_t st, bool pdl);

// Embedding / pass set-up ("begin") kernel modes.
enum BeginMode { BEGIN_TOKENS = 0, BEGIN_AR = 1, BEGIN_DRAFT = 2, BEGIN_EXTRA = 3, BEGIN_VERIFY = 4 };

struct BeginArgs {
  int mode = BEGIN_TOKENS;
  DevState* st = nullptr;
  const int32_t* tokens = nullptr;   // committed tokens [max_seq]
  const int32_t* toks_in = nullptr;  // BEGIN_TOKENS: this pass's tokens
  int M = 1, pos0 = 0;               // BEGIN_TOKENS
  int reset_round = 0;               // BEGIN_TOKENS: set round = 0 (prefill)
  const bf16* embed = nullptr;       // [V][D]
  const float* embed32 = nullptr;    // fp32 models: [V][D] fp32 (embed unused)
  int D = 0;
  float* x = nullptr;                // [16][D]
  float* ss = nullptr;               // [16][D/16]
  const float* bx = nullptr;         // boundary states [16][D] (BEGIN_VERIFY)
  const float* bss = nullptr;
  const float* bxs = nullptr;        // siblings' boundary states [kMaxSide][D]
  const float* bsss = nullptr;
};
cudaError_t launch_begin(const BeginArgs& a, cudaStream_t st, bool pdl);

// Boundary buffers of the draft / extra passes: the chain row's state goes
// to bx slot j (draft) or d (extra pass), a side row's to bxs at its sibling
// index; the pass then continues with the chain row alone.
struct SaveArgs {
  DevState* st = nullptr;
  int use_d = 0;
  const float* x = nullptr;
  const float* ss = nullptr;
  float* bx = nullptr;
  float* bss = nullptr;
  float* bxs = nullptr;
  float* bsss = nullptr;
  int D = 0;
};
cudaError_t launch_save_boundary(const SaveArgs& a, cudaStream_t s, bool pdl);

// Draft-step control: the confidence stop (tau) and, for dynamic
// verification, the sibling rule (tree_tau, tree_max).
struct DraftEndArgs {
  DevState* st = nullptr;
  const RowStats* dstats = nullptr;
  float tau = 0.f, temperature = 0.f;
  float tree_tau = 0.f;
  int tree_max = 0;
};
cudaError_t launch_draft_end(const DraftEndArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_ar_end(DevState* st, int32_t* tokens, const RowStats* vstats, int row_from_M,
                          float temperature, int reset, cudaStream_t s, bool pdl);
cudaError_t launch_accept_greedy(DevState* st, int32_t* tokens, const RowStats* vstats,
                                 cudaStream_t s, bool pdl);
// Device-side generation loop (one graph launch per ssd_generate): the
// conditions of its nodes, set by one-thread kernels from the decoding state.
enum LoopCond {
  LOOP_DRAFT_FIRST = 0,  // enter the draft loop: d_max > 0
  LOOP_DRAFT_NEXT = 1,   // another draft step: no stop and j < d_max
  LOOP_EXTRA = 2,        // the extra pass: the draft loop ended without a stop
  LOOP_WIDE = 3,         // the wide verify graph: d + 1 + siblings > narrow rows
  LOOP_ROUND = 4,        // another round: n < target, n <= limit, no device error
  LOOP_NOP = 5,          // sets nothing (a plain launch that orders the graph)
};
cudaError_t launch_loop_cond(DevState* st, cudaGraphConditionalHandle h, int what, int arg,
                             int limit, cudaStream_t s, bool pdl);

// After a greedy acceptance that took a sibling: its K/V of every layer
// (side slot sib_acc) into the cache at sib_pos.  kc / vc [L][Hkv][max_seq][dh],
// ks / vs [L][Hkv][kMaxSide][dh].  No-op when no sibling was taken.
cudaError_t launch_side_commit(const DevState* st, bf16* kc, bf16* vc, const bf16* ks,
                               const bf16* vs, int L, int Hkv, int max_seq, int dh,
                               cudaStream_t s, bool pdl);

struct AcceptArgs {
  const float* P = nullptr;       // [d+1][V]
  const float* Q = nullptr;       // [d][V]
  const int32_t* drafts = nullptr;
  int d_static = 0;
  const RowStats* pstats = nullptr;  // nullable: lse_t of P rows
  const RowStats* qstats = nullptr;  // nullable: lse_t of Q rows
  int V = 0;
  float temperature = 1.f;
  uint64_t seed = 0;
  int round_static = 0;
  int n_static = 0;
  DevState* st = nullptr;         // state-driven mode when not NULL
  int32_t* tokens = nullptr;      // state-driven: committed tokens
  int32_t* emitted = nullptr;     // op mode outputs
  int32_t* n_emitted = nullptr;
};
cudaError_t launch_accept_stochastic(const AcceptArgs& a, cudaStream_t s, bool pdl);

cudaError_t launch_philox(const uint32_t* ctr, int count, uint64_t key, uint32_t* out,
                          cudaStream_t s);

// ---------------------------------------------------------------------------
// Batched candidate-mask scoring: many-row projections on the tensor cores
// and the scoring forward's other steps (gemm.cu, score.cu).

enum GemmEpi { GEMM_STORE = 0, GEMM_RESID = 1, GEMM_SWIGLU = 2, GEMM_ARGMAX = 3 };

// out[t][r] = sum_k act[t][k] W[r][k] for T rows; W (and W1, the up matrix of
// a SwiGLU pair) in the packed unit layout of launch_pack.
struct GemmArgs {
  const bf16* W0 = nullptr;
  const bf16* W1 = nullptr;
  int R = 0, K = 0, T = 0;
  const bf16* act = nullptr;           // [T][K] in the packed unit layout (packed_off), T padded to 16
  int epi = GEMM_STORE;
  float* y = nullptr;                  // GEMM_STORE [T][R]
  float* x = nullptr;                  // GEMM_RESID: x[rowmap[t]][r] += out[t][r] (16-byte aligned)
  const int32_t* rowmap = nullptr;     // nullable: identity; distinct rows
  bf16* u = nullptr;                   // GEMM_SWIGLU [T][R]: silu(gate) * up
  int u_packed = 0;                    // 1: u in the packed unit layout
  int fast_silu = 0;                   // 1: SiLU with the fast exponential and division
  unsigned long long* best = nullptr;  // GEMM_ARGMAX [T]: atomic max of (value, -index) keys, zero before
  int* err = nullptr;                  // set non-zero if a bounded wait gave up (nullable)
};
cudaError_t launch_gemm_rows(const GemmArgs& a, cudaStream_t s);
// idx[t] = the index of argmax key best[t] (-1 for a row that saw no value)
cudaError_t launch_argmax_index(const unsigned long long* best, int T, int32_t* idx,
                                cudaStream_t s);

struct ScoreAttnArgs {
  const bf16* q = nullptr;    // [T][H][dh] compact rows (RoPE applied)
  const bf16* kc = nullptr;   // the layer's shared cache [Hkv][max_seq][dh]
  const bf16* vc = nullptr;
  const bf16* sk = nullptr;   // window K/V [K * N][Hkv][dh] by physical row
  const bf16* sv = nullptr;
  const int32_t* cand = nullptr;  // [n_active] candidates that keep the layer
  int N = 0, split = 0, max_seq = 0, H = 0, Hkv = 0, dh = 0;
  float scale_log2 = 0.f;     // log2(e) / sqrt(dh)
  bf16* out = nullptr;        // [T][H dh]
  int out_packed = 0;         // 1: out in the packed unit layout (packed_off)
  int w_rows = 0;             // rows of sk / sv
  int* err = nullptr;         // set non-zero if a bounded wait gave up (nullable)
};
cudaError_t launch_score_attn(const ScoreAttnArgs& a, int n_active, cudaStream_t s);
// the tensor-core form (dh 128, N a multiple of 8 up to 128)
bool score_attn_tc_ok(const ScoreAttnArgs& a);
cudaError_t launch_score_attn_tc(const ScoreAttnArgs& a, int n_active, cudaStream_t s);
size_t score_attn_smem(int dh);
cudaError_t launch_score_embed(const bf16* embed, const int32_t* tokens, int split, int N, int rows,
                               int D, float* x, cudaStream_t s);
// out in the packed unit layout (packed_off)
cudaError_t launch_score_norm(const float* x, const int32_t* map, const float* gain, float eps,
                              int T, int D, bf16* out, cudaStream_t s);
// dst = src [T][K] row-major in the packed unit layout, rows T .. 16-padded zero
cudaError_t launch_pack_act(const bf16* src, int T, int K, bf16* dst, cudaStream_t s);
// map nullable (identity); kc / vc nullable: also store k, v into that cache
cudaError_t launch_score_rope(const float* qkv, int T, const int32_t* map, int N, int split, int H,
                              int Hkv, int dh, const float2* rope, bf16* q, bf16* sk, bf16* sv,
                              bf16* kc, bf16* vc, int max_seq, cudaStream_t s);
// compact rows t < T of physical rows map[t] (nullable: identity)
cudaError_t launch_score_match(unsigned long long* best, const int32_t* map, const int32_t* tokens,
                               int split, int N, int T, int32_t* counts, cudaStream_t s);

// AdaInfer exit features of n exit-head row summaries: out [3][n] = top1
// (int bits), top prob p1, gap p1 - p2.
cudaError_t launch_exit_features(const RowStats* st, int n, float* out, cudaStream_t s);

// Runs the device's bounded waits against conditions that never come true
// (never[0] must be 0); *code gets bit 0 if the mbarrier wait gave up, bit 1
// if the counter wait did.
cudaError_t launch_wait_selftest(const unsigned* never, int polls, int32_t* code, cudaStream_t s);

// Sum-of-squares partials of fp32 rows (used by the op entry points to feed
// the norm-fused GEMV from an arbitrary x).
cudaError_t launch_ss_partials(const float* x, int M, int D, float* ss, cudaStream_t s);

}  // namespace ssd
