/*
 * libssd — layer-skipping self-speculative decoding on one GB300 (sm_103a).
 *
 * The calls follow the problem statement of the pages this library is
 * built from:
 *   - LayerSkip blog (marsggbo.github.io, "ACL'24 | LayerSkip ..."),
 *     §3.1 draft_phase, §3.2 verify_phase, §3.3 layerskip_ssd;
 *   - SWIFT: On-the-Fly Self-Speculative Decoding (paperlayer.ai digest),
 *     §4.1/§4.1.2 matchness scoring of candidate layer sets, §4.2
 *     confidence-aware drafting.
 *
 * Model: a Llama-style decoder (RMSNorm, rotate-half RoPE, MHA/GQA
 * attention, SwiGLU MLP, untied LM head).  Weights are bf16, the residual
 * stream fp32; every GEMM input (normed hidden state, attention output,
 * SwiGLU product) and every stored K/V value is rounded to bf16; logits are
 * fp32.
 *
 * Decoding state.  t[0..n-1] are the committed tokens.  The last one,
 * x = t[n-1], is "pending": it has not yet been run through the full model,
 * and K/V at positions < n-1 hold full-model values in every layer.
 *
 * Threading and streams.  A context is used from one host thread at a time.
 * Every call enqueues its work on the context's stream; a call that returns
 * host data (any *_out pointer documented as "host") waits for its stream
 * with a bounded wait (SSD_ERR_TIMEOUT after the context's timeout).
 *
 * Ownership.  The caller owns the weights (device memory) and must keep
 * them alive and unchanged for the context's lifetime.  The context owns its
 * KV cache, workspaces and CUDA graphs.  Host buffers are caller-owned and
 * sized by the documented maxima.
 *
 * Errors.  Every call returns an ssd_status; none aborts the process.
 * ssd_last_error() describes the most recent failure of a context.
 */
#ifndef SSD_H_
#define SSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1, /* bad pointer, size, shape or policy            */
  SSD_ERR_STATE = 2,       /* call made in the wrong order (verify w/o draft)*/
  SSD_ERR_CAPACITY = 3,    /* max_seq, max_draft or scoring capacity exceeded */
  SSD_ERR_OOM = 4,         /* device allocation failed                       */
  SSD_ERR_CUDA = 5,        /* a CUDA runtime call failed                     */
  SSD_ERR_TIMEOUT = 6      /* a bounded host wait on the stream ran out      */
} ssd_status;

typedef struct ssd_ctx ssd_ctx;

/* Model shape and context capacities. */
typedef struct {
  int32_t n_layers;    /* L                                              */
  int32_t d_model;     /* D, multiple of 64                              */
  int32_t n_heads;     /* H                                              */
  int32_t n_kv_heads;  /* Hkv, divides H                                 */
  int32_t head_dim;    /* dh: 64 or 128                                  */
  int32_t ffn_dim;     /* F, multiple of 32                              */
  int32_t vocab;       /* V, multiple of 16                              */
  float rope_theta;    /* RoPE base, e.g. 1e4                            */
  float norm_eps;      /* RMSNorm epsilon, e.g. 1e-5                     */
  int32_t max_seq;     /* KV capacity in positions (multiple of 64)      */
  int32_t max_draft;   /* largest d_max any policy may use, 1..15        */
  int32_t max_score_rows; /* K*N capacity of ssd_score_masks (0: none)   */
  int32_t dtype;       /* SSD_DTYPE_BF16 (0) or SSD_DTYPE_FP32 (1), below */
} ssd_config;

/* Weight and arithmetic precision of a model.  SSD_DTYPE_BF16: projection
 * matrices bf16 in the packed layout, bf16 K/V cache, bf16 rounding at every
 * projection input.  SSD_DTYPE_FP32: every weight fp32 and row-major (tok_embed
 * [V, D], wqkv [(H + 2 Hkv) dh, D], wo [D, H dh], w_gate / w_up [F, D], w_down
 * [D, F], lm_head [V, D]: not packed), fp32 K/V cache, activations and logits
 * with no rounding anywhere; ssd_score_masks, ssd_swift_generate, dynamic
 * verification (tree_tau > 0) and ssd_profile_kernels are for bf16 models
 * only (SSD_ERR_INVALID_ARG). */
enum { SSD_DTYPE_BF16 = 0, SSD_DTYPE_FP32 = 1 };

/* Device pointers of one decoder layer (borrowed), each 16-byte aligned
 * (ssd_create returns SSD_ERR_INVALID_ARG otherwise; the same holds for the
 * pointers of ssd_weights).  Projection matrices are given in the packed
 * layout written by ssd_pack_weight; the shapes below are those of the
 * row-major matrices they were packed from. */
typedef struct {
  const void* attn_norm; /* [D] fp32 RMSNorm gain                          */
  const void* wqkv;      /* packed [(H + 2 Hkv) dh, D] bf16: q, k, v rows  */
  const void* wo;        /* packed [D, H dh] bf16                          */
  const void* mlp_norm;  /* [D] fp32                                       */
  const void* w_gate;    /* packed [F, D] bf16                             */
  const void* w_up;      /* packed [F, D] bf16                             */
  const void* w_down;    /* packed [D, F] bf16                             */
} ssd_layer_weights;

typedef struct {
  const void* tok_embed;  /* [V, D] bf16, row-major (rows are gathered)     */
  const void* final_norm; /* [D] fp32                                       */
  const void* lm_head;    /* packed [V, D] bf16 (shared by draft and verify) */
  const ssd_layer_weights* layers; /* host array of n_layers entries; the
                                      table is copied by ssd_create       */
} ssd_weights;

enum { SSD_MODE_SKIP = 0, SSD_MODE_EXIT = 1 };

/* Draft policy (SWIFT §4.2 / LayerSkip §3.1). */
typedef struct {
  int32_t mode;          /* SSD_MODE_SKIP: draft runs every layer whose bit
                            in skip_mask is clear.  SSD_MODE_EXIT: draft runs
                            layers 0..exit_layer, then the shared final norm
                            and LM head                                      */
  uint64_t skip_mask[4]; /* bit l (word l/64) set: layer l skipped (L<=256) */
  int32_t exit_layer;    /* exit mode: E, 0 <= E < L                         */
  int32_t d_max;         /* draft at most d_max tokens per round (<= max_draft)*/
  float tau;             /* stop drafting when top-1 probability < tau;
                            tau <= 0 never stops                            */
  float temperature;     /* 0: greedy draft and acceptance; > 0: sampled
                            draft from softmax(z/T), min(1,p/q) acceptance  */
  uint64_t seed;         /* Philox4x32-10 key                                */
  /* Skip mode only (SWIFT Fig. 10 skips the two sublayers of a layer
   * separately): bit l set drops only the attention sublayer (attn) or only
   * the MLP sublayer (mlp) of layer l from the draft; a dropped sublayer's
   * residual branch is left out and a layer whose attention is dropped
   * writes no K/V at the draft positions.  A layer in skip_mask drops both.
   * The verify recomputes from the first layer with any dropped sublayer.  */
  uint64_t skip_attn_mask[4];
  uint64_t skip_mlp_mask[4];
  /* Dynamic verification (SWIFT §4.2: the draft's confidence also sets how
   * many candidates are verified; greedy decoding only).  tree_tau <= 0:
   * off.  Otherwise a kept draft y_j whose top-1 probability is below
   * tree_tau gets the draft's second choice s_j as a sibling candidate (at
   * most tree_max per round, 1..8, in depth order; d_max + 1 + tree_max
   * <= 16).  A sibling runs as a side row of the next draft step (or the
   * extra pass) through the layers below s0 and of the verify pass through
   * the rest, attending to the context before its position and to itself.
   * When y_a is rejected and the full model's token there equals s_a, the
   * sibling is taken and the full model's token after it is emitted too
   * (one more token in that round; the output stays the greedy output).
   * Requires temperature 0 (else SSD_ERR_INVALID_ARG).                    */
  float tree_tau;
  int32_t tree_max;
} ssd_policy;

typedef struct {
  int64_t rounds;          /* verify passes                                 */
  int64_t drafted;         /* draft tokens proposed (sum of d)              */
  int64_t accepted;        /* draft tokens accepted                         */
  int64_t emitted;         /* tokens emitted (before truncation to n_tokens)*/
  int64_t draft_steps;     /* draft forward passes run                      */
  int64_t kernel_launches; /* library kernels launched (graph nodes counted) */
  double bytes_streamed;   /* algorithmic HBM bytes: weights + KV read/written */
  /* Device time (CUDA events around each pass; the SWIFT cost coefficient c
   * is draft_ms / draft_steps over ar_ms / AR steps, SWIFT §B.3): */
  double draft_ms;         /* draft steps                                   */
  double verify_ms;        /* extra passes, verify passes and acceptance    */
  double ar_ms;            /* ssd_decode_ar: the autoregressive steps       */
  int64_t side_rows;       /* dynamic verification: siblings verified        */
  int64_t side_accepted;   /* rounds that took a sibling (one more token)   */
} ssd_stats;

/* Fault injection for failure-detection tests: the n-th device allocation
 * (counting from 0) of the calling thread's next ssd_create fails as if the
 * device were out of memory; n < 0 disables it.  ssd_create must then return
 * SSD_ERR_OOM having released everything it allocated. */
ssd_status ssd_debug_fail_alloc(int32_t n);

/* Workspace canaries.  A library built with -DSSD_DEBUG_CHECKS follows every
 * workspace of a context with 256 bytes of 0xA5 and bounds-checks token ids,
 * K/V positions and pass row counts on the device (a failed check records
 * its code, >= 100, and the offending value in the context's state, the
 * access is skipped, and the next call reports SSD_ERR_STATE).  This call
 * counts the canaries (*checked_out; 0 in release builds, which have none)
 * and the canary bytes that no longer hold 0xA5 (*bad_out).  Synchronises
 * the context's stream.  Errors: INVALID_ARG, CUDA, TIMEOUT. */
ssd_status ssd_debug_canaries(ssd_ctx* ctx, int32_t* checked_out, int32_t* bad_out);

/* Converts a row-major bf16 matrix W [R][K] (device memory) into the
 * library's packed layout at dst (device, R*K bf16, must not overlap src).
 * The packed matrix is a sequence of units of 16 rows x 32 columns,
 * row-group-major; inside a unit, element W[16 vr + 8 h + g][32 kb + 8 c + e]
 * sits at unit offset h*256 + (4 g + c)*8 + e (h < 2, g < 8, c < 4, e < 8),
 * which is the register fragment order of the tensor-core MMA, so each unit
 * streams into shared memory with one bulk copy and every projection is one
 * contiguous read.  Requires R % 16 == 0 and K % 32 == 0.  Enqueued on
 * `stream`; returns without waiting.  Errors: INVALID_ARG, CUDA. */
ssd_status ssd_pack_weight(const void* src, void* dst, int32_t R, int32_t K, void* stream);

/* Creates a context for one model on one device (the current device).
 * stream: a cudaStream_t (NULL: the legacy default stream).  Validates the
 * shape (see ssd_config), allocates the KV cache [L][Hkv][max_seq][dh] bf16
 * (K and V) and the workspaces.  Errors: INVALID_ARG, OOM, CUDA. */
ssd_status ssd_create(const ssd_config* cfg, const ssd_weights* weights, void* stream,
                      ssd_ctx** out);

/* Frees everything the context owns.  Waits for its stream.  NULL is OK. */
ssd_status ssd_destroy(ssd_ctx* ctx);

/* Sets the draft policy; (re)builds the CUDA graphs of the draft step, the
 * verify pass and the autoregressive step.  Errors: INVALID_ARG, CAPACITY
 * (d_max > max_draft), CUDA. */
ssd_status ssd_set_policy(ssd_ctx* ctx, const ssd_policy* policy);

/* Runs tokens[0..n-1] (host) through the full model at positions 0..n-1,
 * replacing any previous state, and commits the first new token (argmax, or
 * a sample at T > 0), which it also returns in *first_token_out (host).
 * After the call n_committed = n + 1.  Errors: INVALID_ARG, CAPACITY
 * (n + 1 > max_seq), CUDA, TIMEOUT. */
ssd_status ssd_prefill(ssd_ctx* ctx, const int32_t* tokens, int32_t n, int32_t* first_token_out);

/* LayerSkip §3.1 draft_phase / SWIFT §4.2: drafts up to d_max tokens with
 * the policy's layer subset, feeding x and then each draft token, stopping
 * when top-1 confidence < tau.  draft_out (host, >= d_max) receives
 * y_0..y_{d-1}; conf_out (host, >= d_max + 1, nullable) the confidence of
 * every draft step run (the stopping step included); *d_out = d.
 * Errors: STATE (a draft already pending), CAPACITY (positions would pass
 * max_seq), CUDA, TIMEOUT. */
ssd_status ssd_draft(ssd_ctx* ctx, int32_t* draft_out, float* conf_out, int32_t* d_out);

/* LayerSkip §3.2 verify_phase: the full model over positions n-1..n-1+d,
 * reusing the draft's K/V of layers below s0 (s0 = first skipped layer, or
 * E + 1).  logits_out (host, nullable, [d+1][V] fp32) receives the verify
 * logits.  Errors: STATE (no draft pending), CUDA, TIMEOUT. */
ssd_status ssd_verify(ssd_ctx* ctx, float* logits_out);

/* LayerSkip §3.3: greedy prefix acceptance (T = 0) or min(1, p/q)
 * acceptance with residual / bonus sampling (T > 0); commits the emitted
 * tokens and rolls the KV length back to the accepted prefix.
 * emitted_out (host, >= d_max + 1) and *n_emitted_out (1..d+1).
 * Errors: STATE (no verify pending), CUDA, TIMEOUT. */
ssd_status ssd_accept(ssd_ctx* ctx, int32_t* emitted_out, int32_t* n_emitted_out);

/* One full round (draft, verify, accept) per iteration until n_tokens tokens
 * are emitted; extra tokens of the last round are dropped (the committed
 * length ends exactly n_tokens further).  out (host, nullable, >= n_tokens)
 * receives the tokens; stats (host, nullable) is filled.
 * With the device loop (ssd_set_device_loop, on by default where the device
 * supports the conditional graph nodes it needs) the whole call is one
 * graph launch: the draft loop's stop, the extra pass, the verify width and
 * the next round are decided on the device, and the host reads back once.
 * The tokens and counts are those of the host-driven loop; stats then has
 * draft_ms = verify_ms = 0 and bytes_streamed counts the K/V at the
 * generation's middle position.
 * Errors: CAPACITY, STATE (no prefill), CUDA, TIMEOUT. */
ssd_status ssd_generate(ssd_ctx* ctx, int32_t n_tokens, int32_t* out, ssd_stats* stats);

/* ssd_generate's device loop on (enable != 0, the default) or off (the host
 * drives each draft step, verify and acceptance, and stats carries per-pass
 * device times).  *active_out (host, nullable) = whether the loop graph
 * exists and will be used.  Errors: INVALID_ARG (ctx NULL). */
ssd_status ssd_set_device_loop(ssd_ctx* ctx, int32_t enable, int32_t* active_out);

/* Plain autoregressive decoding with the full model (the baseline the
 * speedup is measured against), same kernels.  out (host, nullable). */
ssd_status ssd_decode_ar(ssd_ctx* ctx, int32_t n_tokens, int32_t* out, ssd_stats* stats);

/* Lossy early exit (LayerSkip blog §3, inference mode one): each step runs
 * the pending token through the policy's draft layers only (exit mode:
 * layers 0..E; skip mode: the kept layers and sublayers) and commits the
 * shared final RMSNorm + LM head's pick (greedy, or at temperature > 0 the
 * Gumbel-max sample an autoregressive step would draw).  No verification:
 * the output is the early model's.  The dropped layers' K/V of those
 * positions are not written, so until the context is rewound to before the
 * first of them (ssd_rewind) or prefilled again, the lossless entry points
 * (ssd_draft, ssd_generate, ssd_decode_ar, ssd_score_masks,
 * ssd_swift_generate, ssd_layer_features) return SSD_ERR_STATE.  A policy
 * whose draft runs every sublayer decodes losslessly and sets no such mark.
 * out (host, nullable, >= n_tokens); stats (host, nullable): rounds =
 * emitted = n_tokens, draft_ms = device time of the steps.
 * Errors: CAPACITY, STATE, CUDA, TIMEOUT. */
ssd_status ssd_decode_lossy(ssd_ctx* ctx, int32_t n_tokens, int32_t* out, ssd_stats* stats);

/* AdaInfer exit features (EE-structure page, steps 1-2): one
 * autoregressive step of the pending token (it commits what ssd_decode_ar
 * would) with the early-exit head (final RMSNorm + LM head) applied to the
 * hidden state after every layer l = min_layer .. L-1.  For entry
 * i = l - min_layer (host arrays of L - min_layer entries): top1[i] = the
 * argmax, top_prob[i] = p1 = max softmax, gap[i] = p1 - p2 (the two largest
 * probabilities).  The label of layer l is top1[i] == top1[L-1-min_layer].
 * Costs one LM-head pass per layer.
 * Errors: INVALID_ARG (min_layer outside 0..L-1, NULL outputs), CAPACITY,
 * STATE, CUDA, TIMEOUT. */
ssd_status ssd_layer_features(ssd_ctx* ctx, int32_t min_layer, int32_t* top1, float* top_prob,
                              float* gap);

/* SWIFT §4.1.2: scores K candidate skip sets by matchness.  Candidate k
 * (masks[4k..4k+3], host, bit l = layer l skipped) runs the window inputs
 * t[n-N-1..n-2] causally through its kept layers, attending to the
 * full-model K/V of positions < n-N-1 and to its own K/V for the window,
 * and predicts t[n-N..n-1] by top-1; matchness_out[k] (host) = matches / N,
 * *best_out = argmax (lowest k on ties).  The shared cache is not modified.
 * Errors: INVALID_ARG, CAPACITY (K*N > max_score_rows, or N + 1 > n - 1),
 * CUDA, TIMEOUT. */
ssd_status ssd_score_masks(ssd_ctx* ctx, const uint64_t* masks, int32_t K, int32_t N,
                           float* matchness_out, int32_t* best_out);

/* Rolls the committed length back to n (2 <= n <= current n).  The token
 * t[n-1] becomes pending again. */
ssd_status ssd_rewind(ssd_ctx* ctx, int32_t n);

/* Copies the committed tokens to out (host, cap entries); *n_out = n. */
ssd_status ssd_get_tokens(ssd_ctx* ctx, int32_t* out, int32_t cap, int32_t* n_out);

/* Per-kernel-class timing of the decode path, measured with CUDA events on
 * the context's stream around every launch of n_steps eager autoregressive
 * steps (the same kernels and launch shapes the captured graphs replay).
 * Class order: 0 qkv, 1 attention, 2 o_proj, 3 gate_up, 4 down, 5 lm_head,
 * 6 control (embedding, acceptance and bookkeeping kernels).  The committed
 * state is restored afterwards.  Errors: STATE (no prefill), CAPACITY, CUDA. */
typedef struct {
  double ms[8];       /* average device time per launch                    */
  double bytes[8];    /* algorithmic HBM bytes per launch (weights + KV)    */
  int64_t launches[8];
} ssd_kernel_times;
ssd_status ssd_profile_decode(ssd_ctx* ctx, int32_t n_steps, ssd_kernel_times* out);

/* Per-kernel-class timing as the captured autoregressive step runs the
 * kernels: for each class, one CUDA graph holding that class's launches for
 * every layer (the LM head: n_layers launches of it) at the step's pass shape
 * (one row at the pending position), chained with programmatic dependent
 * launch as in the step's graph, replayed `reps` times after one warm-up
 * replay between CUDA events on the context's stream.  ms[k] = device time
 * per launch, bytes[k] = algorithmic HBM bytes per launch (weights; K/V of
 * the current context for attention), launches[k] = launches of the class in
 * one autoregressive step (n_layers, 1 for the LM head, 0 for class 6).
 * Entry 7 times attention and o_proj together, one pair per layer launched
 * back to back as the step launches them (ms and bytes per pair, launches 0
 * because the pair repeats classes 1 and 2).  Only
 * scratch buffers and the cache row of the pending position are written; the
 * committed state is restored.  Errors: INVALID_ARG, STATE (no prefill, a
 * round in flight), CAPACITY, CUDA, TIMEOUT. */
ssd_status ssd_profile_kernels(ssd_ctx* ctx, int32_t reps, ssd_kernel_times* out);

/* Host wait limit in milliseconds for calls that return host data
 * (default 120000). */
ssd_status ssd_set_timeout_ms(ssd_ctx* ctx, int32_t ms);

/* SWIFT on-the-fly layer-set optimisation (SWIFT §4: optimisation
 * alternates with confidence-aware acceleration; §4.1.1: uniform layer
 * skipping until the context window is filled; §4.1.2: candidate layer sets
 * proposed by random search, scored by parallel prediction of prior context
 * tokens, the best matchness kept, the phase ending at its step limit or
 * when the best candidate stays unchanged; §B.2: S = 1000, 300 unchanged
 * steps, matchness > 0.95, gamma = 32).  Bayesian optimisation is not
 * included. */
typedef struct {
  int32_t skip_count; /* layers every candidate skips (skip ratio x L), >= 1    */
  int32_t lo_layer;   /* candidates skip layers in [lo_layer, n_layers)          */
  int32_t window;     /* gamma: committed tokens a candidate is scored on       */
  int32_t candidates; /* K per step: the incumbent, then K-1 random proposals;
                         K * window <= max_score_rows                           */
  int32_t max_steps;  /* step limit S                                            */
  int32_t patience;   /* stop after this many consecutive steps the incumbent wins */
  float target;       /* stop after a step whose best matchness exceeds this     */
  uint64_t seed;      /* SplitMix64 (Steele, Lea, Flood 2014) seed of the proposals */
} ssd_swift_params;

typedef struct {
  int32_t steps;        /* optimisation steps run                                */
  int32_t stopped_by;   /* 0: still optimising when the tokens ran out;
                           1: target; 2: step limit; 3: patience                 */
  uint64_t final_mask[4]; /* the incumbent skip set at the end                   */
  int64_t rounds, drafted, accepted, emitted;
  double opt_seconds;   /* host wall time spent in scoring steps                */
  double total_seconds; /* host wall time of the call                           */
} ssd_swift_report;

/* Generates n_tokens after the committed context with SWIFT.  The draft
 * starts from the uniform set (layer lo + floor((2i+1)(L-lo) / (2 count)),
 * i < count); every decoding round with the incumbent set is followed, once
 * window + 1 tokens have been generated and while optimising, by one step
 * that scores the incumbent and K-1 proposals (a partial Fisher-Yates shuffle
 * of the allowed layers per proposal, one SplitMix64 stream drawn in
 * proposal order) with ssd_score_masks over the last `window` committed
 * tokens; the highest matchness wins, the lowest index on ties (the
 * incumbent survives ties).  Optimisation stops after a step whose best
 * exceeds target, after max_steps steps, or after `patience` steps the
 * incumbent won.  Drafting uses the context's policy (skip mode: d_max,
 * tau, temperature, seed) with the incumbent as its skip set, which stays
 * set afterwards.  out (nullable): n_tokens ids.  Per step s < trace_cap
 * (arrays nullable): trace_masks [s][K][4] candidates, trace_scores [s][K]
 * matchness, trace_best [s] the winner.  Errors: INVALID_ARG, STATE (exit
 * mode, no prefill, a round in flight), CAPACITY (tokens or K * window),
 * CUDA, TIMEOUT. */
ssd_status ssd_swift_generate(ssd_ctx* ctx, const ssd_swift_params* params, int32_t n_tokens,
                              int32_t* out, uint64_t* trace_masks, float* trace_scores,
                              int32_t* trace_best, int32_t trace_cap, ssd_swift_report* report);

/* Human-readable description of the context's most recent error ("" if
 * none; a static string for a NULL context). */
const char* ssd_last_error(const ssd_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* SSD_H_ */
