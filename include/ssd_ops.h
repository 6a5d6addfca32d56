/*
 * libssd kernel-level entry points.
 *
 * Each call runs one kernel of the decoding hot path on caller-provided
 * DEVICE buffers, enqueued on `stream` (a cudaStream_t; NULL = legacy
 * default stream), and returns without waiting.  They exist so that each
 * kernel can be checked on its own against the CPU oracle with seeded
 * inputs; the context API in ssd.h runs the same kernels.
 *
 * Common rules: M (rows, i.e. token positions processed together) is
 * 1..16; weight matrices are bf16 in the packed layout of ssd_pack_weight
 * (shapes are given as those of the row-major matrix, R % 16 == 0 and
 * K % 32 == 0); pointers are 16-byte aligned.  Calls that need scratch memory take it
 * from the stream-ordered allocator (cudaMallocAsync) and free it on the
 * same stream.  Errors: SSD_ERR_INVALID_ARG for a bad size or pointer,
 * SSD_ERR_OOM, SSD_ERR_CUDA for a failed launch; the message is available
 * from ssd_ops_last_error().
 *
 * Every kernel's reduction order is fixed by the element's own position and
 * never depends on M or on the other rows: row m of a call with M rows is
 * bit-identical to the same row computed alone.
 */
#ifndef SSD_OPS_H_
#define SSD_OPS_H_

#include <stdint.h>

#include "ssd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Per-row summary of a logits vector z (LM head epilogue). */
typedef struct {
  int32_t top1;   /* argmax z (lowest id on ties)                           */
  int32_t top2;   /* second-largest entry's id                              */
  int32_t sample; /* Gumbel-max sample of softmax(z / T) (T > 0), else top1 */
  int32_t pad;
  float z1;       /* z[top1]                                                */
  float z2;       /* z[top2]                                                */
  float lse;      /* log sum exp z                                          */
  float conf;     /* max softmax(z) = exp(z1 - lse)                         */
  float lse_t;    /* log sum exp (z / T) (T > 0), else lse                  */
  float pad2[3];
} ssd_row_stats;

/* y[m][r] = sum_k W[r][k] * act[m][k].  W bf16 [R][K]; act bf16 [M][K];
 * y fp32 [M][R].  The small-M weight-streaming GEMV of the decoder. */
ssd_status ssd_op_linear(const void* W, int32_t R, int32_t K, const void* act, int32_t M,
                         float* y, void* stream);

/* y = W bf16(rmsnorm(x) * gain): the norm-fused input of the QKV projection
 * and the LM head.  x fp32 [M][K]; gain fp32 [K]; y fp32 [M][R].  When M
 * rows of K do not fit the GEMV's per-CTA activation stage, a RMSNorm pass
 * first writes the bf16 rows (scratch) and the projection reads them; the
 * result is the same.  The same holds for ssd_op_swiglu and ssd_op_lm_head. */
ssd_status ssd_op_rmsnorm_linear(const void* W, int32_t R, int32_t K, const float* x,
                                 const float* gain, float eps, int32_t M, float* y, void* stream);

/* x += W act: o_proj / down_proj with the residual add fused.  x fp32
 * [M][R] (read and written); act bf16 [M][K]. */
ssd_status ssd_op_residual_linear(const void* W, int32_t R, int32_t K, const void* act, int32_t M,
                                  float* x, void* stream);

/* u = bf16(silu(Wg h) * (Wu h)) with h = bf16(rmsnorm(x) * gain).
 * Wg, Wu bf16 [F][K]; x fp32 [M][K]; u bf16 [M][F]. */
ssd_status ssd_op_swiglu(const void* Wg, const void* Wu, int32_t F, int32_t K, const float* x,
                         const float* gain, float eps, int32_t M, void* u, void* stream);

/* Decode / verify attention for M consecutive positions pos0..pos0+M-1.
 * qkv fp32 [M][(H + 2 Hkv) dh] holds the raw projections (q rows, k rows,
 * v rows, before RoPE).  The call applies rotate-half RoPE (base theta) to
 * q and k, stores bf16(k), bf16(v) into k_cache / v_cache ([Hkv][max_seq][dh]
 * bf16) at the M positions, and writes
 *   out[m][h dh ..] = bf16(softmax(q K^T / sqrt(dh), keys <= pos0+m) V)
 * (bf16 [M][H dh]).  Grouped-query: query head h reads K/V head h / (H/Hkv).
 * dh is 64 or 128; pos0 + M <= max_seq. */
ssd_status ssd_op_attention(const float* qkv, int32_t M, int32_t pos0, void* k_cache,
                            void* v_cache, int32_t max_seq, int32_t H, int32_t Hkv, int32_t dh,
                            float theta, void* out, void* stream);

/* Final RMSNorm + LM head with the fused row summary: z = W bf16(rmsnorm(x)
 * * gain) for each of the M rows (W bf16 [V][D], x fp32 [M][D]); writes
 * stats[m] (device) and, if logits is not NULL, z to logits (fp32 [M][V]).
 * At temperature > 0 the row summary includes a Gumbel-max sample drawn with
 * Philox4x32-10 counters (v/4, pos0 + m + 1, round, stream_id), key = seed. */
ssd_status ssd_op_lm_head(const void* W, int32_t V, int32_t D, const float* x, const float* gain,
                          float eps, int32_t M, float temperature, uint64_t seed, int32_t round,
                          int32_t stream_id, int32_t pos0, float* logits, ssd_row_stats* stats,
                          void* stream);

/* LayerSkip §3.3 acceptance at temperature T > 0 for one round.
 * P fp32 [d+1][V] verify logits, Q fp32 [d][V] draft logits, drafts int32 [d]
 * (all device).  Draft j is accepted when u_j < p_j(y_j) / q_j(y_j) with
 * p = softmax(P/T), q = softmax(Q/T) and u_j the Philox uniform at counter
 * (0, n + j, round, 1); on the first rejection a token is drawn from
 * norm(max(0, p_j - q_j)) (from p_j if that is empty), otherwise a bonus
 * from p_d, by Gumbel-max at counters (v/4, n + j, round, 2).
 * Writes emitted (device int32 [d+1]) and n_emitted (device int32 [1]). */
ssd_status ssd_op_accept_stochastic(const float* P, const float* Q, const int32_t* drafts,
                                    int32_t d, int32_t V, float temperature, uint64_t seed,
                                    int32_t round, int32_t n, int32_t* emitted,
                                    int32_t* n_emitted, void* stream);

/* Philox4x32-10 of the library: out[4i..4i+3] = philox(ctr[4i..4i+3], key).
 * ctr, out: device uint32 [4 count]. */
ssd_status ssd_op_philox(const uint32_t* ctr, int32_t count, uint64_t key, uint32_t* out,
                         void* stream);

/* Many-row projection on the tensor cores (the batched candidate-mask
 * scoring forward of SWIFT §4.1.2, where K candidates x N window positions
 * give hundreds of rows): for T >= 1 rows of act (bf16 [T][K]),
 *   epi 0 (store):  out fp32 [T][R] = W act
 *   epi 1 (resid):  out fp32 [*][R]: out[map[t]] += W act[t] (map: device
 *                   int32 [T] of distinct rows, NULL = identity; rows not
 *                   named stay as they are)
 *   epi 2 (swiglu): out bf16 [T][R] = bf16(silu(W act) * (W1 act)), W1 the
 *                   up matrix (same shape as W)
 *   epi 3 (argmax): out int32 [T] = argmax_r (W act)[r], lowest r on ties
 * W, W1 packed (ssd_pack_weight).  With epi | SSD_ROWS_ACT_PACKED, act is
 * already in the packed layout: ssd_pack_weight of the [T'][K] matrix, T'
 * = T rounded up to 16 (the rows beyond T are read and their results
 * dropped); otherwise the call packs a scratch copy first.  Every output
 * sums K in ascending 32-wide steps, whatever T.  This call has no limit of
 * 16 rows. */
#define SSD_ROWS_ACT_PACKED 16
ssd_status ssd_op_linear_rows(const void* W, const void* W1, int32_t R, int32_t K,
                              const void* act, int32_t T, int32_t epi, void* out,
                              const int32_t* map, void* stream);

/* Attention of candidate-mask scoring windows.  For each candidate k in
 * cand (device int32 [n_cand]) and window row i < N (query position
 * split + i), with q bf16 [n_cand N][H][dh] (RoPE applied, row ja N + i for
 * the ja-th candidate of the list):
 *   out[ja N + i][h dh ..] = bf16(softmax(q K^T / sqrt(dh)) V)
 * over the keys of the shared cache k_cache / v_cache ([Hkv][max_seq][dh]
 * bf16) at positions 0..split-1, then candidate k's own window keys
 * wk / wv (bf16 [w_rows][Hkv][dh], row k N + w) for w <= i; every k in cand
 * has k N + N <= w_rows.  split >= 1, split <= max_seq; dh 64 or 128. */
ssd_status ssd_op_score_attention(const void* q, const int32_t* cand, int32_t n_cand, int32_t N,
                                  int32_t split, const void* k_cache, const void* v_cache,
                                  int32_t max_seq, const void* wk, const void* wv, int32_t w_rows,
                                  int32_t H, int32_t Hkv, int32_t dh, void* out, void* stream);

/* Description of the most recent failed op call on this host thread. */
const char* ssd_ops_last_error(void);

/* Failure detection self-test: runs the device-side bounded waits the
 * kernels use (an mbarrier wait, a global-counter wait) against conditions
 * that never come true, each limited to `polls` polls (1..2^20).  Every wait
 * must give up and report instead of hanging: *code_out (host) receives bit
 * 0 if the mbarrier wait gave up and bit 1 if the counter wait did (3 when
 * both behave).  Synchronises the stream.  Errors: INVALID_ARG, CUDA. */
ssd_status ssd_op_wait_selftest(int32_t polls, int32_t* code_out, void* stream);

/* ssd_op_linear for callers that cannot allocate device memory (the pages
 * have no counterpart; this is a library convenience).  Same arguments,
 * layout and result as ssd_op_linear, but the GEMV's scratch (partial sums of
 * row groups split across CTAs, completion counters) comes from a fixed
 * 1 MiB + 4.25 KiB array that the library reserves on every GPU that loads it,
 * held until the process exits; no cudaMalloc, cudaFree or other allocating
 * routine is called.  R must be <= 8192 (SSD_ERR_CAPACITY otherwise).
 * The first call on a device looks up the array's device address with that
 * device current and keeps it; make that first call before any stream
 * capture, and make no call on a device after cudaDeviceReset on it (the
 * reset destroys the array the kept address points to).  Every
 * call on a device shares the one array and clears its counters on entry, so
 * calls whose kernels overlap on the GPU (different streams, or different
 * host threads) race and must be serialised by the caller.  Errors are
 * described by ssd_op_linear_noalloc_last_error(). */
ssd_status ssd_op_linear_noalloc(const void* W, int32_t R, int32_t K, const void* act, int32_t M,
                                 float* y, void* stream);
const char* ssd_op_linear_noalloc_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* SSD_OPS_H_ */
