// Kernel-level C-ABI (ssd_ops.h): each call runs one hot-path kernel on
// caller-provided device buffers, so that every kernel can be checked on
// its own against the CPU oracle.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/ssd_ops.h"
#include "kernels.cuh"

using namespace ssd;

namespace {

thread_local std::string g_op_err;

ssd_status op_fail(ssd_status s, const std::string& m) {
  g_op_err = m;
  return s;
}

bool al16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

ssd_status check_linear(const void* W, int R, int K, int M) {
  if (!al16(W)) return op_fail(SSD_ERR_INVALID_ARG, "W must be non-null and 16-byte aligned");
  if (R <= 0 || R % 16) return op_fail(SSD_ERR_INVALID_ARG, "R must be a positive multiple of 16");
  if (K <= 0 || K % 32) return op_fail(SSD_ERR_INVALID_ARG, "K must be a positive multiple of 32");
  if (M < 1 || M > kMaxRows) return op_fail(SSD_ERR_INVALID_ARG, "M must be in 1..16");
  return SSD_OK;
}

ssd_status cu(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return SSD_OK;
  cudaGetLastError();
  return op_fail(e == cudaErrorMemoryAllocation ? SSD_ERR_OOM : SSD_ERR_CUDA,
                 std::string(what) + ": " + cudaGetErrorString(e));
}

// Stream-ordered scratch that is freed on scope exit.
struct Scratch {
  cudaStream_t s;
  void* p = nullptr;
  Scratch(cudaStream_t st) : s(st) {}
  cudaError_t alloc(size_t bytes) { return cudaMallocAsync(&p, bytes, s); }
  ~Scratch() {
    if (p) cudaFreeAsync(p, s);
  }
};

// Scratch for one GEMV launch (zeroed counters).
struct GemvOpScratch {
  Scratch part, cnt, rec, err;
  explicit GemvOpScratch(cudaStream_t s) : part(s), cnt(s), rec(s), err(s) {}
  ssd_status init(int R, int K, int epi, LinearArgs& a, cudaStream_t s) {
    const GemvScratch gs = gemv_scratch(R, K, epi);
    ssd_status r;
    if ((r = cu(part.alloc(gs.part_floats * 4), "scratch")) != SSD_OK) return r;
    if ((r = cu(cnt.alloc(gs.counters * 4), "scratch")) != SSD_OK) return r;
    if ((r = cu(rec.alloc(gs.rec_floats ? gs.rec_floats * 4 : 16), "scratch")) != SSD_OK) return r;
    if ((r = cu(err.alloc(16), "scratch")) != SSD_OK) return r;
    if ((r = cu(cudaMemsetAsync(cnt.p, 0, gs.counters * 4, s), "memset")) != SSD_OK) return r;
    if ((r = cu(cudaMemsetAsync(err.p, 0, 16, s), "memset")) != SSD_OK) return r;
    a.part = (float*)part.p;
    a.counter = (unsigned*)cnt.p;
    a.rec = (float*)rec.p;
    a.err = (int*)err.p;
    return SSD_OK;
  }
};

// A norm-fused projection: when the rows do not fit the GEMV's activation
// stage, a RMSNorm pre-pass writes bf16 rows and the projection reads those
// (the same bits; what the context runtime does for wide passes).
ssd_status launch_norm_fused(int epi, LinearArgs a, cudaStream_t s, Scratch& xn, const char* what) {
  if (a.M_static <= gemv_stage_rows(a.K)) return cu(launch_gemv(IN_NORM, epi, a, s, false), what);
  ssd_status r;
  if ((r = cu(xn.alloc((size_t)a.M_static * a.K * sizeof(bf16)), "scratch")) != SSD_OK) return r;
  if ((r = cu(launch_norm_rows(a.x, a.ss, a.gain, a.eps, a.M_static, nullptr, a.K, (bf16*)xn.p, s,
                               false),
              "rmsnorm")) != SSD_OK)
    return r;
  a.act = (const bf16*)xn.p;
  a.x = nullptr;
  a.ss = nullptr;
  a.gain = nullptr;
  return cu(launch_gemv(IN_BF16, epi, a, s, false), what);
}

}  // namespace

extern "C" {

const char* ssd_ops_last_error(void) { return g_op_err.c_str(); }

ssd_status ssd_pack_weight(const void* src, void* dst, int32_t R, int32_t K, void* stream) {
  if (!al16(src) || !al16(dst) || src == dst)
    return op_fail(SSD_ERR_INVALID_ARG, "pack: src / dst must be distinct, 16-byte aligned");
  if (R <= 0 || R % 16 || K <= 0 || K % 32)
    return op_fail(SSD_ERR_INVALID_ARG, "pack: R % 16 == 0 and K % 32 == 0 required");
  const char* lo = (const char*)src;
  const char* hi = (const char*)dst;
  const size_t bytes = (size_t)R * K * 2;
  if ((lo < hi && lo + bytes > hi) || (hi < lo && hi + bytes > lo))
    return op_fail(SSD_ERR_INVALID_ARG, "pack: src and dst overlap");
  return cu(launch_pack((const bf16*)src, (bf16*)dst, R, K, (cudaStream_t)stream), "pack");
}

ssd_status ssd_op_linear(const void* W, int32_t R, int32_t K, const void* act, int32_t M,
                         float* y, void* stream) {
  ssd_status r = check_linear(W, R, K, M);
  if (r != SSD_OK) return r;
  if (!al16(act) || !al16(y)) return op_fail(SSD_ERR_INVALID_ARG, "act / y alignment");
  LinearArgs a;
  a.W0 = (const bf16*)W;
  a.R = R;
  a.K = K;
  a.act = (const bf16*)act;
  a.M_static = M;
  a.y = y;
  GemvOpScratch gs((cudaStream_t)stream);
  if ((r = gs.init(R, K, EPI_STORE, a, (cudaStream_t)stream)) != SSD_OK) return r;
  return cu(launch_gemv(IN_BF16, EPI_STORE, a, (cudaStream_t)stream, false), "linear");
}

ssd_status ssd_op_rmsnorm_linear(const void* W, int32_t R, int32_t K, const float* x,
                                 const float* gain, float eps, int32_t M, float* y, void* stream) {
  ssd_status r = check_linear(W, R, K, M);
  if (r != SSD_OK) return r;
  if (!al16(x) || !al16(gain) || !al16(y) || !(eps > 0.f))
    return op_fail(SSD_ERR_INVALID_ARG, "x / gain / y / eps");
  cudaStream_t s = (cudaStream_t)stream;
  Scratch ss(s);
  if ((r = cu(ss.alloc((size_t)M * (K / kSsGroup) * 4), "scratch")) != SSD_OK) return r;
  if ((r = cu(launch_ss_partials(x, M, K, (float*)ss.p, s), "ss")) != SSD_OK) return r;
  LinearArgs a;
  a.W0 = (const bf16*)W;
  a.R = R;
  a.K = K;
  a.x = x;
  a.ss = (const float*)ss.p;
  a.gain = gain;
  a.eps = eps;
  a.M_static = M;
  a.y = y;
  GemvOpScratch gs(s);
  if ((r = gs.init(R, K, EPI_STORE, a, s)) != SSD_OK) return r;
  Scratch xn(s);
  return launch_norm_fused(EPI_STORE, a, s, xn, "rmsnorm_linear");
}

ssd_status ssd_op_residual_linear(const void* W, int32_t R, int32_t K, const void* act, int32_t M,
                                  float* x, void* stream) {
  ssd_status r = check_linear(W, R, K, M);
  if (r != SSD_OK) return r;
  if (!al16(act) || !al16(x)) return op_fail(SSD_ERR_INVALID_ARG, "act / x alignment");
  cudaStream_t s = (cudaStream_t)stream;
  Scratch ss(s);
  if ((r = cu(ss.alloc((size_t)M * (R / kSsGroup) * 4), "scratch")) != SSD_OK) return r;
  LinearArgs a;
  a.W0 = (const bf16*)W;
  a.R = R;
  a.K = K;
  a.act = (const bf16*)act;
  a.M_static = M;
  a.xres = x;
  a.ss_out = (float*)ss.p;
  GemvOpScratch gs(s);
  if ((r = gs.init(R, K, EPI_RESID, a, s)) != SSD_OK) return r;
  return cu(launch_gemv(IN_BF16, EPI_RESID, a, s, false), "residual_linear");
}

ssd_status ssd_op_swiglu(const void* Wg, const void* Wu, int32_t F, int32_t K, const float* x,
                         const float* gain, float eps, int32_t M, void* u, void* stream) {
  ssd_status r = check_linear(Wg, F, K, M);
  if (r != SSD_OK) return r;
  if (!al16(Wu) || !al16(x) || !al16(gain) || !al16(u) || !(eps > 0.f))
    return op_fail(SSD_ERR_INVALID_ARG, "Wu / x / gain / u / eps");
  cudaStream_t s = (cudaStream_t)stream;
  Scratch ss(s);
  if ((r = cu(ss.alloc((size_t)M * (K / kSsGroup) * 4), "scratch")) != SSD_OK) return r;
  if ((r = cu(launch_ss_partials(x, M, K, (float*)ss.p, s), "ss")) != SSD_OK) return r;
  LinearArgs a;
  a.W0 = (const bf16*)Wg;
  a.W1 = (const bf16*)Wu;
  a.R = F;
  a.K = K;
  a.x = x;
  a.ss = (const float*)ss.p;
  a.gain = gain;
  a.eps = eps;
  a.M_static = M;
  a.u = (bf16*)u;
  GemvOpScratch gs(s);
  if ((r = gs.init(F, K, EPI_SWIGLU, a, s)) != SSD_OK) return r;
  Scratch xn(s);
  return launch_norm_fused(EPI_SWIGLU, a, s, xn, "swiglu");
}

ssd_status ssd_op_attention(const float* qkv, int32_t M, int32_t pos0, void* k_cache,
                            void* v_cache, int32_t max_seq, int32_t H, int32_t Hkv, int32_t dh,
                            float theta, void* out, void* stream) {
  if (M < 1 || M > kMaxRows || pos0 < 0 || H <= 0 || Hkv <= 0 || H % Hkv || H / Hkv > 8 ||
      (dh != 64 && dh != 128) || max_seq <= 0 || max_seq % kAttnChunk || pos0 + M > max_seq ||
      !(theta > 0.f))
    return op_fail(SSD_ERR_INVALID_ARG, "attention sizes");
  if (!al16(qkv) || !al16(k_cache) || !al16(v_cache) || !al16(out))
    return op_fail(SSD_ERR_INVALID_ARG, "attention pointers");
  cudaStream_t s = (cudaStream_t)stream;
  ssd_status r;
  Scratch rope(s), part(s), cnt(s), err(s);
  const int half = dh / 2;
  if ((r = cu(rope.alloc((size_t)max_seq * half * sizeof(float2)), "scratch")) != SSD_OK) return r;
  if ((r = cu(part.alloc(attn_part_floats(Hkv, H, dh, max_seq) * 4), "scratch")) != SSD_OK) return r;
  if ((r = cu(cnt.alloc((size_t)Hkv * 4), "scratch")) != SSD_OK) return r;
  if ((r = cu(err.alloc(4), "scratch")) != SSD_OK) return r;
  if ((r = cu(cudaMemsetAsync(cnt.p, 0, (size_t)Hkv * 4, s), "memset")) != SSD_OK) return r;
  if ((r = cu(cudaMemsetAsync(err.p, 0, 4, s), "memset")) != SSD_OK) return r;
  if ((r = cu(launch_rope_table((float2*)rope.p, max_seq, half, (double)theta, s), "rope")) != SSD_OK)
    return r;
  AttnArgs a;
  a.qkv = qkv;
  a.ld_qkv = (H + 2 * Hkv) * dh;
  a.M_static = M;
  a.pos0_static = pos0;
  a.kc = (bf16*)k_cache;
  a.vc = (bf16*)v_cache;
  a.max_seq = max_seq;
  a.H = H;
  a.Hkv = Hkv;
  a.dh = dh;
  a.rope = (const float2*)rope.p;
  a.out = (bf16*)out;
  a.part = (float*)part.p;
  a.counters = (unsigned*)cnt.p;
  a.err = (int*)err.p;
  a.scale = (float)(1.0 / std::sqrt((double)dh));
  if ((r = cu(attn_prepare(a), "attn_prepare")) != SSD_OK) return r;
  return cu(launch_attention(a, s, false), "attention");
}

ssd_status ssd_op_lm_head(const void* W, int32_t V, int32_t D, const float* x, const float* gain,
                          float eps, int32_t M, float temperature, uint64_t seed, int32_t round,
                          int32_t stream_id, int32_t pos0, float* logits, ssd_row_stats* stats,
                          void* stream) {
  ssd_status r = check_linear(W, V, D, M);
  if (r != SSD_OK) return r;
  if (!al16(x) || !al16(gain) || !al16(stats) || (logits && !al16(logits)) || !(eps > 0.f) ||
      !(temperature >= 0.f))
    return op_fail(SSD_ERR_INVALID_ARG, "lm_head pointers / eps / temperature");
  cudaStream_t s = (cudaStream_t)stream;
  Scratch ss(s);
  if ((r = cu(ss.alloc((size_t)M * (D / kSsGroup) * 4), "scratch")) != SSD_OK) return r;
  if ((r = cu(launch_ss_partials(x, M, D, (float*)ss.p, s), "ss")) != SSD_OK) return r;
  LinearArgs a;
  a.W0 = (const bf16*)W;
  a.R = V;
  a.K = D;
  a.x = x;
  a.ss = (const float*)ss.p;
  a.gain = gain;
  a.eps = eps;
  a.M_static = M;
  a.logits = logits;
  a.stats = (RowStats*)stats;
  GemvOpScratch gs(s);
  if ((r = gs.init(V, D, EPI_LMHEAD, a, s)) != SSD_OK) return r;
  a.temperature = temperature;
  a.sample = temperature > 0.f ? 1 : 0;
  a.seed = seed;
  a.round_static = round;
  a.sample_stream = stream_id;
  a.pos0_static = pos0;
  Scratch xn(s);
  return launch_norm_fused(EPI_LMHEAD, a, s, xn, "lm_head");
}

ssd_status ssd_op_accept_stochastic(const float* P, const float* Q, const int32_t* drafts,
                                    int32_t d, int32_t V, float temperature, uint64_t seed,
                                    int32_t round, int32_t n, int32_t* emitted,
                                    int32_t* n_emitted, void* stream) {
  if (!P || (d > 0 && (!Q || !drafts)) || !emitted || !n_emitted || d < 0 || d > kMaxRows - 1 ||
      V <= 0 || !(temperature > 0.f) || n < 0)
    return op_fail(SSD_ERR_INVALID_ARG, "accept arguments");
  AcceptArgs a;
  a.P = P;
  a.Q = Q;
  a.drafts = drafts;
  a.d_static = d;
  a.V = V;
  a.temperature = temperature;
  a.seed = seed;
  a.round_static = round;
  a.n_static = n;
  a.emitted = emitted;
  a.n_emitted = n_emitted;
  return cu(launch_accept_stochastic(a, (cudaStream_t)stream, false), "accept");
}

ssd_status ssd_op_wait_selftest(int32_t polls, int32_t* code_out, void* stream) {
  if (polls < 1 || polls > (1 << 20) || !code_out)
    return op_fail(SSD_ERR_INVALID_ARG, "polls in 1..2^20 and code_out required");
  cudaStream_t s = (cudaStream_t)stream;
  Scratch never(s), code(s);
  ssd_status r;
  if ((r = cu(never.alloc(16), "scratch")) != SSD_OK) return r;
  if ((r = cu(code.alloc(16), "scratch")) != SSD_OK) return r;
  if ((r = cu(cudaMemsetAsync(never.p, 0, 16, s), "memset")) != SSD_OK) return r;
  if ((r = cu(cudaMemsetAsync(code.p, 0xff, 16, s), "memset")) != SSD_OK) return r;
  if ((r = cu(launch_wait_selftest((const unsigned*)never.p, polls, (int32_t*)code.p, s),
              "selftest")) != SSD_OK)
    return r;
  if ((r = cu(cudaMemcpyAsync(code_out, code.p, 4, cudaMemcpyDeviceToHost, s), "copy")) != SSD_OK)
    return r;
  return cu(cudaStreamSynchronize(s), "synchronize");
}

ssd_status ssd_op_philox(const uint32_t* ctr, int32_t count, uint64_t key, uint32_t* out,
                         void* stream) {
  if (count < 0 || (count > 0 && (!al16(ctr) || !al16(out))))
    return op_fail(SSD_ERR_INVALID_ARG, "philox arguments");
  return cu(launch_philox(ctr, count, key, out, (cudaStream_t)stream), "philox");
}

ssd_status ssd_op_linear_rows(const void* W, const void* W1, int32_t R, int32_t K,
                              const void* act, int32_t T, int32_t epi, void* out,
                              const int32_t* map, void* stream) {
  const bool act_packed = (epi & SSD_ROWS_ACT_PACKED) != 0;
  epi &= ~SSD_ROWS_ACT_PACKED;
  if (!al16(W) || (epi == GEMM_SWIGLU && !al16(W1)) || R <= 0 || R % 16 || K <= 0 || K % 32 ||
      T < 1 || !al16(act) || !al16(out) || epi < GEMM_STORE || epi > GEMM_ARGMAX)
    return op_fail(SSD_ERR_INVALID_ARG, "linear_rows arguments");
  cudaStream_t s = (cudaStream_t)stream;
  GemmArgs a;
  a.W0 = (const bf16*)W;
  a.W1 = (const bf16*)W1;
  a.R = R;
  a.K = K;
  a.T = T;
  a.act = (const bf16*)act;
  a.epi = epi;
  Scratch best(s), err(s), packed(s);
  ssd_status r;
  if ((r = cu(err.alloc(16), "scratch")) != SSD_OK) return r;
  if ((r = cu(cudaMemsetAsync(err.p, 0, 16, s), "memset")) != SSD_OK) return r;
  a.err = (int*)err.p;
  // the projection reads its activations in the packed unit layout
  if (!act_packed) {
    const size_t Tp = ((size_t)T + 15) / 16 * 16;
    if ((r = cu(packed.alloc(Tp * K * sizeof(bf16)), "scratch")) != SSD_OK) return r;
    if ((r = cu(launch_pack_act((const bf16*)act, T, K, (bf16*)packed.p, s), "pack_act")) !=
        SSD_OK)
      return r;
    a.act = (const bf16*)packed.p;
  }
  if (epi == GEMM_STORE) a.y = (float*)out;
  if (epi == GEMM_RESID) {
    a.x = (float*)out;
    a.rowmap = map;
  }
  if (epi == GEMM_SWIGLU) a.u = (bf16*)out;
  if (epi == GEMM_ARGMAX) {
    if ((r = cu(best.alloc((size_t)T * 8), "scratch")) != SSD_OK) return r;
    if ((r = cu(cudaMemsetAsync(best.p, 0, (size_t)T * 8, s), "memset")) != SSD_OK) return r;
    a.best = (unsigned long long*)best.p;
  }
  if ((r = cu(launch_gemm_rows(a, s), "linear_rows")) != SSD_OK) return r;
  if (epi == GEMM_ARGMAX)
    return cu(launch_argmax_index(a.best, T, (int32_t*)out, s), "argmax_index");
  return SSD_OK;
}

ssd_status ssd_op_score_attention(const void* q, const int32_t* cand, int32_t n_cand, int32_t N,
                                  int32_t split, const void* k_cache, const void* v_cache,
                                  int32_t max_seq, const void* wk, const void* wv, int32_t w_rows,
                                  int32_t H, int32_t Hkv, int32_t dh, void* out, void* stream) {
  if (!al16(q) || !cand || n_cand < 1 || N < 1 || split < 1 || split > max_seq || w_rows < N ||
      !al16(k_cache) || !al16(v_cache) || !al16(wk) || !al16(wv) || !al16(out) || H < 1 ||
      Hkv < 1 || H % Hkv || (dh != 64 && dh != 128))
    return op_fail(SSD_ERR_INVALID_ARG, "score_attention arguments");
  ScoreAttnArgs a;
  a.q = (const bf16*)q;
  a.kc = (const bf16*)k_cache;
  a.vc = (const bf16*)v_cache;
  a.sk = (const bf16*)wk;
  a.sv = (const bf16*)wv;
  a.cand = cand;
  a.N = N;
  a.split = split;
  a.max_seq = max_seq;
  a.H = H;
  a.Hkv = Hkv;
  a.dh = dh;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)dh));
  a.out = (bf16*)out;
  a.w_rows = w_rows;
  return cu(launch_score_attn(a, n_cand, (cudaStream_t)stream), "score_attention");
}

}  // extern "C"
