// fp32 decoding path (sm_103a): fp32 weights, activations, K/V cache and
// logits, with no rounding anywhere, for models configured with
// SSD_DTYPE_FP32 (the tiny fp32 workload).  The steps are those of the bf16
// path -- RMSNorm-fused projections, attention with RoPE and K/V append,
// o_proj / down with the residual add, SwiGLU, the LM head with its row
// summary -- written as plain CUDA-core kernels: the fp32 models are small
// (their weights sit in L2) and their passes are bound by launch latency,
// not by HBM.
//
// Every reduction has an order fixed by the element's own position (a dot
// product: lane l of the row's warp sums k = l, l + 32, ... in tiles, then a
// butterfly; attention: thread t sums its keys in order, then a fixed tree),
// never by the number of rows processed together, so self-speculative
// greedy output reproduces autoregressive output bit for bit here too.
#include "kernels.cuh"

namespace ssd {

namespace {

constexpr int kTile32 = 512;        // K columns of the input rows staged per step
constexpr int kWarps32 = 8;         // output rows per block (one per warp)
constexpr int kAttnThreads32 = 128;

SSD_DI float warp_sum32(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// y = W act (IN_BF16 here meaning a plain fp32 input) or W rmsnorm(x) g
// (IN_NORM), M <= 16 rows; epilogues: store (rows offset by *row0_dev),
// residual add, SwiGLU (W0 gate, W1 up).
template <int IN, int EPI>
__global__ void __launch_bounds__(kWarps32 * 32) gemv32_kernel(LinearArgs32 a) {
  __shared__ float xs[kMaxRows][kTile32];
  __shared__ float rs[kMaxRows];
  pdl_wait();
  pdl_trigger();
  const int M = rows_of(a.M_static, a.M_dev);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kWarps32 + warp;
  if (IN == IN_NORM) {
    // 1 / sqrt(mean(x^2) + eps) per row: lane-strided sums, then a butterfly
    for (int m = warp; m < M; m += kWarps32) {
      float s = 0.f;
      for (int k = lane; k < a.K; k += 32) {
        const float v = __ldcg(a.x + (size_t)m * a.K + k);
        s = fmaf(v, v, s);
      }
      s = warp_sum32(s);
      if (lane == 0) rs[m] = 1.0f / sqrtf(s / (float)a.K + a.eps);
    }
    __syncthreads();
  }
  float acc[kMaxRows], acc2[kMaxRows];
#pragma unroll
  for (int m = 0; m < kMaxRows; ++m) acc[m] = acc2[m] = 0.f;
  for (int k0 = 0; k0 < a.K; k0 += kTile32) {
    const int tile = min(kTile32, a.K - k0);
    for (int e = threadIdx.x; e < M * tile; e += kWarps32 * 32) {
      const int m = e / tile, k = e % tile;
      xs[m][k] = IN == IN_NORM ? __ldcg(a.x + (size_t)m * a.K + k0 + k) * rs[m] * a.gain[k0 + k]
                               : __ldcg(a.act + (size_t)m * a.K + k0 + k);
    }
    __syncthreads();
    if (r < a.R) {
      const float* w0 = a.W0 + (size_t)r * a.K + k0;
      const float* w1 = EPI == EPI_SWIGLU ? a.W1 + (size_t)r * a.K + k0 : nullptr;
      for (int k = lane; k < tile; k += 32) {
        const float wv = w0[k];
        const float wu = EPI == EPI_SWIGLU ? w1[k] : 0.f;
#pragma unroll
        for (int m = 0; m < kMaxRows; ++m) {
          if (m < M) {
            acc[m] = fmaf(wv, xs[m][k], acc[m]);
            if (EPI == EPI_SWIGLU) acc2[m] = fmaf(wu, xs[m][k], acc2[m]);
          }
        }
      }
    }
    __syncthreads();
  }
  if (r >= a.R) return;
#pragma unroll
  for (int m = 0; m < kMaxRows; ++m) {
    if (m < M) {
      const float v = warp_sum32(acc[m]);
      const float v2 = EPI == EPI_SWIGLU ? warp_sum32(acc2[m]) : 0.f;
      if (lane == 0) {
        if (EPI == EPI_STORE) {
          const int row0 = a.row0_dev ? __ldcg(a.row0_dev) : 0;
          a.y[(size_t)(row0 + m) * a.R + r] = v;
        } else if (EPI == EPI_RESID) {
          float* xp = a.xres + (size_t)m * a.R + r;
          *xp = *xp + v;
        } else if (EPI == EPI_SWIGLU) {
          a.u[(size_t)m * a.R + r] = v / (1.0f + expf(-v)) * v2;
        }
      }
    }
  }
}

// Row summary of logits rows [slot + m], m < M (one block per row): top-1 /
// top-2 (value desc, index asc), lse, conf, lse of z / T and the Gumbel-max
// sample of softmax(z / T) with the noise of (v, pos0 + m + 1, round,
// stream) -- what the bf16 LM head's summary computes.  Each thread takes
// v = t, t + nthr, ... in order; the block combines in a fixed tree.
__global__ void __launch_bounds__(256) lm_summary32_kernel(LmSummaryArgs32 a) {
  __shared__ float sv1[256], sv2[256], sg[256], ssum[256], ssumt[256];
  __shared__ int si1[256], si2[256], sgi[256];
  pdl_wait();
  pdl_trigger();
  const int M = rows_of(a.M_static, a.M_dev);
  const int m = blockIdx.x;
  if (m >= M) return;
  const int slot = a.slot_dev ? __ldcg(a.slot_dev) : 0;
  const int round = a.round_dev ? __ldcg(a.round_dev) : a.round_static;
  const int pos0 = a.pos0_dev ? __ldcg(a.pos0_dev) : a.pos0_static;
  const float T = a.temperature;
  const float* z = a.logits + (size_t)(slot + m) * a.V;
  const int t = threadIdx.x, nt = blockDim.x;
  float v1 = -INFINITY, v2 = -INFINITY, gv = -INFINITY;
  int i1 = 0x7fffffff, i2 = 0x7fffffff, gi = 0x7fffffff;
  for (int v = t; v < a.V; v += nt) {
    const float zv = __ldcg(z + v);
    if (better(zv, v, v1, i1)) {
      v2 = v1; i2 = i1; v1 = zv; i1 = v;
    } else if (better(zv, v, v2, i2)) {
      v2 = zv; i2 = v;
    }
    if (T > 0.f && a.sample) {
      const float sc = zv / T + gumbel_at(a.seed, v, pos0 + m + 1, round, a.stream);
      if (better(sc, v, gv, gi)) { gv = sc; gi = v; }
    }
  }
  sv1[t] = v1; si1[t] = i1; sv2[t] = v2; si2[t] = i2; sg[t] = gv; sgi[t] = gi;
  __syncthreads();
  for (int h = nt / 2; h > 0; h >>= 1) {
    if (t < h) {
      float a1 = sv1[t], a2 = sv2[t];
      int b1 = si1[t], b2 = si2[t];
      const float c1 = sv1[t + h], c2 = sv2[t + h];
      const int d1 = si1[t + h], d2 = si2[t + h];
      // merge two top-2 lists under the total order
      if (better(c1, d1, a1, b1)) {
        if (better(a1, b1, c2, d2)) { a2 = a1; b2 = b1; } else { a2 = c2; b2 = d2; }
        a1 = c1; b1 = d1;
      } else if (better(c1, d1, a2, b2)) {
        a2 = c1; b2 = d1;
      }
      sv1[t] = a1; si1[t] = b1; sv2[t] = a2; si2[t] = b2;
      if (better(sg[t + h], sgi[t + h], sg[t], sgi[t])) { sg[t] = sg[t + h]; sgi[t] = sgi[t + h]; }
    }
    __syncthreads();
  }
  const float z1 = sv1[0];
  float s = 0.f, st = 0.f;
  for (int v = t; v < a.V; v += nt) {
    const float zv = __ldcg(z + v);
    s += expf(zv - z1);
    if (T > 0.f) st += expf(zv / T - z1 / T);
  }
  ssum[t] = s;
  ssumt[t] = st;
  __syncthreads();
  for (int h = nt / 2; h > 0; h >>= 1) {
    if (t < h) {
      ssum[t] += ssum[t + h];
      ssumt[t] += ssumt[t + h];
    }
    __syncthreads();
  }
  if (t == 0) {
    RowStats rsm;
    rsm.top1 = si1[0];
    rsm.top2 = si2[0];
    rsm.sample = T > 0.f && a.sample ? sgi[0] : si1[0];
    rsm.pad = 0;
    rsm.z1 = z1;
    rsm.z2 = sv2[0];
    rsm.lse = z1 + logf(ssum[0]);
    rsm.conf = expf(z1 - rsm.lse);
    rsm.lse_t = T > 0.f ? z1 / T + logf(ssumt[0]) : rsm.lse;
    rsm.pad2[0] = rsm.pad2[1] = rsm.pad2[2] = 0.f;
    a.stats[slot + m] = rsm;
  }
}

// RoPE and append: row m's key (rotate-half at position pos0 + m) and value,
// fp32, into the cache.
__global__ void attn32_append_kernel(AttnArgs32 a) {
  pdl_wait();
  pdl_trigger();
  const int M = rows_of(a.M_static, a.M_dev);
  const int pos0 = a.pos0_dev ? __ldcg(a.pos0_dev) : a.pos0_static;
  const int m = blockIdx.x, kvh = blockIdx.y;
  if (m >= M) return;
  const int half = a.dh / 2, pos = pos0 + m;
  const float* kr = a.qkv + (size_t)m * a.ld_qkv + (size_t)(a.H + kvh) * a.dh;
  const float* vr = kr + (size_t)a.Hkv * a.dh;
  float* kd = a.kc + ((size_t)kvh * a.max_seq + pos) * a.dh;
  float* vd = a.vc + ((size_t)kvh * a.max_seq + pos) * a.dh;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const float2 cs = a.rope[(size_t)pos * half + i];
    const float k0 = __ldcg(kr + i), k1 = __ldcg(kr + i + half);
    kd[i] = k0 * cs.x - k1 * cs.y;
    kd[i + half] = k0 * cs.y + k1 * cs.x;
    vd[i] = __ldcg(vr + i);
    vd[i + half] = __ldcg(vr + i + half);
  }
}

// Causal attention of row m, query head h (one block): keys 0..pos0 + m of
// KV head h / (H / Hkv).
__global__ void __launch_bounds__(kAttnThreads32) attn32_kernel(AttnArgs32 a) {
  extern __shared__ float s32[];  // [dh] query, then [max_seq] scores
  __shared__ float red[kAttnThreads32];
  pdl_wait();
  pdl_trigger();
  const int M = rows_of(a.M_static, a.M_dev);
  const int pos0 = a.pos0_dev ? __ldcg(a.pos0_dev) : a.pos0_static;
  const int h = blockIdx.x, m = blockIdx.y;
  if (m >= M) return;
  const int dh = a.dh, half = dh / 2, t = threadIdx.x, nt = blockDim.x;
  const int kvh = h / (a.H / a.Hkv), pos = pos0 + m, nk = pos + 1;
  float* q = s32;
  float* sc = s32 + dh;
  const float* qr = a.qkv + (size_t)m * a.ld_qkv + (size_t)h * dh;
  for (int i = t; i < half; i += nt) {
    const float2 cs = a.rope[(size_t)pos * half + i];
    const float q0 = __ldcg(qr + i), q1 = __ldcg(qr + i + half);
    q[i] = q0 * cs.x - q1 * cs.y;
    q[i + half] = q0 * cs.y + q1 * cs.x;
  }
  __syncthreads();
  const float* kb = a.kc + (size_t)kvh * a.max_seq * dh;
  const float* vb = a.vc + (size_t)kvh * a.max_seq * dh;
  float mx = -INFINITY;
  for (int j = t; j < nk; j += nt) {
    const float* k = kb + (size_t)j * dh;
    float d = 0.f;
    for (int i = 0; i < dh; ++i) d = fmaf(q[i], __ldcg(k + i), d);
    sc[j] = d * a.scale;
    mx = fmaxf(mx, sc[j]);
  }
  red[t] = mx;
  __syncthreads();
  for (int s = nt / 2; s > 0; s >>= 1) {
    if (t < s) red[t] = fmaxf(red[t], red[t + s]);
    __syncthreads();
  }
  mx = red[0];
  __syncthreads();
  float l = 0.f;
  for (int j = t; j < nk; j += nt) {
    const float p = expf(sc[j] - mx);
    sc[j] = p;
    l += p;
  }
  red[t] = l;
  __syncthreads();
  for (int s = nt / 2; s > 0; s >>= 1) {
    if (t < s) red[t] += red[t + s];
    __syncthreads();
  }
  const float L = red[0];
  for (int dd = t; dd < dh; dd += nt) {
    float o = 0.f;
    for (int j = 0; j < nk; ++j) o = fmaf(sc[j], __ldcg(vb + (size_t)j * dh + dd), o);
    a.out[(size_t)m * a.H * dh + (size_t)h * dh + dd] = o / L;
  }
}

template <class K, class... Args>
cudaError_t launch32(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                     Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, kernel, args...);
}

}  // namespace

cudaError_t launch_gemv32(int in_mode, int epi, const LinearArgs32& a, cudaStream_t st, bool pdl) {
  if (a.R <= 0 || a.K <= 0 || (epi == EPI_SWIGLU && !a.W1)) return cudaErrorInvalidValue;
  const dim3 grid((a.R + kWarps32 - 1) / kWarps32), block(kWarps32 * 32);
#define SSD_GEMV32_CASE(I, E) \
  if (in_mode == I && epi == E) return launch32(gemv32_kernel<I, E>, grid, block, 0, st, pdl, a);
  SSD_GEMV32_CASE(IN_NORM, EPI_STORE)
  SSD_GEMV32_CASE(IN_BF16, EPI_STORE)
  SSD_GEMV32_CASE(IN_BF16, EPI_RESID)
  SSD_GEMV32_CASE(IN_NORM, EPI_SWIGLU)
#undef SSD_GEMV32_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_lm_summary32(const LmSummaryArgs32& a, cudaStream_t st, bool pdl) {
  return launch32(lm_summary32_kernel, dim3(kMaxRows), dim3(256), 0, st, pdl, a);
}

size_t attn32_smem(int dh, int max_seq) { return (size_t)(dh + max_seq) * sizeof(float); }

cudaError_t attn32_prepare(int dh, int max_seq) {
  const size_t smem = attn32_smem(dh, max_seq);
  if (smem <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(attn32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_attention32(const AttnArgs32& a, cudaStream_t st, bool pdl) {
  if (a.dh % 2 || a.H % a.Hkv) return cudaErrorInvalidValue;
  cudaError_t e = launch32(attn32_append_kernel, dim3(kMaxRows, a.Hkv), dim3(64), 0, st, pdl, a);
  if (e != cudaSuccess) return e;
  return launch32(attn32_kernel, dim3(a.H, kMaxRows), dim3(kAttnThreads32),
                  attn32_smem(a.dh, a.max_seq), st, pdl, a);
}

}  // namespace ssd
