// Small-M weight-streaming GEMV on the tensor cores (sm_103a).
//
// y[m][r] = sum_k W[r][k] act[m][k] for M <= 16 rows (token positions).  At
// batch 1 every decoder projection is a matrix-vector product whose cost is
// reading W once from HBM; the same kernel serves the M = d+1 verify pass
// and the 16-row prefill chunks.
//
// Work partition.  W is cut into units of 16 rows x 32 columns (1 KB of
// bf16).  Units are ordered row-group-major and split into equal contiguous
// ranges, one per warp of a fixed grid of kGridCtas CTAs (two resident CTAs
// on each of the 152 SMs), so every warp streams the same number of bytes
// and all CTAs run in a single wave.  A 16-row group whose units span
// several warps ("segments") is finished by the last of those warps to
// complete: it sums the segments' partials in segment order and applies the
// epilogue.  The partition depends only on the matrix shape.
//
// Tensor-core mapping.  One m16n8k16 MMA consumes 16 rows x 16 K of W against
// 16 K x 8 token columns (M <= 8 uses one column tile, M <= 16 two).  The K
// order inside each 32-wide block is permuted consistently for W and the
// activations so that a lane's 16-byte load is exactly its A fragment for
// two MMAs: lane (g, c) holds W[g][8c..8c+7] and W[g+8][8c..8c+7]; the first
// MMA takes elements 0-3, the second 4-7.  Weights stream straight from HBM
// into two register buffers (one in flight while the other feeds the MMAs);
// activations are staged once per CTA in shared memory when they fit.
//
// Reduction order.  Inside a segment each output accumulates its K blocks in
// ascending order; segments are summed in order; nothing depends on M, so a
// column's bits do not change with the number of rows processed together.
// That is what makes self-speculative verification reproduce
// autoregressive decoding bit for bit.
#include "kernels.cuh"

namespace ssd {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kGridCtas = 304;                  // 2 resident CTAs x 152 SMs
constexpr int kTotalWarps = kGridCtas * kWarps;
constexpr int kUnroll = 4;                      // units per pipeline stage
constexpr int kStageBytes = 88 * 1024;          // activation staging budget (2 CTAs/SM)
constexpr int kPad = 8;                         // bf16 row padding in the stage
constexpr int kLmBlock = 32;                    // LM-head row groups per level-2 block

struct Part {
  long long T;  // units = NRG * KB
  int NRG;      // (virtual) 16-row groups
  int KB;       // 32-wide K blocks
  int W;        // warps with work = min(kTotalWarps, T)
  int segmax;   // stride of the partial buffer per row group
};

__host__ __device__ inline long long unit_begin(const Part& p, int w) {
  return (long long)w * p.T / p.W;
}
// first / last warp whose unit range intersects units [a, b)
__host__ __device__ inline int warp_first(const Part& p, long long a) {
  return (int)(((a + 1) * p.W + p.T - 1) / p.T) - 1;
}
__host__ __device__ inline int warp_last(const Part& p, long long b) {
  return (int)((b * p.W + p.T - 1) / p.T) - 1;
}
__host__ __device__ inline int nseg(const Part& p, int vr) {
  return warp_last(p, (long long)(vr + 1) * p.KB) - warp_first(p, (long long)vr * p.KB) + 1;
}

Part make_part(int R, int K, int epi) {
  Part p;
  p.NRG = (epi == EPI_SWIGLU ? 2 : 1) * (R / 16);
  p.KB = K / 32;
  p.T = (long long)p.NRG * p.KB;
  p.W = (int)(p.T < kTotalWarps ? p.T : kTotalWarps);
  p.segmax = (p.W + p.NRG - 1) / p.NRG + 1;
  return p;
}

// B fragment (8 consecutive K of token t) for the permuted MMA layout,
// read from global memory.
template <int IN>
SSD_DI uint4 load_b_global(const LinearArgs& a, int t, int off, const float* rstd) {
  if (IN == IN_BF16) {
    return *reinterpret_cast<const uint4*>(a.act + (size_t)t * a.K + off);
  } else {
    const float4* xp = reinterpret_cast<const float4*>(a.x + (size_t)t * a.K + off);
    const float4* gp = reinterpret_cast<const float4*>(a.gain + off);
    const float4 x0 = xp[0], x1 = xp[1], g0 = gp[0], g1 = gp[1];
    const float r = rstd[t];
    return make_uint4(pack_bf16x2(x0.x * r * g0.x, x0.y * r * g0.y),
                      pack_bf16x2(x0.z * r * g0.z, x0.w * r * g0.w),
                      pack_bf16x2(x1.x * r * g1.x, x1.y * r * g1.y),
                      pack_bf16x2(x1.z * r * g1.z, x1.w * r * g1.w));
  }
}

template <int IN, bool SMEM>
SSD_DI uint4 load_b(const LinearArgs& a, const bf16* stage, int t, int off, bool valid,
                    const float* rstd) {
  if (!valid) return make_uint4(0u, 0u, 0u, 0u);
  if (SMEM) return *reinterpret_cast<const uint4*>(stage + (size_t)t * (a.K + kPad) + off);
  return load_b_global<IN>(a, t, off, rstd);
}

// Row pointer of unit u for lane (g, c): W[row0 + g][kb*32 + 8c].
template <int EPI>
SSD_DI const bf16* unit_ptr(const LinearArgs& a, const Part& p, long long u, int g, int c) {
  const int vr = (int)(u / p.KB);
  const int kb = (int)(u - (long long)vr * p.KB);
  const bf16* W = a.W0;
  int row0 = vr * 16;
  if (EPI == EPI_SWIGLU) {
    W = (vr & 1) ? a.W1 : a.W0;
    row0 = (vr >> 1) * 16;
  }
  return W + (size_t)(row0 + g) * a.K + kb * 32 + 8 * c;
}

struct WBuf {
  uint4 a[kUnroll], b[kUnroll];
};

template <int EPI>
SSD_DI void load_w(WBuf& w, const LinearArgs& a, const Part& p, long long u, long long u1,
                   int lane) {
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int i = 0; i < kUnroll; ++i) {
    if (u + i < u1) {
      const bf16* q = unit_ptr<EPI>(a, p, u + i, g, c);
      w.a[i] = ld_stream_u4(q);
      w.b[i] = ld_stream_u4(q + (size_t)8 * a.K);
    }
  }
}

// ---------------------------------------------------------------- reductions

// Warp-level top-2 merge under the (value desc, index asc) total order.
SSD_DI void top2_insert(float v, int i, float& v1, int& i1, float& v2, int& i2) {
  if (better(v, i, v1, i1)) {
    v2 = v1; i2 = i1; v1 = v; i1 = i;
  } else if (better(v, i, v2, i2)) {
    v2 = v; i2 = i;
  }
}

SSD_DI void top2_warp(float& v1, int& i1, float& v2, int& i2) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov1 = __shfl_xor_sync(0xffffffffu, v1, o);
    const int oi1 = __shfl_xor_sync(0xffffffffu, i1, o);
    const float ov2 = __shfl_xor_sync(0xffffffffu, v2, o);
    const int oi2 = __shfl_xor_sync(0xffffffffu, i2, o);
    top2_insert(ov1, oi1, v1, i1, v2, i2);
    top2_insert(ov2, oi2, v1, i1, v2, i2);
  }
}

SSD_DI void argmax_warp(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

SSD_DI float sum_warp(float s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// LM-head summary record of a set of vocabulary rows for one token:
// {max z, argmax, second z, its id, sum exp(z - max), sum exp(z/T - max/T),
//  best Gumbel score, its id}
struct LmRec {
  float v1, v2, se, set, gv;
  int i1, i2, gi;
};

SSD_DI void lm_store(float* p, const LmRec& r) {
  reinterpret_cast<float4*>(p)[0] = make_float4(r.v1, __int_as_float(r.i1), r.v2, __int_as_float(r.i2));
  reinterpret_cast<float4*>(p)[1] = make_float4(r.se, r.set, r.gv, __int_as_float(r.gi));
}

SSD_DI LmRec lm_load(const float* p) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
  LmRec r;
  r.v1 = a.x; r.i1 = __float_as_int(a.y); r.v2 = a.z; r.i2 = __float_as_int(a.w);
  r.se = b.x; r.set = b.y; r.gv = b.z; r.gi = __float_as_int(b.w);
  return r;
}

SSD_DI LmRec lm_empty() {
  LmRec r;
  r.v1 = r.v2 = r.gv = -INFINITY;
  r.i1 = r.i2 = r.gi = 0x7fffffff;
  r.se = r.set = 0.f;
  return r;
}

// Merge the per-lane records of a warp (a butterfly, identical in every lane).
// Sums are rescaled to the merged maximum before being added.
SSD_DI LmRec lm_merge_warp(LmRec r, float T) {
  float v1 = r.v1, v2 = r.v2, gv = r.gv;
  int i1 = r.i1, i2 = r.i2, gi = r.gi;
  top2_warp(v1, i1, v2, i2);
  argmax_warp(gv, gi);
  const float mx = v1;
  float s = r.v1 == -INFINITY ? 0.f : r.se * expf(r.v1 - mx);
  float st = 0.f;
  if (T > 0.f) st = r.v1 == -INFINITY ? 0.f : r.set * expf(r.v1 / T - mx / T);
  s = sum_warp(s);
  st = sum_warp(st);
  LmRec o;
  o.v1 = v1; o.i1 = i1; o.v2 = v2; o.i2 = i2; o.gv = gv; o.gi = gi; o.se = s; o.set = st;
  return o;
}

// ---------------------------------------------------------------- kernel

template <int IN, int EPI>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(LinearArgs a, Part p) {
  __shared__ float rstd_s[kMaxRows];
  __shared__ float ep[kWarps][2][16][17];   // per-warp epilogue scratch
  extern __shared__ __align__(16) unsigned char stage_raw[];
  bf16* stage = reinterpret_cast<bf16*>(stage_raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int w = blockIdx.x * kWarps + warp;
  const bool has_work = w < p.W;
  const long long u0 = has_work ? unit_begin(p, w) : 0;
  const long long u1 = has_work ? unit_begin(p, w + 1) : 0;

  // Weights do not depend on the preceding kernel: start streaming them
  // before waiting for its results.
  WBuf A, B;
  if (has_work) load_w<EPI>(A, a, p, u0, u1, lane);

  pdl_wait();
  pdl_trigger();

  const int M = rows_of(a.M_static, a.M_dev);
  if (IN == IN_NORM) {
    // 1 / sqrt(mean(x^2) + eps) per row from the producer's partials, in a
    // fixed order: lane l sums partials l, l+32, ... then a butterfly.
    const int NP = a.K / kSsGroup;
    for (int m = warp; m < M; m += kWarps) {
      float s = 0.f;
      for (int q = lane; q < NP; q += 32) s += a.ss[(size_t)m * NP + q];
      s = sum_warp(s);
      if (lane == 0) rstd_s[m] = 1.0f / sqrtf(s / (float)a.K + a.eps);
    }
    __syncthreads();
  }
  const bool use_smem = (size_t)M * (a.K + kPad) * sizeof(bf16) <= (size_t)kStageBytes;
  if (use_smem) {
    const int vpr = a.K / 8;  // 16-byte pieces per row
    for (int e = threadIdx.x; e < M * vpr; e += kThreads) {
      const int m = e / vpr, q = e % vpr;
      reinterpret_cast<uint4*>(stage + (size_t)m * (a.K + kPad))[q] =
          load_b_global<IN>(a, m, q * 8, rstd_s);
    }
    __syncthreads();
  }
  if (!has_work) return;

  const bool two = M > 8;
  const bool v0 = g < M, v1 = two && (g + 8) < M;
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  int cur = (int)(u0 / p.KB);

  // Flush the accumulators of row group `vr` into its segment slot; the last
  // warp to finish the group (or the gate/up pair) runs the epilogue.
  auto flush = [&](int vr) {
    const int seg = w - warp_first(p, (long long)vr * p.KB);
    float* dst = a.part + ((size_t)vr * p.segmax + seg) * 256;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int tok = t * 8 + 2 * c;
      if (tok < M) {
        dst[g * 16 + tok] = acc[t][0];
        dst[(g + 8) * 16 + tok] = acc[t][2];
      }
      if (tok + 1 < M) {
        dst[g * 16 + tok + 1] = acc[t][1];
        dst[(g + 8) * 16 + tok + 1] = acc[t][3];
      }
    }
    __threadfence();
    __syncwarp();
    const int cidx = EPI == EPI_SWIGLU ? vr >> 1 : vr;
    int last = 0;
    if (lane == 0) {
      int expect = nseg(p, vr);
      if (EPI == EPI_SWIGLU) expect += nseg(p, vr ^ 1);
      last = atomicAdd(a.counter + cidx, 1u) == (unsigned)(expect - 1);
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    // sum the segments of the group(s) in segment order
    const int ngrp = EPI == EPI_SWIGLU ? 2 : 1;
    for (int h = 0; h < ngrp; ++h) {
      const int gv = EPI == EPI_SWIGLU ? ((vr & ~1) | h) : vr;
      const int ns = nseg(p, gv);
      const float* src = a.part + (size_t)gv * p.segmax * 256;
      for (int e = lane; e < 16 * M; e += 32) {
        const int row = e / M, tok = e % M;
        float s = 0.f;
        for (int sg = 0; sg < ns; ++sg) s += __ldcg(src + (size_t)sg * 256 + row * 16 + tok);
        ep[warp][h][row][tok] = s;
      }
    }
    __syncwarp();
    if (lane == 0) a.counter[cidx] = 0u;
    if (EPI == EPI_STORE) {
      const int row0 = vr * 16;
      for (int e = lane; e < 16 * M; e += 32) {
        const int row = e / M, tok = e % M;
        a.y[(size_t)tok * a.R + row0 + row] = ep[warp][0][row][tok];
      }
    } else if (EPI == EPI_RESID) {
      const int row0 = vr * 16;
      for (int e = lane; e < 16 * M; e += 32) {
        const int row = e / M, tok = e % M;
        const size_t idx = (size_t)tok * a.R + row0 + row;
        const float xn = a.xres[idx] + ep[warp][0][row][tok];
        a.xres[idx] = xn;
        ep[warp][0][row][tok] = xn;
      }
      __syncwarp();
      if (lane < M) {
        float s = 0.f;
        for (int row = 0; row < 16; ++row) s += ep[warp][0][row][lane] * ep[warp][0][row][lane];
        a.ss_out[(size_t)lane * (a.R / kSsGroup) + vr] = s;
      }
    } else if (EPI == EPI_SWIGLU) {
      const int row0 = (vr >> 1) * 16;
      for (int e = lane; e < 16 * M; e += 32) {
        const int row = e / M, tok = e % M;
        const float gt = ep[warp][0][row][tok];
        const float up = ep[warp][1][row][tok];
        const float sl = gt / (1.0f + expf(-gt));
        a.u[(size_t)tok * a.R + row0 + row] = __float2bfloat16_rn(sl * up);
      }
    } else if (EPI == EPI_LMHEAD) {
      const int slot = a.slot_dev ? *a.slot_dev : 0;
      const int row0 = vr * 16;
      const float T = a.temperature;
      if (a.logits) {
        for (int e = lane; e < 16 * M; e += 32) {
          const int row = e / M, tok = e % M;
          a.logits[(size_t)(slot + tok) * a.R + row0 + row] = ep[warp][0][row][tok];
        }
      }
      const int round = a.round_dev ? *a.round_dev : a.round_static;
      const int pos0 = a.pos0_dev ? *a.pos0_dev : a.pos0_static;
      // level 1: the group's 16 rows, sequentially, one lane per token
      if (lane < M) {
        LmRec r = lm_empty();
        for (int row = 0; row < 16; ++row) {
          const float z = ep[warp][0][row][lane];
          top2_insert(z, row0 + row, r.v1, r.i1, r.v2, r.i2);
          if (T > 0.f) {
            const float sc = z / T + gumbel_at(a.seed, row0 + row, pos0 + lane + 1, round,
                                               a.sample_stream);
            if (better(sc, row0 + row, r.gv, r.gi)) { r.gv = sc; r.gi = row0 + row; }
          }
        }
        for (int row = 0; row < 16; ++row) {
          const float z = ep[warp][0][row][lane];
          r.se += expf(z - r.v1);
          if (T > 0.f) r.set += expf(z / T - r.v1 / T);
        }
        lm_store(a.rec + ((size_t)vr * kMaxRows + lane) * 8, r);
      }
      __threadfence();
      __syncwarp();
      // level 2: blocks of kLmBlock groups
      const int nb = (p.NRG + kLmBlock - 1) / kLmBlock;
      const int blk = vr / kLmBlock;
      const int blk_n = min(kLmBlock, p.NRG - blk * kLmBlock);
      unsigned* c2 = a.counter + p.NRG;
      int last2 = 0;
      if (lane == 0) last2 = atomicAdd(c2 + blk, 1u) == (unsigned)(blk_n - 1);
      last2 = __shfl_sync(0xffffffffu, last2, 0);
      if (!last2) return;
      __threadfence();
      float* rec2 = a.rec + (size_t)p.NRG * kMaxRows * 8;
      for (int tok = 0; tok < M; ++tok) {
        const int gi = blk * kLmBlock + lane;
        LmRec r = lane < blk_n ? lm_load(a.rec + ((size_t)gi * kMaxRows + tok) * 8) : lm_empty();
        r = lm_merge_warp(r, T);
        if (lane == 0) lm_store(rec2 + ((size_t)blk * kMaxRows + tok) * 8, r);
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) c2[blk] = 0u;
      int last3 = 0;
      if (lane == 0) last3 = atomicAdd(c2 + nb, 1u) == (unsigned)(nb - 1);
      last3 = __shfl_sync(0xffffffffu, last3, 0);
      if (!last3) return;
      __threadfence();
      // level 3: all blocks; lane b takes blocks b, b+32, ... in order
      for (int tok = 0; tok < M; ++tok) {
        LmRec r = lm_empty();
        for (int b = lane; b < nb; b += 32) {
          const LmRec q = lm_load(rec2 + ((size_t)b * kMaxRows + tok) * 8);
          const float mx = fmaxf(r.v1, q.v1);
          const float se = (r.v1 == -INFINITY ? 0.f : r.se * expf(r.v1 - mx)) +
                           q.se * expf(q.v1 - mx);
          float set = 0.f;
          if (T > 0.f)
            set = (r.v1 == -INFINITY ? 0.f : r.set * expf(r.v1 / T - mx / T)) +
                  q.set * expf(q.v1 / T - mx / T);
          top2_insert(q.v1, q.i1, r.v1, r.i1, r.v2, r.i2);
          top2_insert(q.v2, q.i2, r.v1, r.i1, r.v2, r.i2);
          if (better(q.gv, q.gi, r.gv, r.gi)) { r.gv = q.gv; r.gi = q.gi; }
          r.se = se;
          r.set = set;
        }
        r = lm_merge_warp(r, T);
        if (lane == 0) {
          RowStats rs;
          rs.top1 = r.i1;
          rs.top2 = r.i2;
          rs.sample = T > 0.f ? r.gi : r.i1;
          rs.pad = 0;
          rs.z1 = r.v1;
          rs.z2 = r.v2;
          rs.lse = r.v1 + logf(r.se);
          rs.conf = expf(r.v1 - rs.lse);
          rs.lse_t = T > 0.f ? r.v1 / T + logf(r.set) : rs.lse;
          rs.pad2[0] = rs.pad2[1] = rs.pad2[2] = 0.f;
          a.stats[slot + tok] = rs;
        }
      }
      if (lane == 0) c2[nb] = 0u;
    }
  };

  // Main loop over this warp's units: two register buffers in flight.
  auto consume = [&](const WBuf& wb, long long u) {
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
      const long long uu = u + i;
      if (uu < u1) {
        const int vr = (int)(uu / p.KB);
        if (vr != cur) {
          flush(cur);
#pragma unroll
          for (int t = 0; t < 2; ++t)
            acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
          cur = vr;
        }
        const int off = (int)(uu - (long long)vr * p.KB) * 32 + 8 * c;
        if (use_smem) {
          const uint4 xa = load_b<IN, true>(a, stage, g, off, v0, rstd_s);
          mma_bf16(acc[0], wb.a[i].x, wb.b[i].x, wb.a[i].y, wb.b[i].y, xa.x, xa.y);
          mma_bf16(acc[0], wb.a[i].z, wb.b[i].z, wb.a[i].w, wb.b[i].w, xa.z, xa.w);
          if (two) {
            const uint4 xb = load_b<IN, true>(a, stage, g + 8, off, v1, rstd_s);
            mma_bf16(acc[1], wb.a[i].x, wb.b[i].x, wb.a[i].y, wb.b[i].y, xb.x, xb.y);
            mma_bf16(acc[1], wb.a[i].z, wb.b[i].z, wb.a[i].w, wb.b[i].w, xb.z, xb.w);
          }
        } else {
          const uint4 xa = load_b<IN, false>(a, stage, g, off, v0, rstd_s);
          mma_bf16(acc[0], wb.a[i].x, wb.b[i].x, wb.a[i].y, wb.b[i].y, xa.x, xa.y);
          mma_bf16(acc[0], wb.a[i].z, wb.b[i].z, wb.a[i].w, wb.b[i].w, xa.z, xa.w);
          if (two) {
            const uint4 xb = load_b<IN, false>(a, stage, g + 8, off, v1, rstd_s);
            mma_bf16(acc[1], wb.a[i].x, wb.b[i].x, wb.a[i].y, wb.b[i].y, xb.x, xb.y);
            mma_bf16(acc[1], wb.a[i].z, wb.b[i].z, wb.a[i].w, wb.b[i].w, xb.z, xb.w);
          }
        }
      }
    }
  };

  long long u = u0;
  while (u < u1) {
    if (u + kUnroll < u1) load_w<EPI>(B, a, p, u + kUnroll, u1, lane);
    consume(A, u);
    u += kUnroll;
    if (u >= u1) break;
    if (u + kUnroll < u1) load_w<EPI>(A, a, p, u + kUnroll, u1, lane);
    consume(B, u);
    u += kUnroll;
  }
  flush(cur);
}

template <int IN, int EPI>
cudaError_t launch_one(const LinearArgs& a, const Part& p, cudaStream_t st, bool pdl) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(gemv_kernel<IN, EPI>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kStageBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(kGridCtas);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = kStageBytes;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, gemv_kernel<IN, EPI>, a, p);
}

}  // namespace

GemvScratch gemv_scratch(int R, int K, int epi) {
  const Part p = make_part(R, K, epi);
  GemvScratch s;
  s.part_floats = (size_t)p.NRG * p.segmax * 256;
  const int nb = (p.NRG + kLmBlock - 1) / kLmBlock;
  s.counters = (size_t)p.NRG + nb + 1;
  s.rec_floats = epi == EPI_LMHEAD ? (size_t)(p.NRG + nb) * kMaxRows * 8 : 0;
  return s;
}

cudaError_t launch_gemv(int in_mode, int epi, const LinearArgs& a, cudaStream_t st, bool pdl) {
  const Part p = make_part(a.R, a.K, epi);
#define SSD_GEMV_CASE(I, E) \
  if (in_mode == I && epi == E) return launch_one<I, E>(a, p, st, pdl);
  SSD_GEMV_CASE(IN_BF16, EPI_STORE)
  SSD_GEMV_CASE(IN_NORM, EPI_STORE)
  SSD_GEMV_CASE(IN_BF16, EPI_RESID)
  SSD_GEMV_CASE(IN_NORM, EPI_SWIGLU)
  SSD_GEMV_CASE(IN_NORM, EPI_LMHEAD)
#undef SSD_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace ssd
