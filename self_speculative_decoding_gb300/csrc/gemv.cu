// Small-M weight-streaming GEMV on the tensor cores (sm_103a).
//
// y[m][r] = sum_k W[r][k] act[m][k] for M <= 16 rows (token positions).  At
// batch 1 every decoder projection is a matrix-vector product whose cost is
// reading W once from HBM; the same kernel serves the M = d+1 verify pass
// and the 16-row prefill chunks.
//
// Mapping.  A warp owns 16 rows of W (one 16-row group) and a contiguous
// slice of K; a CTA of 8 warps owns RG row groups x KS K-slices.  Each lane
// streams 16-byte pieces of two rows straight from HBM into registers, and
// one m16n8k16 tensor-core MMA consumes a 16x16 tile of W against a 16x8
// tile of activations (8 token columns; M <= 8 uses one column tile, M <= 16
// two).  The K order inside each 32-wide block is permuted consistently for
// W and the activations so that a lane's 16-byte load is exactly its A
// fragment for two MMAs: lane (g, c) holds W[g][8c..8c+7] and
// W[g+8][8c..8c+7]; the first MMA takes elements 0-3, the second 4-7.
//
// Reduction order.  Each output element accumulates its K blocks in
// ascending order inside one warp (two MMAs per block), the KS warp partials
// are summed in warp order, and nothing depends on M: a column's bits do not
// change with the number of rows processed together.  That is what makes
// self-speculative verification reproduce autoregressive decoding bit for
// bit.
#include "kernels.cuh"

namespace ssd {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;

// B fragment (8 consecutive K of token t) for the permuted MMA layout.
template <int IN>
SSD_DI uint4 load_b(const LinearArgs& a, int t, int off, bool valid, const float* rstd) {
  if (!valid) return make_uint4(0u, 0u, 0u, 0u);
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

template <int IN, int NT>
SSD_DI void mainloop(const LinearArgs& a, const bf16* __restrict__ wg, const bf16* __restrict__ wg8,
                     int kb0, int kb1, int M, const float* rstd, float (&acc)[2][4], int lane) {
  const int g = lane >> 2, c = lane & 3;
  const bool v0 = g < M;
  const bool v1 = NT == 2 && (g + 8) < M;
  int kb = kb0;
  for (; kb + kUnroll <= kb1; kb += kUnroll) {
    uint4 wa[kUnroll], wb[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int off = (kb + u) * 32 + 8 * c;
      wa[u] = ld_stream_u4(wg + off);
      wb[u] = ld_stream_u4(wg8 + off);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int off = (kb + u) * 32 + 8 * c;
      const uint4 xa = load_b<IN>(a, g, off, v0, rstd);
      mma_bf16(acc[0], wa[u].x, wb[u].x, wa[u].y, wb[u].y, xa.x, xa.y);
      mma_bf16(acc[0], wa[u].z, wb[u].z, wa[u].w, wb[u].w, xa.z, xa.w);
      if (NT == 2) {
        const uint4 xb = load_b<IN>(a, g + 8, off, v1, rstd);
        mma_bf16(acc[1], wa[u].x, wb[u].x, wa[u].y, wb[u].y, xb.x, xb.y);
        mma_bf16(acc[1], wa[u].z, wb[u].z, wa[u].w, wb[u].w, xb.z, xb.w);
      }
    }
  }
  for (; kb < kb1; ++kb) {
    const int off = kb * 32 + 8 * c;
    const uint4 wa = ld_stream_u4(wg + off);
    const uint4 wb = ld_stream_u4(wg8 + off);
    const uint4 xa = load_b<IN>(a, g, off, v0, rstd);
    mma_bf16(acc[0], wa.x, wb.x, wa.y, wb.y, xa.x, xa.y);
    mma_bf16(acc[0], wa.z, wb.z, wa.w, wb.w, xa.z, xa.w);
    if (NT == 2) {
      const uint4 xb = load_b<IN>(a, g + 8, off, v1, rstd);
      mma_bf16(acc[1], wa.x, wb.x, wa.y, wb.y, xb.x, xb.y);
      mma_bf16(acc[1], wa.z, wb.z, wa.w, wb.w, xb.z, xb.w);
    }
  }
}

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

template <int IN, int EPI>
__global__ void __launch_bounds__(kThreads) gemv_kernel(LinearArgs a, int RG, int KS) {
  __shared__ float red[kWarps][16][16];  // [warp][row][token]
  __shared__ float outs[kWarps][16][16]; // [row group][row][token] after the K combine
  __shared__ float rstd_s[kMaxRows];
  __shared__ int last_s;

  pdl_wait();
  pdl_trigger();

  const int M = rows_of(a.M_static, a.M_dev);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (IN == IN_NORM) {
    // 1 / sqrt(mean(x^2) + eps) per row from the producer's partials, in a
    // fixed order: lane l sums partials l, l+32, ... then a butterfly.
    const int NP = a.K / kSsGroup;
    for (int m = warp; m < M; m += kWarps) {
      float s = 0.f;
      for (int p = lane; p < NP; p += 32) s += a.ss[(size_t)m * NP + p];
      s = sum_warp(s);
      if (lane == 0) rstd_s[m] = 1.0f / sqrtf(s / (float)a.K + a.eps);
    }
    __syncthreads();
  }

  const int rg = warp % RG, ks = warp / RG;
  const bf16* W;
  int row0;
  if (EPI == EPI_SWIGLU) {
    const int half = RG / 2;
    W = rg < half ? a.W0 : a.W1;
    row0 = (blockIdx.x * half + (rg % half)) * 16;
  } else {
    W = a.W0;
    row0 = (blockIdx.x * RG + rg) * 16;
  }
  const int KB = a.K / 32;
  const int kb0 = (int)((long long)ks * KB / KS);
  const int kb1 = (int)((long long)(ks + 1) * KB / KS);

  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  const bool rows_ok = row0 < a.R;
  if (rows_ok) {
    const bf16* wg = W + (size_t)(row0 + (lane >> 2)) * a.K;
    const bf16* wg8 = wg + (size_t)8 * a.K;
    if (M > 8)
      mainloop<IN, 2>(a, wg, wg8, kb0, kb1, M, rstd_s, acc, lane);
    else
      mainloop<IN, 1>(a, wg, wg8, kb0, kb1, M, rstd_s, acc, lane);
  }
  {
    const int g = lane >> 2, c = lane & 3;
    red[warp][g][2 * c] = acc[0][0];
    red[warp][g][2 * c + 1] = acc[0][1];
    red[warp][g + 8][2 * c] = acc[0][2];
    red[warp][g + 8][2 * c + 1] = acc[0][3];
    red[warp][g][8 + 2 * c] = acc[1][0];
    red[warp][g][8 + 2 * c + 1] = acc[1][1];
    red[warp][g + 8][8 + 2 * c] = acc[1][2];
    red[warp][g + 8][8 + 2 * c + 1] = acc[1][3];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < RG * 256; e += kThreads) {
    const int r = e >> 8, row = (e >> 4) & 15, tok = e & 15;
    float s = 0.f;
    for (int k = 0; k < KS; ++k) s += red[k * RG + r][row][tok];
    outs[r][row][tok] = s;
  }
  __syncthreads();

  // ---------------- epilogues ----------------
  if (EPI == EPI_STORE) {
    for (int e = threadIdx.x; e < RG * 16 * M; e += kThreads) {
      const int r = e / (16 * M), rem = e % (16 * M), row = rem / M, tok = rem % M;
      const int gr = (blockIdx.x * RG + r) * 16 + row;
      if (gr < a.R) a.y[(size_t)tok * a.R + gr] = outs[r][row][tok];
    }
  } else if (EPI == EPI_RESID) {
    for (int e = threadIdx.x; e < RG * 16 * M; e += kThreads) {
      const int r = e / (16 * M), rem = e % (16 * M), row = rem / M, tok = rem % M;
      const int gr = (blockIdx.x * RG + r) * 16 + row;
      if (gr < a.R) {
        const size_t idx = (size_t)tok * a.R + gr;
        const float xn = a.xres[idx] + outs[r][row][tok];
        a.xres[idx] = xn;
        outs[r][row][tok] = xn;
      }
    }
    __syncthreads();
    const int NP = a.R / kSsGroup;
    for (int e = threadIdx.x; e < RG * M; e += kThreads) {
      const int r = e / M, tok = e % M;
      const int grp = blockIdx.x * RG + r;
      if (grp * 16 < a.R) {
        float s = 0.f;
        for (int row = 0; row < 16; ++row) s += outs[r][row][tok] * outs[r][row][tok];
        a.ss_out[(size_t)tok * NP + grp] = s;
      }
    }
  } else if (EPI == EPI_SWIGLU) {
    const int half = RG / 2;
    for (int e = threadIdx.x; e < half * 16 * M; e += kThreads) {
      const int r = e / (16 * M), rem = e % (16 * M), row = rem / M, tok = rem % M;
      const int gr = (blockIdx.x * half + r) * 16 + row;
      if (gr < a.R) {
        const float gt = outs[r][row][tok];
        const float up = outs[r + half][row][tok];
        const float s = gt / (1.0f + expf(-gt));
        a.u[(size_t)tok * a.R + gr] = __float2bfloat16_rn(s * up);
      }
    }
  } else if (EPI == EPI_LMHEAD) {
    const int slot = a.slot_dev ? *a.slot_dev : 0;
    const int nr = RG * 16;
    const int v0 = blockIdx.x * nr;
    if (a.logits) {
      for (int e = threadIdx.x; e < nr * M; e += kThreads) {
        const int tok = e / nr, i = e % nr;
        if (v0 + i < a.R)
          a.logits[(size_t)(slot + tok) * a.R + v0 + i] = outs[i >> 4][i & 15][tok];
      }
    }
    const float T = a.temperature;
    const int round = a.round_dev ? *a.round_dev : a.round_static;
    const int pos0 = a.pos0_dev ? *a.pos0_dev : a.pos0_static;
    for (int tok = warp; tok < M; tok += kWarps) {
      float v1 = -INFINITY, v2 = -INFINITY, gv = -INFINITY;
      int i1 = 0x7fffffff, i2 = 0x7fffffff, gi = 0x7fffffff;
      for (int i = lane; i < nr; i += 32) {
        if (v0 + i >= a.R) continue;
        const float z = outs[i >> 4][i & 15][tok];
        top2_insert(z, v0 + i, v1, i1, v2, i2);
        if (T > 0.f) {
          const float sc = z / T + gumbel_at(a.seed, v0 + i, pos0 + tok + 1, round, a.sample_stream);
          if (better(sc, v0 + i, gv, gi)) { gv = sc; gi = v0 + i; }
        }
      }
      top2_warp(v1, i1, v2, i2);
      if (T > 0.f) argmax_warp(gv, gi);
      const float mx = v1;
      const float mxt = T > 0.f ? mx / T : mx;
      float se = 0.f, set = 0.f;
      for (int i = lane; i < nr; i += 32) {
        if (v0 + i >= a.R) continue;
        const float z = outs[i >> 4][i & 15][tok];
        se += expf(z - mx);
        if (T > 0.f) set += expf(z / T - mxt);
      }
      se = sum_warp(se);
      set = sum_warp(set);
      if (lane == 0) {
        float* p = a.part + ((size_t)blockIdx.x * kMaxRows + tok) * 8;
        p[0] = mx;
        p[1] = __int_as_float(i1);
        p[2] = v2;
        p[3] = __int_as_float(i2);
        p[4] = se;
        p[5] = set;
        p[6] = gv;
        p[7] = __int_as_float(gi);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned prev = atomicAdd(a.counter, 1u);
      last_s = prev == gridDim.x - 1;
    }
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    const int nC = gridDim.x;
    for (int tok = warp; tok < M; tok += kWarps) {
      float v1 = -INFINITY, v2 = -INFINITY, gv = -INFINITY;
      int i1 = 0x7fffffff, i2 = 0x7fffffff, gi = 0x7fffffff;
      for (int cta = lane; cta < nC; cta += 32) {
        const float* p = a.part + ((size_t)cta * kMaxRows + tok) * 8;
        top2_insert(__ldcg(p + 0), __float_as_int(__ldcg(p + 1)), v1, i1, v2, i2);
        top2_insert(__ldcg(p + 2), __float_as_int(__ldcg(p + 3)), v1, i1, v2, i2);
        const float cg = __ldcg(p + 6);
        const int ci = __float_as_int(__ldcg(p + 7));
        if (better(cg, ci, gv, gi)) { gv = cg; gi = ci; }
      }
      top2_warp(v1, i1, v2, i2);
      argmax_warp(gv, gi);
      const float mx = v1;
      const float mxt = T > 0.f ? mx / T : mx;
      float S = 0.f, St = 0.f;
      for (int cta = lane; cta < nC; cta += 32) {
        const float* p = a.part + ((size_t)cta * kMaxRows + tok) * 8;
        const float cm = __ldcg(p + 0);
        S += __ldcg(p + 4) * expf(cm - mx);
        if (T > 0.f) St += __ldcg(p + 5) * expf(cm / T - mxt);
      }
      S = sum_warp(S);
      St = sum_warp(St);
      if (lane == 0) {
        RowStats rs;
        rs.top1 = i1;
        rs.top2 = i2;
        rs.sample = T > 0.f ? gi : i1;
        rs.pad = 0;
        rs.z1 = mx;
        rs.z2 = v2;
        rs.lse = mx + logf(S);
        rs.conf = expf(mx - rs.lse);
        rs.lse_t = T > 0.f ? mxt + logf(St) : rs.lse;
        rs.pad2[0] = rs.pad2[1] = rs.pad2[2] = 0.f;
        a.stats[slot + tok] = rs;
      }
    }
    if (threadIdx.x == 0) *a.counter = 0u;
  }
}

template <int IN, int EPI>
cudaError_t launch_one(const LinearArgs& a, GemvCfg cfg, int grid, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = 0;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, gemv_kernel<IN, EPI>, a, cfg.RG, cfg.KS);
}

}  // namespace

GemvCfg gemv_pick(int row_groups, int K, int epi) {
  // Prefer more rows per CTA (fewer, larger CTAs) while keeping >= ~2 CTAs
  // per SM and >= 512 K elements per warp; SwiGLU needs an even RG.
  const int cands[3] = {4, 2, 1};
  for (int i = 0; i < 3; ++i) {
    const int RG = cands[i];
    if (epi == EPI_SWIGLU && RG < 2) continue;
    const int per = epi == EPI_SWIGLU ? RG / 2 : RG;
    if (row_groups % per) continue;
    const int ctas = row_groups / per;
    const int KS = kWarps / RG;
    if (ctas >= 300 && K / KS >= 512) return GemvCfg{RG, KS};
  }
  if (epi == EPI_SWIGLU) return GemvCfg{2, kWarps / 2};
  return GemvCfg{1, kWarps};
}

int gemv_grid(int row_groups, GemvCfg cfg, int epi) {
  const int per = epi == EPI_SWIGLU ? cfg.RG / 2 : cfg.RG;
  return (row_groups + per - 1) / per;
}

cudaError_t launch_gemv(int in_mode, int epi, const LinearArgs& a, GemvCfg cfg, cudaStream_t st,
                        bool pdl) {
  const int grid = gemv_grid(a.R / 16, cfg, epi);
#define SSD_GEMV_CASE(I, E) \
  if (in_mode == I && epi == E) return launch_one<I, E>(a, cfg, grid, st, pdl);
  SSD_GEMV_CASE(IN_BF16, EPI_STORE)
  SSD_GEMV_CASE(IN_NORM, EPI_STORE)
  SSD_GEMV_CASE(IN_BF16, EPI_RESID)
  SSD_GEMV_CASE(IN_NORM, EPI_SWIGLU)
  SSD_GEMV_CASE(IN_NORM, EPI_LMHEAD)
#undef SSD_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace ssd
