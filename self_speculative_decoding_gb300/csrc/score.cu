// Batched candidate-mask scoring (SWIFT §4.1.2): K candidate layer sets each
// predict the last N committed tokens in one parallel forward.  Rows are laid
// out candidate-major: physical row p = k * N + i is candidate k's window
// position split + i.  A layer runs only the rows of the candidates that keep
// it; those rows are packed densely (compact row t, row map t -> p) so that
// the projections (gemm.cu) do no work for a skipped layer.
//
// This file holds everything of the scoring forward that is not a
// projection: the embedding of the window tokens, the RMSNorm of mapped rows
// into bf16 activations, RoPE with the window K/V write, the attention of the
// window queries (tensor cores, flash-style online softmax) and the match
// count of the argmax against the committed tokens.
#include "kernels.cuh"

namespace ssd {

namespace {

// x[p] = E[tokens[split + p % N]] (fp32) for p < rows.
__global__ void score_embed_kernel(const bf16* embed, const int32_t* tokens, int split, int N,
                                   int rows, int D, float* x) {
  const size_t n = (size_t)rows * D;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const int p = (int)(e / D), k = (int)(e % D);
    x[e] = __bfloat162float(embed[(size_t)tokens[split + p % N] * D + k]);
  }
}

// out[t] = bf16(rmsnorm(x[map[t]]) * gain), written in the packed unit
// layout the projections read.  One 256-thread block per row.  The row is
// read once, in 8-element chunks held in registers (thread i takes chunks i,
// i + 256, ...); each thread sums the squares of its chunks in that order,
// the block reduces the 256 partial sums in a fixed tree (butterfly within
// each warp, then warp 0 over the 8 warp sums), and every chunk is written
// as one 16-byte piece of the packed layout.
constexpr int kNormChunks = 4;  // chunks per thread: rows of up to 8192
__global__ void __launch_bounds__(256) score_norm_kernel(const float* x, const int32_t* map,
                                                         const float* gain, float eps, int T,
                                                         int D, bf16* out) {
  __shared__ float wsum[8];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* xr = x + (size_t)(map ? map[t] : t) * D;
  const int nc = D / 8;
  float4 va[kNormChunks][2];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kNormChunks; ++i) {
    const int ch = tid + i * 256;
    if (ch < nc) {
      va[i][0] = *reinterpret_cast<const float4*>(xr + 8 * ch);
      va[i][1] = *reinterpret_cast<const float4*>(xr + 8 * ch + 4);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        s += va[i][h].x * va[i][h].x;
        s += va[i][h].y * va[i][h].y;
        s += va[i][h].z * va[i][h].z;
        s += va[i][h].w * va[i][h].w;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) wsum[warp] = s;
  __syncthreads();
  if (warp == 0) {
    float w = lane < 8 ? wsum[lane] : 0.f;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    if (lane == 0) wsum[0] = w;
  }
  __syncthreads();
  const float rs = 1.0f / sqrtf(wsum[0] / (float)D + eps);
#pragma unroll
  for (int i = 0; i < kNormChunks; ++i) {
    const int ch = tid + i * 256;
    if (ch < nc) {
      const float4 g0 = *reinterpret_cast<const float4*>(gain + 8 * ch);
      const float4 g1 = *reinterpret_cast<const float4*>(gain + 8 * ch + 4);
      const float4 v0 = va[i][0], v1 = va[i][1];
      uint4 o;
      o.x = pack_bf16x2(v0.x * rs * g0.x, v0.y * rs * g0.y);
      o.y = pack_bf16x2(v0.z * rs * g0.z, v0.w * rs * g0.w);
      o.z = pack_bf16x2(v1.x * rs * g1.x, v1.y * rs * g1.y);
      o.w = pack_bf16x2(v1.z * rs * g1.z, v1.w * rs * g1.w);
      *reinterpret_cast<uint4*>(out + packed_off(t, 8 * ch, D)) = o;
    }
  }
}

// RoPE (rotate-half pairs (j, j + dh/2)) of the compact rows' q and k at
// position split + p % N (p = map[t], or t without a map); q -> q[t] bf16,
// k and v -> the window cache row p and, when kc is given, also the layer's
// cache [Hkv][max_seq][dh] at that position (the batched prefill).  A thread
// takes four consecutive pairs of one head (16-byte loads, 8-byte stores) or
// eight consecutive values of one v head.
__global__ void score_rope_kernel(const float* qkv, int T, const int32_t* map, int N, int split,
                                  int H, int Hkv, int dh, const float2* rope, bf16* q, bf16* sk,
                                  bf16* sv, bf16* kc, bf16* vc, int max_seq) {
  const int half = dh / 2;
  const int nrot = (H + Hkv) * (half / 4);            // rotation items per row
  const int per_row = nrot + Hkv * (dh / 8);           // + v items
  const int ld = (H + 2 * Hkv) * dh;
  const size_t n = (size_t)T * per_row;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(e / per_row);
    int r = (int)(e % per_row);
    const int p = map ? map[t] : t;
    const int pos = split + p % N;
    const float* row = qkv + (size_t)t * ld;
    if (r < nrot) {
      const int hh = r / (half / 4), j = 4 * (r % (half / 4));
      const float* v = row + (size_t)hh * dh;
      const float4 av = *reinterpret_cast<const float4*>(v + j);
      const float4 bv = *reinterpret_cast<const float4*>(v + j + half);
      const float4 c01 = *reinterpret_cast<const float4*>(rope + (size_t)pos * half + j);
      const float4 c23 = *reinterpret_cast<const float4*>(rope + (size_t)pos * half + j + 2);
      const float a[4] = {av.x, av.y, av.z, av.w}, b[4] = {bv.x, bv.y, bv.z, bv.w};
      const float cx[4] = {c01.x, c01.z, c23.x, c23.z}, cy[4] = {c01.y, c01.w, c23.y, c23.w};
      float ra[4], rb[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        ra[k] = a[k] * cx[k] - b[k] * cy[k];
        rb[k] = a[k] * cy[k] + b[k] * cx[k];
      }
      const uint2 lo = make_uint2(pack_bf16x2(ra[0], ra[1]), pack_bf16x2(ra[2], ra[3]));
      const uint2 hi = make_uint2(pack_bf16x2(rb[0], rb[1]), pack_bf16x2(rb[2], rb[3]));
      bf16* d = hh < H ? q + (size_t)t * H * dh + (size_t)hh * dh
                       : sk + ((size_t)p * Hkv + (hh - H)) * dh;
      *reinterpret_cast<uint2*>(d + j) = lo;
      *reinterpret_cast<uint2*>(d + j + half) = hi;
      if (hh >= H && kc) {
        bf16* e2 = kc + ((size_t)(hh - H) * max_seq + pos) * dh;
        *reinterpret_cast<uint2*>(e2 + j) = lo;
        *reinterpret_cast<uint2*>(e2 + j + half) = hi;
      }
    } else {
      r -= nrot;
      const int kvh = r / (dh / 8), j8 = 8 * (r % (dh / 8));
      const float* v = row + (size_t)(H + Hkv) * dh + (size_t)kvh * dh + j8;
      const float4 v0 = *reinterpret_cast<const float4*>(v);
      const float4 v1 = *reinterpret_cast<const float4*>(v + 4);
      const uint4 vv = make_uint4(pack_bf16x2(v0.x, v0.y), pack_bf16x2(v0.z, v0.w),
                                  pack_bf16x2(v1.x, v1.y), pack_bf16x2(v1.z, v1.w));
      *reinterpret_cast<uint4*>(sv + ((size_t)p * Hkv + kvh) * dh + j8) = vv;
      if (vc) *reinterpret_cast<uint4*>(vc + ((size_t)kvh * max_seq + pos) * dh + j8) = vv;
    }
  }
}

SSD_DI void cp_async16_z(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
SSD_DI void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
SSD_DI void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

SSD_DI void ldsm_x4_trans(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}

constexpr int kSaKeys = 64;  // keys per block

// Window-query attention.  CTA (row block, head h, active candidate ja):
// the row block's 16-row tiles each get two warps, which take the first and
// the second 32 keys of every 64-key block (more warps per SM for the same
// K/V buffers, half the dependent chain per warp).  Keys: the shared cache's
// positions [0, split) then the candidate's own window rows w <= i.  S = Q K^T
// and O += P V run on the tensor cores (bf16 operands, fp32 accumulation); the
// softmax is the online form in base 2 with the running max per row.  Each
// warp sums its key blocks in ascending key order; the two halves' states are
// merged at the end (first half + second half, in that order).
template <int DH>
__global__ void __launch_bounds__(256) score_attn_kernel(ScoreAttnArgs a) {
  extern __shared__ __align__(16) unsigned char sm_raw[];
  constexpr int KT = DH / 16;      // k16 steps of Q K^T
  constexpr int NT = DH / 8;       // n8 tiles of the output
  constexpr int RS = DH + 8;       // padded smem row (bf16)
  bf16* smK = reinterpret_cast<bf16*>(sm_raw);          // [2][64][RS]
  bf16* smV = smK + 2 * kSaKeys * RS;                   // [2][64][RS]
  const int nwr = blockDim.x >> 6;                     // row tiles of the CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rt = warp % nwr, kh = warp / nwr;          // row tile, key half
  const int g = lane >> 2, c = lane & 3;
  const int h = blockIdx.y, ja = blockIdx.z;
  const int kvh = h / (a.H / a.Hkv);
  const int cand = a.cand[ja];
  const int r0 = blockIdx.x * nwr * 16;                // first window row of the CTA
  const int i0 = r0 + rt * 16;                         // first row of the warp
  const int N = a.N;

  // Q fragments (rows beyond N are zero)
  uint32_t qf[KT][4];
  {
    const int ia = i0 + g, ib = i0 + g + 8;
    const bf16* qa = a.q + ((size_t)(ja * N + ia) * a.H + h) * DH;
    const bf16* qb = a.q + ((size_t)(ja * N + ib) * a.H + h) * DH;
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
      const int k0 = kt * 16 + 2 * c;
      qf[kt][0] = ia < N ? *reinterpret_cast<const uint32_t*>(qa + k0) : 0u;
      qf[kt][1] = ib < N ? *reinterpret_cast<const uint32_t*>(qb + k0) : 0u;
      qf[kt][2] = ia < N ? *reinterpret_cast<const uint32_t*>(qa + k0 + 8) : 0u;
      qf[kt][3] = ib < N ? *reinterpret_cast<const uint32_t*>(qb + k0 + 8) : 0u;
    }
  }
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  const int nb_pre = (a.split + kSaKeys - 1) / kSaKeys;
  const int wmax = min(N, r0 + nwr * 16);              // window keys the CTA needs
  const int nb = nb_pre + (wmax + kSaKeys - 1) / kSaKeys;
  const bf16* kc = a.kc + (size_t)kvh * a.max_seq * DH;
  const bf16* vc = a.vc + (size_t)kvh * a.max_seq * DH;

  auto load_block = [&](int b, int buf) {
    constexpr int PR = DH / 8;                         // 16-byte pieces per row
    for (int e = threadIdx.x; e < kSaKeys * PR; e += blockDim.x) {
      const int key = e / PR, q = e % PR;
      const bf16 *ks, *vs;
      bool ok;
      if (b < nb_pre) {
        const int pos = b * kSaKeys + key;
        ok = pos < a.split;
        ks = kc + (size_t)(ok ? pos : 0) * DH;
        vs = vc + (size_t)(ok ? pos : 0) * DH;
      } else {
        const int w = (b - nb_pre) * kSaKeys + key;
        ok = w < wmax;
        const size_t row = ((size_t)cand * N + (ok ? w : 0)) * a.Hkv + kvh;
        ks = a.sk + row * DH;
        vs = a.sv + row * DH;
      }
      cp_async16_z(smK + ((size_t)buf * kSaKeys + key) * RS + q * 8, ks + q * 8, ok);
      cp_async16_z(smV + ((size_t)buf * kSaKeys + key) * RS + q * 8, vs + q * 8, ok);
    }
  };

  load_block(0, 0);
  cp_commit();
  for (int b = 0; b < nb; ++b) {
    const int buf = b & 1;
    if (b + 1 < nb) load_block(b + 1, buf ^ 1);
    cp_commit();
    cp_wait1();
    __syncthreads();
    const bf16* Kb = smK + (size_t)buf * kSaKeys * RS;
    const bf16* Vb = smV + (size_t)buf * kSaKeys * RS;
    // S = Q K^T for this warp's 32 keys of the block
    float s[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      const bf16* kr = Kb + (size_t)(kh * 32 + nt * 8 + g) * RS + 2 * c;
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) {
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr + kt * 16);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + kt * 16 + 8);
        mma_bf16(s[nt], qf[kt][0], qf[kt][1], qf[kt][2], qf[kt][3], b0, b1);
      }
    }
    // mask, scale, online softmax
    const bool pre = b < nb_pre;
    const int kbase = (pre ? b * kSaKeys : (b - nb_pre) * kSaKeys) + kh * 32;
    float bm[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kbase + nt * 8 + 2 * c + (e & 1);
        const int i = i0 + g + 8 * (e >> 1);
        const bool valid = pre ? key < a.split : key <= i && key < N;
        const float v = valid ? s[nt][e] * a.scale_log2 : -INFINITY;
        s[nt][e] = v;
        bm[e >> 1] = fmaxf(bm[e >> 1], v);
      }
    float corr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      bm[r] = fmaxf(bm[r], __shfl_xor_sync(0xffffffffu, bm[r], 1));
      bm[r] = fmaxf(bm[r], __shfl_xor_sync(0xffffffffu, bm[r], 2));
      const float mn = fmaxf(mrow[r], bm[r]);
      corr[r] = mn == -INFINITY ? 1.f : exp2f(mrow[r] - mn);
      mrow[r] = mn;
    }
    float ls[2] = {0.f, 0.f};
    uint32_t pf[2][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float m = mrow[e >> 1];
        pv[e] = m == -INFINITY ? 0.f : exp2f(s[nt][e] - m);
        ls[e >> 1] += pv[e];
      }
      pf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(pv[0], pv[1]);
      pf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(pv[2], pv[3]);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) lrow[r] = lrow[r] * corr[r] + ls[r];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      o[j][0] *= corr[0];
      o[j][1] *= corr[0];
      o[j][2] *= corr[1];
      o[j][3] *= corr[1];
    }
    // O += P V: k16 step kk covers this warp's keys 16kk .. 16kk + 15
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      // A fragment order: (row g, keys 2c..), (row g+8, keys 2c..),
      // (row g, keys 2c+8..), (row g+8, keys 2c+8..)
      const uint32_t a0 = pf[kk][0], a1 = pf[kk][1], a2 = pf[kk][2], a3 = pf[kk][3];
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int j = 0; j < NT; j += 2) {
        uint32_t vb[4];
        ldsm_x4_trans(vb, Vb + (size_t)(kh * 32 + kk * 16 + (mi & 1) * 8 + rr) * RS + j * 8 +
                              (mi >> 1) * 8);
        mma_bf16(o[j], a0, a1, a2, a3, vb[0], vb[1]);
        mma_bf16(o[j + 1], a0, a1, a2, a3, vb[2], vb[3]);
      }
    }
    __syncthreads();
  }
  // row sums over the 4 lanes of a row
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
  }
  // the second key half hands its state to the first (the K/V buffers are
  // free: every warp passed the loop's last barrier)
  constexpr int XS = NT * 4 + 4;                       // floats per lane
  float* xch = reinterpret_cast<float*>(sm_raw) + (size_t)(rt * 32 + lane) * XS;
  if (kh == 1) {
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) xch[j * 4 + e] = o[j][e];
    xch[NT * 4 + 0] = mrow[0];
    xch[NT * 4 + 1] = mrow[1];
    xch[NT * 4 + 2] = lrow[0];
    xch[NT * 4 + 3] = lrow[1];
  }
  __syncthreads();
  if (kh == 1) return;
  float w0[2], w1[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float m1 = xch[NT * 4 + r];
    const float mn = fmaxf(mrow[r], m1);
    w0[r] = mrow[r] == -INFINITY ? 0.f : exp2f(mrow[r] - mn);
    w1[r] = m1 == -INFINITY ? 0.f : exp2f(m1 - mn);
    lrow[r] = lrow[r] * w0[r] + xch[NT * 4 + 2 + r] * w1[r];
  }
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    o[j][0] = o[j][0] * w0[0] + xch[j * 4 + 0] * w1[0];
    o[j][1] = o[j][1] * w0[0] + xch[j * 4 + 1] * w1[0];
    o[j][2] = o[j][2] * w0[1] + xch[j * 4 + 2] * w1[1];
    o[j][3] = o[j][3] * w0[1] + xch[j * 4 + 3] * w1[1];
  }
  // normalise, store
  const int ia = i0 + g, ib = i0 + g + 8;
  const float inva = 1.0f / lrow[0], invb = 1.0f / lrow[1];
  const int HD = a.H * DH;
  const int ta = ja * N + ia, tb = ja * N + ib;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int d = h * DH + j * 8 + 2 * c;
    const size_t offa = a.out_packed ? packed_off(ta, d, HD) : (size_t)ta * HD + d;
    const size_t offb = a.out_packed ? packed_off(tb, d, HD) : (size_t)tb * HD + d;
    if (ia < N) *reinterpret_cast<uint32_t*>(a.out + offa) = pack_bf16x2(o[j][0] * inva, o[j][1] * inva);
    if (ib < N) *reinterpret_cast<uint32_t*>(a.out + offb) = pack_bf16x2(o[j][2] * invb, o[j][3] * invb);
  }
}

// For compact row t of physical row p = map[t]: counts[p / N] += (argmax of
// row t == tokens[split + 1 + p % N]); best[t] is returned to zero.
__global__ void score_match_kernel(unsigned long long* best, const int32_t* map,
                                   const int32_t* tokens, int split, int N, int T,
                                   int32_t* counts) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int p = map ? map[t] : t;
  const unsigned long long key = best[t];
  const int idx = (int)(0xffffffffu - (uint32_t)(key & 0xffffffffull));
  if (key != 0ull && idx == tokens[split + 1 + p % N]) atomicAdd(counts + p / N, 1);
  best[t] = 0ull;
}

}  // namespace

cudaError_t launch_score_embed(const bf16* embed, const int32_t* tokens, int split, int N, int rows,
                               int D, float* x, cudaStream_t s) {
  score_embed_kernel<<<1216, 256, 0, s>>>(embed, tokens, split, N, rows, D, x);
  return cudaGetLastError();
}

cudaError_t launch_score_norm(const float* x, const int32_t* map, const float* gain, float eps,
                              int T, int D, bf16* out, cudaStream_t s) {
  if (D % 64 || D > 8 * 256 * kNormChunks) return cudaErrorInvalidValue;
  score_norm_kernel<<<T, 256, 0, s>>>(x, map, gain, eps, T, D, out);
  return cudaGetLastError();
}

cudaError_t launch_score_rope(const float* qkv, int T, const int32_t* map, int N, int split, int H,
                              int Hkv, int dh, const float2* rope, bf16* q, bf16* sk, bf16* sv,
                              bf16* kc, bf16* vc, int max_seq, cudaStream_t s) {
  if (dh % 8) return cudaErrorInvalidValue;
  score_rope_kernel<<<1216, 256, 0, s>>>(qkv, T, map, N, split, H, Hkv, dh, rope, q, sk, sv, kc, vc,
                                         max_seq);
  return cudaGetLastError();
}

size_t score_attn_smem(int dh) { return (size_t)4 * kSaKeys * (dh + 8) * sizeof(bf16); }

cudaError_t launch_score_attn(const ScoreAttnArgs& a, int n_active, cudaStream_t s) {
  if (n_active <= 0) return cudaSuccess;
  // The tensor-core form runs one CTA per 128 query rows and head through all
  // key blocks in turn (47-52 us at 2048 cached positions up to 12
  // candidates of 32 rows, 13B heads); the mma.sync form one CTA per
  // candidate and head, whose time grows with the candidates (48 us up to 3,
  // 60 us at 4-7, 84 us at 9, 120 us at 12).  The tensor-core form takes
  // passes of 128 rows or more.
#ifndef SSD_SCORE_ATTN_TC_MIN_ROWS
#define SSD_SCORE_ATTN_TC_MIN_ROWS 128
#endif
#ifndef SSD_SCORE_ATTN_MMA_SYNC
  if (score_attn_tc_ok(a) && n_active * a.N >= SSD_SCORE_ATTN_TC_MIN_ROWS)
    return launch_score_attn_tc(a, n_active, s);
#endif
  const int nw = a.N >= 64 ? 4 : (a.N + 15) / 16;     // row tiles per CTA
  dim3 grid((a.N + nw * 16 - 1) / (nw * 16), a.H, n_active);
  const size_t smem = score_attn_smem(a.dh);
  static bool ready128[kDeviceSlots] = {}, ready64[kDeviceSlots] = {};
  const int dv = device_slot();
  cudaError_t e = cudaSuccess;
  if (a.dh == 128) {
    if (dv < 0 || !ready128[dv])
      e = cudaFuncSetAttribute(score_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (e != cudaSuccess) return e;
    if (dv >= 0) ready128[dv] = true;
    score_attn_kernel<128><<<grid, nw * 64, smem, s>>>(a);
  } else if (a.dh == 64) {
    if (dv < 0 || !ready64[dv])
      e = cudaFuncSetAttribute(score_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (e != cudaSuccess) return e;
    if (dv >= 0) ready64[dv] = true;
    score_attn_kernel<64><<<grid, nw * 64, smem, s>>>(a);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_score_match(unsigned long long* best, const int32_t* map, const int32_t* tokens,
                               int split, int N, int T, int32_t* counts, cudaStream_t s) {
  score_match_kernel<<<(T + 255) / 256, 256, 0, s>>>(best, map, tokens, split, N, T, counts);
  return cudaGetLastError();
}

}  // namespace ssd
