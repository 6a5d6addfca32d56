// Decode / verify attention over the KV cache (sm_103a).
//
// A pass carries M <= 16 query rows at consecutive positions pos0..pos0+M-1
// (M = 1 for a draft or autoregressive step, d+1 for the verify pass).  The
// kernel
//   1. applies rotate-half RoPE to the new keys, rounds k and v to bf16 and
//      appends them to the cache at their positions (LayerSkip blog §3.2:
//      the verify pass writes the K/V of every layer it runs);
//   2. splits the keys 0..pos0+M-1 into fixed absolute chunks of 64
//      positions; one work item = (KV head, chunk) computes, for every query
//      head of the group and every row, the chunk's max score, sum of
//      exponentials and unnormalised output (flash-decoding partials);
//   3. the CTA that completes a head's last chunk combines that head's
//      partials in chunk order and writes bf16 outputs.
//
// Causality is per row: row m sees keys <= pos0+m; masked keys contribute
// exact zeros, and a row's partials depend only on its own position, so a
// row computed in a pass of M rows is bit-identical to the same row alone.
#include "kernels.cuh"

namespace ssd {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct Smem {
  bf16* K;     // [64][dh]
  bf16* V;     // [64][dh]
  float* Q;    // [G*16][dh]
  float* S;    // [G*16][64]
};

__global__ void __launch_bounds__(kThreads) attn_kernel(AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int last_s;
  pdl_wait();
  pdl_trigger();

  const int M = rows_of(a.M_static, a.M_dev);
  const int pos0 = a.pos0_dev ? *a.pos0_dev : a.pos0_static;
  const int dh = a.dh, half = dh / 2;
  const int G = a.H / a.Hkv;
  const int rows = G * kMaxRows;
  Smem sm;
  sm.K = reinterpret_cast<bf16*>(smem_raw);
  sm.V = sm.K + kAttnChunk * dh;
  sm.Q = reinterpret_cast<float*>(sm.V + kAttnChunk * dh);
  sm.S = sm.Q + rows * dh;

  const int last_pos = pos0 + M - 1;
  const int n_active = last_pos / kAttnChunk + 1;
  const int n_items = n_active * a.Hkv;
  const int nchunk_max = a.max_seq / kAttnChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t head_stride = (size_t)a.max_seq * dh;
  const int ld_out = a.H * dh;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int c = item / a.Hkv, kvh = item % a.Hkv;
    const int p_begin = c * kAttnChunk;
    const int p_end = min(p_begin + kAttnChunk, last_pos + 1);
    const int nk = p_end - p_begin;
    bf16* kc = a.kc + kvh * head_stride;
    bf16* vc = a.vc + kvh * head_stride;

    // (1) cached keys of this chunk: positions [p_begin, min(p_end, pos0))
    const int n_old = max(0, min(p_end, pos0) - p_begin);
    const int vec_per_row = dh / 8;  // 16-byte pieces
    for (int e = threadIdx.x; e < n_old * vec_per_row; e += kThreads) {
      const int j = e / vec_per_row, q = e % vec_per_row;
      reinterpret_cast<uint4*>(sm.K + j * dh)[q] =
          reinterpret_cast<const uint4*>(kc + (size_t)(p_begin + j) * dh)[q];
      reinterpret_cast<uint4*>(sm.V + j * dh)[q] =
          reinterpret_cast<const uint4*>(vc + (size_t)(p_begin + j) * dh)[q];
    }
    // (2) new keys of this chunk: RoPE, bf16, append to the cache
    const int first_new = max(p_begin, pos0);
    for (int e = threadIdx.x; e < (p_end - first_new) * half; e += kThreads) {
      const int jj = e / half, i = e % half;
      const int pos = first_new + jj, m = pos - pos0, j = pos - p_begin;
      const float* kr = a.qkv + (size_t)m * a.ld_qkv + (size_t)(a.H + kvh) * dh;
      const float* vr = kr + (size_t)a.Hkv * dh;
      const float2 cs = a.rope[(size_t)pos * half + i];
      const float k0 = kr[i], k1 = kr[i + half];
      const bf16 kb0 = __float2bfloat16_rn(k0 * cs.x - k1 * cs.y);
      const bf16 kb1 = __float2bfloat16_rn(k0 * cs.y + k1 * cs.x);
      const bf16 vb0 = __float2bfloat16_rn(vr[i]);
      const bf16 vb1 = __float2bfloat16_rn(vr[i + half]);
      sm.K[j * dh + i] = kb0;
      sm.K[j * dh + i + half] = kb1;
      sm.V[j * dh + i] = vb0;
      sm.V[j * dh + i + half] = vb1;
      kc[(size_t)pos * dh + i] = kb0;
      kc[(size_t)pos * dh + i + half] = kb1;
      vc[(size_t)pos * dh + i] = vb0;
      vc[(size_t)pos * dh + i + half] = vb1;
    }
    // (3) queries of the group, RoPE'd, fp32; row r = gh * 16 + m
    for (int e = threadIdx.x; e < G * M * half; e += kThreads) {
      const int i = e % half, rest = e / half, m = rest % M, gh = rest / M;
      const float* qr = a.qkv + (size_t)m * a.ld_qkv + (size_t)(kvh * G + gh) * dh;
      const float2 cs = a.rope[(size_t)(pos0 + m) * half + i];
      const float q0 = qr[i], q1 = qr[i + half];
      float* qd = sm.Q + (size_t)(gh * kMaxRows + m) * dh;
      qd[i] = q0 * cs.x - q1 * cs.y;
      qd[i + half] = q0 * cs.y + q1 * cs.x;
    }
    __syncthreads();

    // (4) scores: one warp per (row, key); lanes split the head dimension
    const int dpl = dh / 32;
    for (int u = warp; u < G * M * kAttnChunk; u += kWarps) {
      const int j = u % kAttnChunk, rest = u / kAttnChunk, m = rest % M, gh = rest / M;
      const int r = gh * kMaxRows + m;
      float s = -INFINITY;
      if (j < nk && p_begin + j <= pos0 + m) {
        const float* q = sm.Q + (size_t)r * dh + lane * dpl;
        const bf16* k = sm.K + (size_t)j * dh + lane * dpl;
        float acc = 0.f;
        for (int t = 0; t < dpl; t += 2) {
          const uint32_t kk = *reinterpret_cast<const uint32_t*>(k + t);
          acc = fmaf(q[t], bf16_lo(kk), acc);
          acc = fmaf(q[t + 1], bf16_hi(kk), acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        s = acc * a.scale;
      }
      if (lane == 0) sm.S[(size_t)r * kAttnChunk + j] = s;
    }
    __syncthreads();

    // (5) per-row chunk softmax statistics; one warp per row
    float* part_base = a.part + ((size_t)kvh * nchunk_max + c) * rows * (dh + 2);
    for (int rr = warp; rr < G * M; rr += kWarps) {
      const int m = rr % M, gh = rr / M, r = gh * kMaxRows + m;
      float* srow = sm.S + (size_t)r * kAttnChunk;
      const float s0 = srow[lane], s1 = srow[lane + 32];
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float p0 = s0 == -INFINITY ? 0.f : expf(s0 - mx);
      const float p1 = s1 == -INFINITY ? 0.f : expf(s1 - mx);
      float l = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      __syncwarp();
      srow[lane] = p0;
      srow[lane + 32] = p1;
      if (lane == 0) {
        part_base[(size_t)r * (dh + 2) + 0] = mx;
        part_base[(size_t)r * (dh + 2) + 1] = l;
      }
    }
    __syncthreads();
    // (6) unnormalised output of the chunk: sequential over keys
    for (int e = threadIdx.x; e < G * M * dh; e += kThreads) {
      const int dd = e % dh, rest = e / dh, m = rest % M, gh = rest / M;
      const int r = gh * kMaxRows + m;
      const float* p = sm.S + (size_t)r * kAttnChunk;
      float o = 0.f;
      for (int j = 0; j < nk; ++j) o = fmaf(p[j], __bfloat162float(sm.V[j * dh + dd]), o);
      part_base[(size_t)r * (dh + 2) + 2 + dd] = o;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned prev = atomicAdd(a.counters + kvh, 1u);
      last_s = prev == (unsigned)(n_active - 1);
    }
    __syncthreads();
    if (last_s) {
      __threadfence();
      // (7) combine this head's chunks in chunk order
      const float* hb = a.part + (size_t)kvh * nchunk_max * rows * (dh + 2);
      for (int e = threadIdx.x; e < G * M * dh; e += kThreads) {
        const int dd = e % dh, rest = e / dh, m = rest % M, gh = rest / M;
        const int r = gh * kMaxRows + m;
        const int lastc = (pos0 + m) / kAttnChunk;
        float mx = -INFINITY;
        for (int cc = 0; cc <= lastc; ++cc)
          mx = fmaxf(mx, __ldcg(hb + ((size_t)cc * rows + r) * (dh + 2)));
        float L = 0.f, O = 0.f;
        for (int cc = 0; cc <= lastc; ++cc) {
          const float* pc = hb + ((size_t)cc * rows + r) * (dh + 2);
          const float w = expf(__ldcg(pc) - mx);
          L = fmaf(__ldcg(pc + 1), w, L);
          O = fmaf(__ldcg(pc + 2 + dd), w, O);
        }
        a.out[(size_t)m * ld_out + (size_t)(kvh * G + gh) * dh + dd] = __float2bfloat16_rn(O / L);
      }
      if (threadIdx.x == 0) a.counters[kvh] = 0u;
    }
    __syncthreads();
  }
}

}  // namespace

size_t attn_smem(const AttnArgs& a) {
  const int G = a.H / a.Hkv;
  return (size_t)2 * kAttnChunk * a.dh * sizeof(bf16) + (size_t)G * kMaxRows * a.dh * 4 +
         (size_t)G * kMaxRows * kAttnChunk * 4;
}

size_t attn_part_floats(int Hkv, int H, int dh, int max_seq) {
  return (size_t)Hkv * (max_seq / kAttnChunk) * (H / Hkv) * kMaxRows * (dh + 2);
}

static int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = sms;
  }
  return cached[dev];
}

int attn_grid(const AttnArgs& a) {
  // Grid size only sets how many CTAs loop over the (head, chunk) items; it
  // does not change any reduction order.
  const int items = a.Hkv * (a.max_seq / kAttnChunk);
  const int cap = sm_count() * 4;
  return items < cap ? items : cap;
}

cudaError_t attn_prepare(const AttnArgs& a) {
  // the largest geometry this build supports: group of 8, dh 128
  AttnArgs big = a;
  big.H = 8;
  big.Hkv = 1;
  big.dh = 128;
  const size_t smem = attn_smem(big) > attn_smem(a) ? attn_smem(big) : attn_smem(a);
  return cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st, bool pdl) {
  const size_t smem = attn_smem(a);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(attn_grid(a));
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, attn_kernel, a);
}

}  // namespace ssd
