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
constexpr int kKPad = 8;   // bf16 padding per cached key row in shared memory

// Shared-memory layout of one work item (all offsets multiples of 16 B):
//   K [64][dh + 8] bf16 | V [64][dh] bf16 | Q [G*16][dh] f32 | S [G*16][64] f32
//   | combine scratch: m [nchunk], l [nchunk], w [nchunk] f32
struct Smem {
  bf16* K;
  bf16* V;
  float* Q;
  float* S;
  float* cm;
  float* cl;
  float* cw;
};

SSD_DI Smem carve(unsigned char* raw, int dh, int rows, int nchunk) {
  Smem sm;
  sm.K = reinterpret_cast<bf16*>(raw);
  sm.V = sm.K + kAttnChunk * (dh + kKPad);
  sm.Q = reinterpret_cast<float*>(sm.V + kAttnChunk * dh);
  sm.S = sm.Q + rows * dh;
  sm.cm = sm.S + rows * kAttnChunk;
  sm.cl = sm.cm + nchunk;
  sm.cw = sm.cl + nchunk;
  return sm;
}

__global__ void __launch_bounds__(kThreads) attn_kernel(AttnArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int last_s;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  pdl_wait();
  pdl_trigger();

  const int M = rows_of(a.M_static, a.M_dev);
  const int pos0 = a.pos0_dev ? *a.pos0_dev : a.pos0_static;
  const int dh = a.dh, half = dh / 2, krs = dh + kKPad;
  const int G = a.H / a.Hkv;
  const int rows = G * kMaxRows;
  const int nchunk_max = a.max_seq / kAttnChunk;
  const Smem sm = carve(smem_raw, dh, rows, nchunk_max);

  const int last_pos = pos0 + M - 1;
  const int n_active = last_pos / kAttnChunk + 1;
  const int n_items = n_active * a.Hkv;
  const int warp = tid >> 5, lane = tid & 31;
  const size_t head_stride = (size_t)a.max_seq * dh;
  const int ld_out = a.H * dh;
  const int R = G * M;  // active query rows of a head group
  uint32_t phase = 0;
  __syncthreads();

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int c = item / a.Hkv, kvh = item % a.Hkv;
    const int p_begin = c * kAttnChunk;
    const int p_end = min(p_begin + kAttnChunk, last_pos + 1);
    const int nk = p_end - p_begin;
    const int n_old = max(0, min(p_end, pos0) - p_begin);
    bf16* kc = a.kc + kvh * head_stride;
    bf16* vc = a.vc + kvh * head_stride;
    bf16* kc2 = a.kc2 ? a.kc2 + (size_t)kvh * a.scratch_len * dh : nullptr;
    bf16* vc2 = a.vc2 ? a.vc2 + (size_t)kvh * a.scratch_len * dh : nullptr;
    // row of position pos in the shared cache or in the scratch cache
    auto krow = [&](int pos) { return pos < a.split ? kc + (size_t)pos * dh : kc2 + (size_t)(pos - a.split) * dh; };
    auto vrow = [&](int pos) { return pos < a.split ? vc + (size_t)pos * dh : vc2 + (size_t)(pos - a.split) * dh; };

    // (1) cached keys/values of the chunk: bulk copies issued by warp 0 (one
    // per padded K row; V rows in one copy unless the chunk straddles the
    // scratch split)
    if (n_old > 0 && warp == 0) {
      const bool one_v = p_begin + n_old <= a.split || p_begin >= a.split;
      if (lane == 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bar, (uint32_t)(2 * n_old * dh * sizeof(bf16)));
        if (one_v)
          bulk_g2s(sm.V, vrow(p_begin), (uint32_t)(n_old * dh * sizeof(bf16)), &bar);
      }
      __syncwarp();
      for (int j = lane; j < n_old; j += 32) {
        bulk_g2s(sm.K + (size_t)j * krs, krow(p_begin + j), (uint32_t)(dh * sizeof(bf16)), &bar);
        if (!one_v)
          bulk_g2s(sm.V + (size_t)j * dh, vrow(p_begin + j), (uint32_t)(dh * sizeof(bf16)), &bar);
      }
    }
    // (2) new keys of this chunk: RoPE, bf16, append to the cache
    const int first_new = max(p_begin, pos0);
    for (int e = tid; e < (p_end - first_new) * half; e += kThreads) {
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
      sm.K[j * krs + i] = kb0;
      sm.K[j * krs + i + half] = kb1;
      sm.V[j * dh + i] = vb0;
      sm.V[j * dh + i + half] = vb1;
      bf16* kd = krow(pos);
      bf16* vd = vrow(pos);
      kd[i] = kb0;
      kd[i + half] = kb1;
      vd[i] = vb0;
      vd[i + half] = vb1;
    }
    // (3) queries of the group, RoPE'd, fp32; row r = gh * 16 + m
    for (int e = tid; e < R * half; e += kThreads) {
      const int i = e % half, rest = e / half, m = rest % M, gh = rest / M;
      const float* qr = a.qkv + (size_t)m * a.ld_qkv + (size_t)(kvh * G + gh) * dh;
      const float2 cs = a.rope[(size_t)(pos0 + m) * half + i];
      const float q0 = qr[i], q1 = qr[i + half];
      float* qd = sm.Q + (size_t)(gh * kMaxRows + m) * dh;
      qd[i] = q0 * cs.x - q1 * cs.y;
      qd[i + half] = q0 * cs.y + q1 * cs.x;
    }
    if (n_old > 0) {
      if (!mbar_wait(&bar, phase & 1u)) {
        if (tid == 0) atomicExch(a.err, 1);
        return;
      }
      ++phase;
    }
    __syncthreads();

    // (4) scores: 4 lanes per (row, key), each lane a quarter of the head
    // dimension in 8-wide pieces; then a 2-step butterfly (fixed order)
    const int qd = dh / 4;
    for (int u = tid; u < R * kAttnChunk * 4; u += kThreads) {
      const int qt = u & 3, key = (u >> 2) & (kAttnChunk - 1), rr = u >> 8;
      const int m = rr % M, gh = rr / M, r = gh * kMaxRows + m;
      const bool valid = key < nk && p_begin + key <= pos0 + m;
      float acc = 0.f;
      if (valid) {
        const float* q = sm.Q + (size_t)r * dh;
        const bf16* k = sm.K + (size_t)key * krs;
        for (int t = 0; t < qd; t += 8) {
          const int d0 = t * 4 + qt * 8;   // 8 consecutive dims per piece
          const uint4 kk = *reinterpret_cast<const uint4*>(k + d0);
          const float4 qa = *reinterpret_cast<const float4*>(q + d0);
          const float4 qb = *reinterpret_cast<const float4*>(q + d0 + 4);
          acc = fmaf(qa.x, bf16_lo(kk.x), acc);
          acc = fmaf(qa.y, bf16_hi(kk.x), acc);
          acc = fmaf(qa.z, bf16_lo(kk.y), acc);
          acc = fmaf(qa.w, bf16_hi(kk.y), acc);
          acc = fmaf(qb.x, bf16_lo(kk.z), acc);
          acc = fmaf(qb.y, bf16_hi(kk.z), acc);
          acc = fmaf(qb.z, bf16_lo(kk.w), acc);
          acc = fmaf(qb.w, bf16_hi(kk.w), acc);
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (qt == 0) sm.S[(size_t)r * kAttnChunk + key] = valid ? acc * a.scale : -INFINITY;
    }
    __syncthreads();

    // (5) per-row chunk softmax statistics; one warp per row
    float* part_base = a.part + ((size_t)kvh * nchunk_max + c) * rows * (dh + 2);
    for (int rr = warp; rr < R; rr += kWarps) {
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
    for (int e = tid; e < R * dh; e += kThreads) {
      const int dd = e % dh, rest = e / dh, m = rest % M, gh = rest / M;
      const int r = gh * kMaxRows + m;
      const float* p = sm.S + (size_t)r * kAttnChunk;
      float o = 0.f;
      for (int j = 0; j < nk; ++j) o = fmaf(p[j], __bfloat162float(sm.V[j * dh + dd]), o);
      part_base[(size_t)r * (dh + 2) + 2 + dd] = o;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const unsigned prev = atomicAdd(a.counters + kvh, 1u);
      last_s = prev == (unsigned)(n_active - 1);
    }
    __syncthreads();
    if (last_s) {
      __threadfence();
      // (7) combine this head's chunks in chunk order, one row at a time:
      // stage (m_c, l_c), weights w_c = exp(m_c - max), then each output
      // dimension sums o_c * w_c over chunks.
      const float* hb = a.part + (size_t)kvh * nchunk_max * rows * (dh + 2);
      for (int rr = 0; rr < R; ++rr) {
        const int m = rr % M, gh = rr / M, r = gh * kMaxRows + m;
        const int nc = (pos0 + m) / kAttnChunk + 1;
        for (int cc = tid; cc < nc; cc += kThreads) {
          const float* pc = hb + ((size_t)cc * rows + r) * (dh + 2);
          sm.cm[cc] = __ldcg(pc);
          sm.cl[cc] = __ldcg(pc + 1);
        }
        __syncthreads();
        float mx = -INFINITY;
        for (int cc = 0; cc < nc; ++cc) mx = fmaxf(mx, sm.cm[cc]);
        for (int cc = tid; cc < nc; cc += kThreads) sm.cw[cc] = expf(sm.cm[cc] - mx);
        __syncthreads();
        float L = 0.f;
        for (int cc = 0; cc < nc; ++cc) L = fmaf(sm.cl[cc], sm.cw[cc], L);
        for (int dd = tid; dd < dh; dd += kThreads) {
          float O = 0.f;
          int cc = 0;
          for (; cc + 4 <= nc; cc += 4) {
            const float o0 = __ldcg(hb + ((size_t)(cc + 0) * rows + r) * (dh + 2) + 2 + dd);
            const float o1 = __ldcg(hb + ((size_t)(cc + 1) * rows + r) * (dh + 2) + 2 + dd);
            const float o2 = __ldcg(hb + ((size_t)(cc + 2) * rows + r) * (dh + 2) + 2 + dd);
            const float o3 = __ldcg(hb + ((size_t)(cc + 3) * rows + r) * (dh + 2) + 2 + dd);
            O = fmaf(o0, sm.cw[cc + 0], O);
            O = fmaf(o1, sm.cw[cc + 1], O);
            O = fmaf(o2, sm.cw[cc + 2], O);
            O = fmaf(o3, sm.cw[cc + 3], O);
          }
          for (; cc < nc; ++cc)
            O = fmaf(__ldcg(hb + ((size_t)cc * rows + r) * (dh + 2) + 2 + dd), sm.cw[cc], O);
          a.out[(size_t)m * ld_out + (size_t)(kvh * G + gh) * dh + dd] = __float2bfloat16_rn(O / L);
        }
        __syncthreads();
      }
      if (tid == 0) a.counters[kvh] = 0u;
    }
    // the next item's bulk copies overwrite this item's shared memory
    fence_proxy_async_smem();
    __syncthreads();
  }
}

}  // namespace

size_t attn_smem(const AttnArgs& a) {
  const int G = a.H / a.Hkv;
  return (size_t)kAttnChunk * (a.dh + kKPad) * sizeof(bf16) +
         (size_t)kAttnChunk * a.dh * sizeof(bf16) + (size_t)G * kMaxRows * a.dh * 4 +
         (size_t)G * kMaxRows * kAttnChunk * 4 + (size_t)3 * (a.max_seq / kAttnChunk) * 4;
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
  // raise the kernel's dynamic shared-memory limit to what this geometry needs
  static size_t set_to = 0;
  const size_t smem = attn_smem(a);
  if (smem <= set_to) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) set_to = smem;
  return e;
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
