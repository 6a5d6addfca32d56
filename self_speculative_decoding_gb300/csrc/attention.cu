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
#include "attn_dev.cuh"

namespace ssd {

namespace {

__global__ void __launch_bounds__(attn::kGroupThreads, 4) attn_kernel(AttnArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int flag;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // The pass shape was written by kernels that completed before this one was
  // launched, and the cached rows before pos0 by earlier passes: the first
  // item's bulk copies go out before the wait on the preceding kernel (the
  // projection that produces q, k, v).
  const int M = a.M_dev ? __ldcg(a.M_dev) : a.M_static;
  const int pos0 = a.pos0_dev ? __ldcg(a.pos0_dev) : a.pos0_static;
  const int ns = a.ns_dev ? __ldcg(a.ns_dev) : 0;  // side rows (after the chain rows)
  {
    // debug builds: the pass's rows and positions lie inside the cache
    int* e = blockIdx.x == 0 && tid == 0 ? a.err : nullptr;
    bool ok = SSD_CHECK_W(e, a.err_val, M >= 1 && M <= kMaxRows && ns >= 0 && ns <= kMaxSide &&
                                            ns < M, DBG_ROWS, M);
    ok = ok && SSD_CHECK_W(e, a.err_val, pos0 >= 0 && pos0 + M - ns <= a.max_seq, DBG_POS,
                           pos0 + M - ns);
    for (int i = 0; ok && i < ns; ++i) {
      const int sp = __ldcg(a.side_pos + i);
      ok = SSD_CHECK_W(e, a.err_val, sp >= 0 && sp < pos0 + M - ns, DBG_POS, sp);
    }
    if (!ok) return;
  }
  const attn::Smem sm = attn::carve(smem_raw, a.dh, a.max_seq / kAttnChunk);
  const int n_items = ((pos0 + M - ns - 1) / kAttnChunk + 1) * a.Hkv;
  uint32_t phase = 0;
  if ((int)blockIdx.x < n_items) attn::issue(a, M - ns, pos0, blockIdx.x, sm, &bar, tid);
  pdl_wait();
  pdl_trigger();
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    if (it != (int)blockIdx.x) attn::issue(a, M - ns, pos0, it, sm, &bar, tid);
    attn::body(a, M, ns, pos0, it, sm, &bar, phase, &flag, tid, [] { __syncthreads(); });
  }
}

}  // namespace

size_t attn_smem(const AttnArgs& a) { return attn::smem_bytes(a.dh, a.max_seq / kAttnChunk); }

size_t attn_part_floats(int Hkv, int H, int dh, int max_seq) {
  return (size_t)Hkv * (max_seq / kAttnChunk) * (H / Hkv) * kMaxRows * (dh + attn::kRecPad);
}

static int sm_count() {
  static int cached[kDeviceSlots] = {0};
  const int dv = device_slot();
  if (dv >= 0 && cached[dv]) return cached[dv];
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (dv >= 0) cached[dv] = sms;
  return sms;
}

int attn_grid(const AttnArgs& a) {
  // Grid size only sets how many CTAs loop over the (head, chunk) items; it
  // does not change any reduction order.
  const int items = a.Hkv * (a.max_seq / kAttnChunk);
  const int cap = sm_count() * 4;  // resident CTAs per SM (launch bounds)
  return items < cap ? items : cap;
}

cudaError_t attn_prepare(const AttnArgs& a) {
  // raise the kernel's dynamic shared-memory limit to what this geometry needs
  static size_t set_to[kDeviceSlots] = {};
  const size_t smem = attn_smem(a);
  const int dv = device_slot();
  if (dv >= 0 && smem <= set_to[dv]) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess && dv >= 0) set_to[dv] = smem;
  return e;
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st, bool pdl) {
  const size_t smem = attn_smem(a);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(attn_grid(a));
  lc.blockDim = dim3(attn::kGroupThreads);
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
