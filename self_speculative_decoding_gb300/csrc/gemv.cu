// Small-M weight-streaming GEMV on the tensor cores (sm_103a).
//
// y[m][r] = sum_k W[r][k] act[m][k] for M <= 16 rows (token positions).  At
// batch 1 every decoder projection is a matrix-vector product whose cost is
// reading W once from HBM; the same kernel serves the M = d+1 verify pass
// and the 16-row prefill chunks.
//
// Weight layout.  W is stored in "units" of 16 rows x 32 columns (1 KB),
// row-group-major, each unit in tensor-core fragment order (see
// ssd_pack_weight): the matrix is one contiguous stream and a unit is exactly
// the A operand of two m16n8k16 MMAs for one warp.
//
// Data movement.  Each CTA owns a contiguous range of units: whole row
// groups (whole gate/up pairs) in equal numbers where the matrix has enough
// of them, else an equal share of single units (at most kGridCtas CTAs, two
// per SM, one wave).  A producer warp streams the range into a ring of
// shared-memory slots with bulk (TMA) copies of up to 16 units, completing on
// mbarriers; eight consumer warps take two units each per slot (warp w units
// w and w + 8), read their fragments with conflict-free 16-byte shared loads
// and run the MMAs.  The ring has 3 slots of 16 KB, plus, when a launch's
// rows leave part of the activation stage unused (one-row passes), the whole
// 16 KB slots that fit there.  Activations (the B operand: 8 or 16 token
// columns) are staged once per CTA in shared memory (normalised with the
// RMSNorm statistics for the norm-fused input); wide passes whose CTAs own
// whole row groups copy them window by window (K-outer batches), other wide
// passes read them from global memory a chunk ahead.
//
// Reduction order.  A row group's sum is the sum, in CTA order, of its CTAs'
// partials; a partial is the sum, in warp order, of the consumer warps'
// accumulators; each warp accumulates its units in ascending K order.  The
// partition depends only on the matrix shape and nothing depends on M, so a
// column's bits do not change with the number of rows processed together —
// which is what makes self-speculative verification reproduce
// autoregressive decoding bit for bit.
#include "gemv_dev.cuh"

namespace ssd {

using namespace gemv;

namespace {

template <int IN, int EPI>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) gemv_kernel(LinearArgs a, Part p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  GemvSmem& sm = *reinterpret_cast<GemvSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots + kStageBytes / kSlotBytes; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumers);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.rfull[s], kConsumers);
      mbar_init(&sm.rempty[s], 1);
    }
    mbar_init(&sm.foldbar, 1);
    mbar_init(&sm.lastbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  RingPos rp;
  rp.nslots = ring_slots(a, kouter_order<IN, EPI>(a, p));
  if (warp == kProducer) {
    // weights do not depend on the preceding kernel: no wait before streaming
    producer_phase<IN, EPI>(a, p, sm, b, lane, rp);
    return;
  }
  pdl_wait();
  pdl_trigger();
  int M = rows_of(a.M_static, a.M_dev);
  if (!SSD_CHECK_W(b == 0 && warp == 0 && lane == 0 ? a.err : nullptr, a.err_val,
                   M >= 1 && M <= kMaxRows, DBG_ROWS, M))
    M = M < 1 ? 1 : kMaxRows;
  // the staged rows must stay clear of the ring slots borrowed from the stage
  if (rp.nslots > kSlots) {
    const int room = (kStageBytes - (rp.nslots - kSlots) * kSlotBytes) / ((a.K + kPad) * (int)sizeof(bf16));
    if (M > room) {
      if (b == 0 && warp == 0 && lane == 0) atomicExch(a.err, 10);
      M = room;
    }
  }
  if (warp == kEpilogue) {
    LmRec run = lm_empty();
    epilogue_phase<IN, EPI>(a, p, sm, b, M, lane, rp, run);
    if (EPI == EPI_LMHEAD) lm_end(a, p, sm, b, M, warp, lane, rp, run, true);
    return;
  }
  consumer_phase<IN, EPI>(a, p, sm, b, M, warp, lane, rp);
  if (EPI == EPI_LMHEAD) lm_end(a, p, sm, b, M, warp, lane, rp, lm_empty(), false);
}

template <int IN, int EPI>
cudaError_t launch_one(const LinearArgs& a, const Part& p, cudaStream_t st, bool pdl) {
  static bool attr_set[kDeviceSlots] = {};
  const int smem = (int)sizeof(GemvSmem) + 128;
  const int dv = device_slot();
  if (dv < 0 || !attr_set[dv]) {
    const cudaError_t e = cudaFuncSetAttribute(
        gemv_kernel<IN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dv >= 0) attr_set[dv] = true;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(p.C);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, gemv_kernel<IN, EPI>, a, p);
}

// Packs W [R][K] row-major into units of 16 rows x 32 columns: unit
// (vr, kb) = 512 bf16; half h holds rows vr*16 + 8h .. + 7, row g at
// [h*256 + 32g], its 16-byte chunk c (columns kb*32 + 8c .. + 7) at
// position c ^ ((g >> 1) & 3) of the row (the 64-byte swizzle).
__global__ void pack_kernel(const bf16* __restrict__ src, bf16* __restrict__ dst, int R, int K) {
  const long long n = (long long)R * K / 8;  // 16-byte pieces
  const int KB = K / 32;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long unit = i / 64;
    const int within = (int)(i % 64);
    const int h = within / 32, L = within % 32;
    const int gg = L >> 2, cc = (L & 3) ^ ((gg >> 1) & 3);
    const long long vr = unit / KB;
    const int kb = (int)(unit % KB);
    const long long row = vr * 16 + 8 * h + gg;
    reinterpret_cast<uint4*>(dst)[i] =
        *reinterpret_cast<const uint4*>(src + row * K + (long long)kb * 32 + 8 * cc);
  }
}

// RMSNorm of the pass's rows into bf16: out[m][k] = bf16(x[m][k] * r_m * g[k])
// with r_m = 1 / sqrt(mean(x_m^2) + eps) from the sum-of-squares partials.
// Every warp of a block computes r_m itself, in the consumer warps' order
// (lane l sums partials l, l+32, ..., then a butterfly), and the products are
// rounded as the staged layout rounds them, so a projection fed from this
// buffer computes the bits the norm-fused input computes.
__global__ void __launch_bounds__(256) norm_rows_kernel(const float* x, const float* ss,
                                                        const float* gain, float eps, int M_static,
                                                        const int32_t* M_dev, int K, bf16* out) {
  pdl_wait();
  pdl_trigger();
  const int M = M_dev ? __ldcg(M_dev) : M_static;
  const int m = blockIdx.x;
  if (m >= M) return;
  const int lane = threadIdx.x & 31;
  const int NP = K / kSsGroup;
  float s2 = 0.f;
#pragma unroll 8
  for (int q = lane; q < NP; q += 32) s2 += __ldcg(ss + (size_t)m * NP + q);
  s2 = sum_warp(s2);
  const float rs = 1.0f / sqrtf(s2 / (float)K + eps);
  const int k0 = (blockIdx.y * 256 + threadIdx.x) * 8;
  if (k0 >= K) return;
  const float4* xp = reinterpret_cast<const float4*>(x + (size_t)m * K + k0);
  const float4* gp = reinterpret_cast<const float4*>(gain + k0);
  const float4 x0 = __ldcg(xp), x1 = __ldcg(xp + 1), g0 = gp[0], g1 = gp[1];
  *reinterpret_cast<uint4*>(out + (size_t)m * K + k0) =
      make_uint4(pack_bf16x2(x0.x * rs * g0.x, x0.y * rs * g0.y),
                 pack_bf16x2(x0.z * rs * g0.z, x0.w * rs * g0.w),
                 pack_bf16x2(x1.x * rs * g1.x, x1.y * rs * g1.y),
                 pack_bf16x2(x1.z * rs * g1.z, x1.w * rs * g1.w));
}

}  // namespace

int gemv_stage_rows(int K) { return kStageBytes / ((K + kPad) * (int)sizeof(bf16)); }

cudaError_t launch_norm_rows(const float* x, const float* ss, const float* gain, float eps,
                             int M_static, const int32_t* M_dev, int K, bf16* out, cudaStream_t st,
                             bool pdl) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(kMaxRows, (K + 2047) / 2048);
  lc.blockDim = dim3(256);
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, norm_rows_kernel, x, ss, gain, eps, M_static, M_dev, K, out);
}

GemvScratch gemv_scratch(int R, int K, int epi) {
  const Part p = make_part(R, K, epi);
  GemvScratch s;
  s.part_floats = (size_t)p.NRG * p.segmax * 256;
  s.counters = (size_t)p.NRG + 1;
  s.rec_floats = epi == EPI_LMHEAD ? (size_t)p.C * kMaxRows * 8 : 0;
  return s;
}

cudaError_t launch_gemv(int in_mode, int epi, const LinearArgs& a0, cudaStream_t st, bool pdl) {
  if (!part_fits(a0.R, a0.K)) return cudaErrorInvalidValue;
  // norm-fused rows must fit the activation stage (callers with more rows
  // run the RMSNorm pre-pass and a bf16-input projection)
  if (in_mode == IN_NORM && a0.M_static > gemv_stage_rows(a0.K)) return cudaErrorInvalidValue;
  LinearArgs a = a0;
  if (!a.M_dev && a.M_static > gemv_stage_rows(a.K)) a.wide = 1;
  const Part p = make_part(a.R, a.K, epi);
#define SSD_GEMV_CASE(I, E) \
  if (in_mode == I && epi == E) return launch_one<I, E>(a, p, st, pdl);
  SSD_GEMV_CASE(IN_BF16, EPI_STORE)
  SSD_GEMV_CASE(IN_NORM, EPI_STORE)
  SSD_GEMV_CASE(IN_BF16, EPI_RESID)
  SSD_GEMV_CASE(IN_NORM, EPI_SWIGLU)
  SSD_GEMV_CASE(IN_NORM, EPI_LMHEAD)
  SSD_GEMV_CASE(IN_BF16, EPI_SWIGLU)
  SSD_GEMV_CASE(IN_BF16, EPI_LMHEAD)
#undef SSD_GEMV_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_pack(const bf16* src, bf16* dst, int R, int K, cudaStream_t st) {
  const long long n = (long long)R * K / 8;
  long long blocks = (n + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  pack_kernel<<<(int)blocks, 256, 0, st>>>(src, dst, R, K);
  return cudaGetLastError();
}

}  // namespace ssd
