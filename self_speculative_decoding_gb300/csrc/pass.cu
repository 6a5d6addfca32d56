// Persistent pass kernel (sm_103a): one launch runs a whole decoding pass.
//
// A pass (a draft step, the verify pass, an autoregressive step) is a chain
// of dependent steps: embedding, then per layer the norm-fused QKV GEMV,
// attention, the O projection, the gate/up GEMV and the down projection,
// then the LM head and the draft-control step.  As separate kernels every
// step pays a launch, a ramp-up of the weight stream and a drain; here the
// grid stays resident and runs the steps as a program of phases:
//
//   * the producer warp of every CTA streams its share of each GEMV phase's
//     weights into the shared-memory ring back to back, across phase
//     boundaries and during attention (weights never depend on activations);
//   * the consumer warps start phase k once phase k-1 has signalled all of
//     its completions (row groups finished, attention heads combined, the
//     control step done) on a device counter; one thread per CTA polls it;
//   * the epilogue warp finishes row groups as in the single-GEMV kernel.
//
// Every phase runs the same device code as its single-step kernel (the GEMV
// roles, the attention work item, the control bodies) with the same
// partition, so a pass computes exactly the bits the multi-kernel path
// computes.  All CTAs of the fixed grid are resident at once (cooperative
// launch); every wait is bounded and an abort flag ends all of them.
#include "attn_dev.cuh"
#include "control_dev.cuh"
#include "gemv_dev.cuh"

namespace ssd {

using namespace gemv;

namespace {

struct __align__(16) PassSmem {
  GemvSmem g;
  uint64_t abar;   // attention bulk-copy barrier
  int flag;        // attention: this item combined its head
  int epoch;       // last phase this CTA has seen complete
  int epoch_ok;
  int s_M[2];
  int s_tok[kMaxRows];
};

SSD_DI int ld_volatile(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

SSD_DI void raise_abort(const PassProg& P, int code) {
  atomicExch(P.abort, 1);
  atomicCAS(P.err, 0, code);
}

// Phase k complete (all its completions signalled)?  Bounded; polls tightly
// at first, then backs off.  False on abort or time-out.
SSD_DI bool poll_done(const PassProg& P, int k) {
  const unsigned target = P.ph[k].target;
  for (int i = 0; i < (1 << 22); ++i) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(P.done + k) : "memory");
    if (v >= target) return true;
    if ((i & 63) == 63 && ld_volatile(P.abort)) return false;
    if (i > 1024) __nanosleep(64);
  }
  raise_abort(P, 7);
  return false;
}

// Epilogue warp: wait until this CTA's consumers have seen phase k complete.
SSD_DI bool epoch_wait(const PassProg& P, PassSmem& S, int k) {
  for (int i = 0; i < (1 << 24); ++i) {
    if (ld_volatile(&S.epoch) >= k) return true;
    if (ld_volatile(&S.epoch_ok) == 0 || ((i & 255) == 255 && ld_volatile(P.abort))) return false;
    if (i > 1024) __nanosleep(32);
  }
  raise_abort(P, 8);
  return false;
}

SSD_DI void signal(const PassProg& P, int k) {
  __threadfence();
  atomicAdd(P.done + k, 1u);
}

// Waits for the bulk copies this CTA's producer issued and nobody consumed
// (only after an error: normally every copy has been consumed).
SSD_DI void drain(GemvSmem& sm, const RingPos& rp) {
  const int n = rp.t < kSlots ? rp.t : kSlots;
  int slot = rp.slot;
  uint32_t ph = rp.ph;
  for (int i = 0; i < n; ++i) {
    if (--slot < 0) { slot = kSlots - 1; ph ^= 1u; }
    mbar_wait(&sm.full[slot], ph);
  }
}

__device__ __noinline__ void producer_any(int epi, const LinearArgs& a, GemvSmem& sm, int b, int lane, RingPos& rp) {
  const Part p = make_part(a.R, a.K, epi);
  switch (epi) {
    case EPI_STORE: producer_phase<EPI_STORE>(a, p, sm, b, lane, rp); break;
    case EPI_RESID: producer_phase<EPI_RESID>(a, p, sm, b, lane, rp); break;
    case EPI_SWIGLU: producer_phase<EPI_SWIGLU>(a, p, sm, b, lane, rp); break;
    case EPI_LMHEAD: producer_phase<EPI_LMHEAD>(a, p, sm, b, lane, rp); break;
  }
}

__device__ __noinline__ void epilogue_any(int epi, const LinearArgs& a, GemvSmem& sm, int b, int M, int lane,
                         RingPos& rp, unsigned* done) {
  const Part p = make_part(a.R, a.K, epi);
  switch (epi) {
    case EPI_STORE: epilogue_phase<EPI_STORE>(a, p, sm, b, M, lane, rp, done); break;
    case EPI_RESID: epilogue_phase<EPI_RESID>(a, p, sm, b, M, lane, rp, done); break;
    case EPI_SWIGLU: epilogue_phase<EPI_SWIGLU>(a, p, sm, b, M, lane, rp, done); break;
    case EPI_LMHEAD: epilogue_phase<EPI_LMHEAD>(a, p, sm, b, M, lane, rp, done); break;
  }
}

// One out-of-line function per GEMV variant: each gets its own register
// allocation, as in the single-GEMV kernel.
template <int IN, int EPI>
__device__ __noinline__ void consumer_one(const LinearArgs& a, GemvSmem& sm, int b, int M,
                                          int warp, int lane, RingPos& rp) {
  const Part p = make_part(a.R, a.K, EPI);
  consumer_phase<IN, EPI>(a, p, sm, b, M, warp, lane, rp);
}

SSD_DI void consumer_any(int in, int epi, const LinearArgs& a, GemvSmem& sm, int b, int M,
                         int warp, int lane, RingPos& rp) {
  if (in == IN_NORM && epi == EPI_STORE) consumer_one<IN_NORM, EPI_STORE>(a, sm, b, M, warp, lane, rp);
  else if (in == IN_NORM && epi == EPI_SWIGLU) consumer_one<IN_NORM, EPI_SWIGLU>(a, sm, b, M, warp, lane, rp);
  else if (in == IN_NORM && epi == EPI_LMHEAD) consumer_one<IN_NORM, EPI_LMHEAD>(a, sm, b, M, warp, lane, rp);
  else if (in == IN_BF16 && epi == EPI_STORE) consumer_one<IN_BF16, EPI_STORE>(a, sm, b, M, warp, lane, rp);
  else if (in == IN_BF16 && epi == EPI_RESID) consumer_one<IN_BF16, EPI_RESID>(a, sm, b, M, warp, lane, rp);
  else rp.ok = false;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) pass_kernel(PassProg P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  PassSmem& S = *reinterpret_cast<PassSmem*>(smem_raw);
  GemvSmem& sm = S.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumers);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.rfull[s], kConsumers);
      mbar_init(&sm.rempty[s], 1);
    }
    mbar_init(&S.abar, 1);
    fence_mbar_init();
    S.epoch = -1;
    S.epoch_ok = 1;
  }
  __syncthreads();
  RingPos rp;

  if (warp == kProducer) {
    // ---- weight stream of every GEMV phase, in program order
    if (lane == 0) {
      for (int k = 0; k < P.n && rp.ok; ++k) {
        const PassPhase ph = P.ph[k];
        if (ph.kind != PK_GEMV) continue;
        if (ld_volatile(P.abort)) break;
        const LinearArgs& a = P.lin[ph.idx];
        producer_any(ph.epi, a, sm, b, lane, rp);
      }
      if (!rp.ok || ld_volatile(P.abort)) {
        raise_abort(P, 2);
        drain(sm, rp);
      }
    }
  } else if (warp == kEpilogue) {
    // ---- row-group epilogues of every GEMV phase
    for (int k = 0; k < P.n; ++k) {
      const PassPhase ph = P.ph[k];
      if (ph.kind != PK_GEMV) continue;
      int ok = 1;
      if (lane == 0) ok = k == 0 || epoch_wait(P, S, k - 1);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int M = __ldcg(&P.st->M);
      const LinearArgs& a = P.lin[ph.idx];
      epilogue_any(ph.epi, a, sm, b, M, lane, rp, P.done + k);
      if (!rp.ok) {
        if (lane == 0) raise_abort(P, 4);
        break;
      }
    }
  } else {
    // ---- consumer warps: MMAs, attention items, control steps
    const int tid = threadIdx.x;
    uint32_t aphase = 0;
    for (int k = 0; k < P.n; ++k) {
      const PassPhase ph = P.ph[k];
      if (k > 0) {
        // one decision for all consumer warps: a warp that failed in the
        // previous phase still takes part in this barrier
        if (tid == 0) {
          if (ld_volatile(&S.epoch_ok) != 0 && poll_done(P, k - 1)) {
            *reinterpret_cast<volatile int*>(&S.epoch) = k - 1;
          } else {
            *reinterpret_cast<volatile int*>(&S.epoch_ok) = 0;
          }
        }
        consumer_sync();
        if (ld_volatile(&S.epoch_ok) == 0) break;
      }
      if (ph.kind == PK_GEMV) {
        const int M = __ldcg(&P.st->M);
        const LinearArgs& a = P.lin[ph.idx];
        consumer_any(ph.in, ph.epi, a, sm, b, M, warp, lane, rp);
        if (!rp.ok && lane == 0) {
          raise_abort(P, 3);
          *reinterpret_cast<volatile int*>(&S.epoch_ok) = 0;
        }
      } else if (ph.kind == PK_ATTN) {
        const AttnArgs& a = P.att[ph.idx];
        const int M = __ldcg(&P.st->M), pos0 = __ldcg(&P.st->pos0);
        const int ns = a.ns_dev ? __ldcg(a.ns_dev) : 0;
        const attn::Smem asm_ = attn::carve(reinterpret_cast<unsigned char*>(sm.stage), a.dh,
                                            a.max_seq / kAttnChunk);
        // the staging area was last written through the generic proxy
        fence_proxy_async_smem();
        consumer_sync();
        const int n_items = ((pos0 + M - ns - 1) / kAttnChunk + 1) * a.Hkv;
        for (int it = b; it < n_items; it += gridDim.x) {
          const bool fin = attn::item(a, M, ns, pos0, it, asm_, &S.abar, aphase, &S.flag, tid,
                                      [] { consumer_sync(); });
          if (fin && tid == 0) signal(P, k);
        }
      } else if (b == 0) {
        if (ph.kind == PK_BEGIN) {
          ctl::begin(P.beg[ph.idx], tid, kConsumers * 32, S.s_M, S.s_tok,
                     [] { consumer_sync(); });
          consumer_sync();
        } else if (ph.kind == PK_SAVE) {
          SaveArgs sa;
          sa.st = P.st;
          sa.use_d = ph.use_d;
          sa.x = P.x;
          sa.ss = P.ss;
          sa.bx = P.bx;
          sa.bss = P.bss;
          sa.bxs = P.bxs;
          sa.bsss = P.bsss;
          sa.D = P.D;
          ctl::save_boundary(sa, tid, kConsumers * 32, [] { consumer_sync(); });
          consumer_sync();
        } else if (ph.kind == PK_DRAFT_END) {
          if (tid == 0) {
            DraftEndArgs da;
            da.st = P.st;
            da.dstats = P.dstats;
            da.tau = ph.tau;
            da.temperature = ph.temperature;
            da.tree_tau = ph.tree_tau;
            da.tree_max = ph.tree_max;
            ctl::draft_end(da);
          }
        } else if (ph.kind == PK_AR_END) {
          if (tid == 0)
            ctl::ar_end(P.st, P.tokens, P.vstats, ph.row_from_M, ph.temperature, ph.reset);
        }
        if (tid == 0) signal(P, k);
      }
    }
  }

  // ---- the last CTA out returns the counters to zero for the next launch
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(P.exit_count, 1u) == gridDim.x - 1) {
      for (int k = 0; k < P.n; ++k) P.done[k] = 0u;
      *P.exit_count = 0u;
      __threadfence();
    }
  }
}

int g_pass_ready = -1;  // -1 unknown, 0 unusable, 1 ready

}  // namespace

bool pass_supported(int dh, int max_seq) {
  return attn::smem_bytes(dh, max_seq / kAttnChunk) <= (size_t)kStageBytes;
}

cudaError_t pass_prepare() {
  if (g_pass_ready == 1) return cudaSuccess;
  const int smem = (int)sizeof(PassSmem) + 128;
  cudaError_t e = cudaFuncSetAttribute(pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pass_kernel, kThreads, smem)) !=
      cudaSuccess)
    return e;
  if (per_sm * sms < kGridCtas) {
    g_pass_ready = 0;
    return cudaErrorCooperativeLaunchTooLarge;
  }
  g_pass_ready = 1;
  return cudaSuccess;
}

cudaError_t launch_pass(const PassProg& p, cudaStream_t st) {
  const int smem = (int)sizeof(PassSmem) + 128;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(kGridCtas);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, pass_kernel, p);
}

}  // namespace ssd
