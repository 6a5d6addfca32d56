// Many-row projection on the 5th-generation tensor cores (tcgen05, sm_103a):
// the batched candidate-mask scoring forward (SWIFT §4.1.2: every candidate
// layer set predicts the last N context tokens in one parallel forward; K
// candidates give K * N rows).
//
// D[r][t] = sum_k W[r][k] act[t][k] over T rows t (tokens) and R outputs r.
// With hundreds of rows every weight tile is used by every token tile, so the
// work is a dense contraction.
//
// CTA tile: 128 outputs (8 packed row groups; for SwiGLU 4 gate/up pairs,
// virtual group 2p = gate, 2p + 1 = up) x NT tokens (NT <= 256, a multiple
// of 16 chosen per launch so that the token tiles split T evenly).  The
// accumulator lives in tensor memory: 128 lanes (outputs) x NT columns
// (tokens) of fp32.
//
// Operands are staged in shared memory in the K-major 64-byte-swizzle
// layout the MMA descriptors read: the weights' packed units already are in
// that layout (an 8-row half of a unit is one 512-byte swizzle atom), so a
// unit is copied as is; activation rows are placed chunk by chunk with the
// same swizzle.  A stage holds 64 K columns; all 128 threads fill stages
// with 16-byte cp.async copies, one thread issues the MMAs of a stage
// (4 x K16) and commits them to the stage's mbarrier, which frees the stage
// for the copies three stages ahead.  Every output sums its K in ascending
// order in one accumulator, so the result depends on the shapes only.
//
// Epilogue: each warp reads its 32 TMEM lanes (tcgen05.ld, 16 columns at a
// time): store fp32; residual add into the rows named by a row map; SwiGLU to
// bf16 (gate and up rows exchanged across half-warps); per-token argmax
// (largest value, lowest index) through a 64-bit atomic max of an
// order-preserving key, independent of the order CTAs finish in.
//
// Waits are bounded: a stage barrier that never completes sets the error
// word, and the CTA drains its own copies, frees its tensor memory and
// returns.
#include "kernels.cuh"

namespace ssd {

namespace {

constexpr int kTcM = 128;          // outputs per tile
constexpr int kTcGroups = 8;       // 16-row groups per tile
constexpr int kTcKbs = 2;          // 32-wide K blocks per stage
constexpr int kTcStages = 4;
constexpr int kTcThreads = 128;
constexpr int kTcMaxN = 256;
constexpr int kTcABytes = kTcKbs * kTcGroups * 1024;   // weights of one stage
constexpr int kWaitPolls = 1 << 24;

SSD_DI void cp16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
SSD_DI void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
SSD_DI void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
SSD_DI void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- tcgen05 helpers
SSD_DI void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
SSD_DI void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
SSD_DI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SSD_DI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 64-byte swizzle, 8-row atoms of
// 512 bytes stacked densely along M/N (stride 512 bytes).
SSD_DI uint64_t sw64_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                             // leading offset (unused here)
  d |= (uint64_t)(512 >> 4) << 32;                    // stride offset
  d |= (uint64_t)1 << 46;                             // descriptor version
  d |= (uint64_t)4 << 61;                             // 64-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

SSD_DI void mma_bf16_tc(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
SSD_DI void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}
SSD_DI void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// float -> uint32 with the same order (argmax keys)
SSD_DI uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TcShape {
  int NT;        // tokens per tile (multiple of 16, <= 256)
  int tiles;     // token tiles
  int ncols;     // tensor-memory columns allocated (power of 2, >= 32)
  size_t smem;   // dynamic shared memory
};

TcShape tc_shape(int T) {
  TcShape s;
  s.tiles = (T + kTcMaxN - 1) / kTcMaxN;
  const int per = (T + s.tiles - 1) / s.tiles;
  s.NT = ((per + 15) / 16) * 16;
  s.ncols = 32;
  while (s.ncols < s.NT) s.ncols <<= 1;
  const size_t stage = (size_t)kTcABytes + (size_t)kTcKbs * s.NT * 64;
  s.smem = 1024 + kTcStages * stage + 256;
  return s;
}

__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(GemmArgs a, int NT, int ncols) {
  extern __shared__ unsigned char sm_raw[];
  // 1024-byte aligned stage area (the swizzle pattern repeats every 512 bytes
  // of the absolute shared-memory address)
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
  const int stage_bytes = kTcABytes + kTcKbs * NT * 64;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kTcStages * stage_bytes);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + kTcStages);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KB = a.K / 32;
  const int nkb = (KB + kTcKbs - 1) / kTcKbs;                         // stages of K
  const bool swiglu = a.epi == GEMM_SWIGLU;
  const int NRG = (swiglu ? 2 : 1) * (a.R / 16);
  const int rg0 = blockIdx.y * kTcGroups;
  const int t0 = blockIdx.x * NT;

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) mbar_init(&bar[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, (uint32_t)ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  auto unit_src = [&](int v, int kb) -> const unsigned char* {
    if (swiglu) {
      const bf16* W = (v & 1) ? a.W1 : a.W0;
      return reinterpret_cast<const unsigned char*>(W) + ((size_t)(v >> 1) * KB + kb) * 1024;
    }
    return reinterpret_cast<const unsigned char*>(a.W0) + ((size_t)v * KB + kb) * 1024;
  };
  // fill stage st with the K blocks of step s
  auto load_stage = [&](int s, int st) {
    unsigned char* A = sm + st * stage_bytes;
    unsigned char* B = A + kTcABytes;
    for (int e = tid; e < kTcKbs * kTcGroups * 64; e += kTcThreads) {
      const int kbl = e / (kTcGroups * 64), rem = e % (kTcGroups * 64);
      const int u = rem / 64, q = rem % 64;
      const int kb = s * kTcKbs + kbl, v = rg0 + u;
      const bool ok = kb < KB && v < NRG;
      cp16(A + kbl * (kTcGroups * 1024) + u * 1024 + q * 16,
           ok ? unit_src(v, kb) + q * 16 : reinterpret_cast<const unsigned char*>(a.W0), ok);
    }
    for (int e = tid; e < kTcKbs * NT * 4; e += kTcThreads) {
      const int kbl = e / (NT * 4), rem = e % (NT * 4);
      const int n = rem / 4, c = rem % 4;
      const int kb = s * kTcKbs + kbl, t = t0 + n;
      const bool ok = kb < KB && t < a.T;
      const int r8 = n & 7;
      cp16(B + kbl * (NT * 64) + (n >> 3) * 512 + r8 * 64 + ((c ^ ((r8 >> 1) & 3)) << 4),
           ok ? a.act + (size_t)t * a.K + (size_t)kb * 32 + c * 8 : a.act, ok);
    }
  };

  const uint32_t idesc = idesc_bf16(kTcM, NT);
  bool ok = true;
#pragma unroll
  for (int s = 0; s < kTcStages - 1; ++s) {
    if (s < nkb) load_stage(s, s);
    cp_commit();
  }
  for (int s = 0; s < nkb; ++s) {
    const int st = s % kTcStages;
    cp_wait<kTcStages - 2>();
    fence_async_smem();
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    if (tid == 0) {
      tc_fence_after();
      const uint32_t A = smem_addr(sm + st * stage_bytes);
      const uint32_t B = A + kTcABytes;
#pragma unroll
      for (int kbl = 0; kbl < kTcKbs; ++kbl) {
        if (s * kTcKbs + kbl < KB) {
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            const uint64_t ad = sw64_desc(A + kbl * (kTcGroups * 1024) + ks * 32);
            const uint64_t bd = sw64_desc(B + kbl * (NT * 64) + ks * 32);
            mma_bf16_tc(tmem, ad, bd, idesc, (s | kbl | ks) != 0);
          }
        }
      }
      mma_commit(&bar[st]);
    }
    // the stage refilled next was read by the MMAs of step s - 1
    const int nxt = s + kTcStages - 1;
    if (s >= 1 && nxt < nkb) {
      const int ps = (s - 1) % kTcStages;
      if (!mbar_wait_n(&bar[ps], (uint32_t)(((s - 1) / kTcStages) & 1), kWaitPolls)) ok = false;
    }
    if (ok && nxt < nkb) load_stage(nxt, nxt % kTcStages);
    cp_commit();
  }
  // every MMA done (a commit tracks all MMAs issued before it)
  if (ok) {
    const int ls = (nkb - 1) % kTcStages;
    if (!mbar_wait_n(&bar[ls], (uint32_t)(((nkb - 1) / kTcStages) & 1), kWaitPolls)) ok = false;
  }
  ok = __syncthreads_and(ok) != 0;
  if (!ok) {
    if (tid == 0 && a.err) atomicExch(a.err, 5);
    cp_wait<0>();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, (uint32_t)ncols);
    return;
  }
  tc_fence_after();

  // ---- epilogue: warp w owns tile rows 32w .. 32w + 31 (TMEM lanes)
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  const int vrow = rg0 * 16 + warp * 32 + lane;   // (virtual) output row
  for (int c0 = 0; c0 < NT; c0 += 16) {
    float v[16];
    tmem_ld16(trow + (uint32_t)c0, v);
    if (a.epi == GEMM_ARGMAX) {
      const bool rv = vrow < a.R;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int tok = t0 + c0 + j;
        float bv = rv ? v[j] : -INFINITY;
        int bi = rv ? vrow : 0x7fffffff;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0 && tok < a.T && bi != 0x7fffffff)
          atomicMax(a.best + tok, ((unsigned long long)order_key(bv) << 32) |
                                      (unsigned long long)(0xffffffffu - (uint32_t)bi));
      }
    } else if (swiglu) {
      // lanes 0-15: gate rows of pair p, lanes 16-31: the matching up rows
      const int pair = (rg0 >> 1) + warp;
      const bool pv = 2 * pair + 1 < NRG;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float up = __shfl_xor_sync(0xffffffffu, v[j], 16);
        const int tok = t0 + c0 + j;
        if (lane < 16 && pv && tok < a.T) {
          const float gt = v[j];
          const float sl = gt / (1.0f + expf(-gt));
          a.u[(size_t)tok * a.R + pair * 16 + lane] = __float2bfloat16_rn(sl * up);
        }
      }
    } else if (vrow < a.R) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int tok = t0 + c0 + j;
        if (tok < a.T) {
          if (a.epi == GEMM_STORE) {
            a.y[(size_t)tok * a.R + vrow] = v[j];
          } else {
            const size_t orow = a.rowmap ? (size_t)a.rowmap[tok] : (size_t)tok;
            a.x[orow * a.R + vrow] += v[j];
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, (uint32_t)ncols);
}

// idx[t] = the index held by an argmax key.
__global__ void argmax_index_kernel(const unsigned long long* best, int T, int32_t* idx) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T) idx[t] = best[t] ? (int)(0xffffffffu - (uint32_t)(best[t] & 0xffffffffull)) : -1;
}

}  // namespace

cudaError_t launch_argmax_index(const unsigned long long* best, int T, int32_t* idx,
                                cudaStream_t s) {
  argmax_index_kernel<<<(T + 255) / 256, 256, 0, s>>>(best, T, idx);
  return cudaGetLastError();
}

cudaError_t launch_gemm_rows(const GemmArgs& a, cudaStream_t s) {
  if (a.R % 16 || a.K % 32 || a.T <= 0) return cudaErrorInvalidValue;
  const TcShape sh = tc_shape(a.T);
  static size_t smem_set = 0;
  if (sh.smem > smem_set) {
    const cudaError_t e = cudaFuncSetAttribute(
        gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sh.smem);
    if (e != cudaSuccess) return e;
    smem_set = sh.smem;
  }
  const int NRG = (a.epi == GEMM_SWIGLU ? 2 : 1) * (a.R / 16);
  dim3 grid(sh.tiles, (NRG + kTcGroups - 1) / kTcGroups);
  gemm_tc_kernel<<<grid, kTcThreads, sh.smem, s>>>(a, sh.NT, sh.ncols);
  return cudaGetLastError();
}

}  // namespace ssd
