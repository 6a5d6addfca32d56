// Many-row projection on the 5th-generation tensor cores (tcgen05, sm_103a):
// the batched candidate-mask scoring forward (SWIFT §4.1.2: every candidate
// layer set predicts the last N context tokens in one parallel forward; K
// candidates give K * N rows).
//
// D[r][t] = sum_k W[r][k] act[t][k] over T rows t (tokens) and R outputs r.
// With hundreds of rows every weight tile is used by every token tile, so the
// work is a dense contraction.
//
// CTA tile: 128 outputs (8 packed row groups) x NT tokens (NT <= 256, a
// multiple of 16 chosen per launch from a cost model of CTA rounds and bytes
// streamed).  Accumulators live in tensor memory: 128 lanes (outputs) x NT
// columns (tokens) of fp32, up to four side by side, their number fixed by
// the matrix (not by T).  A SwiGLU tile holds 128 features: the gate rows
// accumulate in columns [0, NT), the up rows of the same features in
// [NT, 2 NT), so one thread sees both halves of its feature.  Other tiles use
// one accumulator, or four that take the K16 steps j of every stage by
// j mod 4 and are added in order in the epilogue.
//
// Operands are staged in shared memory in the K-major 64-byte-swizzle layout
// the MMA descriptors read.  Weights and activations are both stored in the
// packed unit layout (16 rows x 32 columns; each 8-row half is one 512-byte
// swizzle atom), which a tensor map views as a 3-D tensor of 8-byte
// elements (the 1 KB of a unit, 16-row groups, K blocks): one tiled TMA copy
// brings 8 row groups of all the K blocks of a stage ([K block][group][unit],
// 8 KB per K block), another the token tile's K blocks (NT x 64 bytes per K
// block), rows beyond the matrix and K blocks beyond K zero-filled.  Thread 0
// issues the copies (stage barrier `full`, transaction bytes): the copy
// engine accepts one tiled copy every 75-110 ns per SM, so a copy per
// operand per stage rather than per K block keeps the loads ahead of the
// MMAs.  One thread per accumulator, each in its own warp, issues the MMAs
// (a single thread issues M = 128 MMAs at the tensor core's own rate, about
// N / 2 cycles each).  Each commits its MMAs of a stage to the stage's
// `empty` barrier (one arrival per issuer frees it for the copies `stages`
// steps ahead), and last to `done`.  All loops advance their slot and phase
// parity incrementally (no division in the issue path).  Every accumulator
// sums its K steps in ascending order, so the result depends on the shapes
// only.
//
// Epilogue: each warp reads its 32 TMEM lanes (tcgen05.ld, 16 columns at a
// time): store fp32; residual add into the rows named by a row map; SwiGLU to
// bf16; per-token argmax (largest value, lowest index) through a 64-bit
// atomic max of an order-preserving key, independent of the order CTAs
// finish in.
//
// Waits are bounded: a barrier that never completes sets the error word,
// and the CTA waits (bounded) for its own copies, frees its tensor memory and
// returns.
#include <cuda.h>

#include "kernels.cuh"
#include "tc_dev.cuh"

namespace ssd {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no
// link-time dependency on the driver library); null if unavailable.
EncodeTiled tma_encoder() {
  static EncodeTiled fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

namespace {

using namespace tc;

constexpr int kTcM = 128;          // outputs per tile
constexpr int kTcGroups = 8;       // 16-row groups per tile
constexpr int kTcMaxStages = 16;
constexpr int kTcThreads = 160;    // warp 0: copies; warps 1-4: MMA issuers; warps 0-3: epilogue
constexpr int kTcMaxN = 256;
constexpr int kTcManyTiles = 100;  // 128-row tiles from which a matrix uses one accumulator
#ifndef SSD_TC_SMEM_KB
#define SSD_TC_SMEM_KB 224
#endif
#ifndef SSD_TC_KBS
#define SSD_TC_KBS 0  // K blocks per stage; 0: chosen per shape
#endif
// stage memory of a CTA alone on its SM, and of each of two CTAs on an SM
// (227 KB per CTA at most; two CTAs share 228 KB less 1 KB each)
constexpr int kTcSmemBudget1 = SSD_TC_SMEM_KB * 1024;
constexpr int kTcSmemBudget2 = 108 * 1024;
constexpr int kWaitPolls = 1 << 24;

// Barrier of the four epilogue warps (threads 0 .. 127).
SSD_DI void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// float -> uint32 with the same order (argmax keys)
SSD_DI uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}


struct TcShape {
  int NT;          // tokens per tile (multiple of 16, <= 256)
  int tiles;       // token tiles
  int ncols;       // tensor-memory columns allocated (power of 2, >= 32)
  int nacc;        // accumulators = MMA-issuing threads (1, 2 or 4)
  int kbs;         // 32-wide K blocks per stage (2 or 4)
  int stages;      // pipeline depth
  int stage_bytes; // kTcKbs x (weights (8 KB, 16 KB for SwiGLU) + activations (NT x 64 B))
  size_t smem;     // dynamic shared memory
};

// Accumulators (= MMA-issuing threads) depend on the matrix only, never on
// T, so that a row's bits do not depend on how many rows are processed
// together: SwiGLU 2 (gate, up); matrices with few 128-row tiles 4 (the K16
// steps dealt by j mod 4; tiles of at most 128 tokens keep 4 accumulators in
// tensor memory); matrices with many tiles 1 (their grids want two CTAs per
// SM, which one accumulator of up to 256 columns allows).
// Token tiling: among the tile counts from the fewest the column limit
// allows up to tiles of 32 tokens, the one with the least (CTA rounds x
// bytes a CTA streams per K block: its weights plus NT tokens).
TcShape tc_shape(int T, bool swiglu, int m_tiles, int sms) {
  TcShape s;
  s.nacc = swiglu ? 2 : (m_tiles < kTcManyTiles ? 4 : 1);
  const int max_n = s.nacc == 4 ? 128 : kTcMaxN;
  const int wcols = (swiglu ? 2 : 1) * 128;   // weight bytes per K block / 64
  long best = -1;
  for (int tiles = (T + max_n - 1) / max_n;; ++tiles) {
    const int NT = ((T + tiles - 1) / tiles + 15) / 16 * 16;
    const int n = (T + NT - 1) / NT;
    const long cost = (long)((m_tiles * n + sms - 1) / sms) * (NT + wcols);
    if (best < 0 || cost < best) {
      best = cost;
      s.NT = NT;
      s.tiles = n;
    }
    if (NT <= 32) break;
  }
  auto pow2 = [](int c) { int n = 32; while (n < c) n <<= 1; return n; };
  s.ncols = pow2(s.nacc * s.NT);
  const int kb_bytes = (swiglu ? 2 : 1) * kTcGroups * 1024 + s.NT * 64;
  // shared memory sized so that the whole grid is resident at once when it
  // fits (up to 2 CTAs per SM; tensor memory allows 512 / ncols)
  int per_sm = (m_tiles * s.tiles + sms - 1) / sms;
  if (per_sm > 2) per_sm = 2;
  if (per_sm > 512 / s.ncols) per_sm = 512 / s.ncols;
  if (per_sm < 1) per_sm = 1;
  // deeper stages (4 K blocks) amortise each issuer's per-stage barrier
  // wait, fence and commit when at least 3 of them still fit
  const int budget = per_sm == 1 ? kTcSmemBudget1 : kTcSmemBudget2;
  s.kbs = budget / (4 * kb_bytes) >= 3 ? 4 : 2;
  // a stage's 2 kbs K16 steps are dealt to the issuers of a matrix by j mod
  // per, so kbs is 2 or 4 (the deal is then the step's index mod per)
  if (SSD_TC_KBS == 2 || SSD_TC_KBS == 4) s.kbs = SSD_TC_KBS;
  // no copy box above 32 KB (a 64 KB box of activations failed to encode)
  if (s.kbs == 4 && 4 * s.NT * 64 > 32768) s.kbs = 2;
  s.stage_bytes = s.kbs * kb_bytes;
  s.stages = budget / s.stage_bytes;
  if (s.stages > kTcMaxStages) s.stages = kTcMaxStages;
  if (s.stages < 2) s.stages = 2;
  s.smem = 1024 + (size_t)s.stages * s.stage_bytes + 512;
  return s;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mW0, const __grid_constant__ CUtensorMap mW1,
                   const __grid_constant__ CUtensorMap mAct, GemmArgs a, int NT, int ncols,
                   int stages, int stage_bytes, int tx_stage, int nacc, int kbs, int kbox,
                   int wsplit) {
  extern __shared__ unsigned char sm_raw[];
  // 1024-byte aligned stage area (the swizzle pattern repeats every 512 bytes
  // of the absolute shared-memory address)
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + stages * stage_bytes);
  uint64_t* empty = full + kTcMaxStages;
  uint64_t* done = empty + kTcMaxStages;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  int* fail = reinterpret_cast<int*>(tslot + 1);
  int* issued = fail + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KB = a.K / 32;
  const bool swiglu = a.epi == GEMM_SWIGLU;
  constexpr int wkb = kTcGroups * 1024;                    // one matrix's bytes per K block
  const int a_kb = (swiglu ? 2 : 1) * wkb;                 // weight bytes per K block
  const int rg0 = blockIdx.y * kTcGroups;
  const int t0 = blockIdx.x * NT;

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nacc);   // one commit per MMA issuer
    }
    mbar_init(done, nacc);
    *fail = 0;
    *issued = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, (uint32_t)ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  // A stage holds kbs K blocks: the weights [kbl][8 KB] (SwiGLU: all the
  // gate blocks, then all the up blocks), then the activations
  // [kbl][NT x 64 B].  Slots and phase parities advance incrementally.
  const int nst = (KB + kbs - 1) / kbs;
  if (warp == 0 && lane == 0) {
    // producer: per stage one box of kbox K blocks of 8 weight row groups
    // (one per K block for matrices of fewer row groups; two matrices for
    // SwiGLU) and one box of the tile's tokens
    asm volatile("prefetch.tensormap [%0];" ::"l"(&mW0) : "memory");
    if (swiglu) asm volatile("prefetch.tensormap [%0];" ::"l"(&mW1) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&mAct) : "memory");
    int s = 0, st = 0;
    uint32_t par = 0;
    unsigned char* S = sm;
    for (; s < nst; ++s) {
      if (s >= stages && !mbar_wait_n(&empty[st], par ^ 1u, kWaitPolls)) {
        atomicExch(fail, 1);
        break;
      }
      const int kb0 = s * kbs;
      mbar_arrive_expect_tx(&full[st], (uint32_t)tx_stage);
      if (!wsplit) {
        tma_load_3d(S, &mW0, 0, rg0, kb0, &full[st]);
        if (swiglu) tma_load_3d(S + kbs * wkb, &mW1, 0, rg0, kb0, &full[st]);
      } else {
        for (int kbl = 0; kbl < kbox; ++kbl) {
          tma_load_3d(S + kbl * wkb, &mW0, 0, rg0, kb0 + kbl, &full[st]);
          if (swiglu) tma_load_3d(S + (kbs + kbl) * wkb, &mW1, 0, rg0, kb0 + kbl, &full[st]);
        }
      }
      tma_load_3d(S + kbs * a_kb, &mAct, 0, t0 / 16, kb0, &full[st]);
      if (++st == stages) {
        st = 0;
        par ^= 1u;
        S = sm;
      } else {
        S += stage_bytes;
      }
    }
    *issued = s;
  } else if (warp >= 1 && warp <= nacc && lane == 0) {
    // MMA issuers (one thread's issue rate alone cannot keep the tensor core
    // busy), each into its own accumulator of NT columns: the K16 steps j
    // of a stage (j = 2 kbl + ks) are dealt to the `per` issuers of a matrix
    // by j mod per; for SwiGLU issuers 0 .. per-1 take the gate rows and
    // per .. 2 per-1 the up rows.  Descriptors advance by adding the byte
    // offset / 16 to the start field.
    const int who = warp - 1;
    const int per = swiglu ? nacc / 2 : nacc;
    const int r = who % per;
    const uint32_t idesc = idesc_bf16(kTcM, NT);
    const uint64_t d0 = sw64_desc(smem_addr(sm));
    const uint32_t dcol = tmem + (uint32_t)(who * NT);
    const uint32_t wofs = swiglu && who >= per ? (uint32_t)(kbs * wkb >> 4) : 0u;
    int st = 0;
    uint32_t par = 0, off = 0;
    for (int s = 0; s < nst; ++s) {
      if (!mbar_wait_n(&full[st], par, kWaitPolls)) {
        atomicExch(fail, 1);
        break;
      }
      tc_fence_after();
      const int nj = 2 * min(kbs, KB - s * kbs);
      for (int j = r; j < nj; j += per) {
        const int kbl = j >> 1, ks = j & 1;
        const uint64_t da = d0 + ((off + kbl * wkb) >> 4) + wofs + 2 * ks;
        const uint64_t db = d0 + ((off + kbs * a_kb + kbl * (NT * 64)) >> 4) + 2 * ks;
        mma_bf16_tc(dcol, da, db, idesc, (s != 0 || j != r) ? 1u : 0u);
      }
      mma_commit(&empty[st]);
      if (++st == stages) {
        st = 0;
        par ^= 1u;
        off = 0;
      } else {
        off += stage_bytes;
      }
    }
    // arrives once every MMA this thread issued has completed
    mma_commit(done);
  }
  __syncwarp();
  bool ok = mbar_wait_n(done, 0u, kWaitPolls);
  __syncthreads();
  ok = __syncthreads_and(ok && *reinterpret_cast<volatile int*>(fail) == 0) != 0;
  if (!ok) {
    if (tid == 0) {
      if (a.err) atomicExch(a.err, 5);
      // let this CTA's copies still in flight land before the memory is released
      const int n = *issued;
      for (int s = n - 1; s >= 0 && s >= n - stages; --s)  // stage steps issued last
        mbar_wait_n(&full[s % stages], (uint32_t)((s / stages) & 1), 1 << 20);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, (uint32_t)ncols);
    return;
  }
  tc_fence_after();

  // ---- epilogue: warp w < 4 owns tile rows 32w .. 32w + 31 (TMEM lanes).
  // A matrix's value is the sum of its issuers' accumulators in issuer
  // order; an issuer that received no K16 step (2 KB < per) holds nothing.
  if (warp >= 4) {
    tc_fence_before();
    __syncthreads();
    return;
  }
  const int per = swiglu ? nacc / 2 : nacc;
  const int nsum = min(per, 2 * KB);
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  const int row = rg0 * 16 + warp * 32 + lane;   // output row (feature for SwiGLU)
  const bool rv = row < a.R;
  // Residual add: the tile's residual rows are staged in the stage memory
  // (idle once every MMA has completed) with 16-byte asynchronous copies, all
  // in flight at once, in passes of as many tokens as it holds: xs[t][128]
  // floats, then the pass's map rows.
  const bool resid = a.epi == GEMM_RESID;
  const int ns_max = min(NT, ((stages * stage_bytes - 1024) / 512) & ~15);
  float* xs = reinterpret_cast<float*>(sm);
  int* orow_s = reinterpret_cast<int*>(sm + (size_t)ns_max * 512);
  const int rows_here = min(kTcM, a.R - rg0 * 16);  // tile rows inside the matrix (multiple of 16)
  const int pass = resid ? ns_max : NT;
  for (int p0 = 0; p0 < NT; p0 += pass) {
    const int np = min(pass, NT - p0);
    if (resid) {
      epi_sync();  // the previous pass's reads of xs are done
      for (int t = tid; t < np; t += kTcM) {
        const int tok = t0 + p0 + t;
        orow_s[t] = tok < a.T ? (a.rowmap ? __ldg(a.rowmap + tok) : tok) : -1;
      }
      epi_sync();
      for (int e = tid; e < np * 32; e += kTcM) {
        const int t = e >> 5, q = e & 31;
        const int om = orow_s[t];
        if (om >= 0 && q * 4 < rows_here)
          cp_async16(xs + t * kTcM + q * 4, a.x + (size_t)om * a.R + rg0 * 16 + q * 4);
      }
      cp_async_wait_all();
      epi_sync();
    }
    // 16 columns at a time (32 for a single accumulator without SwiGLU): every
    // TMEM load of the step is issued before one wait; a matrix's value is
    // its issuers' accumulators added in issuer order
    for (int cs = p0; cs < p0 + np;) {
      const bool two = nsum == 1 && !swiglu && cs + 32 <= p0 + np;
      float vv[2][16], upv[16];
      {
        uint32_t r0[16], r1[16], r2[16], r3[16];
        tmem_ld16_nw(trow + (uint32_t)cs, r0);
        if (two || nsum > 1) tmem_ld16_nw(trow + (uint32_t)((two ? 0 : NT) + cs + (two ? 16 : 0)), r1);
        if (nsum > 2) tmem_ld16_nw(trow + (uint32_t)(2 * NT + cs), r2);
        if (nsum > 3) tmem_ld16_nw(trow + (uint32_t)(3 * NT + cs), r3);
        if (swiglu) tmem_ld16_nw(trow + (uint32_t)(per * NT + cs), r3);  // per == nsum == 1
        tmem_wait_ld();
        tmem_pin16(r0);
        if (two || nsum > 1) tmem_pin16(r1);
        if (nsum > 2) tmem_pin16(r2);
        if (nsum > 3 || swiglu) tmem_pin16(r3);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float x = __uint_as_float(r0[j]);
          if (!two && nsum > 1) x += __uint_as_float(r1[j]);
          if (nsum > 2) x += __uint_as_float(r2[j]);
          if (nsum > 3) x += __uint_as_float(r3[j]);
          vv[0][j] = x;
          vv[1][j] = __uint_as_float(r1[j]);
          upv[j] = __uint_as_float(r3[j]);
        }
      }
      for (int hh = 0; hh < (two ? 2 : 1); ++hh) {
      const int c0 = cs + 16 * hh;
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = vv[hh][j];
      if (a.epi == GEMM_ARGMAX) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = t0 + c0 + j;
          float bv = rv ? v[j] : -INFINITY;
          int bi = rv ? row : 0x7fffffff;
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
        const float* up = upv;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = t0 + c0 + j;
          if (rv && tok < a.T) {
            // silu; the scoring forward takes the fast exponential and division
            // (the full-precision pair costs most of its epilogue, and the product
            // is rounded to bf16), the prefill the full-precision pair
            const float gt = v[j];
            const float sl = a.fast_silu ? __fdividef(gt, 1.0f + __expf(-gt))
                                         : gt / (1.0f + expf(-gt));
            a.u[a.u_packed ? packed_off(tok, row, a.R) : (size_t)tok * a.R + row] =
                __float2bfloat16_rn(sl * up[j]);
          }
        }
      } else if (resid) {
        if (rv) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = c0 - p0 + j;
            const int om = orow_s[t];
            if (om >= 0) a.x[(size_t)om * a.R + row] = xs[t * kTcM + warp * 32 + lane] + v[j];
          }
        }
      } else if (rv) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = t0 + c0 + j;
          if (tok < a.T) a.y[(size_t)tok * a.R + row] = v[j];
        }
      }
      }
      cs += two ? 32 : 16;
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

// dst (packed unit layout) = src [T][K] row-major; rows T .. 16-padded are zero.
__global__ void pack_act_kernel(const bf16* src, int T, int K, bf16* dst) {
  const int Tp = (T + 15) & ~15;
  const size_t n = (size_t)Tp * K / 8;  // 16-byte chunks
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / (K / 8)), k = (int)(i % (K / 8)) * 8;
    const uint4 v = t < T ? *reinterpret_cast<const uint4*>(src + (size_t)t * K + k)
                          : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(dst + packed_off(t, k, K)) = v;
  }
}

// ---- host: tensor maps over the packed layout

// A packed [groups * 16][K] bf16 matrix seen as (128 8-byte elements of a
// 1 KB unit, groups, K / 32 K blocks); boxes of (128, box_groups, box_kb):
// box_kb K blocks of box_groups row groups, landing K block by K block as
// consecutive 1 KB units.
bool packed_map(CUtensorMap* m, const void* base, int K, int groups, int box_groups, int box_kb) {
  EncodeTiled enc = tma_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {128, (cuuint64_t)groups, (cuuint64_t)(K / 32)};
  const cuuint64_t strides[2] = {(cuuint64_t)(K / 32) * 1024, 1024};
  const cuuint32_t box[3] = {128, (cuuint32_t)box_groups, (cuuint32_t)box_kb};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_pack_act(const bf16* src, int T, int K, bf16* dst, cudaStream_t s) {
  if (K % 32 || T <= 0) return cudaErrorInvalidValue;
  pack_act_kernel<<<1216, 256, 0, s>>>(src, T, K, dst);
  return cudaGetLastError();
}

cudaError_t launch_argmax_index(const unsigned long long* best, int T, int32_t* idx,
                                cudaStream_t s) {
  argmax_index_kernel<<<(T + 255) / 256, 256, 0, s>>>(best, T, idx);
  return cudaGetLastError();
}

cudaError_t launch_gemm_rows(const GemmArgs& a, cudaStream_t s) {
  if (a.R % 16 || a.K % 32 || a.T <= 0) return cudaErrorInvalidValue;
  const bool swiglu = a.epi == GEMM_SWIGLU;
  if (((uintptr_t)a.W0 | (uintptr_t)a.act | (swiglu ? (uintptr_t)a.W1 : 0) |
       (a.epi == GEMM_RESID ? (uintptr_t)a.x : 0)) & 15)
    return cudaErrorInvalidValue;
  static int sms_of[kDeviceSlots] = {};
  const int dv0 = device_slot();
  int sms = dv0 >= 0 ? sms_of[dv0] : 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      sms = 1;
    if (dv0 >= 0) sms_of[dv0] = sms;
  }
  const int m_tiles = (a.R / 16 + kTcGroups - 1) / kTcGroups;
  const TcShape sh = tc_shape(a.T, swiglu, m_tiles, sms);
  // boxes no larger than the tensors; the bytes a stage receives
  CUtensorMap m0, m1, mx;
  const int groups = a.R / 16, tgroups = (a.T + 15) / 16;
  const int wbox = groups < kTcGroups ? groups : kTcGroups;
  const int xbox = tgroups < sh.NT / 16 ? tgroups : sh.NT / 16;
  // K blocks per box: a stage's worth (fewer when K is shorter); a matrix of
  // fewer than 8 row groups takes one box per K block, so that each K block
  // still starts 8 KB after the previous one
  const int kbox = sh.kbs < a.K / 32 ? sh.kbs : a.K / 32;
  const int wsplit = wbox < kTcGroups ? 1 : 0;
  if (!packed_map(&m0, a.W0, a.K, groups, wbox, wsplit ? 1 : kbox) ||
      !packed_map(&m1, swiglu ? a.W1 : a.W0, a.K, groups, wbox, wsplit ? 1 : kbox) ||
      !packed_map(&mx, a.act, a.K, tgroups, xbox, kbox))
    return cudaErrorInvalidValue;
  const int tx = kbox * ((swiglu ? 2 : 1) * wbox + xbox) * 1024;
  static size_t smem_set[kDeviceSlots] = {};
  const int dv = device_slot();
  if (dv < 0 || sh.smem > smem_set[dv]) {
    const cudaError_t e = cudaFuncSetAttribute(
        gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sh.smem);
    if (e != cudaSuccess) return e;
    if (dv >= 0) smem_set[dv] = sh.smem;
  }
  dim3 grid(sh.tiles, (groups + kTcGroups - 1) / kTcGroups);
  gemm_tc_kernel<<<grid, kTcThreads, sh.smem, s>>>(m0, m1, mx, a, sh.NT, sh.ncols, sh.stages,
                                                   sh.stage_bytes, tx, sh.nacc, sh.kbs, kbox,
                                                   wsplit);
  return cudaGetLastError();
}

}  // namespace ssd
