// Window-query attention of candidate-mask scoring on the 5th-generation
// tensor cores (SWIFT §4.1.2: every candidate layer set predicts the last N
// committed tokens; window row i of a candidate attends to the shared cache
// below the window and to its own candidate's window rows w <= i).
//
// CTA = (group of G = 128 / N candidates, head h): the group's G N query rows
// (compact rows of consecutive candidates) are one M = 128 tile.  Keys come
// in blocks of 128: the shared prefix [0, split) in ceil(split / 128) blocks,
// then one block holding the G candidates' own window keys (key column
// c N + w for candidate c).  Per block:
//   S = Q K^T            tcgen05 (M = 128, N = 128 keys, K = dh), S in
//                        tensor memory, double-buffered;
//   online softmax       eight warps, two threads per query row (TMEM lane),
//                        each over 64 of the block's keys: mask, row max
//                        (the pair's maxima exchanged in shared memory),
//                        2^x on the special-function unit, partial sums
//                        added in a fixed order (base 2);
//   O *= exp2(m - m')    in tensor memory, each thread of the pair over half
//                        of O's columns, and only in warps where some row's
//                        maximum grew (the factor is otherwise exactly 1);
//   P, V^T               bf16 into shared memory in the K-major 128-byte
//                        swizzle layout the MMA reads (V transposed by
//                        ldmatrix and stmatrix.trans);
//   O += P V             tcgen05 (M = 128, N = dh, K = 128 keys).
// Warp 8 issues the TMA copies (Q once; K and V blocks in a 2-stage ring,
// 128-byte swizzle, cache rows at or beyond split zero-filled; a stage is
// refilled once its block's P and V^T are written), warp 9 the
// MMAs (S of block j + 2 goes out as soon as block j's P is in).  Every wait
// is bounded; a wait that gives up flags the CTA, every role then runs out,
// the copies and MMAs in flight are waited for and the error word is set.
#include "kernels.cuh"
#include "tc_dev.cuh"

namespace ssd {
namespace {

using namespace tc;

constexpr int kAtKeys = 128;                    // keys per block
constexpr int kAtRegion = 128 * 128;            // [128 rows][64] bf16, 128-byte swizzle
constexpr int kOffQ = 0;                        // Q: 2 regions (dh halves)
constexpr int kOffK = 2 * kAtRegion;            // K: 2 stages x 2 regions (dh halves)
constexpr int kOffV = 6 * kAtRegion;            // V: 2 stages x 2 regions (dh halves)
constexpr int kOffP = 10 * kAtRegion;           // P: 2 regions (key halves)
constexpr int kOffVt = 12 * kAtRegion;          // V^T: 2 regions (key halves)
constexpr int kOffX = 14 * kAtRegion;           // exchange of the row pairs: [2][128] floats
constexpr int kOffBar = kOffX + 1024;           // barriers, TMEM slot, flag
constexpr int kAtThreads = 320;                 // warps 0-7 softmax, 8 copies, 9 MMAs
constexpr int kSoftThreads = 256;
constexpr int kAtPolls = 1 << 22;
constexpr uint32_t kColO = 256;                 // TMEM: S buffers [0, 256), O [256, 384)
constexpr uint32_t kAtCols = 512;

// Byte offset of (row, col) in a [rows][64] bf16 region, 128-byte swizzle
// (16-byte chunk index XOR row mod 8; 8-row atoms of 1024 bytes).
SSD_DI uint32_t sw128_off(int row, int col) {
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((((col >> 3) ^ row) & 7) << 4) +
                    (col & 7) * 2);
}

// Four 8x8 b16 tiles: lanes 8t .. 8t + 7 give the row addresses of tile t.
SSD_DI void ldsm_x4(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}
// The same four tiles stored transposed (row addresses of the destination).
SSD_DI void stsm_x4_t(uint32_t saddr, const uint32_t (&r)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(saddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}

SSD_DI bool flagged(const int* f) { return *reinterpret_cast<const volatile int*>(f) != 0; }
// 2^x by the special-function unit (ex2.approx: relative error about 2^-22;
// the probabilities are rounded to bf16 before the PV MMA).
SSD_DI float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Barrier of the eight softmax warps.
SSD_DI void soft_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__global__ void __launch_bounds__(kAtThreads, 1)
    score_attn_tc_kernel(const __grid_constant__ CUtensorMap mQ,
                         const __grid_constant__ CUtensorMap mK,
                         const __grid_constant__ CUtensorMap mV,
                         const __grid_constant__ CUtensorMap mWK,
                         const __grid_constant__ CUtensorMap mWV, ScoreAttnArgs a, int n_active,
                         int cpg, int qrows, int kbox) {
  extern __shared__ unsigned char sm_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* qfull = bars;
  uint64_t* full = bars + 1;    // [2] K and V block landed
  uint64_t* sfull = bars + 5;   // [2] S buffer written
  uint64_t* pready = bars + 7;  // P, V^T written and O rescaled (256 arrivals)
  uint64_t* pvdone = bars + 8;  // PV completed
  uint64_t* mdone = bars + 9;   // every MMA of the CTA completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 10);
  int* fail = reinterpret_cast<int*>(tslot + 1);
  int* last_blk = fail + 1;     // [2] last block copied into each stage, -1 none

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  const int N = a.N, kvh = h / (a.H / a.Hkv);
  const int c_first = blockIdx.x * cpg;
  const int ncand = min(cpg, n_active - c_first);
  const int nbp = (a.split + kAtKeys - 1) / kAtKeys;  // prefix blocks
  const int nb = nbp + 1;                             // and the window block

  if (tid == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sfull[s], 1);
      last_blk[s] = -1;
    }
    mbar_init(pready, kSoftThreads);
    mbar_init(pvdone, 1);
    mbar_init(mdone, 1);
    *fail = 0;
    fence_mbar_init();
  }
  // Q, K and V buffers start at zero: rows a block does not fill (absent
  // candidates, query rows beyond the tensor) must hold finite values, since
  // P = 0 meets them in the MMA and 0 x NaN is NaN
  for (int e = tid; e < 10 * kAtRegion / 16; e += kAtThreads)
    reinterpret_cast<uint4*>(sm + kOffQ)[e] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 0) tmem_alloc(tslot, kAtCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 8) {
    // ---- copies
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&mQ) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&mK) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&mV) : "memory");
      mbar_arrive_expect_tx(qfull, 2u * 128u * (uint32_t)qrows);
      tma_load_3d(sm + kOffQ, &mQ, 0, h, c_first * N, qfull);
      tma_load_3d(sm + kOffQ + kAtRegion, &mQ, 64, h, c_first * N, qfull);
      for (int j = 0; j < nb; ++j) {
        const int st = j & 1;
        // the stage's previous block (j - 2) is consumed once its P and V^T
        // are written: S has read its K, the transposition its V
        if (j >= 2 && !mbar_wait_n(pready, (uint32_t)(j & 1), kAtPolls)) {
          atomicExch(fail, 1);
          break;
        }
        if (flagged(fail)) break;
        unsigned char* K = sm + kOffK + st * 2 * kAtRegion;
        unsigned char* V = sm + kOffV + st * 2 * kAtRegion;
        reinterpret_cast<volatile int*>(last_blk)[st] = j;
        if (j < nbp) {
          mbar_arrive_expect_tx(&full[st], 4u * 128u * (uint32_t)kbox);
          for (int hf = 0; hf < 2; ++hf) {
            tma_load_3d(K + hf * kAtRegion, &mK, hf * 64, j * kAtKeys, kvh, &full[st]);
            tma_load_3d(V + hf * kAtRegion, &mV, hf * 64, j * kAtKeys, kvh, &full[st]);
          }
        } else {
          mbar_arrive_expect_tx(&full[st], 4u * 128u * (uint32_t)(ncand * N));
          for (int c = 0; c < ncand; ++c) {
            const int cand = __ldg(a.cand + c_first + c);
            for (int hf = 0; hf < 2; ++hf) {
              tma_load_3d(K + hf * kAtRegion + c * N * 128, &mWK, hf * 64, kvh, cand * N, &full[st]);
              tma_load_3d(V + hf * kAtRegion + c * N * 128, &mWV, hf * 64, kvh, cand * N, &full[st]);
            }
          }
        }
      }
    }
  } else if (warp == 9) {
    // ---- MMAs
    if (lane == 0) {
      const uint32_t id = idesc_bf16(128, 128);
      const uint32_t qa = smem_addr(sm + kOffQ);
      bool ok = mbar_wait_n(qfull, 0u, kAtPolls);
      auto issue_s = [&](int j) -> bool {  // S of block j into S buffer j & 1
        const int st = j & 1;
        if (!mbar_wait_n(&full[st], (uint32_t)((j >> 1) & 1), kAtPolls)) return false;
        tc_fence_after();
        const uint32_t ka = smem_addr(sm + kOffK + st * 2 * kAtRegion);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t rg = (uint32_t)(ks >> 2) * kAtRegion;
          const uint64_t da = sw128_desc(qa + rg) + 2 * (ks & 3);
          const uint64_t db = sw128_desc(ka + rg) + 2 * (ks & 3);
          mma_bf16_tc(tmem + (uint32_t)(st * 128), da, db, id, ks > 0 ? 1u : 0u);
        }
        mma_commit(&sfull[st]);
        return true;
      };
      ok = ok && issue_s(0);
      ok = ok && (nb < 2 || issue_s(1));
      const uint32_t pa = smem_addr(sm + kOffP), va = smem_addr(sm + kOffVt);
      for (int j = 0; ok && j < nb; ++j) {
        if (!mbar_wait_n(pready, (uint32_t)(j & 1), kAtPolls) || flagged(fail)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t rg = (uint32_t)(ks >> 2) * kAtRegion;
          const uint64_t da = sw128_desc(pa + rg) + 2 * (ks & 3);
          const uint64_t db = sw128_desc(va + rg) + 2 * (ks & 3);
          mma_bf16_tc(tmem + kColO, da, db, id, (j > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(pvdone);
        if (j + 2 < nb) ok = issue_s(j + 2);
      }
      if (!ok) atomicExch(fail, 1);
      // every MMA issued has completed before the memory is released
      mma_commit(mdone);
      mbar_wait_n(mdone, 0u, kAtPolls);
    }
  } else {
    // ---- softmax, rescale, P and V^T, epilogue: query row r, key half hh.
    // Every block runs the same sequence of barriers in all 256 threads; a
    // wait that gives up (or a CTA already flagged) only skips the work that
    // needed it, so no thread is ever left at a barrier the others skip.
    const int r = tid & 127, hh = tid >> 7;
    const int c = r / N, i = r - c * N;
    const bool rvalid = c < ncand;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    float* xch = reinterpret_cast<float*>(sm + kOffX);  // [2][128]
    const float scale = a.scale_log2;
    float m = -INFINITY, l = 0.f;                      // l: this thread's half of the sum
    // bounded wait, warp-uniform result, nothing waited for once flagged
    auto wait_w = [&](uint64_t* bar, uint32_t parity) -> bool {
      bool okw = !flagged(fail) && mbar_wait_n(bar, parity, kAtPolls);
      okw = __all_sync(0xffffffffu, okw);
      if (!okw && lane == 0) atomicExch(fail, 1);
      return okw;
    };
    for (int j = 0; j < nb; ++j) {
      const int st = j & 1;
      const uint32_t par = (uint32_t)((j >> 1) & 1);
      uint32_t sr[2][32];
      if (wait_w(&sfull[st], par)) {
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q)
          tmem_ld32_nw(trow + (uint32_t)(st * 128 + hh * 64 + q * 32), sr[q]);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 2; ++q) tmem_pin32(sr[q]);
      } else {
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int e = 0; e < 32; ++e) sr[q][e] = 0u;
      }
      // mask (partial prefix block, window block: masked scores -inf); this
      // half's maximum in four independent chains
      const int kb = j * kAtKeys + hh * 64;             // first key of this half
      const bool full_pre = j < nbp && kb + 64 <= a.split;
      float bmx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float v = __uint_as_float(sr[q][e]);
          if (!full_pre) {
            const int k = hh * 64 + q * 32 + e;
            bool valid;
            if (j < nbp) {
              valid = kb + q * 32 + e < a.split;
            } else {
              const int cc = k / N, w = k - cc * N;
              valid = rvalid && cc == c && w <= i;
            }
            if (!valid) v = -INFINITY;
          }
          sr[q][e] = __float_as_uint(v);
          bmx[e & 3] = fmaxf(bmx[e & 3], v);
        }
      float bm = fmaxf(fmaxf(bmx[0], bmx[1]), fmaxf(bmx[2], bmx[3])) * scale;
      // the row's block maximum over both halves (scaled, base 2)
      xch[hh * 128 + r] = bm;
      soft_sync();
      bm = fmaxf(bm, xch[(hh ^ 1) * 128 + r]);
      soft_sync();  // the exchange slots are free for the next block
      const float mn = fmaxf(m, bm);
      const float corr = (m == -INFINITY || mn == -INFINITY) ? 1.f : ex2(m - mn);
      // p = 2^(s scale - m'), masked keys 0; four partial sums, added in a
      // fixed order
      const float nmn = mn == -INFINITY ? 0.f : -mn;
      float lsx[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[2][16];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float s0 = __uint_as_float(sr[q][e]), s1 = __uint_as_float(sr[q][e + 1]);
          const float p0 = ex2(fmaf(s0, scale, nmn));
          const float p1 = ex2(fmaf(s1, scale, nmn));
          lsx[(e >> 1) & 3] += p0 + p1;
          pk[q][e >> 1] = pack_bf16x2(p0, p1);
        }
      const float ls = (lsx[0] + lsx[1]) + (lsx[2] + lsx[3]);
      l = l * corr + ls;
      m = mn;
      // the previous block's PV has completed: O, P and V^T may be touched
      if (j > 0 && wait_w(pvdone, (uint32_t)((j - 1) & 1))) {
        tc_fence_after();
        if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t o[32];
            const uint32_t col = kColO + (uint32_t)(hh * 64 + q * 32);
            tmem_ld32_nw(trow + col, o);
            tmem_wait_ld();
            tmem_pin32(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st32(trow + col, o);
          }
          tmem_wait_st();
        }
      }
      // P row r, keys of this half: 8 chunks of 8
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        const uint4 v = make_uint4(pk[q8 >> 2][(q8 & 3) * 4], pk[q8 >> 2][(q8 & 3) * 4 + 1],
                                   pk[q8 >> 2][(q8 & 3) * 4 + 2], pk[q8 >> 2][(q8 & 3) * 4 + 3]);
        *reinterpret_cast<uint4*>(sm + kOffP + hh * kAtRegion + sw128_off(r, q8 * 8)) = v;
      }
      // V^T: warp w takes dh rows 16w .. 16w + 15 of the block's V: 8x8 tiles
      // read with ldmatrix (rows = keys) and written back transposed with
      // stmatrix.trans (rows = dh)
      if (wait_w(&full[st], par)) {
        const unsigned char* Vb = sm + kOffV + st * 2 * kAtRegion;
        const int tq = lane >> 3, tr8 = lane & 7;      // tile of this lane's row address
        const int d0 = warp * 16 + (tq & 1) * 8;        // dh of the tile
#pragma unroll 4
        for (int kt = 0; kt < 16; kt += 2) {
          const int k0 = (kt + (tq >> 1)) * 8;          // keys of the tile
          uint32_t t4[4];
          ldsm_x4(t4, smem_addr(Vb + (d0 >> 6) * kAtRegion + sw128_off(k0 + tr8, d0 & 63)));
          stsm_x4_t(smem_addr(sm + kOffVt + (k0 >> 6) * kAtRegion + sw128_off(d0 + tr8, k0 & 63)), t4);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_cta(pready);
    }
    // epilogue: O / l (the two halves' sums added), bf16; each thread of the
    // pair writes half of the row's columns
    const bool ok = wait_w(pvdone, (uint32_t)((nb - 1) & 1));
    xch[hh * 128 + r] = l;
    soft_sync();
    const float lt = hh == 0 ? l + xch[128 + r] : xch[r] + l;
    if (ok) {
      tc_fence_after();
      const float inv = lt > 0.f ? 1.0f / lt : 0.f;
      const int HD = a.H * 128;
      const int t = (c_first + c) * N + i;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t o[32];
        const int cbase = hh * 64 + q * 32;
        tmem_ld32_nw(trow + kColO + (uint32_t)cbase, o);
        tmem_wait_ld();
        tmem_pin32(o);
        if (rvalid) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int d = h * 128 + cbase + u * 8;
            const uint4 v = make_uint4(
                pack_bf16x2(__uint_as_float(o[u * 8 + 0]) * inv, __uint_as_float(o[u * 8 + 1]) * inv),
                pack_bf16x2(__uint_as_float(o[u * 8 + 2]) * inv, __uint_as_float(o[u * 8 + 3]) * inv),
                pack_bf16x2(__uint_as_float(o[u * 8 + 4]) * inv, __uint_as_float(o[u * 8 + 5]) * inv),
                pack_bf16x2(__uint_as_float(o[u * 8 + 6]) * inv, __uint_as_float(o[u * 8 + 7]) * inv));
            const size_t off = a.out_packed ? packed_off(t, d, HD) : (size_t)t * HD + d;
            *reinterpret_cast<uint4*>(a.out + off) = v;
          }
        }
      }
    }
  }
  // teardown: the copies still in flight land before the memory is released
  if (warp == 8 && lane == 0) {
    for (int s = 0; s < 2; ++s) {
      const int j = reinterpret_cast<volatile int*>(last_blk)[s];
      if (j >= 0) mbar_wait_n(&full[s], (uint32_t)((j >> 1) & 1), kAtPolls);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && flagged(fail) && a.err) atomicExch(a.err, 7);
  if (warp == 0) tmem_dealloc(tmem, kAtCols);
}

}  // namespace

// The tensor-core path takes dh 128 and windows of N <= 128 rows with N a
// multiple of 8 (a candidate's window keys start on a 1024-byte swizzle atom).
bool score_attn_tc_ok(const ScoreAttnArgs& a) {
  return a.dh == 128 && a.N >= 8 && a.N <= 128 && a.N % 8 == 0 && a.w_rows >= a.N &&
         a.split >= 1 && tma_encoder() != nullptr;
}

cudaError_t launch_score_attn_tc(const ScoreAttnArgs& a, int n_active, cudaStream_t s) {
  if (!score_attn_tc_ok(a)) return cudaErrorInvalidValue;
  if (((uintptr_t)a.q | (uintptr_t)a.kc | (uintptr_t)a.vc | (uintptr_t)a.sk | (uintptr_t)a.sv |
       (uintptr_t)a.out) & 15)
    return cudaErrorInvalidValue;
  EncodeTiled enc = tma_encoder();
  const int cpg = 128 / a.N;
  const int rows_q = n_active * a.N;
  const int qrows = rows_q < 128 ? rows_q : 128;
  const int kbox = a.split < 128 ? a.split : 128;
  auto map3 = [&](CUtensorMap* m, const void* base, cuuint64_t d1, cuuint64_t d2, cuuint64_t s1,
                  cuuint64_t s2, cuuint32_t b1, cuuint32_t b2) {
    const cuuint64_t dims[3] = {128, d1, d2};
    const cuuint64_t strides[2] = {s1, s2};
    const cuuint32_t box[3] = {64, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
  };
  const cuuint64_t row = 128 * sizeof(bf16);
  CUtensorMap mQ, mK, mV, mWK, mWV;
  // q [rows][H][128]; cache [Hkv][max_seq][128] seen as keys < split;
  // window [w_rows][Hkv][128]
  if (!map3(&mQ, a.q, a.H, rows_q, row, row * a.H, 1, qrows) ||
      !map3(&mK, a.kc, a.split, a.Hkv, row, row * a.max_seq, kbox, 1) ||
      !map3(&mV, a.vc, a.split, a.Hkv, row, row * a.max_seq, kbox, 1) ||
      !map3(&mWK, a.sk, a.Hkv, a.w_rows, row, row * a.Hkv, 1, a.N) ||
      !map3(&mWV, a.sv, a.Hkv, a.w_rows, row, row * a.Hkv, 1, a.N))
    return cudaErrorInvalidValue;
  const size_t smem = (size_t)kOffBar + 128 + 1024;
  static bool ready[kDeviceSlots] = {};
  const int dv = device_slot();
  if (dv < 0 || !ready[dv]) {
    const cudaError_t e = cudaFuncSetAttribute(
        score_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dv >= 0) ready[dv] = true;
  }
  dim3 grid((n_active + cpg - 1) / cpg, a.H);
  score_attn_tc_kernel<<<grid, kAtThreads, smem, s>>>(mQ, mK, mV, mWK, mWV, a, n_active, cpg,
                                                      qrows, kbox);
  return cudaGetLastError();
}

}  // namespace ssd
