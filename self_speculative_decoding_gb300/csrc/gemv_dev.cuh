// Device side of the small-M weight-streaming GEMV: the packed-unit
// partition, the producer / consumer / epilogue warp roles, and the
// epilogues of the GEMV kernel (gemv.cu).
//
// Loads of data written by the preceding kernel or by other CTAs of this one
// (the residual stream, its sum-of-squares partials, activations, split-group
// partials) go through L2 (ld.global.cg).
#pragma once

#include "kernels.cuh"

namespace ssd {
namespace gemv {

#ifndef SSD_GEMV_CONSUMERS
#define SSD_GEMV_CONSUMERS 8
#endif
#ifndef SSD_GEMV_CPS
#define SSD_GEMV_CPS 2
#endif
#ifndef SSD_GEMV_CTAS
#define SSD_GEMV_CTAS (152 * SSD_GEMV_CPS)
#endif
#ifndef SSD_GEMV_STAGE_KB
#define SSD_GEMV_STAGE_KB 44
#endif
constexpr int kConsumers = SSD_GEMV_CONSUMERS;   // consumer warps
constexpr int kProducer = kConsumers;            // warp that issues the bulk copies
constexpr int kEpilogue = kConsumers + 1;        // warp that finishes row groups
constexpr int kThreads = (kConsumers + 2) * 32;
constexpr int kCtasPerSm = SSD_GEMV_CPS;         // resident CTAs per SM
#ifndef SSD_GEMV_CHUNK
#define SSD_GEMV_CHUNK 16
#endif
#ifndef SSD_GEMV_SLOTS
#define SSD_GEMV_SLOTS 3
#endif
constexpr int kGridCtas = SSD_GEMV_CTAS;         // kCtasPerSm resident CTAs x 152 SMs
constexpr int kChunk = SSD_GEMV_CHUNK;           // units per ring slot (<= kConsumers * k)
constexpr int kSlots = SSD_GEMV_SLOTS;           // ring depth
constexpr int kUPW = (kChunk + kConsumers - 1) / kConsumers;  // units per warp per chunk
constexpr int kUnitBytes = 1024;
constexpr int kSlotBytes = kChunk * kUnitBytes;
constexpr int kRingBytes = kSlots * kSlotBytes;
// Activations (the B operand, bf16 and already normalised for the norm-fused
// input) are staged once per CTA when M rows of K fit in this budget; this
// covers every single-token pass of the 7B and 13B shapes.
constexpr int kStageBytes = SSD_GEMV_STAGE_KB * 1024;
constexpr int kPad = 8;                          // bf16 row padding of the stage

// Partition of a GEMV's T units over C CTAs: CTA b owns the contiguous
// granules [b*Tg/C, (b+1)*Tg/C), a granule being G units.  Where the matrix
// has enough row groups, a granule is a whole row group (a whole gate/up
// pair for SwiGLU) and C is chosen so that every CTA gets the same number of
// granules: no row group is then split across CTAs and every epilogue runs
// from shared memory.  Matrices with too few row groups for that use single
// units (G = 1, C = kGridCtas) and combine split groups across CTAs.
constexpr int kMinWholeCtas = 200;

struct Part {
  int T;       // units = NRG * KB
  int Tg;      // granules = T / G
  int NRG;     // (virtual) 16-row groups
  int KB;      // 32-wide K blocks
  int G;       // units per granule
  int C;       // CTAs with work = min(kGridCtas, Tg)
  int segmax;  // stride of the partial buffer per row group
};

// All partition arithmetic is 32-bit unsigned: launch_gemv refuses shapes
// with T * (kGridCtas + 1) >= 2^32 (far beyond any decoder projection).
__host__ __device__ inline int unit_begin(const Part& p, int b) {
  return (int)((unsigned)b * (unsigned)p.Tg / (unsigned)p.C) * p.G;
}
// first CTA whose range contains unit a / last CTA whose range meets [.., b)
__host__ __device__ inline int cta_first(const Part& p, int a) {
  const unsigned ga = (unsigned)(a / p.G);
  return (int)(((ga + 1u) * (unsigned)p.C + (unsigned)p.Tg - 1u) / (unsigned)p.Tg) - 1;
}
__host__ __device__ inline int cta_last(const Part& p, int b) {
  const unsigned gb = (unsigned)((b + p.G - 1) / p.G);
  return (int)((gb * (unsigned)p.C + (unsigned)p.Tg - 1u) / (unsigned)p.Tg) - 1;
}
__host__ __device__ inline int nseg(const Part& p, int vr) {
  return cta_last(p, (vr + 1) * p.KB) - cta_first(p, vr * p.KB) + 1;
}
// row group vr lies entirely in CTA b's range
__host__ __device__ inline bool owns(const Part& p, int vr, int b) {
  return cta_first(p, vr * p.KB) == b && cta_last(p, (vr + 1) * p.KB) == b;
}

__host__ __device__ inline Part make_part(int R, int K, int epi) {
  Part p;
  p.NRG = (epi == EPI_SWIGLU ? 2 : 1) * (R / 16);
  p.KB = K / 32;
  p.T = p.NRG * p.KB;
  const int gu = (epi == EPI_SWIGLU ? 2 : 1) * p.KB;  // units of a whole group / pair
  const int ng = p.T / gu;
  const int per = (ng + kGridCtas - 1) / kGridCtas;   // granules per CTA
  const int cw = (ng + per - 1) / per;                // CTAs with equal shares
  if (epi == EPI_LMHEAD || cw >= kMinWholeCtas) {
    p.G = gu;
    p.Tg = ng;
    p.C = cw;
  } else {
    p.G = 1;
    p.Tg = p.T;
    p.C = p.T < kGridCtas ? p.T : kGridCtas;
  }
  p.segmax = (p.C + p.NRG - 1) / p.NRG + 1;
  return p;
}

// Shapes whose partition arithmetic fits 32 bits.
inline bool part_fits(int R, int K) {
  const unsigned long long T = 2ull * (unsigned long long)(R / 16) * (unsigned long long)(K / 32);
  return T * (unsigned long long)(kGridCtas + 1) < (1ull << 32);
}

// Unit (vr, kb) in the packed stream of its matrix.
template <int EPI>
SSD_DI const bf16* unit_src(const LinearArgs& a, const Part& p, int vr, int kb) {
  if (EPI == EPI_SWIGLU) {
    const bf16* W = (vr & 1) ? a.W1 : a.W0;
    return W + ((size_t)(vr >> 1) * p.KB + kb) * (kUnitBytes / 2);
  }
  return a.W0 + ((size_t)vr * p.KB + kb) * (kUnitBytes / 2);
}

// Raw B operand (8 consecutive K of one token): loaded one chunk ahead so
// that the global-memory latency is off the critical path.  For the
// norm-fused input the RMSNorm is applied when the operand is used.
template <int IN>
struct BRaw {
  uint4 v;
};
template <>
struct BRaw<IN_NORM> {
  float4 x0, x1, g0, g1;
};

template <int IN>
SSD_DI void b_issue(BRaw<IN>& r, const LinearArgs& a, int t, int off, bool valid) {
  if (IN == IN_BF16) {
    auto& q = reinterpret_cast<BRaw<IN_BF16>&>(r);
    q.v = valid ? __ldcg(reinterpret_cast<const uint4*>(a.act + (size_t)t * a.K + off))
                : make_uint4(0u, 0u, 0u, 0u);
  } else {
    auto& q = reinterpret_cast<BRaw<IN_NORM>&>(r);
    if (valid) {
      const float4* xp = reinterpret_cast<const float4*>(a.x + (size_t)t * a.K + off);
      const float4* gp = reinterpret_cast<const float4*>(a.gain + off);
      q.x0 = __ldcg(xp); q.x1 = __ldcg(xp + 1); q.g0 = gp[0]; q.g1 = gp[1];
    } else {
      q.x0 = q.x1 = q.g0 = q.g1 = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

template <int IN>
SSD_DI uint4 b_finish(const BRaw<IN>& r, float rs) {
  if (IN == IN_BF16) {
    return reinterpret_cast<const BRaw<IN_BF16>&>(r).v;
  } else {
    const auto& q = reinterpret_cast<const BRaw<IN_NORM>&>(r);
    return make_uint4(pack_bf16x2(q.x0.x * rs * q.g0.x, q.x0.y * rs * q.g0.y),
                      pack_bf16x2(q.x0.z * rs * q.g0.z, q.x0.w * rs * q.g0.w),
                      pack_bf16x2(q.x1.x * rs * q.g1.x, q.x1.y * rs * q.g1.y),
                      pack_bf16x2(q.x1.z * rs * q.g1.z, q.x1.w * rs * q.g1.w));
  }
}

SSD_DI void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory"); }

SSD_DI void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// ---------------------------------------------------------------- reductions

// Top-2 merge under the (value desc, index asc) total order.
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

// LM-head summary of a set of vocabulary rows for one token: max z and its
// id, second z and its id, sum exp(z - max), sum exp(z/T - max/T), best
// Gumbel score and its id.
struct LmRec {
  float v1, v2, se, set, gv;
  int i1, i2, gi;
};

SSD_DI void lm_store(float* p, const LmRec& r) {
  reinterpret_cast<float4*>(p)[0] =
      make_float4(r.v1, __int_as_float(r.i1), r.v2, __int_as_float(r.i2));
  reinterpret_cast<float4*>(p)[1] = make_float4(r.se, r.set, r.gv, __int_as_float(r.gi));
}

SSD_DI LmRec lm_load(const float* p) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
  LmRec r;
  r.v1 = a.x; r.i1 = __float_as_int(a.y); r.v2 = a.z; r.i2 = __float_as_int(a.w);
  r.se = b.x; r.set = b.y; r.gv = b.z; r.gi = __float_as_int(b.w);
  return r;
}

SSD_DI LmRec lm_empty() {
  LmRec r;
  r.v1 = r.v2 = r.gv = -INFINITY;
  r.i1 = r.i2 = r.gi = 0x7fffffff;
  r.se = r.set = 0.f;
  return r;
}

// Merge one record per lane (a butterfly, identical in every lane); the sums
// are rescaled to the merged maximum before being added.
SSD_DI LmRec lm_merge_warp(LmRec r, float T) {
  float v1 = r.v1, v2 = r.v2, gv = r.gv;
  int i1 = r.i1, i2 = r.i2, gi = r.gi;
  top2_warp(v1, i1, v2, i2);
  argmax_warp(gv, gi);
  const float mx = v1;
  float s = r.v1 == -INFINITY ? 0.f : r.se * expf(r.v1 - mx);
  float st = 0.f;
  if (T > 0.f) st = r.v1 == -INFINITY ? 0.f : r.set * expf(r.v1 / T - mx / T);
  s = sum_warp(s);
  st = sum_warp(st);
  LmRec o;
  o.v1 = v1; o.i1 = i1; o.v2 = v2; o.i2 = i2; o.gv = gv; o.gi = gi; o.se = s; o.set = st;
  return o;
}

// ---------------------------------------------------------------- epilogues

// Residual entries lane + 32 i of a row group (EPI_RESID), loaded ahead of
// the group's completion so that their latency is off the tail.
struct XPre {
  float v[kMaxRows * 16 / 32];
};

template <int EPI>
SSD_DI void xres_prefetch(const LinearArgs& a, int vr, int M, int lane, XPre& xp) {
  if (EPI == EPI_RESID) {
#pragma unroll
    for (int i = 0; i < kMaxRows * 16 / 32; ++i) {
      const int e = lane + 32 * i;
      if (e < 16 * M) {
        const int row = e / M, tok = e % M;
        xp.v[i] = __ldcg(a.xres + (size_t)tok * a.R + vr * 16 + row);
      }
    }
  }
}

// Runs in one warp once row group vr (or the gate/up pair containing it) is
// complete; ep[h][row][tok] holds the finished sums.  Projections only (the
// LM head goes through lm_group / lm_finish).
template <int EPI>
SSD_DI void epilogue(const LinearArgs& a, const Part& p, int vr, float (*ep)[16][17], int M,
                     int lane, const XPre& xp) {
  if (EPI == EPI_STORE) {
    const int row0 = vr * 16;
    for (int e = lane; e < 16 * M; e += 32) {
      const int row = e / M, tok = e % M;
      a.y[(size_t)tok * a.R + row0 + row] = ep[0][row][tok];
    }
  } else if (EPI == EPI_RESID) {
    const int row0 = vr * 16;
#pragma unroll
    for (int i = 0; i < kMaxRows * 16 / 32; ++i) {
      const int e = lane + 32 * i;
      if (e < 16 * M) {
        const int row = e / M, tok = e % M;
        const float xn = xp.v[i] + ep[0][row][tok];
        a.xres[(size_t)tok * a.R + row0 + row] = xn;
        ep[0][row][tok] = xn;
      }
    }
    __syncwarp();
    if (lane < M) {
      float s = 0.f;
      for (int row = 0; row < 16; ++row) s += ep[0][row][lane] * ep[0][row][lane];
      a.ss_out[(size_t)lane * (a.R / kSsGroup) + vr] = s;
    }
  } else if (EPI == EPI_SWIGLU) {
    const int row0 = (vr >> 1) * 16;
    for (int e = lane; e < 16 * M; e += 32) {
      const int row = e / M, tok = e % M;
      const float gt = ep[0][row][tok];
      const float up = ep[1][row][tok];
      const float sl = gt / (1.0f + expf(-gt));
      a.u[(size_t)tok * a.R + row0 + row] = __float2bfloat16_rn(sl * up);
    }
  }
}

// Folds record q into r: top-2 and the Gumbel argmax under the total order,
// the exponential sums rescaled to the larger maximum.
SSD_DI void lm_combine(LmRec& r, const LmRec& q, float T) {
  if (q.v1 == -INFINITY) return;
  const float mx = fmaxf(r.v1, q.v1);
  const float se = (r.v1 == -INFINITY ? 0.f : r.se * expf(r.v1 - mx)) + q.se * expf(q.v1 - mx);
  float set = 0.f;
  if (T > 0.f)
    set = (r.v1 == -INFINITY ? 0.f : r.set * expf(r.v1 / T - mx / T)) +
          q.set * expf(q.v1 / T - mx / T);
  top2_insert(q.v1, q.i1, r.v1, r.i1, r.v2, r.i2);
  top2_insert(q.v2, q.i2, r.v1, r.i1, r.v2, r.i2);
  if (better(q.gv, q.gi, r.gv, r.gi)) { r.gv = q.gv; r.gi = q.gi; }
  r.se = se;
  r.set = set;
}

// LM head, one finished row group (16 vocabulary rows in ep[0]): optional
// logits, then lane tok < M folds the group's rows, in row order, into its
// running record `run` (the CTA's vocabulary range so far).
// LM head, token tok's record of one finished row group (vocabulary rows
// row0 .. row0 + 15, logit of row r at z[r * zstride]), rows in order.
SSD_DI LmRec lm_group_rec(const LinearArgs& a, int row0, const float* z, int zstride, int tok,
                          int round, int pos0) {
  const float T = a.temperature;
  LmRec r = lm_empty();
  const bool draw = T > 0.f && a.sample;
  for (int rb = 0; rb < 16; rb += 4) {
    float g[4] = {0.f, 0.f, 0.f, 0.f};
    if (draw) gumbel4(a.seed, (row0 + rb) >> 2, pos0 + tok + 1, round, a.sample_stream, g);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int row = rb + w;
      const float zz = z[row * zstride];
      top2_insert(zz, row0 + row, r.v1, r.i1, r.v2, r.i2);
      if (draw) {
        const float sc = zz / T + g[w];
        if (better(sc, row0 + row, r.gv, r.gi)) { r.gv = sc; r.gi = row0 + row; }
      }
    }
  }
  for (int row = 0; row < 16; ++row) {
    const float zz = z[row * zstride];
    r.se += expf(zz - r.v1);
    if (T > 0.f) r.set += expf(zz / T - r.v1 / T);
  }
  return r;
}

SSD_DI void lm_group(const LinearArgs& a, int vr, float (*ep)[16][17], int M, int lane, int slot,
                     int round, int pos0, LmRec& run) {
  const int row0 = vr * 16;
  if (a.logits) {
    for (int e = lane; e < 16 * M; e += 32) {
      const int row = e / M, tok = e % M;
      a.logits[(size_t)(slot + tok) * a.R + row0 + row] = ep[0][row][tok];
    }
  }
  if (lane < M) lm_combine(run, lm_group_rec(a, row0, &ep[0][0][lane], 17, lane, round, pos0), a.temperature);
}

// LM head, end of CTA b's range: publish the CTA's records (one per token,
// stored [tok][b]).  Returns (in every lane) whether this CTA published
// last, i.e. every CTA's records are in.
SSD_DI bool lm_publish(const LinearArgs& a, const Part& p, int b, int M, int lane,
                       const LmRec& run) {
  if (lane < M) lm_store(a.rec + ((size_t)lane * p.C + b) * 8, run);
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(a.counter, 1u) == (unsigned)(p.C - 1);
  return __shfl_sync(0xffffffffu, last, 0) != 0;
}

// LM head, token tok's row summary from all C records (one warp): the
// records go to `stage` (C x 32 bytes of shared memory, this warp's own)
// with 16-byte asynchronous copies, all in flight at once; lane l folds
// CTAs l, l+32, ... in order, then a butterfly.  The order depends on C
// alone, so a token's summary does not depend on how many tokens the pass
// carries or on which warp folds it.
SSD_DI void lm_fold(const LinearArgs& a, const Part& p, int tok, int lane, int slot, float* stage) {
  const float T = a.temperature;
  const float4* src = reinterpret_cast<const float4*>(a.rec + (size_t)tok * p.C * 8);
  float4* dst = reinterpret_cast<float4*>(stage);
  for (int i = lane; i < 2 * p.C; i += 32) cp_async16(dst + i, src + i);
  cp_async_wait_all();
  __syncwarp();
  LmRec r = lm_empty();
  for (int c = lane; c < p.C; c += 32) {
    const float4 x0 = dst[2 * c], x1 = dst[2 * c + 1];
    LmRec q;
    q.v1 = x0.x; q.i1 = __float_as_int(x0.y); q.v2 = x0.z; q.i2 = __float_as_int(x0.w);
    q.se = x1.x; q.set = x1.y; q.gv = x1.z; q.gi = __float_as_int(x1.w);
    lm_combine(r, q, T);
  }
  r = lm_merge_warp(r, T);
  if (lane == 0) {
    RowStats rs;
    rs.top1 = r.i1;
    rs.top2 = r.i2;
    rs.sample = T > 0.f && a.sample ? r.gi : r.i1;
    rs.pad = 0;
    rs.z1 = r.v1;
    rs.z2 = r.v2;
    rs.lse = r.v1 + logf(r.se);
    rs.conf = expf(r.v1 - rs.lse);
    rs.lse_t = T > 0.f ? r.v1 / T + logf(r.set) : rs.lse;
    rs.pad2[0] = rs.pad2[1] = rs.pad2[2] = 0.f;
    a.stats[slot + tok] = rs;
  }
  __syncwarp();
}

// ---------------------------------------------------------------- kernel

struct __align__(16) GemvSmem {
  unsigned char ring[kRingBytes];
  float red[2][kConsumers][16][16];  // per-warp partials, double-buffered per row group
  float ep[2][16][17];               // epilogue operands
  float rstd[kMaxRows];
  uint64_t full[kSlots + kStageBytes / kSlotBytes];   // slot filled by the bulk copy
  uint64_t empty[kSlots + kStageBytes / kSlotBytes];  // slot consumed by all consumer warps
  uint64_t rfull[2];                 // partial buffer written by all consumer warps
  uint64_t rempty[2];                // partial buffer read by the epilogue warp
  uint64_t foldbar;                  // LM head: the epilogue warp knows whether this CTA folds
  uint64_t lastbar;                  // LM head: the consumers' records of the last batch are in
  int fold_last;
  __align__(16) bf16 stage[kStageBytes / 2];
};
// LM head fold: each of the kConsumers + 1 folding warps stages C records
// (at most kGridCtas x 32 bytes) in its own part of the ring and the stage.
constexpr int kFoldBytes = 10240;
static_assert(kGridCtas * 32 <= kFoldBytes, "a warp's fold staging holds every CTA's record");
constexpr int kFoldInRing = kRingBytes / kFoldBytes;    // folding warps staged in the ring
constexpr int kFoldInStage = kStageBytes / kFoldBytes;  // then in the stage, then in red
static_assert(kFoldInRing + kFoldInStage + (int)(sizeof(float) * 2 * kConsumers * 256 >= kFoldBytes) >=
                  kConsumers + 1,
              "the folding warps' staging fits the ring and the stage");

// Position of a warp role in the slot ring and in the partial hand-off
// sequence; persists across the GEMV phases of one kernel.
struct RingPos {
  int nslots = kSlots;  // ring depth of this launch (ring_slots)
  int slot = 0;
  uint32_t ph = 0;   // parity of the current ring pass
  int t = 0;         // chunks issued so far (producer)
  int fl = 0;        // row-group segments handed over so far
  bool ok = true;
};

// Slots of the ring: kSlots in the ring proper, then slots borrowed from the
// end of the activation stage when the most rows of the launch leave it free
// (one-row passes stage 8 KB of their 44 KB at K = 4096): more weight bytes
// in flight per CTA.  Never while the stage holds the K-outer windows.
SSD_HD int ring_slots(const LinearArgs& a, bool kouter) {
  if (kouter) return kSlots;
  const int mm = a.m_max > 0 ? a.m_max : (a.M_dev ? kMaxRows : a.M_static);
  const long need = (long)mm * (a.K + kPad) * (long)sizeof(bf16);
  if (need > kStageBytes) return kSlots;
  return kSlots + (int)((kStageBytes - need) / kSlotBytes);
}
SSD_DI unsigned char* slot_ptr(GemvSmem& sm, int slot) {
  return slot < kSlots ? sm.ring + slot * kSlotBytes
                       : reinterpret_cast<unsigned char*>(sm.stage) + kStageBytes -
                             (slot - kSlots + 1) * kSlotBytes;
}

// Length of the next chunk: at most kChunk units, never crossing a row group.
SSD_DI int chunk_len(const Part& p, int kb, int left) {
  return min(kChunk, min(p.KB - kb, left));
}

// Consumer warps: take the ring's slots in order, kUPW units per warp per
// slot, and hand each finished row-group segment to the epilogue warp.
template <int IN, int EPI, bool STAGED>
SSD_DI void consume(const LinearArgs& a, const Part& p, GemvSmem& sm, int U0, int U1,
                    int M, int warp, int lane, RingPos& rp) {
  const int g = lane >> 2, c = lane & 3;
  const bool two = M > 8;
  const bool v0 = g < M, v1 = two && (g + 8) < M;
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  const float rs0 = IN == IN_NORM && v0 && !STAGED ? sm.rstd[g] : 0.f;
  const float rs1 = IN == IN_NORM && v1 && !STAGED ? sm.rstd[g + 8] : 0.f;
  int vr = U0 / p.KB, kb = U0 % p.KB, left = U1 - U0;
  int n = left > 0 ? chunk_len(p, kb, left) : 0;
  BRaw<IN> ra[kUPW], rb[kUPW];
  if (!STAGED) {
#pragma unroll
    for (int i = 0; i < kUPW; ++i) {
      const int un = warp + i * kConsumers;
      b_issue<IN>(ra[i], a, g, (kb + un) * 32 + 8 * c, v0 && un < n);
      if (two) b_issue<IN>(rb[i], a, g + 8, (kb + un) * 32 + 8 * c, v1 && un < n);
    }
  }
  int slot = rp.slot;
  uint32_t ph = rp.ph;
  int fl = rp.fl;
  while (left > 0) {
    // position of the next chunk; its B operands are requested now
    int kb2 = kb + n, vr2 = vr;
    const int left2 = left - n;
    if (kb2 == p.KB) { kb2 = 0; ++vr2; }
    const int n2 = left2 > 0 ? chunk_len(p, kb2, left2) : 0;
    BRaw<IN> na[kUPW], nb[kUPW];
    if (!STAGED) {
#pragma unroll
      for (int i = 0; i < kUPW; ++i) {
        const int un = warp + i * kConsumers;
        b_issue<IN>(na[i], a, g, (kb2 + un) * 32 + 8 * c, v0 && un < n2);
        if (two) b_issue<IN>(nb[i], a, g + 8, (kb2 + un) * 32 + 8 * c, v1 && un < n2);
      }
    }

    if (!mbar_wait(&sm.full[slot], ph)) {
      if (lane == 0) atomicExch(a.err, 3);
      rp.ok = false;
      return;
    }
#pragma unroll
    for (int i = 0; i < kUPW; ++i) {
      const int un = warp + i * kConsumers;
      if (un < n) {
        const unsigned char* base = slot_ptr(sm, slot) + un * kUnitBytes;
        const uint4 wa = *reinterpret_cast<const uint4*>(base + unit_slot(lane));
        const uint4 wb = *reinterpret_cast<const uint4*>(base + 512 + unit_slot(lane));
        const int off = (kb + un) * 32 + 8 * c;
        const uint4 xa = STAGED ? (v0 ? *reinterpret_cast<const uint4*>(sm.stage + (size_t)g * (a.K + kPad) + off)
                                      : make_uint4(0u, 0u, 0u, 0u))
                                : b_finish<IN>(ra[i], rs0);
        mma_bf16(acc[0], wa.x, wb.x, wa.y, wb.y, xa.x, xa.y);
        mma_bf16(acc[0], wa.z, wb.z, wa.w, wb.w, xa.z, xa.w);
        if (two) {
          const uint4 xb = STAGED ? (v1 ? *reinterpret_cast<const uint4*>(sm.stage + (size_t)(g + 8) * (a.K + kPad) + off)
                                        : make_uint4(0u, 0u, 0u, 0u))
                                  : b_finish<IN>(rb[i], rs1);
          mma_bf16(acc[1], wa.x, wb.x, wa.y, wb.y, xb.x, xb.y);
          mma_bf16(acc[1], wa.z, wb.z, wa.w, wb.w, xb.z, xb.w);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[slot]);
    if (++slot == rp.nslots) { slot = 0; ph ^= 1u; }
    const bool group_done = kb2 == 0 || left2 == 0;
    vr = vr2;
    kb = kb2;
    left = left2;
    n = n2;
    if (!STAGED) {
#pragma unroll
      for (int i = 0; i < kUPW; ++i) {
        ra[i] = na[i];
        if (two) rb[i] = nb[i];
      }
    }
    if (!group_done) continue;
    // ---- the CTA's part of a row group is done: hand the accumulators to
    // the epilogue warp through the double-buffered partial area
    {
      const int buf = fl & 1;
      if (fl >= 2 && !mbar_wait(&sm.rempty[buf], ((fl >> 1) - 1) & 1)) {
        if (lane == 0) atomicExch(a.err, 5);
        rp.ok = false;
        return;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int tok = h * 8 + 2 * c;
        sm.red[buf][warp][g][tok] = acc[h][0];
        sm.red[buf][warp][g][tok + 1] = acc[h][1];
        sm.red[buf][warp][g + 8][tok] = acc[h][2];
        sm.red[buf][warp][g + 8][tok + 1] = acc[h][3];
        acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.rfull[buf]);
      ++fl;
    }
  }
  rp.slot = slot;
  rp.ph = ph;
  rp.fl = fl;
}

// Batched K-outer order (bf16 input, whole-group partition, passes whose rows
// may not fit the stage: LinearArgs::wide).  A CTA takes its row groups in
// batches of up to kBatch (whole gate/up pairs for SwiGLU); within a batch it
// goes through K in windows of kWinUnits units (512 columns), and within a
// window through the batch's groups, each in chunks of up to kChunk units.
// The activations of a window (the pass's rows x 512 columns) are copied to
// shared memory once per batch with cp.async into a ring of as many buffers
// of M rows as the stage holds (at most kWinBufs), all but one of them ahead
// of the window being consumed.  The chunks, the unit each
// warp takes and the order in which a warp accumulates a group's units are
// those of the staged layout, so every row's bits are the same in both.
constexpr int kWinUnits = 16;
constexpr int kWinRow = kWinUnits * 32 * 2 + 64;   // bytes per row; rows 16 banks apart
constexpr int kWinBytes = kMaxRows * kWinRow;
#ifndef SSD_GEMV_WINBUFS
#define SSD_GEMV_WINBUFS 4
#endif
constexpr int kWinBufs = SSD_GEMV_WINBUFS;         // most window buffers (2 .. 4)
#ifndef SSD_GEMV_BATCH
#define SSD_GEMV_BATCH 4
#endif
constexpr int kBatch = SSD_GEMV_BATCH;             // row groups per batch (even: whole pairs)
static_assert(2 * kWinBytes <= kStageBytes, "two windows of kMaxRows rows fit the stage");
static_assert(kWinBufs >= 2 && kWinBufs <= 4, "window ring depth");
// window buffers of M rows in the stage
SSD_HD int win_bufs(int M) {
  const int n = kStageBytes / (M * kWinRow);
  return n < kWinBufs ? n : kWinBufs;
}
static_assert(kWinUnits % kChunk == 0, "windows hold whole chunks");
static_assert(kBatch % 2 == 0, "a batch holds whole gate/up pairs");
static_assert(sizeof(float) * kBatch * (kConsumers + 1) * 256 + sizeof(LmRec) * kBatch * kMaxRows <=
                  (size_t)kStageBytes,
              "the last batch's warp sums, outputs and records fit the stage");

template <int IN, int EPI>
SSD_HD bool kouter_order(const LinearArgs& a, const Part& p) {
  return IN == IN_BF16 && a.wide && p.G == p.KB * (EPI == EPI_SWIGLU ? 2 : 1);
}

// Calls f(vr, kb, n) for every chunk of CTA range [U0, U1) (whole groups) in
// the batched K-outer order.
template <class F>
SSD_DI void kouter_chunks(const Part& p, int U0, int U1, F&& f) {
  const int KB = p.KB, g_end = U1 / KB;
  for (int g0 = U0 / KB; g0 < g_end; g0 += kBatch) {
    const int nb = min(kBatch, g_end - g0);
    for (int kw = 0; kw < KB; kw += kWinUnits) {
      const int ke = min(kw + kWinUnits, KB);
      for (int gi = 0; gi < nb; ++gi)
        for (int kb = kw; kb < ke; kb += kChunk) f(g0 + gi, kb, min(kChunk, ke - kb));
    }
  }
}

// First row group of the batch that holds the last group of [g_begin,
// g_end) in the batched K-outer order.
SSD_HD int kouter_last_batch(int g_begin, int g_end) {
  return g_begin + ((g_end - g_begin - 1) / kBatch) * kBatch;
}

// The last batch of a K-outer CTA range, finished by the consumer warps
// (threads 0 .. kConsumers * 32 - 1) once their MMAs are done, so that the
// kernel's tail is not one warp working through several 13-row groups.
// part[gi][w][row][tok] holds warp w's sums of group g0 + gi; every output
// is finished with the arithmetic of `epilogue` (the warps' sums added in
// warp order, then the epilogue's own operations), so the bits are those
// of the epilogue warp's path.  Projections only (not the LM head).
template <int EPI>
SSD_DI void final_batch_epilogue(const LinearArgs& a, const float* part, float* epv, int g0,
                                 int nb, int M, int tid) {
  constexpr int kT = kConsumers * 32;
  for (int e = tid; e < nb * 16 * M; e += kT) {
    const int gi = e / (16 * M), rem = e % (16 * M), row = rem / M, tok = rem % M;
    float s2 = 0.f;
    for (int w2 = 0; w2 < kConsumers; ++w2) s2 += part[((gi * kConsumers + w2) * 16 + row) * 16 + tok];
    epv[(gi * 16 + row) * 16 + tok] = 0.f + s2;
  }
  consumer_sync();
  if (EPI == EPI_LMHEAD) {
    // logits, then every (group, token) record of lm_group; the epilogue
    // warp folds the records into its running records in group order
    const int slot = a.slot_dev ? __ldcg(a.slot_dev) : 0;
    const int round = a.round_dev ? __ldcg(a.round_dev) : a.round_static;
    const int pos0 = a.pos0_dev ? __ldcg(a.pos0_dev) : a.pos0_static;
    if (a.logits)
      for (int e = tid; e < nb * 16 * M; e += kT) {
        const int gi = e / (16 * M), rem = e % (16 * M), row = rem / M, tok = rem % M;
        a.logits[(size_t)(slot + tok) * a.R + (g0 + gi) * 16 + row] = epv[(gi * 16 + row) * 16 + tok];
      }
    LmRec* recs = reinterpret_cast<LmRec*>(epv + nb * 256);  // [gi][tok]
    for (int e = tid; e < nb * M; e += kT) {
      const int gi = e / M, tok = e % M;
      recs[gi * kMaxRows + tok] = lm_group_rec(a, (g0 + gi) * 16, epv + gi * 256 + tok, 16, tok,
                                               round, pos0);
    }
    return;
  }
  if (EPI == EPI_STORE) {
    for (int e = tid; e < nb * 16 * M; e += kT) {
      const int gi = e / (16 * M), rem = e % (16 * M), row = rem / M, tok = rem % M;
      a.y[(size_t)tok * a.R + (g0 + gi) * 16 + row] = epv[(gi * 16 + row) * 16 + tok];
    }
  } else if (EPI == EPI_RESID) {
    for (int e = tid; e < nb * 16 * M; e += kT) {
      const int gi = e / (16 * M), rem = e % (16 * M), row = rem / M, tok = rem % M;
      float* xp = a.xres + (size_t)tok * a.R + (g0 + gi) * 16 + row;
      const float xn = __ldcg(xp) + epv[(gi * 16 + row) * 16 + tok];
      *xp = xn;
      epv[(gi * 16 + row) * 16 + tok] = xn;
    }
    consumer_sync();
    for (int e = tid; e < nb * M; e += kT) {
      const int gi = e / M, tok = e % M;
      float s = 0.f;
      for (int row = 0; row < 16; ++row) {
        const float v = epv[(gi * 16 + row) * 16 + tok];
        s += v * v;
      }
      a.ss_out[(size_t)tok * (a.R / kSsGroup) + g0 + gi] = s;
    }
  } else if (EPI == EPI_SWIGLU) {
    // groups g0 + gi (gate, gi even) and g0 + gi + 1 (up) are one feature block
    for (int e = tid; e < (nb / 2) * 16 * M; e += kT) {
      const int pi = e / (16 * M), rem = e % (16 * M), row = rem / M, tok = rem % M;
      const float gt = epv[(2 * pi * 16 + row) * 16 + tok];
      const float up = epv[((2 * pi + 1) * 16 + row) * 16 + tok];
      const float sl = gt / (1.0f + expf(-gt));
      a.u[(size_t)tok * a.R + ((g0 + 2 * pi) >> 1) * 16 + row] = __float2bfloat16_rn(sl * up);
    }
  }
}

template <int EPI>
SSD_DI void consume_win(const LinearArgs& a, const Part& p, GemvSmem& sm, int U0, int U1, int M,
                        int warp, int lane, RingPos& rp) {
  const int tid = threadIdx.x;  // consumer threads are 0 .. kConsumers * 32 - 1
  const int g = lane >> 2, c = lane & 3;
  const bool two = M > 8;
  const bool v0 = g < M, v1 = two && (g + 8) < M;
  unsigned char* wb = reinterpret_cast<unsigned char*>(sm.stage);
  const int KB = p.KB;
  const int nwin = (KB + kWinUnits - 1) / kWinUnits;  // windows per batch
  const int g_begin = U0 / KB, g_end = U1 / KB;
  const int nbatch = (g_end - g_begin + kBatch - 1) / kBatch;
  const int total = nbatch * nwin;                    // windows this CTA consumes
  // window q (K window q % nwin of batch q / nwin) into buffer q % nbuf;
  // one commit per window, empty past the end, so the group count is uniform
  const int nbuf = win_bufs(M), wstride = M * kWinRow;
  auto issue = [&](int q) {
    if (q < total) {
      const int kw = q % nwin;
      const int wu = min(kWinUnits, KB - kw * kWinUnits);
      unsigned char* dst = wb + (q % nbuf) * wstride;
      const bf16* src = a.act + (size_t)kw * kWinUnits * 32;
      for (int e = tid; e < M * kWinUnits * 4; e += kConsumers * 32) {
        const int m = e / (kWinUnits * 4), qq = e % (kWinUnits * 4);
        if (qq < wu * 4) cp_async16(dst + m * kWinRow + qq * 16, src + (size_t)m * a.K + qq * 8);
      }
    }
    cp_async_commit();
  };
  for (int q0 = 0; q0 < nbuf - 1; ++q0) issue(q0);
  float acc[kBatch][2][4];
#pragma unroll
  for (int gi = 0; gi < kBatch; ++gi)
#pragma unroll
    for (int h = 0; h < 2; ++h) acc[gi][h][0] = acc[gi][h][1] = acc[gi][h][2] = acc[gi][h][3] = 0.f;
  int slot = rp.slot;
  uint32_t ph = rp.ph;
  int fl = rp.fl;
  // A failed wait does not leave the loop: every consumer warp must take part
  // in every window barrier, so a warp that gave up runs on without waiting.
  bool okw = rp.ok;
  int q = 0;
  for (int g0 = g_begin; g0 < g_end; g0 += kBatch) {
    const int nb = min(kBatch, g_end - g0);
    for (int kw = 0; kw < nwin; ++kw, ++q) {
      // window q has landed (for every thread's copies) and every warp is
      // done with window q - 1, whose buffer window q + nbuf - 1 now takes
      if (nbuf == 2) cp_async_wait_group<0>();
      else if (nbuf == 3) cp_async_wait_group<1>();
      else cp_async_wait_group<2>();
      consumer_sync();
      issue(q + nbuf - 1);
      const unsigned char* wbase = wb + (q % nbuf) * wstride;
      const int kb0 = kw * kWinUnits, ke = min(kb0 + kWinUnits, KB);
#pragma unroll
      for (int gi = 0; gi < kBatch; ++gi) {
        if (gi >= nb) break;
        for (int kb = kb0; kb < ke; kb += kChunk) {
          const int n = min(kChunk, ke - kb);
          if (okw && !mbar_wait(&sm.full[slot], ph)) {
            if (lane == 0) atomicExch(a.err, 3);
            okw = false;
          }
#pragma unroll
          for (int i = 0; i < kUPW; ++i) {
            const int un = warp + i * kConsumers;
            if (un < n) {
              const unsigned char* base = slot_ptr(sm, slot) + un * kUnitBytes;
              const uint4 wa = *reinterpret_cast<const uint4*>(base + unit_slot(lane));
              const uint4 wbv = *reinterpret_cast<const uint4*>(base + 512 + unit_slot(lane));
              const int col = ((kb - kb0) + un) * 64 + c * 16;  // bytes into the row
              const uint4 xa = v0 ? *reinterpret_cast<const uint4*>(wbase + g * kWinRow + col)
                                  : make_uint4(0u, 0u, 0u, 0u);
              mma_bf16(acc[gi][0], wa.x, wbv.x, wa.y, wbv.y, xa.x, xa.y);
              mma_bf16(acc[gi][0], wa.z, wbv.z, wa.w, wbv.w, xa.z, xa.w);
              if (two) {
                const uint4 xb = v1 ? *reinterpret_cast<const uint4*>(wbase + (g + 8) * kWinRow + col)
                                    : make_uint4(0u, 0u, 0u, 0u);
                mma_bf16(acc[gi][1], wa.x, wbv.x, wa.y, wbv.y, xb.x, xb.y);
                mma_bf16(acc[gi][1], wa.z, wbv.z, wa.w, wbv.w, xb.z, xb.w);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.empty[slot]);
          if (++slot == rp.nslots) { slot = 0; ph ^= 1u; }
        }
      }
    }
    if (g0 == kouter_last_batch(g_begin, g_end)) {
      // the last batch: every consumer warp is done with the windows and the
      // ring, so the stage takes the warps' sums and the consumer warps
      // finish the batch themselves (the epilogue warp stops before it)
      consumer_sync();
      float* part = reinterpret_cast<float*>(sm.stage);
#pragma unroll
      for (int gi = 0; gi < kBatch; ++gi) {
        if (gi >= nb) break;
        float* pw = part + (size_t)(gi * kConsumers + warp) * 256;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int tok = h * 8 + 2 * c;
          pw[g * 16 + tok] = acc[gi][h][0];
          pw[g * 16 + tok + 1] = acc[gi][h][1];
          pw[(g + 8) * 16 + tok] = acc[gi][h][2];
          pw[(g + 8) * 16 + tok + 1] = acc[gi][h][3];
        }
      }
      consumer_sync();
      final_batch_epilogue<EPI>(a, part, part + (size_t)nb * kConsumers * 256, g0, nb, M,
                                threadIdx.x);
      if (EPI == EPI_LMHEAD) {
        consumer_sync();
        if (threadIdx.x == 0) mbar_arrive(&sm.lastbar);
      }
      break;
    }
    // the batch's groups are done: hand them to the epilogue warp in order
#pragma unroll
    for (int gi = 0; gi < kBatch; ++gi) {
      if (gi >= nb) break;
      const int buf = fl & 1;
      if (okw && fl >= 2 && !mbar_wait(&sm.rempty[buf], ((fl >> 1) - 1) & 1)) {
        if (lane == 0) atomicExch(a.err, 5);
        okw = false;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int tok = h * 8 + 2 * c;
        sm.red[buf][warp][g][tok] = acc[gi][h][0];
        sm.red[buf][warp][g][tok + 1] = acc[gi][h][1];
        sm.red[buf][warp][g + 8][tok] = acc[gi][h][2];
        sm.red[buf][warp][g + 8][tok + 1] = acc[gi][h][3];
        acc[gi][h][0] = acc[gi][h][1] = acc[gi][h][2] = acc[gi][h][3] = 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.rfull[buf]);
      ++fl;
    }
  }
  cp_async_wait_all();
  rp.slot = slot;
  rp.ph = ph;
  rp.fl = fl;
  rp.ok = okw;
}

// Producer warp (lane 0 issues): streams CTA b's units of one GEMV into the
// ring, in the order the consumers take them (row groups in turn, or the
// batched K-outer order).  Weights never depend on earlier phases, so the
// producer runs ahead of the consumers, bounded only by free ring slots.
template <int IN, int EPI>
SSD_DI void producer_phase(const LinearArgs& a, const Part& p, GemvSmem& sm, int b, int lane,
                           RingPos& rp) {
  if (b >= p.C || lane != 0 || !rp.ok) return;
  // the RMSNorm gain is the one input the consumers read from DRAM: bring
  // it into L2 ahead of this CTA's weight stream
  if (a.gain && b == 0) bulk_prefetch_l2(a.gain, (uint32_t)(a.K * sizeof(float)));
  const int U0 = unit_begin(p, b), U1 = unit_begin(p, b + 1);
  auto put = [&](int vr, int kb, int n) {
    if (!rp.ok) return;
    if (rp.t >= rp.nslots && !mbar_wait(&sm.empty[rp.slot], rp.ph ^ 1u)) {
      atomicExch(a.err, 2);
      rp.ok = false;
      return;
    }
    mbar_arrive_expect_tx(&sm.full[rp.slot], (uint32_t)(n * kUnitBytes));
    bulk_g2s(slot_ptr(sm, rp.slot), unit_src<EPI>(a, p, vr, kb), (uint32_t)(n * kUnitBytes),
             &sm.full[rp.slot]);
    if (++rp.slot == rp.nslots) { rp.slot = 0; rp.ph ^= 1u; }
    ++rp.t;
  };
  if (kouter_order<IN, EPI>(a, p)) {
    kouter_chunks(p, U0, U1, put);
    return;
  }
  int vr = U0 / p.KB, kb = U0 % p.KB, left = U1 - U0;
  while (left > 0 && rp.ok) {
    const int n = chunk_len(p, kb, left);
    put(vr, kb, n);
    kb += n;
    left -= n;
    if (kb == p.KB) { kb = 0; ++vr; }
  }
}

// Epilogue warp: receives CTA b's row-group segments of one GEMV in order.
// A row group that lies wholly in this CTA (for SwiGLU: both groups of the
// gate/up pair) is finished straight from shared memory.  A group split
// across CTAs is finished by the last CTA to complete it: each CTA stores its
// partial, and the finisher sums the partials in CTA order.  Either way a
// group's sum is its CTAs' partials added in CTA order, each partial being
// the consumer warps' sums added in warp order, so the result depends on the
// matrix shape only.  The LM head (whole-group partition) folds its groups
// into one running record per token and publishes it at the end.
template <int IN, int EPI>
SSD_DI void epilogue_phase(const LinearArgs& a, const Part& p, GemvSmem& sm, int b, int M,
                           int lane, RingPos& rp, LmRec& run) {
  if (b >= p.C || !rp.ok) return;
  const int U0 = unit_begin(p, b), U1 = unit_begin(p, b + 1);
  int vr = U0 / p.KB, kb = U0 % p.KB, left = U1 - U0;
  // K-outer ranges: the consumer warps finish the last batch
  const bool kouter = kouter_order<IN, EPI>(a, p);
  const int g_last = kouter ? kouter_last_batch(U0 / p.KB, U1 / p.KB) : 0;
  if (kouter) left = g_last * p.KB - U0;
  int slot = 0, round = 0, pos0 = 0;
  if (EPI == EPI_LMHEAD) {
    slot = a.slot_dev ? __ldcg(a.slot_dev) : 0;
    round = a.round_dev ? __ldcg(a.round_dev) : a.round_static;
    pos0 = a.pos0_dev ? __ldcg(a.pos0_dev) : a.pos0_static;
  }
  for (; left > 0; ++rp.fl) {
    const int fl = rp.fl;
    const int gvr = vr;
    left -= p.KB - kb < left ? p.KB - kb : left;
    kb = 0;
    ++vr;
    const int buf = fl & 1;
    XPre xp;
    xres_prefetch<EPI>(a, gvr, M, lane, xp);
    if (!mbar_wait(&sm.rfull[buf], (fl >> 1) & 1)) {
      if (lane == 0) atomicExch(a.err, 4);
      rp.ok = false;
      return;
    }
    const bool whole = EPI == EPI_LMHEAD ||
                       (owns(p, gvr, b) && (EPI != EPI_SWIGLU || owns(p, gvr ^ 1, b)));
    if (whole) {
      const int h = EPI == EPI_SWIGLU ? (gvr & 1) : 0;
      for (int e = lane; e < 16 * M; e += 32) {
        const int row = e / M, tok = e % M;
        float s2 = 0.f;
        for (int w2 = 0; w2 < kConsumers; ++w2) s2 += sm.red[buf][w2][row][tok];
        sm.ep[h][row][tok] = 0.f + s2;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.rempty[buf]);
      if (EPI == EPI_SWIGLU && h == 0) continue;  // the up group follows
      if (EPI == EPI_LMHEAD)
        lm_group(a, gvr, sm.ep, M, lane, slot, round, pos0, run);
      else
        epilogue<EPI>(a, p, gvr, sm.ep, M, lane, xp);
      __syncwarp();
      continue;
    }
    // ---- split group (pair): every CTA stores its partial; the CTA that
    // holds the first unit (F) finishes, the others only publish.  F's own
    // segments of the group are its last ones and the others' are their
    // first ones, so F waits for work that needs nothing from F.
    const int seg = b - cta_first(p, gvr * p.KB);
    float* dst = a.part + ((size_t)gvr * p.segmax + seg) * 256;
    for (int e = lane; e < 16 * M; e += 32) {
      const int row = e / M, tok = e % M;
      float s2 = 0.f;
      for (int w2 = 0; w2 < kConsumers; ++w2) s2 += sm.red[buf][w2][row][tok];
      dst[row * 16 + tok] = s2;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.rempty[buf]);
    const int g0 = EPI == EPI_SWIGLU ? (gvr & ~1) : gvr;
    const int F = cta_first(p, g0 * p.KB);
    const int cidx = EPI == EPI_SWIGLU ? gvr >> 1 : gvr;
    if (b != F) {
      __threadfence();
      __syncwarp();
      if (lane == 0) red_release_add(a.counter + cidx, 1u);
      continue;
    }
    if (EPI == EPI_SWIGLU && (gvr & 1) == 0 && left > 0) continue;  // F's up segment follows
    const int ngrp = EPI == EPI_SWIGLU ? 2 : 1;
    int expect = 0;
    for (int hh = 0; hh < ngrp; ++hh) {
      const int gv = g0 + hh;
      expect += nseg(p, gv) - (cta_first(p, gv * p.KB) == F ? 1 : 0);
    }
    int ok = 1;
    if (lane == 0) ok = wait_count(a.counter + cidx, (unsigned)expect);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) atomicExch(a.err, 6);
      rp.ok = false;
      return;
    }
    // sum the CTAs' partials of the group(s) in CTA order; the loads of up
    // to four segments of both groups are issued before any is used
    int ns[2];
    ns[0] = nseg(p, g0);
    ns[1] = ngrp > 1 ? nseg(p, g0 + 1) : 0;
    for (int e = lane; e < 16 * M; e += 32) {
      const int row = e / M, tok = e % M;
      float v[2][4];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float* src = a.part + (size_t)(g0 + hh) * p.segmax * 256 + row * 16 + tok;
#pragma unroll
        for (int q = 0; q < 4; ++q) v[hh][q] = q < ns[hh] ? __ldcg(src + (size_t)q * 256) : 0.f;
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (hh >= ngrp) break;
        const float* src = a.part + (size_t)(g0 + hh) * p.segmax * 256 + row * 16 + tok;
        float s2 = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q < ns[hh]) s2 += v[hh][q];
        for (int q = 4; q < ns[hh]; ++q) s2 += __ldcg(src + (size_t)q * 256);
        sm.ep[hh][row][tok] = s2;
      }
    }
    __syncwarp();
    if (lane == 0) a.counter[cidx] = 0u;
    epilogue<EPI>(a, p, gvr, sm.ep, M, lane, xp);
    __syncwarp();
  }
  if (EPI == EPI_LMHEAD && kouter) {
    // the last batch's records, computed by the consumer warps, in group order
    if (!mbar_wait(&sm.lastbar, 0u)) {
      if (lane == 0) atomicExch(a.err, 8);
      rp.ok = false;
      return;
    }
    const LmRec* recs = reinterpret_cast<const LmRec*>(
        reinterpret_cast<const float*>(sm.stage) + (size_t)(U1 / p.KB - g_last) * (kConsumers + 1) * 256);
    if (lane < M)
      for (int gi = 0; gi < U1 / p.KB - g_last; ++gi)
        lm_combine(run, recs[gi * kMaxRows + lane], a.temperature);
  }
}

// LM head, end of the kernel for the epilogue warp (is_epi, holding the
// CTA's running records) and the consumer warps: the epilogue warp publishes
// and tells the others through foldbar whether this CTA published last; if
// so the kConsumers + 1 warps fold the pass's tokens, token t by warp
// t mod (kConsumers + 1).  Every wait is bounded.
SSD_DI void lm_end(const LinearArgs& a, const Part& p, GemvSmem& sm, int b, int M, int warp,
                   int lane, const RingPos& rp, const LmRec& run, bool is_epi) {
  int last = 0;
  if (is_epi) {
    if (rp.ok && b < p.C) last = lm_publish(a, p, b, M, lane, run);
    if (lane == 0) {
      sm.fold_last = last;
      mbar_arrive(&sm.foldbar);
    }
    if (last && lane == 0) a.counter[0] = 0u;  // every CTA has counted
  } else {
    if (!mbar_wait(&sm.foldbar, 0u)) {
      if (lane == 0) atomicExch(a.err, 7);
      return;
    }
    last = *reinterpret_cast<volatile int*>(&sm.fold_last);
  }
  if (!last) return;
  __threadfence();
  const int slot = a.slot_dev ? __ldcg(a.slot_dev) : 0;
  const int wi = is_epi ? kConsumers : warp;
  float* stage =
      wi < kFoldInRing ? reinterpret_cast<float*>(sm.ring + wi * kFoldBytes)
      : wi < kFoldInRing + kFoldInStage
          ? reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(sm.stage) +
                                     (wi - kFoldInRing) * kFoldBytes)
          : &sm.red[0][0][0][0];
  for (int tok = wi; tok < M; tok += kConsumers + 1) lm_fold(a, p, tok, lane, slot, stage);
}

// Consumer warps: RMSNorm statistics, activation staging and the MMAs for
// CTA b's units of one GEMV.
template <int IN, int EPI>
SSD_DI void consumer_phase(const LinearArgs& a, const Part& p, GemvSmem& sm, int b, int M,
                           int warp, int lane, RingPos& rp) {
  if (b >= p.C) return;
  const int U0 = unit_begin(p, b), U1 = unit_begin(p, b + 1);
  if (!rp.ok) return;
  const bool kouter = kouter_order<IN, EPI>(a, p);
  const bool staged = !kouter && (size_t)M * (a.K + kPad) * sizeof(bf16) <= (size_t)kStageBytes;
  const int vpr = a.K / 8;  // 16-byte pieces per row
  const int nst = staged ? M * vpr : 0;
  constexpr int kPre = IN == IN_NORM ? 2 : 4;
  constexpr int kStride = kConsumers * 32;
  // the first pieces' loads go out together with the statistics' loads
  BRaw<IN> pre[kPre];
  int e0 = threadIdx.x;
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int e = e0 + i * kStride;
    if (e < nst) b_issue<IN>(pre[i], a, e / vpr, (e % vpr) * 8, true);
  }
  if (IN == IN_NORM) {
    // 1 / sqrt(mean(x^2) + eps) per row from the producer's partials, in a
    // fixed order: lane l sums partials l, l+32, ... then a butterfly.
    const int NP = a.K / kSsGroup;
    for (int m = warp; m < M; m += kConsumers) {
      float s2 = 0.f;
#pragma unroll 8
      for (int q = lane; q < NP; q += 32) s2 += __ldcg(a.ss + (size_t)m * NP + q);
      s2 = sum_warp(s2);
      if (lane == 0) sm.rstd[m] = 1.0f / sqrtf(s2 / (float)a.K + a.eps);
    }
    consumer_sync();
  }
  if (staged) {
    for (;;) {
#pragma unroll
      for (int i = 0; i < kPre; ++i) {
        const int e = e0 + i * kStride;
        if (e < nst) {
          const int m = e / vpr;
          const float rs = IN == IN_NORM ? sm.rstd[m] : 0.f;
          *reinterpret_cast<uint4*>(sm.stage + (size_t)m * (a.K + kPad) + (e % vpr) * 8) =
              b_finish<IN>(pre[i], rs);
        }
      }
      e0 += kPre * kStride;
      if (e0 >= nst) break;
#pragma unroll
      for (int i = 0; i < kPre; ++i) {
        const int e = e0 + i * kStride;
        if (e < nst) b_issue<IN>(pre[i], a, e / vpr, (e % vpr) * 8, true);
      }
    }
    consumer_sync();
    consume<IN, EPI, true>(a, p, sm, U0, U1, M, warp, lane, rp);
  } else if (kouter) {
    consume_win<EPI>(a, p, sm, U0, U1, M, warp, lane, rp);
  } else if constexpr (IN == IN_NORM) {
    // norm-fused rows always fit the stage (the host refuses more and runs
    // the RMSNorm pre-pass with a bf16-input pass instead)
    if (lane == 0) atomicExch(a.err, 9);
    rp.ok = false;
  } else {
    consume<IN, EPI, false>(a, p, sm, U0, U1, M, warp, lane, rp);
  }
}



}  // namespace gemv
}  // namespace ssd
