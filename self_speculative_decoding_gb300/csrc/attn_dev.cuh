// Decode / verify attention: one work item = (KV head, 64-position chunk).
//
// A pass carries M <= 16 query rows at consecutive positions pos0..pos0+M-1.
// The item
//   1. brings the chunk's cached keys / values into shared memory with bulk
//      copies;
//   2. applies rotate-half RoPE to the chunk's new keys, rounds k and v to
//      bf16 and appends them to the cache (LayerSkip blog §3.2: every pass
//      writes the K/V of the layers it runs);
//   3. for every query head of the group and every row computes the chunk's
//      maximum score, sum of exponentials and unnormalised output;
//   4. the item that completes a head's last chunk combines that head's
//      chunks in chunk order and writes bf16 outputs.
// Causality is per row: row m sees keys <= pos0+m; masked keys contribute
// exact zeros, and a row's values depend only on its own position, so a row
// computed in a pass of M rows is bit-identical to the same row alone.
#pragma once

#include "kernels.cuh"

namespace ssd {
namespace attn {

constexpr int kGroupThreads = 256;  // threads that execute an item
constexpr int kGroupWarps = kGroupThreads / 32;
// A chunk's partial record per (head, row): max score, sum of exponentials,
// two pad words, then the unnormalised output (16-byte aligned).
constexpr int kRecPad = 4;

// Shared memory of one item (offsets multiples of 16 B):
//   K [64][dh] bf16 | V [64][dh] bf16 | Q [16][dh] f32 | S [16][64] f32
//   | combine scratch: m, l, w [nchunk] f32
//   | rows' positions [16] i32 | side rows' own-key weights [16] f32
//   | side rows' own keys / values [kMaxSide][dh] bf16 each
// The combine reuses the region from K up to the end of the scratch arrays;
// the tail after it survives the combine.
struct Smem {
  bf16* K;
  bf16* V;
  float* Q;
  float* S;
  float* cm;
  float* cl;
  float* cw;
  int* rpos;
  float* sp;
  bf16* SK;
  bf16* SV;
};

__host__ __device__ inline size_t main_bytes(int dh, int nchunk) {
  const size_t b = (size_t)kAttnChunk * dh * 2 + (size_t)kAttnChunk * dh * 2 +
                   (size_t)kMaxRows * dh * 4 + (size_t)kMaxRows * kAttnChunk * 4 +
                   (size_t)3 * nchunk * 4;
  return (b + 15) & ~(size_t)15;
}

__host__ __device__ inline size_t smem_bytes(int dh, int nchunk) {
  return main_bytes(dh, nchunk) + (size_t)kMaxRows * 4 * 2 + (size_t)kMaxSide * dh * 2 * 2;
}

SSD_DI Smem carve(unsigned char* raw, int dh, int nchunk) {
  Smem sm;
  sm.K = reinterpret_cast<bf16*>(raw);
  sm.V = sm.K + kAttnChunk * dh;
  sm.Q = reinterpret_cast<float*>(sm.V + kAttnChunk * dh);
  sm.S = sm.Q + kMaxRows * dh;
  sm.cm = sm.S + kMaxRows * kAttnChunk;
  sm.cl = sm.cm + nchunk;
  sm.cw = sm.cl + nchunk;
  sm.rpos = reinterpret_cast<int*>(raw + main_bytes(dh, nchunk));
  sm.sp = reinterpret_cast<float*>(sm.rpos + kMaxRows);
  sm.SK = reinterpret_cast<bf16*>(sm.sp + kMaxRows);
  sm.SV = sm.SK + kMaxSide * dh;
  return sm;
}

// Position p's cached key / value row.
SSD_DI const bf16* cache_row(const bf16* c, const AttnArgs& a, int kvh, int pos) {
  return c + (size_t)kvh * a.max_seq * a.dh + (size_t)pos * a.dh;
}

// Step (1) of work item `item`: the bulk copies of the chunk's cached keys
// and values (positions before pos0): one copy each for the K rows and the V
// rows (consecutive positions are contiguous in the cache), issued by one
// thread and completing on `bar`.  The cache rows before pos0 were written by earlier
// passes, so this may run before the wait on the preceding kernel.
SSD_DI void issue(const AttnArgs& a, int M, int pos0, int item, const Smem& sm, uint64_t* bar,
                  int tid) {
  const int dh = a.dh;
  const int c = item / a.Hkv, kvh = item % a.Hkv;
  const int p_begin = c * kAttnChunk;
  const int p_end = min(p_begin + kAttnChunk, pos0 + M);
  const int n_old = max(0, min(p_end, pos0) - p_begin);
  if (n_old > 0 && tid == 0) {
    const uint32_t bytes = (uint32_t)(n_old * dh * sizeof(bf16));
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, 2 * bytes);
    bulk_g2s(sm.K, cache_row(a.kc, a, kvh, p_begin), bytes, bar);
    bulk_g2s(sm.V, cache_row(a.vc, a, kvh, p_begin), bytes, bar);
  }
}

// Steps (2)-(4) of work item `item`, after issue() for the same item, with
// threads tid < kGroupThreads; `sync()` is the barrier of those threads.
// `bar` is an initialised mbarrier whose phase parity is tracked in `phase`;
// `flag` is one shared int.  Returns true if this item combined its head
// (the head's output is complete).
//
// Side rows (the pass's last ns rows, dynamic verification): row Mc + i sits
// at position side_pos[i] <= the last chain position.  It sees the keys
// before its position (cache and chain keys) and its own key, which stands
// where the cache would hold it; its own value enters the chunk's output as
// the last term, after the masked keys' exact zeros, so the row gets the
// bits the same token would get as an ordinary row at that position.  Its
// K/V go to its side slot, not to the cache.
template <class Sync>
SSD_DI bool body(const AttnArgs& a, int M, int ns, int pos0, int item, const Smem& sm,
                 uint64_t* bar, uint32_t& phase, int* flag, int tid, Sync sync) {
  const int dh = a.dh, half = dh / 2;
  const int G = a.H / a.Hkv;
  const int rows = G * kMaxRows;
  const int nchunk_max = a.max_seq / kAttnChunk;
  const int Mc = M - ns;                    // chain rows
  const int last_pos = pos0 + Mc - 1;
  const int n_active = last_pos / kAttnChunk + 1;
  const int warp = tid >> 5, lane = tid & 31;
  const int ld_out = a.H * dh;

  const int c = item / a.Hkv, kvh = item % a.Hkv;
  const int p_begin = c * kAttnChunk;
  const int p_end = min(p_begin + kAttnChunk, last_pos + 1);
  const int nk = p_end - p_begin;
  const int n_old = max(0, min(p_end, pos0) - p_begin);
  if (tid < M) sm.rpos[tid] = tid < Mc ? pos0 + tid : __ldcg(a.side_pos + (tid - Mc));
  // (2) new keys of this chunk: RoPE, bf16, append to the cache
  const int first_new = max(p_begin, pos0);
  for (int e = tid; e < (p_end - first_new) * half; e += kGroupThreads) {
    const int jj = e / half, i = e % half;
    const int pos = first_new + jj, m = pos - pos0, j = pos - p_begin;
    const float* kr = a.qkv + (size_t)m * a.ld_qkv + (size_t)(a.H + kvh) * dh;
    const float* vr = kr + (size_t)a.Hkv * dh;
    const float2 cs = a.rope[(size_t)pos * half + i];
    const float k0 = __ldcg(kr + i), k1 = __ldcg(kr + i + half);
    const bf16 kb0 = __float2bfloat16_rn(k0 * cs.x - k1 * cs.y);
    const bf16 kb1 = __float2bfloat16_rn(k0 * cs.y + k1 * cs.x);
    const bf16 vb0 = __float2bfloat16_rn(__ldcg(vr + i));
    const bf16 vb1 = __float2bfloat16_rn(__ldcg(vr + i + half));
    sm.K[j * dh + i] = kb0;
    sm.K[j * dh + i + half] = kb1;
    sm.V[j * dh + i] = vb0;
    sm.V[j * dh + i + half] = vb1;
    bf16* kd = const_cast<bf16*>(cache_row(a.kc, a, kvh, pos));
    bf16* vd = const_cast<bf16*>(cache_row(a.vc, a, kvh, pos));
    kd[i] = kb0;
    kd[i + half] = kb1;
    vd[i] = vb0;
    vd[i + half] = vb1;
  }
  // (2') side rows whose position lies in this chunk: own key and value
  // (same RoPE and rounding) to shared memory and to the side slot
  if (ns > 0) {
    const int side0 = __ldcg(a.side0);
    for (int e = tid; e < ns * half; e += kGroupThreads) {
      const int si = e / half, i = e % half;
      const int pos = __ldcg(a.side_pos + si);
      if (pos / kAttnChunk != c) continue;
      const float* kr = a.qkv + (size_t)(Mc + si) * a.ld_qkv + (size_t)(a.H + kvh) * dh;
      const float* vr = kr + (size_t)a.Hkv * dh;
      const float2 cs = a.rope[(size_t)pos * half + i];
      const float k0 = __ldcg(kr + i), k1 = __ldcg(kr + i + half);
      const bf16 kb0 = __float2bfloat16_rn(k0 * cs.x - k1 * cs.y);
      const bf16 kb1 = __float2bfloat16_rn(k0 * cs.y + k1 * cs.x);
      const bf16 vb0 = __float2bfloat16_rn(__ldcg(vr + i));
      const bf16 vb1 = __float2bfloat16_rn(__ldcg(vr + i + half));
      sm.SK[si * dh + i] = kb0;
      sm.SK[si * dh + i + half] = kb1;
      sm.SV[si * dh + i] = vb0;
      sm.SV[si * dh + i + half] = vb1;
      bf16* kd = a.ks + ((size_t)kvh * kMaxSide + side0 + si) * dh;
      bf16* vd = a.vs + ((size_t)kvh * kMaxSide + side0 + si) * dh;
      kd[i] = kb0;
      kd[i + half] = kb1;
      vd[i] = vb0;
      vd[i + half] = vb1;
    }
  }
  if (n_old > 0) {
    if (!mbar_wait(bar, phase & 1u)) {
      if (tid == 0) atomicExch(a.err, 1);
      return false;
    }
    ++phase;
  }

  float* part_base = a.part + ((size_t)kvh * nchunk_max + c) * rows * (dh + kRecPad);
  for (int gh = 0; gh < G; ++gh) {
    sync();  // K/V complete; the previous head's S and Q are no longer read
    // (3) queries of this head, RoPE'd, fp32
    for (int e = tid; e < M * half; e += kGroupThreads) {
      const int i = e % half, m = e / half;
      const float* qr = a.qkv + (size_t)m * a.ld_qkv + (size_t)(kvh * G + gh) * dh;
      const float2 cs = a.rope[(size_t)sm.rpos[m] * half + i];
      const float q0 = __ldcg(qr + i), q1 = __ldcg(qr + i + half);
      float* qd = sm.Q + (size_t)m * dh;
      qd[i] = q0 * cs.x - q1 * cs.y;
      qd[i + half] = q0 * cs.y + q1 * cs.x;
    }
    sync();
    // (4) scores.  Row m's dot product with key j is taken by an aligned
    // group of 8 lanes: lane q8 sums the 8-element pieces q8, q8 + 8, ... of
    // the head dimension in that order, then a 3-step butterfly (fixed
    // order).  One warp instruction reads 4 key rows of 128 contiguous bytes
    // (no bank conflict).  A warp task is one row and a run of 4-key groups;
    // the row's query pieces stay in registers over the run.  Only the
    // assignment of tasks to warps depends on M, never the order of a sum.
    {
      const int gpt = M <= 4 ? 2 : 4;        // 4-key groups per task
      const int tpr = kAttnChunk / 4 / gpt;  // tasks per row
      const int q8 = lane & 7, ks = lane >> 3;
      const bool two = dh > 64;              // pieces per lane: 1 (dh 64) or 2 (dh 128)
      for (int task = warp; task < M * tpr; task += kGroupWarps) {
        const int m = task / tpr, kg0 = (task % tpr) * gpt;
        const float* q = sm.Q + (size_t)m * dh + q8 * 8;
        const float4 qa0 = *reinterpret_cast<const float4*>(q);
        const float4 qb0 = *reinterpret_cast<const float4*>(q + 4);
        float4 qa1 = qa0, qb1 = qb0;
        if (two) {
          qa1 = *reinterpret_cast<const float4*>(q + 64);
          qb1 = *reinterpret_cast<const float4*>(q + 68);
        }
        const int pm = sm.rpos[m];
        const bf16* own = sm.SK + (size_t)(m >= Mc ? m - Mc : 0) * dh + q8 * 8;  // side rows
        for (int kg = kg0; kg < kg0 + gpt; ++kg) {
          const int key = kg * 4 + ks;
          const bool valid = key < nk && p_begin + key <= pm;
          float acc = 0.f;
          if (valid) {
            const bf16* k = m >= Mc && p_begin + key == pm ? own : sm.K + (size_t)key * dh + q8 * 8;
            acc = dot8(qa0, qb0, *reinterpret_cast<const uint4*>(k), acc);
            if (two) acc = dot8(qa1, qb1, *reinterpret_cast<const uint4*>(k + 64), acc);
          }
          acc += __shfl_xor_sync(0xffffffffu, acc, 1);
          acc += __shfl_xor_sync(0xffffffffu, acc, 2);
          acc += __shfl_xor_sync(0xffffffffu, acc, 4);
          if (q8 == 0) sm.S[(size_t)m * kAttnChunk + key] = valid ? acc * a.scale : -INFINITY;
        }
      }
    }
    sync();
    // (5) per-row chunk softmax statistics; one warp per row
    for (int m = warp; m < M; m += kGroupWarps) {
      const int r = gh * kMaxRows + m;
      float* srow = sm.S + (size_t)m * kAttnChunk;
      const float s0 = srow[lane], s1 = srow[lane + 32];
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float p0 = s0 == -INFINITY ? 0.f : expf(s0 - mx);
      float p1 = s1 == -INFINITY ? 0.f : expf(s1 - mx);
      float l = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      __syncwarp();
      if (m >= Mc) {
        // a side row's own-key weight is kept aside; its slot in the row's
        // weights becomes an exact zero for the chain value there
        const int jo = sm.rpos[m] - p_begin;
        if (jo == lane) { sm.sp[m] = p0; p0 = 0.f; }
        if (jo == lane + 32) { sm.sp[m] = p1; p1 = 0.f; }
      }
      srow[lane] = p0;
      srow[lane + 32] = p1;
      if (lane == 0) {
        part_base[(size_t)r * (dh + kRecPad) + 0] = mx;
        part_base[(size_t)r * (dh + kRecPad) + 1] = l;
      }
    }
    sync();
    // (6) unnormalised output of the chunk: output (m, dd) sums p_j v_j[dd]
    // over the keys in order.  When every output has a thread of its own
    // (M dh <= threads), thread t takes column t % dh of row t / dh.
    // Otherwise thread t takes the column pair t % (dh/2) and the rows
    // t / (dh/2) + r (kGroupThreads / (dh/2)), r = 0, 1, ...; per 4 keys it
    // reads one bf16 pair per key and one float4 of p per row.
    if (M * dh <= kGroupThreads) {
      const int dd = tid % dh, m = tid / dh;
      if (m < M) {
        const bf16* vcol = sm.V + dd;
        const float* p = sm.S + (size_t)m * kAttnChunk;
        float o = 0.f;
        int j = 0;
        for (; j + 4 <= nk; j += 4) {
          const float4 pp = *reinterpret_cast<const float4*>(p + j);
          o = fmaf(pp.x, __bfloat162float(vcol[(size_t)j * dh]), o);
          o = fmaf(pp.y, __bfloat162float(vcol[(size_t)(j + 1) * dh]), o);
          o = fmaf(pp.z, __bfloat162float(vcol[(size_t)(j + 2) * dh]), o);
          o = fmaf(pp.w, __bfloat162float(vcol[(size_t)(j + 3) * dh]), o);
        }
        for (; j < nk; ++j) o = fmaf(p[j], __bfloat162float(vcol[(size_t)j * dh]), o);
        if (m >= Mc) {
          const int jo = sm.rpos[m] - p_begin;
          if (jo >= 0 && jo < kAttnChunk)
            o = fmaf(sm.sp[m], __bfloat162float(sm.SV[(size_t)(m - Mc) * dh + dd]), o);
        }
        part_base[(size_t)(gh * kMaxRows + m) * (dh + kRecPad) + kRecPad + dd] = o;
      }
    } else {
      const int h2 = dh / 2;
      const int nrg = kGroupThreads / h2;    // 4 (dh 128) or 8 (dh 64)
      const int cp = tid % h2, rg = tid / h2;
      const int nr = M > rg ? (M - rg + nrg - 1) / nrg : 0;  // <= kMaxRows / 4
      float o[kMaxRows / 4][2];
#pragma unroll
      for (int r = 0; r < kMaxRows / 4; ++r) o[r][0] = o[r][1] = 0.f;
      const __nv_bfloat162* vcol = reinterpret_cast<const __nv_bfloat162*>(sm.V) + cp;
      int j = 0;
      for (; j + 4 <= nk; j += 4) {
        float2 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = __bfloat1622float2(vcol[(size_t)(j + q) * h2]);
#pragma unroll
        for (int r = 0; r < kMaxRows / 4; ++r) {
          if (r < nr) {
            const float4 p = *reinterpret_cast<const float4*>(sm.S + (size_t)(rg + r * nrg) * kAttnChunk + j);
            o[r][0] = fmaf(p.x, v[0].x, o[r][0]);
            o[r][1] = fmaf(p.x, v[0].y, o[r][1]);
            o[r][0] = fmaf(p.y, v[1].x, o[r][0]);
            o[r][1] = fmaf(p.y, v[1].y, o[r][1]);
            o[r][0] = fmaf(p.z, v[2].x, o[r][0]);
            o[r][1] = fmaf(p.z, v[2].y, o[r][1]);
            o[r][0] = fmaf(p.w, v[3].x, o[r][0]);
            o[r][1] = fmaf(p.w, v[3].y, o[r][1]);
          }
        }
      }
      for (; j < nk; ++j) {
        const float2 v = __bfloat1622float2(vcol[(size_t)j * h2]);
#pragma unroll
        for (int r = 0; r < kMaxRows / 4; ++r) {
          if (r < nr) {
            const float p = sm.S[(size_t)(rg + r * nrg) * kAttnChunk + j];
            o[r][0] = fmaf(p, v.x, o[r][0]);
            o[r][1] = fmaf(p, v.y, o[r][1]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kMaxRows / 4; ++r) {
        const int m = rg + r * nrg;
        if (r < nr && m >= Mc) {
          const int jo = sm.rpos[m] - p_begin;
          if (jo >= 0 && jo < kAttnChunk) {
            const __nv_bfloat162 sv =
                reinterpret_cast<const __nv_bfloat162*>(sm.SV + (size_t)(m - Mc) * dh)[cp];
            const float2 v = __bfloat1622float2(sv);
            o[r][0] = fmaf(sm.sp[m], v.x, o[r][0]);
            o[r][1] = fmaf(sm.sp[m], v.y, o[r][1]);
          }
        }
        if (r < nr) {
          const int rr = gh * kMaxRows + m;
          *reinterpret_cast<float2*>(part_base + (size_t)rr * (dh + kRecPad) + kRecPad + 2 * cp) =
              make_float2(o[r][0], o[r][1]);
        }
      }
    }
  }
  __threadfence();
  sync();
  if (tid == 0) {
    const unsigned prev = atomicAdd(a.counters + kvh, 1u);
    *flag = prev == (unsigned)(n_active - 1);
  }
  sync();
  const bool last = *flag != 0;
  if (last) {
    __threadfence();
    // (7) combine this head's chunks in chunk order.  Per row: w_c =
    // exp(m_c - max_c m_c), L = sum_c l_c w_c and O = sum_c o_c w_c, each sum
    // in chunk order.  All rows at once when their (m, l, w) fit in this
    // item's shared memory, else one row at a time.
    const float* hb = a.part + (size_t)kvh * nchunk_max * rows * (dh + kRecPad);
    const int R = G * M;
    float* CM = reinterpret_cast<float*>(sm.K);
    float* CL = CM + R * n_active;
    float* CW = CL + R * n_active;
    float* LR = CW + R * n_active;
    const size_t need = ((size_t)3 * R * n_active + R) * sizeof(float);
    if (need <= main_bytes(dh, nchunk_max)) {
      // The chunks' output vectors of a batch of rows go to shared memory with
      // 16-byte asynchronous copies, all in flight at once (thread t copies
      // piece t % (dh/4) of (row, chunk) records t / (dh/4), ...); the first
      // batch is requested before the (m, l) loads so that the two L2 round
      // trips overlap.  Then every output sums its chunks in chunk order.
      const size_t cs = (size_t)rows * (dh + kRecPad);
      const size_t used = ((size_t)3 * R * n_active + R + 3) & ~(size_t)3;  // floats, 16 B aligned
      float* OB = CM + used;
      const size_t row_floats = (size_t)n_active * dh;
      const int per_batch = (int)((main_bytes(dh, nchunk_max) / sizeof(float) - used) / row_floats);
      auto fetch = [&](int r0) {
        const int nb = min(per_batch, R - r0);
        const int h4 = dh / 4;
        const int q = tid % h4;
        for (int rc = tid / h4; rc < nb * n_active; rc += kGroupThreads / h4) {
          const int rb = rc / n_active, cc = rc % n_active;
          const int rr = r0 + rb;
          const int m = rr % M, r = (rr / M) * kMaxRows + m;
          if (cc <= sm.rpos[m] / kAttnChunk)
            cp_async16(OB + (size_t)rb * row_floats + (size_t)cc * dh + 4 * q,
                       hb + cc * cs + (size_t)r * (dh + kRecPad) + kRecPad + 4 * q);
        }
      };
      if (per_batch >= 1) fetch(0);
      for (int e = tid; e < R * n_active; e += kGroupThreads) {
        const int rr = e / n_active, cc = e % n_active;
        const int m = rr % M, r = (rr / M) * kMaxRows + m;
        if (cc <= sm.rpos[m] / kAttnChunk) {
          const float* pc = hb + ((size_t)cc * rows + r) * (dh + kRecPad);
          CM[e] = __ldcg(pc);
          CL[e] = __ldcg(pc + 1);
        }
      }
      sync();
      // each row's maximum, then every (row, chunk) weight in parallel, then
      // each row's sum in chunk order
      for (int rr = tid; rr < R; rr += kGroupThreads) {
        const int m = rr % M;
        const int nc = sm.rpos[m] / kAttnChunk + 1;
        const float* cm = CM + rr * n_active;
        float mx = -INFINITY;
        for (int cc = 0; cc < nc; ++cc) mx = fmaxf(mx, cm[cc]);
        LR[rr] = mx;
      }
      sync();
      for (int e = tid; e < R * n_active; e += kGroupThreads) {
        const int rr = e / n_active, cc = e % n_active;
        if (cc <= sm.rpos[rr % M] / kAttnChunk) CW[e] = expf(CM[e] - LR[rr]);
      }
      sync();
      for (int rr = tid; rr < R; rr += kGroupThreads) {
        const int nc = sm.rpos[rr % M] / kAttnChunk + 1;
        float L = 0.f;
        for (int cc = 0; cc < nc; ++cc) L = fmaf(CL[rr * n_active + cc], CW[rr * n_active + cc], L);
        LR[rr] = L;
      }
      sync();
      if (per_batch >= 1) {
        for (int r0 = 0; r0 < R; r0 += per_batch) {
          const int nb = min(per_batch, R - r0);
          if (r0 > 0) fetch(r0);
          cp_async_wait_all();
          sync();
          for (int e = tid; e < nb * dh; e += kGroupThreads) {
            const int rb = e / dh, dd = e % dh;
            const int rr = r0 + rb;
            const int m = rr % M, gh = rr / M;
            const int nc = sm.rpos[m] / kAttnChunk + 1;
            const float* w = CW + rr * n_active;
            const float* ob = OB + (size_t)rb * row_floats + dd;
            float O = 0.f;
            for (int cc = 0; cc < nc; ++cc) O = fmaf(ob[(size_t)cc * dh], w[cc], O);
            a.out[(size_t)m * ld_out + (size_t)(kvh * G + gh) * dh + dd] =
                __float2bfloat16_rn(O / LR[rr]);
          }
          sync();
        }
      } else {
        for (int e = tid; e < R * dh; e += kGroupThreads) {
          const int rr = e / dh, dd = e % dh;
          const int m = rr % M, gh = rr / M, r = gh * kMaxRows + m;
          const int nc = sm.rpos[m] / kAttnChunk + 1;
          const float* w = CW + rr * n_active;
          const float* ob = hb + (size_t)r * (dh + kRecPad) + kRecPad + dd;
          float O = 0.f;
          int cc = 0;
          for (; cc + 4 <= nc; cc += 4) {
            float o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) o[q] = __ldcg(ob + (size_t)(cc + q) * cs);
#pragma unroll
            for (int q = 0; q < 4; ++q) O = fmaf(o[q], w[cc + q], O);
          }
          for (; cc < nc; ++cc) O = fmaf(__ldcg(ob + (size_t)cc * cs), w[cc], O);
          a.out[(size_t)m * ld_out + (size_t)(kvh * G + gh) * dh + dd] =
              __float2bfloat16_rn(O / LR[rr]);
        }
        sync();
      }
    } else {
      for (int rr = 0; rr < R; ++rr) {
        const int m = rr % M, gh = rr / M, r = gh * kMaxRows + m;
        const int nc = sm.rpos[m] / kAttnChunk + 1;
        for (int cc = tid; cc < nc; cc += kGroupThreads) {
          const float* pc = hb + ((size_t)cc * rows + r) * (dh + kRecPad);
          sm.cm[cc] = __ldcg(pc);
          sm.cl[cc] = __ldcg(pc + 1);
        }
        sync();
        float mx = -INFINITY;
        for (int cc = 0; cc < nc; ++cc) mx = fmaxf(mx, sm.cm[cc]);
        for (int cc = tid; cc < nc; cc += kGroupThreads) sm.cw[cc] = expf(sm.cm[cc] - mx);
        sync();
        float L = 0.f;
        for (int cc = 0; cc < nc; ++cc) L = fmaf(sm.cl[cc], sm.cw[cc], L);
        for (int dd = tid; dd < dh; dd += kGroupThreads) {
          float O = 0.f;
          for (int cc = 0; cc < nc; ++cc)
            O = fmaf(__ldcg(hb + ((size_t)cc * rows + r) * (dh + kRecPad) + kRecPad + dd), sm.cw[cc], O);
          a.out[(size_t)m * ld_out + (size_t)(kvh * G + gh) * dh + dd] =
              __float2bfloat16_rn(O / L);
        }
        sync();
      }
    }
    if (tid == 0) a.counters[kvh] = 0u;
  }
  // the next item's bulk copies overwrite this item's shared memory
  fence_proxy_async_smem();
  sync();
  return last;
}

// A whole work item: issue() then body().
template <class Sync>
SSD_DI bool item(const AttnArgs& a, int M, int ns, int pos0, int item, const Smem& sm,
                 uint64_t* bar, uint32_t& phase, int* flag, int tid, Sync sync) {
  issue(a, M - ns, pos0, item, sm, bar, tid);
  return body(a, M, ns, pos0, item, sm, bar, phase, flag, tid, sync);
}

}  // namespace attn
}  // namespace ssd
