// Device helpers shared by the libssd kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define SSD_HD __host__ __device__ __forceinline__
#define SSD_DI __device__ __forceinline__

namespace ssd {

typedef __nv_bfloat16 bf16;

// Per-device one-time host set-up (a kernel's dynamic shared-memory limit
// applies to the device that is current when it is set): the index of the
// current device into tables of kDeviceSlots entries, or -1 for a device
// beyond them (whose set-up then runs on every call).
constexpr int kDeviceSlots = 64;
inline int device_slot() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kDeviceSlots) return -1;
  return d;
}

// Largest number of rows (token positions) one pass processes together.
constexpr int kMaxRows = 16;
// Attention key chunk: keys are split into fixed absolute chunks of this many
// positions; partial softmax statistics are combined in chunk order.  The
// chunking depends only on absolute positions, never on how many query rows
// a pass carries.
constexpr int kAttnChunk = 64;
// Columns of the residual stream covered by one sum-of-squares partial (one
// 16-row group of the producing projection).
constexpr int kSsGroup = 16;
// Dynamic verification (SWIFT §4.2): at most this many sibling candidates per
// round, each a side row of the passes that carry it.
constexpr int kMaxSide = 8;

// Per-row logits summary (same layout as ssd_row_stats in ssd_ops.h).
struct RowStats {
  int32_t top1, top2, sample, pad;
  float z1, z2, lse, conf, lse_t, pad2[3];
};
static_assert(sizeof(RowStats) == 48, "RowStats layout");

// Decoding state kept in device memory so that captured CUDA graphs can be
// replayed for every step: kernels read the pass shape (rows, first
// position, input tokens) from here instead of from launch arguments.
struct DevState {
  int32_t n;        // committed length; tokens[n-1] is pending
  int32_t round;    // decoding round counter (Philox counter word 2)
  int32_t j;        // draft steps run in the current round
  int32_t d;        // draft tokens kept in the current round
  int32_t stop;     // the confidence stop fired in the current round
  int32_t M;        // rows of the current pass (chain rows, then side rows)
  int32_t pos0;     // position of row 0 of the current pass
  int32_t slot;     // output slot of the current pass (draft step index)
  int32_t n_emitted;
  int32_t accepted;
  int32_t err;      // non-zero: a device-side wait gave up (its code)
  int32_t ns;       // side rows of the current pass (its last ns rows)
  int32_t side0;    // sibling index (side K/V slot) of the first side row
  int32_t n_sib;    // siblings recorded in the current round
  int32_t sib_acc;  // sibling taken by the last acceptance (-1: none)
  int32_t sib_pos;  // its position
  int32_t in_tok[kMaxRows];
  int32_t draft_tok[kMaxRows];
  float draft_conf[kMaxRows];
  int32_t emitted[kMaxRows + 1];
  int32_t sib_depth[kMaxSide];  // sibling i stands for draft y_j, j = sib_depth[i] (position n + j)
  int32_t sib_tok[kMaxSide];
  int32_t side_pos[kMaxSide];   // positions of the current pass's side rows
  // device-side generation loop: its target length, the kept drafts of the
  // last accepted round, and running counts of the loop's work
  int32_t target_n;
  int32_t last_d;
  int32_t acc_rounds, acc_drafted, acc_accepted, acc_emitted;
  int32_t acc_steps, acc_extra, acc_side_rows, acc_side_acc;
  // debug builds (SSD_DEBUG_CHECKS): the value that failed the bounds check
  // recorded in err (codes >= kDbgCodeBase), and the bounds the checks use
  int32_t err_val;
  int32_t vocab, max_seq;
  int32_t pad2[2];
};
static_assert(sizeof(DevState) % 16 == 0, "DevState layout");

// Debug builds (compiled with -DSSD_DEBUG_CHECKS): device-side bounds checks
// on token ids, KV positions and pass row counts.  A failed check records
// its code and the offending value in the state's error words (the first
// failure wins) and the caller skips or clamps the access; nothing traps.
// Release builds compile every check to `true`.
constexpr int kDbgCodeBase = 100;
enum DbgCode {
  DBG_TOKEN = 101,     // a token id outside [0, vocab)
  DBG_POS = 102,       // a K/V position outside [0, max_seq)
  DBG_ROWS = 103,      // a pass row count outside [1, 16]
  DBG_COMMIT = 104,    // committed tokens beyond max_seq
};
#ifdef SSD_DEBUG_CHECKS
SSD_DI bool dbg_check(DevState* st, bool ok, int code, int value) {
  if (ok) return true;
  if (st && atomicCAS(&st->err, 0, code) == 0) st->err_val = value;
  return false;
}
// The same for kernels given the error words (err, err_val) instead of the
// state.
SSD_DI bool dbg_check_words(int* err, int* err_val, bool ok, int code, int value) {
  if (ok) return true;
  if (err && atomicCAS(err, 0, code) == 0 && err_val) *err_val = value;
  return false;
}
#define SSD_CHECK(st, cond, code, value) ::ssd::dbg_check((st), (cond), (code), (int)(value))
#define SSD_CHECK_W(err, err_val, cond, code, value) \
  ::ssd::dbg_check_words((err), (err_val), (cond), (code), (int)(value))
#else
#define SSD_CHECK(st, cond, code, value) true
#define SSD_CHECK_W(err, err_val, cond, code, value) true
#endif


// ---------------------------------------------------------------------------
// loads / stores

// Weights are read exactly once per pass: keep them out of L1.
SSD_DI uint4 ld_stream_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

SSD_DI uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

SSD_DI float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
SSD_DI float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// acc + sum_i q_i k_i over 8 elements (q = qa, qb; k = 8 bf16), in element order.
SSD_DI float dot8(const float4& qa, const float4& qb, const uint4& k, float acc) {
  acc = fmaf(qa.x, bf16_lo(k.x), acc);
  acc = fmaf(qa.y, bf16_hi(k.x), acc);
  acc = fmaf(qa.z, bf16_lo(k.y), acc);
  acc = fmaf(qa.w, bf16_hi(k.y), acc);
  acc = fmaf(qb.x, bf16_lo(k.z), acc);
  acc = fmaf(qb.y, bf16_hi(k.z), acc);
  acc = fmaf(qb.z, bf16_lo(k.w), acc);
  acc = fmaf(qb.w, bf16_hi(k.w), acc);
  return acc;
}

// D += A * B on the tensor cores, m16n8k16, bf16 inputs, fp32 accumulate.
SSD_DI void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                     uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Programmatic dependent launch: wait for the preceding kernel's memory, and
// let the following kernel start its launch.
SSD_DI void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
SSD_DI void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

SSD_DI int rows_of(int M_static, const int32_t* M_dev) { return M_dev ? *M_dev : M_static; }

// ---------------------------------------------------------------------------
// mbarrier + bulk (TMA) copies

SSD_DI uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SSD_DI void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

SSD_DI void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same memory.
SSD_DI void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

SSD_DI void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Bulk global -> shared copy (bytes and both addresses multiples of 16),
// completing on `bar`.
SSD_DI void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 16-byte asynchronous global -> shared copy through L2 (both addresses
// 16-byte aligned); completes at cp_async_wait_all().
SSD_DI void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
SSD_DI void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Closes this thread's group of cp.async copies issued since the last commit.
SSD_DI void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's committed groups are still in flight.
template <int N>
SSD_DI void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Bulk prefetch of global memory into L2 (address and size multiples of 16).
SSD_DI void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Bounded wait for the phase with the given parity; false if it never
// completed (the caller records an error instead of hanging).
SSD_DI bool mbar_wait_n(uint64_t* bar, uint32_t parity, int polls) {
  const uint32_t addr = smem_addr(bar);
  for (int i = 0; i < polls; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
SSD_DI bool mbar_wait(uint64_t* bar, uint32_t parity) { return mbar_wait_n(bar, parity, 1 << 22); }

// Adds v to a global counter with release semantics (no value returned).
SSD_DI void red_release_add(unsigned* c, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(c), "r"(v) : "memory");
}

// Bounded wait until a global counter reaches target (acquire); false if it
// never did (the caller records an error instead of hanging).
SSD_DI bool wait_count_n(const unsigned* c, unsigned target, int polls) {
  for (int i = 0; i < polls; ++i) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    if (v >= target) return true;
  }
  return false;
}
SSD_DI bool wait_count(const unsigned* c, unsigned target) { return wait_count_n(c, target, 1 << 24); }

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64 multiplies on a 128-bit counter with a Weyl-bumped 64-bit key.

SSD_DI uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Uniform in (0, 1), exact in fp32: ((r >> 9) + 0.5) * 2^-23.
SSD_DI float u01(uint32_t r) { return (float(r >> 9) + 0.5f) * (1.0f / 8388608.0f); }

SSD_DI uint32_t word_of(uint4 v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Gumbel noise -log(-log u) for vocabulary entry v at (pos, round, stream).
SSD_DI float gumbel_at(uint64_t seed, int v, int pos, int round, int stream) {
  const uint4 r = philox4x32_10(make_uint4((uint32_t)(v >> 2), (uint32_t)pos, (uint32_t)round,
                                           (uint32_t)stream),
                                (uint32_t)seed, (uint32_t)(seed >> 32));
  return -logf(-logf(u01(word_of(r, v & 3))));
}

// The Gumbel noise of entries 4 b .. 4 b + 3 from one Philox call (the four
// words of counter block b): g[w] == gumbel_at(seed, 4 b + w, ...).
SSD_DI void gumbel4(uint64_t seed, int b, int pos, int round, int stream, float (&g)[4]) {
  const uint4 r = philox4x32_10(make_uint4((uint32_t)b, (uint32_t)pos, (uint32_t)round,
                                           (uint32_t)stream),
                                (uint32_t)seed, (uint32_t)(seed >> 32));
  g[0] = -logf(-logf(u01(r.x)));
  g[1] = -logf(-logf(u01(r.y)));
  g[2] = -logf(-logf(u01(r.z)));
  g[3] = -logf(-logf(u01(r.w)));
}

// Packed weight unit (16 rows x 32 columns bf16, 1 KB): each 8-row half is
// row-major with 64-byte rows whose four 16-byte chunks are stored in the
// 64-byte swizzle order (chunk c of row r at position c ^ ((r >> 1) & 3)),
// which the tensor cores' shared-memory descriptors read directly.  Byte
// offset, within a half, of the chunk that mma.sync lane L = 4g + c needs
// (row g, columns 8c .. 8c + 7).
SSD_DI int unit_slot(int lane) { return (lane ^ ((lane >> 3) & 3)) << 4; }

// Element offset of (row t, column k) of a [T][K] bf16 matrix stored in the
// packed unit layout (units ordered (t / 16, k / 32); T padded to 16 rows).
// The many-row projection reads its activations in this layout, one bulk
// copy per unit.
SSD_HD size_t packed_off(int t, int k, int K) {
  const int r = t & 15;
  return ((size_t)(t >> 4) * (size_t)(K >> 5) + (size_t)(k >> 5)) * 512 + (size_t)r * 32 +
         (size_t)(((((k >> 3) & 3) ^ (((r & 7) >> 1) & 3))) << 3) + (size_t)(k & 7);
}

// Total order used by every argmax: larger value first, then lower index.
SSD_DI bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

}  // namespace ssd
