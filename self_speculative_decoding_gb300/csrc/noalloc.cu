// ssd_op_linear_noalloc: the small-M GEMV of ssd_op_linear for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they need the
// projection: a serving runtime that reserved all of the GPU's memory for its
// own pool when it started, or a latency-critical step that must not risk an
// out-of-memory failure or the device-wide synchronisation an allocation or
// free can trigger.  ssd_op_linear takes its scratch (the partial sums of row
// groups split across CTAs, and their completion counters) from the
// stream-ordered allocator; this variant takes it from a fixed array that the
// library reserves in device memory on every GPU that loads it, and calls no
// allocating routine at all.
#include <mutex>
#include <string>

#include "../../include/ssd_ops.h"
#include "kernels.cuh"

using namespace ssd;

namespace {

// Largest row count accepted: R <= 8192 needs at most 1 MiB of partial sums
// (512 row groups, two segments each) and 2.1 KiB of counters.
constexpr int kNoAllocMaxRows = 8192;
constexpr size_t kPartOffset = 0;
constexpr size_t kPartCapacity = 1024 * 1024;
constexpr size_t kCounterOffset = kPartCapacity;
constexpr size_t kCounterCapacity = 4096;
constexpr size_t kErrOffset = kCounterOffset + kCounterCapacity;
constexpr size_t kNoAllocBytes = kErrOffset + 256;  // 1 MiB + 4.25 KiB

// Held by every GPU that loads the library until the process exits.
static __device__ __align__(256) unsigned char g_linear_scratch[kNoAllocBytes];

// Device address of g_linear_scratch, per device.  In host code the symbol
// names a host-side stand-in, so the address is looked up once per device
// with that device current.  cudaDeviceReset destroys the context that holds
// the array, so the cached address is not valid after it.
std::mutex g_mu;
void* g_scratch_addr[64] = {};

thread_local std::string g_err;

ssd_status fail(ssd_status s, const std::string& m) {
  g_err = m;
  return s;
}

}  // namespace

extern "C" {

const char* ssd_op_linear_noalloc_last_error(void) { return g_err.c_str(); }

ssd_status ssd_op_linear_noalloc(const void* W, int32_t R, int32_t K, const void* act, int32_t M,
                                 float* y, void* stream) {
  if (!W || !act || !y || (((uintptr_t)W | (uintptr_t)act | (uintptr_t)y) & 15u))
    return fail(SSD_ERR_INVALID_ARG, "W, act and y must be non-null and 16-byte aligned");
  if (R <= 0 || R % 16 || K <= 0 || K % 32 || M < 1 || M > kMaxRows)
    return fail(SSD_ERR_INVALID_ARG, "need R % 16 == 0, K % 32 == 0, 1 <= M <= 16");
  if (R > kNoAllocMaxRows)
    return fail(SSD_ERR_CAPACITY,
                "ssd_op_linear_noalloc accepts at most 8192 rows (its fixed scratch is 1 MiB)");
  const GemvScratch gs = gemv_scratch(R, K, EPI_STORE);
  if (gs.part_floats * sizeof(float) > kPartCapacity ||
      gs.counters * sizeof(unsigned) > kCounterCapacity)
    return fail(SSD_ERR_CAPACITY, "shape needs more scratch than the fixed array holds");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SSD_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(SSD_ERR_INVALID_ARG, "device index out of range");
  unsigned char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_linear_scratch);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SSD_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      }
      g_scratch_addr[dev] = p;
    }
    base = static_cast<unsigned char*>(g_scratch_addr[dev]);
  }
  cudaStream_t s = (cudaStream_t)stream;
  // The counters (and the error word) must start at zero; the array keeps
  // whatever the previous call left there.
  e = cudaMemsetAsync(base + kCounterOffset, 0, kCounterCapacity + 256, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(SSD_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
  }

  LinearArgs a;
  a.W0 = (const bf16*)W;
  a.R = R;
  a.K = K;
  a.act = (const bf16*)act;
  a.M_static = M;
  a.y = y;
  a.part = reinterpret_cast<float*>(base + kPartOffset);
  a.counter = reinterpret_cast<unsigned*>(base + kCounterOffset);
  a.err = reinterpret_cast<int*>(base + kErrOffset);
  e = launch_gemv(IN_BF16, EPI_STORE, a, s, false);
  if (e != cudaSuccess) {
    cudaGetLastError();  // the error is reported here, not to the caller's next check
    return fail(SSD_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e));
  }
  return SSD_OK;
}

}  // extern "C"
