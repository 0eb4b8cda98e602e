// qgemm_w4a16_noalloc: the dense W4A16 GEMM without a caller-provided workspace.
//
// Some callers cannot allocate device memory for a workspace: a serving framework whose
// allocator has already reserved the whole device and hands out no extra buffers, or a
// latency-critical caller that must not trigger the device-wide synchronization that
// cudaMalloc/cudaFree can cause.  For them the split-K scratch lives in one file-scope
// device array, sized at build time, that every GPU loading this library keeps until the
// process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"
#include "qgemm.h"

namespace {

// The shared split-K scratch (partial sums and tile counters) of qgemm_w4a16_noalloc.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QGEMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once per device.
// In host code `g_noalloc_scratch` names a host-side stand-in, never the device memory,
// so the address must come from cudaGetSymbolAddress with that device current.
qgemm_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return QGEMM_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return QGEMM_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return QGEMM_OK;
}

}  // namespace

extern "C" qgemm_status qgemm_w4a16_noalloc(const qgemm_wdesc* desc, const void* packed,
                                            const void* X, int64_t M, int64_t ldx,
                                            const float* chan_scale, void* Y, int64_t ldy,
                                            void* stream) {
  // This call's own schedule decides the scratch it needs; every argument is checked
  // before anything is enqueued.
  int64_t need = 0, counter_off = 0, counter_bytes = 0;
  qgemm_status s = qgemm::dense_a16_scratch(desc, packed, X, M, ldx, chan_scale, Y, ldy,
                                            int64_t(QGEMM_NOALLOC_SCRATCH_BYTES), &need,
                                            &counter_off, &counter_bytes);
  if (s != QGEMM_OK || M == 0) return s;
  if (need > int64_t(QGEMM_NOALLOC_SCRATCH_BYTES)) return QGEMM_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    if ((s = scratch_address(&scratch)) != QGEMM_OK) return s;
    // The array keeps whatever the previous call left; the partial-sum slots are written
    // before they are read, but the tile arrival counters must start at zero.
    if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + counter_off, 0,
                        size_t(counter_bytes), static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return QGEMM_ERR_CUDA;
  }
  return qgemm_w4a16(desc, packed, X, M, ldx, chan_scale, nullptr, Y, ldy, scratch, size_t(need),
                     stream);
}
