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
  if (qgemm_check_desc(desc) != QGEMM_OK) return QGEMM_ERR_INVALID_ARG;
  if (M <= 0)   // M == 0 is a no-op, M < 0 an argument error: no scratch involved
    return qgemm_w4a16(desc, packed, X, M, ldx, chan_scale, Y, ldy, nullptr, 0, stream);
  const size_t need = qgemm_workspace_bytes(desc, M);
  if (need > size_t(QGEMM_NOALLOC_SCRATCH_BYTES)) return QGEMM_ERR_WORKSPACE;
  void* scratch = nullptr;
  const qgemm_status s = scratch_address(&scratch);
  if (s != QGEMM_OK) return s;
  // The array keeps whatever the previous call left; the split-K tile counters must
  // start at zero.
  if (need > 0 && cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return QGEMM_ERR_CUDA;
  return qgemm_w4a16(desc, packed, X, M, ldx, chan_scale, Y, ldy, scratch,
                     size_t(QGEMM_NOALLOC_SCRATCH_BYTES), stream);
}
