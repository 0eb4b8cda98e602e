// qgemm_w4a16_host: the dense W4A16 GEMM with X and Y in (page-locked) host memory.
//
// The rows are cut into up to sixteen chunks of at least 512 rows (measured on a GB300: the
// more chunks, the less of the first copy in and the last copy out stays exposed, down to
// chunks whose GEMM runs markedly less efficiently).  Each chunk's X rows are copied in on a library
// stream, multiplied on the caller's stream, and its Y rows copied out on a second library
// stream.  Two device staging buffers alternate between chunks, so that while chunk i runs
// on the tensor cores, chunk i + 1 is being copied in and chunk i - 1 copied out.  Events
// order each buffer's reuse after its previous readers.  The caller's stream waits for the
// last copy out, so work ordered after the call on that stream sees Y in host memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "qgemm.h"

namespace {

constexpr int kMaxDevices = 64;
#ifndef QGEMM_HOST_MIN_ROWS
#define QGEMM_HOST_MIN_ROWS 512
#endif
#ifndef QGEMM_HOST_CHUNKS
#define QGEMM_HOST_CHUNKS 16
#endif
constexpr int64_t kMinChunkRows = QGEMM_HOST_MIN_ROWS;  // shorter chunks lose GEMM efficiency
constexpr int kMaxChunks = QGEMM_HOST_CHUNKS;

// Library streams and events of one device, created on first use and kept until exit.
struct HostPipe {
  bool init = false;
  bool ok = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, copied_in[2] = {}, computed[2] = {}, copied_out[2] = {};
  std::mutex mu;                          // one call enqueues at a time (events are reused)
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_init_mu;

HostPipe* pipe_of_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_init_mu);
  HostPipe& p = g_pipe[dev];
  if (!p.init) {
    p.init = true;
    bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess;
    for (int b = 0; b < 2 && ok; ++b)
      ok = cudaEventCreateWithFlags(&p.copied_in[b], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.computed[b], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.copied_out[b], cudaEventDisableTiming) == cudaSuccess;
    p.ok = ok;
  }
  return p.ok ? &p : nullptr;
}

int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

// Rows per chunk for M rows: all of them up to kMinChunkRows, else M / kMaxChunks rounded
// up to a multiple of 256, at least kMinChunkRows.  Non-decreasing in M, so the staging
// size for M_max covers every smaller M.
int64_t chunk_rows(int64_t M) {
  if (M <= kMinChunkRows) return M;
  const int64_t q = round_up((M + kMaxChunks - 1) / kMaxChunks, 256);
  return q < kMinChunkRows ? kMinChunkRows : q;
}

int64_t x_stage_bytes(const qgemm_wdesc* d, int64_t rows) { return round_up(rows * d->K * 2, 256); }
int64_t y_stage_bytes(const qgemm_wdesc* d, int64_t rows) { return round_up(rows * d->N * 2, 256); }

}  // namespace

extern "C" {

size_t qgemm_host_staging_bytes(const qgemm_wdesc* desc, int64_t M_max) {
  if (qgemm_check_desc(desc) != QGEMM_OK || M_max <= 0) return 0;
  const int64_t rows = chunk_rows(M_max);
  return size_t(2 * (x_stage_bytes(desc, rows) + y_stage_bytes(desc, rows)));
}

qgemm_status qgemm_w4a16_host(const qgemm_wdesc* desc, const void* packed, const void* X_host,
                              int64_t M, int64_t ldx, const float* chan_scale, const float* bias,
                              void* Y_host,
                              int64_t ldy, void* staging, size_t staging_bytes, void* ws,
                              size_t ws_bytes, void* stream) {
  if (qgemm_check_desc(desc) != QGEMM_OK) return QGEMM_ERR_INVALID_ARG;
  if (desc->afmt != QGEMM_A_BF16) return QGEMM_ERR_INVALID_ARG;
  if (M < 0 || X_host == nullptr || Y_host == nullptr || ldx < desc->K || ldy < desc->N)
    return QGEMM_ERR_INVALID_ARG;
  if (M == 0) return QGEMM_OK;
  if (staging == nullptr || staging_bytes < qgemm_host_staging_bytes(desc, M))
    return QGEMM_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(staging) % 256 != 0) return QGEMM_ERR_ALIGNMENT;
  HostPipe* p = pipe_of_current_device();
  if (p == nullptr) return QGEMM_ERR_NO_DEVICE;

  const int64_t K = desc->K, N = desc->N;
  const int64_t rows = chunk_rows(M);
  const int64_t nch = (M + rows - 1) / rows;
  uint8_t* base = static_cast<uint8_t*>(staging);
  uint8_t* xs[2] = {base, base + x_stage_bytes(desc, rows)};
  uint8_t* ys[2] = {base + 2 * x_stage_bytes(desc, rows),
                    base + 2 * x_stage_bytes(desc, rows) + y_stage_bytes(desc, rows)};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint8_t* xh = static_cast<const uint8_t*>(X_host);
  uint8_t* yh = static_cast<uint8_t*>(Y_host);

  if (nch == 1) {
    // nothing to overlap: copy in, multiply and copy out in order on the caller's stream
    if (cudaMemcpy2DAsync(xs[0], size_t(K) * 2, xh, size_t(ldx) * 2, size_t(K) * 2, size_t(M),
                          cudaMemcpyHostToDevice, st) != cudaSuccess)
      return QGEMM_ERR_CUDA;
    const qgemm_status s = qgemm_w4a16(desc, packed, xs[0], M, K, chan_scale, bias, ys[0], N, ws,
                                       ws_bytes, stream);
    if (s != QGEMM_OK) return s;
    if (cudaMemcpy2DAsync(yh, size_t(ldy) * 2, ys[0], size_t(N) * 2, size_t(N) * 2, size_t(M),
                          cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return QGEMM_ERR_CUDA;
    return QGEMM_OK;
  }
  std::lock_guard<std::mutex> lk(p->mu);
  // Nothing of this call starts before the work already ordered on the caller's stream.
  if (cudaEventRecord(p->start, st) != cudaSuccess ||
      cudaStreamWaitEvent(p->in, p->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(p->out, p->start, 0) != cudaSuccess)
    return QGEMM_ERR_CUDA;
  for (int64_t i = 0; i < nch; ++i) {
    const int b = int(i & 1);
    const int64_t r0 = i * rows;
    const int64_t m = (M - r0) < rows ? (M - r0) : rows;
    // copy in, once the GEMM of chunk i - 2 has read this buffer
    if (i >= 2 && cudaStreamWaitEvent(p->in, p->computed[b], 0) != cudaSuccess) return QGEMM_ERR_CUDA;
    if (cudaMemcpy2DAsync(xs[b], size_t(K) * 2, xh + r0 * ldx * 2, size_t(ldx) * 2,
                          size_t(K) * 2, size_t(m), cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
        cudaEventRecord(p->copied_in[b], p->in) != cudaSuccess)
      return QGEMM_ERR_CUDA;
    // multiply, once X is in and the copy out of chunk i - 2 has read this Y buffer
    if (cudaStreamWaitEvent(st, p->copied_in[b], 0) != cudaSuccess) return QGEMM_ERR_CUDA;
    if (i >= 2 && cudaStreamWaitEvent(st, p->copied_out[b], 0) != cudaSuccess) return QGEMM_ERR_CUDA;
    const qgemm_status s = qgemm_w4a16(desc, packed, xs[b], m, K, chan_scale, bias, ys[b], N, ws,
                                       ws_bytes, stream);
    if (s != QGEMM_OK) return s;
    if (cudaEventRecord(p->computed[b], st) != cudaSuccess) return QGEMM_ERR_CUDA;
    // copy out
    if (cudaStreamWaitEvent(p->out, p->computed[b], 0) != cudaSuccess ||
        cudaMemcpy2DAsync(yh + r0 * ldy * 2, size_t(ldy) * 2, ys[b], size_t(N) * 2, size_t(N) * 2,
                          size_t(m), cudaMemcpyDeviceToHost, p->out) != cudaSuccess ||
        cudaEventRecord(p->copied_out[b], p->out) != cudaSuccess)
      return QGEMM_ERR_CUDA;
  }
  // the caller's stream resumes after the last copy out (the out stream runs in order)
  if (cudaStreamWaitEvent(st, p->copied_out[(nch - 1) & 1], 0) != cudaSuccess) return QGEMM_ERR_CUDA;
  return QGEMM_OK;
}

}  // extern "C"
