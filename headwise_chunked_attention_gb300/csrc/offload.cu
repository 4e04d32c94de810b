// libupipe host side of the offload of block inputs to host memory and their
// prefetch back (include/upipe.h, upipe_offload / upipe_prefetch /
// upipe_copy_join).  The pages' memory stack moves each transformer block's
// input off the GPU while it is not needed and prefetches it before the
// backward reaches that block, so the copies hide under compute (memeeeeeex.com
// article, the stack section on CPU offload; aipmzone.com article; liquidgold.cc
// talk transcript).  Each copy runs on a library-owned copy stream of the
// device, after everything enqueued on the caller's stream so far (an event
// orders it after the producer), as one cudaMemcpyAsync; the ticket it returns
// is the event recorded after the copy, which upipe_copy_join makes the
// consumer's stream wait on and then releases.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/upipe.h"
#include "internal.h"

namespace upipe {
namespace {

constexpr int kMaxCopyDevices = 64;
cudaStream_t g_copy_stream[kMaxCopyDevices] = {};
std::mutex g_copy_mu;

// the current device's copy stream, created on first use
int copy_stream(cudaStream_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxCopyDevices)
    return UPIPE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_copy_mu);
  if (!g_copy_stream[dev] &&
      cudaStreamCreateWithFlags(&g_copy_stream[dev], cudaStreamNonBlocking) != cudaSuccess) {
    g_copy_stream[dev] = nullptr;
    return UPIPE_ERR_CUDA;
  }
  *out = g_copy_stream[dev];
  return UPIPE_OK;
}

// kind of memory behind p: 1 device memory of the current device, 2 page-
// locked host memory, 0 anything else (pageable host memory, managed memory,
// another device's memory)
int memory_kind(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (a.type == cudaMemoryTypeDevice) {
    int dev = -1;
    return (cudaGetDevice(&dev) == cudaSuccess && dev == a.device) ? 1 : 0;
  }
  return a.type == cudaMemoryTypeHost ? 2 : 0;
}

int start_copy(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, void* stream,
               void** ticket) {
  if (!ticket) return UPIPE_ERR_INVALID_ARG;
  *ticket = nullptr;
  if (!dst || !src || bytes == 0) return UPIPE_ERR_INVALID_ARG;
  const bool to_host = kind == cudaMemcpyDeviceToHost;
  if (memory_kind(to_host ? src : dst) != 1 || memory_kind(to_host ? dst : src) != 2)
    return UPIPE_ERR_INVALID_ARG;
  cudaStream_t cs = nullptr;
  const int rc = copy_stream(&cs);
  if (rc != UPIPE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaEvent_t ready = nullptr, done = nullptr;
  if (cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) != cudaSuccess)
    return UPIPE_ERR_CUDA;
  if (cudaEventCreateWithFlags(&done, cudaEventDisableTiming) != cudaSuccess) {
    cudaEventDestroy(ready);
    return UPIPE_ERR_CUDA;
  }
  // the copy starts after the caller's stream has produced the source
  const bool ok = cudaEventRecord(ready, st) == cudaSuccess &&
                  cudaStreamWaitEvent(cs, ready, 0) == cudaSuccess &&
                  cudaMemcpyAsync(dst, src, bytes, kind, cs) == cudaSuccess &&
                  cudaEventRecord(done, cs) == cudaSuccess;
  cudaEventDestroy(ready);   // allowed while pending: released on completion
  if (!ok) {
    cudaEventDestroy(done);
    return UPIPE_ERR_CUDA;
  }
  *ticket = done;
  return UPIPE_OK;
}

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" int upipe_offload(const void* dev_src, void* host_dst, size_t bytes, void* stream,
                             void** ticket) {
  NvtxRange range("upipe_offload");
  return start_copy(host_dst, dev_src, bytes, cudaMemcpyDeviceToHost, stream, ticket);
}

extern "C" int upipe_prefetch(const void* host_src, void* dev_dst, size_t bytes, void* stream,
                              void** ticket) {
  NvtxRange range("upipe_prefetch");
  return start_copy(dev_dst, host_src, bytes, cudaMemcpyHostToDevice, stream, ticket);
}

extern "C" int upipe_copy_join(void* ticket, void* stream) {
  if (!ticket) return UPIPE_ERR_INVALID_ARG;
  cudaEvent_t done = static_cast<cudaEvent_t>(ticket);
  const bool ok = cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), done, 0) == cudaSuccess;
  cudaEventDestroy(done);
  return ok ? UPIPE_OK : UPIPE_ERR_CUDA;
}
