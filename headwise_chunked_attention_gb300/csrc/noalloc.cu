// upipe_attn_fwd_noalloc: the layer forward for callers that cannot allocate
// device memory (see include/upipe.h).  Its workspace is one file-scope
// static __device__ array of UPIPE_STATIC_SCRATCH_BYTES; the layer forward
// runs on it with every launch on the caller's stream (it creates no events
// and uses no side stream).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/upipe.h"
#include "internal.h"

namespace {

// The scratch every call of upipe_attn_fwd_noalloc uses, on every device that
// loads this library (held until the process exits).
static __device__ __align__(256) unsigned char g_static_scratch[UPIPE_STATIC_SCRATCH_BYTES];

// In host code g_static_scratch names a host-side stand-in, not device memory:
// its device address is looked up once per device, with that device current.
constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return UPIPE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return UPIPE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return UPIPE_OK;
}

}  // namespace

extern "C" int upipe_attn_fwd_noalloc(const upipe_shape_t* shape, const upipe_bf16* x,
                                      const upipe_bf16* Wq, const upipe_bf16* Wk,
                                      const upipe_bf16* Wv, const upipe_bf16* Wo,
                                      const float* q_norm_w, const float* k_norm_w, float* out,
                                      float* lse, void* stream) {
  const size_t need = upipe_workspace_bytes(shape, 0);
  if (need == 0)  // invalid or unsupported shape: report its own code, launch nothing
    return upipe::attn_fwd_unforked(shape, x, Wq, Wk, Wv, Wo, q_norm_w, k_norm_w, out, lse,
                                    nullptr, 0, stream);
  if (need > (size_t)UPIPE_STATIC_SCRATCH_BYTES) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const int rc = static_scratch(&scratch);
  if (rc != UPIPE_OK) return rc;
  // Nothing in the scratch has to start at zero: every byte the forward reads
  // is written earlier in the same call.  The forward is given exactly the
  // minimal (mode 0) workspace size, so it always takes the mode-0 layout
  // whatever else would fit in the array.
  return upipe::attn_fwd_unforked(shape, x, Wq, Wk, Wv, Wo, q_norm_w, k_norm_w, out, lse, scratch,
                                  need, stream);
}
