// libupipe host side of the sequence-tiled cross-entropy loss (include/upipe.h,
// upipe_loss_*): the language-model loss over a vocabulary of V words computed
// over tiles of ``tile_rows`` tokens, so that no [S, V] logits buffer exists
// (the pages' stack tiles the loss along the sequence, as it does the MLPs:
// memeeeeeex.com article, the stack section on Arctic sequence-length
// training; liquidgold.cc talk transcript).  Per tile of rows R:
//   forward   z = h_R W^T never stored: the GEMM epilogue keeps, per row and
//             vocabulary tile, the (max, sum of exp) partial of the
//             log-sum-exp and the target's logit (EPI_LSE_PART); one small
//             kernel combines the partials into lse_R and the losses
//   backward  z recomputed; dz = scale (softmax - onehot) in bf16
//             (EPI_DLOGITS); dh_R = dz W; dW += dz^T h_R (split-K)
// The tile's partials (forward) or dz (backward) are the workspace, reused
// by every tile.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <initializer_list>

#include "../../include/upipe.h"
#include "internal.h"

namespace upipe {
namespace {

constexpr size_t kLossAlign = 256;
inline size_t loss_align(size_t v) { return (v + kLossAlign - 1) / kLossAlign * kLossAlign; }

struct LossLayout {
  size_t part, zt, dz, total;
};

int check_loss_shape(const upipe_loss_shape_t* sh) {
  if (!sh) return UPIPE_ERR_INVALID_ARG;
  if (sh->S < 1 || sh->S > (int64_t)INT32_MAX - 256 || sh->hidden <= 0 || sh->vocab <= 0 ||
      sh->tile_rows <= 0)
    return UPIPE_ERR_INVALID_ARG;
  if (sh->hidden % 128 != 0 || sh->vocab % 128 != 0 || sh->tile_rows % 128 != 0)
    return UPIPE_ERR_UNSUPPORTED;
  if (sh->hidden > 65536 || sh->vocab > (1 << 24)) return UPIPE_ERR_UNSUPPORTED;
  return UPIPE_OK;
}

int64_t loss_tile(const upipe_loss_shape_t* sh) { return std::min<int64_t>(sh->tile_rows, sh->S); }

// vocabulary tile width of the logits GEMMs
int vocab_bn(const upipe_loss_shape_t* sh) { return sh->vocab % 256 == 0 ? 256 : 128; }

LossLayout loss_plan(const upipe_loss_shape_t* sh, int mode) {
  LossLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += loss_align(bytes);
    return at;
  };
  const size_t T = (size_t)loss_tile(sh), V = (size_t)sh->vocab;
  L.part = L.zt = L.dz = (size_t)-1;
  if (mode == 0) {
    L.part = take(T * (V / vocab_bn(sh)) * sizeof(float2));
    L.zt = take(T * sizeof(float));
  } else {
    L.dz = take(T * V * 2);
  }
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define LOSS_TRY(expr)                \
  do {                                \
    int _rc = (expr);                 \
    if (_rc != UPIPE_OK) return _rc;  \
  } while (0)
#define LOSS_CUDA(expr) \
  do { if ((expr) != cudaSuccess) return UPIPE_ERR_CUDA; } while (0)
#define LOSS_MAP(...) \
  do { if (!make_tmap_bf16(__VA_ARGS__)) return UPIPE_ERR_CUDA; } while (0)
#define LOSS_MAP32(...) \
  do { if (!make_tmap_f32(__VA_ARGS__)) return UPIPE_ERR_CUDA; } while (0)

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

int validate(const upipe_loss_shape_t* sh, std::initializer_list<const void*> required,
             const void* workspace, size_t ws_bytes, int mode) {
  LOSS_TRY(check_loss_shape(sh));
  for (const void* p : required)
    if (!p || !aligned16(p)) return UPIPE_ERR_INVALID_ARG;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % kLossAlign)
    return UPIPE_ERR_INVALID_ARG;
  if (ws_bytes < loss_plan(sh, mode).total) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  return UPIPE_OK;
}

// the logits GEMM of one tile with the loss epilogue ``epi``: A = h_R, B = W
int logits_gemm(const upipe_loss_shape_t* sh, const bf16* h_rows, int64_t rows,
                const CUtensorMap& wmap, EpiKind epi, const EpiParams& ep, int* err, int sms,
                cudaStream_t st) {
  CUtensorMap hm;
  LOSS_MAP(&hm, h_rows, (uint64_t)rows, sh->hidden, sh->hidden, 128, 64);
  GemmArgs ga{(int)rows, sh->vocab, sh->hidden, 1, 128};
  // the h tile (A) is far smaller than W (B): row blocks fastest keeps it in
  // L2 and reads W once per tile
  ga.m_fastest = 1;
  LOSS_CUDA(launch_gemm(vocab_bn(sh), false, false, epi, &hm, 1, &wmap, 1, ga, ep, err, sms, st));
  return UPIPE_OK;
}

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" size_t upipe_loss_workspace_bytes(const upipe_loss_shape_t* shape, int mode) {
  if (mode < 0 || mode > 1 || check_loss_shape(shape) != UPIPE_OK) return 0;
  return loss_plan(shape, mode).total;
}

extern "C" int upipe_loss_fwd(const upipe_loss_shape_t* shape, const upipe_bf16* h_,
                              const upipe_bf16* W_, const int32_t* targets, float* loss_rows,
                              float* lse, void* workspace, size_t ws_bytes, void* stream) {
  LOSS_TRY(validate(shape, {h_, W_, targets, loss_rows, lse}, workspace, ws_bytes, 0));
  NvtxRange call_range("upipe_loss_fwd");
  const bf16* h = reinterpret_cast<const bf16*>(h_);
  const bf16* W = reinterpret_cast<const bf16*>(W_);
  int* err = nullptr;
  int sms = 0;
  LOSS_TRY(device_context(&err, &sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const LossLayout L = loss_plan(shape, 0);
  float2* part = at<float2>(workspace, L.part);
  float* zt = at<float>(workspace, L.zt);
  const int H = shape->hidden, V = shape->vocab, bn = vocab_bn(shape);
  const int64_t S = shape->S, T = loss_tile(shape);
  CUtensorMap wmap;
  LOSS_MAP(&wmap, W, V, H, H, bn, 64);
  for (int64_t t0 = 0; t0 < S; t0 += T) {
    NvtxRange tile_range("upipe_loss_fwd", (int)(t0 / T));
    const int64_t rows = std::min(T, S - t0);
    EpiParams ep{};
    ep.targets = targets + t0;
    ep.part = part;
    ep.ld_part = V / bn;
    ep.zt = zt;
    LOSS_TRY(logits_gemm(shape, h + t0 * H, rows, wmap, EPI_LSE_PART, ep, err, sms, st));
    LOSS_CUDA(launch_loss_rows(part, V / bn, zt, targets + t0, V, rows, lse + t0, loss_rows + t0,
                               st, err));
  }
  return UPIPE_OK;
}

extern "C" int upipe_loss_bwd(const upipe_loss_shape_t* shape, const upipe_bf16* h_,
                              const upipe_bf16* W_, const int32_t* targets, const float* lse,
                              float scale, float* dh, float* dW, void* workspace, size_t ws_bytes,
                              void* stream) {
  LOSS_TRY(validate(shape, {h_, W_, targets, lse, dh, dW}, workspace, ws_bytes, 1));
  NvtxRange call_range("upipe_loss_bwd");
  const bf16* h = reinterpret_cast<const bf16*>(h_);
  const bf16* W = reinterpret_cast<const bf16*>(W_);
  int* err = nullptr;
  int sms = 0;
  LOSS_TRY(device_context(&err, &sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const LossLayout L = loss_plan(shape, 1);
  bf16* dz = at<bf16>(workspace, L.dz);
  const int H = shape->hidden, V = shape->vocab, bn = vocab_bn(shape);
  const int64_t S = shape->S, T = loss_tile(shape);
  LOSS_CUDA(cudaMemsetAsync(dW, 0, sizeof(float) * (size_t)V * H, st));
  CUtensorMap wmap, w_mn;
  LOSS_MAP(&wmap, W, V, H, H, bn, 64);      // B of the logits, K-major
  LOSS_MAP(&w_mn, W, V, H, H, 64, 64);      // B of dh = dz W: [K = vocab, N = hidden]
  const int hbn = (H % 256 == 0) ? 256 : 128;
  for (int64_t t0 = 0; t0 < S; t0 += T) {
    NvtxRange tile_range("upipe_loss_bwd", (int)(t0 / T));
    const int64_t rows = std::min(T, S - t0);
    const bf16* h_t = h + t0 * H;
    // 1. z recomputed, dz = scale (softmax - onehot)  [rows, V] bf16
    {
      EpiParams ep{};
      ep.targets = targets + t0;
      ep.lse_rows = lse + t0;
      ep.dz = dz;
      ep.ld_dz = V;
      ep.loss_scale = scale;
      LOSS_TRY(logits_gemm(shape, h_t, rows, wmap, EPI_DLOGITS, ep, err, sms, st));
    }
    // 2. dh_R = dz W  (K = vocab)
    {
      CUtensorMap am, dhm;
      LOSS_MAP(&am, dz, (uint64_t)rows, V, V, 128, 64);
      LOSS_MAP32(&dhm, dh + t0 * H, (uint64_t)rows, H, H, 32, 32);
      EpiParams ep{};
      ep.C = dh + t0 * H;
      ep.ldc = H;
      GemmArgs ga{(int)rows, H, V, 1, 128};
      LOSS_CUDA(launch_gemm(hbn, false, true, EPI_F32, &am, 1, &w_mn, 1, ga, ep, err, sms, st,
                            &dhm));
    }
    // 3. dW += dz^T h_R  (M = vocab, N = hidden, K = rows; split-K)
    {
      CUtensorMap dz_mn, h_mn;
      LOSS_MAP(&dz_mn, dz, (uint64_t)rows, V, V, 64, 64);
      LOSS_MAP(&h_mn, h_t, (uint64_t)rows, H, H, 64, 64);
      EpiParams ep{};
      ep.C = dW;
      ep.ldc = H;
      GemmArgs ga{V, H, (int)rows, wgrad_splits(rows, V, H, hbn, sms), 128};
      LOSS_CUDA(launch_gemm(hbn, true, true, EPI_F32_ATOMIC, &dz_mn, 1, &h_mn, 1, ga, ep, err, sms,
                            st));
    }
  }
  return UPIPE_OK;
}
