// libupipe host side of the sequence-tiled MLP (include/upipe.h,
// upipe_mlp_*): the SwiGLU MLP of the decoder layer computed over tiles of
// ``tile_rows`` tokens, so that no buffer as long as the sequence exists for
// its [S, ffn] intermediates (the pages' stack tiles the MLP and the loss
// along the sequence: memeeeeeex.com article, the stack section on Arctic
// sequence-length training; liquidgold.cc talk transcript).  Per tile t of
// rows R = [t0, t0 + T):
//   forward   a_t = silu(x_R Wg^T) * (x_R Wu^T)      one GEMM, EPI_SWIGLU
//             y_R = a_t Wd^T                         one GEMM, fp32 TMA store
//   backward  dA_t = dy_R Wd                         one GEMM, fp32 TMA store
//             g, u recomputed; dg_t, du_t, a_t       one GEMM, EPI_SWIGLU_BWD
//             dx_R = dg_t Wg + du_t Wu                one K-segmented GEMM
//             dWd += dy_R^T a_t                      split-K, red.global.add
//             dWg += dg_t^T x_R,  dWu += du_t^T x_R  one M-segmented split-K GEMM
// Every tile reuses the same workspace views; stream order alone makes the
// reuse safe.  Tiling is exact: a token's MLP output depends on that token
// alone, so the forward's rows do not depend on tile_rows.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <initializer_list>

#include "../../include/upipe.h"
#include "internal.h"

namespace upipe {
namespace {

constexpr size_t kMlpAlign = 256;
inline size_t mlp_align(size_t v) { return (v + kMlpAlign - 1) / kMlpAlign * kMlpAlign; }

struct MlpLayout {
  size_t act, dA, dG, dU, total;
};

int check_mlp_shape(const upipe_mlp_shape_t* sh) {
  if (!sh) return UPIPE_ERR_INVALID_ARG;
  if (sh->S < 1 || sh->S > (int64_t)INT32_MAX - 256 || sh->hidden <= 0 || sh->ffn <= 0 ||
      sh->tile_rows <= 0)
    return UPIPE_ERR_INVALID_ARG;
  // 128-row / 128-column tiles throughout, 256-wide gate/up output tiles
  if (sh->hidden % 128 != 0 || sh->ffn % 128 != 0 || sh->tile_rows % 128 != 0)
    return UPIPE_ERR_UNSUPPORTED;
  if ((int64_t)sh->ffn * 2 > (int64_t)INT32_MAX / 2 || sh->hidden > 65536 || sh->ffn > 262144)
    return UPIPE_ERR_UNSUPPORTED;
  return UPIPE_OK;
}

// rows of one tile: tile_rows, or S when the sequence is shorter
int64_t tile_of(const upipe_mlp_shape_t* sh) {
  return std::min<int64_t>(sh->tile_rows, sh->S);
}

MlpLayout mlp_plan(const upipe_mlp_shape_t* sh, int mode) {
  MlpLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += mlp_align(bytes);
    return at;
  };
  const size_t T = (size_t)tile_of(sh), F = (size_t)sh->ffn;
  L.act = take(T * F * 2);
  L.dA = L.dG = L.dU = (size_t)-1;
  if (mode == 1) {
    L.dA = take(T * F * 4);
    L.dG = take(T * F * 2);
    L.dU = take(T * F * 2);
  }
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define MLP_TRY(expr)                 \
  do {                                \
    int _rc = (expr);                 \
    if (_rc != UPIPE_OK) return _rc;  \
  } while (0)
#define MLP_CUDA(expr) \
  do { if ((expr) != cudaSuccess) return UPIPE_ERR_CUDA; } while (0)
#define MLP_MAP(...) \
  do { if (!make_tmap_bf16(__VA_ARGS__)) return UPIPE_ERR_CUDA; } while (0)
#define MLP_MAP32(...) \
  do { if (!make_tmap_f32(__VA_ARGS__)) return UPIPE_ERR_CUDA; } while (0)

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// a = silu(x_R Wg^T) * (x_R Wu^T) for the tile's rows (EPI_SWIGLU), or the
// same recomputed with dg, du from dA (EPI_SWIGLU_BWD)
int gate_up(const upipe_mlp_shape_t* sh, const bf16* x_rows, int64_t rows, const CUtensorMap& gmap,
            const CUtensorMap& umap, EpiKind epi, bf16* act, const float* dA, bf16* dG, bf16* dU,
            int* err, int sms, cudaStream_t st) {
  CUtensorMap xm, bm[2] = {gmap, umap};
  MLP_MAP(&xm, x_rows, (uint64_t)rows, sh->hidden, sh->hidden, 128, 64);
  EpiParams ep{};
  ep.act = act;
  ep.ld_act = sh->ffn;
  ep.dA = dA;
  ep.ld_da = sh->ffn;
  ep.dG = dG;
  ep.dU = dU;
  ep.ld_dg = sh->ffn;
  GemmArgs ga{(int)rows, 2 * sh->ffn, sh->hidden, 1, 128};
  // the x tile (A) is far smaller than Wg and Wu together (B): row blocks
  // fastest, in groups of 16 (2 MB of x per 128-row block at hidden 4096:
  // a group stays in L2 while the columns are swept)
  ga.m_fastest = 16;
  MLP_CUDA(launch_gemm(256, false, false, epi, &xm, 1, bm, 2, ga, ep, err, sms, st));
  return UPIPE_OK;
}

int validate(const upipe_mlp_shape_t* sh, std::initializer_list<const void*> required,
             const void* workspace, size_t ws_bytes, int mode) {
  MLP_TRY(check_mlp_shape(sh));
  for (const void* p : required)
    if (!p || !aligned16(p)) return UPIPE_ERR_INVALID_ARG;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % kMlpAlign)
    return UPIPE_ERR_INVALID_ARG;
  if (ws_bytes < mlp_plan(sh, mode).total) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  return UPIPE_OK;
}

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" size_t upipe_mlp_workspace_bytes(const upipe_mlp_shape_t* shape, int mode) {
  if (mode < 0 || mode > 1 || check_mlp_shape(shape) != UPIPE_OK) return 0;
  return mlp_plan(shape, mode).total;
}

extern "C" int upipe_mlp_fwd(const upipe_mlp_shape_t* shape, const upipe_bf16* x_,
                             const upipe_bf16* Wg_, const upipe_bf16* Wu_, const upipe_bf16* Wd_,
                             float* y, void* workspace, size_t ws_bytes, void* stream) {
  MLP_TRY(validate(shape, {x_, Wg_, Wu_, Wd_, y}, workspace, ws_bytes, 0));
  NvtxRange call_range("upipe_mlp_fwd");
  const bf16* x = reinterpret_cast<const bf16*>(x_);
  const bf16* Wg = reinterpret_cast<const bf16*>(Wg_);
  const bf16* Wu = reinterpret_cast<const bf16*>(Wu_);
  const bf16* Wd = reinterpret_cast<const bf16*>(Wd_);
  int* err = nullptr;
  int sms = 0;
  MLP_TRY(device_context(&err, &sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const MlpLayout L = mlp_plan(shape, 0);
  bf16* act = at<bf16>(workspace, L.act);
  const int H = shape->hidden, F = shape->ffn;
  const int64_t S = shape->S, T = tile_of(shape);
  CUtensorMap gmap, umap, dmap, amap;
  MLP_MAP(&gmap, Wg, F, H, H, 128, 64);     // B of the gate rows, K-major
  MLP_MAP(&umap, Wu, F, H, H, 128, 64);     // B of the up rows
  const int ybn = (H % 256 == 0) ? 256 : 128;
  MLP_MAP(&dmap, Wd, H, F, F, ybn, 64);     // B of y = a Wd^T, K-major
  for (int64_t t0 = 0; t0 < S; t0 += T) {
    NvtxRange tile_range("upipe_mlp_fwd", (int)(t0 / T));
    const int64_t rows = std::min(T, S - t0);
    MLP_TRY(gate_up(shape, x + t0 * H, rows, gmap, umap, EPI_SWIGLU, act, nullptr, nullptr,
                    nullptr, err, sms, st));
    CUtensorMap ymap;
    MLP_MAP(&amap, act, (uint64_t)rows, F, F, 128, 64);
    MLP_MAP32(&ymap, y + t0 * H, (uint64_t)rows, H, H, 32, 32);
    EpiParams ep{};
    ep.C = y + t0 * H;
    ep.ldc = H;
    ep.beta = 0;
    GemmArgs ga{(int)rows, H, F, 1, 128};
    MLP_CUDA(launch_gemm(ybn, false, false, EPI_F32, &amap, 1, &dmap, 1, ga, ep, err, sms, st,
                         &ymap));
  }
  return UPIPE_OK;
}

extern "C" int upipe_mlp_bwd(const upipe_mlp_shape_t* shape, const upipe_bf16* x_,
                             const upipe_bf16* Wg_, const upipe_bf16* Wu_, const upipe_bf16* Wd_,
                             const upipe_bf16* dy_, float* dx, float* dWg, float* dWu, float* dWd,
                             void* workspace, size_t ws_bytes, void* stream) {
  MLP_TRY(validate(shape, {x_, Wg_, Wu_, Wd_, dy_, dx, dWg, dWu, dWd}, workspace, ws_bytes, 1));
  NvtxRange call_range("upipe_mlp_bwd");
  const bf16* x = reinterpret_cast<const bf16*>(x_);
  const bf16* Wg = reinterpret_cast<const bf16*>(Wg_);
  const bf16* Wu = reinterpret_cast<const bf16*>(Wu_);
  const bf16* Wd = reinterpret_cast<const bf16*>(Wd_);
  const bf16* dy = reinterpret_cast<const bf16*>(dy_);
  int* err = nullptr;
  int sms = 0;
  MLP_TRY(device_context(&err, &sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const MlpLayout L = mlp_plan(shape, 1);
  bf16* act = at<bf16>(workspace, L.act);
  float* dA = at<float>(workspace, L.dA);
  bf16* dG = at<bf16>(workspace, L.dG);
  bf16* dU = at<bf16>(workspace, L.dU);
  const int H = shape->hidden, F = shape->ffn;
  const int64_t S = shape->S, T = tile_of(shape);
  MLP_CUDA(cudaMemsetAsync(dWg, 0, sizeof(float) * (size_t)F * H, st));
  MLP_CUDA(cudaMemsetAsync(dWu, 0, sizeof(float) * (size_t)F * H, st));
  MLP_CUDA(cudaMemsetAsync(dWd, 0, sizeof(float) * (size_t)H * F, st));
  CUtensorMap gmap, umap, wd_mn, wg_mn, wu_mn;
  MLP_MAP(&gmap, Wg, F, H, H, 128, 64);     // gate/up recompute, K-major
  MLP_MAP(&umap, Wu, F, H, H, 128, 64);
  MLP_MAP(&wd_mn, Wd, H, F, F, 64, 64);     // B of dA = dy Wd: [K = hidden, N = ffn]
  MLP_MAP(&wg_mn, Wg, F, H, H, 64, 64);     // B of dx = dg Wg + du Wu: [K = ffn, N = hidden]
  MLP_MAP(&wu_mn, Wu, F, H, H, 64, 64);
  const int da_bn = (F % 256 == 0) ? 256 : 128;
  const int dx_bn = (H % 256 == 0) ? 256 : 128;
  for (int64_t t0 = 0; t0 < S; t0 += T) {
    NvtxRange tile_range("upipe_mlp_bwd", (int)(t0 / T));
    const int64_t rows = std::min(T, S - t0);
    const bf16* x_t = x + t0 * H;
    const bf16* dy_t = dy + t0 * H;
    // 1. dA = dy_R Wd  [rows, ffn] fp32
    {
      CUtensorMap dym, dam;
      MLP_MAP(&dym, dy_t, (uint64_t)rows, H, H, 128, 64);
      MLP_MAP32(&dam, dA, (uint64_t)rows, F, F, 32, 32);
      EpiParams ep{};
      ep.C = dA;
      ep.ldc = F;
      GemmArgs ga{(int)rows, F, H, 1, 128};
      ga.m_fastest = 16;  // groups of 16 dy row blocks stay in L2 while Wd (B) is swept
      MLP_CUDA(launch_gemm(da_bn, false, true, EPI_F32, &dym, 1, &wd_mn, 1, ga, ep, err, sms, st,
                           &dam));
    }
    // 2. g, u recomputed: dg, du and a of the tile (bf16)
    MLP_TRY(gate_up(shape, x_t, rows, gmap, umap, EPI_SWIGLU_BWD, act, dA, dG, dU, err, sms, st));
    // 3. dx_R = dg Wg + du Wu: two K segments into one accumulator
    {
      CUtensorMap am[2], bm[2] = {wg_mn, wu_mn}, dxm;
      MLP_MAP(&am[0], dG, (uint64_t)rows, F, F, 128, 64);
      MLP_MAP(&am[1], dU, (uint64_t)rows, F, F, 128, 64);
      MLP_MAP32(&dxm, dx + t0 * H, (uint64_t)rows, H, H, 32, 32);
      GemmArgs ga{(int)rows, H, 2 * F, 1, 128};
      ga.nkseg = 2;
      ga.kseg_end[0] = F / 64;
      ga.kseg_end[1] = 2 * F / 64;
      ga.kseg_a[0] = 0;
      ga.kseg_a[1] = 1;
      ga.kseg_b[0] = 0;
      ga.kseg_b[1] = 1;
      EpiParams ep{};
      ep.C = dx + t0 * H;
      ep.ldc = H;
      MLP_CUDA(launch_gemm(dx_bn, false, true, EPI_F32, am, 2, bm, 2, ga, ep, err, sms, st, &dxm));
    }
    // 4. dWd += dy_R^T a  (M = hidden, N = ffn, K = rows; split-K)
    {
      CUtensorMap dy_mn, a_mn;
      MLP_MAP(&dy_mn, dy_t, (uint64_t)rows, H, H, 64, 64);
      MLP_MAP(&a_mn, act, (uint64_t)rows, F, F, 64, 64);
      EpiParams ep{};
      ep.C = dWd;
      ep.ldc = F;
      const int bn = (F % 256 == 0) ? 256 : 128;
      GemmArgs ga{H, F, (int)rows, wgrad_splits(rows, H, F, bn, sms), 128};
      ga.m_fastest = 1;   // dy^T (A) stays in L2, a^T (B) is read once
      MLP_CUDA(launch_gemm(bn, true, true, EPI_F32_ATOMIC, &dy_mn, 1, &a_mn, 1, ga, ep, err, sms,
                           st));
    }
    // 5. dWg += dg^T x_R, dWu += du^T x_R: two M segments, x read once
    {
      CUtensorMap am[2], x_mn;
      MLP_MAP(&am[0], dG, (uint64_t)rows, F, F, 64, 64);
      MLP_MAP(&am[1], dU, (uint64_t)rows, F, F, 64, 64);
      MLP_MAP(&x_mn, x_t, (uint64_t)rows, H, H, 64, 64);
      const int bn = (H % 256 == 0) ? 256 : 128;
      GemmArgs ga{2 * F, H, (int)rows, 1, 128};
      ga.nmseg = 2;
      ga.mseg_t0[0] = 0;
      ga.mseg_t0[1] = F / 128;
      ga.mseg_t0[2] = 2 * F / 128;
      ga.mseg_rows[0] = F;
      ga.mseg_rows[1] = F;
      ga.mseg_a[0] = 0;
      ga.mseg_a[1] = 1;
      ga.ksplit = wgrad_splits(rows, 2 * F, H, bn, sms);
      EpiParams ep{};
      ep.ldc = H;
      ep.mseg_c[0] = dWg;
      ep.mseg_c[1] = dWu;
      MLP_CUDA(launch_gemm(bn, true, true, EPI_F32_ATOMIC, am, 2, &x_mn, 1, ga, ep, err, sms,
                           st));
    }
  }
  return UPIPE_OK;
}
