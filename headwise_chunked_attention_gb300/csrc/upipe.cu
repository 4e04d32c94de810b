// libupipe host side: argument validation, the workspace planner and the
// head-chunk scheduler behind the C ABI of include/upipe.h.
//
// The chunk loop is the UPipe loop (memeeeeeex.com article, "Untied Ulysses
// (UPipe)"; liquidgold.cc talk transcript: divide the heads into chunks and
// reuse all the buffers): for chunk c of ``chunk_heads`` query heads, project
// the chunk's Q (and its KV group's K/V when the chunk starts a new group)
// into the workspace, run causal attention for those heads over the whole
// sequence, and add the chunk's Wo-slice partial result into ``out``.  Every
// chunk reuses the same workspace views; stream order alone makes the reuse
// safe, there is no host synchronisation inside the loop.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/upipe.h"
#include "internal.h"

namespace upipe {

__device__ int g_device_error = 0;

// NVTX ranges (internal.h): one per entry point and per chunk, so that a
// timeline tool shows the chunk loop.
NvtxRange::NvtxRange(const char* what, int chunk) {
  if (chunk < 0) {
    nvtxRangePushA(what);
  } else {
    char name[64];
    std::snprintf(name, sizeof name, "%s chunk %d", what, chunk);
    nvtxRangePushA(name);
  }
}
NvtxRange::~NvtxRange() { nvtxRangePop(); }

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// --------------------------------------------------------- device state --

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int* err = nullptr;
  // highest-priority stream on which the forward runs each chunk's Wo-slice
  // accumulate beside the next chunk's attention; created by the first
  // forward that forks (nullptr: not yet, or not available)
  bool side_tried = false;
  cudaStream_t side = nullptr;
};

// measurement hook (upipe_profile_attach)
struct Profile {
  int kernel = -1;
  void* const* starts = nullptr;
  void* const* ends = nullptr;
  int capacity = 0;
  int count = 0;
};
Profile g_prof;

inline void prof_begin(int kernel, cudaStream_t st) {
  if (g_prof.kernel == kernel && g_prof.count < g_prof.capacity)
    cudaEventRecord(static_cast<cudaEvent_t>(g_prof.starts[g_prof.count]), st);
}
inline void prof_end(int kernel, cudaStream_t st) {
  if (g_prof.kernel == kernel && g_prof.count < g_prof.capacity)
    cudaEventRecord(static_cast<cudaEvent_t>(g_prof.ends[g_prof.count++]), st);
}

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return UPIPE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return UPIPE_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return UPIPE_ERR_CUDA;
    s.err = static_cast<int*>(p);
    s.ready = true;
  }
  *out = &s;
  return UPIPE_OK;
}

// The side stream of the current device (set up by device_state), created on
// first use; nullptr if it cannot be created (the forward then runs serially).
cudaStream_t side_stream(DeviceState* s) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!s->side_tried) {
    s->side_tried = true;
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&s->side, cudaStreamNonBlocking, greatest) != cudaSuccess) {
      s->side = nullptr;
      cudaGetLastError();
    }
  }
  return s->side;
}

// ---------------------------------------------------------- tensor maps --

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                    uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_f32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                   uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 4};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// ------------------------------------------------------------ validation --

struct Geo {
  long long S;
  int hidden, Hq, Hkv, d, ch, g, kvc, nchunks;
  bool norm;
};

int check_shape(const upipe_shape_t* sh, Geo* geo) {
  if (!sh) return UPIPE_ERR_INVALID_ARG;
  if (sh->S < 1 || sh->S > (int64_t)INT32_MAX - 256) return UPIPE_ERR_INVALID_ARG;
  if (sh->hidden <= 0 || sh->Hq <= 0 || sh->Hkv <= 0 || sh->d <= 0 || sh->chunk_heads <= 0)
    return UPIPE_ERR_INVALID_ARG;
  if (sh->Hq % sh->Hkv != 0 || sh->Hq % sh->chunk_heads != 0) return UPIPE_ERR_INVALID_ARG;
  const int g = sh->Hq / sh->Hkv;
  if (!(sh->chunk_heads % g == 0 || g % sh->chunk_heads == 0)) return UPIPE_ERR_INVALID_ARG;
  if (!(sh->rope_theta > 0.0) || !std::isfinite(sh->rope_theta)) return UPIPE_ERR_INVALID_ARG;
  if (sh->qk_norm != 0 && sh->qk_norm != 1) return UPIPE_ERR_INVALID_ARG;
  if (sh->qk_norm && !(sh->norm_eps >= 0.f)) return UPIPE_ERR_INVALID_ARG;
  if (sh->d != 64 && sh->d != 128) return UPIPE_ERR_UNSUPPORTED;
  if (sh->hidden % 128 != 0) return UPIPE_ERR_UNSUPPORTED;
  if ((long long)sh->Hq * sh->d > 65536) return UPIPE_ERR_UNSUPPORTED;
  geo->S = sh->S;
  geo->hidden = sh->hidden;
  geo->Hq = sh->Hq;
  geo->Hkv = sh->Hkv;
  geo->d = sh->d;
  geo->ch = sh->chunk_heads;
  geo->g = g;
  geo->kvc = sh->chunk_heads >= g ? sh->chunk_heads / g : 1;
  geo->nchunks = sh->Hq / sh->chunk_heads;
  geo->norm = sh->qk_norm != 0;
  return UPIPE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ----------------------------------------------------------- workspace --

struct Layout {
  size_t rope_hi, rope_lo, rope_lo_t, q, k, v, o, flush;     // forward
  size_t o2;                                               // forward, mode 2
  size_t dO, D, dq, dk, dv, dklo, dvlo, yq, rq, yk, rk, sc;  // backward
  size_t total;
};

Layout plan(const Geo& g, int mode) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off += align_up(bytes);
    return at;
  };
  const size_t S = (size_t)g.S, d = (size_t)g.d, ch = (size_t)g.ch, kvc = (size_t)g.kvc;
  L.rope_hi = take((((size_t)g.S >> 10) + 1) * (d / 2) * sizeof(float2));
  L.rope_lo = take(1024 * (d / 2) * sizeof(float2));
  L.rope_lo_t = take(1024 * (d / 2) * sizeof(float2));
  L.q = take(S * ch * d * 2);
  L.k = take(S * kvc * d * 2);
  L.v = take(S * kvc * d * 2);
  // mode 3 (the fused forward) adds each chunk's partial result into out
  // from the attention kernel: no O buffer
  L.o = mode == 3 ? (size_t)-1 : take(S * ch * d * 2);
  // per-SM fp32 rows into which long attention rows fold their O accumulator
  L.flush = S > (size_t)kFlushTiles * 128 ? take((size_t)kFlushSlots * 256 * d * 4) : (size_t)-1;
  // mode 2: a third chunk buffer, last so that every other offset is mode 0's
  L.o2 = mode == 2 ? take(S * ch * d * 2) : (size_t)-1;
  if (mode == 1) {
    L.dO = take(S * ch * d * 2);
    L.D = take(ch * S * 4);
    L.dq = take(S * ch * d * 4);
    L.dk = take(S * kvc * d * 4);
    L.dv = take(S * kvc * d * 4);
    L.dklo = take(S * kvc * d * 2);
    L.dvlo = take(S * kvc * d * 2);
    if (g.norm) {
      L.yq = take(S * ch * d * 4);
      L.rq = take(ch * S * 4);
      L.yk = take(S * kvc * d * 4);
      L.rk = take(kvc * S * 4);
    }
    // the fp16 gradient scales' norm maxima: [Mdout, Wcol, Vmax per KV head
    // that starts a group, MdO' per chunk] (internal.h)
    L.sc = take((size_t)(2 + g.Hkv + g.nchunks) * sizeof(float));
  }
  L.total = off;
  return L;
}

// UPIPE_VERBOSE=1 in the environment prints the CUDA error behind an
// UPIPE_ERR_CUDA return to stderr.
int cuda_fail_at(cudaError_t e, const char* what, int line) {
  if (e == cudaSuccess) return UPIPE_OK;
  static const bool verbose = [] {
    const char* v = std::getenv("UPIPE_VERBOSE");
    return v && *v && *v != '0';
  }();
  if (verbose)
    std::fprintf(stderr, "upipe: %s failed (upipe.cu:%d): %s\n", what, line,
                 cudaGetErrorString(e));
  return UPIPE_ERR_CUDA;
}

#define UPIPE_TRY(expr)                 \
  do {                                  \
    int _rc = (expr);                   \
    if (_rc != UPIPE_OK) return _rc;    \
  } while (0)
#define UPIPE_CUDA(expr) UPIPE_TRY(cuda_fail_at((expr), #expr, __LINE__))
#define UPIPE_MAP(...) \
  do { if (!make_tmap_bf16(__VA_ARGS__)) return UPIPE_ERR_CUDA; } while (0)

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// Events of one forward call's fork/join with the side stream.  Destroying an
// event whose record is still pending is allowed: CUDA frees it on completion.
// If the call leaves early (an error after work was forked), the destructor
// still orders the caller's stream after everything enqueued on the side
// stream, so the caller never sees the side stream's work outlive the call.
struct Events {
  cudaEvent_t proj = nullptr, out[2] = {nullptr, nullptr};
  cudaStream_t side = nullptr, caller = nullptr;  // set once work is forked
  bool joined = false;
  cudaError_t create() {
    for (cudaEvent_t* e : {&proj, &out[0], &out[1]}) {
      const cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  }
  ~Events() {
    if (side && !joined && proj && cudaEventRecord(proj, side) == cudaSuccess)
      cudaStreamWaitEvent(caller, proj, 0);
    for (cudaEvent_t e : {proj, out[0], out[1]})
      if (e) cudaEventDestroy(e);
  }
};

}  // namespace

// Split-K partitions of a weight-gradient GEMM (K = S tokens, M x N output in
// 128 x bn tiles): about one partition per 8192 tokens (at most 64), moved
// within a factor of two of that to the count whose tiles fill the last wave
// of SMs best (ties: the count nearest the base), keeping >= 1024 tokens per
// partition.
int wgrad_splits(int64_t S, int M, int N, int bn, int sms) {
  const long long mn = (long long)((M + 127) / 128) * (N / bn);
  const int base = (int)std::max<int64_t>(1, std::min<int64_t>(64, (S + 8191) / 8192));
  int best = base;
  double best_eff = -1.0;
  for (int k = std::max(1, base / 2); k <= std::min(64, 2 * base); ++k) {
    if (k > 1 && S / k < 1024) continue;
    const long long tiles = mn * k;
    const long long waves = (tiles + sms - 1) / sms;
    const double eff = (double)tiles / (double)(waves * sms);
    if (eff > best_eff + 1e-9 ||
        (eff > best_eff - 1e-9 && std::abs(k - base) < std::abs(best - base))) {
      best = k;
      best_eff = eff;
    }
  }
  return best;
}

namespace {

// Longest query walk (sub-tiles of 64 queries) of one attention-backward CTA,
// whose dK / dV accumulate in TMEM over the walk: the whole walk up to 1M
// tokens (16384 sub-tiles, as many accumulation steps as the forward's O takes
// over 1M keys), else segments of 8192 sub-tiles.  UPIPE_BWD_WALK (an even
// number >= 2) overrides it, e.g. to run the segmented walk on short
// sequences.
int bwd_walk(int64_t S) {
  static const int forced = [] {
    const char* v = std::getenv("UPIPE_BWD_WALK");
    const int w = v ? std::atoi(v) : 0;
    return (w >= 2 && w % 2 == 0) ? w : 0;
  }();
  if (forced) return forced;
  const int64_t nu = (S + 63) / 64;
  return nu <= 16384 ? (int)((nu + 1) / 2 * 2) : 8192;
}

// SMs given to a Wo-slice accumulate that runs beside an attention launch: it
// is bound by HBM (a read-modify-write of the fp32 layer output), which a
// fifth of the SMs can nearly saturate, and the rest keep the tensor cores of
// the attention busy.
inline int side_sms(int num_sms) { return std::max(8, num_sms / 5); }

// Fused projection of one chunk: Q heads [h0, h0+ch) and, when the chunk
// starts a new KV group, K and V heads [kv0, kv0+kvc).  Each 128-row x d
// output tile is one head, so a head's values never depend on chunk_heads.
// Q, K, V are written in fp16 (the attention kernels' operand type).  vmax:
// nullptr, or where the running max of the V rows' norms goes (backward).
int project_chunk(const Geo& g, const DeviceState* ds, cudaStream_t st, const CUtensorMap& xmap,
                  const bf16* Wq, const bf16* Wk, const bf16* Wv, const float* qgw,
                  const float* kgw, float eps, int h0, int kv0, bool new_group, __half* Q,
                  __half* K, __half* V, const float2* rhi, const float2* rlo_t, float* yq,
                  float* rq, float* yk, float* rk, float* vmax = nullptr) {
  const int d = g.d;
  CUtensorMap bm[3];
  EpiParams ep{};
  ep.rope_hi = rhi;
  ep.rope_lo_t = rlo_t;
  ep.eps = eps;
  const int qk_mode = g.norm ? PROJ_NORM_ROPE : PROJ_ROPE;
  int n = 0, ns = 0;
  UPIPE_MAP(&bm[0], Wq, (uint64_t)g.Hq * d, g.hidden, g.hidden, d, 64);
  ep.seg[ns++] =
      ProjSeg{n, n + g.ch * d, 0, h0 * d, Q, g.ch * d, 0, qk_mode, qgw, yq, g.ch * d, rq, nullptr};
  n += g.ch * d;
  if (new_group) {
    UPIPE_MAP(&bm[1], Wk, (uint64_t)g.Hkv * d, g.hidden, g.hidden, d, 64);
    UPIPE_MAP(&bm[2], Wv, (uint64_t)g.Hkv * d, g.hidden, g.hidden, d, 64);
    ep.seg[ns++] = ProjSeg{n, n + g.kvc * d, 1, kv0 * d, K, g.kvc * d, 0, qk_mode, kgw, yk,
                           g.kvc * d, rk, nullptr};
    n += g.kvc * d;
    ep.seg[ns++] = ProjSeg{n, n + g.kvc * d, 2, kv0 * d, V, g.kvc * d, 0, PROJ_PLAIN, nullptr,
                           nullptr, 0, nullptr, vmax};
    n += g.kvc * d;
  }
  ep.nseg = ns;
  GemmArgs ga{(int)g.S, n, g.hidden, 1, d};
  UPIPE_CUDA(launch_gemm(d, false, false, EPI_PROJ, &xmap, 1, bm, new_group ? 3 : 1, ga, ep, ds->err,
                         ds->num_sms, st));
  return UPIPE_OK;
}

// dO / D (the backward's recompute): also form D' = dO' . o per row from the
// kernel's fp32 o (see AttnFwdArgs).
// womap / outmap (the fused forward): the kernel adds the chunk's partial
// result into out itself and stores no o (O must be nullptr).
int attention_chunk(const Geo& g, const DeviceState* ds, cudaStream_t st, const __half* Q,
                    const __half* K, const __half* V, int h0, int kv0, bf16* O, int ldo,
                    float* lse, float* flush, const __half* dO = nullptr, int ld_do = 0,
                    float* D = nullptr, const CUtensorMap* womap = nullptr,
                    const CUtensorMap* outmap = nullptr, const float* lse_in = nullptr) {
  const int d = g.d;
  CUtensorMap qm, km, vm;
  UPIPE_MAP(&qm, Q, g.S, (uint64_t)g.ch * d, (uint64_t)g.ch * d, 128, 64);
  UPIPE_MAP(&km, K, g.S, (uint64_t)g.kvc * d, (uint64_t)g.kvc * d, 128, 64);
  UPIPE_MAP(&vm, V, g.S, (uint64_t)g.kvc * d, (uint64_t)g.kvc * d, 128, 64);
  AttnFwdArgs a{};
  a.S = (int)g.S;
  a.heads = g.ch;
  a.group = g.g;
  a.h0 = h0;
  a.kv0 = kv0;
  a.O = O;
  a.ldo = ldo;
  a.lse = lse;
  a.lse_stride = g.S;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
  a.flush = flush;
  a.dO = dO;
  a.ld_do = ld_do;
  a.D = D;
  a.wo_tiles = womap ? g.hidden / 128 : 0;
  a.lse_in = lse_in;
  const int timer = womap ? 5 : 0;
  prof_begin(timer, st);
  const cudaError_t e = launch_attn_fwd(qm, km, vm, a, d, ds->err, st, womap, outmap);
  prof_end(timer, st);
  UPIPE_CUDA(e);
  return UPIPE_OK;
}

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" size_t upipe_workspace_bytes(const upipe_shape_t* shape, int mode) {
  Geo g;
  if (mode < 0 || mode > 3) return 0;
  if (check_shape(shape, &g) != UPIPE_OK) return 0;
  return plan(g, mode).total;
}

// The forward of both entry points.  fork: run each chunk's Wo-slice
// accumulate on the device's side stream beside the next chunk's attention
// (three events per call); false keeps every launch on the caller's stream
// and creates nothing.
static int attn_fwd_impl(const upipe_shape_t* shape, const upipe_bf16* x_,
                         const upipe_bf16* Wq_, const upipe_bf16* Wk_, const upipe_bf16* Wv_,
                         const upipe_bf16* Wo_, const float* q_norm_w, const float* k_norm_w,
                         float* out, float* lse, void* workspace, size_t ws_bytes,
                         upipe_bf16* attn_o, void* stream, bool fork) {
  Geo g;
  UPIPE_TRY(check_shape(shape, &g));
  NvtxRange call_range("upipe_attn_fwd");
  const bf16* x = reinterpret_cast<const bf16*>(x_);
  const bf16* Wq = reinterpret_cast<const bf16*>(Wq_);
  const bf16* Wk = reinterpret_cast<const bf16*>(Wk_);
  const bf16* Wv = reinterpret_cast<const bf16*>(Wv_);
  const bf16* Wo = reinterpret_cast<const bf16*>(Wo_);
  bf16* o_all = reinterpret_cast<bf16*>(attn_o);
  if (!x || !Wq || !Wk || !Wv || !Wo || !out || !lse || !workspace) return UPIPE_ERR_INVALID_ARG;
  for (const void* p : {(const void*)x, (const void*)Wq, (const void*)Wk, (const void*)Wv,
                        (const void*)Wo, (const void*)out, (const void*)lse, (const void*)o_all,
                        (const void*)q_norm_w, (const void*)k_norm_w})
    if (p && !aligned16(p)) return UPIPE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return UPIPE_ERR_INVALID_ARG;
  if (ws_bytes < plan(g, 0).total) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  const bool third = ws_bytes >= plan(g, 2).total;
  const Layout L = plan(g, third ? 2 : 0);
  DeviceState* ds = nullptr;
  UPIPE_TRY(device_state(&ds));
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  float2* rhi = at<float2>(workspace, L.rope_hi);
  float2* rlo = at<float2>(workspace, L.rope_lo);
  float2* rlo_t = at<float2>(workspace, L.rope_lo_t);
  bf16* Q = at<bf16>(workspace, L.q);
  __half* K = at<__half>(workspace, L.k);
  __half* V = at<__half>(workspace, L.v);
  bf16* Ows = at<bf16>(workspace, L.o);
  float* flush = L.flush == (size_t)-1 ? nullptr : at<float>(workspace, L.flush);
  UPIPE_CUDA(launch_rope_table(rhi, rlo, rlo_t, g.S, g.d, shape->rope_theta, st, ds->err));

  CUtensorMap xmap, outmap;
  UPIPE_MAP(&xmap, x, g.S, g.hidden, g.hidden, 128, 64);
  if (!make_tmap_f32(&outmap, out, g.S, g.hidden, g.hidden, 32, 32)) return UPIPE_ERR_CUDA;
  const int out_bn = (g.hidden % 256 == 0) ? 256 : 128;

  // Chunk c projects Q (fp16) into buffer c % 2 and the attention writes O
  // (bf16) over it in place (each Q tile is read only by the CTA that writes
  // the same O rows, and before it writes them).  With more than one chunk, the Wo-slice accumulate
  // of chunk c - 1 runs on the side stream with a few SMs, after the projection
  // of chunk c and beside its attention; the projection of chunk c + 1 waits
  // for it, since it overwrites that buffer.  The last accumulate runs on the
  // caller's stream with every SM, after the side stream's work.  Without the
  // side stream each accumulate follows its chunk's attention on the caller's
  // stream.
  // Paired accumulates: with three or more chunks, a side stream and room
  // for the chunks' O (a third buffer, or the caller's attn_o), one GEMM adds
  // chunks c - 2 and c - 1 (K = 2 ch d) beside chunk c's attention, which
  // halves the fp32 read-modify-write passes over out.  Chunk c then projects
  // into buffer c % 3, whose previous chunk c - 3 belongs to the pair added
  // beside chunk c - 1 or c - 2.
  bf16* QO[3] = {Q, Ows, third ? at<bf16>(workspace, L.o2) : nullptr};
  cudaStream_t side = (fork && g.nchunks > 1) ? side_stream(ds) : nullptr;
  const bool overlap = side != nullptr;
  const bool pair = overlap && g.nchunks >= 3 && (o_all || third);
  const int nbuf = (pair && !o_all) ? 3 : 2;
  Events ev;
  if (overlap) {
    UPIPE_CUDA(ev.create());
    ev.side = side;
    ev.caller = st;
  }
  // timed: the measurement hook's kernel 2 covers the accumulates that run on
  // the call's stream with every SM, not the ones beside the next attention
  auto out_gemm = [&](int c, cudaStream_t s, int sms, bool timed) -> int {
    const int h0 = c * g.ch;
    const bf16* O = o_all ? o_all + (size_t)h0 * g.d : QO[c % nbuf];
    const int ldo = o_all ? g.Hq * g.d : g.ch * g.d;
    // out (+)= O_c Wo[:, h0*d : (h0+ch)*d]^T  (the chunk's partial result)
    CUtensorMap om, wom;
    UPIPE_MAP(&om, O, g.S, (uint64_t)g.ch * g.d, ldo, 128, 64);
    UPIPE_MAP(&wom, Wo + (size_t)h0 * g.d, g.hidden, (uint64_t)g.ch * g.d,
              (uint64_t)g.Hq * g.d, out_bn, 64);
    EpiParams ep{};
    ep.C = out;
    ep.ldc = g.hidden;
    ep.beta = c > 0;
    GemmArgs ga{(int)g.S, g.hidden, g.ch * g.d, 1, g.d};
    if (timed) prof_begin(2, s);
    UPIPE_CUDA(launch_gemm(out_bn, false, false, EPI_F32, &om, 1, &wom, 1, ga, ep, ds->err, sms, s,
                           &outmap));
    if (timed) prof_end(2, s);
    return UPIPE_OK;
  };
  // out (+)= O_c0 Wo_c0^T + O_c0+1 Wo_c0+1^T: two K segments, one per chunk
  auto out_gemm_pair = [&](int c0, cudaStream_t s, int sms, bool timed) -> int {
    CUtensorMap om[2], wom[2];
    for (int i = 0; i < 2; ++i) {
      const int h0 = (c0 + i) * g.ch;
      const bf16* O = o_all ? o_all + (size_t)h0 * g.d : QO[(c0 + i) % nbuf];
      const int ldo = o_all ? g.Hq * g.d : g.ch * g.d;
      UPIPE_MAP(&om[i], O, g.S, (uint64_t)g.ch * g.d, ldo, 128, 64);
      UPIPE_MAP(&wom[i], Wo + (size_t)h0 * g.d, g.hidden, (uint64_t)g.ch * g.d,
                (uint64_t)g.Hq * g.d, out_bn, 64);
    }
    EpiParams ep{};
    ep.C = out;
    ep.ldc = g.hidden;
    ep.beta = c0 > 0;
    GemmArgs ga{(int)g.S, g.hidden, 2 * g.ch * g.d, 1, g.d};
    ga.nkseg = 2;
    ga.kseg_end[0] = g.ch * g.d / 64;
    ga.kseg_end[1] = 2 * g.ch * g.d / 64;
    ga.kseg_a[0] = 0;
    ga.kseg_a[1] = 1;
    ga.kseg_b[0] = 0;
    ga.kseg_b[1] = 1;
    if (timed) prof_begin(2, s);
    UPIPE_CUDA(launch_gemm(out_bn, false, false, EPI_F32, om, 2, wom, 2, ga, ep, ds->err, sms, s,
                           &outmap));
    if (timed) prof_end(2, s);
    return UPIPE_OK;
  };
  for (int c = 0; c < g.nchunks; ++c) {
    NvtxRange chunk_range("upipe_attn_fwd", c);
    const int h0 = c * g.ch;
    const int kv0 = h0 / g.g;
    const bool new_group = (g.ch >= g.g) || (h0 % g.g == 0);
    bf16* Qc = QO[c % nbuf];
    if (pair) {
      // buffer c % 3 last held O of chunk c - 3: wait for its pair's accumulate
      if (!o_all && c >= 3 && (c - 3) % 2 == 0)
        UPIPE_CUDA(cudaStreamWaitEvent(st, ev.out[((c - 3) / 2) & 1], 0));
    } else if (overlap && c >= 2) {
      UPIPE_CUDA(cudaStreamWaitEvent(st, ev.out[c & 1], 0));
    }
    __half* Qh = reinterpret_cast<__half*>(Qc);
    UPIPE_TRY(project_chunk(g, ds, st, xmap, Wq, Wk, Wv, q_norm_w, k_norm_w, shape->norm_eps, h0,
                            kv0, new_group, Qh, K, V, rhi, rlo_t, nullptr, nullptr, nullptr,
                            nullptr));
    if (pair && c >= 2 && c % 2 == 0) {
      UPIPE_CUDA(cudaEventRecord(ev.proj, st));
      UPIPE_CUDA(cudaStreamWaitEvent(side, ev.proj, 0));
      UPIPE_TRY(out_gemm_pair(c - 2, side, side_sms(ds->num_sms), false));
      UPIPE_CUDA(cudaEventRecord(ev.out[((c - 2) / 2) & 1], side));
    } else if (!pair && overlap && c >= 1) {
      UPIPE_CUDA(cudaEventRecord(ev.proj, st));
      UPIPE_CUDA(cudaStreamWaitEvent(side, ev.proj, 0));
      UPIPE_TRY(out_gemm(c - 1, side, side_sms(ds->num_sms), false));
      UPIPE_CUDA(cudaEventRecord(ev.out[(c - 1) & 1], side));
    }
    bf16* O = o_all ? o_all + (size_t)h0 * g.d : Qc;
    const int ldo = o_all ? g.Hq * g.d : g.ch * g.d;
    UPIPE_TRY(attention_chunk(g, ds, st, Qh, K, V, h0, kv0, O, ldo, lse + (size_t)h0 * g.S,
                              flush));
    if (!overlap && c + 1 < g.nchunks) UPIPE_TRY(out_gemm(c, st, ds->num_sms, true));
  }
  if (pair) {
    // pairs 0 .. np - 1 went to the side stream (chunks 0 .. 2 np - 1); the
    // one or two chunks left follow on the caller's stream with every SM
    const int np = (g.nchunks - 1) / 2;
    UPIPE_CUDA(cudaStreamWaitEvent(st, ev.out[(np - 1) & 1], 0));
    ev.joined = true;
    if (g.nchunks - 2 * np == 2) UPIPE_TRY(out_gemm_pair(2 * np, st, ds->num_sms, true));
    else UPIPE_TRY(out_gemm(g.nchunks - 1, st, ds->num_sms, true));
    return UPIPE_OK;
  }
  if (overlap) {
    UPIPE_CUDA(cudaStreamWaitEvent(st, ev.out[(g.nchunks - 2) & 1], 0));
    ev.joined = true;
  }
  UPIPE_TRY(out_gemm(g.nchunks - 1, st, ds->num_sms, true));
  return UPIPE_OK;
}

extern "C" int upipe_attn_fwd(const upipe_shape_t* shape, const upipe_bf16* x,
                              const upipe_bf16* Wq, const upipe_bf16* Wk, const upipe_bf16* Wv,
                              const upipe_bf16* Wo, const float* q_norm_w, const float* k_norm_w,
                              float* out, float* lse, void* workspace, size_t ws_bytes,
                              upipe_bf16* attn_o, void* stream) {
  return attn_fwd_impl(shape, x, Wq, Wk, Wv, Wo, q_norm_w, k_norm_w, out, lse, workspace,
                       ws_bytes, attn_o, stream, true);
}

// Forward with the Wo-slice accumulate fused into the attention kernel.  One
// Q buffer serves every chunk: the projection of chunk c + 1 follows chunk
// c's attention on the same stream.  out starts from zero (the chunks' CTAs
// add into it in no fixed order).
extern "C" int upipe_attn_fwd_fused(const upipe_shape_t* shape, const upipe_bf16* x_,
                                    const upipe_bf16* Wq_, const upipe_bf16* Wk_,
                                    const upipe_bf16* Wv_, const upipe_bf16* Wo_,
                                    const float* q_norm_w, const float* k_norm_w, float* out,
                                    float* lse, void* workspace, size_t ws_bytes, void* stream) {
  Geo g;
  UPIPE_TRY(check_shape(shape, &g));
  NvtxRange call_range("upipe_attn_fwd_fused");
  const bf16* x = reinterpret_cast<const bf16*>(x_);
  const bf16* Wq = reinterpret_cast<const bf16*>(Wq_);
  const bf16* Wk = reinterpret_cast<const bf16*>(Wk_);
  const bf16* Wv = reinterpret_cast<const bf16*>(Wv_);
  const bf16* Wo = reinterpret_cast<const bf16*>(Wo_);
  if (!x || !Wq || !Wk || !Wv || !Wo || !out || !lse || !workspace) return UPIPE_ERR_INVALID_ARG;
  for (const void* p : {(const void*)x, (const void*)Wq, (const void*)Wk, (const void*)Wv,
                        (const void*)Wo, (const void*)out, (const void*)lse,
                        (const void*)q_norm_w, (const void*)k_norm_w})
    if (p && !aligned16(p)) return UPIPE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return UPIPE_ERR_INVALID_ARG;
  const Layout L = plan(g, 3);
  if (ws_bytes < L.total) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  DeviceState* ds = nullptr;
  UPIPE_TRY(device_state(&ds));
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  float2* rhi = at<float2>(workspace, L.rope_hi);
  float2* rlo = at<float2>(workspace, L.rope_lo);
  float2* rlo_t = at<float2>(workspace, L.rope_lo_t);
  __half* Q = at<__half>(workspace, L.q);
  __half* K = at<__half>(workspace, L.k);
  __half* V = at<__half>(workspace, L.v);
  float* flush = L.flush == (size_t)-1 ? nullptr : at<float>(workspace, L.flush);
  UPIPE_CUDA(launch_rope_table(rhi, rlo, rlo_t, g.S, g.d, shape->rope_theta, st, ds->err));

  CUtensorMap xmap, outmap, womap;
  UPIPE_MAP(&xmap, x, g.S, g.hidden, g.hidden, 128, 64);
  if (!make_tmap_f32(&outmap, out, g.S, g.hidden, g.hidden, 32, 32)) return UPIPE_ERR_CUDA;
  UPIPE_MAP(&womap, Wo, g.hidden, (uint64_t)g.Hq * g.d, (uint64_t)g.Hq * g.d, 128, 64);
  UPIPE_CUDA(cudaMemsetAsync(out, 0, (size_t)g.S * g.hidden * sizeof(float), st));
  for (int c = 0; c < g.nchunks; ++c) {
    NvtxRange chunk_range("upipe_attn_fwd_fused", c);
    const int h0 = c * g.ch;
    const int kv0 = h0 / g.g;
    const bool new_group = (g.ch >= g.g) || (h0 % g.g == 0);
    UPIPE_TRY(project_chunk(g, ds, st, xmap, Wq, Wk, Wv, q_norm_w, k_norm_w, shape->norm_eps, h0,
                            kv0, new_group, Q, K, V, rhi, rlo_t, nullptr, nullptr, nullptr,
                            nullptr));
    UPIPE_TRY(attention_chunk(g, ds, st, Q, K, V, h0, kv0, nullptr, 0, lse + (size_t)h0 * g.S,
                              flush, nullptr, 0, nullptr, &womap, &outmap));
  }
  return UPIPE_OK;
}

namespace upipe {
int attn_fwd_unforked(const upipe_shape_t* shape, const upipe_bf16* x, const upipe_bf16* Wq,
                      const upipe_bf16* Wk, const upipe_bf16* Wv, const upipe_bf16* Wo,
                      const float* q_norm_w, const float* k_norm_w, float* out, float* lse,
                      void* workspace, size_t ws_bytes, void* stream) {
  return attn_fwd_impl(shape, x, Wq, Wk, Wv, Wo, q_norm_w, k_norm_w, out, lse, workspace,
                       ws_bytes, nullptr, stream, false);
}
}  // namespace upipe

// The backward of both entry points.  o_saved: nullptr (recompute each
// chunk's attention output in the workspace) or the forward's per-head
// attention output [S, Hq*d] bf16.
static int attn_bwd_impl(const upipe_shape_t* shape, const upipe_bf16* x_,
                         const upipe_bf16* Wq_, const upipe_bf16* Wk_, const upipe_bf16* Wv_,
                         const upipe_bf16* Wo_, const float* q_norm_w, const float* k_norm_w,
                         const upipe_bf16* dout_, const float* lse, const upipe_bf16* o_saved_,
                         float* dx, float* dWq, float* dWk, float* dWv, float* dWo,
                         float* dq_norm_w, float* dk_norm_w, void* workspace, size_t ws_bytes,
                         void* stream) {
  Geo g;
  UPIPE_TRY(check_shape(shape, &g));
  NvtxRange call_range("upipe_attn_bwd");
  const bf16* o_saved = reinterpret_cast<const bf16*>(o_saved_);
  if (o_saved && !aligned16(o_saved)) return UPIPE_ERR_INVALID_ARG;
  const bf16* x = reinterpret_cast<const bf16*>(x_);
  const bf16* Wq = reinterpret_cast<const bf16*>(Wq_);
  const bf16* Wk = reinterpret_cast<const bf16*>(Wk_);
  const bf16* Wv = reinterpret_cast<const bf16*>(Wv_);
  const bf16* Wo = reinterpret_cast<const bf16*>(Wo_);
  const bf16* dout = reinterpret_cast<const bf16*>(dout_);
  if (!x || !Wq || !Wk || !Wv || !Wo || !dout || !lse || !dx || !dWq || !dWk || !dWv || !dWo ||
      !workspace)
    return UPIPE_ERR_INVALID_ARG;
  if (g.norm && (!dq_norm_w || !dk_norm_w)) return UPIPE_ERR_INVALID_ARG;
  for (const void* p : {(const void*)x, (const void*)Wq, (const void*)Wk, (const void*)Wv,
                        (const void*)Wo, (const void*)dout, (const void*)lse, (const void*)dx,
                        (const void*)dWq, (const void*)dWk, (const void*)dWv, (const void*)dWo,
                        (const void*)q_norm_w, (const void*)k_norm_w, (const void*)dq_norm_w,
                        (const void*)dk_norm_w})
    if (p && !aligned16(p)) return UPIPE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return UPIPE_ERR_INVALID_ARG;
  const Layout L = plan(g, 1);
  if (ws_bytes < L.total) return UPIPE_ERR_WORKSPACE_TOO_SMALL;
  DeviceState* ds = nullptr;
  UPIPE_TRY(device_state(&ds));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int d = g.d;
  const size_t S = (size_t)g.S;

  float2* rhi = at<float2>(workspace, L.rope_hi);
  float2* rlo = at<float2>(workspace, L.rope_lo);
  float2* rlo_t = at<float2>(workspace, L.rope_lo_t);
  // Q, K, V and dO' hold fp16 operands of the attention kernels; once those
  // are done, their buffers take the bf16 hi parts of the gradients
  __half* Q = at<__half>(workspace, L.q);
  __half* K = at<__half>(workspace, L.k);
  __half* V = at<__half>(workspace, L.v);
  bf16* Ows = at<bf16>(workspace, L.o);
  float* flush = L.flush == (size_t)-1 ? nullptr : at<float>(workspace, L.flush);
  __half* dO = at<__half>(workspace, L.dO);
  bf16* dO_hi = reinterpret_cast<bf16*>(dO);
  bf16* K_hi = reinterpret_cast<bf16*>(K);
  bf16* V_hi = reinterpret_cast<bf16*>(V);
  float* sc = at<float>(workspace, L.sc);
  float* Dv = at<float>(workspace, L.D);
  float* dQ = at<float>(workspace, L.dq);
  float* dK = at<float>(workspace, L.dk);
  float* dV = at<float>(workspace, L.dv);
  bf16* dKlo = at<bf16>(workspace, L.dklo);
  bf16* dVlo = at<bf16>(workspace, L.dvlo);
  float* yq = g.norm ? at<float>(workspace, L.yq) : nullptr;
  float* rq = g.norm ? at<float>(workspace, L.rq) : nullptr;
  float* yk = g.norm ? at<float>(workspace, L.yk) : nullptr;
  float* rk = g.norm ? at<float>(workspace, L.rk) : nullptr;

  UPIPE_CUDA(launch_rope_table(rhi, rlo, rlo_t, g.S, d, shape->rope_theta, st, ds->err));
  // the fp16 gradient scales: norm maxima start at zero; the dO scale's
  // bound (max ||dout_i||, max ||Wo[:, j]||) is taken once per call
  UPIPE_CUDA(cudaMemsetAsync(sc, 0, sizeof(float) * (size_t)(2 + g.Hkv + g.nchunks), st));
  UPIPE_CUDA(launch_grad_bound(dout, g.S, g.hidden, Wo, g.Hq * d, sc, st, ds->err));
  // split-K weight gradients accumulate with reductions: start from zero
  UPIPE_CUDA(cudaMemsetAsync(dWq, 0, sizeof(float) * (size_t)g.Hq * d * g.hidden, st));
  UPIPE_CUDA(cudaMemsetAsync(dWk, 0, sizeof(float) * (size_t)g.Hkv * d * g.hidden, st));
  UPIPE_CUDA(cudaMemsetAsync(dWv, 0, sizeof(float) * (size_t)g.Hkv * d * g.hidden, st));
  UPIPE_CUDA(cudaMemsetAsync(dWo, 0, sizeof(float) * (size_t)g.Hq * d * g.hidden, st));
  if (g.norm) {
    UPIPE_CUDA(cudaMemsetAsync(dq_norm_w, 0, sizeof(float) * d, st));
    UPIPE_CUDA(cudaMemsetAsync(dk_norm_w, 0, sizeof(float) * d, st));
  }

  CUtensorMap xmap, x_mn, dout_k, dout_mn, dxmap;
  if (!make_tmap_f32(&dxmap, dx, g.S, g.hidden, g.hidden, 32, 32)) return UPIPE_ERR_CUDA;
  UPIPE_MAP(&xmap, x, g.S, g.hidden, g.hidden, 128, 64);       // A, K-major
  UPIPE_MAP(&x_mn, x, g.S, g.hidden, g.hidden, 64, 64);        // B of dW = dA^T x (MN-major)
  UPIPE_MAP(&dout_k, dout, g.S, g.hidden, g.hidden, 128, 64);  // A of dO = dout Wo_c
  UPIPE_MAP(&dout_mn, dout, g.S, g.hidden, g.hidden, 64, 64);  // A of dWo = dout^T O
  const int dx_bn = (g.hidden % 256 == 0) ? 256 : 128;
  bool dx_started = false;

  // dx (+)= sum_s dA_s W_s: one GEMM whose K range runs through the chunk's
  // projection-output gradients (each as a bf16 hi and lo half) in turn, so
  // that dx is read and written once per chunk.  W_s is the weight slice
  // [ncols_s rows, hidden] that produced dA_s [S, ncols_s].
  struct DxSeg {
    const bf16* dA;
    int ncols;
    const bf16* W;
  };
  auto dx_gemm = [&](const DxSeg* segs, int nseg) -> int {
    CUtensorMap am[kMaxASegs], bm[kMaxBMaps];
    GemmArgs ga{(int)g.S, g.hidden, 0, 1, d};
    ga.nkseg = nseg;
    const bf16* bw[kMaxBMaps] = {};  // weight slice behind each B map
    int nb = 0, kb = 0;
    for (int s = 0; s < nseg; ++s) {
      UPIPE_MAP(&am[s], segs[s].dA, g.S, (uint64_t)segs[s].ncols, (uint64_t)segs[s].ncols, 128,
                64);
      int b = 0;
      while (b < nb && bw[b] != segs[s].W) ++b;
      if (b == nb) {
        if (nb == kMaxBMaps) return UPIPE_ERR_INVALID_ARG;
        UPIPE_MAP(&bm[nb], segs[s].W, (uint64_t)segs[s].ncols, g.hidden, g.hidden, 64, 64);
        bw[nb++] = segs[s].W;
      }
      kb += segs[s].ncols / 64;
      ga.kseg_end[s] = kb;
      ga.kseg_a[s] = s;
      ga.kseg_b[s] = b;
    }
    ga.K = kb * 64;
    EpiParams ep{};
    ep.C = dx;
    ep.ldc = g.hidden;
    ep.beta = dx_started ? 1 : 0;
    UPIPE_CUDA(launch_gemm(dx_bn, false, true, EPI_F32, am, nseg, bm, nb, ga, ep, ds->err,
                           ds->num_sms, st, &dxmap));
    dx_started = true;
    return UPIPE_OK;
  };
  // dW (+)= dA^T x for every part of the chunk in one split-K GEMM: the parts
  // are M segments (one A map and one output each; a weight's hi and lo parts
  // add into the same rows), so the chunk reads x once, not once per part.
  struct DwSeg {
    const bf16* dA;  // [S, ncols] bf16
    int ncols;
    float* dW;       // [ncols rows, hidden] fp32
  };
  auto dw_gemm = [&](const DwSeg* segs, int nseg) -> int {
    CUtensorMap am[kMaxASegs];
    GemmArgs ga{0, g.hidden, (int)g.S, 1, d};
    EpiParams ep{};
    ep.ldc = g.hidden;
    ga.nmseg = nseg;
    int tiles = 0;
    for (int s = 0; s < nseg; ++s) {
      UPIPE_MAP(&am[s], segs[s].dA, g.S, (uint64_t)segs[s].ncols, (uint64_t)segs[s].ncols, 64,
                64);
      ga.mseg_t0[s] = tiles;
      ga.mseg_rows[s] = segs[s].ncols;
      ga.mseg_a[s] = s;
      ep.mseg_c[s] = segs[s].dW;
      tiles += (segs[s].ncols + 127) / 128;
    }
    ga.mseg_t0[nseg] = tiles;
    ga.M = tiles * 128;
    // 256-wide tiles: two operands MN-major at BN = 128 bring 128 bytes into
    // the SM per tensor-core cycle, more than the TMA path feeds
    const int bn = (g.hidden % 256 == 0) ? 256 : 128;
    ga.ksplit = wgrad_splits(g.S, ga.M, g.hidden, bn, ds->num_sms);
    UPIPE_CUDA(launch_gemm(bn, true, true, EPI_F32_ATOMIC, am, nseg, &x_mn, 1, ga, ep, ds->err,
                           ds->num_sms, st));
    return UPIPE_OK;
  };

  for (int c = 0; c < g.nchunks; ++c) {
    NvtxRange chunk_range("upipe_attn_bwd", c);
    const int h0 = c * g.ch;
    const int kv0 = h0 / g.g;
    const bool new_group = (g.ch >= g.g) || (h0 % g.g == 0);
    const bool last_of_group = (g.ch >= g.g) || ((h0 + g.ch) % g.g == 0);
    // 1. recompute Q (and K, V) of the chunk
    float* vmax = sc + 2 + kv0;     // the norm maximum of this group's V rows
    float* do_max = sc + 2 + g.Hkv + c;
    UPIPE_TRY(project_chunk(g, ds, st, xmap, Wq, Wk, Wv, q_norm_w, k_norm_w, shape->norm_eps, h0,
                            kv0, new_group, Q, K, V, rhi, rlo_t, yq, rq, yk, rk, vmax));
    if (new_group) {
      UPIPE_CUDA(cudaMemsetAsync(dK, 0, sizeof(float) * S * g.kvc * d, st));
      UPIPE_CUDA(cudaMemsetAsync(dV, 0, sizeof(float) * S * g.kvc * d, st));
    }
    // the chunk's attention output: recomputed into the workspace, or the
    // forward's saved copy
    const bf16* Oc = o_saved ? o_saved + (size_t)h0 * d : Ows;
    const int ldo = o_saved ? g.Hq * d : g.ch * d;
    // 2. dO'_c = sigma dout Wo_c; D' = rowsum(dO' * O): with the saved O from
    //    its bf16 copy here, else from the fp32 o inside the recomputed
    //    attention (3.), whose fp16 V the attention backward's dP' uses too
    {
      CUtensorMap wom;
      UPIPE_MAP(&wom, Wo + (size_t)h0 * d, g.hidden, (uint64_t)g.ch * d, (uint64_t)g.Hq * d, 64,
                64);
      EpiParams ep{};
      ep.dO = dO;
      ep.ld_do = g.ch * d;
      ep.O = o_saved ? Oc : nullptr;
      ep.ld_o = ldo;
      ep.D = Dv;
      ep.bound = sc;
      ep.do_max = do_max;
      GemmArgs ga{(int)g.S, g.ch * d, g.hidden, 1, d};
      UPIPE_CUDA(launch_gemm(d, false, true, EPI_DO, &dout_k, 1, &wom, 1, ga, ep, ds->err,
                             ds->num_sms, st));
    }
    // 3. the recomputed attention output (and D'), with the forward's LSE:
    //    p = exp(s - lse) needs no online max or row sum
    if (!o_saved)
      UPIPE_TRY(attention_chunk(g, ds, st, Q, K, V, h0, kv0, Ows, g.ch * d, nullptr, flush, dO,
                                g.ch * d, Dv, nullptr, nullptr, lse + (size_t)h0 * g.S));
    // 4. dWo_c = dout^T O_c
    {
      CUtensorMap om;
      UPIPE_MAP(&om, Oc, g.S, (uint64_t)g.ch * d, (uint64_t)ldo, 64, 64);
      EpiParams ep2{};
      ep2.C = dWo + (size_t)h0 * d;
      ep2.ldc = (long long)g.Hq * d;
      const int bn = (g.ch * d) % 128 == 0 ? 128 : 64;
      GemmArgs gb{g.hidden, g.ch * d, (int)g.S,
                  wgrad_splits(g.S, g.hidden, g.ch * d, bn, ds->num_sms), d};
      UPIPE_CUDA(launch_gemm(bn, true, true, EPI_F32_ATOMIC, &dout_mn, 1, &om, 1, gb, ep2, ds->err,
                             ds->num_sms, st));
    }
    // 5. attention backward: dQ_c (fresh), dK/dV (accumulated over the group)
    UPIPE_CUDA(cudaMemsetAsync(dQ, 0, sizeof(float) * S * g.ch * d, st));
    {
      AttnBwdArgs a{};
      a.S = (int)g.S;
      a.heads = g.ch;
      a.group = g.g;
      a.h0 = h0;
      a.kv0 = kv0;
      a.d = d;
      a.Q = Q;
      a.ldq = g.ch * d;
      a.K = K;
      a.V = V;
      a.ldkv = g.kvc * d;
      a.dO = dO;
      a.ld_do = g.ch * d;
      a.lse = lse + (size_t)h0 * S;
      a.lse_stride = g.S;
      a.D = Dv;
      a.dQ = dQ;
      a.ld_dq = g.ch * d;
      a.dK = dK;
      a.dV = dV;
      a.ld_dkv = g.kvc * d;
      a.scale = (float)(1.0 / std::sqrt((double)d));
      a.bound = sc;
      a.vmax = vmax;
      a.do_max = do_max;
      a.walk = bwd_walk(g.S);
      prof_begin(1, st);
      const cudaError_t e = launch_attn_bwd(a, ds->err, st);
      prof_end(1, st);
      UPIPE_CUDA(e);
    }
    // 6. dQ -> gradient of the Q projection output (RoPE^T, RMSNorm backward)
    //    as bf16 hi (into the dO buffer: dO is dead now) + lo (into the O
    //    buffer: O is dead after the dO / dWo GEMMs); dx += dA_q Wq_c;
    //    dWq_c = dA_q^T x, each as a hi and a lo GEMM
    {
      QkBwdArgs q{};
      q.err = ds->err;
      q.S = g.S;
      q.heads = g.ch;
      q.d = d;
      q.g = dQ;
      q.ld_g = g.ch * d;
      q.out = dO_hi;
      q.out_lo = Ows;
      q.ld_out = g.ch * d;
      q.mode = g.norm ? PROJ_NORM_ROPE : PROJ_ROPE;
      q.yhat = yq;
      q.ld_yhat = g.ch * d;
      q.rstd = rq;
      q.gamma = q_norm_w;
      q.dgamma = dq_norm_w;
      q.rope_hi = rhi;
      q.rope_lo = rlo;
      prof_begin(3, st);
      UPIPE_CUDA(launch_qk_bwd(q, st));
      prof_end(3, st);
    }
    const bf16* Wq_c = Wq + (size_t)h0 * d * g.hidden;
    DxSeg dxs[kMaxASegs] = {{dO_hi, g.ch * d, Wq_c}, {Ows, g.ch * d, Wq_c}};
    float* dWq_c = dWq + (size_t)h0 * d * g.hidden;
    DwSeg dws[kMaxASegs] = {{dO_hi, g.ch * d, dWq_c}, {Ows, g.ch * d, dWq_c}};
    int ndx = 2;
    // 7. at the group's last chunk: dK -> dA_k (hi over K, lo beside it),
    //    dV -> hi over V and lo beside it
    if (last_of_group) {
      QkBwdArgs q{};
      q.err = ds->err;
      q.S = g.S;
      q.heads = g.kvc;
      q.d = d;
      q.g = dK;
      q.ld_g = g.kvc * d;
      q.out = K_hi;
      q.out_lo = dKlo;
      q.ld_out = g.kvc * d;
      q.mode = g.norm ? PROJ_NORM_ROPE : PROJ_ROPE;
      q.yhat = yk;
      q.ld_yhat = g.kvc * d;
      q.rstd = rk;
      q.gamma = k_norm_w;
      q.dgamma = dk_norm_w;
      q.rope_hi = rhi;
      q.rope_lo = rlo;
      prof_begin(3, st);
      UPIPE_CUDA(launch_qk_bwd(q, st));
      prof_end(3, st);
      prof_begin(4, st);
      UPIPE_CUDA(launch_f32_to_bf16x2(dV, g.kvc * d, V_hi, dVlo, g.kvc * d, g.S, g.kvc * d, st,
                                      ds->err));
      prof_end(4, st);
      const bf16* Wk_g = Wk + (size_t)kv0 * d * g.hidden;
      const bf16* Wv_g = Wv + (size_t)kv0 * d * g.hidden;
      float* dWk_g = dWk + (size_t)kv0 * d * g.hidden;
      float* dWv_g = dWv + (size_t)kv0 * d * g.hidden;
      for (int part = 0; part < 2; ++part) {
        const bf16* gk = part ? dKlo : K_hi;
        const bf16* gv = part ? dVlo : V_hi;
        dws[ndx] = {gk, g.kvc * d, dWk_g};
        dxs[ndx++] = {gk, g.kvc * d, Wk_g};
        dws[ndx] = {gv, g.kvc * d, dWv_g};
        dxs[ndx++] = {gv, g.kvc * d, Wv_g};
      }
    }
    // 8. dWq (and the group's dWk, dWv) and dx (+)= the chunk's Q part (and
    //    the group's K and V parts), each as one GEMM over all parts
    UPIPE_TRY(dw_gemm(dws, ndx));
    UPIPE_TRY(dx_gemm(dxs, ndx));
  }
  return UPIPE_OK;
}

extern "C" int upipe_attn_bwd(const upipe_shape_t* shape, const upipe_bf16* x,
                              const upipe_bf16* Wq, const upipe_bf16* Wk, const upipe_bf16* Wv,
                              const upipe_bf16* Wo, const float* q_norm_w, const float* k_norm_w,
                              const upipe_bf16* dout, const float* lse, float* dx, float* dWq,
                              float* dWk, float* dWv, float* dWo, float* dq_norm_w,
                              float* dk_norm_w, void* workspace, size_t ws_bytes, void* stream) {
  return attn_bwd_impl(shape, x, Wq, Wk, Wv, Wo, q_norm_w, k_norm_w, dout, lse, nullptr, dx, dWq,
                       dWk, dWv, dWo, dq_norm_w, dk_norm_w, workspace, ws_bytes, stream);
}

extern "C" int upipe_attn_bwd_saved_o(const upipe_shape_t* shape, const upipe_bf16* x,
                                      const upipe_bf16* Wq, const upipe_bf16* Wk,
                                      const upipe_bf16* Wv, const upipe_bf16* Wo,
                                      const float* q_norm_w, const float* k_norm_w,
                                      const upipe_bf16* dout, const float* lse,
                                      const upipe_bf16* attn_o, float* dx, float* dWq, float* dWk,
                                      float* dWv, float* dWo, float* dq_norm_w, float* dk_norm_w,
                                      void* workspace, size_t ws_bytes, void* stream) {
  if (!attn_o) return UPIPE_ERR_INVALID_ARG;
  return attn_bwd_impl(shape, x, Wq, Wk, Wv, Wo, q_norm_w, k_norm_w, dout, lse, attn_o, dx, dWq,
                       dWk, dWv, dWo, dq_norm_w, dk_norm_w, workspace, ws_bytes, stream);
}

extern "C" void upipe_profile_attach(int kernel, void* const* start_events,
                                     void* const* end_events, int capacity) {
  g_prof.kernel = capacity > 0 ? kernel : -1;
  g_prof.starts = start_events;
  g_prof.ends = end_events;
  g_prof.capacity = capacity > 0 ? capacity : 0;
  g_prof.count = 0;
}

extern "C" int upipe_profile_count(void) { return g_prof.count; }

extern "C" int upipe_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us <= 0 || limit_us > 1000000) return UPIPE_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  UPIPE_TRY(device_state(&ds));
  UPIPE_CUDA(launch_selftest_wait(ds->err, (unsigned long long)limit_us * 1000ull,
                                  static_cast<cudaStream_t>(stream)));
  return UPIPE_OK;
}

namespace upipe {
int device_context(int** err, int* num_sms) {
  DeviceState* ds = nullptr;
  UPIPE_TRY(device_state(&ds));
  *err = ds->err;
  *num_sms = ds->num_sms;
  return UPIPE_OK;
}
}  // namespace upipe

extern "C" int upipe_debug_bounds(void) {
#ifdef UPIPE_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

extern "C" int upipe_selftest_bounds(void* stream, int* written) {
  if (!written) return UPIPE_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  UPIPE_TRY(device_state(&ds));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  UPIPE_CUDA(launch_selftest_bounds(ds->err, st));
  UPIPE_CUDA(cudaStreamSynchronize(st));
  UPIPE_CUDA(selftest_bounds_probe_written(written));
  return UPIPE_OK;
}

extern "C" int upipe_last_error(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return UPIPE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return UPIPE_ERR_CUDA;
  const int zero = 0;
  if (v != 0 && cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess)
    return UPIPE_ERR_CUDA;
  return v;
}

extern "C" const char* upipe_strerror(int code) {
  switch (code) {
    case UPIPE_OK: return "ok";
    case UPIPE_ERR_INVALID_ARG: return "invalid argument";
    case UPIPE_ERR_UNSUPPORTED: return "unsupported shape";
    case UPIPE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case UPIPE_ERR_CUDA: return "CUDA error";
    case UPIPE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case UPIPE_ERR_RANGE: return "projected value outside the fp16 range";
    case UPIPE_ERR_BOUNDS: return "device bounds check failed (debug build)";
    case UPIPE_ERR_TARGET: return "loss target outside the vocabulary";
    default: return "unknown error";
  }
}
