// Internal (not exported) interfaces between the translation units of
// libupipe: kernel launchers and their parameter blocks.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/upipe.h"

namespace upipe {

// Sets a kernel's dynamic shared memory limit once per device (thread-safe:
// concurrent first calls both set it, which is harmless).  ``done`` is the
// kernel's own bit mask of devices already set up.
template <typename Kernel>
cudaError_t smem_attr_once(Kernel* kernel, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

using bf16 = __nv_bfloat16;

// ----------------------------------------------------------- tensor maps --

// Encode a 2-D tensor map of 16-bit elements over a row-major matrix [rows,
// cols] with leading dimension ``ld`` elements, box [box_rows, box_cols]
// (box_cols * 2 must be 128: 128-byte swizzle).  The map is declared bf16; it
// carries fp16 data as well (TMA copies the bits, and its zero fill is zero in
// both types).  Returns false when the driver refuses.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint64_t ld, uint32_t box_rows, uint32_t box_cols);

// The same for an fp32 matrix; box_cols * 4 must be 128 (128-byte swizzle).
bool make_tmap_f32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                   uint64_t ld, uint32_t box_rows, uint32_t box_cols);

// ------------------------------------------------- backward fp16 scales --
//
// The attention backward runs its MMAs in fp16 (11 significant bits), whose
// range (normal numbers 2^-14 .. 65504) is far narrower than bf16's.  Three
// quantities pass through fp16 there, each with a power-of-two factor chosen
// on the device from exact norms, so that nothing overflows and small values
// stay normal; the factors are exact and are divided out of dQ, dK and dV:
//   P''  = rho * P,       rho = 2^14  (0 <= P <= 1, so P'' <= 2^14)
//   dO'  = sigma * dO,    sigma = 2^(13 - floor(log2(Mdout * Wcol)))
//          with Mdout = max_i ||dout_i||_2 and Wcol = max_j ||Wo[:, j]||_2, so
//          |dO'_ij| <= sigma * ||dout_i|| ||Wo[:, j]|| < 2^14
//   dS'' = P'' (lambda dP' - lambda D') = lambda rho sigma dS,
//          lambda = 2^(-1 - floor(log2(MdO' * Vmax))), MdO' = max ||dO'_i||_2
//          over the chunk's rows and heads, Vmax = max_j ||v_j||_2 of its
//          KV group: |dP'_ij| <= MdO' Vmax and |D'_i| <= MdO' max||o_i|| <=
//          MdO' Vmax, so |dS''| <= rho * 2 * lambda MdO' Vmax < 2^15.
// The scalars live in the backward workspace, zeroed at the start of a call:
//   [0] Mdout   [1] Wcol   [2 + kv0] Vmax of the group starting at kv head kv0
//   [2 + Hkv + c] MdO' of chunk c
constexpr float kGradRho = 16384.0f;   // rho, and its log2 below
constexpr float kGradRhoLog2 = 14.0f;

// 2^e as a float for |e| <= 100.
__host__ __device__ inline float pow2i(int e) {
  e = e < -100 ? -100 : (e > 100 ? 100 : e);
  union { unsigned int u; float f; } v;
  v.u = (unsigned int)(e + 127) << 23;
  return v.f;
}

// floor(log2(v)) for a finite v > 0 (subnormals count as 2^-127).
__host__ __device__ inline int floor_log2(float v) {
  union { float f; unsigned int u; } b;
  b.f = v;
  return (int)((b.u >> 23) & 255u) - 127;
}

// 2^(top - floor(log2(m))) for a finite m > 0; 1 otherwise (all-zero or
// non-finite inputs: the factor then does not matter).
__host__ __device__ inline float pow2_scale_for(float m, int top) {
  if (!(m > 0.f) || !(m <= 3.0e38f)) return 1.f;
  return pow2i(top - floor_log2(m));
}

__host__ __device__ inline float grad_sigma(const float* bound) {
  return pow2_scale_for(bound[0] * bound[1], 13);
}
__host__ __device__ inline float grad_lambda(float do_max, float vmax) {
  return pow2_scale_for(do_max * vmax, -1);
}

// max_i ||dout_i||_2 -> bound[0] and max_j ||Wo[:, j]||_2 -> bound[1]
// (atomic maxima: bound must start at zero).
cudaError_t launch_grad_bound(const bf16* dout, long long S, int hidden, const bf16* Wo,
                              int ncols, float* bound, cudaStream_t stream, int* err);

// ------------------------------------------------------------------ GEMM --

enum EpiKind : int {
  EPI_PROJ = 0,        // fp16 store with optional per-head RMSNorm and RoPE
  EPI_F32 = 1,         // fp32 store (beta = 0) or read-modify-write add (beta = 1)
  EPI_DO = 2,          // scaled fp16 store of dO plus D = rowsum(dO * O) per head
  EPI_F32_ATOMIC = 3,  // fp32 reduction-add (split-K partial sums)
  EPI_SWIGLU = 4,      // MLP gate/up: a = silu(g) * u, bf16 store
  EPI_SWIGLU_BWD = 5,  // MLP gate/up recomputed: dg, du (from dA) and a, bf16 stores
  EPI_LSE_PART = 6,    // loss logits: per row and column tile, (max, sum of exp) partials
  EPI_DLOGITS = 7,     // loss logits recomputed: dz = scale (softmax - onehot), bf16 store
};

enum ProjMode : int { PROJ_PLAIN = 0, PROJ_ROPE = 1, PROJ_NORM_ROPE = 2 };

// One contiguous run of output columns of the fused projection GEMM.  The
// GEMM's N range [n_begin, n_end) comes from B map ``bmap`` starting at
// weight row ``b_row0`` and lands in ``out`` (row stride ``ld``) starting at
// column ``col0``, as fp16 (the attention kernels' operand type).  A value
// outside fp16's range sets kErrRange in the error word.
struct ProjSeg {
  int n_begin, n_end;
  int bmap;
  int b_row0;
  __half* out;
  int ld;
  int col0;
  int mode;
  const float* gamma;  // RMSNorm gain [d], nullptr means ones
  float* yhat;         // optional: normalised, pre-gain, pre-RoPE values (fp32)
  int ld_yhat;
  float* rstd;         // optional: 1/sqrt(mean(a^2)+eps) per (head, row): [heads][rows]
  float* norm_max;     // optional: running max over rows and heads of ||row||_2
};

struct EpiParams {
  // EPI_PROJ
  ProjSeg seg[3];
  int nseg;
  const float2* rope_hi;  // [(S >> 10) + 1][d/2] (cos, sin) of (pos & ~1023) * w_i
  const float2* rope_lo_t;  // [d/2][1024]        (cos, sin) of (pos & 1023) * w_i
  float eps;
  // EPI_F32 / EPI_F32_ATOMIC
  float* C;
  long long ldc;
  int beta;          // EPI_F32: 0 store, 1 add (both through the C tensor map)
  // EPI_F32_ATOMIC with M segments: output base of each segment (row 0)
  float* mseg_c[6];
  // EPI_DO: dO' = sigma * dO in fp16 with sigma = grad_sigma(bound), the
  // running max of ||dO'_row||_2 over rows and heads in *do_max, and (when O
  // is given: the saved-O backward) D' = rowsum(dO' * O) from the stored fp16
  // dO'
  __half* dO;
  int ld_do;
  const bf16* O;
  int ld_o;
  float* D;  // [heads][M]
  const float* bound;   // [Mdout, Wcol] (backward fp16 scales, above)
  float* do_max;
  // EPI_SWIGLU / EPI_SWIGLU_BWD: B map 0 holds the gate weights Wg, B map 1
  // the up weights Wu ([ffn, K] each); output tile n of N = 2 ffn is gate rows
  // and up rows [128 n, 128 n + 128), i.e. columns [128 n, 128 n + 128) of
  // a = silu(g) * u [M, ffn] (bf16, row stride ld_act).  EPI_SWIGLU_BWD also
  // reads dA [M, ffn] fp32 (row stride ld_da) and stores
  //   dg = dA * u * silu'(g),  du = dA * silu(g)   (bf16, row stride ld_dg)
  bf16* act;
  long long ld_act;
  const float* dA;
  long long ld_da;
  bf16* dG;
  bf16* dU;
  long long ld_dg;
  // EPI_LSE_PART / EPI_DLOGITS (the tiled loss; N = vocabulary, z = logits):
  // targets [M] int32 of the tile's rows.  EPI_LSE_PART stores, for row m and
  // column tile j, part[m * ld_part + j] = (max_v z*log2e, sum_v 2^(z*log2e - max))
  // over the tile's columns, and zt[m] = z[m, targets[m]] from the tile that
  // holds the target.  EPI_DLOGITS reads lse_rows [M] (natural log) and stores
  // dz[m, v] = loss_scale * (exp(z - lse) - [v == target]) in bf16.
  const int* targets;
  float2* part;
  int ld_part;
  float* zt;
  const float* lse_rows;
  bf16* dz;
  long long ld_dz;
  float loss_scale;
};

constexpr int kMaxASegs = 6;  // A tensor maps of one GEMM
constexpr int kMaxBMaps = 3;  // B tensor maps of one GEMM

struct GemmArgs {
  int M, N, K;      // C[M, N] = sum_k A[m, k] * B[n, k]
  int ksplit;       // number of K partitions (EPI_F32_ATOMIC only)
  int head_dim;     // d (EPI_PROJ / EPI_DO)
  // K segments (nkseg > 0): the K range is a concatenation of nkseg runs of
  // 64-wide K blocks; run s ends at block kseg_end[s] (exclusive), reads A from
  // A map kseg_a[s] and B from B map kseg_b[s], each from K coordinate 0.  So
  // C = sum_s A_s B_s^T in one accumulator.  K is then 64 * kseg_end[nkseg-1].
  int nkseg;
  int kseg_end[kMaxASegs];
  int kseg_a[kMaxASegs];
  int kseg_b[kMaxASegs];
  // M segments (nmseg > 0, EPI_F32_ATOMIC): the M range is a concatenation of
  // nmseg runs of 128-row tiles; run s covers tiles [mseg_t0[s], mseg_t0[s+1]),
  // reads A from A map mseg_a[s] (rows from 0) and adds its mseg_rows[s] rows
  // into EpiParams::mseg_c[s] (row stride ldc).  M is then 128 * mseg_t0[nmseg].
  int nmseg;
  int mseg_t0[kMaxASegs + 1];
  int mseg_rows[kMaxASegs];
  int mseg_a[kMaxASegs];
  // tile order: 0 column tiles fastest (the default: A row blocks are
  // reused, B cycles), 1 row blocks fastest (B column tiles are reused and A
  // cycles: the order for an A much smaller than B, which then stays in L2),
  // G > 1 row blocks fastest within groups of G row blocks (B read once per
  // group; for an A too large to stay in L2 as a whole)
  int m_fastest;
};

// a_mn / b_mn: operand stored MN-major (A as [K, M] row-major, B as [K, N]).
// amaps: 1..kMaxASegs maps for A (more than one only with K segments).
// bmaps: 1..kMaxBMaps maps for B (EPI_PROJ may use one per segment, K
// segments one per run).
// cmap: for EPI_F32, an fp32 tensor map over C with box 32 x 32 (128-byte
// swizzle); the epilogue stores (beta 0) or reduce-adds (beta 1) through it.
cudaError_t launch_gemm(int bn, bool a_mn, bool b_mn, EpiKind epi, const CUtensorMap* amaps,
                        int namaps, const CUtensorMap* bmaps, int nbmaps, const GemmArgs& g,
                        const EpiParams& ep, int* err, int num_sms, cudaStream_t stream,
                        const CUtensorMap* cmap = nullptr);

// ------------------------------------------------------------- attention --

// Q, K, V: fp16 [S, heads*d] / [S, kv heads*d] through the tensor maps.
struct AttnFwdArgs {
  int S;
  int heads;        // query heads in this launch
  int group;        // query heads per kv head (GQA)
  int h0;           // global index of the first query head (kv map)
  int kv0;          // global index of the first kv head held in K/V buffers
  bf16* O;          // [S, ldo] bf16, head i at column i*d
  int ldo;
  float* lse;       // [heads][S] natural-log LSE (nullptr: not written)
  long long lse_stride;
  float scale_log2; // log2(e) / sqrt(d)
  float* flush;     // nullptr, or [kFlushSlots][256 rows][d] fp32 per-SM O accumulators
  // optional (the backward's recompute): D'_i = dO'_i . o_i from the fp32 o
  // before its bf16 rounding, so that D' matches the dP' = dO' v^T the
  // attention backward forms from the same fp16 V
  const __half* dO; int ld_do;  // [S, ld_do] fp16, head i at column i*d
  float* D;                     // [heads][S]
  // fused Wo-slice accumulate (launch with womap / outmap; O and dO null):
  // the hidden / 128 column blocks of out each CTA adds its rows into
  int wo_tiles;
  // nullptr, or the forward's LSE of these heads ([heads][lse_stride],
  // natural log; then lse must be nullptr): the backward's recompute takes
  // p = exp(s - lse) directly instead of the online softmax
  const float* lse_in;
};

// The attention forward folds its TMEM O accumulator into an fp32 row in
// global memory every kFlushTiles KV tiles (see attn_fwd.cu); the scratch has
// one slot per SM id and is needed only when S > kFlushTiles * 128.
constexpr int kFlushTiles = 512;
constexpr int kFlushSlots = 256;

// womap / outmap: nullptr (o is stored to a.O), or both (fused Wo-slice
// accumulate): womap over Wo [hidden, Hq*d] bf16 with box [128 rows][64
// cols], outmap over out [S, hidden] fp32 with box [32 rows][32 cols].
cudaError_t launch_attn_fwd(const CUtensorMap& qmap, const CUtensorMap& kmap,
                            const CUtensorMap& vmap, const AttnFwdArgs& a, int d, int* err,
                            cudaStream_t stream, const CUtensorMap* womap = nullptr,
                            const CUtensorMap* outmap = nullptr);

struct AttnBwdArgs {
  int S, heads, group, h0, kv0, d;
  const __half* Q; int ldq;     // [S, ldq] fp16
  const __half* K; const __half* V; int ldkv;
  const __half* dO; int ld_do;  // dO' = sigma * dO, fp16
  const float* lse; long long lse_stride;   // caller's LSE, rows of this chunk
  const float* D;               // [heads][S]
  float* dQ; int ld_dq;         // fp32 [S, ld_dq], accumulated
  float* dK; float* dV; int ld_dkv;  // fp32, accumulated across the group's chunks
  float scale;                  // 1/sqrt(d)
  const float* bound;           // GradScales [0], [1] (sigma)
  const float* vmax;            // Vmax of the chunk's KV group
  const float* do_max;          // MdO' of the chunk (lambda)
  int walk;                     // max query sub-tiles (of 64) one CTA walks; even
};

cudaError_t launch_attn_bwd(const AttnBwdArgs& a, int* err, cudaStream_t stream);

// ---------------------------------------------------------- elementwise --

// hi [(S >> 10) + 1][d/2], lo [1024][d/2] and lo_t [d/2][1024] (lo transposed)
cudaError_t launch_rope_table(float2* hi, float2* lo, float2* lo_t, long long S, int d,
                              double theta, cudaStream_t stream, int* err);

// Backward of (RMSNorm ->) RoPE for one block of heads: g (fp32, gradient of
// the rotated values) -> bf16 gradient of the projection output; optionally
// accumulates the gain gradient.
struct QkBwdArgs {
  long long S;
  int heads, d;
  const float* g; int ld_g;          // [S, ld_g] fp32
  bf16* out; int ld_out;             // [S, ld_out] bf16, high part
  bf16* out_lo;                      // [S, ld_out] bf16, low part (value - high)
  int mode;                          // PROJ_ROPE or PROJ_NORM_ROPE
  const float* yhat; int ld_yhat;    // saved normalised values (norm mode, fp32)
  const float* rstd;                 // [heads][S]
  const float* gamma;                // [d] or nullptr
  float* dgamma;                     // [d] accumulated (norm mode)
  const float2* rope_hi; const float2* rope_lo;
  int* err;                          // device error word (debug bounds checks)
};
cudaError_t launch_qk_bwd(const QkBwdArgs& a, cudaStream_t stream);

// fp32 [S, ld_in] -> bf16 high part and bf16 low part (value - high),
// [S, ld_out] each, for ``cols`` columns: hi + lo carries ~16 significant bits.
cudaError_t launch_f32_to_bf16x2(const float* in, int ld_in, bf16* hi, bf16* lo, int ld_out,
                                 long long S, int cols, cudaStream_t stream, int* err);

// The tiled loss's per-row log-sum-exp (natural log) and loss lse - z[target]
// from the logits GEMM's per-tile partials [rows][ntiles] and target logits.
cudaError_t launch_loss_rows(const float2* part, int ntiles, const float* zt, const int* targets,
                             int vocab, long long rows, float* lse, float* loss,
                             cudaStream_t stream, int* err);

// The current device's error word and SM count (created on first use).
int device_context(int** err, int* num_sms);

// Split-K factor for a weight-gradient GEMM with K = S and an [M, N] output of
// BN-wide tiles on ``sms`` SMs.
int wgrad_splits(int64_t S, int M, int N, int bn, int sms);

// NVTX range over the host-side enqueue of one entry point or one chunk
// (header-only NVTX: without a tool attached each push/pop is a no-op call).
struct NvtxRange {
  explicit NvtxRange(const char* what, int chunk = -1);
  ~NvtxRange();
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// upipe_attn_fwd with every launch on the caller's stream: no side stream,
// no events (the static-scratch entry point, which must create nothing).
int attn_fwd_unforked(const upipe_shape_t* shape, const upipe_bf16* x, const upipe_bf16* Wq,
                      const upipe_bf16* Wk, const upipe_bf16* Wv, const upipe_bf16* Wo,
                      const float* q_norm_w, const float* k_norm_w, float* out, float* lse,
                      void* workspace, size_t ws_bytes, void* stream);

// One-CTA kernel whose waits expire after limit_ns (failure-detection test).
cudaError_t launch_selftest_wait(int* err, unsigned long long limit_ns, cudaStream_t stream);
// One-thread kernel whose write lies one element past a declared view (inside
// its array): debug builds refuse it (UPIPE_ERR_BOUNDS); *written after a
// synchronisation tells whether the write happened.
cudaError_t launch_selftest_bounds(int* err, cudaStream_t stream);
cudaError_t selftest_bounds_probe_written(int* written);

}  // namespace upipe
