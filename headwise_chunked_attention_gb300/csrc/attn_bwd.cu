// Causal attention backward for one head chunk (warp-level mma.sync bf16).
//
// For the chunk's heads, given Q, K, V (recomputed in the workspace), dO, the
// forward LSE and D_i = sum_c dO_ic O_ic:
//   P_ij  = exp(q_i . k_j / sqrt(d) - lse_i)            (j <= i)
//   dV_j += sum_i P_ij dO_i
//   dS_ij = P_ij (dO_i . v_j - D_i)
//   dK_j += sum_i dS_ij q_i / sqrt(d),   dQ_i += sum_j dS_ij k_j / sqrt(d)
// (the backward that activation recomputation needs: aipmzone.com /
// dimanyen.com "activation checkpointing"; per-chunk recomputation,
// memeeeeeex.com "Untied Ulysses (UPipe)").
//
// One CTA owns 64 keys of one head and walks the query tiles at or after its
// diagonal.  Each of the 4 warps keeps dK and dV of 16 keys in registers; dQ
// is reduced into fp32 global memory with red.global.add, and dK/dV too at the
// end because the heads of a GQA group (and the chunks of a group) share them.
// Shared-memory tiles use a 16-byte-chunk XOR swizzle so that ldmatrix rows of
// one 8x8 matrix hit distinct banks.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {

namespace {

constexpr int BR = 64;  // queries per step
constexpr int BC = 64;  // keys per CTA
constexpr int kThreads = 128;

__device__ __forceinline__ uint32_t swz(int row, int chunk) { return (uint32_t)(chunk ^ (row & 7)); }

// byte offset of (row, col) in a [rows][COLS] bf16 tile with swizzled 16 B chunks
template <int COLS>
__device__ __forceinline__ uint32_t toff(int row, int col) {
  return (uint32_t)(row * COLS * 2) + (swz(row, col >> 3) << 4) + (uint32_t)((col & 7) * 2);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Load a [64][COLS] bf16 tile (rows r0.., row stride ld elements) into
// swizzled shared memory; rows >= nrows are zero-filled.
template <int COLS>
__device__ __forceinline__ void load_tile(uint32_t sbase, const bf16* g, long long ld, int r0,
                                          int nrows) {
  constexpr int CH = COLS / 8;
  for (int t = threadIdx.x; t < 64 * CH; t += kThreads) {
    const int row = t / CH, ch = t % CH;
    const bool valid = r0 + row < nrows;
    const bf16* src = g + (long long)(valid ? r0 + row : 0) * ld + ch * 8;
    cp_async16(sbase + toff<COLS>(row, ch * 8), src, valid);
  }
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads) attn_bwd_kernel(const AttnBwdArgs a) {
  constexpr int TILE = 64 * D * 2;
  constexpr int NT_D = D / 8;  // n-tiles of 8 along d
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sK = smem_u32(smem);
  const uint32_t sV = sK + TILE;
  const uint32_t sQ = sV + TILE;          // [2] stages
  const uint32_t sdO = sQ + 2 * TILE;     // [2] stages
  const uint32_t sdS = sdO + 2 * TILE;    // [64 keys][64 queries]
  float* s_lse = reinterpret_cast<float*>(smem + 6 * TILE + 64 * 64 * 2);  // [2][64]
  float* s_D = s_lse + 2 * BR;                                             // [2][64]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int jt = blockIdx.x;
  const int head = blockIdx.y;
  const int kvh = (a.h0 + head) / a.group - a.kv0;
  const int S = a.S;
  const int k0 = jt * BC;
  const int nq = (S + BR - 1) / BR;
  const float sl2 = a.scale * 1.4426950408889634f;

  const bf16* Qg = a.Q + head * D;
  const bf16* dOg = a.dO + head * D;
  const bf16* Kg = a.K + kvh * D;
  const bf16* Vg = a.V + kvh * D;
  const float* lse_g = a.lse + (long long)head * a.lse_stride;
  const float* D_g = a.D + (long long)head * S;

  load_tile<D>(sK, Kg, a.ldkv, k0, S);
  load_tile<D>(sV, Vg, a.ldkv, k0, S);
  auto load_q = [&](int it, int stage) {
    const int q0 = it * BR;
    load_tile<D>(sQ + stage * TILE, Qg, a.ldq, q0, S);
    load_tile<D>(sdO + stage * TILE, dOg, a.ld_do, q0, S);
    for (int r = threadIdx.x; r < BR; r += kThreads) {
      const bool v = q0 + r < S;
      s_lse[stage * BR + r] = v ? lse_g[q0 + r] * 1.4426950408889634f : INFINITY;
      s_D[stage * BR + r] = v ? D_g[q0 + r] : 0.f;
    }
  };
  const int i_begin = jt;  // BR == BC: first query tile that sees key k0
  load_q(i_begin, 0);
  cp_async_commit();

  float dk[NT_D][4], dv[NT_D][4];
#pragma unroll
  for (int n = 0; n < NT_D; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[n][e] = dv[n][e] = 0.f;

  const int kw = warp * 16;           // this warp's keys within the tile
  const int lr = lane >> 2;           // fragment row
  const int lc = (lane & 3) * 2;      // fragment column pair

  for (int it = i_begin; it < nq; ++it) {
    const int stage = (it - i_begin) & 1;
    cp_async_wait<0>();
    __syncthreads();
    if (it + 1 < nq) load_q(it + 1, stage ^ 1);
    cp_async_commit();
    const uint32_t q_s = sQ + stage * TILE, do_s = sdO + stage * TILE;
    const float* lse_s = s_lse + stage * BR;
    const float* D_s = s_D + stage * BR;
    const int q0 = it * BR;

    // S^T (16 keys x 64 queries) and dP^T
    float st[8][4], dpt[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[n][e] = dpt[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t ak[4], av[4];
      const int arow = kw + (lane & 15), acol = kk * 16 + (lane >> 4) * 8;
      ldsm_x4(sK + toff<D>(arow, acol), ak[0], ak[1], ak[2], ak[3]);
      ldsm_x4(sV + toff<D>(arow, acol), av[0], av[1], av[2], av[3]);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int brow = p * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int bcol = kk * 16 + ((lane >> 3) & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(q_s + toff<D>(brow, bcol), b0, b1, b2, b3);
        mma16816(st[2 * p], ak, b0, b1);
        mma16816(st[2 * p + 1], ak, b2, b3);
        ldsm_x4(do_s + toff<D>(brow, bcol), b0, b1, b2, b3);
        mma16816(dpt[2 * p], av, b0, b1);
        mma16816(dpt[2 * p + 1], av, b2, b3);
      }
    }
    // P^T, dS^T
    const bool diag = (q0 == k0);
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kw + lr + ((e >> 1) << 3);
        const int q = n * 8 + lc + (e & 1);
        float p = ex2(fmaf(st[n][e], sl2, -lse_s[q]));
        if (diag && key > q) p = 0.f;
        st[n][e] = p;
        dpt[n][e] = p * (dpt[n][e] - D_s[q]);
      }
    // dV += P^T dO ; dK += dS^T Q   (k = queries)
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t ap[4], ad[4];
      ap[0] = pack_bf16(st[2 * kt][0], st[2 * kt][1]);
      ap[1] = pack_bf16(st[2 * kt][2], st[2 * kt][3]);
      ap[2] = pack_bf16(st[2 * kt + 1][0], st[2 * kt + 1][1]);
      ap[3] = pack_bf16(st[2 * kt + 1][2], st[2 * kt + 1][3]);
      ad[0] = pack_bf16(dpt[2 * kt][0], dpt[2 * kt][1]);
      ad[1] = pack_bf16(dpt[2 * kt][2], dpt[2 * kt][3]);
      ad[2] = pack_bf16(dpt[2 * kt + 1][0], dpt[2 * kt + 1][1]);
      ad[3] = pack_bf16(dpt[2 * kt + 1][2], dpt[2 * kt + 1][3]);
#pragma unroll
      for (int dt = 0; dt < D / 16; ++dt) {
        const int brow = kt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int bcol = dt * 16 + (lane >> 4) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(do_s + toff<D>(brow, bcol), b0, b1, b2, b3);
        mma16816(dv[2 * dt], ap, b0, b1);
        mma16816(dv[2 * dt + 1], ap, b2, b3);
        ldsm_x4_t(q_s + toff<D>(brow, bcol), b0, b1, b2, b3);
        mma16816(dk[2 * dt], ad, b0, b1);
        mma16816(dk[2 * dt + 1], ad, b2, b3);
      }
      // dS^T rows (keys) kw + lr (+8), query columns kt*16 + lc (+8)
      uint8_t* ds = smem + 6 * TILE;
      *reinterpret_cast<uint32_t*>(ds + toff<64>(kw + lr, kt * 16 + lc)) = ad[0];
      *reinterpret_cast<uint32_t*>(ds + toff<64>(kw + lr + 8, kt * 16 + lc)) = ad[1];
      *reinterpret_cast<uint32_t*>(ds + toff<64>(kw + lr, kt * 16 + 8 + lc)) = ad[2];
      *reinterpret_cast<uint32_t*>(ds + toff<64>(kw + lr + 8, kt * 16 + 8 + lc)) = ad[3];
    }
    __syncthreads();
    // dQ (queries 16w..16w+15) += dS K  (k = keys)
    {
      float dq[NT_D][4];
#pragma unroll
      for (int n = 0; n < NT_D; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) dq[n][e] = 0.f;
      const int qw = warp * 16;
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        uint32_t as[4];
        // A = dS [query][key] from dS^T stored [key][query]: transposed load
        const int srow = kt * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int scol = qw + ((lane >> 3) & 1) * 8;
        ldsm_x4_t(sdS + toff<64>(srow, scol), as[0], as[1], as[2], as[3]);
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt) {
          const int brow = kt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int bcol = dt * 16 + (lane >> 4) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sK + toff<D>(brow, bcol), b0, b1, b2, b3);
          mma16816(dq[2 * dt], as, b0, b1);
          mma16816(dq[2 * dt + 1], as, b2, b3);
        }
      }
#pragma unroll
      for (int n = 0; n < NT_D; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = q0 + qw + lr + h * 8;
          if (q < S) {
            float* p = a.dQ + (long long)q * a.ld_dq + head * D + n * 8 + lc;
            red_add_f32(p, dq[n][2 * h] * a.scale);
            red_add_f32(p + 1, dq[n][2 * h + 1] * a.scale);
          }
        }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  // dK, dV of this warp's 16 keys
#pragma unroll
  for (int n = 0; n < NT_D; ++n)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int key = k0 + kw + lr + h * 8;
      if (key < S) {
        const long long off = (long long)key * a.ld_dkv + kvh * D + n * 8 + lc;
        red_add_f32(a.dK + off, dk[n][2 * h] * a.scale);
        red_add_f32(a.dK + off + 1, dk[n][2 * h + 1] * a.scale);
        red_add_f32(a.dV + off, dv[n][2 * h]);
        red_add_f32(a.dV + off + 1, dv[n][2 * h + 1]);
      }
    }
}

template <int D>
static cudaError_t launch_bwd_t(const AttnBwdArgs& a, cudaStream_t stream) {
  constexpr int SMEM = 6 * 64 * D * 2 + 64 * 64 * 2 + 4 * 64 * 4;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((a.S + BC - 1) / BC, a.heads);
  attn_bwd_kernel<D><<<grid, kThreads, SMEM, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const AttnBwdArgs& a, cudaStream_t stream) {
  if (a.S <= 0 || a.heads <= 0) return cudaSuccess;
  if (a.d == 128) return launch_bwd_t<128>(a, stream);
  if (a.d == 64) return launch_bwd_t<64>(a, stream);
  return cudaErrorNotSupported;
}

}  // namespace upipe
