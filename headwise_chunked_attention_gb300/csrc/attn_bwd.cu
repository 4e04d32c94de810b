// Causal attention backward for one head chunk on tcgen05.
//
// For the chunk's heads, given Q, K, V (recomputed in the workspace), dO, the
// forward LSE and D_i = sum_c dO_ic O_ic:
//   P_ij  = exp(q_i . k_j / sqrt(d) - lse_i)            (j <= i)
//   dV_j += sum_i P_ij dO_i
//   dS_ij = P_ij (dO_i . v_j - D_i)
//   dK_j += sum_i dS_ij q_i / sqrt(d),   dQ_i += sum_j dS_ij k_j / sqrt(d)
// (the backward that activation recomputation needs: aipmzone.com /
// dimanyen.com "activation checkpointing"; per-chunk recomputation of the
// heads, memeeeeeex.com "Untied Ulysses (UPipe)").
//
// One CTA owns 128 keys (one KV tile) of one head and walks the 128-query
// tiles from its diagonal to the end of the sequence.
//   warps 0-3  softmax-gradient warps: one key row (TMEM lane) per thread;
//              P^T and dS^T from S^T and dP^T, the dQ read-out and its fp32
//              reduction into global memory, the final dK/dV reduction
//   warp 4     TMEM owner and tcgen05.mma issuer
//   warp 5     TMA producer: K, V once, then Q_i, dO_i through 2 stages
// TMEM (512 columns):
//   [  0,128)  S^T = K Q_i^T (fp32); then P^T (bf16, cols 0..63) and
//              dS^T (bf16, cols 64..127), the A operands of the dV / dK MMAs
//   [128,256)  dP^T = V dO_i^T (fp32); then dQ_i = dS K (fp32, D columns)
//   [256,384)  dV accumulator (D columns)     [384,512) dK accumulator
// dS^T is also written to shared memory (128-byte swizzle, query-contiguous)
// where it is the MN-major A operand of dQ = dS K.  Per query tile the tensor
// core runs 5 MMAs of 128 x 128 x {d or 128}; MMAs issued by one thread
// complete in order, which makes the reuse of the TMEM regions safe.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {

namespace {

constexpr int kThreads = 192;
constexpr int BT = 128;  // keys per CTA = queries per step

template <int D>
struct BwdCfg {
  static constexpr uint32_t TILE = BT * D * 2;           // K, V, Q or dO tile
  static constexpr uint32_t BLOCK = BT * 64 * 2;         // one 64-column swizzled block
  static constexpr uint32_t K_OFF = 0;
  static constexpr uint32_t V_OFF = TILE;
  static constexpr uint32_t Q_OFF = 2 * TILE;            // [2] stages
  static constexpr uint32_t DO_OFF = 4 * TILE;           // [2] stages
  static constexpr uint32_t DS_OFF = 6 * TILE;           // dS^T [128 keys][128 queries] bf16
  static constexpr uint32_t BAR_OFF = DS_OFF + BT * BT * 2;
  static constexpr uint32_t SMEM_BYTES = BAR_OFF + 128 + 1024;
  static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 384;
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_kernel(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap domap,
    const AttnBwdArgs a, int* __restrict__ err) {
  using Cfg = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;    // [2]
  uint64_t* q_empty = bars + 3;   // [2]
  uint64_t* s_full = bars + 5;
  uint64_t* p_ready = bars + 6;
  uint64_t* dq_full = bars + 7;
  uint64_t* dq_free = bars + 8;
  uint64_t* mma_done = bars + 9;
  uint64_t* drain_bar = bars + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = a.S;
  const int jt = blockIdx.x;
  const int head = blockIdx.y;
  const int kvh = (a.h0 + head) / a.group - a.kv0;
  const int k0 = jt * BT;
  const int n_it = (S + BT - 1) / BT - jt;  // query tiles jt .. end

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_ready, 4);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 4);
    mbar_init(mma_done, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5 && lane == 0) {
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    prefetch_tmap(&domap);
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 5) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t issued = 0, issued_phase = 0;
      mbar_expect_tx(kv_full, 2 * Cfg::TILE);
      for (int b = 0; b < D / 64; ++b) {
        tma_load_2d(smem + Cfg::K_OFF + b * Cfg::BLOCK, &kmap, kv_full, kvh * D + 64 * b, k0);
        tma_load_2d(smem + Cfg::V_OFF + b * Cfg::BLOCK, &vmap, kv_full, kvh * D + 64 * b, k0);
      }
      for (int it = 0; it < n_it; ++it) {
        const int st = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&q_empty[st], ph ^ 1, err, abort_flag)) break;
        mbar_expect_tx(&q_full[st], 2 * Cfg::TILE);
        const int q0 = (jt + it) * BT;
        for (int b = 0; b < D / 64; ++b) {
          tma_load_2d(smem + Cfg::Q_OFF + st * Cfg::TILE + b * Cfg::BLOCK, &qmap, &q_full[st],
                      head * D + 64 * b, q0);
          tma_load_2d(smem + Cfg::DO_OFF + st * Cfg::TILE + b * Cfg::BLOCK, &domap, &q_full[st],
                      head * D + 64 * b, q0);
        }
        issued |= 1u << st;
        issued_phase = (issued_phase & ~(1u << st)) | (ph << st);
      }
      if (*abort_flag) {
        mbar_wait_drain(kv_full, 0);
        for (int s = 0; s < 2; ++s)
          if (issued & (1u << s)) mbar_wait_drain(&q_full[s], (issued_phase >> s) & 1u);
      }
    }
  } else if (warp == 4) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t ID_ACC = idesc_bf16(128, D, false, true);   // dV, dK (A in TMEM)
      constexpr uint32_t ID_DQ = idesc_bf16(128, D, true, true);     // dQ = dS K
      const uint32_t kb = smem_u32(smem + Cfg::K_OFF);
      const uint32_t vb = smem_u32(smem + Cfg::V_OFF);
      const uint32_t dsb = smem_u32(smem + Cfg::DS_OFF);
      bool ok = mbar_wait(kv_full, 0, err, abort_flag);
      for (int it = 0; it < n_it && ok; ++it) {
        const int st = it & 1;
        if (!mbar_wait(&q_full[st], (it >> 1) & 1, err, abort_flag)) break;
        tc_fence_after();
        const uint32_t qb = smem_u32(smem + Cfg::Q_OFF + st * Cfg::TILE);
        const uint32_t dob = smem_u32(smem + Cfg::DO_OFF + st * Cfg::TILE);
        // S^T = K Q^T  (k over d)
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * Cfg::BLOCK + (k % 4) * 32;
          mma_ss(tmem + Cfg::COL_S, sdesc_sw128(kb + off, 16, 1024),
                 sdesc_sw128(qb + off, 16, 1024), ID_S, k > 0);
        }
        // dP^T = V dO^T, into the region dQ of the previous step used
        if (it > 0) {
          if (!mbar_wait(dq_free, (it - 1) & 1, err, abort_flag)) break;
          tc_fence_after();
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * Cfg::BLOCK + (k % 4) * 32;
          mma_ss(tmem + Cfg::COL_DP, sdesc_sw128(vb + off, 16, 1024),
                 sdesc_sw128(dob + off, 16, 1024), ID_S, k > 0);
        }
        mma_commit(s_full);
        if (!mbar_wait(p_ready, it & 1, err, abort_flag)) break;
        tc_fence_after();
        // dQ = dS K  (k over keys; A = dS from dS^T in smem, MN-major)
#pragma unroll
        for (int k = 0; k < BT / 16; ++k)
          mma_ss(tmem + Cfg::COL_DP, sdesc_sw128(dsb + k * 2048, Cfg::BLOCK, 1024),
                 sdesc_sw128(kb + k * 2048, Cfg::BLOCK, 1024), ID_DQ, k > 0);
        mma_commit(dq_full);
        // dV += P^T dO ; dK += dS^T Q  (k over queries; A in TMEM)
#pragma unroll
        for (int k = 0; k < BT / 16; ++k) {
          const uint32_t acc = (it > 0 || k > 0) ? 1u : 0u;
          mma_ts(tmem + Cfg::COL_DV, tmem + Cfg::COL_S + k * 8,
                 sdesc_sw128(dob + k * 2048, Cfg::BLOCK, 1024), ID_ACC, acc);
          mma_ts(tmem + Cfg::COL_DK, tmem + Cfg::COL_S + 64 + k * 8,
                 sdesc_sw128(qb + k * 2048, Cfg::BLOCK, 1024), ID_ACC, acc);
        }
        mma_commit(&q_empty[st]);
      }
      mma_commit(mma_done);
    }
  } else {
    // ------------------------------------- softmax gradient + epilogue warps
    const int r = warp * 32 + lane;  // key row within the tile (TMEM lane)
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float sl2 = a.scale * 1.4426950408889634f;
    const float* lse_g = a.lse + (long long)head * a.lse_stride;
    const float* D_g = a.D + (long long)head * S;
    uint8_t* ds_row = smem + Cfg::DS_OFF + r * 128;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int q0 = (jt + it) * BT;
      // lse (log2 units) and D of this tile's 128 queries: lane l holds
      // queries l + 32m; a column's value is broadcast with a shuffle whose
      // source lane and register are compile-time constants
      float lse_r[4], dd_r[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int q = q0 + 32 * m + lane;
        lse_r[m] = q < S ? lse_g[q] * 1.4426950408889634f : INFINITY;
        dd_r[m] = q < S ? D_g[q] : 0.f;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(s_full, it & 1, err, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const bool diag = (it == 0);
      float p[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_off + Cfg::COL_S + 32 * c, rr);
        tmem_ld_wait(rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int q = 32 * c + i;
          const float lq = __shfl_sync(0xffffffffu, lse_r[c], i);
          float v = ex2(fmaf(__uint_as_float(rr[i]), sl2, -lq));
          if (diag && r > q) v = 0.f;
          p[q] = v;
        }
      }
      // P^T (bf16) over the first half of S^T
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = pack_bf16(p[64 * h + 2 * i], p[64 * h + 2 * i + 1]);
        tmem_st32(tmem + lane_off + Cfg::COL_S + 32 * h, pk);
      }
      // dS^T = P^T (dP^T - D): TMEM (second half of S^T) and shared memory
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_off + Cfg::COL_DP + 64 * h + 32 * c, rr);
          tmem_ld_wait(rr);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int q = 64 * h + 32 * c + 2 * i;
            const float D0 = __shfl_sync(0xffffffffu, dd_r[q >> 5], q & 31);
            const float D1 = __shfl_sync(0xffffffffu, dd_r[(q + 1) >> 5], (q + 1) & 31);
            const float d0 = p[q] * (__uint_as_float(rr[2 * i]) - D0);
            const float d1 = p[q + 1] * (__uint_as_float(rr[2 * i + 1]) - D1);
            pk[16 * c + i] = pack_bf16(d0, d1);
          }
        }
        tmem_st32(tmem + lane_off + Cfg::COL_S + 64 + 32 * h, pk);
        uint8_t* blk = ds_row + h * Cfg::BLOCK;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          *reinterpret_cast<uint4*>(blk + ((ch ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready);
      // dQ rows (query q0 + r): read out, free the region, reduce to global
      ok = __all_sync(0xffffffffu, mbar_wait(dq_full, it & 1, err, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float dq[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_off + Cfg::COL_DP + 32 * c, rr);
        tmem_ld_wait(rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) dq[32 * c + i] = __uint_as_float(rr[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
      if (q0 + r < S) {
        float* dst = a.dQ + (long long)(q0 + r) * a.ld_dq + head * D;
#pragma unroll
        for (int i = 0; i < D; i += 4)
          red_add_v4_f32(dst + i, dq[i] * a.scale, dq[i + 1] * a.scale, dq[i + 2] * a.scale,
                         dq[i + 3] * a.scale);
      }
    }
    // final dK, dV of this CTA's keys
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(mma_done, 0, err, abort_flag));
    if (ok) {
      tc_fence_after();
      const int key = k0 + r;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rv[32], rk[32];
        tmem_ld32(tmem + lane_off + Cfg::COL_DV + 32 * c, rv);
        tmem_ld_wait(rv);
        tmem_ld32(tmem + lane_off + Cfg::COL_DK + 32 * c, rk);
        tmem_ld_wait(rk);
        if (key < S) {
          const long long off = (long long)key * a.ld_dkv + kvh * D + 32 * c;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            red_add_v4_f32(a.dV + off + i, __uint_as_float(rv[i]), __uint_as_float(rv[i + 1]),
                           __uint_as_float(rv[i + 2]), __uint_as_float(rv[i + 3]));
            red_add_v4_f32(a.dK + off + i, __uint_as_float(rk[i]) * a.scale,
                           __uint_as_float(rk[i + 1]) * a.scale,
                           __uint_as_float(rk[i + 2]) * a.scale,
                           __uint_as_float(rk[i + 3]) * a.scale);
          }
        }
      }
    }
  }

  // --------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    if (*abort_flag) {
      if (lane == 0) {
        mma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0);
      }
      __syncwarp();
    }
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
static cudaError_t launch_bwd_t(const AttnBwdArgs& a, int* err, cudaStream_t stream) {
  using Cfg = BwdCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap qm, km, vm, dm;
  if (!make_tmap_bf16(&qm, a.Q, a.S, (uint64_t)a.heads * D, a.ldq, BT, 64) ||
      !make_tmap_bf16(&km, a.K, a.S, (uint64_t)a.ldkv, a.ldkv, BT, 64) ||
      !make_tmap_bf16(&vm, a.V, a.S, (uint64_t)a.ldkv, a.ldkv, BT, 64) ||
      !make_tmap_bf16(&dm, a.dO, a.S, (uint64_t)a.heads * D, a.ld_do, BT, 64))
    return cudaErrorInvalidValue;
  dim3 grid((a.S + BT - 1) / BT, a.heads);
  attn_bwd_kernel<D><<<grid, kThreads, Cfg::SMEM_BYTES, stream>>>(qm, km, vm, dm, a, err);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const AttnBwdArgs& a, int* err, cudaStream_t stream) {
  if (a.S <= 0 || a.heads <= 0) return cudaSuccess;
  if (a.d == 128) return launch_bwd_t<128>(a, err, stream);
  if (a.d == 64) return launch_bwd_t<64>(a, err, stream);
  return cudaErrorNotSupported;
}

}  // namespace upipe
