// Causal online-softmax attention forward on tcgen05 (one head chunk).
//
// This is the per-head attention that every chunk of the head-chunked loop
// runs over the whole sequence: for query row i,
//   s_ij = q_i . k_j / sqrt(d)  (j <= i),
//   lse_i = log sum_j exp(s_ij),   o_i = sum_j exp(s_ij - lse_i) v_j.
// (Untied Ulysses, memeeeeeex.com "Untied Ulysses (UPipe)": per chunk the
// heads' attention is computed, then the partial result is stored; the
// attention itself is FlashAttention-style over the full sequence per head,
// "DeepSpeed Ulysses" section.)
//
// One CTA = 256 query rows (two 128-row tiles t = 0, 1) of one head.  The two
// tiles ping-pong on the tensor core: while the softmax warps of one tile turn
// S into P, the tensor core runs the other tile's PV and next QK^T.
//   warps 0-3   softmax + epilogue of tile 0 (TMEM lanes 0..127, one row each)
//   warps 4-7   softmax + epilogue of tile 1
//   warp 8      TMEM owner and tcgen05.mma issuer
//   warp 9      TMA producer (Q once, then K_j, V_j through a 4-slot ring)
//   warps 10-11 idle (they complete warpgroup 2 for register reallocation)
// setmaxnreg gives the softmax warpgroups 216 registers a thread and
// warpgroup 2 72: 2 x 128 x 216 + 128 x 72 = 64512 = 384 threads x 168, the
// registers the block is launched with.
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1.  P_t (fp16) is written over the
// first half of S_t and fed to the PV MMA straight from TMEM.
// Operands: Q, K, V arrive in fp16 and P is stored in fp16 (11 significant
// bits; bf16 has 8), so QK^T and PV both run as fp16 MMAs with fp32
// accumulation.  P carries a fixed factor 2^kPShift: a probability p relative
// to the row max is stored as p * 2^8, so every p >= 2^-22 is a normal fp16
// number (long rows hold millions of small p; without the shift those below
// 2^-14 would lose precision or flush to zero).  l and O carry the same factor,
// which cancels in O / l and is taken out of the LSE.
// Softmax runs in base 2 with the row max taken only on demand: P is computed
// with the running max m, and while m is the row's max every p <= 1, so the
// tile's row sum is at most 128.  Only a sum above 128 (or inf / NaN on a
// row's first tile, where m = -inf) makes the thread take the tile's max,
// rescale O and l to it and recompute P.  Growth that keeps the sum within
// 128 keeps m (p <= 128, so p * 2^8 <= 2^15 stays inside fp16's range), so
// almost every step skips both the max and the O read-modify-write.
// The diagonal KV tile of each query tile is the only one masked; KV tiles
// beyond it are never loaded (causal skipping).
// Grid: heaviest query blocks first, all heads of a block together.
// Long rows: the tensor core's fp32 accumulation of O drifts over hundreds of
// thousands of MMA steps (measured: the error grows linearly with position
// past ~1M keys), so every kFlushTiles KV tiles each softmax thread folds its
// O row out of TMEM into an fp32 row in global memory (IEEE adds, rescaled to
// the current row max) and the next PV MMA restarts the TMEM accumulator.  The
// rows live in a per-SM slot (one CTA per SM), so the scratch is bounded.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {

namespace {

constexpr int kThreads = 384;
constexpr int kSlots = 4;

__device__ __forceinline__ uint32_t sm_id() {
  uint32_t v;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
  return v;
}
constexpr float kPShift = 8.0f;       // P is stored as p * 2^kPShift (see above)
// shifted row sum of one tile's p that asks for a new max (128 * 2^kPShift)
constexpr float kSumLimit = 128.0f * 256.0f;

template <int D>
struct FwdCfg {
  static constexpr uint32_t TILE_BYTES = 128 * D * 2;     // one Q, K or V tile
  static constexpr uint32_t BLOCK_BYTES = 128 * 64 * 2;   // one 64-column swizzled block
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t SLOT_OFF = 2 * TILE_BYTES;
  static constexpr uint32_t BAR_OFF = SLOT_OFF + kSlots * TILE_BYTES;
  static constexpr uint32_t SMEM_BYTES = BAR_OFF + 256 + 1024;
  static constexpr uint32_t O_COL = 256;  // O_t at TMEM column O_COL + t * D
};

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const AttnFwdArgs a,
                    int* __restrict__ err) {
  using Cfg = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
  uint64_t* q_full = bars + 0;
  uint64_t* slot_full = bars + 1;             // [kSlots]
  uint64_t* slot_empty = bars + 1 + kSlots;   // [kSlots]
  uint64_t* s_full = bars + 1 + 2 * kSlots;   // [2]
  uint64_t* p_full = s_full + 2;              // [2]
  uint64_t* o_done = p_full + 2;              // [2]
  uint64_t* drain_bar = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int nqb = (a.S + 255) / 256;
  const int qb = nqb - 1 - (int)(blockIdx.x / a.heads);
  const int head = (int)(blockIdx.x % a.heads);
  const int kvh = (a.h0 + head) / a.group - a.kv0;
  const int q0 = qb * 256;
  const int n_kv = 2 * qb + 2;  // KV tiles of query tile 1; tile 0 has n_kv - 1
  // folding of long rows (see above): only when the scratch exists, the rows
  // are long enough, and this SM id has a slot
  const bool folding = a.flush != nullptr && n_kv > kFlushTiles && sm_id() < (uint32_t)kFlushSlots;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&slot_full[s], 1);
      mbar_init(&slot_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
      mbar_init(&o_done[t], 1);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9 && lane == 0) {
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
  setmaxnreg_dec<72>();
  if (warp == 9) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t issued = 0, issued_phase = 0;
      mbar_expect_tx(q_full, 2 * Cfg::TILE_BYTES);
      for (int t = 0; t < 2; ++t)
        for (int b = 0; b < D / 64; ++b)
          tma_load_2d(smem + Cfg::Q_OFF + t * Cfg::TILE_BYTES + b * Cfg::BLOCK_BYTES, &qmap,
                      q_full, head * D + 64 * b, q0 + 128 * t);
      for (int idx = 0; idx < 2 * n_kv; ++idx) {
        const int slot = idx % kSlots;
        const uint32_t ph = (idx / kSlots) & 1;
        if (!mbar_wait(&slot_empty[slot], ph ^ 1, err, abort_flag)) break;
        mbar_expect_tx(&slot_full[slot], Cfg::TILE_BYTES);
        const CUtensorMap* map = (idx & 1) ? &vmap : &kmap;
        uint8_t* dst = smem + Cfg::SLOT_OFF + slot * Cfg::TILE_BYTES;
        for (int b = 0; b < D / 64; ++b)
          tma_load_2d(dst + b * Cfg::BLOCK_BYTES, map, &slot_full[slot], kvh * D + 64 * b,
                      128 * (idx >> 1));
        issued |= 1u << slot;
        issued_phase = (issued_phase & ~(1u << slot)) | (ph << slot);
      }
      if (*abort_flag) {
        mbar_wait_drain(q_full, 0);
        for (int s = 0; s < kSlots; ++s)
          if (issued & (1u << s)) mbar_wait_drain(&slot_full[s], (issued_phase >> s) & 1u);
      }
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------- MMA issue
    {  // whole warp; one elected lane issues
      constexpr uint32_t IDESC_S = idesc_f16(128, 128, false, false);
      constexpr uint32_t IDESC_O = idesc_f16(128, D, false, true);
      const uint32_t q_base = smem_u32(smem + Cfg::Q_OFF);
      const uint32_t slot_base = smem_u32(smem + Cfg::SLOT_OFF);
      uint32_t p_phase[2] = {0, 0};
      const int n0 = n_kv - 1;
      bool ok = mbar_wait_warp(q_full, 0, err, abort_flag);
      for (int j = 0; j <= n_kv && ok; ++j) {
        const int kidx = 2 * j;
        const int vidx = 2 * j - 1;  // V_{j-1}
        const uint32_t k_addr = slot_base + (kidx % kSlots) * Cfg::TILE_BYTES;
        const int vslot = j >= 1 ? vidx % kSlots : 0;
        const uint32_t v_addr = slot_base + vslot * Cfg::TILE_BYTES;
        if (j < n_kv) {
          if (!mbar_wait_warp(&slot_full[kidx % kSlots], (kidx / kSlots) & 1, err, abort_flag)) break;
        }
        if (j >= 1) {
          if (!mbar_wait_warp(&slot_full[vslot], (vidx / kSlots) & 1, err, abort_flag)) break;
        }
        tc_fence_after();
        for (int t = 0; t < 2 && ok; ++t) {
          const int nt = t == 0 ? n0 : n_kv;
          // O_t += P_t(j-1) V_{j-1}
          if (j >= 1 && j - 1 < nt) {
            if (!mbar_wait_warp(&p_full[t], p_phase[t], err, abort_flag)) { ok = false; break; }
            p_phase[t] ^= 1;
            tc_fence_after();
            const uint32_t o_tmem = tmem + Cfg::O_COL + t * D;
            const uint32_t p_tmem = tmem + 128 * t;
            const uint32_t acc0 =
                ((j - 1 == 0) || (folding && (j - 1) % kFlushTiles == 0)) ? 0u : 1u;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t bd = sdesc_sw128(v_addr + k * 2048, Cfg::BLOCK_BYTES, 1024);
              mma_ts_w(o_tmem, p_tmem + k * 8, bd, IDESC_O, k > 0 ? 1u : acc0);
            }
            if (t == 1) mma_commit_w(&slot_empty[vslot]);
            if (j - 1 == nt - 1) mma_commit_w(&o_done[t]);
          }
          // S_t = Q_t K_j^T
          if (j < nt) {
            const uint32_t s_tmem = tmem + 128 * t;
            const uint32_t qa = q_base + t * Cfg::TILE_BYTES;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t off = (k / 4) * Cfg::BLOCK_BYTES + (k % 4) * 32;
              const uint64_t ad = sdesc_sw128(qa + off, 16, 1024);
              const uint64_t bd = sdesc_sw128(k_addr + off, 16, 1024);
              mma_ss_w(s_tmem, ad, bd, IDESC_S, k > 0 ? 1u : 0u);
            }
            mma_commit_w(&s_full[t]);
            if (t == 1) mma_commit_w(&slot_empty[kidx % kSlots]);
          }
        }
      }
    }
  }
  } else {
    // --------------------------------------------------- softmax (tile t)
    setmaxnreg_inc<216>();
    const int t = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qpos = q0 + 128 * t + r;
    const int nt = (t == 0) ? n_kv - 1 : n_kv;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + 128 * t + lane_off;
    const uint32_t o_tmem = tmem + Cfg::O_COL + t * D + lane_off;
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY;
    float l_run = 0.f;
    float m_acc = -INFINITY;  // row max of the folded part of O (-inf: nothing folded)
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      // warp-uniform: the tcgen05.ld/st below are warp-collective
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], j & 1, err, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float s[128];
      {
        uint32_t rr[128];
        tmem_ld128(s_tmem, rr);
        tmem_ld_wait(rr);
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(rr[i]);
      }
      if (j == nt - 1) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > r) s[c] = -INFINITY;
      }
      // p = 2^(s * scale_log2 - m_run + kPShift) with the running max: pairs
      // through one packed FMA each, the row sum in four packed partial sums
      // (depth 16).  Writes P (fp16) over S in TMEM and returns the row sum.
      const float2 sc2 = make_float2(sl2, sl2);
      auto p_tile = [&](float m) -> float {
        const float2 nm2 = make_float2(kPShift - m, kPShift - m);
        float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float2 x = ffma2(make_float2(s[64 * h + 2 * i], s[64 * h + 2 * i + 1]), sc2, nm2);
            x.x = ex2(x.x);
            x.y = ex2(x.y);
            ps[i & 3] = fadd2(ps[i & 3], x);
            pk[i] = pack_f16(x.x, x.y);
          }
          tmem_st32(s_tmem + 32 * h, pk);
        }
        const float2 s01 = fadd2(ps[0], ps[1]);
        const float2 s23 = fadd2(ps[2], ps[3]);
        return (s01.x + s23.x) + (s01.y + s23.y);
      };
      float l_tile = p_tile(m_run);
      // Every p <= 1 while m_run is the row's max, so a row sum above
      // kSumLimit (or inf / NaN: the first tile, m_run = -inf) means the
      // max has grown.  Only then is the row max taken; O and l are rescaled
      // to it and P is recomputed.  A smaller growth keeps m_run: its shifted
      // p stay below kSumLimit = 2^15, inside the range of fp16 P.
      const bool grow = !(l_tile <= kSumLimit);
      if (__any_sync(0xffffffffu, grow)) {
        float m_new = m_run;
        if (grow) {
          // four independent three-input chains (depth 16, not 127)
          float mq[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) mq[k] = fmaxf(s[2 * k], s[2 * k + 1]);
#pragma unroll
          for (int c = 8; c < 128; c += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k) mq[k] = fmax3(mq[k], s[c + 2 * k], s[c + 2 * k + 1]);
          const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
          m_new = fmaxf(m_run, mx * sl2);
        }
        if (j > 0) {
          const float alpha = grow ? ex2(m_run - m_new) : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(o_tmem + 32 * c, rr);
            tmem_ld_wait(rr);
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
            tmem_st32(o_tmem + 32 * c, rr);
          }
        }
        if (grow) {
          l_run *= ex2(m_run - m_new);
          m_run = m_new;
        }
        tmem_st_wait();   // the first P's stores land before they are rewritten
        l_tile = p_tile(m_run);
      }
      l_run += l_tile;
      if (folding && j > 0 && j % kFlushTiles == 0) {
        // O in TMEM holds PV(0 .. j-1) since the last fold, in units of m_run
        const bool have_acc = m_acc != -INFINITY;
        const float keep = have_acc ? ex2(m_acc - m_run) : 0.f;
        float* acc_row = a.flush + ((size_t)sm_id() * 256 + 128 * t + r) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(o_tmem + 32 * c, rr);
          tmem_ld_wait(rr);
          float* ap = acc_row + 32 * c;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float4 v = make_float4(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1]),
                                   __uint_as_float(rr[i + 2]), __uint_as_float(rr[i + 3]));
            if (have_acc) {
              const float4 o = *reinterpret_cast<const float4*>(ap + i);
              v.x = fmaf(o.x, keep, v.x); v.y = fmaf(o.y, keep, v.y);
              v.z = fmaf(o.z, keep, v.z); v.w = fmaf(o.w, keep, v.w);
            }
            *reinterpret_cast<float4*>(ap + i) = v;
          }
        }
        m_acc = m_run;
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    // ------------------------------------------------------------ epilogue
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_done[t], 0, err, abort_flag));
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      const bool live = qpos < a.S;
      const bool have_acc = m_acc != -INFINITY;
      const float keep = have_acc ? ex2(m_acc - m_run) : 0.f;
      const float* acc_row =
          have_acc ? a.flush + ((size_t)sm_id() * 256 + 128 * t + r) * D : nullptr;
      bf16* op = a.O + (long long)qpos * a.ldo + head * D;
      const __half* dop = a.dO ? a.dO + (long long)qpos * a.ld_do + head * D : nullptr;
      float dot = 0.f;  // D' = dO' . o over the fp32 o (the backward's recompute)
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(o_tmem + 32 * c, rr);
        tmem_ld_wait(rr);
        if (have_acc) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            rr[i] = __float_as_uint(fmaf(acc_row[32 * c + i], keep, __uint_as_float(rr[i])));
        }
        if (live && dop) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            const uint4 dv = *reinterpret_cast<const uint4*>(dop + 32 * c + i);
            const uint32_t* dw = &dv.x;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 g = unpack_f16(dw[j]);
              dot = fmaf(g.x, __uint_as_float(rr[i + 2 * j]) * inv_l, dot);
              dot = fmaf(g.y, __uint_as_float(rr[i + 2 * j + 1]) * inv_l, dot);
            }
          }
        }
        if (live) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(rr[i + 0]) * inv_l, __uint_as_float(rr[i + 1]) * inv_l);
            w.y = pack_bf16(__uint_as_float(rr[i + 2]) * inv_l, __uint_as_float(rr[i + 3]) * inv_l);
            w.z = pack_bf16(__uint_as_float(rr[i + 4]) * inv_l, __uint_as_float(rr[i + 5]) * inv_l);
            w.w = pack_bf16(__uint_as_float(rr[i + 6]) * inv_l, __uint_as_float(rr[i + 7]) * inv_l);
            *reinterpret_cast<uint4*>(op + 32 * c + i) = w;
          }
        }
      }
      if (live && a.lse)
        a.lse[(long long)head * a.lse_stride + qpos] =
            (m_run - kPShift + __log2f(l_run)) * 0.69314718055994531f;
      if (live && dop) a.D[(long long)head * a.S + qpos] = dot;
    }
  }

  // --------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
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
static cudaError_t launch_fwd_t(const CUtensorMap& qmap, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, const AttnFwdArgs& a, int* err,
                                cudaStream_t stream) {
  using Cfg = FwdCfg<D>;
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t ea = smem_attr_once(attn_fwd_kernel<D>, (int)Cfg::SMEM_BYTES, attr_done);
  if (ea != cudaSuccess) return ea;
  const long long nqb = (a.S + 255) / 256;
  const long long grid = nqb * a.heads;
  attn_fwd_kernel<D><<<(unsigned)grid, kThreads, Cfg::SMEM_BYTES, stream>>>(qmap, kmap, vmap, a,
                                                                           err);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const CUtensorMap& qmap, const CUtensorMap& kmap,
                            const CUtensorMap& vmap, const AttnFwdArgs& a, int d, int* err,
                            cudaStream_t stream) {
  if (a.S <= 0 || a.heads <= 0) return cudaSuccess;
  if (d == 128) return launch_fwd_t<128>(qmap, kmap, vmap, a, err, stream);
  if (d == 64) return launch_fwd_t<64>(qmap, kmap, vmap, a, err, stream);
  return cudaErrorNotSupported;
}

}  // namespace upipe
