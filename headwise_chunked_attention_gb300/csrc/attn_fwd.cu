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
// Known LSE (the backward's recompute): with the forward's LSE of each row the
// kernel takes p = 2^(s * scale_log2 - lse_2 + kPShift) directly, p <= 2^8, so
// it skips the row sum and the max test and O needs no division by l.
// Long rows: the tensor core's fp32 accumulation of O drifts over hundreds of
// thousands of MMA steps (measured: the error grows linearly with position
// past ~1M keys), so every kFlushTiles KV tiles each softmax thread folds its
// O row out of TMEM into an fp32 row in global memory (IEEE adds, rescaled to
// the current row max) and the next PV MMA restarts the TMEM accumulator.  The
// rows live in a per-SM slot (one CTA per SM), so the scratch is bounded.
//
// Fused Wo-slice accumulate (FUSE): instead of storing o, the CTA adds its
// rows' partial result out[rows] += o_h Wo[:, h*d:(h+1)*d]^T itself (each
// chunk keeps its heads' contribution to the layer output, memeeeeeex.com
// "Untied Ulysses (UPipe)", here without an attention-output buffer).  After the attention loop the softmax warps write o
// (bf16) over their Q tile in shared memory, the K/V ring is reused for two
// 128-row tiles of the head's Wo slice and for fp32 staging, and for each
// 128-column block n of out the MMA warp computes the two 128 x 128 products
// into TMEM (double-buffered: S_t for even n, O_t's columns for odd n) while
// the softmax warps stage the previous block and add it into out with TMA
// reduce-adds (the read-modify-write runs in L2).
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

constexpr int kStgBufs = 2;                    // fp32 staging buffers per softmax warp (FUSE)
constexpr uint32_t kStgBytes = 32 * 32 * 4;    // [32 rows][32 cols] fp32, 128-byte swizzled

// Kernel modes: o stored to a.O (the forward, and the backward's recompute
// without a known LSE); the fused Wo-slice accumulate; the backward's
// recompute with the forward's LSE given.
constexpr int kModeStore = 0;
constexpr int kModeFused = 1;
constexpr int kModeKnownLse = 2;

template <int D, bool FUSE>
struct FwdCfg {
  static constexpr uint32_t TILE_BYTES = 128 * D * 2;     // one Q, K or V tile
  static constexpr uint32_t BLOCK_BYTES = 128 * 64 * 2;   // one 64-column swizzled block
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t SLOT_OFF = 2 * TILE_BYTES;
  static constexpr uint32_t RING_END = SLOT_OFF + kSlots * TILE_BYTES;
  // FUSE, after the attention loop: two Wo tiles [128 outputs][D] over the
  // first two ring slots, then the softmax warps' staging buffers
  static constexpr uint32_t WO_OFF = SLOT_OFF;
  static constexpr uint32_t STG_OFF = SLOT_OFF + 2 * TILE_BYTES;
  static constexpr uint32_t STG_END = STG_OFF + 8 * kStgBufs * kStgBytes;
  static constexpr uint32_t BAR_OFF = (FUSE && STG_END > RING_END) ? STG_END : RING_END;
  static constexpr uint32_t SMEM_BYTES = BAR_OFF + 256 + 1024;
  static constexpr uint32_t O_COL = 256;  // O_t at TMEM column O_COL + t * D
  static_assert(WO_OFF % 1024 == 0 && STG_OFF % 1024 == 0, "swizzled tiles need 1 KB alignment");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per block");
};

}  // namespace

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap,
                    const __grid_constant__ CUtensorMap womap,
                    const __grid_constant__ CUtensorMap outmap, const AttnFwdArgs a,
                    int* __restrict__ err) {
  constexpr bool FUSE = MODE == kModeFused;
  constexpr bool KNOWN = MODE == kModeKnownLse;
  using Cfg = FwdCfg<D, FUSE>;
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
  // FUSE: o of both tiles in shared memory (8 softmax warps); Wo tiles
  // loaded / consumed; product block in TMEM / read out (8 softmax warps)
  uint64_t* o_stored = drain_bar + 1;
  uint64_t* wo_full = o_stored + 1;           // [2]
  uint64_t* wo_empty = wo_full + 2;           // [2]
  uint64_t* acc_full = wo_empty + 2;          // [2]
  uint64_t* acc_empty = acc_full + 2;         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
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
    mbar_init(o_stored, 8);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&wo_full[b], 1);
      mbar_init(&wo_empty[b], 1);
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9 && lane == 0) {
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    if constexpr (FUSE) {
      prefetch_tmap(&womap);
      prefetch_tmap(&outmap);
    }
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
      uint32_t wo_issued = 0, wo_phase = 0;
      if constexpr (FUSE) {
        // the ring is free once both tiles' o is in shared memory (that
        // follows the last PV MMA, which read the last V tile)
        if (!*abort_flag && mbar_wait(o_stored, 0, err, abort_flag)) {
          const int wcol = (a.h0 + head) * D;
          for (int n = 0; n < a.wo_tiles; ++n) {
            const int b = n & 1;
            const uint32_t ph = (n >> 1) & 1;
            if (!mbar_wait(&wo_empty[b], ph ^ 1, err, abort_flag)) break;
            mbar_expect_tx(&wo_full[b], Cfg::TILE_BYTES);
            uint8_t* dst = smem + Cfg::WO_OFF + b * Cfg::TILE_BYTES;
            for (int k = 0; k < D / 64; ++k)
              tma_load_2d(dst + k * Cfg::BLOCK_BYTES, &womap, &wo_full[b], wcol + 64 * k, 128 * n);
            wo_issued |= 1u << b;
            wo_phase = (wo_phase & ~(1u << b)) | (ph << b);
          }
        }
      }
      if (*abort_flag) {
        mbar_wait_drain(q_full, 0);
        for (int s = 0; s < kSlots; ++s)
          if (issued & (1u << s)) mbar_wait_drain(&slot_full[s], (issued_phase >> s) & 1u);
        for (int b = 0; b < 2; ++b)
          if (wo_issued & (1u << b)) mbar_wait_drain(&wo_full[b], (wo_phase >> b) & 1u);
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
      if constexpr (FUSE) {
        // out block n = o_t Wo_h[128 n : 128 n + 128, :]^T for both tiles,
        // into S_t (n even) or the columns of O_t (n odd)
        constexpr uint32_t IDESC_W = idesc_bf16(128, 128, false, false);
        const uint32_t wo_base = smem_u32(smem + Cfg::WO_OFF);
        if (ok && !*abort_flag) ok = mbar_wait_warp(o_stored, 0, err, abort_flag);
        for (int n = 0; n < a.wo_tiles && ok; ++n) {
          const int b = n & 1;
          if (!mbar_wait_warp(&wo_full[b], (n >> 1) & 1, err, abort_flag)) break;
          if (n >= 2 && !mbar_wait_warp(&acc_empty[b], ((n >> 1) - 1) & 1, err, abort_flag)) break;
          tc_fence_after();
          const uint32_t w_addr = wo_base + b * Cfg::TILE_BYTES;
          for (int t = 0; t < 2; ++t) {
            const uint32_t acc = tmem + (b ? Cfg::O_COL : 0u) + 128 * t;
            const uint32_t oa = q_base + t * Cfg::TILE_BYTES;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t off = (k / 4) * Cfg::BLOCK_BYTES + (k % 4) * 32;
              mma_ss_w(acc, sdesc_sw128(oa + off, 16, 1024), sdesc_sw128(w_addr + off, 16, 1024),
                       IDESC_W, k > 0 ? 1u : 0u);
            }
          }
          mma_commit_w(&wo_empty[b]);
          mma_commit_w(&acc_full[b]);
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
    if constexpr (KNOWN) {
      // the row's max is replaced by its log-sum-exp (base 2, scaled): every
      // p is then final, p * 2^kPShift <= 2^kPShift, and no tile changes it
      // (rows past S take 0: their values are never stored)
      const long long li = (long long)head * a.lse_stride + qpos;
      m_run = (qpos < a.S && dbg_in(li, li, (long long)a.heads * a.lse_stride, err))
                  ? a.lse_in[li] * 1.4426950408889634f
                  : 0.f;
    }
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
      if constexpr (!KNOWN) {
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
      }
      if (folding && j > 0 && j % kFlushTiles == 0) {
        // O in TMEM holds PV(0 .. j-1) since the last fold, in units of m_run
        const bool have_acc = m_acc != -INFINITY;
        const float keep = have_acc ? ex2(m_acc - m_run) : 0.f;
        const long long row_off = ((long long)sm_id() * 256 + 128 * t + r) * D;
        const bool row_ok = dbg_in(row_off, row_off + D - 1, (long long)kFlushSlots * 256 * D, err);
        float* acc_row = a.flush + row_off;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(o_tmem + 32 * c, rr);
          tmem_ld_wait(rr);
          if (!row_ok) continue;
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
      // with the known LSE, sum_j p_j = 1: O carries just the 2^kPShift factor
      const float inv_l = KNOWN ? 1.f / (float)(1 << (int)kPShift) : 1.f / l_run;
      const bool live = qpos < a.S;
      const long long row_off = ((long long)sm_id() * 256 + 128 * t + r) * D;
      const bool have_acc = m_acc != -INFINITY &&
          dbg_in(row_off, row_off + D - 1, (long long)kFlushSlots * 256 * D, err);
      const float keep = have_acc ? ex2(m_acc - m_run) : 0.f;
      const float* acc_row = have_acc ? a.flush + row_off : nullptr;
      // o and dO' rows of this head: columns [head * D, head * D + D) of
      // [S, ldo] and [S, ld_do]
      const long long o_off = (long long)qpos * a.ldo + head * D;
      const long long do_off = (long long)qpos * a.ld_do + head * D;
      const bool o_ok = FUSE || !live || dbg_in2(qpos, a.S, head * D, head * D + D - 1, a.ldo, err);
      const bool do_ok = !a.dO || !live ||
          dbg_in2(qpos, a.S, head * D, head * D + D - 1, a.ld_do, err);
      bf16* op = FUSE ? nullptr : a.O + o_off;
      const __half* dop = (a.dO && do_ok) ? a.dO + do_off : nullptr;
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
        if (FUSE || (live && o_ok)) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(rr[i + 0]) * inv_l, __uint_as_float(rr[i + 1]) * inv_l);
            w.y = pack_bf16(__uint_as_float(rr[i + 2]) * inv_l, __uint_as_float(rr[i + 3]) * inv_l);
            w.z = pack_bf16(__uint_as_float(rr[i + 4]) * inv_l, __uint_as_float(rr[i + 5]) * inv_l);
            w.w = pack_bf16(__uint_as_float(rr[i + 6]) * inv_l, __uint_as_float(rr[i + 7]) * inv_l);
            if constexpr (FUSE) {
              // row r of the tile's K-major, 128-byte swizzled A operand (the
              // layout TMA gave Q): 16-byte chunk q of a 64-column block at
              // (q ^ (r & 7))
              const int col = 32 * c + i;
              const int q = (col & 63) >> 3;
              *reinterpret_cast<uint4*>(smem + Cfg::Q_OFF + t * Cfg::TILE_BYTES +
                                        (col >> 6) * Cfg::BLOCK_BYTES + r * 128 +
                                        ((q ^ (r & 7)) << 4)) = w;
            } else {
              *reinterpret_cast<uint4*>(op + 32 * c + i) = w;
            }
          }
        }
      }
      const long long l_off = (long long)head * a.lse_stride + qpos;
      if (live && a.lse && dbg_in(l_off, l_off, (long long)a.heads * a.lse_stride, err))
        a.lse[l_off] = (m_run - kPShift + __log2f(l_run)) * 0.69314718055994531f;
      const long long d_off = (long long)head * a.S + qpos;
      if (live && dop && dbg_in(d_off, d_off, (long long)a.heads * a.S, err)) a.D[d_off] = dot;
    }
    if constexpr (FUSE) {
      // o is in shared memory (for the async proxy) and every TMEM read of
      // O_t is done: hand both to the MMA warp
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(o_stored);
      // the staging buffers lie over the ring, which the other tile's last
      // PV MMA may still read until its O is done
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_done[1 - t], 0, err, abort_flag));
      uint8_t* stg = smem + Cfg::STG_OFF + warp * kStgBufs * kStgBytes;
      const int row0 = q0 + 128 * t + 32 * quarter;
      const bool rows_live = row0 < a.S;   // rows past S: the TMA reduce drops them
      uint32_t round = 0;
#pragma unroll 1
      for (int n = 0; n < a.wo_tiles && ok; ++n) {
        const int b = n & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[b], (n >> 1) & 1, err, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint32_t acc = tmem + (b ? Cfg::O_COL : 0u) + 128 * t + lane_off;
#pragma unroll 1
        for (int c = 0; c < 4; ++c, ++round) {
          // two 16-column loads: a 32-column load here made ptxas spill in
          // the softmax loop
          uint32_t lo[16], hi[16];
          tmem_ld16(acc + 32 * c, lo);
          tmem_ld16(acc + 32 * c + 16, hi);
          tmem_ld_wait(lo);
          tmem_ld_wait(hi);
          if (c == 3) {  // the block is read out: the MMA warp may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
          }
          if (rows_live) {
            uint8_t* buf = stg + (round % kStgBufs) * kStgBytes;
            if (lane == 0) bulk_wait_read<kStgBufs - 1>();   // buf's previous reduce has read it
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t* v = k < 4 ? lo + 4 * k : hi + 4 * (k - 4);
              *reinterpret_cast<uint4*>(buf + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                  make_uint4(v[0], v[1], v[2], v[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d(&outmap, buf, 128 * n + 32 * c, row0);
              bulk_commit();
            }
          }
        }
      }
      if (lane == 0) bulk_wait_all();
      __syncwarp();
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

template <int D, int MODE>
static cudaError_t launch_fwd_t(const CUtensorMap& qmap, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, const CUtensorMap& womap,
                                const CUtensorMap& outmap, const AttnFwdArgs& a, int* err,
                                cudaStream_t stream) {
  using Cfg = FwdCfg<D, MODE == kModeFused>;
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t ea =
      smem_attr_once(attn_fwd_kernel<D, MODE>, (int)Cfg::SMEM_BYTES, attr_done);
  if (ea != cudaSuccess) return ea;
  const long long nqb = (a.S + 255) / 256;
  const long long grid = nqb * a.heads;
  attn_fwd_kernel<D, MODE><<<(unsigned)grid, kThreads, Cfg::SMEM_BYTES, stream>>>(
      qmap, kmap, vmap, womap, outmap, a, err);
  return cudaGetLastError();
}

template <int MODE>
static cudaError_t launch_fwd_d(int d, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, const CUtensorMap& womap,
                                const CUtensorMap& outmap, const AttnFwdArgs& a, int* err,
                                cudaStream_t stream) {
  if (d == 128) return launch_fwd_t<128, MODE>(qmap, kmap, vmap, womap, outmap, a, err, stream);
  if (d == 64) return launch_fwd_t<64, MODE>(qmap, kmap, vmap, womap, outmap, a, err, stream);
  return cudaErrorNotSupported;
}

cudaError_t launch_attn_fwd(const CUtensorMap& qmap, const CUtensorMap& kmap,
                            const CUtensorMap& vmap, const AttnFwdArgs& a, int d, int* err,
                            cudaStream_t stream, const CUtensorMap* womap,
                            const CUtensorMap* outmap) {
  if (a.S <= 0 || a.heads <= 0) return cudaSuccess;
  const bool fuse = womap != nullptr;
  if (fuse != (outmap != nullptr) || (fuse && (a.wo_tiles <= 0 || a.O || a.dO || a.lse_in)))
    return cudaErrorInvalidValue;
  if (fuse) return launch_fwd_d<kModeFused>(d, qmap, kmap, vmap, *womap, *outmap, a, err, stream);
  // the unused map parameters are passed as copies of the Q map
  if (a.lse_in) {
    if (a.lse) return cudaErrorInvalidValue;   // the LSE is an input here
    return launch_fwd_d<kModeKnownLse>(d, qmap, kmap, vmap, qmap, qmap, a, err, stream);
  }
  return launch_fwd_d<kModeStore>(d, qmap, kmap, vmap, qmap, qmap, a, err, stream);
}

}  // namespace upipe
