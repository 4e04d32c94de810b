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
// Precision: Q, K, V and dO arrive in fp16 and P and dS are written in fp16,
// so every MMA here is an fp16 MMA with fp32 accumulation (11 significant bits
// in each operand; bf16 has 8).  fp16's range is narrow, so P, dO and dS carry
// exact power-of-two factors (see "backward fp16 scales" in internal.h):
//   P'' = rho P (rho = 2^14, folded into the LSE), dO' = sigma dO (applied by
//   the dO GEMM), dS'' = P'' (lambda dP' - lambda D') (lambda folded into the
//   packed FMA that subtracts D), so dV'' = rho sigma dV and dQ'', dK'' =
//   lambda rho sigma dQ, dK; the epilogue divides the factors out.
//
// One CTA owns 128 keys (one KV tile) of one head and walks the queries from
// its diagonal to the end of the sequence in sub-tiles of 64.  Two TMEM slots
// alternate between sub-tiles, each with its own warpgroup, so that the
// softmax-gradient work of one slot overlaps the tensor core's work on the
// other slot and the two warpgroups overlap each other.
//   warps 0-3    warpgroup of slot 0 (even sub-tiles), warps 4-7 of slot 1 (odd):
//                softmax gradient with one key row (TMEM lane) per thread
//                (P^T, dS^T from S^T, dP^T)
//   warps 8-11   epilogue warpgroup: dQ^T read-out of every sub-tile with one
//                d index per thread, staged in shared memory as [16 queries x
//                32 d] fp32 blocks and added into global dQ by TMA reduce-add
//                (the reduction runs in L2); at the end dK and dV
//   warp 12      TMEM owner and tcgen05.mma issuer
//   warp 13      TMA producer: K, V once, then Q_u, dO_u through 3 stages
//   warps 14-15  idle (they complete warpgroup 3 for register reallocation)
// Registers are moved with setmaxnreg from warpgroups 2 and 3 to the two
// softmax warpgroups: 168 + 168 + 104 + 72 per thread, x 128 threads each =
// 65536, the registers the block is launched with (512 threads x 128).
// TMEM (512 columns), slot s in {0, 1} at column 128 s, two 64-column blocks
// per slot; for sub-tile u, with b = (u >> 1) & 1:
//   block b     S^T_u = K Q_u^T (fp32); then P^T_u (fp16, +0..31) and
//               dS^T_u (fp16, +32..63), A operands of the dV / dK MMAs; then
//               dQ^T_u = K^T dS^T_u (fp32)
//   block 1-b   dP^T_u = V dO_u^T (fp32)
//   [256, 256+d) dV accumulator      [384, 384+d) dK accumulator
// The blocks swap roles on every use of a slot: S^T of sub-tile u + 2 goes
// into the block of dP^T_u (dead once its softmax has run) and is computed
// while the epilogue still reads dQ^T_u; only dP^T_{u+2} waits for that read.
// dS^T_u is also written to shared memory (one 128-byte swizzled row per key)
// where it is the MN-major B operand of dQ^T = K^T dS^T.  MMAs issued by one
// thread complete in order, which makes the reuse of the TMEM slots safe.
// Long walks: dK and dV accumulate in TMEM over every query sub-tile of a
// CTA's walk, and the tensor core's fp32 accumulation drifts over hundreds of
// thousands of steps (the forward's O drifted out of bounds past ~1M keys,
// 65536 accumulation steps).  A CTA therefore walks at most a.walk sub-tiles:
// a longer walk is cut into segments that separate CTAs run, each adding its
// dK / dV partial into the fp32 global accumulators (which every CTA does
// anyway).  Up to 1M tokens (16384 sub-tiles) the host passes the whole walk,
// so every key tile is one CTA; beyond, segments of 8192 sub-tiles.  Grid
// order: segment 0 of every key tile (ascending, heaviest first), then
// segment 1 of the key tiles that have one, and so on.
// For d = 64 the dQ^T MMA still runs with M = 128: its A operand reads past
// the 64-wide K tile into the V tile (inside this CTA's shared memory) and
// the extra 64 output rows are never stored.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {

namespace {

constexpr int kThreads = 512;
constexpr int kWarpMma = 12;
constexpr int kWarpTma = 13;
constexpr int BK = 128;  // keys per CTA
constexpr int BQ = 64;   // queries per sub-tile
constexpr int NST = 3;   // Q/dO stages
constexpr int DQR = 16;  // query rows per dQ staging round

template <int D>
struct BwdCfg {
  static constexpr uint32_t KV_TILE = BK * D * 2;
  static constexpr uint32_t KV_BLOCK = BK * 64 * 2;      // 64-column block of K or V
  static constexpr uint32_t Q_TILE = BQ * D * 2;
  static constexpr uint32_t Q_BLOCK = BQ * 64 * 2;       // 64-column block of Q or dO
  static constexpr uint32_t K_OFF = 0;
  static constexpr uint32_t V_OFF = KV_TILE;
  static constexpr uint32_t ST_OFF = 2 * KV_TILE;        // NST x (Q tile, dO tile)
  static constexpr uint32_t ST_BYTES = 2 * Q_TILE;
  static constexpr uint32_t DS_OFF = ST_OFF + NST * ST_BYTES;   // 2 x [128 keys][64 q] fp16
  static constexpr uint32_t DS_BYTES = BK * BQ * 2;
  // 4 epilogue warps x 4 buffers x [16 q][32 d] fp32
  static constexpr uint32_t DQS_OFF = DS_OFF + 2 * DS_BYTES;
  static constexpr uint32_t DQS_BYTES = DQR * 32 * 4;
  static constexpr int NDQS = 4;
  // 2 warpgroups x 2 parities x (64 lse + 64 D)
  static constexpr uint32_t LD_OFF = DQS_OFF + 4 * NDQS * DQS_BYTES;
  static constexpr uint32_t BAR_OFF = LD_OFF + 2 * 2 * 2 * BQ * 4;
  // the dynamic shared memory base is 1024-byte aligned (checked at entry)
  static constexpr uint32_t SMEM_BYTES = BAR_OFF + 256;
};

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_kernel(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap domap,
    const __grid_constant__ CUtensorMap dqmap, const AttnBwdArgs a, int* __restrict__ err) {
  using Cfg = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem) & 1023u) {  // swizzled tiles need 1024-byte alignment: refuse, no access
    if (threadIdx.x == 0) atomicCAS(err, 0, kErrDeviceTimeout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;            // [NST]
  uint64_t* q_empty = q_full + NST;       // [NST]
  uint64_t* s_full = q_empty + NST;       // [2]
  uint64_t* p_ready = s_full + 2;         // [2]
  uint64_t* dq_full = p_ready + 2;        // [2]
  uint64_t* dq_free = dq_full + 2;        // [2]
  uint64_t* mma_done = dq_free + 2;
  uint64_t* drain_bar = mma_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = a.S;
  const int head = blockIdx.y;
  const int kvh = (a.h0 + head) / a.group - a.kv0;
  // (key tile, segment) of this CTA: key tile jt walks n_u(jt) = NU0 - 2 jt
  // sub-tiles from its diagonal; segment kseg of it exists while
  // n_u(jt) > kseg * walk, i.e. for the first ceil((NU0 - kseg walk) / 2)
  // key tiles
  const int NU0 = (S + BQ - 1) / BQ;
  const int NT = (S + BK - 1) / BK;
  int jt = (int)blockIdx.x, kseg = 0;
  for (;;) {
    const int over = NU0 - kseg * a.walk;
    const int J = over > 0 ? min(NT, (over + 1) / 2) : 0;
    if (J == 0) { jt = -1; break; }   // past the grid the host computed: no work
    if (jt < J) break;
    jt -= J;
    ++kseg;
  }
  if (jt < 0) return;
  const int k0 = jt * BK;
  const int u0 = kseg * a.walk;                        // first sub-tile of the segment
  const int n_u = min(a.walk, NU0 - 2 * jt - u0);      // query sub-tiles of this CTA
  const int qs0 = k0 + u0 * BQ;                        // its first query

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_ready[s], 4);
      mbar_init(&dq_full[s], 1);
      mbar_init(&dq_free[s], 4);   // the 4 epilogue warps
    }
    mbar_init(mma_done, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpTma && lane == 0) {
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    prefetch_tmap(&domap);
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int wgroup = warp >> 2;
  if (wgroup == 3) {
  setmaxnreg_dec<72>();
  if (warp == kWarpTma) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t issued = 0, issued_phase = 0;
      mbar_expect_tx(kv_full, 2 * Cfg::KV_TILE);
      for (int b = 0; b < D / 64; ++b) {
        tma_load_2d(smem + Cfg::K_OFF + b * Cfg::KV_BLOCK, &kmap, kv_full, kvh * D + 64 * b, k0);
        tma_load_2d(smem + Cfg::V_OFF + b * Cfg::KV_BLOCK, &vmap, kv_full, kvh * D + 64 * b, k0);
      }
      for (int u = 0; u < n_u; ++u) {
        const int st = u % NST;
        const uint32_t ph = (u / NST) & 1;
        if (!mbar_wait(&q_empty[st], ph ^ 1, err, abort_flag)) break;
        mbar_expect_tx(&q_full[st], Cfg::ST_BYTES);
        const int q0 = qs0 + u * BQ;
        uint8_t* base = smem + Cfg::ST_OFF + st * Cfg::ST_BYTES;
        for (int b = 0; b < D / 64; ++b) {
          tma_load_2d(base + b * Cfg::Q_BLOCK, &qmap, &q_full[st], head * D + 64 * b, q0);
          tma_load_2d(base + Cfg::Q_TILE + b * Cfg::Q_BLOCK, &domap, &q_full[st],
                      head * D + 64 * b, q0);
        }
        issued |= 1u << st;
        issued_phase = (issued_phase & ~(1u << st)) | (ph << st);
      }
      if (*abort_flag) {
        mbar_wait_drain(kv_full, 0);
        for (int s = 0; s < NST; ++s)
          if (issued & (1u << s)) mbar_wait_drain(&q_full[s], (issued_phase >> s) & 1u);
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issue
    {  // whole warp; one elected lane issues
      constexpr uint32_t ID_S = idesc_f16(128, BQ, false, false);   // S^T, dP^T
      constexpr uint32_t ID_ACC = idesc_f16(128, D, false, true);   // dV, dK (A in TMEM)
      constexpr uint32_t ID_DQ = idesc_f16(128, BQ, true, true);    // dQ^T = K^T dS^T
      const uint32_t kb = smem_u32(smem + Cfg::K_OFF);
      const uint32_t vb = smem_u32(smem + Cfg::V_OFF);
      bool ok = mbar_wait_warp(kv_full, 0, err, abort_flag);
      for (int u = 0; u <= n_u && ok; ++u) {
        if (u < n_u) {
          const int s = u & 1, st = u % NST, p = (u >> 1) & 1;
          if (!mbar_wait_warp(&q_full[st], (u / NST) & 1, err, abort_flag)) break;
          tc_fence_after();
          const uint32_t qb = smem_u32(smem + Cfg::ST_OFF + st * Cfg::ST_BYTES);
          const uint32_t dob = qb + Cfg::Q_TILE;
          const uint32_t slot = tmem + 128 * s;
          // S^T into the block that held dP^T of sub-tile u - 2 (read by its
          // softmax before its dV / dK MMAs were issued)
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t ko = (k / 4) * Cfg::KV_BLOCK + (k % 4) * 32;
            const uint32_t qo = (k / 4) * Cfg::Q_BLOCK + (k % 4) * 32;
            mma_ss_w(slot + 64 * p, sdesc_sw128(kb + ko, 16, 1024),
                     sdesc_sw128(qb + qo, 16, 1024), ID_S, k > 0);
          }
          // dP^T into the block of dQ^T of sub-tile u - 2: wait for its
          // read-out, which overlaps the S^T MMAs above
          if (u >= 2 && !mbar_wait_warp(&dq_free[s], ((u - 2) >> 1) & 1, err, abort_flag)) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t ko = (k / 4) * Cfg::KV_BLOCK + (k % 4) * 32;
            const uint32_t qo = (k / 4) * Cfg::Q_BLOCK + (k % 4) * 32;
            mma_ss_w(slot + 64 * (1 - p), sdesc_sw128(vb + ko, 16, 1024),
                     sdesc_sw128(dob + qo, 16, 1024), ID_S, k > 0);
          }
          mma_commit_w(&s_full[s]);
        }
        if (u >= 1) {
          const int v = u - 1, sv = v & 1, stv = v % NST, pv = (v >> 1) & 1;
          if (!mbar_wait_warp(&p_ready[sv], (v >> 1) & 1, err, abort_flag)) break;
          tc_fence_after();
          const uint32_t qb = smem_u32(smem + Cfg::ST_OFF + stv * Cfg::ST_BYTES);
          const uint32_t dob = qb + Cfg::Q_TILE;
          const uint32_t slot = tmem + 128 * sv + 64 * pv;  // P^T | dS^T, then dQ^T
          const uint32_t dsb = smem_u32(smem + Cfg::DS_OFF + sv * Cfg::DS_BYTES);
          // dV += P^T dO ; dK += dS^T Q   (k over the sub-tile's 64 queries)
#pragma unroll
          for (int k = 0; k < BQ / 16; ++k) {
            const uint32_t acc = (v > 0 || k > 0) ? 1u : 0u;
            mma_ts_w(tmem + 256, slot + k * 8, sdesc_sw128(dob + k * 2048, Cfg::Q_BLOCK, 1024),
                   ID_ACC, acc);
            mma_ts_w(tmem + 384, slot + 32 + k * 8,
                   sdesc_sw128(qb + k * 2048, Cfg::Q_BLOCK, 1024), ID_ACC, acc);
          }
          // dQ^T = K^T dS^T  (k over the 128 keys; both operands MN-major),
          // over P^T / dS^T: the dV / dK MMAs above read them first
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_ss_w(slot, sdesc_sw128(kb + k * 2048, Cfg::KV_BLOCK, 1024),
                   sdesc_sw128(dsb + k * 2048, Cfg::Q_BLOCK, 1024), ID_DQ, k > 0);
          mma_commit_w(&dq_full[sv]);
          mma_commit_w(&q_empty[stv]);
        }
      }
      mma_commit_w(mma_done);
    }
  }
  } else if (wgroup < 2) {
    // ------------------------------- slot warpgroups: softmax gradient
    setmaxnreg_inc<168>();
    const int wg = wgroup;           // slot served by this warpgroup
    const int qw = warp & 3;
    const int r = qw * 32 + lane;    // TMEM lane: key row of S^T/dP^T, d index of dQ^T
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    const uint32_t slot = tmem + lane_off + 128 * wg;
    const float sl2 = a.scale * 1.4426950408889634f;
    const float2 sl2x2 = make_float2(sl2, sl2);
    const float lam = grad_lambda(*a.do_max, *a.vmax);
    const float2 lam2 = make_float2(lam, lam);
    const float* lse_g = a.lse + (long long)head * a.lse_stride;
    const float* D_g = a.D + (long long)head * S;
    // lse/D of the current sub-tile, shared by the warpgroup and double-buffered
    // by sub-tile parity (every warp writes the same values before reading)
    float* ld_wg = reinterpret_cast<float*>(smem + Cfg::LD_OFF) + wg * 2 * (2 * BQ);
    uint8_t* ds_rows = smem + Cfg::DS_OFF + wg * Cfg::DS_BYTES + r * 128;
    // lse (log2 units) and D of the queries of a sub-tile, loaded one sub-tile
    // of this slot ahead: lane l holds queries l and l + 32
    float nl[2], nd[2];
    auto fetch = [&](int u) {
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int q = min(qs0 + u * BQ + 32 * m + lane, S - 1);  // clamp: masked below
        const bool ok_l = dbg_in2(head, a.heads, q, q, a.lse_stride, err);
        const bool ok_d = dbg_in2(head, a.heads, q, q, S, err);
        nl[m] = ok_l ? ld_nc_f32(lse_g + q) : 0.f;
        nd[m] = ok_d ? ld_nc_f32(D_g + q) : 0.f;
      }
    };
    if (wg < n_u) fetch(wg);
    bool ok = true;
    for (int u = wg; u < n_u; u += 2) {
      const uint32_t ph = (u >> 1) & 1;
      float* ld_w = ld_wg + ph * (2 * BQ);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const bool live = qs0 + u * BQ + 32 * m + lane < S;  // queries past S: P = 0
        // stored negated, as the packed FMAs below take them: -lse (log2
        // units) + log2(rho), so that exp2 gives P'' = rho P; and -lambda D'
        ld_w[32 * m + lane] = live ? kGradRhoLog2 - nl[m] * 1.4426950408889634f : -INFINITY;
        ld_w[BQ + 32 * m + lane] = live ? -lam * nd[m] : 0.f;
      }
      __syncwarp();
      if (u + 2 < n_u) fetch(u + 2);
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[wg], ph, err, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const float4* lse4 = reinterpret_cast<const float4*>(ld_w);
      const float4* dd4 = reinterpret_cast<const float4*>(ld_w + BQ);
      // columns c < mask_from hold key > query: masked (first segment only)
      const int mask_from = r - (u0 + u) * BQ;
      uint8_t* row = ds_rows;
      // the slot's two 64-column blocks swap roles on every use of the slot
      const uint32_t sblk = slot + 64 * ph, pblk = slot + 64 * (ph ^ 1);
      // two halves of 32 queries: P^T, then dS^T = P^T (dP^T - D).  dS^T goes
      // over the second half of S^T, so the first half's dS^T is stored to
      // TMEM only after the second half of S^T has been read.
      uint32_t ds0[16];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float p[32];
        {
          uint32_t rr[32];
          tmem_ld32(sblk + 32 * h, rr);
          tmem_ld_wait(rr);
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 l4 = lse4[(32 * h + i) / 4];  // log2(rho) - lse (log2 units)
            const float2 x0 = ffma2(make_float2(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])),
                                    sl2x2, make_float2(l4.x, l4.y));
            const float2 x1 = ffma2(make_float2(__uint_as_float(rr[i + 2]), __uint_as_float(rr[i + 3])),
                                    sl2x2, make_float2(l4.z, l4.w));
            p[i] = ex2(x0.x);
            p[i + 1] = ex2(x0.y);
            p[i + 2] = ex2(x1.x);
            p[i + 3] = ex2(x1.y);
          }
        }
        if (h == 1) tmem_st16(sblk + 32, ds0);  // S^T fully read now
        if (mask_from > 32 * h) {  // only the two sub-tiles on the diagonal
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * h + i < mask_from) p[i] = 0.f;
        }
        {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack_f16(p[2 * i], p[2 * i + 1]);
          tmem_st16(sblk + 16 * h, pk);
        }
        {
          uint32_t rr[32], pk[16];
          tmem_ld32(pblk + 32 * h, rr);
          tmem_ld_wait(rr);
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 d4 = dd4[(32 * h + i) / 4];  // -lambda D'
            // dS'' = P'' (lambda dP' - lambda D')
            const float2 g0 = fmul2(make_float2(p[i], p[i + 1]),
                                    ffma2(make_float2(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])),
                                          lam2, make_float2(d4.x, d4.y)));
            const float2 g1 = fmul2(make_float2(p[i + 2], p[i + 3]),
                                    ffma2(make_float2(__uint_as_float(rr[i + 2]), __uint_as_float(rr[i + 3])),
                                          lam2, make_float2(d4.z, d4.w)));
            pk[i / 2] = pack_f16(g0.x, g0.y);
            pk[i / 2 + 1] = pack_f16(g1.x, g1.y);
          }
          if (h == 0) {
#pragma unroll
            for (int i = 0; i < 16; ++i) ds0[i] = pk[i];
          } else {
            tmem_st16(sblk + 48, pk);
          }
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const int c = 4 * h + ch;  // 16-byte chunk of the 128-byte row
            *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
          }
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_ready[wg]);

    }
  } else {
    // ------------------------------------------ epilogue: dQ, then dK / dV
    setmaxnreg_dec<104>();
    const int qw = warp & 3;
    const int t = qw * 32 + lane;    // TMEM lane: d index of dQ^T, key row of dK/dV
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    uint8_t* stage_w = smem + Cfg::DQS_OFF + qw * Cfg::NDQS * Cfg::DQS_BYTES;
    uint32_t round = 0;  // dQ staging rounds issued by this warp
    // the exact power-of-two factors to divide out: dQ'' and dK'' carry
    // lambda rho sigma, dV'' carries rho sigma (and dQ, dK take 1/sqrt(d))
    const double rs = (double)kGradRho * (double)grad_sigma(a.bound);
    const float dq_mul = (float)((double)a.scale / (rs * (double)grad_lambda(*a.do_max, *a.vmax)));
    const float dv_mul = (float)(1.0 / rs);
    bool ok = true;
    for (int u = 0; u < n_u; ++u) {
      const int s = u & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&dq_full[s], (u >> 1) & 1, err, abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t lo[32], hi[32];
      const uint32_t dqb = tmem + lane_off + 128 * s + 64 * ((u >> 1) & 1);
      tmem_ld32(dqb, lo);
      tmem_ld_wait(lo);
      tmem_ld32(dqb + 32, hi);
      tmem_ld_wait(hi);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dq_free[s]);
      if (qw * 32 < D) {
        const int q0 = qs0 + u * BQ;
        const uint32_t cb = (uint32_t)(lane >> 2), cw = (uint32_t)(lane & 3) * 4;
#pragma unroll
        for (int rd = 0; rd < BQ / DQR; ++rd, ++round) {
          uint8_t* buf = stage_w + (round % Cfg::NDQS) * Cfg::DQS_BYTES;
          if (lane == 0) bulk_wait_read<Cfg::NDQS - 1>();   // buf's previous reduce has read it
          __syncwarp();
#pragma unroll
          for (int c = 0; c < DQR; ++c) {
            const int q = rd * DQR + c;   // compile-time after unrolling
            *reinterpret_cast<float*>(buf + c * 128 + ((cb ^ (c & 7)) << 4) + cw) =
                __uint_as_float(q < 32 ? lo[q & 31] : hi[q & 31]) * dq_mul;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_2d(&dqmap, buf, head * D + 32 * qw, q0 + rd * DQR);
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(mma_done, 0, err, abort_flag));
    if (ok) {
      tc_fence_after();
      const int key = k0 + t;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rv[32], rk[32];
        tmem_ld32(tmem + lane_off + 256 + 32 * c, rv);
        tmem_ld_wait(rv);
        tmem_ld32(tmem + lane_off + 384 + 32 * c, rk);
        tmem_ld_wait(rk);
        if (key < S && dbg_in2(key, S, kvh * D + 32 * c, kvh * D + 32 * c + 31, a.ld_dkv, err)) {
          const long long off = (long long)key * a.ld_dkv + kvh * D + 32 * c;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            red_add_v4_f32(a.dV + off + i, __uint_as_float(rv[i]) * dv_mul,
                           __uint_as_float(rv[i + 1]) * dv_mul,
                           __uint_as_float(rv[i + 2]) * dv_mul,
                           __uint_as_float(rv[i + 3]) * dv_mul);
            red_add_v4_f32(a.dK + off + i, __uint_as_float(rk[i]) * dq_mul,
                           __uint_as_float(rk[i + 1]) * dq_mul,
                           __uint_as_float(rk[i + 2]) * dq_mul,
                           __uint_as_float(rk[i + 3]) * dq_mul);
          }
        }
      }
    }
  }

  // --------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
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
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t ea = smem_attr_once(attn_bwd_kernel<D>, (int)Cfg::SMEM_BYTES, attr_done);
  if (ea != cudaSuccess) return ea;
  CUtensorMap qm, km, vm, dm, dqm;
  if (!make_tmap_f32(&dqm, a.dQ, a.S, (uint64_t)a.ld_dq, a.ld_dq, DQR, 32) ||
      !make_tmap_bf16(&qm, a.Q, a.S, (uint64_t)a.heads * D, a.ldq, BQ, 64) ||
      !make_tmap_bf16(&km, a.K, a.S, (uint64_t)a.ldkv, a.ldkv, BK, 64) ||
      !make_tmap_bf16(&vm, a.V, a.S, (uint64_t)a.ldkv, a.ldkv, BK, 64) ||
      !make_tmap_bf16(&dm, a.dO, a.S, (uint64_t)a.heads * D, a.ld_do, BQ, 64))
    return cudaErrorInvalidValue;
  // CTAs: segment k of the walks for the key tiles whose walk is longer than
  // k * walk sub-tiles (see the kernel)
  const long long NU0 = (a.S + BQ - 1) / BQ, NT = (a.S + BK - 1) / BK;
  long long ctas = 0;
  for (long long k = 0; NU0 - k * a.walk > 0; ++k)
    ctas += std::min(NT, (NU0 - k * a.walk + 1) / 2);
  if (a.walk <= 0 || a.walk % 2 != 0 || ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  dim3 grid((unsigned)ctas, a.heads);
  attn_bwd_kernel<D><<<grid, kThreads, Cfg::SMEM_BYTES, stream>>>(qm, km, vm, dm, dqm, a, err);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const AttnBwdArgs& a, int* err, cudaStream_t stream) {
  if (a.S <= 0 || a.heads <= 0) return cudaSuccess;
  if (a.d == 128) return launch_bwd_t<128>(a, err, stream);
  if (a.d == 64) return launch_bwd_t<64>(a, err, stream);
  return cudaErrorNotSupported;
}

}  // namespace upipe
