// Persistent tcgen05 GEMM with fused epilogues.
//
//   C[M, N] = sum_k A[m, k] * B[n, k]       (bf16 operands, fp32 in TMEM)
//
// One CTA per SM walks the output tiles (MT x 128 rows x BN columns) with a
// static stride.  Warp roles:
//   warp 0      TMA producer: 128-byte-swizzled 64-wide K slabs of A (MT
//               128-row tiles) and B into a ring of shared-memory stages;
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma M=128, N=BN, K=16 per
//               128-row part (MT = 2: two parts share each B slab, halving
//               the B bytes loaded and read per FLOP), accumulating into one
//               of two TMEM accumulator sets, so that the epilogue of tile i
//               overlaps the main loop of tile i+1;
//   warps 2..5  epilogue: tcgen05.ld of one accumulator row per thread,
//               then the fused operation and the global store.
// Operands may be K-major (row-major [M,K] / [N,K]) or MN-major ([K,M] /
// [K,N]); the layout is chosen by the instruction descriptor's transpose bits
// and the shared-memory descriptors, the data is never transposed.
// K segments: the K range may run through several (A, B) tensor-map pairs
// into one accumulator (dx += sum of a chunk's gradient parts times their
// weight slices).  M segments: 128-row tile runs may each take their own A
// map and output pointer (a chunk's split-K weight gradients in one launch).
//
// Epilogues (what the attention layer needs around the attention kernel):
//   EPI_PROJ        Q/K/V projection of one head chunk: optional per-head
//                   RMSNorm (Qwen3 geometry), RoPE, fp16 store to workspace
//                   (the attention kernels' operand type);
//   EPI_F32         Wo-slice partial result: out (+)= O_c Wo_c^T in fp32,
//                   staged per warp in shared memory and written by TMA store
//                   (first chunk) or TMA reduce-add (later chunks: the
//                   read-modify-write runs in L2, the SM never reads out);
//   EPI_DO          dO_c = dOut Wo_c, scaled and stored in fp16 (and, given
//                   O, D = rowsum(dO * O) per head);
//   EPI_F32_ATOMIC  split-K weight gradients, reduced with red.global.add
//                   after a transpose through shared memory (whole
//                   128-byte row segments per instruction);
//   EPI_SWIGLU      the sequence-tiled MLP's gate and up projections: each
//                   256-wide output tile is 128 gate rows and the same 128 up
//                   rows (two B maps, one 128-row TMA box each into one B
//                   stage), and the epilogue stores a = silu(g) * u in bf16;
//   EPI_SWIGLU_BWD  the same recomputed, with dA read for the tile and
//                   dg = dA u silu'(g), du = dA silu(g) and a stored in bf16;
//   EPI_LSE_PART    the sequence-tiled loss's logits z = h W^T: per row and
//                   vocabulary tile the (max, sum of exp) partial of the
//                   log-sum-exp, and the target's logit; z is never stored;
//   EPI_DLOGITS     the same recomputed: dz = scale (softmax - onehot), bf16.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;                      // one 128-byte swizzle atom of bf16
constexpr int kThreads = 192;
constexpr uint32_t A_STAGE_BYTES = BM * BK * 2;  // 16 KB

constexpr int kEpiBufs = 2;                       // staging buffers per epilogue warp
constexpr uint32_t EPI_BUF_BYTES = 32 * 32 * 4;   // [32 rows][32 cols] fp32

// MT: 128-row A tiles per output tile (MT = 2: two accumulators share each
// B tile, halving the B bytes loaded and read per FLOP)
template <int BN, int MT = 1>
struct GemmCfg {
  static constexpr uint32_t B_STAGE_BYTES = BN * BK * 2;
  static constexpr uint32_t STAGE_BYTES = MT * A_STAGE_BYTES + B_STAGE_BYTES;
  static constexpr int STAGES = (STAGE_BYTES > 32768) ? 4 : 6;
  static constexpr uint32_t TMEM_COLS = (2 * MT * BN < 32) ? 32 : 2 * MT * BN;
  static constexpr uint32_t EPI_OFF = STAGES * STAGE_BYTES;
  static constexpr uint32_t BAR_OFF = EPI_OFF + 4 * kEpiBufs * EPI_BUF_BYTES;
  static constexpr uint32_t SMEM_BYTES = BAR_OFF + 1024 /*align*/ + 256 /*bars*/;
};

struct TileCoord {
  int m0, n0, kb0, kb1;
};

// Every tensor map of one launch, passed as one __grid_constant__ parameter
// (TMA reads a map straight from parameter space).
struct GemmMaps {
  CUtensorMap a[kMaxASegs];
  CUtensorMap b[kMaxBMaps];
  CUtensorMap c;
};

// Tile order: column tiles fastest (consecutive tiles share an A row block;
// the B operand cycles), or with m_fastest = 1 row blocks fastest
// (consecutive tiles share a B column tile; A cycles and should be the
// operand that stays in L2), or with m_fastest = G > 1 the same within groups
// of G row blocks, group after group (B is read once per group, and only a
// group's A rows cycle).
// (Host and device: the host copy backs upipe_gemm_tile_order.)
__host__ __device__ __forceinline__ TileCoord tile_coord(int t, int num_m, int num_n, int kb_total,
                                                         int ksplit, int tile_rows, int m_fastest) {
  const int per_split = num_m * num_n;
  const int ks = t / per_split;
  const int r = t - ks * per_split;
  TileCoord c;
  if (m_fastest > 1) {
    // groups of m_fastest row blocks: within a group row blocks fastest, then
    // columns, then the next group (only a group's A rows need stay in L2)
    const int group = r / (m_fastest * num_n);
    const int rem = r - group * m_fastest * num_n;
    const int left = num_m - group * m_fastest;   // row blocks in this group
    const int gm = left < m_fastest ? left : m_fastest;
    c.m0 = (group * m_fastest + rem % gm) * tile_rows;
    c.n0 = rem / gm;
  } else if (m_fastest) {
    c.m0 = (r % num_m) * tile_rows;
    c.n0 = r / num_m;
  } else {
    c.m0 = (r / num_n) * tile_rows;
    c.n0 = (r % num_n);
  }
  const int kb_per = (kb_total + ksplit - 1) / ksplit;
  c.kb0 = ks * kb_per;
  c.kb1 = kb_total < c.kb0 + kb_per ? kb_total : c.kb0 + kb_per;
  return c;
}

// ---- epilogue helpers -------------------------------------------------

// cos/sin of pos * w_i from the two-level table: angle = hi part + lo part.
// The lo part comes from the transposed table, so that the warp's threads
// (consecutive rows) read consecutive entries.
__device__ __forceinline__ void rope_cs(const float2* __restrict__ hi,
                                        const float2* __restrict__ lo_t, long long pos, int half,
                                        int i, float& c, float& s) {
  const float2 a = __ldg(hi + (pos >> 10) * half + i);
  const float2 b = __ldg(lo_t + (long long)i * 1024 + (pos & 1023));
  c = a.x * b.x - a.y * b.y;
  s = a.y * b.x + a.x * b.y;
}

// sigmoid(v) = 1 / (1 + e^-v) with the fast exponential and reciprocal
// division; the exponent is clamped at 80 so that the divisor stays below
// 2^126, where the fast division is exact to its error bound (for v < -80,
// sigmoid(v) < 2e-35 either way)
__device__ __forceinline__ float sigmoid_fast(float v) {
  return __fdividef(1.f, 1.f + __expf(fminf(-v, 80.f)));
}

// Stores a warp's [32 rows x 32 cols] bf16 block, held one row per thread as
// four 16-byte chunks w[0..3], through ``buf`` (2 KB of this warp's shared
// memory): each instruction then writes 8 whole 64-byte row segments (lane:
// row 8k + l/4, chunk l%4) instead of 16-byte pieces of 32 rows.  Chunks are
// swizzled by row pair, which keeps both the row-per-thread writes and the
// row-segment reads free of bank conflicts.  Rows at or past ``rows`` are not
// stored.
__device__ __forceinline__ void warp_store_rows_bf16(uint8_t* buf, int lane, const uint4 (&w)[4],
                                                     bf16* dst, long long ld, long long row0,
                                                     long long rows, long long col, int* err) {
  __syncwarp();   // the previous block's reads of buf are done
  const int pr = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ pr) << 4)) = w[j];
  __syncwarp();
  const int sq = lane & 3, sr = lane >> 2;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int rr = 8 * k + sr;
    const long long row = row0 + rr;
    // streaming store: the block is read once, by a later GEMM
    if (row < rows && dbg_in2(row, rows, col, col + 31, ld, err))
      __stcs(reinterpret_cast<uint4*>(dst + row * ld + col + 8 * sq),
             *reinterpret_cast<const uint4*>(buf + rr * 64 + ((sq ^ ((rr >> 1) & 3)) << 4)));
  }
}

template <int D>
__device__ __forceinline__ void epi_proj_row(const EpiParams& ep, const ProjSeg& sg, long long m,
                                             long long M, int n_local, float (&v)[D], int* err) {
  constexpr int H = D / 2;
  if (sg.mode == PROJ_NORM_ROPE) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < D; ++i) ss = fmaf(v[i], v[i], ss);
    const float rs = rsqrtf(ss * (1.0f / D) + ep.eps);
    if (sg.yhat && dbg_in2(m, M, n_local, n_local + D - 1, sg.ld_yhat, err)) {
      float* yp = sg.yhat + m * sg.ld_yhat + n_local;
#pragma unroll
      for (int i = 0; i < D; i += 4)
        *reinterpret_cast<float4*>(yp + i) =
            make_float4(v[i] * rs, v[i + 1] * rs, v[i + 2] * rs, v[i + 3] * rs);
    }
#pragma unroll
    for (int i = 0; i < D; ++i) {
      const float gmul = sg.gamma ? __ldg(sg.gamma + i) : 1.f;
      v[i] = v[i] * rs * gmul;
    }
  }
  if (sg.mode != PROJ_PLAIN) {
#pragma unroll
    for (int i = 0; i < H; ++i) {
      float c, s;
      rope_cs(ep.rope_hi, ep.rope_lo_t, m, H, i, c, s);
      const float a = v[i], b = v[i + H];
      v[i] = a * c - b * s;
      v[i + H] = b * c + a * s;
    }
  }
  // fp16 store: values beyond its range (|v| > 65504) would become inf; the
  // error word reports them (UPIPE_ERR_RANGE).  The optional row norm feeds
  // the backward's fp16 scale of dS.
  float amax = 0.f, ss = 0.f;
#pragma unroll
  for (int i = 0; i < D; ++i) {
    amax = fmaxf(amax, fabsf(v[i]));
    if (sg.norm_max) ss = fmaf(v[i], v[i], ss);
  }
  if (amax > 65504.f) atomicCAS(err, 0, kErrRange);
  if (sg.norm_max) atomic_max_nonneg(sg.norm_max, sqrtf(ss));
  if (!dbg_in2(m, M, sg.col0 + n_local, sg.col0 + n_local + D - 1, sg.ld, err)) return;
  __half* op = sg.out + m * sg.ld + sg.col0 + n_local;
#pragma unroll
  for (int i = 0; i < D; i += 8) {
    uint4 w;
    w.x = pack_f16(v[i + 0], v[i + 1]);
    w.y = pack_f16(v[i + 2], v[i + 3]);
    w.z = pack_f16(v[i + 4], v[i + 5]);
    w.w = pack_f16(v[i + 6], v[i + 7]);
    *reinterpret_cast<uint4*>(op + i) = w;
  }
}

}  // namespace

template <int BN, bool A_MN, bool B_MN, int EPI, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs g, const EpiParams ep,
                int* __restrict__ err) {
  using Cfg = GemmCfg<BN, MT>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int num_m = g.nmseg > 0 ? g.mseg_t0[g.nmseg] : (g.M + BM * MT - 1) / (BM * MT);
  const int num_n = g.N / BN;
  const int kb_total = g.nkseg > 0 ? g.kseg_end[g.nkseg - 1] : (g.K + BK - 1) / BK;
  const int ksplit = g.ksplit > 0 ? g.ksplit : 1;
  const int num_tiles = num_m * num_n * ksplit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.a[0]);
    prefetch_tmap(&maps.b[0]);
    if (EPI == EPI_PROJ) {
      prefetch_tmap(&maps.b[1]);
      prefetch_tmap(&maps.b[2]);
    }
    if (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD) prefetch_tmap(&maps.b[1]);
    for (int s = 1; s < g.nkseg; ++s) {
      prefetch_tmap(&maps.a[g.kseg_a[s]]);
      prefetch_tmap(&maps.b[g.kseg_b[s]]);
    }
    for (int s = 1; s < g.nmseg; ++s) prefetch_tmap(&maps.a[g.mseg_a[s]]);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_phase = 0;  // per-stage bit masks
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, num_m, num_n, kb_total, ksplit, BM * MT, g.m_fastest);
        const int n0 = tc.n0 * BN;
        const CUtensorMap* am = &maps.a[0];
        const CUtensorMap* bm = &maps.b[0];
        int brow = n0;
        int arow = tc.m0;  // first row of the A tile in its tensor map
        if (g.nmseg > 0) {
          const int mt = tc.m0 / BM;
          int s = 0;
          while (s + 1 < g.nmseg && mt >= g.mseg_t0[s + 1]) ++s;
          am = &maps.a[g.mseg_a[s]];
          arow = (mt - g.mseg_t0[s]) * BM;
        }
        if (EPI == EPI_PROJ) {
          int s = 0;
          while (s + 1 < ep.nseg && n0 >= ep.seg[s].n_end) ++s;
          bm = &maps.b[ep.seg[s].bmap];
          brow = ep.seg[s].b_row0 + (n0 - ep.seg[s].n_begin);
        }
        // K segment holding block kb (always segment 0 without K segments)
        int ks = 0, ks_kb0 = 0;
        for (int kb = tc.kb0; kb < tc.kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, err, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * Cfg::STAGE_BYTES;
          uint8_t* sb = sa + MT * A_STAGE_BYTES;
          mbar_expect_tx(&full[stage], Cfg::STAGE_BYTES);
          if (g.nkseg > 0) {
            while (kb >= g.kseg_end[ks]) ks_kb0 = g.kseg_end[ks++];
            am = &maps.a[g.kseg_a[ks]];
            bm = &maps.b[g.kseg_b[ks]];
          }
          const int k0 = (kb - ks_kb0) * BK;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            uint8_t* sam = sa + mt * A_STAGE_BYTES;
            if (!A_MN) {
              tma_load_2d(sam, am, &full[stage], k0, arow + BM * mt);
            } else {
              tma_load_2d(sam, am, &full[stage], arow + BM * mt, k0);
              tma_load_2d(sam + 8192, am, &full[stage], arow + BM * mt + 64, k0);
            }
          }
          if (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD) {
            // gate rows, then the same up rows: one 256-row K-major B tile
            tma_load_2d(sb, &maps.b[0], &full[stage], k0, brow / 2);
            tma_load_2d(sb + (BN / 2) * BK * 2, &maps.b[1], &full[stage], k0, brow / 2);
          } else if (!B_MN) {
            tma_load_2d(sb, bm, &full[stage], k0, brow);
          } else {
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(sb + i * 8192, bm, &full[stage], brow + 64 * i, k0);
          }
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (*abort_flag) {
        // leave no bulk copy in flight into this CTA's shared memory
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) mbar_wait_drain(&full[s], (issued_phase >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue
    {  // whole warp; one elected lane issues
      constexpr uint32_t IDESC = idesc_bf16(BM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++it) {
        const TileCoord tc = tile_coord(t, num_m, num_n, kb_total, ksplit, BM * MT, g.m_fastest);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_warp(&acc_empty[acc], acc_phase ^ 1, err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * (MT * BN);
        for (int kb = tc.kb0; kb < tc.kb1; ++kb) {
          if (!mbar_wait_warp(&full[stage], phase, err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::STAGE_BYTES);
          const uint32_t sb = sa + MT * A_STAGE_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            uint64_t bd;
            if (!B_MN) bd = sdesc_sw128(sb + k * 32, 16, 1024);
            else bd = sdesc_sw128(sb + k * 2048, 8192, 1024);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const uint32_t sam = sa + mt * A_STAGE_BYTES;
              uint64_t ad;
              if (!A_MN) ad = sdesc_sw128(sam + k * 32, 16, 1024);
              else ad = sdesc_sw128(sam + k * 2048, 8192, 1024);
              mma_ss_w(d_tmem + mt * BN, ad, bd, IDESC, (kb > tc.kb0 || k > 0) ? 1u : 0u);
            }
          }
          mma_commit_w(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        // an empty K range (split-K remainder) commits without MMAs; the
        // epilogue skips such tiles by the same test
        mma_commit_w(&acc_full[acc]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int it = 0;
    uint32_t epi_round = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const TileCoord tc = tile_coord(t, num_m, num_n, kb_total, ksplit, BM * MT, g.m_fastest);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      // warp-uniform: the tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[acc], acc_phase, err, abort_flag))) break;
      tc_fence_after();
#pragma unroll 1
      for (int mt = 0; mt < MT; ++mt) {
      const int m0t = tc.m0 + BM * mt;  // first row of this 128-row part
      const uint32_t tbase =
          tmem_base + acc * (MT * BN) + mt * BN + ((uint32_t)(quarter * 32) << 16);
      const long long m = (long long)m0t + row;
      const int n0 = tc.n0 * BN;
      const bool live = (m < g.M) && (tc.kb1 > tc.kb0);

      if constexpr (EPI == EPI_PROJ) {
        constexpr int D = BN;  // one head per tile
        float v[D];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[c * 32 + i] = __uint_as_float(r[i]);
        }
        if (live) {
          int s = 0;
          while (s + 1 < ep.nseg && n0 >= ep.seg[s].n_end) ++s;
          const ProjSeg& sg = ep.seg[s];
          const int n_local = n0 - sg.n_begin;
          if (sg.mode == PROJ_NORM_ROPE && sg.rstd &&
              dbg_in2(n_local / D, (sg.n_end - sg.n_begin) / D, m, m, g.M, err)) {
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < D; ++i) ss = fmaf(v[i], v[i], ss);
            sg.rstd[(long long)(n_local / D) * g.M + m] = rsqrtf(ss * (1.0f / D) + ep.eps);
          }
          epi_proj_row<D>(ep, sg, m, g.M, n_local, v, err);
        }
      } else if constexpr (EPI == EPI_DO) {
        constexpr int D = BN;
        float dot = 0.f, ss = 0.f;
        const int head = n0 / D;
        const float sigma = grad_sigma(ep.bound);
        // this row's D columns of dO' [M, ld_do] and O [M, ld_o]
        const bool row_ok = live && dbg_in2(m, g.M, n0, n0 + D - 1, ep.ld_do, err) &&
                            (!ep.O || dbg_in2(m, g.M, n0, n0 + D - 1, ep.ld_o, err));
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          tmem_ld_wait(r);
          if (row_ok) {
            __half* dp = ep.dO + m * ep.ld_do + n0 + c * 32;
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 w;
              uint32_t* wp = &w.x;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                // D' and the norm use the fp16 dO' the attention backward
                // will read, so that sum_j dS_ij stays consistent with dP
                wp[j] = pack_f16(__uint_as_float(r[i + 2 * j]) * sigma,
                                 __uint_as_float(r[i + 2 * j + 1]) * sigma);
                const float2 dv = unpack_f16(wp[j]);
                ss = fmaf(dv.x, dv.x, ss);
                ss = fmaf(dv.y, dv.y, ss);
              }
              if (ep.O) {
                const uint4 ov = *reinterpret_cast<const uint4*>(ep.O + m * ep.ld_o + n0 + c * 32 + i);
                const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const float2 dv = unpack_f16(wp[j]);
                  const float2 of = __bfloat1622float2(o2[j]);
                  dot = fmaf(dv.x, of.x, dot);
                  dot = fmaf(dv.y, of.y, dot);
                }
              }
              *reinterpret_cast<uint4*>(dp + i) = w;
            }
          }
        }
        if (row_ok) {
          if (ep.O && dbg_in2(head, g.N / D, m, m, g.M, err)) ep.D[(long long)head * g.M + m] = dot;
          atomic_max_nonneg(ep.do_max, sqrtf(ss));
        }
      } else if constexpr (EPI == EPI_SWIGLU) {
        // accumulator columns [0, 128): g, [128, 256): u of output columns
        // [c0, c0 + 128) of this row; a = silu(g) u leaves through shared
        // memory as whole row segments
        constexpr int H = BN / 2;
        const long long c0 = n0 / 2;
        uint8_t* buf0 = smem + Cfg::EPI_OFF + quarter * kEpiBufs * EPI_BUF_BYTES;
        const long long wrow0 = (long long)m0t + quarter * 32;   // first row of this warp
        const bool warp_live = (tc.kb1 > tc.kb0) && wrow0 < g.M;
#pragma unroll 1
        for (int c = 0; c < H / 32; ++c) {
          uint32_t rg[32], ru[32];
          tmem_ld32(tbase + 32 * c, rg);
          tmem_ld_wait(rg);
          tmem_ld32(tbase + H + 32 * c, ru);
          tmem_ld_wait(ru);
          if (!warp_live) continue;   // warp-uniform
          uint4 w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t* wp = &w[q].x;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int i = 8 * q + 2 * j;
              const float g0 = __uint_as_float(rg[i]), g1 = __uint_as_float(rg[i + 1]);
              const float u0 = __uint_as_float(ru[i]), u1 = __uint_as_float(ru[i + 1]);
              wp[j] = pack_bf16(g0 * sigmoid_fast(g0) * u0, g1 * sigmoid_fast(g1) * u1);
            }
          }
          warp_store_rows_bf16(buf0, lane, w, ep.act, ep.ld_act, wrow0, g.M, c0 + 32 * c, err);
        }
      } else if constexpr (EPI == EPI_SWIGLU_BWD) {
        // The same accumulator layout.  dA comes in and dg, du and a go out
        // through this warp's two shared-memory buffers, so that every global
        // access is a whole row segment: the [32 rows x 32 cols] fp32 block of
        // dA arrives 4 rows x 128 bytes per instruction (lane: row 4k + l/8,
        // 16-byte chunk l%8) into buf0, 128-byte swizzled, and each thread
        // takes its own row; the three [32 x 32] bf16 outputs (64 bytes a row,
        // 16-byte chunks swizzled by row pair) leave 8 rows x 64 bytes per
        // instruction (lane: row 8k + l/4, chunk l%4).  dg and du are staged
        // in buf1, a in buf0 once dA has been read out of it.
        constexpr int H = BN / 2;
        const long long c0 = n0 / 2;
        uint8_t* buf0 = smem + Cfg::EPI_OFF + quarter * kEpiBufs * EPI_BUF_BYTES;
        uint8_t* buf1 = buf0 + EPI_BUF_BYTES;
        const long long wrow0 = (long long)m0t + quarter * 32;   // first row of this warp
        const bool warp_live = (tc.kb1 > tc.kb0) && wrow0 < g.M;
        const int lq = lane & 7, lr = lane >> 3;   // dA loads
        const int sq = lane & 3, sr = lane >> 2;   // output stores
        const int pr = (lane >> 1) & 3;            // this thread's row-pair swizzle
#pragma unroll 1
        for (int c = 0; c < H / 32; ++c) {
          uint32_t rg[32], ru[32];
          tmem_ld32(tbase + 32 * c, rg);
          tmem_ld_wait(rg);
          tmem_ld32(tbase + H + 32 * c, ru);
          tmem_ld_wait(ru);
          if (!warp_live) continue;   // warp-uniform
          const long long col = c0 + 32 * c;   // first output column of the block
          __syncwarp();   // the previous block's reads of buf0 and buf1 are done
          {
            // all 8 loads in flight at once; dA is read once (streaming)
            float4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const long long row = wrow0 + 4 * k + lr;
              v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (row < g.M && dbg_in2(row, g.M, col, col + 31, ep.ld_da, err))
                v[k] = __ldcs(reinterpret_cast<const float4*>(ep.dA + row * ep.ld_da + col) + lq);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int rr = 4 * k + lr;
              *reinterpret_cast<float4*>(buf0 + rr * 128 + ((lq ^ (rr & 7)) << 4)) = v[k];
            }
          }
          __syncwarp();
          float da[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 d4 =
                *reinterpret_cast<const float4*>(buf0 + lane * 128 + ((k ^ (lane & 7)) << 4));
            da[4 * k] = d4.x;
            da[4 * k + 1] = d4.y;
            da[4 * k + 2] = d4.z;
            da[4 * k + 3] = d4.w;
          }
          __syncwarp();   // every row of dA is out of buf0 before a goes in
#pragma unroll
          for (int j = 0; j < 4; ++j) {   // columns 8j..8j+7: one 16-byte chunk of each output
            uint32_t wg[4], wu[4], wa[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float og[2], ou[2], oa[2];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int i = 8 * j + 2 * e + h;
                const float gv = __uint_as_float(rg[i]), uv = __uint_as_float(ru[i]);
                const float sg = sigmoid_fast(gv);
                const float sl = gv * sg;                      // silu(g)
                og[h] = da[i] * uv * (sg * (1.f + gv * (1.f - sg)));
                ou[h] = da[i] * sl;
                oa[h] = sl * uv;
              }
              wg[e] = pack_bf16(og[0], og[1]);
              wu[e] = pack_bf16(ou[0], ou[1]);
              wa[e] = pack_bf16(oa[0], oa[1]);
            }
            const uint32_t off = lane * 64 + ((j ^ pr) << 4);
            *reinterpret_cast<uint4*>(buf1 + off) = make_uint4(wg[0], wg[1], wg[2], wg[3]);
            *reinterpret_cast<uint4*>(buf1 + 2048 + off) = make_uint4(wu[0], wu[1], wu[2], wu[3]);
            *reinterpret_cast<uint4*>(buf0 + off) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int rr = 8 * k + sr;
            const long long row = wrow0 + rr;
            if (row < g.M && dbg_in2(row, g.M, col, col + 31, ep.ld_dg, err) &&
                dbg_in2(row, g.M, col, col + 31, ep.ld_act, err)) {
              const uint32_t off = rr * 64 + ((sq ^ ((rr >> 1) & 3)) << 4);
              const long long og = row * ep.ld_dg + col + 8 * sq;
              // streaming stores: each output is read once, by a later GEMM
              __stcs(reinterpret_cast<uint4*>(ep.dG + og), *reinterpret_cast<const uint4*>(buf1 + off));
              __stcs(reinterpret_cast<uint4*>(ep.dU + og),
                     *reinterpret_cast<const uint4*>(buf1 + 2048 + off));
              __stcs(reinterpret_cast<uint4*>(ep.act + row * ep.ld_act + col + 8 * sq),
                     *reinterpret_cast<const uint4*>(buf0 + off));
            }
          }
        }
      } else if constexpr (EPI == EPI_LSE_PART) {
        // the row's max and sum of exponentials over this column tile, base 2
        constexpr float kL2E = 1.4426950408889634f;
        const int jt = n0 / BN;
        const int tcol = live ? __ldg(ep.targets + m) - n0 : -1;   // target in this tile?
        float mx = -INFINITY, sm = 0.f, zt = 0.f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tbase + 32 * c, r);
          tmem_ld_wait(r);
          float cmax = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i) cmax = fmaxf(cmax, __uint_as_float(r[i]));
          const float mnew = fmaxf(mx, cmax * kL2E);
          float cs = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) cs += ex2(fmaf(__uint_as_float(r[i]), kL2E, -mnew));
          sm = sm * ex2(mx - mnew) + cs;
          mx = mnew;
          if (tcol >= 32 * c && tcol < 32 * c + 32) {
            // the target's logit, picked without indexing the register array
            // by a run-time value (which would move it to local memory)
            const int k = tcol - 32 * c;
#pragma unroll
            for (int i = 0; i < 32; ++i) zt = fmaf(i == k ? 1.f : 0.f, __uint_as_float(r[i]), zt);
          }
        }
        if (live && dbg_in2(m, g.M, jt, jt, ep.ld_part, err))
          ep.part[m * ep.ld_part + jt] = make_float2(mx, sm);
        if (live && tcol >= 0 && tcol < BN && dbg_in(m, m, g.M, err)) ep.zt[m] = zt;
      } else if constexpr (EPI == EPI_DLOGITS) {
        // dz = scale (softmax - onehot) over this column tile, bf16, leaving
        // through shared memory as whole row segments
        constexpr float kL2E = 1.4426950408889634f;
        uint8_t* buf0 = smem + Cfg::EPI_OFF + quarter * kEpiBufs * EPI_BUF_BYTES;
        const long long wrow0 = (long long)m0t + quarter * 32;   // first row of this warp
        const bool warp_live = (tc.kb1 > tc.kb0) && wrow0 < g.M;
        const int tcol = live ? __ldg(ep.targets + m) - n0 : -1;
        const float lse2 = live ? __ldg(ep.lse_rows + m) * kL2E : 0.f;
        const float sc = ep.loss_scale;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tbase + 32 * c, r);
          tmem_ld_wait(r);
          if (!warp_live) continue;   // warp-uniform
          uint4 w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t* wp = &w[q].x;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int i = 8 * q + 2 * j;
              const int col = 32 * c + i;
              const float p0 = ex2(fmaf(__uint_as_float(r[i]), kL2E, -lse2));
              const float p1 = ex2(fmaf(__uint_as_float(r[i + 1]), kL2E, -lse2));
              wp[j] = pack_bf16(sc * (p0 - (col == tcol ? 1.f : 0.f)),
                                sc * (p1 - (col + 1 == tcol ? 1.f : 0.f)));
            }
          }
          // dz (tile x vocabulary) is stored streaming, so that it does not
          // push the h tile out of L2
          warp_store_rows_bf16(buf0, lane, w, ep.dz, ep.ld_dz, wrow0, g.M, n0 + 32 * c, err);
        }
      } else if constexpr (EPI == EPI_F32) {
        // [32 rows x 32 cols] fp32 blocks of this warp's rows, 128-byte
        // swizzled in shared memory, then one TMA store / reduce-add each
        uint8_t* bufs = smem + Cfg::EPI_OFF + quarter * kEpiBufs * EPI_BUF_BYTES;
        const bool any_live = (m0t + quarter * 32 < g.M) && (tc.kb1 > tc.kb0);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c, ++epi_round) {
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          tmem_ld_wait(r);
          if (any_live) {
            uint8_t* buf = bufs + (epi_round % kEpiBufs) * EPI_BUF_BYTES;
            if (lane == 0) bulk_wait_read<kEpiBufs - 1>();  // buf's previous copy has read it
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<uint4*>(buf + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                  make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (ep.beta) tma_reduce_add_2d(&maps.c, buf, n0 + 32 * c, m0t + quarter * 32);
              else tma_store_2d(&maps.c, buf, n0 + 32 * c, m0t + quarter * 32);
              bulk_commit();
            }
          }
        }
      } else {
        // [32 rows x 32 cols] fp32 blocks of this warp's rows go through its
        // shared-memory buffer (128-byte swizzled) and are reduce-added back
        // by rows: lanes 8j..8j+7 cover one row's 128 contiguous bytes, so an
        // instruction adds 4 whole row segments instead of 16-byte pieces of
        // 32 rows.  Lane l adds column chunk q = l & 7 of rows 4k + (l >> 3).
        uint8_t* buf = smem + Cfg::EPI_OFF + quarter * kEpiBufs * EPI_BUF_BYTES;
        const int q = lane & 7;
        const int r_lane = lane >> 3;
        // the rows of this warp's 32 start at warp_row0 (tile-local row index
        // quarter * 32 within the 128-row part); with M segments the tile's
        // segment holds them all, and rows are counted within it
        const long long warp_row0 = (long long)m0t + quarter * 32;
        float* cbase;
        long long row0, row_end;   // first row of the warp, one past the last live row
        if (g.nmseg > 0) {
          const int mtile = m0t / BM;
          int s = 0;
          while (s + 1 < g.nmseg && mtile >= g.mseg_t0[s + 1]) ++s;
          cbase = ep.mseg_c[s];
          row0 = warp_row0 - (long long)g.mseg_t0[s] * BM;
          row_end = g.mseg_rows[s];
        } else {
          cbase = ep.C;
          row0 = warp_row0;
          row_end = g.M;
        }
        const bool tile_live = (tc.kb1 > tc.kb0) && row0 < row_end;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          tmem_ld_wait(r);
          if (!tile_live) continue;   // warp-uniform
          __syncwarp();               // the previous block's reads of buf are done
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4*>(buf + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rr = 4 * k + r_lane;   // row within the warp's 32
            const long long row = row0 + rr;
            if (row < row_end && dbg_in2(row, row_end, n0, n0 + BN - 1, g.N, err)) {
              const uint4 v = *reinterpret_cast<const uint4*>(buf + rr * 128 + ((q ^ (rr & 7)) << 4));
              red_add_v4_f32(cbase + row * ep.ldc + n0 + 32 * c + 4 * q, __uint_as_float(v.x),
                             __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
            }
          }
        }
      }
      }  // mt
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
    if constexpr (EPI == EPI_F32) {
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }

  // --------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (*abort_flag) {
      // make sure no MMA issued by this CTA still writes TMEM
      if (lane == 0) {
        mma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0);
      }
      __syncwarp();
    }
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host --

template <int BN, bool A_MN, bool B_MN, int EPI, int MT = 1>
static cudaError_t launch_t(const GemmMaps& maps, const GemmArgs& g, const EpiParams& ep,
                            int* err, int num_sms, cudaStream_t stream) {
  using Cfg = GemmCfg<BN, MT>;
  auto kfn = gemm_kernel<BN, A_MN, B_MN, EPI, MT>;
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t ea = smem_attr_once(kfn, (int)Cfg::SMEM_BYTES, attr_done);
  if (ea != cudaSuccess) return ea;
  if (MT > 1 && g.nmseg > 0) return cudaErrorInvalidValue;
  const int num_m = g.nmseg > 0 ? g.mseg_t0[g.nmseg] : (g.M + BM * MT - 1) / (BM * MT);
  const long long tiles = (long long)num_m * (g.N / BN) * std::max(1, g.ksplit);
  const int grid = (int)std::max(1LL, std::min<long long>(tiles, num_sms));
  kfn<<<grid, kThreads, Cfg::SMEM_BYTES, stream>>>(maps, g, ep, err);
  return cudaGetLastError();
}

cudaError_t launch_gemm(int bn, bool a_mn, bool b_mn, EpiKind epi, const CUtensorMap* amaps,
                        int na, const CUtensorMap* bmaps, int nb, const GemmArgs& g,
                        const EpiParams& ep, int* err, int num_sms, cudaStream_t stream,
                        const CUtensorMap* cmap) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  if (g.N % bn != 0) return cudaErrorInvalidValue;
  if (na < 1 || na > kMaxASegs || nb < 1 || nb > kMaxBMaps) return cudaErrorInvalidValue;
  if (epi == EPI_F32 && !cmap) return cudaErrorInvalidValue;
  if (g.nkseg < 0 || g.nkseg > kMaxASegs) return cudaErrorInvalidValue;
  if (g.nmseg < 0 || g.nmseg > kMaxASegs || (g.nmseg > 0 && epi != EPI_F32_ATOMIC))
    return cudaErrorInvalidValue;
  for (int s = 0; s < g.nmseg; ++s)
    if (g.mseg_a[s] < 0 || g.mseg_a[s] >= na || g.mseg_t0[s + 1] <= g.mseg_t0[s] ||
        g.mseg_rows[s] <= 0 || g.mseg_rows[s] > (g.mseg_t0[s + 1] - g.mseg_t0[s]) * BM ||
        !ep.mseg_c[s])
      return cudaErrorInvalidValue;
  for (int s = 0; s < g.nkseg; ++s)
    if (g.kseg_a[s] < 0 || g.kseg_a[s] >= na || g.kseg_b[s] < 0 || g.kseg_b[s] >= nb ||
        g.kseg_end[s] <= (s ? g.kseg_end[s - 1] : 0))
      return cudaErrorInvalidValue;
  GemmMaps maps;
  for (int i = 0; i < kMaxASegs; ++i) maps.a[i] = amaps[i < na ? i : 0];
  for (int i = 0; i < kMaxBMaps; ++i) maps.b[i] = bmaps[i < nb ? i : 0];
  maps.c = cmap ? *cmap : bmaps[0];
#define UPIPE_GEMM_CASE(BN_, AMN, BMN, E)                                              \
  if (bn == BN_ && a_mn == AMN && b_mn == BMN && epi == E)                             \
    return launch_t<BN_, AMN, BMN, E>(maps, g, ep, err, num_sms, stream);
  // projections (one head per tile: BN = d; at d = 128 each tile holds 256
  // rows in two accumulators that share the weight tile)
  UPIPE_GEMM_CASE(64, false, false, EPI_PROJ)
  if (bn == 128 && !a_mn && !b_mn && epi == EPI_PROJ)
    return launch_t<128, false, false, EPI_PROJ, 2>(maps, g, ep, err, num_sms, stream);
  // Wo-slice accumulate
  UPIPE_GEMM_CASE(128, false, false, EPI_F32)
  UPIPE_GEMM_CASE(256, false, false, EPI_F32)
  // dO = dOut Wo_c (+ D); at d = 128 also 256 rows per tile
  UPIPE_GEMM_CASE(64, false, true, EPI_DO)
  if (bn == 128 && !a_mn && b_mn && epi == EPI_DO)
    return launch_t<128, false, true, EPI_DO, 2>(maps, g, ep, err, num_sms, stream);
  // dX += dQKV W
  UPIPE_GEMM_CASE(128, false, true, EPI_F32)
  UPIPE_GEMM_CASE(256, false, true, EPI_F32)
  // weight gradients (K = S, split)
  UPIPE_GEMM_CASE(256, true, true, EPI_F32_ATOMIC)
  UPIPE_GEMM_CASE(128, true, true, EPI_F32_ATOMIC)
  UPIPE_GEMM_CASE(64, true, true, EPI_F32_ATOMIC)
  // the sequence-tiled MLP's gate/up projections (two B maps)
  if ((epi == EPI_SWIGLU || epi == EPI_SWIGLU_BWD) && (bn != 256 || a_mn || b_mn || nb < 2))
    return cudaErrorInvalidValue;
  UPIPE_GEMM_CASE(256, false, false, EPI_SWIGLU)
  UPIPE_GEMM_CASE(256, false, false, EPI_SWIGLU_BWD)
  // the sequence-tiled loss's logits (vocabulary tiles of 256 or 128)
  UPIPE_GEMM_CASE(256, false, false, EPI_LSE_PART)
  UPIPE_GEMM_CASE(128, false, false, EPI_LSE_PART)
  UPIPE_GEMM_CASE(256, false, false, EPI_DLOGITS)
  UPIPE_GEMM_CASE(128, false, false, EPI_DLOGITS)
#undef UPIPE_GEMM_CASE
  return cudaErrorNotSupported;
}

}  // namespace upipe

extern "C" int upipe_gemm_tile_order(int num_m, int num_n, int kb_total, int ksplit,
                                     int m_fastest, int32_t* out, int64_t out_len) {
  if (num_m < 1 || num_n < 1 || kb_total < 1 || ksplit < 1 || m_fastest < 0 || !out)
    return UPIPE_ERR_INVALID_ARG;
  const long long tiles = (long long)num_m * num_n * ksplit;
  // the walk forms m_fastest * num_n in int
  if (tiles > INT32_MAX || (long long)m_fastest * num_n > INT32_MAX || out_len < 4 * tiles)
    return UPIPE_ERR_INVALID_ARG;
  for (int t = 0; t < (int)tiles; ++t) {
    const upipe::TileCoord c = upipe::tile_coord(t, num_m, num_n, kb_total, ksplit, 1, m_fastest);
    out[4 * t] = c.m0;
    out[4 * t + 1] = c.n0;
    out[4 * t + 2] = c.kb0;
    out[4 * t + 3] = c.kb1;
  }
  return UPIPE_OK;
}
