// HBM-bound elementwise kernels around the attention layer:
//   * the RoPE angle table (built in float64, stored as fp32 cos/sin pairs);
//   * the backward of the q/k post-processing: RoPE transpose, then (Qwen3
//     geometry) the RMSNorm backward with its gain gradient;
//   * fp32 -> bf16 hi/lo split of an accumulated gradient;
//   * the norm bounds behind the backward's fp16 gradient scale.
// Gradients leave these kernels as two bf16 tensors, hi = bf16(v) and
// lo = bf16(v - hi), which the dX / dW GEMMs consume as two bf16 operands: the
// tensor cores then see ~16 significant bits of the fp32 gradient instead of 8.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace upipe {

// ------------------------------------------------------------ RoPE table --
// RoPE rotates the pair (i, i + d/2) by pos * w_i, w_i = theta^(-2i/d).  At
// positions up to millions a float32 angle pos * w_i has an ulp near 0.5 rad,
// so the angle is split: pos = hi + lo with hi = pos & ~1023, lo = pos & 1023;
// hi[b][i] = (cos, sin)(b * 1024 * w_i), lo[p][i] = (cos, sin)(p * w_i), both
// evaluated in float64 and rounded once; the consumer combines them with one
// complex multiplication (error ~1e-7).  lo is also written transposed,
// lo_t[i][p], for consumers whose threads walk positions (one row each).
__global__ void rope_table_kernel(float2* __restrict__ hi, float2* __restrict__ lo,
                                  float2* __restrict__ lo_t, long long nhi, int half,
                                  double theta, int* __restrict__ err) {
  const long long total = (nhi + 1024) * half;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long row = t / half;
    const int i = (int)(t - row * half);
    const double w = pow(theta, -2.0 * i / (2.0 * half));
    double ang;
    float2* dst;
    bool ok;
    if (row < nhi) {
      ang = (double)(row * 1024) * w;
      dst = hi + row * half + i;
      ok = dbg_in2(row, nhi, i, i, half, err);
    } else {
      ang = (double)(row - nhi) * w;
      dst = lo + (row - nhi) * half + i;
      ok = dbg_in2(row - nhi, 1024, i, i, half, err);
    }
    double s, c;
    sincos(ang, &s, &c);
    if (ok) *dst = make_float2((float)c, (float)s);
    if (row >= nhi && dbg_in2(i, half, row - nhi, row - nhi, 1024, err))
      lo_t[(long long)i * 1024 + (row - nhi)] = make_float2((float)c, (float)s);
  }
}

cudaError_t launch_rope_table(float2* hi, float2* lo, float2* lo_t, long long S, int d,
                              double theta, cudaStream_t stream, int* err) {
  const long long nhi = (S >> 10) + 1;
  const long long total = (nhi + 1024) * (d / 2);
  const int threads = 256;
  const int blocks = (int)std::min<long long>((total + threads - 1) / threads, 4096);
  rope_table_kernel<<<blocks, threads, 0, stream>>>(hi, lo, lo_t, nhi, d / 2, theta, err);
  return cudaGetLastError();
}

// ------------------------------------------------------ q/k post backward --
// D/8 lanes per (row, head) item, so a warp takes 32 / (D/8) items per pass.
// Lane j of an item owns elements 4j..4j+3 and their RoPE partners
// H+4j..H+4j+3 (H = D/2): every pair (i, i + H) stays inside one lane and each
// access is one 16-byte load (fp32) or 8-byte store (bf16).
//   dy = R^T g                       (RoPE transpose)
//   norm mode, with yhat = a / r saved by the forward projection:
//     dgamma += dy * yhat;  dyhat = dy * gamma;
//     da = (dyhat - yhat * mean(dyhat * yhat)) * rstd
template <int D, bool NORM>
__global__ void __launch_bounds__(256) qk_bwd_kernel(const QkBwdArgs a) {
  constexpr int H = D / 2;
  int* err = a.err;
  constexpr int LPR = D / 8;      // lanes per item
  constexpr int IPW = 32 / LPR;   // items per warp pass
  __shared__ float sg[D];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int j = lane % LPR;
  const int sub = lane / LPR;
  constexpr bool norm = NORM;
  if constexpr (norm) {
    for (int i = threadIdx.x; i < D; i += blockDim.x) sg[i] = 0.f;
    __syncthreads();
  }
  // element k < 4 is column 4j + k, element 4 + k is column H + 4j + k
  float gam[8], dgam[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    gam[k] = (norm && a.gamma) ? a.gamma[4 * j + k] : 1.f;
    gam[4 + k] = (norm && a.gamma) ? a.gamma[H + 4 * j + k] : 1.f;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) dgam[k] = 0.f;
  const long long items = a.S * a.heads;
  const long long step = (long long)gridDim.x * (blockDim.x >> 5) * IPW;
  for (long long base = ((long long)blockIdx.x * (blockDim.x >> 5) + wib) * IPW; base < items;
       base += step) {
    // every lane runs the body (the norm mode reduces across the item's
    // lanes); an item past the end recomputes the last one and stores nothing
    const long long it0 = base + sub;
    const bool live = it0 < items;
    const long long it = live ? it0 : items - 1;
    const long long s0 = it / a.heads;
    const int h0 = (int)(it - s0 * a.heads);
    // this lane's columns of row s: [h D + 4j, h D + 4j + 3] and the same + H
    // in g, yhat and the outputs; entries [4j, 4j + 3] (float2) of rows
    // s & 1023 and s >> 10 of the RoPE tables.
    // A failed check (debug builds) reads item 0 instead and stores nothing;
    // every lane still runs the body for the shuffles below.
    const bool in_ok = dbg_in2(s0, a.S, h0 * D + 4 * j, h0 * D + H + 4 * j + 3, a.ld_g, err) &&
                       dbg_in2(s0 & 1023, 1024, 4 * j, 4 * j + 3, H, err) &&
                       dbg_in2(s0 >> 10, (a.S >> 10) + 1, 4 * j, 4 * j + 3, H, err) &&
                       (!norm || (dbg_in2(s0, a.S, h0 * D + 4 * j, h0 * D + H + 4 * j + 3,
                                          a.ld_yhat, err) &&
                                  dbg_in2(h0, a.heads, s0, s0, a.S, err)));
    const long long s = in_ok ? s0 : 0;
    const int h = in_ok ? h0 : 0;
    const float* gp = a.g + s * a.ld_g + h * D + 4 * j;
    const float4 ga4 = *reinterpret_cast<const float4*>(gp);
    const float4 gb4 = *reinterpret_cast<const float4*>(gp + H);
    const float4* lo4 = reinterpret_cast<const float4*>(a.rope_lo + (s & 1023) * H + 4 * j);
    const float4* hi4 = reinterpret_cast<const float4*>(a.rope_hi + (s >> 10) * H + 4 * j);
    const float4 l01 = __ldg(lo4), l23 = __ldg(lo4 + 1);
    const float4 h01 = __ldg(hi4), h23 = __ldg(hi4 + 1);
    const float lc[4] = {l01.x, l01.z, l23.x, l23.z}, ls[4] = {l01.y, l01.w, l23.y, l23.w};
    const float hc[4] = {h01.x, h01.z, h23.x, h23.z}, hs[4] = {h01.y, h01.w, h23.y, h23.w};
    const float ga[4] = {ga4.x, ga4.y, ga4.z, ga4.w}, gb[4] = {gb4.x, gb4.y, gb4.z, gb4.w};
    float dy[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float c = hc[k] * lc[k] - hs[k] * ls[k];
      const float sn = hs[k] * lc[k] + hc[k] * ls[k];
      dy[k] = ga[k] * c + gb[k] * sn;
      dy[4 + k] = gb[k] * c - ga[k] * sn;
    }
    if constexpr (norm) {
      const float* yp = a.yhat + s * a.ld_yhat + h * D + 4 * j;
      const float4 ya4 = *reinterpret_cast<const float4*>(yp);
      const float4 yb4 = *reinterpret_cast<const float4*>(yp + H);
      const float yh[8] = {ya4.x, ya4.y, ya4.z, ya4.w, yb4.x, yb4.y, yb4.z, yb4.w};
      const float rs = a.rstd[(long long)h * a.S + s];
      float dot = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (live) dgam[k] = fmaf(dy[k], yh[k], dgam[k]);
        dot = fmaf(dy[k] * gam[k], yh[k], dot);
      }
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      const float mean = dot * (1.0f / D);
#pragma unroll
      for (int k = 0; k < 8; ++k) dy[k] = (dy[k] * gam[k] - yh[k] * mean) * rs;
    }
    if (live && in_ok && dbg_in2(s, a.S, h * D + 4 * j, h * D + H + 4 * j + 3, a.ld_out, err)) {
      const long long o = s * a.ld_out + h * D + 4 * j;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float* v = dy + 4 * half;
        uint2 wh, wl;
        wh.x = pack_bf16(v[0], v[1]);
        wh.y = pack_bf16(v[2], v[3]);
        const float2 h0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wh.x));
        const float2 h1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wh.y));
        wl.x = pack_bf16(v[0] - h0.x, v[1] - h0.y);
        wl.y = pack_bf16(v[2] - h1.x, v[3] - h1.y);
        *reinterpret_cast<uint2*>(a.out + o + half * H) = wh;
        *reinterpret_cast<uint2*>(a.out_lo + o + half * H) = wl;
      }
    }
  }
  if constexpr (norm) {
    if (!a.dgamma) return;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      atomicAdd(&sg[4 * j + k], dgam[k]);
      atomicAdd(&sg[H + 4 * j + k], dgam[4 + k]);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < D; i += blockDim.x) atomicAdd(a.dgamma + i, sg[i]);
  }
}

cudaError_t launch_qk_bwd(const QkBwdArgs& a, cudaStream_t stream) {
  if (a.S <= 0 || a.heads <= 0) return cudaSuccess;
  if (a.d != 128 && a.d != 64) return cudaErrorNotSupported;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long items = a.S * a.heads;
  const long long per_block = 8LL * (32 / (a.d / 8));   // 8 warps, 32 / (d/8) items each
  const int blocks =
      (int)std::min<long long>((items + per_block - 1) / per_block, (long long)sms * 8);
  const bool norm = a.mode == PROJ_NORM_ROPE;
  if (a.d == 128 && norm) qk_bwd_kernel<128, true><<<blocks, 256, 0, stream>>>(a);
  else if (a.d == 128) qk_bwd_kernel<128, false><<<blocks, 256, 0, stream>>>(a);
  else if (norm) qk_bwd_kernel<64, true><<<blocks, 256, 0, stream>>>(a);
  else qk_bwd_kernel<64, false><<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------- fp32->bf16x2 --
// Each thread converts float4 groups t and t + stride per pass: both loads
// are issued before either result is stored.
__device__ __forceinline__ void split_store(const float4 v, bf16* hi, bf16* lo) {
  uint2 wh, wl;
  wh.x = pack_bf16(v.x, v.y);
  wh.y = pack_bf16(v.z, v.w);
  const float2 h0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wh.x));
  const float2 h1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wh.y));
  wl.x = pack_bf16(v.x - h0.x, v.y - h0.y);
  wl.y = pack_bf16(v.z - h1.x, v.w - h1.y);
  *reinterpret_cast<uint2*>(hi) = wh;
  *reinterpret_cast<uint2*>(lo) = wl;
}

__global__ void f32_to_bf16x2_kernel(const float* __restrict__ in, int ld_in,
                                     bf16* __restrict__ hi, bf16* __restrict__ lo, int ld_out,
                                     long long S, int cols4, int* __restrict__ err) {
  const long long total = S * cols4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += 2 * stride) {
    const long long t2 = t + stride;
    const long long r = t / cols4;
    const int c = (int)(t - r * cols4) * 4;
    const bool ok = dbg_in2(r, S, c, c + 3, ld_in, err) && dbg_in2(r, S, c, c + 3, ld_out, err);
    const float4 v = ok ? *reinterpret_cast<const float4*>(in + r * ld_in + c)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    long long r2 = 0;
    int c2 = 0;
    float4 v2 = make_float4(0.f, 0.f, 0.f, 0.f);
    bool ok2 = false;
    if (t2 < total) {
      r2 = t2 / cols4;
      c2 = (int)(t2 - r2 * cols4) * 4;
      ok2 = dbg_in2(r2, S, c2, c2 + 3, ld_in, err) && dbg_in2(r2, S, c2, c2 + 3, ld_out, err);
      if (ok2) v2 = *reinterpret_cast<const float4*>(in + r2 * ld_in + c2);
    }
    if (ok) split_store(v, hi + r * ld_out + c, lo + r * ld_out + c);
    if (ok2) split_store(v2, hi + r2 * ld_out + c2, lo + r2 * ld_out + c2);
  }
}

cudaError_t launch_f32_to_bf16x2(const float* in, int ld_in, bf16* hi, bf16* lo, int ld_out,
                                 long long S, int cols, cudaStream_t stream, int* err) {
  if (S <= 0 || cols <= 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long total = S * (cols / 4);
  const int blocks = (int)std::min<long long>((total + 511) / 512, (long long)sms * 8);
  f32_to_bf16x2_kernel<<<blocks, 256, 0, stream>>>(in, ld_in, hi, lo, ld_out, S, cols / 4, err);
  return cudaGetLastError();
}

// ------------------------------------------------------- gradient bounds --
// The backward's fp16 scale of dO (internal.h, "backward fp16 scales") needs
// max_i ||dout_i||_2 and max_j ||Wo[:, j]||_2.  Blocks [0, row_blocks) take
// dout rows, one warp per row with 16-byte loads (hidden is a multiple of
// 128); each later block takes 32 columns of Wo with 8 warps over its rows
// (consecutive columns per warp: coalesced), then reduces the 8 partial sums.
__global__ void __launch_bounds__(256)
    grad_bound_kernel(const bf16* __restrict__ dout, long long S, int hidden,
                      const bf16* __restrict__ Wo, int ncols, int row_blocks,
                      float* __restrict__ bound, int* __restrict__ err) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if ((int)blockIdx.x < row_blocks) {
    float mx = 0.f;
    for (long long r = (long long)blockIdx.x * 8 + warp; r < S; r += (long long)row_blocks * 8) {
      const bf16* row = dout + r * hidden;
      float ss = 0.f;
      for (int c = lane * 8; c < hidden; c += 256) {
        if (!dbg_in2(r, S, c, c + 7, hidden, err)) continue;
        const uint4 v = *reinterpret_cast<const uint4*>(row + c);
        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(p2[k]);
          ss = fmaf(f.x, f.x, ss);
          ss = fmaf(f.y, f.y, ss);
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      mx = fmaxf(mx, ss);
    }
    if (lane == 0) atomic_max_nonneg(bound, sqrtf(mx));
  } else {
    __shared__ float part[8][32];
    const int col = ((int)blockIdx.x - row_blocks) * 32 + lane;
    float ss = 0.f;
    if (col < ncols)
      for (int r = warp; r < hidden; r += 8) {
        if (!dbg_in2(r, hidden, col, col, ncols, err)) continue;
        const float v = __bfloat162float(Wo[(long long)r * ncols + col]);
        ss = fmaf(v, v, ss);
      }
    part[warp][lane] = ss;
    __syncthreads();
    if (warp == 0) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) t += part[w][lane];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, off));
      if (lane == 0) atomic_max_nonneg(bound + 1, sqrtf(t));
    }
  }
}

cudaError_t launch_grad_bound(const bf16* dout, long long S, int hidden, const bf16* Wo,
                              int ncols, float* bound, cudaStream_t stream, int* err) {
  if (S <= 0 || hidden <= 0 || ncols <= 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int row_blocks = (int)std::min<long long>((S + 7) / 8, (long long)sms * 8);
  const int col_blocks = (ncols + 31) / 32;
  grad_bound_kernel<<<row_blocks + col_blocks, 256, 0, stream>>>(dout, S, hidden, Wo, ncols,
                                                                 row_blocks, bound, err);
  return cudaGetLastError();
}

// ------------------------------------------------------ tiled loss rows --
// The sequence-tiled loss: each row's log-sum-exp over the vocabulary from
// the (max, sum of exp) partials of its column tiles (base 2, written by the
// logits GEMM's epilogue), and the row's loss lse - z[target].  One warp per
// row; lane l combines tiles l, l + 32, ...; a target outside [0, vocab)
// gives a NaN loss and UPIPE_ERR_TARGET.
__global__ void __launch_bounds__(256)
    loss_rows_kernel(const float2* __restrict__ part, int ntiles, const float* __restrict__ zt,
                     const int* __restrict__ targets, int vocab, long long rows,
                     float* __restrict__ lse, float* __restrict__ loss, int* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;   // warp-uniform
  float mx = -INFINITY;
  for (int j = lane; j < ntiles; j += 32)
    if (dbg_in2(row, rows, j, j, ntiles, err)) mx = fmaxf(mx, part[row * ntiles + j].x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float sm = 0.f;
  for (int j = lane; j < ntiles; j += 32) {
    if (!dbg_in2(row, rows, j, j, ntiles, err)) continue;
    const float2 p = part[row * ntiles + j];
    sm += p.y * exp2f(p.x - mx);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off);
  if (lane == 0) {
    const float l = (mx + log2f(sm)) * 0.69314718055994531f;
    const int t = targets[row];
    lse[row] = l;
    if (t < 0 || t >= vocab) {
      loss[row] = __int_as_float(0x7fc00000);   // NaN
      atomicCAS(err, 0, kErrTarget);
    } else {
      loss[row] = l - zt[row];
    }
  }
}

cudaError_t launch_loss_rows(const float2* part, int ntiles, const float* zt, const int* targets,
                             int vocab, long long rows, float* lse, float* loss,
                             cudaStream_t stream, int* err) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;
  loss_rows_kernel<<<(unsigned)blocks, 256, 0, stream>>>(part, ntiles, zt, targets, vocab, rows,
                                                          lse, loss, err);
  return cudaGetLastError();
}

}  // namespace upipe
