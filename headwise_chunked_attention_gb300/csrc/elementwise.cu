// HBM-bound elementwise kernels around the attention layer:
//   * the RoPE angle table (built in float64, stored as fp32 cos/sin pairs);
//   * the backward of the q/k post-processing: RoPE transpose, then (Qwen3
//     geometry) the RMSNorm backward with its gain gradient;
//   * fp32 -> bf16 hi/lo split of an accumulated gradient.
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
                                  double theta) {
  const long long total = (nhi + 1024) * half;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long row = t / half;
    const int i = (int)(t - row * half);
    const double w = pow(theta, -2.0 * i / (2.0 * half));
    double ang;
    float2* dst;
    if (row < nhi) {
      ang = (double)(row * 1024) * w;
      dst = hi + row * half + i;
    } else {
      ang = (double)(row - nhi) * w;
      dst = lo + (row - nhi) * half + i;
    }
    double s, c;
    sincos(ang, &s, &c);
    *dst = make_float2((float)c, (float)s);
    if (row >= nhi) lo_t[(long long)i * 1024 + (row - nhi)] = make_float2((float)c, (float)s);
  }
}

cudaError_t launch_rope_table(float2* hi, float2* lo, float2* lo_t, long long S, int d,
                              double theta, cudaStream_t stream) {
  const long long nhi = (S >> 10) + 1;
  const long long total = (nhi + 1024) * (d / 2);
  const int threads = 256;
  const int blocks = (int)std::min<long long>((total + threads - 1) / threads, 4096);
  rope_table_kernel<<<blocks, threads, 0, stream>>>(hi, lo, lo_t, nhi, d / 2, theta);
  return cudaGetLastError();
}

// ------------------------------------------------------ q/k post backward --
// One warp per (row, head).  Lane l owns elements l + 32k, k < D/32, which
// holds each RoPE pair (i, i + D/2) inside one lane.
//   dy = R^T g                       (RoPE transpose)
//   norm mode, with yhat = a / r saved by the forward projection:
//     dgamma += dy * yhat;  dyhat = dy * gamma;
//     da = (dyhat - yhat * mean(dyhat * yhat)) * rstd
template <int D>
__global__ void __launch_bounds__(256) qk_bwd_kernel(const QkBwdArgs a) {
  constexpr int E = D / 32;
  constexpr int H = D / 2;
  __shared__ float sg[D];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const bool norm = a.mode == PROJ_NORM_ROPE;
  if (norm)
    for (int i = threadIdx.x; i < D; i += blockDim.x) sg[i] = 0.f;
  __syncthreads();
  float gam[E], dgam[E];
#pragma unroll
  for (int k = 0; k < E; ++k) {
    gam[k] = (norm && a.gamma) ? a.gamma[lane + 32 * k] : 1.f;
    dgam[k] = 0.f;
  }
  const long long items = a.S * a.heads;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long it = blockIdx.x * (long long)(blockDim.x >> 5) + wib; it < items; it += warps) {
    const long long s = it / a.heads;
    const int h = (int)(it - s * a.heads);
    const float* gp = a.g + s * a.ld_g + h * D;
    float g[E], dy[E];
#pragma unroll
    for (int k = 0; k < E; ++k) g[k] = gp[lane + 32 * k];
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
      const int i = lane + 32 * k;  // first half index, partner i + H
      const float2 lo = __ldg(a.rope_lo + (s & 1023) * H + i);
      const float2 hi = __ldg(a.rope_hi + (s >> 10) * H + i);
      const float c = hi.x * lo.x - hi.y * lo.y;
      const float sn = hi.y * lo.x + hi.x * lo.y;
      const float ga = g[k], gb = g[k + E / 2];
      dy[k] = ga * c + gb * sn;
      dy[k + E / 2] = gb * c - ga * sn;
    }
    bf16* op = a.out + s * a.ld_out + h * D;
    bf16* lp = a.out_lo + s * a.ld_out + h * D;
    if (norm) {
      const float* yp = a.yhat + s * a.ld_yhat + h * D;
      const float rs = a.rstd[(long long)h * a.S + s];
      float yh[E], dot = 0.f;
#pragma unroll
      for (int k = 0; k < E; ++k) {
        yh[k] = yp[lane + 32 * k];
        dgam[k] = fmaf(dy[k], yh[k], dgam[k]);
        dot = fmaf(dy[k] * gam[k], yh[k], dot);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      const float mean = dot * (1.0f / D);
#pragma unroll
      for (int k = 0; k < E; ++k) dy[k] = (dy[k] * gam[k] - yh[k] * mean) * rs;
    }
#pragma unroll
    for (int k = 0; k < E; ++k) {
      const bf16 hi = __float2bfloat16(dy[k]);
      op[lane + 32 * k] = hi;
      lp[lane + 32 * k] = __float2bfloat16(dy[k] - __bfloat162float(hi));
    }
  }
  if (norm && a.dgamma) {
#pragma unroll
    for (int k = 0; k < E; ++k) atomicAdd(&sg[lane + 32 * k], dgam[k]);
    __syncthreads();
    for (int i = threadIdx.x; i < D; i += blockDim.x) atomicAdd(a.dgamma + i, sg[i]);
  }
}

cudaError_t launch_qk_bwd(const QkBwdArgs& a, cudaStream_t stream) {
  if (a.S <= 0 || a.heads <= 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long items = a.S * a.heads;
  const int blocks = (int)std::min<long long>((items + 7) / 8, (long long)sms * 8);
  if (a.d == 128) qk_bwd_kernel<128><<<blocks, 256, 0, stream>>>(a);
  else if (a.d == 64) qk_bwd_kernel<64><<<blocks, 256, 0, stream>>>(a);
  else return cudaErrorNotSupported;
  return cudaGetLastError();
}

// ---------------------------------------------------------- fp32->bf16x2 --
__global__ void f32_to_bf16x2_kernel(const float* __restrict__ in, int ld_in,
                                     bf16* __restrict__ hi, bf16* __restrict__ lo, int ld_out,
                                     long long S, int cols4) {
  const long long total = S * cols4;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long r = t / cols4;
    const int c = (int)(t - r * cols4) * 4;
    const float4 v = *reinterpret_cast<const float4*>(in + r * ld_in + c);
    uint2 wh, wl;
    wh.x = pack_bf16(v.x, v.y);
    wh.y = pack_bf16(v.z, v.w);
    const float2 h0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wh.x));
    const float2 h1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wh.y));
    wl.x = pack_bf16(v.x - h0.x, v.y - h0.y);
    wl.y = pack_bf16(v.z - h1.x, v.w - h1.y);
    *reinterpret_cast<uint2*>(hi + r * ld_out + c) = wh;
    *reinterpret_cast<uint2*>(lo + r * ld_out + c) = wl;
  }
}

cudaError_t launch_f32_to_bf16x2(const float* in, int ld_in, bf16* hi, bf16* lo, int ld_out,
                                 long long S, int cols, cudaStream_t stream) {
  if (S <= 0 || cols <= 0) return cudaSuccess;
  const long long total = S * (cols / 4);
  const int blocks = (int)std::min<long long>((total + 255) / 256, 152 * 16);
  f32_to_bf16x2_kernel<<<blocks, 256, 0, stream>>>(in, ld_in, hi, lo, ld_out, S, cols / 4);
  return cudaGetLastError();
}

}  // namespace upipe
