// Kernels of the flash_block wrapper around the layer ("Transformer Quality
// in Linear Time", flash_block pseudocode: pre-norm, RoPE on the four heads,
// residual): the pre-norm of X into the workspace region xn, for both io
// types, and for fp32 the RoPE rotation of the heads in place (the bf16
// projection rotates them in its epilogue, the output epilogues add the
// residual).
#include <cuda_bf16.h>

#include "flash_gau_internal.h"
#include "sm103_ptx.cuh"

namespace flashgau {
namespace {

using ptx::griddep_launch_dependents;
using ptx::griddep_wait;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per row of X: LayerNorm ((x - mean) / sqrt(var + eps) * g + b,
// biased variance) or ScaleNorm (g * x / max(||x||, eps)), fp32 statistics
// from two passes over the row (the second reads it from L1).
template <typename T>
__global__ void __launch_bounds__(256) norm_rows(const T *__restrict__ X, T *__restrict__ xn,
                                                 long long M, int d, int kind,
                                                 const float *__restrict__ g,
                                                 const float *__restrict__ b, float eps) {
  // xn was read by the previous forward's projection, which has completed
  // once this wait returns
  griddep_wait();
  griddep_launch_dependents();
  const long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const T *x = X + row * d;
  T *y = xn + row * d;
  float mean = 0.f;
  if (kind == FLASH_GAU_NORM_LAYER) {
    float s1 = 0.f;
    for (int k = lane; k < d; k += 32) s1 += to_f(x[k]);
    mean = warp_sum(s1) / (float)d;
  }
  float s2 = 0.f;
  for (int k = lane; k < d; k += 32) {
    const float v = to_f(x[k]) - mean;
    s2 += v * v;
  }
  s2 = warp_sum(s2);
  const float scale = kind == FLASH_GAU_NORM_LAYER ? 1.0f / sqrtf(s2 / (float)d + eps)
                                                   : g[0] / fmaxf(sqrtf(s2), eps);
  for (int k = lane; k < d; k += 32) {
    float v = (to_f(x[k]) - mean) * scale;
    if (kind == FLASH_GAU_NORM_LAYER) v = fmaf(v, g[k], b ? b[k] : 0.f);
    y[k] = from_f<T>(v);
  }
}

// fp32 heads [4][M][s] rotated in place: thread = (head, token, pair).
__global__ void __launch_bounds__(256) rope_heads_f32(float *__restrict__ heads, long long M,
                                                      int T, int s, double log2_base,
                                                      int pos_offset) {
  const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const int half = s / 2;
  if (idx >= 4 * M * half) return;
  const int i = (int)(idx % half);
  const long long hm = idx / half;  // h * M + m
  const long long m = hm % M;
  float cs, sn;
  rope_sincos((double)(m % T + pos_offset), i, s, log2_base, &sn, &cs);
  float *h = heads + hm * s + 2 * i;
  const float x0 = h[0], x1 = h[1];
  h[0] = x0 * cs - x1 * sn;
  h[1] = x0 * sn + x1 * cs;
}

inline unsigned cdiv(long long a, long long b) { return (unsigned)((a + b - 1) / b); }

}  // namespace

cudaError_t block_norm(const Problem &p) {
  const unsigned grid = cdiv(p.M * 32, 256);
  if (p.dtype == FLASH_GAU_BF16)
    return launch_pdl(norm_rows<__nv_bfloat16>, dim3(grid), dim3(256), 0, p.stream,
                      (const __nv_bfloat16 *)p.X, (__nv_bfloat16 *)p.xn, p.M, p.d, p.norm,
                      p.norm_g, p.norm_b, p.norm_eps);
  return launch_pdl(norm_rows<float>, dim3(grid), dim3(256), 0, p.stream, (const float *)p.X,
                    (float *)p.xn, p.M, p.d, p.norm, p.norm_g, p.norm_b, p.norm_eps);
}

cudaError_t simt_rope_heads_f32(const Problem &p) {
  rope_heads_f32<<<cdiv(4 * p.M * (p.s / 2), 256), 256, 0, p.stream>>>(
      (float *)p.heads, p.M, p.T, p.s, log2((double)p.rope_base), p.pos_offset);
  return cudaGetLastError();
}

}  // namespace flashgau
