// Kernels of the flash_block wrapper around the layer ("Transformer Quality
// in Linear Time", flash_block pseudocode: pre-norm, RoPE on the four heads,
// residual): the pre-norm of X into the workspace region xn, for both io
// types, and for fp32 the RoPE rotation of the heads in place (the bf16
// projection rotates them in its epilogue, the output epilogues add the
// residual).  Also the RoPE construction of the relative position bias for
// long windows (appendix D, Code 4): the table of the layer's bias from two
// learned vectors.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

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

// cos / sin of every (pair, position): the table the bf16 projection's heads
// epilogue reads, [s / 2][T] half2 (cos, sin), pair-major so that a warp's 32
// consecutive positions of one pair are one coalesced load (fp16 keeps them
// to 2^-11, well below the bf16 rounding of the heads).  Block `blk` of
// the job fills entries blk * blockDim.x + threadIdx.x.
struct RopeJob {
  __half2 *tab;  // null: no table
  int T, s, pos_offset;
  RopeTable phi;
};
__device__ __forceinline__ void rope_table_part(const RopeJob &r, unsigned blk) {
  if (!r.tab) return;
  const long long idx = (long long)blk * blockDim.x + threadIdx.x;
  if (idx >= (long long)r.T * (r.s / 2)) return;
  const int t = (int)(idx % r.T);
  const int i = (int)(idx / r.T);
  float sn, cs;
  rope_sincos((float)(t + r.pos_offset), r.phi.phi[i], &sn, &cs);
  r.tab[idx] = __floats2half2_rn(cs, sn);
}

__global__ void __launch_bounds__(256) rope_table_kernel(const RopeJob r) {
  griddep_wait();  // the previous forward's projection has read the table
  rope_table_part(r, blockIdx.x);
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
  // once this wait returns.  No early trigger: the projection's CTAs would
  // take the SMs and wait there while the rows still need them.
  griddep_wait();
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

// bf16 rows with d % 8 == 0 and d <= 32 * 8 * NV: one warp per row, the row
// read once into registers as 16-byte vectors, kept packed (lane l holds
// elements 256 k + 8 l .. +7, k < NV) and unpacked in each pass, so that
// registers stay few and many rows are in flight per SM; 16-byte stores.
// NV is the smallest that holds the row.  Blocks past the rows compute the
// RoPE table when the block needs one (rope_table), in the same launch.
constexpr int kNormVec = 16;
template <int NV>
__global__ void __launch_bounds__(256) norm_rows_bf16x8(const uint4 *__restrict__ X,
                                                        uint4 *__restrict__ xn, long long M,
                                                        int d, int kind,
                                                        const float *__restrict__ g,
                                                        const float *__restrict__ b, float eps,
                                                        RopeJob rope) {
  griddep_wait();  // as norm_rows
  const long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= M) {
    rope_table_part(rope, blockIdx.x - (unsigned)((M * 32 + blockDim.x - 1) / blockDim.x));
    return;
  }
  const int d8 = d / 8;  // 16-byte vectors per row
  const uint4 *x = X + row * d8;
  uint4 *y = xn + row * d8;
  uint4 raw[NV];
  auto val = [&](int k, int q) {  // element 8 (32 k + lane) + q, as float
    const __nv_bfloat162 h = reinterpret_cast<const __nv_bfloat162 *>(&raw[k])[q >> 1];
    return (q & 1) ? __high2float(h) : __low2float(h);
  };
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int j = k * 32 + lane;  // vector index
    raw[k] = j < d8 ? __ldg(x + j) : make_uint4(0, 0, 0, 0);
  }
  float s1 = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int q = 0; q < 8; ++q) s1 += val(k, q);  // zeros past the row
  const float mean = kind == FLASH_GAU_NORM_LAYER ? warp_sum(s1) / (float)d : 0.f;
  float s2 = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (k * 32 + lane < d8)
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float c = val(k, q) - mean;
        s2 += c * c;
      }
  s2 = warp_sum(s2);
  const float scale = kind == FLASH_GAU_NORM_LAYER ? 1.0f / sqrtf(s2 / (float)d + eps)
                                                   : g[0] / fmaxf(sqrtf(s2), eps);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int j = k * 32 + lane;
    if (j < d8) {
      // the scale and shift of this lane's 8 columns, as two float4 each
      float gv[8], bv[8];
      if (kind == FLASH_GAU_NORM_LAYER) {
        const float4 *g4 = reinterpret_cast<const float4 *>(g) + 2 * j;
        const float4 g0 = __ldg(g4), g1 = __ldg(g4 + 1);
        gv[0] = g0.x; gv[1] = g0.y; gv[2] = g0.z; gv[3] = g0.w;
        gv[4] = g1.x; gv[5] = g1.y; gv[6] = g1.z; gv[7] = g1.w;
        if (b) {
          const float4 *b4 = reinterpret_cast<const float4 *>(b) + 2 * j;
          const float4 b0 = __ldg(b4), b1 = __ldg(b4 + 1);
          bv[0] = b0.x; bv[1] = b0.y; bv[2] = b0.z; bv[3] = b0.w;
          bv[4] = b1.x; bv[5] = b1.y; bv[6] = b1.z; bv[7] = b1.w;
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) bv[q] = 0.f;
        }
      }
      uint4 u;
      __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float a = (val(k, 2 * q) - mean) * scale, c = (val(k, 2 * q + 1) - mean) * scale;
        if (kind == FLASH_GAU_NORM_LAYER) {
          a = fmaf(a, gv[2 * q], bv[2 * q]);
          c = fmaf(c, gv[2 * q + 1], bv[2 * q + 1]);
        }
        h[q] = __floats2bfloat162_rn(a, c);
      }
      y[j] = u;
    }
  }
}

// fp32 heads [4][M][s] rotated in place: thread = (head, token, pair).
__global__ void __launch_bounds__(256) rope_heads_f32(float *__restrict__ heads, long long M,
                                                      int T, int s, const RopeTable tab,
                                                      int pos_offset) {
  const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const int half = s / 2;
  if (idx >= 4 * M * half) return;
  const int i = (int)(idx % half);
  const long long hm = idx / half;  // h * M + m
  const long long m = hm % M;
  float cs, sn;
  rope_sincos((float)(m % T + pos_offset), tab.phi[i], &sn, &cs);
  float *h = heads + hm * s + 2 * i;
  const float x0 = h[0], x1 = h[1];
  h[0] = x0 * cs - x1 * sn;
  h[1] = x0 * sn + x1 * cs;
}


inline unsigned cdiv(long long a, long long b) { return (unsigned)((a + b - 1) / b); }

RopeJob rope_job(const Problem &p) {
  RopeJob r;
  r.tab = (p.rope && p.dtype == FLASH_GAU_BF16) ? (__half2 *)p.rope_cs : nullptr;
  r.T = p.T;
  r.s = p.s;
  r.pos_offset = p.pos_offset;
  r.phi = p.rope_tab;
  return r;
}
unsigned rope_blocks(const RopeJob &r) { return r.tab ? cdiv((long long)r.T * (r.s / 2), 256) : 0; }

template <int NV>
cudaError_t launch_norm_bf16x8(const Problem &p, unsigned grid) {
  const int nv = (p.d / 8 + 31) / 32;
  if (nv > NV) return launch_norm_bf16x8<NV * 2 <= kNormVec ? NV * 2 : kNormVec>(p, grid);
  const RopeJob r = rope_job(p);
  return launch_pdl(norm_rows_bf16x8<NV>, dim3(grid + rope_blocks(r)), dim3(256), 0, p.stream,
                    (const uint4 *)p.X, (uint4 *)p.xn, p.M, p.d, p.norm, p.norm_g, p.norm_b,
                    p.norm_eps, r);
}

// whether block_norm's launch also fills the RoPE table
bool norm_fills_rope_table(const Problem &p) {
  auto al16 = [](const void *q) { return ((uintptr_t)q & 15) == 0; };
  return p.dtype == FLASH_GAU_BF16 && p.d % 8 == 0 && p.d <= 32 * 8 * kNormVec && al16(p.X) &&
         (p.norm != FLASH_GAU_NORM_LAYER || (al16(p.norm_g) && al16(p.norm_b)));
}

// relpos[k] = rope(a)_i . rope(b)_j for any i, j with j - i = k - (C - 1):
// rotating a by i and b by j leaves a . R(j - i) b, per pair
// (a0 b0 + a1 b1) cos(delta) + (a1 b0 - a0 b1) sin(delta), delta = (j - i)
// times the pair's frequency.  One warp per entry, the lanes taking pairs
// q = lane, lane + 32, ..., fp32 partial sums added by a butterfly; the
// angles from the same exact-turns method as the heads' RoPE.
__global__ void __launch_bounds__(256)
rope_toeplitz_kernel(const float *__restrict__ a, const float *__restrict__ b, int pairs, int C,
                     const RopeTable phi, float *__restrict__ relpos) {
  const int k = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x % 32;
  if (k >= 2 * C - 1) return;
  const float off = (float)(k - (C - 1));  // exact: |off| < 2^24
  float acc = 0.f;
  for (int q = lane; q < pairs; q += 32) {
    float sn, cs;
    rope_sincos(off, phi.phi[q], &sn, &cs);
    const float a0 = a[2 * q], a1 = a[2 * q + 1], b0 = b[2 * q], b1 = b[2 * q + 1];
    acc = fmaf(fmaf(a0, b0, a1 * b1), cs, acc);
    acc = fmaf(fmaf(a1, b0, -a0 * b1), sn, acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) relpos[k] = acc;
}

}  // namespace

cudaError_t block_norm(const Problem &p) {
  const unsigned grid = cdiv(p.M * 32, 256);
  // 16-byte loads of X (and of the LayerNorm scale and shift) need 16-byte
  // aligned caller pointers; otherwise the scalar kernel runs
  if (norm_fills_rope_table(p))
    return launch_norm_bf16x8<1>(p, grid);
  if (p.dtype == FLASH_GAU_BF16)
    return launch_pdl(norm_rows<__nv_bfloat16>, dim3(grid), dim3(256), 0, p.stream,
                      (const __nv_bfloat16 *)p.X, (__nv_bfloat16 *)p.xn, p.M, p.d, p.norm,
                      p.norm_g, p.norm_b, p.norm_eps);
  return launch_pdl(norm_rows<float>, dim3(grid), dim3(256), 0, p.stream, (const float *)p.X,
                    (float *)p.xn, p.M, p.d, p.norm, p.norm_g, p.norm_b, p.norm_eps);
}

cudaError_t rope_table_stage(const Problem &p) {
  // done inside the norm's launch when that runs the fast kernel
  if (p.norm != FLASH_GAU_NORM_NONE && norm_fills_rope_table(p)) return cudaSuccess;
  const RopeJob r = rope_job(p);
  return launch_pdl(rope_table_kernel, dim3(rope_blocks(r)), dim3(256), 0, p.stream, r);
}

cudaError_t rope_toeplitz_bias(const float *a, const float *b, int m, int C, float base,
                               float *relpos, cudaStream_t stream) {
  RopeTable phi;
  rope_table(&phi, m, base);
  const unsigned n = (unsigned)(2 * C - 1);  // entries, one warp each, 8 a block
  rope_toeplitz_kernel<<<(n + 7) / 8, 256, 0, stream>>>(a, b, m / 2, C, phi, relpos);
  return cudaGetLastError();
}

cudaError_t simt_rope_heads_f32(const Problem &p) {
  rope_heads_f32<<<cdiv(4 * p.M * (p.s / 2), 256), 256, 0, p.stream>>>(
      (float *)p.heads, p.M, p.T, p.s, p.rope_tab, p.pos_offset);
  return cudaGetLastError();
}

}  // namespace flashgau
