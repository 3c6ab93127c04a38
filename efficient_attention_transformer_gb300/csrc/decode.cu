// Autoregressive decode step of the FLASH GAU layer: one new token for each
// of B sequences, in constant work per token ("Transformer Quality in
// Linear Time", §3.2.1: decoding keeps the global term as a single running
// matrix and attends locally within the current chunk only).  Per sequence
// the state holds
//   pos      tokens consumed so far (the new one sits at i = pos mod C of
//            its chunk)
//   Prefix   [s, e] fp32, the sum of K_lin^T V over completed chunks
//   caches   the current chunk's K_quad, K_lin [C, s] and V [C, e] rows
// and a step runs five launches, chained by programmatic dependent launch:
//   project  x W_uvz in depth slices (pos += 1)
//   scores   z = swish(sum of the Z slices), the four heads, and
//            a_j = relu(q_quad . k_quad_j / C + relpos[j - i + C - 1])^2
//            (j <= i), once per sequence
//   attend   u, v = swish(sum of the slices); vhat = sum_j a_j v_j +
//            lin_scale q_lin Prefix, gated = u * vhat; the token's rows go
//            into the caches
//   output   gated W_o in depth slices
//   finish   out = the slices' sum; at a chunk's last token
//            Prefix += K_lin,chunk^T V_chunk
// The projections stream the weights once per step for all B sequences.
// For bf16 io they run on the tcgen05 tensor cores: y^T = W^T x^T with 128
// weight columns in the TMEM lanes and the sequences as the MMA's N (up to
// 256), split over the depth in about 150 blocks, the weight tiles loaded by
// TMA before the step's input is ready (programmatic dependent launch).  For
// fp32 io they are split-K matrix-vector products on the CUDA cores with
// 16-byte weight loads.  Sums, scores and caches are fp32.  The step is
// latency-bound: the kernels keep several independent loads in flight per
// thread.
#include <cuda_bf16.h>

#include "flash_gau_internal.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

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
__device__ __forceinline__ float swish(float x) { return x / (1.0f + expf(-x)); }

constexpr int kGroup = 8;       // sequences per pass of a matrix-vector kernel
constexpr int kWarps = 8;
constexpr int kTileN = 256;     // output columns per block: 8 per lane
// dynamic shared memory of the matrix-vector kernel: the group's input rows
// and the warps' partial sums
constexpr size_t kGemvSmem = sizeof(float) * (kGroup * 128 + kWarps * kGroup * (kTileN + 4));

// 8 consecutive weights of row k from column c (c % 8 == 0), as floats
__device__ __forceinline__ void load8(const __nv_bfloat16 *W, long long o, float (&w)[8]) {
  const uint4 q = *reinterpret_cast<const uint4 *>(W + o);
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    w[2 * i] = f.x;
    w[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float *W, long long o, float (&w)[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(W + o);
  const float4 b = *reinterpret_cast<const float4 *>(W + o + 4);
  w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w, w[4] = b.x, w[5] = b.y, w[6] = b.z, w[7] = b.w;
}

// Split-K matrix-vector products: part[slice][b][c] = sum over the slice's
// ks rows k of x[b][k] W[k][c], for all B sequences.  Block (column tile,
// slice, group of 8 sequences); a lane owns 8 consecutive columns (16-byte loads of a weight row,
// 512 coalesced bytes per warp), the warps share the slice's rows, and the
// warps' sums meet in shared memory.  Consumers add the slices in a fixed
// order, so the results do not depend on scheduling.
template <typename Tx, typename Tw>
__global__ void __launch_bounds__(256)
gemv_splitk(const Tx *__restrict__ x, int B, const Tw *__restrict__ W, int K, int N, int ks,
            float *__restrict__ part, int *pos) {
  extern __shared__ float dsm[];
  float(*sx)[128] = reinterpret_cast<float(*)[128]>(dsm);
  float(*red)[kGroup][kTileN + 4] =
      reinterpret_cast<float(*)[kGroup][kTileN + 4]>(dsm + kGroup * 128);
  griddep_launch_dependents();
  griddep_wait();  // x comes from the kernel before (or the step before)
  if (pos && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
    for (int b = threadIdx.x; b < B; b += blockDim.x) pos[b] += 1;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = blockIdx.x * kTileN + lane * 8;
  const int k0 = blockIdx.y * ks, k1 = min(K, k0 + ks);
  const int rows = (k1 - k0 + kWarps - 1) / kWarps;  // rows per warp
  // this block's group of up to kGroup sequences (the groups run in parallel)
  {
    const int b0 = blockIdx.z * kGroup;
    const int nb = min(kGroup, B - b0);
    for (int i = threadIdx.x; i < kGroup * ks; i += blockDim.x) {
      const int b = i / ks, k = i - b * ks;
      sx[b][k] = (b < nb && k0 + k < k1) ? to_f(x[(long long)(b0 + b) * K + k0 + k]) : 0.f;
    }
    __syncthreads();
    float acc[kGroup][8];
#pragma unroll
    for (int b = 0; b < kGroup; ++b)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[b][j] = 0.f;
    if (c < N) {
      const int kw0 = k0 + warp * rows, kw1 = min(k1, kw0 + rows);
#pragma unroll 4
      for (int k = kw0; k < kw1; ++k) {
        float w[8];
        load8(W, (long long)k * N + c, w);
#pragma unroll
        for (int b = 0; b < kGroup; ++b) {
          const float xv = sx[b][k - k0];
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[b][j] = fmaf(xv, w[j], acc[b][j]);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kGroup; ++b)
#pragma unroll
      for (int j = 0; j < 8; ++j) red[warp][b][lane * 8 + j] = acc[b][j];
    __syncthreads();
    for (int o = threadIdx.x; o < nb * kTileN; o += blockDim.x) {
      const int b = o / kTileN, cc = o - b * kTileN;
      const int col = blockIdx.x * kTileN + cc;
      if (col >= N) continue;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += red[w][b][cc];
      part[((long long)blockIdx.y * B + b0 + b) * N + col] = v;
    }
    __syncthreads();
  }
}

// Split-K product on the tensor cores, bf16 operands, fp32 accumulation:
// part[slice][b][c] = sum over the slice's rows k of x[b][k] W[k][c], as
// y^T = W^T x^T.  Block (128 weight columns, depth slice of kbs 64-row
// k-blocks): A = the W tile, two 64-column boxes per k-block read M-major;
// B = the sequences' x rows (npad = B rounded up to 16, rows past B read as
// zeros), K-major; D = [128 columns, npad sequences] fp32 in TMEM.  Thread 0
// issues the weight loads before waiting for the kernel before (the weights
// are inputs), then the x loads and the MMAs; each of the four warps drains
// its 32 columns (thread = column, registers = sequences), so the stores of
// one sequence's columns are coalesced.  Every wait is bounded.
constexpr int kTcCols = 128;
constexpr int kTcMaxKb = 4;
constexpr int kTcW = 64 * 64 * 2;  // one 64 x 64 weight box
__host__ __device__ constexpr size_t tc_stage_bytes(int npad) { return 2 * kTcW + (size_t)npad * 128; }

__global__ void __launch_bounds__(128, 1)
decode_tc_gemm(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
               int B, int npad, int K, int N, int kbs, float *__restrict__ part, int *pos,
               int *status) {
  using namespace ptx;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *tiles = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_w, bar_x, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ int failed;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n0 = blockIdx.x * kTcCols;
  const int nkb_all = (K + 63) / 64, kb0 = blockIdx.y * kbs;
  const int nkb = min(kbs, nkb_all - kb0);
  const uint32_t tcols = npad <= 32 ? 32 : npad <= 64 ? 64 : npad <= 128 ? 128 : 256;
  const size_t stage = tc_stage_bytes(npad);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar_w), 1);
    mbar_init(smem_u32(&bar_x), 1);
    mbar_init(smem_u32(&bar_mma), 1);
    failed = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base), tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    // the weight tiles: inputs, loaded while the kernel before still runs
    mbar_arrive_expect_tx(smem_u32(&bar_w), (uint32_t)(nkb * 2 * kTcW));
    for (int k = 0; k < nkb; ++k)
      for (int h = 0; h < 2; ++h)
        tma_load_2d(smem_u32(tiles + k * stage + h * kTcW), &tmW, smem_u32(&bar_w), n0 + 64 * h,
                    (kb0 + k) * 64);
  }
  griddep_launch_dependents();
  griddep_wait();  // x comes from the kernel before
  if (pos && blockIdx.x == 0 && blockIdx.y == 0)
    for (int b = threadIdx.x; b < B; b += blockDim.x) pos[b] += 1;
  const uint32_t idesc = idesc_bf16_f32(kTcCols, npad, 1, 0);
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(smem_u32(&bar_x), (uint32_t)(nkb * npad * 128));
    for (int k = 0; k < nkb; ++k)
      tma_load_2d(smem_u32(tiles + k * stage + 2 * kTcW), &tmX, smem_u32(&bar_x), (kb0 + k) * 64, 0);
    if (mbar_wait(smem_u32(&bar_w), 0) && mbar_wait(smem_u32(&bar_x), 0)) {
      tc_fence_after();
      for (int k = 0; k < nkb; ++k) {
        // A: W^T, M-major, the two 64-column boxes 8 KB apart, 16 rows of
        // 128 B per step; B: x rows, K-major, 32 B per step
        const uint64_t da = sw128_desc(smem_u32(tiles + k * stage), kTcW, 1024);
        const uint64_t db = sw128_desc(smem_u32(tiles + k * stage + 2 * kTcW), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16_ss(tmem_base, desc_advance(da, kk * 2048), desc_advance(db, kk * 32), idesc,
                     (k | kk) != 0);
      }
      mma_commit(smem_u32(&bar_mma));
    } else {
      failed = 1;
      atomicExch(status, FLASH_GAU_ETIMEOUT);
    }
  }
  __syncthreads();
  bool ok = !failed && mbar_wait(smem_u32(&bar_mma), 0);
  ok = __all_sync(0xffffffffu, ok);
  if (ok) {
    tc_fence_after();
    const int col = n0 + warp * 32 + lane;
    const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16);
    float *dst = part + (size_t)blockIdx.y * B * N + col;
    for (int c0 = 0; c0 < npad; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(taddr + c0, v);
      tmem_ld_wait();
      if (col < N)
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c0 + j < B) dst[(size_t)(c0 + j) * N] = __uint_as_float(v[j]);
    }
  } else if (lane == 0) {
    atomicExch(status, FLASH_GAU_ETIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tcols);
  }
}

// The chunk weights of the new token, once per sequence: block (32-key
// tile, sequence), 8 warps of 4 keys each.  Each block forms z = swish of
// the projection's Z slices and the two quadratic heads it needs; block 0
// of a sequence also stores all four heads for the attend kernel.  A warp
// issues the loads of its 4 cached key rows together, then reduces the 4
// dot products; a_j = local_scale relu(q_quad . k_quad_j / C +
// relpos[j - i + C - 1])^2 for j <= i (key i is the new token's own).
constexpr int kKeyTile = 32;
constexpr int kMaxS = 256;
__global__ void __launch_bounds__(256)
decode_scores(DecodeLayout L, const float *__restrict__ gamma, const float *__restrict__ beta,
              const float *__restrict__ relpos, int B, int C, int e, int s, int slices,
              float local_scale) {
  __shared__ float qq[kMaxS], kq_new[kMaxS];
  griddep_launch_dependents();
  griddep_wait();
  const int b = blockIdx.y, j0 = blockIdx.x * kKeyTile;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int N = 2 * e + s;
  const int i = (L.pos[b] - 1) % C;
  if (j0 > i && blockIdx.x != 0) return;
  const float *yp = L.proj + (long long)b * N;
  const long long sstride = (long long)B * N;
  const float *kq_c = L.kq + (long long)b * C * s;
  constexpr int KW = kKeyTile / 8;  // keys per warp
  constexpr int MS = kMaxS / 32;    // key elements per lane
  float kv[KW][MS];
  // the cached keys first: they do not depend on this step's projection
#pragma unroll
  for (int t = 0; t < KW; ++t) {
    const int j = j0 + warp * KW + t;
#pragma unroll
    for (int m = 0; m < MS; ++m) {
      const int k = lane + 32 * m;
      kv[t][m] = 0.f;
      if (j < i && k < s) kv[t][m] = kq_c[(long long)j * s + k];
    }
  }
  for (int k = threadIdx.x; k < s; k += blockDim.x) {
    float pz = 0.f;
    for (int q = 0; q < slices; ++q) pz += yp[q * sstride + 2 * e + k];
    const float z = swish(pz);
    qq[k] = fmaf(z, gamma[k], beta[k]);
    kq_new[k] = fmaf(z, gamma[s + k], beta[s + k]);
    if (blockIdx.x == 0)
      for (int h = 0; h < 4; ++h)
        L.heads[((long long)b * 4 + h) * s + k] = fmaf(z, gamma[h * s + k], beta[h * s + k]);
  }
  __syncthreads();
  if (j0 > i) return;
  const float inv_c = 1.0f / (float)C;
#pragma unroll
  for (int t = 0; t < KW; ++t) {
    const int j = j0 + warp * KW + t;
#pragma unroll
    for (int m = 0; m < MS; ++m) {
      const int k = lane + 32 * m;
      if (j == i && k < s) kv[t][m] = kq_new[k];
    }
  }
#pragma unroll
  for (int t = 0; t < KW; ++t) {
    const int j = j0 + warp * KW + t;
    float dot = 0.f;
#pragma unroll
    for (int m = 0; m < MS; ++m) {
      const int k = lane + 32 * m;
      if (k < s) dot = fmaf(qq[k], kv[t][m], dot);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0 && j <= i) {
      const float r = fmaxf(fmaf(dot, inv_c, relpos[j - i + C - 1]), 0.f);
      L.score[(long long)b * C + j] = local_scale * r * r;
    }
  }
}

// one block per (128 value columns, sequence), 8 warps: gathers the
// projection's slices into this block's U and V columns, then the weighted
// sum over the chunk's cached V rows (weights a_j) and the rows of the
// linear cache (weights lin_scale q_lin), each lane on 4 consecutive
// columns (16-byte loads): warp w takes rows w, w + 8, .. of each, eight
// loads in flight per lane.  MANY (many sequences, more than two blocks an
// SM): the eight rows land in registers before one accumulator takes them
// (64 registers, four blocks an SM); else each row has an accumulator of its
// own (two blocks an SM, but shorter dependences per warp).  Then the gate.
// The warps' sums meet in a fixed order.
constexpr int kAttW = 8;
constexpr int kAttCols = 128;  // value columns per block: 4 per lane
constexpr int kAttBatch = 8;   // loads in flight per lane
__device__ __forceinline__ float4 fma4(float a, float4 v, float4 acc) {
  return make_float4(fmaf(a, v.x, acc.x), fmaf(a, v.y, acc.y), fmaf(a, v.z, acc.z),
                     fmaf(a, v.w, acc.w));
}
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

template <bool MANY>
__global__ void __launch_bounds__(32 * kAttW)
decode_attend(DecodeLayout L, int B, int C, int e, int s, int slices, float lin_scale,
              __nv_bfloat16 *gated_io) {
  __shared__ float4 red[kAttW][32];
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int b = blockIdx.y, c = blockIdx.x * kAttCols + lane * 4;  // 4 columns a lane
  const int N = 2 * e + s;
  const int i = (L.pos[b] - 1) % C;
  const float *yp = L.proj + (long long)b * N;
  const long long sstride = (long long)B * N;
  const float *ql = L.heads + ((long long)b * 4 + 2) * s;
  const float *sa = L.score + (long long)b * C;
  float *v_c = L.vc + (long long)b * C * e;
  const float *pre = L.prefix + (long long)b * s * e + c;
  const bool on = c < e;  // e is a multiple of 8: all 4 columns or none
  float4 pu = make_float4(0.f, 0.f, 0.f, 0.f), pv = pu;
  if (on)
    for (int q = 0; q < slices; ++q) {
      pu = add4(pu, *reinterpret_cast<const float4 *>(yp + q * sstride + c));
      pv = add4(pv, *reinterpret_cast<const float4 *>(yp + q * sstride + e + c));
    }
  const float4 u = make_float4(swish(pu.x), swish(pu.y), swish(pu.z), swish(pu.w));
  const float4 vnew = make_float4(swish(pv.x), swish(pv.y), swish(pv.z), swish(pv.w));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (on) {
    if constexpr (MANY) {
      // the chunk's cached V rows j < i, then the linear cache's rows
      for (int j0 = warp; j0 < i; j0 += kAttBatch * kAttW) {
        float4 v[kAttBatch];
        float a[kAttBatch];
#pragma unroll
        for (int t = 0; t < kAttBatch; ++t) {
          const int j = j0 + t * kAttW;
          v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
          a[t] = 0.f;
          if (j < i) {
            v[t] = *reinterpret_cast<const float4 *>(v_c + (long long)j * e + c);
            a[t] = sa[j];
          }
        }
#pragma unroll
        for (int t = 0; t < kAttBatch; ++t) acc = fma4(a[t], v[t], acc);
      }
      if (i % kAttW == warp) acc = fma4(sa[i], vnew, acc);
      for (int k0 = warp; k0 < s; k0 += kAttBatch * kAttW) {
        float4 v[kAttBatch];
        float a[kAttBatch];
#pragma unroll
        for (int t = 0; t < kAttBatch; ++t) {
          const int k = k0 + t * kAttW;
          v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
          a[t] = 0.f;
          if (k < s) {
            v[t] = *reinterpret_cast<const float4 *>(pre + (long long)k * e);
            a[t] = ql[k];
          }
        }
#pragma unroll
        for (int t = 0; t < kAttBatch; ++t) acc = fma4(lin_scale * a[t], v[t], acc);
      }
    } else {
      float4 a8[kAttBatch], l8[kAttBatch];
#pragma unroll
      for (int t = 0; t < kAttBatch; ++t) a8[t] = l8[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j0 = warp; j0 < i; j0 += kAttBatch * kAttW) {
#pragma unroll
        for (int t = 0; t < kAttBatch; ++t) {
          const int j = j0 + t * kAttW;
          if (j < i)
            a8[t] = fma4(sa[j], *reinterpret_cast<const float4 *>(v_c + (long long)j * e + c),
                         a8[t]);
        }
      }
      if (i % kAttW == warp) a8[0] = fma4(sa[i], vnew, a8[0]);
      for (int k0 = warp; k0 < s; k0 += kAttBatch * kAttW) {
#pragma unroll
        for (int t = 0; t < kAttBatch; ++t) {
          const int k = k0 + t * kAttW;
          if (k < s)
            l8[t] = fma4(ql[k], *reinterpret_cast<const float4 *>(pre + (long long)k * e), l8[t]);
        }
      }
      float4 l = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int t = 0; t < kAttBatch; ++t) {
        acc = add4(acc, a8[t]);
        l = add4(l, l8[t]);
      }
      acc = fma4(lin_scale, l, acc);
    }
  }
  red[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && on) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kAttW; ++w) v = add4(v, red[w][lane]);
    const float4 g = make_float4(u.x * v.x, u.y * v.y, u.z * v.z, u.w * v.w);
    *reinterpret_cast<float4 *>(L.gated + (long long)b * e + c) = g;
    if (gated_io) {
      // bf16 copy: the tensor-core output projection's operand
      __nv_bfloat162 h2[2] = {__floats2bfloat162_rn(g.x, g.y), __floats2bfloat162_rn(g.z, g.w)};
      *reinterpret_cast<uint2 *>(gated_io + (long long)b * e + c) =
          *reinterpret_cast<const uint2 *>(h2);
    }
    // the token's row, for the chunk's later keys
    *reinterpret_cast<float4 *>(v_c + (long long)i * e + c) = vnew;
  }
  if (blockIdx.x == 0) {
    const float *h = L.heads + (long long)b * 4 * s;
    float *kq_c = L.kq + (long long)b * C * s, *kl_c = L.kl + (long long)b * C * s;
    for (int k = threadIdx.x; k < s; k += blockDim.x) {
      kq_c[(long long)i * s + k] = h[s + k];
      kl_c[(long long)i * s + k] = h[3 * s + k];
    }
  }
}

// the output's slices into out (io type): blocks with blockIdx.y == 0, one
// thread per column; and, at a chunk's last token,
// Prefix += K_lin,chunk^T V_chunk: one thread per column c for kFoldRows
// rows k, blocks (256 columns, row group, sequence).  Away from a chunk's
// end the row-group blocks return at once, so there are few of them.
constexpr int kFoldRows = 16;
template <typename T>
__global__ void __launch_bounds__(256)
decode_finish(DecodeLayout L, T *__restrict__ out, int B, int C, int d, int e, int s, int slices) {
  griddep_launch_dependents();
  griddep_wait();
  const int b = blockIdx.z, k0 = blockIdx.y * kFoldRows;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (blockIdx.y == 0 && c < d) {
    float v = 0.f;
#pragma unroll 8
    for (int q = 0; q < slices; ++q) v += L.outp[((long long)q * B + b) * d + c];
    out[(long long)b * d + c] = from_f<T>(v);
  }
  if ((L.pos[b] - 1) % C != C - 1 || c >= e) return;
  const float *kl_c = L.kl + (long long)b * C * s, *v_c = L.vc + (long long)b * C * e;
  const int k1 = k0 + kFoldRows < s ? k0 + kFoldRows : s;
  float acc[kFoldRows];
#pragma unroll
  for (int t = 0; t < kFoldRows; ++t) acc[t] = 0.f;
  for (int j = 0; j < C; ++j) {
    const float v = v_c[(long long)j * e + c];
#pragma unroll
    for (int t = 0; t < kFoldRows; ++t)
      if (k0 + t < k1) acc[t] = fmaf(kl_c[(long long)j * s + k0 + t], v, acc[t]);
  }
#pragma unroll
  for (int t = 0; t < kFoldRows; ++t)
    if (k0 + t < k1) L.prefix[((long long)b * s + k0 + t) * e + c] += acc[t];
}

// One tensor-core split-K product: part[slices][B][N] from x [B, K] (bf16)
// and W [K, N] (bf16); slices from decode_tc_slices.
cudaError_t tc_product(const void *x, const void *W, int B, int K, int N, float *part, int *pos,
                       int *status, cudaStream_t stream) {
  const int npad = (B + 15) / 16 * 16;
  int kbs = 0;
  const int slices = decode_tc_slices(K, N, &kbs);
  CUtensorMap tW, tX;
  cudaError_t err;
  if ((err = make_tmap_bf16_2d(&tW, W, K, N, N, 64, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tX, x, B, K, K, npad, 64)) != cudaSuccess) return err;
  const size_t smem = kbs * tc_stage_bytes(npad) + 1024;
  static unsigned long long configured = 0;  // shared-memory ceiling, per device
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!(configured & (1ull << dev))) {
    if ((err = cudaFuncSetAttribute(decode_tc_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)(kTcMaxKb * tc_stage_bytes(kDecodeTcMaxB) + 1024))) !=
        cudaSuccess)
      return err;
    configured |= 1ull << dev;
  }
  return launch_pdl(decode_tc_gemm, dim3((N + kTcCols - 1) / kTcCols, slices), dim3(128), smem,
                    stream, tW, tX, B, npad, K, N, kbs, part, pos, status);
}

template <typename T>
cudaError_t step(const DecodeProblem &q) {
  cudaError_t err;
  const int N = 2 * q.e + q.s;
  // bf16: the projections on the tensor cores
  const bool tc = sizeof(T) == 2 && q.B <= kDecodeTcMaxB;
  const int sp = tc ? decode_tc_slices(q.d, N, nullptr) : decode_slices(q.d, N);
  const int so = tc ? decode_tc_slices(q.e, q.d, nullptr) : decode_slices(q.e, q.d);
  const int ksp = (q.d + sp - 1) / sp, kso = (q.e + so - 1) / so;

  static unsigned long long configured = 0;  // shared-memory ceilings, per device
  static int sms[64];                         // and SM counts
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!(configured & (1ull << dev))) {
    if ((err = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev)) !=
        cudaSuccess)
      return err;
    if ((err = cudaFuncSetAttribute(gemv_splitk<T, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kGemvSmem)) != cudaSuccess ||
        (err = cudaFuncSetAttribute(gemv_splitk<float, T>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kGemvSmem)) != cudaSuccess)
      return err;
    configured |= 1ull << dev;
  }
  const int groups = (q.B + kGroup - 1) / kGroup;
  if (tc)
    err = tc_product(q.x, q.W_uvz, q.B, q.d, N, q.L.proj, q.L.pos, q.L.status, q.stream);
  else
    err = launch_pdl(gemv_splitk<T, T>, dim3((N + kTileN - 1) / kTileN, sp, groups), dim3(256),
                     kGemvSmem, q.stream, (const T *)q.x, q.B, (const T *)q.W_uvz, q.d, N, ksp,
                     q.L.proj, q.L.pos);
  if (err != cudaSuccess) return err;
  if ((err = launch_pdl(decode_scores, dim3((q.C + kKeyTile - 1) / kKeyTile, q.B), dim3(256), 0,
                        q.stream, q.L, q.gamma, q.beta, q.relpos, q.B, q.C, q.e, q.s, sp,
                        q.local_scale)) != cudaSuccess)
    return err;
  // more attention blocks than two an SM: the few-register form
  const dim3 agrid((q.e + kAttCols - 1) / kAttCols, q.B);
  const bool many = (long long)agrid.x * agrid.y > 2LL * sms[dev];
  if ((err = launch_pdl(many ? decode_attend<true> : decode_attend<false>, agrid,
                        dim3(32 * kAttW), 0, q.stream, q.L, q.B, q.C, q.e, q.s, sp, q.lin_scale,
                        tc ? (__nv_bfloat16 *)q.L.gated_io : (__nv_bfloat16 *)nullptr)) !=
      cudaSuccess)
    return err;
  if (tc)
    err = tc_product(q.L.gated_io, q.W_o, q.B, q.e, q.d, q.L.outp, nullptr, q.L.status, q.stream);
  else
    err = launch_pdl(gemv_splitk<float, T>, dim3((q.d + kTileN - 1) / kTileN, so, groups),
                     dim3(256), kGemvSmem, q.stream, (const float *)q.L.gated, q.B,
                     (const T *)q.W_o, q.e, q.d, kso, q.L.outp, (int *)nullptr);
  if (err != cudaSuccess) return err;
  const int fx = ((q.e > q.d ? q.e : q.d) + 255) / 256;
  return launch_pdl(decode_finish<T>, dim3(fx, (q.s + kFoldRows - 1) / kFoldRows, q.B),
                    dim3(256), 0, q.stream,
                    q.L, (T *)q.out, q.B, q.C, q.d, q.e, q.s, so);
}

}  // namespace

cudaError_t decode_step_f32(const DecodeProblem &q) { return step<float>(q); }
cudaError_t decode_step_bf16(const DecodeProblem &q) { return step<__nv_bfloat16>(q); }

}  // namespace flashgau
