// CUDA-core (FFMA) kernels of the FLASH GAU forward.  They compute in true
// fp32 (no TF32) and serve the fp32 io type, whose tolerance the tensor cores'
// reduced-precision inputs could not meet.
//
// Stages ("Transformer Quality in Linear Time", Method and eq. 7/8):
//   projection   [U|V|Z] = swish(X W_uvz), heads = Z*gamma_h + beta_h
//   chunk state  State_g = K_lin,g^T V_g
//   prefix scan  Prefix_g = lin_scale * sum_{h<g} State_h  (or the total)
//   attention    gated = U * (relu^2(Qq Kq^T/C + b) V + Q_lin Prefix_g)
//   output       O = gated W_o
#include <cuda_bf16.h>

#include "flash_gau_internal.h"
#include "sm103_ptx.cuh"

namespace flashgau {
using ptx::griddep_launch_dependents;
using ptx::griddep_wait;
namespace {

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

// ---------------------------------------------------------------- GEMM ----
// C[m, n] = sum_k A(m, k) B(k, n) for one batch (blockIdx.z), 64x64 tiles,
// 256 threads with a 4x4 register block each.  Operands are addressed by
// explicit element strides so that transposed views need no copy.
constexpr int kTile = 64;
constexpr int kTileK = 16;

template <typename Tin, typename Epi>
__global__ void __launch_bounds__(256)
simt_gemm(int M, int N, int K, const Tin *__restrict__ A, long long sam,
          long long sak, long long sab, const Tin *__restrict__ Bm, long long sbk,
          long long sbn, long long sbb, Epi epi) {
  // launched with programmatic dependent launch (see the stage functions)
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float As[kTileK][kTile + 1];
  __shared__ float Bs[kTileK][kTile + 1];
  const int batch = blockIdx.z;
  const int m0 = blockIdx.y * kTile, n0 = blockIdx.x * kTile;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  A += batch * sab;
  Bm += batch * sbb;
  float acc[4][4] = {};
  // each thread's share of a k-tile (4 A and 4 B elements), loaded into
  // registers one k-tile ahead so the loads overlap the products
  constexpr int kPer = kTile * kTileK / 256;
  float ra[kPer], rb[kPer];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int t = 0; t < kPer; ++t) {
      const int idx = threadIdx.x + t * 256;
      const int kk = idx % kTileK, mm = idx / kTileK;
      const int gm = m0 + mm, gk = k0 + kk;
      ra[t] = (gm < M && gk < K) ? to_f(A[gm * sam + gk * sak]) : 0.f;
      const int nn = idx % kTile, kb = idx / kTile;
      const int gn = n0 + nn, gk2 = k0 + kb;
      rb[t] = (gn < N && gk2 < K) ? to_f(Bm[gk2 * sbk + gn * sbn]) : 0.f;
    }
  };
  fetch(0);
  for (int k0 = 0; k0 < K; k0 += kTileK) {
#pragma unroll
    for (int t = 0; t < kPer; ++t) {
      const int idx = threadIdx.x + t * 256;
      As[idx % kTileK][idx / kTileK] = ra[t];
      Bs[idx / kTile][idx % kTile] = rb[t];
    }
    __syncthreads();
    if (k0 + kTileK < K) fetch(k0 + kTileK);
#pragma unroll
    for (int kk = 0; kk < kTileK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int gm = m0 + ty * 4 + i, gn = n0 + tx * 4 + j;
      if (gm < M && gn < N) epi(batch, gm, gn, acc[i][j]);
    }
}

// Projection epilogue: columns [0,e) -> U, [e,2e) -> V, [2e,2e+s) -> heads.
template <typename T>
struct ProjEpi {
  T *U, *V, *heads;
  const float *gamma, *beta;
  long long M;
  int e, s;
  __device__ void operator()(int, int m, int n, float acc) const {
    float y = swish(acc);
    if (n < e) {
      U[(long long)m * e + n] = from_f<T>(y);
    } else if (n < 2 * e) {
      V[(long long)m * e + (n - e)] = from_f<T>(y);
    } else {
      int c = n - 2 * e;
#pragma unroll
      for (int h = 0; h < 4; ++h)
        heads[(long long)h * M * s + (long long)m * s + c] =
            from_f<T>(fmaf(y, gamma[h * s + c], beta[h * s + c]));
    }
  }
};

template <typename T>
struct StateEpi {  // batch = b*G + g; State_g[si, ej]
  T *state;
  int s, e;
  __device__ void operator()(int batch, int m, int n, float acc) const {
    state[((long long)batch * s + m) * e + n] = from_f<T>(acc);
  }
};

template <typename T>
struct StoreEpi {
  T *out;
  int ld;
  const T *residual;  // added when not null (the block's shortcut)
  __device__ void operator()(int, int m, int n, float acc) const {
    const long long i = (long long)m * ld + n;
    out[i] = from_f<T>(residual ? acc + to_f(residual[i]) : acc);
  }
};

// ---------------------------------------------------------- prefix scan ----
// One thread per (b, s*e element): the G-step running sum of chunk states.
// With segment ids (a change of id between neighbouring chunks starts a
// segment) the sums restart at each segment, and a non-causal prefix is the
// segment's total, one per chunk; `average` divides each sum by its number
// of chunks (an empty sum stays zero).
template <typename T>
__global__ void simt_prefix_scan(const T *__restrict__ state, T *__restrict__ prefix,
                                 int B, int G, long long se, int causal, float lin_scale,
                                 const int *__restrict__ seg_ids, int average, int per_chunk) {
  griddep_wait();
  griddep_launch_dependents();
  long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (idx >= B * se) return;
  long long b = idx / se, r = idx % se;
  const T *st = state + b * G * se + r;
  const int *seg = seg_ids ? seg_ids + b * G : nullptr;
  T *pre = prefix + (per_chunk ? b * G * se : b * se) + r;
  float run = 0.f;
  int start = 0;
  auto write_total = [&](int end) {
    const float v = (average ? lin_scale / (float)(end - start) : lin_scale) * run;
    for (int h = start; h < end; ++h) pre[h * se] = from_f<T>(v);
  };
  for (int g = 0; g < G; ++g) {
    if (seg && g > 0 && seg[g] != seg[g - 1]) {
      if (!causal) write_total(g);
      run = 0.f;
      start = g;
    }
    if (causal) {
      const int n = g - start;
      const float sc = average ? (n > 0 ? lin_scale / (float)n : 0.f) : lin_scale;
      pre[g * se] = from_f<T>(sc * run);
    }
    run += to_f(st[g * se]);
  }
  if (!causal) {
    if (per_chunk) write_total(G);
    else pre[0] = from_f<T>((average ? lin_scale / (float)G : lin_scale) * run);
  }
}

// ------------------------------------------------------ chunk attention ----
// Block = (chunk b*G+g, 32 query rows, 64 value columns).  Score rows are
// built 64 keys at a time in shared memory and consumed immediately; the
// C x C matrix never exists in global memory.
constexpr int kAttRows = 32;
constexpr int kAttKeys = 64;
constexpr int kAttCols = 64;

template <typename T>
__global__ void __launch_bounds__(256)
simt_chunk_attention(const T *__restrict__ U, const T *__restrict__ V,
                     const T *__restrict__ heads, const T *__restrict__ prefix,
                     const float *__restrict__ relpos, T *__restrict__ gated,
                     long long M, int C, int G, int e, int s, int causal, float local_scale,
                     int per_chunk) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ float sm[];
  const int sp = s + 1;
  float *q = sm;                          // [32][s+1]
  float *kk = q + kAttRows * sp;          // [64][s+1]
  float *pw = kk + kAttKeys * sp;         // [32][65]
  float *vv = pw + kAttRows * (kAttKeys + 1);  // [64][65]

  const int chunk = blockIdx.z;  // b*G + g
  const int g = chunk % G;
  const long long tok0 = (long long)chunk * C;  // first token of the chunk
  const int i0 = blockIdx.y * kAttRows;          // row offset inside the chunk
  const int c0 = blockIdx.x * kAttCols;          // value column offset
  const T *Qq = heads, *Kq = heads + M * s, *Ql = heads + 2 * M * s;
  const int tid = threadIdx.x;
  const int r = tid / 8, cg = (tid % 8) * 8;  // this thread: row r, cols cg..cg+7
  float acc[8] = {};

  for (int idx = tid; idx < kAttRows * s; idx += 256) {
    int rr = idx / s, k = idx % s;
    q[rr * sp + k] = (i0 + rr < C) ? to_f(Qq[(tok0 + i0 + rr) * s + k]) : 0.f;
  }
  const float inv_c = 1.0f / (float)C;
  // no keys at all when the local term is switched off
  const int key_end = local_scale == 0.f ? 0 : causal ? min(C, i0 + kAttRows) : C;
  for (int j0 = 0; j0 < key_end; j0 += kAttKeys) {
    __syncthreads();
    for (int idx = tid; idx < kAttKeys * s; idx += 256) {
      int jj = idx / s, k = idx % s;
      kk[jj * sp + k] = (j0 + jj < C) ? to_f(Kq[(tok0 + j0 + jj) * s + k]) : 0.f;
    }
    for (int idx = tid; idx < kAttKeys * kAttCols; idx += 256) {
      int jj = idx / kAttCols, cc = idx % kAttCols;
      vv[jj * (kAttCols + 1) + cc] = (j0 + jj < C && c0 + cc < e)
                                         ? to_f(V[(tok0 + j0 + jj) * e + c0 + cc])
                                         : 0.f;
    }
    __syncthreads();
    for (int idx = tid; idx < kAttRows * kAttKeys; idx += 256) {
      int rr = idx / kAttKeys, jj = idx % kAttKeys;
      int i = i0 + rr, j = j0 + jj;
      float sc = 0.f;
      for (int k = 0; k < s; ++k) sc = fmaf(q[rr * sp + k], kk[jj * sp + k], sc);
      float a = 0.f;
      if (i < C && j < C && !(causal && j > i)) {
        float x = fmaf(sc, inv_c, relpos[j - i + C - 1]);
        x = fmaxf(x, 0.f);
        a = local_scale * x * x;
      }
      pw[rr * (kAttKeys + 1) + jj] = a;
    }
    __syncthreads();
    for (int jj = 0; jj < kAttKeys; ++jj) {
      float a = pw[r * (kAttKeys + 1) + jj];
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = fmaf(a, vv[jj * (kAttCols + 1) + cg + c], acc[c]);
    }
  }

  // global term: Q_lin rows times the chunk's prefix state (already scaled)
  __syncthreads();
  for (int idx = tid; idx < kAttRows * s; idx += 256) {
    int rr = idx / s, k = idx % s;
    q[rr * sp + k] = (i0 + rr < C) ? to_f(Ql[(tok0 + i0 + rr) * s + k]) : 0.f;
  }
  const long long se = (long long)s * e;
  const T *pre = prefix + (per_chunk ? (long long)chunk * se : (long long)(chunk / G) * se);
  (void)g;
  for (int k0 = 0; k0 < s; k0 += kAttKeys) {
    __syncthreads();
    for (int idx = tid; idx < kAttKeys * kAttCols; idx += 256) {
      int kk2 = idx / kAttCols, cc = idx % kAttCols;
      vv[kk2 * (kAttCols + 1) + cc] =
          (k0 + kk2 < s && c0 + cc < e) ? to_f(pre[(long long)(k0 + kk2) * e + c0 + cc]) : 0.f;
    }
    __syncthreads();
    const int kn = min(kAttKeys, s - k0);
    for (int k2 = 0; k2 < kn; ++k2) {
      float a = q[r * sp + k0 + k2];
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = fmaf(a, vv[k2 * (kAttCols + 1) + cg + c], acc[c]);
    }
  }

  const int i = i0 + r;
  if (i < C) {
    const long long row = tok0 + i;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      int col = c0 + cg + c;
      if (col < e) gated[row * e + col] = from_f<T>(to_f(U[row * e + col]) * acc[c]);
    }
  }
}

inline unsigned cdiv(long long a, long long b) { return (unsigned)((a + b - 1) / b); }

template <typename T>
cudaError_t projection(const Problem &p) {
  const int N = 2 * p.e + p.s;
  dim3 grid(cdiv(N, kTile), cdiv(p.M, kTile), 1);
  ProjEpi<T> epi{(T *)p.U, (T *)p.V, (T *)p.heads, p.gamma, p.beta, p.M, p.e, p.s};
  return launch_pdl(simt_gemm<T, ProjEpi<T>>, grid, dim3(256), 0, p.stream, (int)p.M, N, p.d,
                    (const T *)p.A_in, (long long)p.d, 1LL, 0LL, (const T *)p.W_uvz, (long long)N,
                    1LL, 0LL, epi);
}

template <typename T>
cudaError_t chunk_state(const Problem &p) {
  // batch = b*G+g; A(m = si, k = t) = K_lin[t, si]; B(k = t, n) = V[t, n]
  const T *Kl = (const T *)p.heads + 3 * p.M * p.s;
  dim3 grid(cdiv(p.e, kTile), cdiv(p.s, kTile), p.B * p.G);
  StateEpi<T> epi{(T *)p.state, p.s, p.e};
  return launch_pdl(simt_gemm<T, StateEpi<T>>, grid, dim3(256), 0, p.stream, p.s, p.e, p.C, Kl,
                    1LL, (long long)p.s, (long long)p.C * p.s, (const T *)p.V, (long long)p.e, 1LL,
                    (long long)p.C * p.e, epi);
}

template <typename T>
cudaError_t prefix_scan(const Problem &p) {
  long long se = (long long)p.s * p.e;
  return launch_pdl(simt_prefix_scan<T>, dim3(cdiv(p.B * se, 256)), dim3(256), 0, p.stream,
                    (const T *)p.state, (T *)p.prefix, p.B, p.G, se, p.causal, p.lin_scale,
                    p.seg_ids, p.chunk_average, p.per_chunk);
}

size_t attention_smem(int s) {
  const size_t sp = (size_t)s + 1;
  return sizeof(float) * (kAttRows * sp + kAttKeys * sp + (size_t)kAttRows * (kAttKeys + 1) +
                          (size_t)kAttKeys * (kAttCols + 1));
}

template <typename T>
cudaError_t chunk_attention(const Problem &p) {
  const size_t smem = attention_smem(p.s);
  // the shared-memory ceiling for the widest head (s = 128), once per device
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!(configured & (1ull << dev))) {
    err = cudaFuncSetAttribute(simt_chunk_attention<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)attention_smem(128));
    if (err != cudaSuccess) return err;
    configured |= 1ull << dev;
  }
  dim3 grid(cdiv(p.e, kAttCols), cdiv(p.C, kAttRows), p.B * p.G);
  return launch_pdl(simt_chunk_attention<T>, grid, dim3(256), smem, p.stream, (const T *)p.U,
                    (const T *)p.V, (const T *)p.heads, (const T *)p.prefix, p.relpos,
                    (T *)p.gated, p.M, p.C, p.G, p.e, p.s, p.causal, p.local_scale,
                    p.per_chunk);
}

template <typename T>
cudaError_t output(const Problem &p) {
  dim3 grid(cdiv(p.d, kTile), cdiv(p.M, kTile), 1);
  StoreEpi<T> epi{(T *)p.out, p.d, (const T *)p.residual};
  return launch_pdl(simt_gemm<T, StoreEpi<T>>, grid, dim3(256), 0, p.stream, (int)p.M, p.d, p.e,
                    (const T *)p.gated, (long long)p.e, 1LL, 0LL, (const T *)p.W_o, (long long)p.d,
                    1LL, 0LL, epi);
}

}  // namespace

cudaError_t simt_projection_f32(const Problem &p) { return projection<float>(p); }
cudaError_t simt_chunk_state_f32(const Problem &p) { return chunk_state<float>(p); }
cudaError_t simt_prefix_scan_f32(const Problem &p) { return prefix_scan<float>(p); }
cudaError_t simt_chunk_attention_f32(const Problem &p) { return chunk_attention<float>(p); }
cudaError_t simt_output_f32(const Problem &p) { return output<float>(p); }

}  // namespace flashgau
