// Backward pass of the FLASH GAU layer: the gradients of sum(dO * O) with
// respect to X and every parameter ("Transformer Quality in Linear Time",
// Method, eq. 5, eq. 7, eq. 8 and the display after it, differentiated by
// the chain rule).  For bf16 io whose shapes tile, every contraction runs
// on the tcgen05 tensor cores (bf16 operands, fp32 accumulation); fp32 io
// and bf16 shapes that do not tile run them on the CUDA cores in fp32
// (bf16 operands widened as they are loaded):
//
//   recompute  Pre = X W_uvz;  U, V, Z = swish(Pre);  heads = Z gamma + beta
//              S = Qq Kq^T / C + b,  P = relu(S)^2 (masked)      per chunk
//              Vh = l P V + lin_scale Q_lin Prefix_g,  A = U * Vh
//              (l = local_scale)
//   output     dW_o = A^T dO,  dA = dO W_o^T,  dU = dA * Vh,  dVh = dA * U
//   local      dP = l dVh V^T,  dV = l P^T dVh,  dS = 2 relu(S) dP (masked),
//              dQq = dS Kq / C,  dKq = dS^T Qq / C,  db[j-i] += dS[i, j]
//   global     dQl = lin_scale dVh Prefix^T,  dPrefix = lin_scale Ql^T dVh,
//              dState_h = sum_{g>h} dPrefix_g (or the total),
//              dKl = V dState^T,  dV += Kl dState
//   heads      dZ = sum_k dhead_k gamma_k,  dgamma, dbeta = column sums
//   input      dPre = d(U|V|Z) * swish'(Pre),  dX = dPre W_uvz^T,
//              dW_uvz = X^T dPre
//
// The contractions run on one batched, strided GEMM kernel (64 x 64 tiles,
// 4 x 4 per thread), so transposed views cost no copies; the rest are
// elementwise or column-reduction kernels.  For bf16 io, when the shapes
// tile, every contraction runs on the tensor cores instead: the five large
// ones (Pre, dW_o, dA, dX, dW_uvz) on the 2-SM pair GEMM or the general one
// (tc_gemm_pair.cu, tc_gemm_any.cu) and, batched over the chunks, the
// chunk-level ones, with their operands (the gated product, dPre, V, the
// heads, P, dS, dVh, the prefix states and their gradients) rounded to
// bf16 by the kernels that produce them.  There the elementwise steps that
// follow a contraction run in its epilogue: V, Z and the heads in the
// recompute's, A = U * Vh in Vh's, the gate's gradient in dA's (dA is not
// stored), dV * swish'(Pre_v) in dV's; sums and scans stay fp32.
#include <cuda_bf16.h>

#include "flash_gau_internal.h"
#include "sm103_ptx.cuh"

namespace flashgau {
namespace {

// Every kernel of the backward is launched with programmatic dependent
// launch: it may be scheduled while the previous one drains, waits for it
// before touching memory, and lets the next one be scheduled at once.
__device__ __forceinline__ void pdl_enter() {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
}


__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float sigmoid(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float swish(float x) { return x * sigmoid(x); }
__device__ __forceinline__ float swish_grad(float x) {
  const float sg = sigmoid(x);
  return sg * (1.0f + x * (1.0f - sg));
}

// four bf16 values as floats, and back (8-byte accesses)
struct Bf4 {
  __nv_bfloat162 a, b;
};
__device__ __forceinline__ float4 load_bf4(const __nv_bfloat16 *p) {
  const Bf4 v = *reinterpret_cast<const Bf4 *>(p);
  const float2 x = __bfloat1622float2(v.a), y = __bfloat1622float2(v.b);
  return make_float4(x.x, x.y, y.x, y.y);
}
__device__ __forceinline__ void store_bf4(__nv_bfloat16 *p, float a, float b, float c, float d) {
  Bf4 v;
  v.a = __floats2bfloat162_rn(a, b);
  v.b = __floats2bfloat162_rn(c, d);
  *reinterpret_cast<Bf4 *>(p) = v;
}

// ------------------------------------------------------------------ GEMM --
// C[z](m, n) = sum_k A[z / adiv](m, k) B[z / bdiv](k, n), handed to the
// epilogue per element.  Element strides: A(m, k) at m * sam + k * sak, B(k,
// n) at k * sbk + n * sbn; batches z = blockIdx.z.
constexpr int kTile = 64;
constexpr int kTileK = 16;

struct Operand {
  long long sm, sk, sb;  // for B: sm is the k stride and sk the n stride
  int div;
};

template <typename TA, typename TB, typename Epi>
__global__ void __launch_bounds__(256)
bw_gemm(int M, int N, int K, const TA *__restrict__ A, Operand oa, const TB *__restrict__ Bm,
        Operand ob, Epi epi) {
  pdl_enter();
  __shared__ float As[kTileK][kTile + 1];
  __shared__ float Bs[kTileK][kTile + 1];
  const int z = blockIdx.z;
  const int m0 = blockIdx.y * kTile, n0 = blockIdx.x * kTile;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  A += (long long)(z / oa.div) * oa.sb;
  Bm += (long long)(z / ob.div) * ob.sb;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kTileK) {
    for (int idx = threadIdx.x; idx < kTile * kTileK; idx += 256) {
      const int kk = idx % kTileK, mm = idx / kTileK;
      const int gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < M && gk < K) ? to_f(A[gm * oa.sm + gk * oa.sk]) : 0.f;
      const int nn = idx % kTile, kb = idx / kTile;
      const int gn = n0 + nn, gk2 = k0 + kb;
      Bs[kb][nn] = (gn < N && gk2 < K) ? to_f(Bm[gk2 * ob.sm + gn * ob.sk]) : 0.f;
    }
    __syncthreads();
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
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < M && n < N) epi(z, m, n, acc[i][j]);
    }
}

// C[z](m, n) = alpha * acc (+ C when accumulating), fp32
struct StoreF32 {
  float *C;
  long long scm, scn, scb;
  float alpha;
  int accumulate;
  __device__ void operator()(int z, int m, int n, float v) const {
    float *p = C + z * scb + m * scm + n * scn;
    *p = accumulate ? *p + alpha * v : alpha * v;
  }
};

// dX in the io type
template <typename T>
struct StoreIo;
template <>
struct StoreIo<float> {
  float *C;
  long long ld;
  __device__ void operator()(int, int m, int n, float v) const { C[m * ld + n] = v; }
};
template <>
struct StoreIo<__nv_bfloat16> {
  __nv_bfloat16 *C;
  long long ld;
  __device__ void operator()(int, int m, int n, float v) const {
    C[m * ld + n] = __float2bfloat16_rn(v);
  }
};

// scores of chunk z: S = acc / C + relpos[j - i + C - 1], P = relu(S)^2,
// zero above the diagonal when causal
struct ScoreEpi {
  float *S, *P;
  const float *relpos;
  int C, causal;
  float inv_c;
  __device__ void operator()(int z, int i, int j, float v) const {
    const float s = fmaf(v, inv_c, relpos[j - i + C - 1]);
    const long long o = ((long long)z * C + i) * C + j;
    S[o] = s;
    const float r = fmaxf(s, 0.f);
    P[o] = (causal && j > i) ? 0.f : r * r;
  }
};

template <typename TA, typename TB, typename Epi>
cudaError_t gemm(cudaStream_t st, int M, int N, int K, int batches, const TA *A, Operand oa,
                 const TB *Bm, Operand ob, Epi epi) {
  if (M <= 0 || N <= 0 || batches <= 0) return cudaSuccess;
  dim3 grid((N + kTile - 1) / kTile, (M + kTile - 1) / kTile, batches);
  return launch_pdl(bw_gemm<TA, TB, Epi>, grid, dim3(256), 0, st, M, N, K, A, oa, Bm, ob, epi);
}

Operand op(long long sm, long long sk, long long sb = 0, int div = 1) { return {sm, sk, sb, div}; }

// ------------------------------------------------------------ elementwise --
// U, V, Z = swish(Pre) and the four heads Z gamma_k + beta_k (CUDA-core
// path: fp32 Pre, any widths).  V and H are written in fp32 when given, and
// as bf16 copies when V_io / H_io are.
__global__ void act_heads(const float *__restrict__ pre, float *__restrict__ U,
                          float *__restrict__ V, float *__restrict__ Z, float *__restrict__ H,
                          const float *__restrict__ gamma, const float *__restrict__ beta,
                          long long M, int e, int s, __nv_bfloat16 *__restrict__ V_io,
                          __nv_bfloat16 *__restrict__ H_io) {
  pdl_enter();
  const int N = 2 * e + s;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < M * N;
       i += (long long)gridDim.x * blockDim.x) {
    const long long m = i / N;
    const int c = (int)(i - m * N);
    const float y = swish(pre[i]);
    if (c < e) {
      U[m * e + c] = y;
    } else if (c < 2 * e) {
      if (V) V[m * e + c - e] = y;
      if (V_io) V_io[m * e + c - e] = __float2bfloat16_rn(y);
    } else {
      const int k = c - 2 * e;
      Z[m * s + k] = y;
      for (int h = 0; h < 4; ++h) {
        const float v = fmaf(y, gamma[h * s + k], beta[h * s + k]);
        if (H) H[(h * M + m) * s + k] = v;
        if (H_io) H_io[(h * M + m) * s + k] = __float2bfloat16_rn(v);
      }
    }
  }
}

// A = U * Vh (fp32 when A is set, a bf16 copy when A_io is)
__global__ void gate(const float *__restrict__ U, const float *__restrict__ Vh,
                     float *__restrict__ A, __nv_bfloat16 *__restrict__ A_io, long long n) {
  pdl_enter();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float a = U[i] * Vh[i];
    if (A) A[i] = a;
    if (A_io) A_io[i] = __float2bfloat16_rn(a);
  }
}

// dU = dA * Vh, dVh = dA * U (fp32 when dVh is set, a bf16 copy when dVh_io is)
__global__ void gate_grad(const float *__restrict__ dA, const float *__restrict__ U,
                          const float *__restrict__ Vh, float *__restrict__ dU,
                          float *__restrict__ dVh, long long n,
                          __nv_bfloat16 *__restrict__ dVh_io) {
  pdl_enter();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    dU[i] = dA[i] * Vh[i];
    const float g = dA[i] * U[i];
    if (dVh) dVh[i] = g;
    if (dVh_io) dVh_io[i] = __float2bfloat16_rn(g);
  }
}

// the scores from the raw products R = Qq Kq^T of chunk z (in place):
// S = R / C + relpos[j - i + C - 1], and P = relu(S)^2 (zero above the
// diagonal when causal) as a bf16 operand
// Four columns per thread (C a multiple of 4), over the rows z*C + i of the
// [B*G*C, C] score matrices.
// (P_io carries the factor l = local_scale: both contractions that read it
// multiply P by l)
__global__ void score_act(float *__restrict__ S, __nv_bfloat16 *__restrict__ P_io,
                          const float *__restrict__ relpos, long long rows, int C, int causal,
                          float inv_c, float l) {
  pdl_enter();
  const int C4 = C / 4;
  for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < rows * C4;
       q += (long long)gridDim.x * blockDim.x) {
    const long long row = q / C4;
    const int j = 4 * (int)(q - row * C4), i = (int)(row % C);
    float4 v = reinterpret_cast<float4 *>(S)[q];
    const float *rp = relpos + C - 1 - i + j;
    v.x = fmaf(v.x, inv_c, rp[0]);
    v.y = fmaf(v.y, inv_c, rp[1]);
    v.z = fmaf(v.z, inv_c, rp[2]);
    v.w = fmaf(v.w, inv_c, rp[3]);
    reinterpret_cast<float4 *>(S)[q] = v;
    const float r0 = fmaxf(v.x, 0.f), r1 = fmaxf(v.y, 0.f), r2 = fmaxf(v.z, 0.f),
                r3 = fmaxf(v.w, 0.f);
    const bool m = causal != 0;
    store_bf4(P_io + 4LL * q, (m && j > i) ? 0.f : l * (r0 * r0),
              (m && j + 1 > i) ? 0.f : l * (r1 * r1), (m && j + 2 > i) ? 0.f : l * (r2 * r2),
              (m && j + 3 > i) ? 0.f : l * (r3 * r3));
  }
}

// dS = 2 relu(S) dP, zero above the diagonal when causal (in place over dP)
// (blocks along y take the rows of the score matrices)
__global__ void score_grad(const float *__restrict__ S, float *__restrict__ dP, long long rows,
                           int C, int causal, __nv_bfloat16 *__restrict__ dS_io) {
  pdl_enter();
  for (long long row = blockIdx.y; row < rows; row += gridDim.y) {
  const int i = (int)(row % C);
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < C; j += gridDim.x * blockDim.x) {
    const long long o = row * C + j;
    const float v = (causal && j > i) ? 0.f : 2.f * fmaxf(S[o], 0.f) * dP[o];
    dP[o] = v;
    if (dS_io) dS_io[o] = __float2bfloat16_rn(v);
  }
  }
}

// Tensor-core path: dS = 2 relu(S) dP (zero above the diagonal when causal)
// as the bf16 operand of the next contractions, and its diagonal sums
// drelpos[j - i + C - 1] (zeroed first) in one pass.  Four columns per
// thread (C a multiple of 4); a block takes a contiguous range of rows,
// bins its values by offset in shared memory and adds its bins to drelpos.
__global__ void __launch_bounds__(256)
score_grad_relpos(const float *__restrict__ S, const float *__restrict__ dP,
                  __nv_bfloat16 *__restrict__ dS_io, float *__restrict__ drelpos, long long rows,
                  int C, int causal, long long rows_per_block) {
  pdl_enter();
  extern __shared__ float bins[];  // [2C - 1]
  for (int k = threadIdx.x; k < 2 * C - 1; k += blockDim.x) bins[k] = 0.f;
  __syncthreads();
  const int C4 = C / 4;
  const long long r0 = blockIdx.x * rows_per_block;
  const long long r1 = r0 + rows_per_block < rows ? r0 + rows_per_block : rows;
  for (long long q = r0 * C4 + threadIdx.x; q < r1 * C4; q += blockDim.x) {
    const long long row = q / C4;
    const int j = 4 * (int)(q - row * C4), i = (int)(row % C);
    const float4 sv = reinterpret_cast<const float4 *>(S)[q];
    const float4 pv = reinterpret_cast<const float4 *>(dP)[q];
    const bool m = causal != 0;
    const float d0 = (m && j > i) ? 0.f : 2.f * fmaxf(sv.x, 0.f) * pv.x;
    const float d1 = (m && j + 1 > i) ? 0.f : 2.f * fmaxf(sv.y, 0.f) * pv.y;
    const float d2 = (m && j + 2 > i) ? 0.f : 2.f * fmaxf(sv.z, 0.f) * pv.z;
    const float d3 = (m && j + 3 > i) ? 0.f : 2.f * fmaxf(sv.w, 0.f) * pv.w;
    store_bf4(dS_io + 4 * q, d0, d1, d2, d3);
    float *bk = bins + (j - i + C - 1);
    if (d0 != 0.f) atomicAdd(bk, d0);
    if (d1 != 0.f) atomicAdd(bk + 1, d1);
    if (d2 != 0.f) atomicAdd(bk + 2, d2);
    if (d3 != 0.f) atomicAdd(bk + 3, d3);
  }
  __syncthreads();
  for (int k = threadIdx.x; k < 2 * C - 1; k += blockDim.x)
    if (bins[k] != 0.f) atomicAdd(drelpos + k, bins[k]);
}

// drelpos[k] = sum over chunks and over (i, j) with j - i = k - (C - 1).
// A block takes kRelRows consecutive rows of the [B*G*C, C] matrix dS, reads
// them along j (coalesced) into 2C - 1 shared bins by offset, then adds its
// bins to drelpos (zeroed first) with one atomic per bin.
constexpr int kRelRows = 32;
__global__ void relpos_grad(const float *__restrict__ dS, float *__restrict__ drelpos,
                            long long rows, int C) {
  pdl_enter();
  extern __shared__ float bins[];  // [2C - 1]
  for (int k = threadIdx.x; k < 2 * C - 1; k += blockDim.x) bins[k] = 0.f;
  __syncthreads();
  const long long r0 = (long long)blockIdx.x * kRelRows;
  for (int rr = 0; rr < kRelRows && r0 + rr < rows; ++rr) {
    const long long row = r0 + rr;
    const int i = (int)(row % C);
    for (int j = threadIdx.x; j < C; j += blockDim.x)
      atomicAdd(&bins[j - i + C - 1], dS[row * C + j]);
  }
  __syncthreads();
  for (int k = threadIdx.x; k < 2 * C - 1; k += blockDim.x)
    if (bins[k] != 0.f) atomicAdd(drelpos + k, bins[k]);
}

// prefix[b][g] = lin_scale * (exclusive sum over chunks, or the total), in
// fp32 when prefix is set and as bf16 when prefix_io is
__global__ void scan_forward(const float *__restrict__ state, float *__restrict__ prefix, int B,
                             int G, long long se, int causal, float lin_scale,
                             __nv_bfloat16 *__restrict__ prefix_io) {
  pdl_enter();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < B * se;
       i += (long long)gridDim.x * blockDim.x) {
    const long long b = i / se, r = i - b * se;
    float run = 0.f;
    for (int g = 0; g < G; ++g) {
      if (causal) {
        const long long o = (b * G + g) * se + r;
        if (prefix) prefix[o] = lin_scale * run;
        if (prefix_io) prefix_io[o] = __float2bfloat16_rn(lin_scale * run);
      }
      run += state[(b * G + g) * se + r];
    }
    if (!causal) {
      if (prefix) prefix[b * se + r] = lin_scale * run;
      if (prefix_io) prefix_io[b * se + r] = __float2bfloat16_rn(lin_scale * run);
    }
  }
}

// dState_h = sum_{g>h} dPrefix_g (causal) or the total (in place), with the
// lin_scale factor already inside dPrefix
// (with dstate_io set, dState goes only there, as bf16, and dPrefix is left
// as it is)
__global__ void scan_backward(float *__restrict__ dpre, int B, int G, long long se, int causal,
                              __nv_bfloat16 *__restrict__ dstate_io) {
  pdl_enter();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < B * se;
       i += (long long)gridDim.x * blockDim.x) {
    const long long b = i / se, r = i - b * se;
    if (causal) {
      // groups of 8 chunks, last first: the 8 loads issue together
      float run = 0.f;
      for (int g1 = G; g1 > 0; g1 -= 8) {
        const int g0 = g1 - 8 > 0 ? g1 - 8 : 0;
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (g0 + k < g1) v[k] = dpre[(b * G + g0 + k) * se + r];
#pragma unroll
        for (int k = 7; k >= 0; --k) {
          if (g0 + k >= g1) continue;
          const long long o = (b * G + g0 + k) * se + r;
          if (dstate_io) dstate_io[o] = __float2bfloat16_rn(run);
          else dpre[o] = run;
          run += v[k];
        }
      }
    } else {
      float tot = 0.f;
      for (int g = 0; g < G; ++g) tot += dpre[(b * G + g) * se + r];
      for (int g = 0; g < G; ++g) {
        if (dstate_io) dstate_io[(b * G + g) * se + r] = __float2bfloat16_rn(tot);
        else dpre[(b * G + g) * se + r] = tot;
      }
    }
  }
}

// The tensor-core path's scans: four consecutive state elements per thread
// (se a multiple of 4), the loads of 8 chunks issued together, bf16 out.
// prefix_io[b][g] = lin_scale * (exclusive sum over chunks, or the total)
__global__ void scan_forward4(const float4 *__restrict__ state, int B, int G, long long se4,
                              int causal, float lin_scale, __nv_bfloat16 *__restrict__ prefix_io) {
  pdl_enter();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < B * se4;
       i += (long long)gridDim.x * blockDim.x) {
    const long long b = i / se4, r = i - b * se4;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g0 = 0; g0 < G; g0 += 8) {
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (g0 + k < G) v[k] = state[(b * G + g0 + k) * se4 + r];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (g0 + k >= G) continue;
        if (causal)
          store_bf4(prefix_io + 4 * ((b * G + g0 + k) * se4 + r), lin_scale * run.x,
                    lin_scale * run.y, lin_scale * run.z, lin_scale * run.w);
        run = make_float4(run.x + v[k].x, run.y + v[k].y, run.z + v[k].z, run.w + v[k].w);
      }
    }
    if (!causal)
      store_bf4(prefix_io + 4 * (b * se4 + r), lin_scale * run.x, lin_scale * run.y,
                lin_scale * run.z, lin_scale * run.w);
  }
}

// dState_h = sum_{g>h} dPrefix_g (causal) or the total, as bf16
__global__ void scan_backward4(const float4 *__restrict__ dpre, int B, int G, long long se4,
                               int causal, __nv_bfloat16 *__restrict__ dstate_io) {
  pdl_enter();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < B * se4;
       i += (long long)gridDim.x * blockDim.x) {
    const long long b = i / se4, r = i - b * se4;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!causal)
      for (int g = 0; g < G; ++g) {
        const float4 v = dpre[(b * G + g) * se4 + r];
        run = make_float4(run.x + v.x, run.y + v.y, run.z + v.z, run.w + v.w);
      }
    for (int g1 = G; g1 > 0; g1 -= 8) {
      const int g0 = g1 - 8 > 0 ? g1 - 8 : 0;
      float4 v[8];
      if (causal)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (g0 + k < g1) v[k] = dpre[(b * G + g0 + k) * se4 + r];
#pragma unroll
      for (int k = 7; k >= 0; --k) {
        if (g0 + k >= g1) continue;
        store_bf4(dstate_io + 4 * ((b * G + g0 + k) * se4 + r), run.x, run.y, run.z, run.w);
        if (causal) run = make_float4(run.x + v[k].x, run.y + v[k].y, run.z + v[k].z, run.w + v[k].w);
      }
    }
  }
}

// dZ = sum_k dH_k * gamma_k; dgamma, dbeta as column sums of dH_k * Z, dH_k
// (per block partial sums over its rows, added atomically; 256 threads)
__global__ void __launch_bounds__(256)
heads_grad(const float *__restrict__ dH, const float *__restrict__ Z,
           const float *__restrict__ gamma, float *__restrict__ dZ, float *__restrict__ dgamma,
           float *__restrict__ dbeta, long long M, int s, int rows_per_block) {
  pdl_enter();
  // two row parities x 128 columns; the parities meet in shared memory
  __shared__ float red[8][128];
  const int par = threadIdx.x / 128, cl = threadIdx.x % 128;
  const long long r0 = (long long)blockIdx.x * rows_per_block;
  const long long r1 = r0 + rows_per_block < M ? r0 + rows_per_block : M;
  for (int c0 = 0; c0 < s; c0 += 128) {
    const int c = c0 + cl;
    float bsum[4] = {0.f, 0.f, 0.f, 0.f}, gsum[4] = {0.f, 0.f, 0.f, 0.f};
    if (c < s) {
      float g[4];
      for (int k = 0; k < 4; ++k) g[k] = gamma[k * s + c];
#pragma unroll 4
      for (long long m = r0 + par; m < r1; m += 2) {
        const float z = Z[m * s + c];
        float dz = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float dh = dH[((long long)k * M + m) * s + c];
          dz = fmaf(dh, g[k], dz);
          gsum[k] = fmaf(dh, z, gsum[k]);
          bsum[k] += dh;
        }
        dZ[m * s + c] = dz;
      }
    }
    if (par == 1)
      for (int k = 0; k < 4; ++k) {
        red[k][cl] = gsum[k];
        red[4 + k][cl] = bsum[k];
      }
    __syncthreads();
    if (par == 0 && c < s)
      for (int k = 0; k < 4; ++k) {
        atomicAdd(dgamma + k * s + c, gsum[k] + red[k][cl]);
        atomicAdd(dbeta + k * s + c, bsum[k] + red[4 + k][cl]);
      }
    __syncthreads();
  }
}

// dPre = d(U | V | Z) * swish'(Pre), in place over Pre (and its bf16 copy
// when pre_io is set)
__global__ void pre_grad(float *__restrict__ pre, __nv_bfloat16 *__restrict__ pre_io,
                         const float *__restrict__ dU, const float *__restrict__ dV,
                         const float *__restrict__ dZ, long long M, int e, int s) {
  pdl_enter();
  const int N = 2 * e + s;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < M * N;
       i += (long long)gridDim.x * blockDim.x) {
    const long long m = i / N;
    const int c = (int)(i - m * N);
    const float g = c < e ? dU[m * e + c] : c < 2 * e ? dV[m * e + c - e] : dZ[m * s + c - 2 * e];
    const float v = g * swish_grad(pre[i]);
    pre[i] = v;
    if (pre_io) pre_io[i] = __float2bfloat16_rn(v);
  }
}

// act_heads with a bf16 Pre (tensor-core recompute, CUDA-core chunk path)
__global__ void act_heads_bf16(const __nv_bfloat16 *__restrict__ pre, float *__restrict__ U,
                               float *__restrict__ V, float *__restrict__ Z,
                               float *__restrict__ H, const float *__restrict__ gamma,
                               const float *__restrict__ beta, long long M, int e, int s) {
  pdl_enter();
  const int N = 2 * e + s;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < M * N;
       i += (long long)gridDim.x * blockDim.x) {
    const long long m = i / N;
    const int c = (int)(i - m * N);
    const float y = swish(__bfloat162float(pre[i]));
    if (c < e) {
      U[m * e + c] = y;
    } else if (c < 2 * e) {
      V[m * e + c - e] = y;
    } else {
      const int k = c - 2 * e;
      Z[m * s + k] = y;
      for (int h = 0; h < 4; ++h) H[(h * M + m) * s + k] = fmaf(y, gamma[h * s + k], beta[h * s + k]);
    }
  }
}

// The tensor-core path's forms of the kernels above: Pre comes as bf16
// (the recompute GEMM's output, in the dPre buffer), four columns per
// thread (e and s multiples of 4), the sigmoid from the fast exponential
// and division intrinsics (their errors are far below the bf16 rounding of
// Pre), and only the bf16 operands that the tensor-core contractions read
// are written besides Z.

// The tensor-core path keeps no U: U = swish(Pre_u) is recomputed from
// the bf16 Pre wherever it is needed (the values are those that U held,
// swish of the same bf16 inputs).  act_heads_vz writes the V and Z parts'
// operands (V and the heads in bf16, Z in fp32).
__global__ void act_heads_vz(const __nv_bfloat16 *__restrict__ pre, float *__restrict__ Z,
                             const float *__restrict__ gamma, const float *__restrict__ beta,
                             long long M, int e, int s, __nv_bfloat16 *__restrict__ V_io,
                             __nv_bfloat16 *__restrict__ H_io) {
  pdl_enter();
  const int N = 2 * e + s, W4 = (e + s) / 4, e4 = e / 4;  // the V and Z columns
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long i0 = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  long long m = i0 / W4;
  int c4 = (int)(i0 - m * W4);
  const long long dm = stride / W4;
  const int dc = (int)(stride - dm * W4);
  for (long long i = i0; i < M * W4; i += stride) {
    const float4 x = load_bf4(pre + m * N + e + 4 * c4);
    const float4 y = make_float4(swish_fast(x.x), swish_fast(x.y), swish_fast(x.z), swish_fast(x.w));
    if (c4 < e4) {
      store_bf4(V_io + m * e + 4 * c4, y.x, y.y, y.z, y.w);
    } else {
      const int k = 4 * (c4 - e4);
      reinterpret_cast<float4 *>(Z + m * s)[k / 4] = y;
      for (int h = 0; h < 4; ++h) {
        const float *g = gamma + h * s + k, *b = beta + h * s + k;
        store_bf4(H_io + (h * M + m) * s + k, fmaf(y.x, __ldg(g), __ldg(b)),
                  fmaf(y.y, __ldg(g + 1), __ldg(b + 1)), fmaf(y.z, __ldg(g + 2), __ldg(b + 2)),
                  fmaf(y.w, __ldg(g + 3), __ldg(b + 3)));
      }
    }
    m += dm;
    c4 += dc;
    if (c4 >= W4) {
      c4 -= W4;
      ++m;
    }
  }
}

// The Z part of dPre = dZ * swish'(Pre_z), bf16, in place (Pre row stride
// 2e + s; the U and V parts come from the epilogues of the contractions
// that produce dU and dV)
__global__ void pre_grad_z(__nv_bfloat16 *__restrict__ pre_io, const float *__restrict__ dZ,
                           long long M, int e, int s) {
  pdl_enter();
  const int N = 2 * e + s, s4 = s / 4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < M * s4; i += stride) {
    const long long m = i / s4;
    const int c4 = (int)(i - m * s4);
    const float4 g = reinterpret_cast<const float4 *>(dZ)[i];
    __nv_bfloat16 *pz = pre_io + m * N + 2 * e + 4 * c4;
    const float4 x = load_bf4(pz);
    store_bf4(pz, g.x * swish_grad_fast(x.x), g.y * swish_grad_fast(x.y),
              g.z * swish_grad_fast(x.z), g.w * swish_grad_fast(x.w));
  }
}

// A = U * Vh as bf16 only; n4 = elements / 4
__global__ void gate_v4(const float4 *__restrict__ U, const float4 *__restrict__ Vh,
                        __nv_bfloat16 *__restrict__ A_io, long long n4) {
  pdl_enter();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 u = U[i], v = Vh[i];
    store_bf4(A_io + 4 * i, u.x * v.x, u.y * v.y, u.z * v.z, u.w * v.w);
  }
}

// dPre = d(U | V | Z) * swish'(Pre), bf16, in place over the bf16 Pre
__global__ void pre_grad_v4(__nv_bfloat16 *__restrict__ pre_io, const float *__restrict__ dU,
                            const float *__restrict__ dV, const float *__restrict__ dZ,
                            long long M, int e, int s) {
  pdl_enter();
  const int N4 = (2 * e + s) / 4, e4 = e / 4, s4 = s / 4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long i0 = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  long long m = i0 / N4;
  int c4 = (int)(i0 - m * N4);
  const long long dm = stride / N4;
  const int dc = (int)(stride - dm * N4);
  for (long long i = i0; i < M * N4; i += stride) {
    const float4 g = c4 < e4       ? reinterpret_cast<const float4 *>(dU)[m * e4 + c4]
                     : c4 < 2 * e4 ? reinterpret_cast<const float4 *>(dV)[m * e4 + c4 - e4]
                                   : reinterpret_cast<const float4 *>(dZ)[m * s4 + c4 - 2 * e4];
    const float4 x = load_bf4(pre_io + 4 * i);
    store_bf4(pre_io + 4 * i, g.x * swish_grad_fast(x.x), g.y * swish_grad_fast(x.y),
              g.z * swish_grad_fast(x.z), g.w * swish_grad_fast(x.w));
    m += dm;
    c4 += dc;
    if (c4 >= N4) {
      c4 -= N4;
      ++m;
    }
  }
}

// a tensor-core contraction of the backward (bf16 operands)
GemmAnyArgs tc_args(const BackwardProblem &q, const void *A, long long lda, int a_mn,
                    const void *B, long long ldb, int b_km, void *C, int c_bf16, int M, int N,
                    int K, int allow_split) {
  GemmAnyArgs g;
  g.A = A;
  g.lda = lda;
  g.a_mn = a_mn;
  g.B = B;
  g.ldb = ldb;
  g.b_km = b_km;
  g.C = C;
  g.c_bf16 = c_bf16;
  g.M = M;
  g.N = N;
  g.K = K;
  g.accumulate = 0;
  g.allow_split = allow_split;
  g.num_sms = q.num_sms;
  g.status = q.L.status;
  return g;
}

// The gradients summed by atomic or TMA reduce-adds start from zero, all in
// one launch: three small ones element by element, and (the tensor-core
// path's split-K weight gradients, 16-byte aligned, sizes multiples of 4)
// two large ones in 16-byte stores.
__global__ void zero_sums(float *a, int na, float *b, int nb, float *c, int nc, float4 *w1,
                          long long n1, float4 *w2, long long n2) {
  pdl_enter();
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long i0 = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  for (long long i = i0; i < na + nb + nc; i += stride) {
    if (i < na) a[i] = 0.f;
    else if (i < na + nb) b[i - na] = 0.f;
    else c[i - na - nb] = 0.f;
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = i0; i < n1; i += stride) w1[i] = z;
  for (long long i = i0; i < n2; i += stride) w2[i] = z;
}


// blocks of 256 threads over the columns of a row, each block looping over
// rows: at most 2048 blocks along y
dim3 rows_grid(int cols, long long rows) {
  const int bx = (cols + 255) / 256;
  return dim3(bx < 8 ? bx : 8, (unsigned)(rows < 2048 ? rows : 2048));
}

unsigned blocks_for(long long n) {
  const long long b = (n + 255) / 256;
  return (unsigned)(b < 16384 ? b : 16384);
}

template <typename T>
cudaError_t run(const BackwardProblem &q) {
  cudaStream_t st = q.stream;
  const long long M = q.M;
  const int d = q.d, e = q.e, s = q.s, C = q.C, G = q.G, N = 2 * e + s;
  const long long BG = (long long)q.B * G, se = (long long)s * e;
  const T *X = (const T *)q.X, *Wuvz = (const T *)q.W_uvz, *Wo = (const T *)q.W_o;
  const T *dO = (const T *)q.dO;
  const BackwardLayout &L = q.L;
  float *pre = L.pre, *U = L.U, *V = L.V, *Z = L.Z, *H = L.H, *S = L.S, *P = L.P;
  float *Vh = L.Vh, *Ag = L.A, *state = L.state, *prefix = L.prefix, *dA = L.dA, *dU = L.dU;
  float *dVh = L.dVh, *dV = L.dV, *dP = L.dP, *dH = L.dH, *dpre = L.dprefix, *dZ = L.dZ;
  const long long Ms = M * s;
  cudaError_t err;
#define BW_TRY(x)                          \
  do {                                     \
    if ((err = (x)) != cudaSuccess) return err; \
  } while (0)
#define LAUNCH(...) BW_TRY(launch_pdl(__VA_ARGS__));
  // the five large contractions on the tensor cores: bf16 io, shapes that
  // tile 128 x 64 (rows of every output, depths) and 64-wide columns
  const bool tc = sizeof(T) == 2 && M % 128 == 0 && d % 128 == 0 && e % 128 == 0 &&
                  N % 64 == 0 && L.A_io && L.dpre_io;
  __nv_bfloat16 *A_io = tc ? (__nv_bfloat16 *)L.A_io : nullptr;
  __nv_bfloat16 *dpre_io = tc ? (__nv_bfloat16 *)L.dpre_io : nullptr;
  // the chunk-level contractions on the tensor cores too, batched over the
  // chunks: chunks and heads of whole 128-row tiles
  const bool tcc = tc && C % 128 == 0 && s % 128 == 0 && L.H_io && L.V_io && L.P_io &&
                   L.prefix_io && L.dVh_io && L.dS_io && L.dstate_io;
  typedef __nv_bfloat16 bf;
  bf *H_io = tcc ? (bf *)L.H_io : nullptr, *V_io = tcc ? (bf *)L.V_io : nullptr;
  bf *P_io = (bf *)L.P_io, *pre_io = tcc ? (bf *)L.prefix_io : nullptr;
  bf *dVh_io = tcc ? (bf *)L.dVh_io : nullptr, *dS_io = tcc ? (bf *)L.dS_io : nullptr;
  bf *dst_io = tcc ? (bf *)L.dstate_io : nullptr;
  const bf *Qq_io = H_io, *Kq_io = H_io + (tcc ? Ms : 0), *Ql_io = H_io + (tcc ? 2 * Ms : 0);
  const bf *Kl_io = H_io + (tcc ? 3 * Ms : 0);
  // C[z] (+)= alpha A[z] B[z / b_div] for the BG chunks z
  auto bt = [&](const void *A, long long lda, int a_mn, const void *Bm, long long ldb, int b_km,
                float *Cm, int m, int n, int k, int b_div, float alpha, int acc) {
    GemmAnyArgs g = tc_args(q, A, lda, a_mn, Bm, ldb, b_km, Cm, 0, m, n, k, 0);
    g.batches = (int)BG;
    g.b_div = b_div;
    g.alpha = alpha;
    g.accumulate = acc;
    return tc_gemm_any(g, st);
  };
  const int pdiv = q.causal ? 1 : G;  // chunks sharing one prefix state
  // the summed gradients start from zero (the split-K weight gradients of
  // the tensor-core path too, so those contractions need no zeroing)
  {
    const long long n1 = tc ? (long long)e * d / 4 : 0, n2 = tc ? (long long)d * N / 4 : 0;
    LAUNCH(zero_sums, blocks_for(n2 > 2 * C + 8 * s ? n2 : 2 * C + 8 * s), 256, 0, st, q.drelpos,
                      2 * C - 1, q.dgamma, 4 * s, q.dbeta, 4 * s, (float4 *)q.dW_o, n1,
                      (float4 *)q.dW_uvz, n2)
  }
  // ---- recompute the forward
  // (the tensor-core path keeps Pre in bf16, in the buffer of dPre)
  // the forward's 2-SM pair GEMM: with e a multiple of 256 its epilogue also
  // forms V, Z and the heads (then no separate activation pass)
  const bool fused_act = tcc && e % 256 == 0 && s == 128;
  if (fused_act)
    BW_TRY(pair_recompute_bf16(X, Wuvz, q.gamma, q.beta, dpre_io, V_io, Z, H_io, (int)M, d, e, s,
                               L.status, q.num_sms, st));
  else if (tcc)
    BW_TRY(pair_gemm_bf16(X, Wuvz, 0, dpre_io, (int)M, N, d, L.status, q.num_sms, st));
  else if (tc)
    BW_TRY(tc_gemm_any(tc_args(q, X, d, 0, Wuvz, N, 0, dpre_io, 1, (int)M, N, d, 0), st));
  else
    BW_TRY(gemm(st, (int)M, N, d, 1, X, op(d, 1), Wuvz, op(N, 1), StoreF32{pre, N, 1, 0, 1.f, 0}));
  if (fused_act) {
  } else if (tcc)
    LAUNCH(act_heads_vz, blocks_for(M * (e + s) / 4), 256, 0, st, dpre_io, Z, q.gamma, q.beta, M, e,
                                                                  s, V_io, H_io)
  else if (tc)  // bf16 Pre, fp32 heads and V for the CUDA-core chunk contractions
    LAUNCH(act_heads_bf16, blocks_for(M * N), 256, 0, st, dpre_io, U, V, Z, H, q.gamma, q.beta, M, e,
                                                      s)
  else
    LAUNCH(act_heads, blocks_for(M * N), 256, 0, st, pre, U, V, Z, H, q.gamma, q.beta, M, e, s,
                                                 nullptr, nullptr)
  const float *Qq = H, *Kq = H + Ms, *Ql = H + 2 * Ms, *Kl = H + 3 * Ms;
  // per chunk z: rows z*C .. of the [M, *] matrices
  if (tcc) {
    BW_TRY(bt(Qq_io, s, 0, Kq_io, s, 1, S, C, C, s, 1, 1.f, 0));  // raw Qq Kq^T
    LAUNCH(score_act, blocks_for(BG * C * C / 4), 256, 0, st, S, P_io, q.relpos, BG * C, C, q.causal,
                                                           1.f / C, q.local_scale)
    BW_TRY(bt(Kl_io, s, 1, V_io, e, 0, state, s, e, C, 1, 1.f, 0));
  } else {
    BW_TRY(gemm(st, C, C, s, (int)BG, Qq, op(s, 1, (long long)C * s), Kq,
                op(1, s, (long long)C * s), ScoreEpi{S, P, q.relpos, C, q.causal, 1.f / C}));
    BW_TRY(gemm(st, C, e, C, (int)BG, P, op(C, 1, (long long)C * C), V,
                op(e, 1, (long long)C * e), StoreF32{Vh, e, 1, (long long)C * e, q.local_scale, 0}));
    BW_TRY(gemm(st, s, e, C, (int)BG, Kl, op(1, s, (long long)C * s), V,
                op(e, 1, (long long)C * e), StoreF32{state, e, 1, se, 1.f, 0}));
  }
  if (tcc)
    LAUNCH(scan_forward4, blocks_for(q.B * se / 4), 256, 0, st, (const float4 *)state, q.B, G, se / 4,
                                                         q.causal, q.lin_scale, pre_io)
  else
    LAUNCH(scan_forward, blocks_for(q.B * se), 256, 0, st, state, prefix, q.B, G, se, q.causal,
                                                        q.lin_scale, pre_io)
  // Vh (+)= Q_lin Prefix (a chunk's prefix, or its batch row's total)
  if (tcc) {
    // Vh = (l P) V + Q_lin Prefix as one two-product contraction
    // bf16 Vh, and in the epilogue the gated product A = swish(Pre_u) * Vh
    GemmAnyArgs g = tc_args(q, P_io, C, 0, V_io, e, 0, Vh, 1, C, e, C, 0);
    g.batches = (int)BG;
    g.A2 = Ql_io;
    g.lda2 = s;
    g.a2_mn = 0;
    g.B2 = pre_io;
    g.ldb2 = e;
    g.K2 = s;
    g.b2_div = pdiv;
    g.epi = kEpiGate;
    g.E = dpre_io;  // Pre's U columns
    g.lde = N;
    g.D = A_io;
    g.ldd = e;
    BW_TRY(tc_gemm_any(g, st));
  } else {
    const Operand opre = q.causal ? op(e, 1, se) : op(e, 1, se, G);
    BW_TRY(gemm(st, C, e, s, (int)BG, Ql, op(s, 1, (long long)C * s), prefix, opre,
                StoreF32{Vh, e, 1, (long long)C * e, 1.f, 1}));
  }
  if (tcc) {
    // the gate was applied in the epilogue above
  } else if (tc)
    LAUNCH(gate_v4, blocks_for(M * e / 4), 256, 0, st, (const float4 *)U, (const float4 *)Vh, A_io,
                                                    M * e / 4)
  else
    LAUNCH(gate, blocks_for(M * e), 256, 0, st, U, Vh, Ag, nullptr, M * e)
  // ---- output projection and gate
  if (tc) {
    // dW_o = A^T dO: A the transpose of the stored [M, e] gated product
    {
      GemmAnyArgs g = tc_args(q, A_io, e, 1, dO, d, 0, q.dW_o, 0, e, d, (int)M, 1);
      g.c_zeroed = 1;
      BW_TRY(tc_gemm_any(g, st));
    }
    // dA = dO W_o^T: B the transpose of the stored [e, d] W_o.  The
    // tensor-core chunk path forms it on the pair GEMM, whose epilogue
    // takes it straight into the gate's gradient (dVh, and dPre_u over Pre_u)
    if (tcc)
      BW_TRY(pair_gate_grad_bf16(dO, Wo, dpre_io, Vh, dVh_io, (int)M, e, s, d, L.status,
                                 q.num_sms, st));
    else
      BW_TRY(tc_gemm_any(tc_args(q, dO, d, 0, Wo, d, 1, dA, 0, (int)M, e, d, 0), st));
  } else {
    BW_TRY(gemm(st, e, d, (int)M, 1, Ag, op(1, e), dO, op(d, 1),
                StoreF32{q.dW_o, d, 1, 0, 1.f, 0}));
    BW_TRY(gemm(st, (int)M, e, d, 1, dO, op(d, 1), Wo, op(1, d), StoreF32{dA, e, 1, 0, 1.f, 0}));
  }
  if (!tcc)
    LAUNCH(gate_grad, blocks_for(M * e), 256, 0, st, dA, U, Vh, dU, dVh, M * e, nullptr)
  // ---- local part
  if (tcc) {
    // dV = (l P)^T dVh + K_lin dState comes after the reverse scan
    BW_TRY(bt(dVh_io, e, 0, V_io, e, 1, dP, C, C, e, 1, q.local_scale, 0));
  } else {
    BW_TRY(gemm(st, C, C, e, (int)BG, dVh, op(e, 1, (long long)C * e), V,
                op(1, e, (long long)C * e),
                StoreF32{dP, C, 1, (long long)C * C, q.local_scale, 0}));
    BW_TRY(gemm(st, C, e, C, (int)BG, P, op(1, C, (long long)C * C), dVh,
                op(e, 1, (long long)C * e),
                StoreF32{dV, e, 1, (long long)C * e, q.local_scale, 0}));
  }
  if (tcc) {
    const long long rpb = 32;  // rows per block
    LAUNCH(score_grad_relpos, (unsigned)((BG * C + rpb - 1) / rpb), 256, (2 * C - 1) * sizeof(float), st, S, dP, dS_io, q.drelpos, BG * C, C, q.causal, rpb)
  } else {
    LAUNCH(score_grad, rows_grid(C, BG * C), 256, 0, st, S, dP, BG * C, C, q.causal, nullptr)
    LAUNCH(relpos_grad, (unsigned)((BG * C + kRelRows - 1) / kRelRows), 256, (2 * C - 1) * sizeof(float), st, dP, q.drelpos, BG * C, C)
  }
  float *dQq = dH, *dKq = dH + Ms, *dQl = dH + 2 * Ms, *dKl = dH + 3 * Ms;
  if (tcc) {
    BW_TRY(bt(dS_io, C, 0, Kq_io, s, 0, dQq, C, s, C, 1, 1.f / C, 0));
    BW_TRY(bt(dS_io, C, 1, Qq_io, s, 0, dKq, C, s, C, 1, 1.f / C, 0));
  } else {
    BW_TRY(gemm(st, C, s, C, (int)BG, dP, op(C, 1, (long long)C * C), Kq,
                op(s, 1, (long long)C * s), StoreF32{dQq, s, 1, (long long)C * s, 1.f / C, 0}));
    BW_TRY(gemm(st, C, s, C, (int)BG, dP, op(1, C, (long long)C * C), Qq,
                op(s, 1, (long long)C * s), StoreF32{dKq, s, 1, (long long)C * s, 1.f / C, 0}));
  }
  // ---- global part
  if (tcc) {
    BW_TRY(bt(dVh_io, e, 0, pre_io, e, 1, dQl, C, s, e, pdiv, 1.f, 0));
    BW_TRY(bt(Ql_io, s, 1, dVh_io, e, 0, dpre, s, e, C, 1, q.lin_scale, 0));
  } else {
    const Operand opreT = q.causal ? op(1, e, se) : op(1, e, se, G);
    BW_TRY(gemm(st, C, s, e, (int)BG, dVh, op(e, 1, (long long)C * e), prefix, opreT,
                StoreF32{dQl, s, 1, (long long)C * s, 1.f, 0}));
    BW_TRY(gemm(st, s, e, C, (int)BG, Ql, op(1, s, (long long)C * s), dVh,
                op(e, 1, (long long)C * e), StoreF32{dpre, e, 1, se, q.lin_scale, 0}));
  }
  if (tcc)
    LAUNCH(scan_backward4, blocks_for(q.B * se / 4), 256, 0, st, (const float4 *)dpre, q.B, G,
                                                          se / 4, q.causal, dst_io)
  else
    LAUNCH(scan_backward, blocks_for(q.B * se), 256, 0, st, dpre, q.B, G, se, q.causal, dst_io)
  if (tcc) {
    BW_TRY(bt(V_io, e, 0, dst_io, e, 1, dKl, C, s, e, 1, 1.f, 0));
    // dV = (l P)^T dVh + K_lin dState as one two-product contraction; its
    // epilogue writes the V part of dPre = dV * swish'(Pre_v) in place over
    // Pre_v (bf16), so dV itself is never stored
    GemmAnyArgs g = tc_args(q, P_io, C, 1, dVh_io, e, 0, nullptr, 1, C, e, C, 0);
    g.batches = (int)BG;
    g.A2 = Kl_io;
    g.lda2 = s;
    g.a2_mn = 0;
    g.B2 = dst_io;
    g.ldb2 = e;
    g.K2 = s;
    g.b2_div = 1;
    g.epi = kEpiSwishGrad;
    g.E = dpre_io + e;
    g.lde = N;
    g.D = dpre_io + e;
    g.ldd = N;
    BW_TRY(tc_gemm_any(g, st));
  } else {
    BW_TRY(gemm(st, C, s, e, (int)BG, V, op(e, 1, (long long)C * e), dpre, op(1, e, se),
                StoreF32{dKl, s, 1, (long long)C * s, 1.f, 0}));
    BW_TRY(gemm(st, C, e, s, (int)BG, Kl, op(s, 1, (long long)C * s), dpre, op(e, 1, se),
                StoreF32{dV, e, 1, (long long)C * e, 1.f, 1}));
  }
  // ---- heads
  const int rows = 32;  // about 3 blocks a SM at the long workload's 16k rows
  LAUNCH(heads_grad, (unsigned)((M + rows - 1) / rows), 256, 0, st, dH, Z, q.gamma, dZ, q.dgamma,
                                                                q.dbeta, M, s, rows)
  // ---- input side
  if (tcc)  // the U part came from the dA contraction, the V part from the dV one
    LAUNCH(pre_grad_z, blocks_for(M * s / 4), 256, 0, st, dpre_io, dZ, M, e, s)
  else if (tc)
    LAUNCH(pre_grad_v4, blocks_for(M * N / 4), 256, 0, st, dpre_io, dU, dV, dZ, M, e, s)
  else
    LAUNCH(pre_grad, blocks_for(M * N), 256, 0, st, pre, nullptr, dU, dV, dZ, M, e, s)
  if (tc) {
    // dX = dPre W_uvz^T (bf16 out); dW_uvz = X^T dPre
    if (tcc)  // on the pair GEMM (d a multiple of 128)
      BW_TRY(pair_gemm_bf16(dpre_io, Wuvz, 1, q.dX, (int)M, d, N, L.status, q.num_sms, st));
    else
      BW_TRY(tc_gemm_any(tc_args(q, dpre_io, N, 0, Wuvz, N, 1, q.dX, 1, (int)M, d, N, 0), st));
    GemmAnyArgs g = tc_args(q, X, d, 1, dpre_io, N, 0, q.dW_uvz, 0, d, N, (int)M, 1);
    g.c_zeroed = 1;
    BW_TRY(tc_gemm_any(g, st));
  } else {
    BW_TRY(gemm(st, (int)M, d, N, 1, (const float *)pre, op(N, 1), Wuvz, op(1, N),
                StoreIo<T>{(T *)q.dX, d}));
    BW_TRY(gemm(st, d, N, (int)M, 1, X, op(1, d), (const float *)pre, op(N, 1),
                StoreF32{q.dW_uvz, N, 1, 0, 1.f, 0}));
  }
#undef LAUNCH
#undef BW_TRY
  return cudaGetLastError();
}

}  // namespace

cudaError_t backward_f32(const BackwardProblem &q) { return run<float>(q); }
cudaError_t backward_bf16(const BackwardProblem &q) { return run<__nv_bfloat16>(q); }

}  // namespace flashgau
