// Internal declarations shared by the translation units of libflashgau.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/flash_gau.h"

namespace flashgau {

// RoPE of pair i at position pos: the angle pos * base^(-2i/s).  Positions
// reach the thousands, so a plain fp32 product would lose the angle's low
// bits, and fp64 arithmetic is slow on this GPU.  The host gives each
// pair's frequency in turns, phi_i = base^(-2i/s) / (2 pi), as an fp32
// hi + lo pair (computed in double); pos * phi is formed exactly enough
// with an fma-based product, its integer turns dropped, and the fraction
// goes to sincospif.
constexpr int kMaxRopePairs = 64;
struct RopeTable {
  float2 phi[kMaxRopePairs];  // (hi, lo) of base^(-2i/s) / (2 pi)
};
__device__ __forceinline__ void rope_sincos(float pos, float2 phi, float *sn, float *cs) {
  const float t_hi = pos * phi.x;
  const float t_lo = fmaf(pos, phi.y, fmaf(pos, phi.x, -t_hi));  // exact product error
  const float f = (t_hi - rintf(t_hi)) + t_lo;                   // turns, |f| <~ 0.5
  sincospif(2.0f * f, sn, cs);
}
// Fills the table for head width s and the given base (host side).
void rope_table(RopeTable *tab, int s, float base);

// Keeps the message of a failed CUDA call for flash_gau_strerror and returns
// FLASH_GAU_ECUDA.
int record_cuda(cudaError_t err);

// Every host-side check of one forward call before its first launch:
// pointers and factors, the shape (filling *L with the workspace layout),
// out against X, and the current device (filling *num_sms).  With a
// non-null workspace, also its size, alignment and overlap with out.
int check_forward(const void *X, const flash_gau_weights *w, int B, int T, int C, int causal,
                  int dtype, const void *out, const void *workspace, size_t workspace_bytes,
                  flash_gau_workspace_layout *L, int *num_sms);

// One forward call, with every device pointer resolved.
struct Problem {
  int B, T, C, G, d, e, s, causal, dtype;
  long long M;  // B * T tokens
  float lin_scale;
  float local_scale;  // factor on the local term; 0 = global term only
  // bf16 without a chunk mask whose global term is zero for every chunk
  // (lin_scale 0, or causal with a single chunk, where the only prefix is
  // the empty sum) and whose local term is not: no chunk states, no prefix
  int lin_off;
  // chunk mask of the global term: segment ids [B, G] (null: one segment)
  // and row normalisation; per_chunk: a prefix state per chunk (causal or
  // segmented), else one per batch row
  const int *seg_ids;
  int chunk_average, per_chunk;
  const void *X;
  const void *W_uvz;
  const void *W_o;
  const float *gamma;
  const float *beta;
  const float *relpos;
  void *out;
  // workspace regions
  int *status;
  void *U;
  void *V;
  void *heads;  // [4][M][s]
  void *state;  // [B, G, s, e] io type
  void *prefix;
  void *gated;
  float *bias;  // [2C-1] relpos, causal entries of offset j-i >= 1 set to -inf
  // flash_block options: the projection reads A_in (X, or the normalised
  // input xn); rope rotates the heads; residual (X or null) is added to O
  const void *A_in;
  void *xn;
  int norm;
  const float *norm_g, *norm_b;
  float norm_eps;
  int rope;
  float rope_base;
  int pos_offset;
  RopeTable rope_tab;  // filled when rope is set
  void *rope_cs;       // [s / 2][T] half2 (cos, sin), bf16 path
  const void *residual;
  cudaStream_t stream;
  int num_sms;
};

// The status word's 256-byte workspace slot also holds, at these int
// offsets, the work counter of the chunk-attention kernel and the arrival
// counter of the chunk-state kernel's grid barrier; the projection kernel
// zeroes both.
constexpr int kNextUnitWord = 16;

// The bf16 path keeps V, the chunk states and the prefix states in 64 x 64
// blocks, row-block-major: block (i, j) of a [rows, cols] matrix is 8 KB of
// row-major data at block index i * (cols / 64) + j.  Seen as a flat matrix
// of 128-byte rows ([rows * cols / 64, 64]), element (r, c) sits in flat row
// rb64_row(r, c, cols / 64), column c % 64; 64 rows of 64 k adjacent column
// blocks are 64 k consecutive flat rows, one contiguous TMA box.
__host__ __device__ inline long long rb64_row(long long r, long long c, long long ncb) {
  return ((r >> 6) * ncb + (c >> 6)) * 64 + (r & 63);
}
constexpr int kGridBarrierWord = 17;


// General tcgen05 GEMM (tc_gemm_any.cu): C[M, N] = A B, bf16 operands.
enum { kEpiNone = 0, kEpiGate = 1, kEpiSwishGrad = 2 };

#ifdef __CUDACC__
// The backward's activation arithmetic: the sigmoid from the fast
// exponential and reciprocal
__device__ __forceinline__ float sigmoid_fast(float x) {
  return __fdividef(1.0f, 1.0f + __expf(-x));
}
__device__ __forceinline__ float swish_fast(float x) { return x * sigmoid_fast(x); }
__device__ __forceinline__ float swish_grad_fast(float x) {
  const float sg = sigmoid_fast(x);
  return sg * (1.0f + x * (1.0f - sg));
}
#endif

struct GemmAnyArgs {
  const void *A;
  long long lda;
  int a_mn;  // A is the transpose of a row-major [K, M] matrix
  const void *B;
  long long ldb;
  int b_km;  // B is the transpose of a row-major [N, K] matrix
  void *C;   // row-major [M, N], leading dimension N
  int c_bf16;
  int M, N, K;
  int accumulate;   // fp32: add into C
  int allow_split;  // fp32: split K across CTAs when the tiles are few
  int c_zeroed = 0; // C is known to be zero: a split needs no zeroing first
  int num_sms;
  int *status;
  // batched: `batches` independent products, each operand's batch z stored
  // right after batch z-1 (A: M or K rows, B: K or N rows, C: M rows, as
  // the operand is stored); B's batch is z / b_div (a shared operand)
  int batches = 1;
  int b_div = 1;
  float alpha = 1.f;  // fp32 output: C (+)= alpha * A B
  // optional second product summed into the same tile: C = A B + A2 B2,
  // K2 deep (a multiple of 64), A2 of its own majorness, B2 stored as B,
  // batched like A and B (B2's batch z / b2_div); K2 = 0: none
  const void *A2 = nullptr;
  long long lda2 = 0;
  int a2_mn = 0;
  const void *B2 = nullptr;
  long long ldb2 = 0;
  int K2 = 0;
  int b2_div = 1;
  // optional elementwise epilogue (bf16 C only) with an operand E and a
  // result D, both bf16 with C's rows and columns (leading dimensions lde,
  // ldd): kEpiGate stores C and D = swish(E) * C; kEpiSwishGrad stores
  // D = C * swish'(E) only (C is then not written, and D may be E itself).
  // C's values enter as rounded to bf16.
  int epi = 0;
  const void *E = nullptr;
  long long lde = 0;
  void *D = nullptr;
  long long ldd = 0;
};
cudaError_t tc_gemm_any(const GemmAnyArgs &g, cudaStream_t stream);

// C[M, N] = A[M, K] B[K, N], bf16 operands and output, on the 2-SM pair
// GEMM of the forward (tc_gemm_pair.cu): A and C row-major, B a row-major
// [K, N] matrix or (b_km) the transpose of a row-major [N, K] one; M a
// multiple of 128, N of 128, K of 64.
cudaError_t pair_gemm_bf16(const void *A, const void *B, int b_km, void *C, int M, int N, int K,
                           int *status, int num_sms, cudaStream_t stream);
// The backward's recompute on the pair GEMM: Pre = X W_uvz as bf16 [M,
// 2e + s], and from its bf16 values V_io = swish (bf16 [M, e]), Z = swish
// (fp32 [M, s]) and the four heads H_io = Z gamma_h + beta_h (bf16 [4, M,
// s]); M a multiple of 128, e of 256, s = 128.
// dVh = dA * swish(Pre_u) and dPre_u = (dA * Vh) * swish'(Pre_u) (over Pre_u
// in place, Pre's rows 2e + s wide) with dA = dO W_o^T formed on the pair
// GEMM and not stored; M a multiple of 128, e of 128, d of 64
cudaError_t pair_gate_grad_bf16(const void *dO, const void *W_o, void *pre, const void *Vh,
                                void *dVh, int M, int e, int s, int d, int *status, int num_sms,
                                cudaStream_t stream);
cudaError_t pair_recompute_bf16(const void *X, const void *W_uvz, const float *gamma,
                                const float *beta, void *pre, void *V_io, float *Z, void *H_io,
                                int M, int d, int e, int s, int *status, int num_sms,
                                cudaStream_t stream);

// Decode step (decode.cu): the per-sequence state, all fp32 but pos.
struct DecodeLayout {
  int *status;     // the state's first slot
  int *pos;        // [B] tokens consumed
  float *prefix;   // [B, s, e] sum of completed chunks' K_lin^T V
  float *kq, *kl;  // [B, C, s] the current chunk's K_quad, K_lin rows
  float *vc;       // [B, C, e] the current chunk's V rows
  float *proj;     // [slices, B, 2e+s] this step's x W_uvz, by depth slice
  float *gated;    // [B, e]
  void *gated_io;  // [B, e] io-type copy of gated (bf16: the tensor-core projection's operand)
  float *outp;     // [slices, B, d] this step's gated W_o, by depth slice
  float *heads;    // [B, 4, s] this step's four heads
  float *score;    // [B, C] this step's chunk weights a_j (local_scale included)
};
// Depth slices of the decode step's split-K matrix-vector product with a
// [K, N] weight: about 150 blocks of 256 columns x one slice, but at most 16
// slices (their consumers add the slices one after another), at most 128
// rows a slice.
inline int decode_slices(int K, int N) {
  const int tiles = (N + 255) / 256;
  int sl = (150 + tiles - 1) / tiles;
  if (sl > 16) sl = 16;
  const int lo = (K + 127) / 128, hi = (K + 7) / 8;
  if (sl < lo) sl = lo;
  if (sl > hi) sl = hi;
  return sl < 1 ? 1 : sl;
}
// The bf16 decode step's projections on the tensor cores: y^T = W^T x^T,
// 128 weight columns (TMEM lanes) x the sequences (up to 256, padded to 16)
// per block, over a depth slice of kbs 64-row k-blocks (at most 4), about
// 150 blocks; returns the number of slices.
constexpr int kDecodeTcMaxB = 256;
inline int decode_tc_slices(int K, int N, int *kbs) {
  const int nkb = (K + 63) / 64, tiles = (N + 127) / 128;
  int sl = (150 + tiles - 1) / tiles;
  if (sl > nkb) sl = nkb;
  int kb = (nkb + sl - 1) / sl;
  if (kb > 4) kb = 4;
  if (kbs) *kbs = kb;
  return (nkb + kb - 1) / kb;
}
struct DecodeProblem {
  int B, C, d, e, s;
  float lin_scale, local_scale;
  const void *x, *W_uvz, *W_o;
  const float *gamma, *beta, *relpos;
  void *out;
  DecodeLayout L;
  cudaStream_t stream;
};
cudaError_t decode_step_f32(const DecodeProblem &q);
cudaError_t decode_step_bf16(const DecodeProblem &q);

// Backward pass (backward.cu): fp32 work buffers in the caller's workspace.
struct BackwardLayout {
  int *status;    // the workspace's first slot: FLASH_GAU_ETIMEOUT on a timed-out wait
  float *pre;     // [M, 2e+s] X W_uvz, then its gradient
  float *U, *V;   // [M, e]
  float *Z;       // [M, s]
  float *H;       // [4, M, s] Q_quad, K_quad, Q_lin, K_lin
  float *S, *P;   // [B*G, C, C] scores, relu^2 weights
  float *Vh, *A;  // [M, e] V_quad + V_lin, the gated product
  float *state;   // [B*G, s, e]
  float *prefix;  // [B*G or B, s, e], lin_scale included
  float *dA, *dU, *dVh, *dV;  // [M, e]
  float *dP;      // [B*G, C, C], then dS
  float *dH;      // [4, M, s]
  float *dprefix; // [B*G, s, e], then dState
  float *dZ;      // [M, s]
  void *A_io;     // [M, e] bf16 copy of the gated product (tensor-core path)
  void *dpre_io;  // [M, 2e+s] bf16 copy of dPre (tensor-core path)
  // bf16 operand copies of the chunk-level contractions (tensor-core path)
  void *H_io;       // [4, M, s]
  void *V_io;       // [M, e]
  void *P_io;       // [B*G, C, C]
  void *prefix_io;  // [B*G or B, s, e]
  void *dVh_io;     // [M, e]
  void *dS_io;      // [B*G, C, C]
  void *dstate_io;  // [B*G, s, e]
};
struct BackwardProblem {
  int B, T, C, G, d, e, s, causal;
  long long M;
  float lin_scale, local_scale;
  const void *X, *dO, *W_uvz, *W_o;
  const float *gamma, *beta, *relpos;
  void *dX;
  float *dW_uvz, *dW_o, *dgamma, *dbeta, *drelpos;
  BackwardLayout L;
  cudaStream_t stream;
  int num_sms;
};
cudaError_t backward_f32(const BackwardProblem &q);
cudaError_t backward_bf16(const BackwardProblem &q);

using StageFn = cudaError_t (*)(const Problem &);

// Launches `kernel` on the problem's stream with programmatic stream
// serialisation, so that it may start while the previous kernel drains; the
// kernel itself waits (griddepcontrol.wait) before touching data that the
// previous kernels produce or consume.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

struct Stage {
  const char *name;
  StageFn fn;
};

// flash_block stages (block_kernels.cu): the pre-norm into xn, and for fp32
// the RoPE rotation of the heads in place
cudaError_t block_norm(const Problem &p);
cudaError_t rope_table_stage(const Problem &p);
cudaError_t simt_rope_heads_f32(const Problem &p);
// the relative-position table of the RoPE bias construction (block_kernels.cu)
cudaError_t rope_toeplitz_bias(const float *a, const float *b, int m, int C, float base,
                               float *relpos, cudaStream_t stream);

// fp32 SIMT stages (simt_kernels.cu)
cudaError_t simt_projection_f32(const Problem &p);
cudaError_t simt_chunk_state_f32(const Problem &p);
cudaError_t simt_prefix_scan_f32(const Problem &p);
cudaError_t simt_chunk_attention_f32(const Problem &p);
cudaError_t simt_output_f32(const Problem &p);

// bf16 tensor-core stages: projection and output (tc_gemm_pair.cu), chunk
// states followed by their prefix scan (tc_gemm.cu)
cudaError_t tc_projection_bf16(const Problem &p);
cudaError_t tc_chunk_state_scan_bf16(const Problem &p);
cudaError_t tc_output_bf16(const Problem &p);

// bf16 tensor-core chunk attention (chunk_attention.cu)
cudaError_t tc_chunk_attention_bf16(const Problem &p);

}  // namespace flashgau
