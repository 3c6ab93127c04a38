// Internal declarations shared by the translation units of libflashgau.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/flash_gau.h"

namespace flashgau {

// One forward call, with every device pointer resolved.
struct Problem {
  int B, T, C, G, d, e, s, causal, dtype;
  long long M;  // B * T tokens
  float lin_scale;
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
  float *state;
  void *prefix;
  void *gated;
  cudaStream_t stream;
  int num_sms;
};

using StageFn = cudaError_t (*)(const Problem &);

struct Stage {
  const char *name;
  StageFn fn;
};

// fp32 SIMT stages (simt_kernels.cu)
cudaError_t simt_projection_f32(const Problem &p);
cudaError_t simt_chunk_state_f32(const Problem &p);
cudaError_t simt_prefix_scan_f32(const Problem &p);
cudaError_t simt_chunk_attention_f32(const Problem &p);
cudaError_t simt_output_f32(const Problem &p);

// bf16 tensor-core stages (tc_gemm.cu)
cudaError_t tc_projection_bf16(const Problem &p);
cudaError_t tc_chunk_state_bf16(const Problem &p);
cudaError_t tc_output_bf16(const Problem &p);

// bf16 tensor-core chunk attention (chunk_attention.cu)
cudaError_t tc_chunk_attention_bf16(const Problem &p);

// bf16 CUDA-core stages
cudaError_t simt_projection_bf16(const Problem &p);
cudaError_t simt_chunk_state_bf16(const Problem &p);
cudaError_t simt_prefix_scan_bf16(const Problem &p);
cudaError_t simt_chunk_attention_bf16(const Problem &p);
cudaError_t simt_output_bf16(const Problem &p);

}  // namespace flashgau
