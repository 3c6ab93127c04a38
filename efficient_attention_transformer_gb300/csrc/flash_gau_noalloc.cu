// flash_gau_forward_noalloc: the forward pass with its workspace in a static
// device array instead of caller memory, for callers that cannot allocate
// device memory where they run the layer.  It runs the unchanged
// flash_gau_forward on that array.
#include <mutex>

#include "flash_gau_internal.h"

using namespace flashgau;

namespace {

constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FLASH_GAU_NOALLOC_SCRATCH_BYTES];

void *g_scratch_addr[kMaxDevices];  // device address per device ordinal
std::mutex g_scratch_mu;

}  // namespace

extern "C" int flash_gau_forward_noalloc(const void *X, const flash_gau_weights *w, int B, int T,
                                         int C, int causal, int dtype, void *out, void *stream) {
  causal = causal ? 1 : 0;
  // Every argument check of flash_gau_forward comes first, so that a
  // rejected call leaves the shared array (and its status word) untouched.
  flash_gau_workspace_layout L;
  int num_sms = 0;
  int st = check_forward(X, w, B, T, C, causal, dtype, out, nullptr, 0, &L, &num_sms);
  if (st != FLASH_GAU_OK) return st;
  if (L.total_bytes > FLASH_GAU_NOALLOC_SCRATCH_BYTES) return FLASH_GAU_EWORKSPACE;

  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return record_cuda(err);
  if (dev < 0 || dev >= kMaxDevices) return FLASH_GAU_EDEVICE;
  void *scratch = nullptr;
  {
    // once per device, with that device current
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void *ptr = nullptr;
      err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (err != cudaSuccess) return record_cuda(err);
      if (!ptr) return FLASH_GAU_ECUDA;
      g_scratch_addr[dev] = ptr;
    }
    scratch = g_scratch_addr[dev];
  }
  st = check_forward(X, w, B, T, C, causal, dtype, out, scratch, FLASH_GAU_NOALLOC_SCRATCH_BYTES,
                     &L, &num_sms);
  if (st != FLASH_GAU_OK) return st;
  // The status word is the only part of the workspace that must start at
  // zero; every intermediate is fully rewritten by the kernels.
  err = cudaMemsetAsync(static_cast<char *>(scratch) + L.status, 0, sizeof(int),
                        static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return record_cuda(err);
  return flash_gau_forward(X, w, B, T, C, causal, dtype, out, scratch,
                           FLASH_GAU_NOALLOC_SCRATCH_BYTES, stream);
}
