// Self-test of the bounded waits: one thread waits on something that nothing
// will ever signal and must give up, writing FLASH_GAU_ETIMEOUT into a status
// word, instead of hanging the GPU.  The two forms are the ones the kernels
// use: a shared-memory mbarrier (the TMA / tensor-core pipelines) and a flag
// in global memory (the grid barrier of the chunk-state kernel).
#include "flash_gau_internal.h"
#include "sm103_ptx.cuh"

namespace flashgau {
namespace {

using namespace ptx;

__global__ void bounded_wait_probe(int which, int *words) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  if (which == 0) {
    mbar_init(smem_u32(&bar), 1);  // one arrival expected, none made
    fence_mbar_init();
    if (!mbar_wait(smem_u32(&bar), 0)) atomicExch(&words[0], FLASH_GAU_ETIMEOUT);
  } else {
    const uint64_t t0 = globaltimer();
    while (ld_acquire_gpu(&words[1]) == 0) {  // a flag nothing sets
      if (globaltimer() - t0 > kWaitLimitNs) {
        atomicExch(&words[0], FLASH_GAU_ETIMEOUT);
        break;
      }
      __nanosleep(256);
    }
  }
}

}  // namespace
}  // namespace flashgau

extern "C" int flash_gau_selftest_bounded_wait(int which, int *words, void *stream) {
  if (!words || (which != 0 && which != 1)) return FLASH_GAU_EINVAL;
  flashgau::bounded_wait_probe<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(which, words);
  return cudaGetLastError() == cudaSuccess ? FLASH_GAU_OK : FLASH_GAU_ECUDA;
}
