// flash_gau_forward_host: the forward pass on host buffers.  The input is
// copied to the device, the layer runs, and the output is copied back, with
// the copies of one part of the batch overlapping the computation of
// another: batch rows are independent problems, so the batch is cut into up
// to kMaxParts parts, and
//   copy stream     X part 0 in | X part 1 in | ...
//   caller stream               | layer part 0 | layer part 1 | ...
//   copy stream 2                              | O part 0 out | O part 1 out
// The caller's stream is joined to the last output copy before the call
// returns, so synchronising that stream covers everything; work queued on
// it before the call happens first.  The two copy streams and the events
// are created once per device (no device memory) and shared by the calls
// on that device, under a lock held while a call enqueues its work.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "flash_gau_internal.h"

namespace flashgau {
namespace {

constexpr int kMaxParts = 4;
constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct HostResources {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in_done[kMaxParts] = {}, comp_done[kMaxParts] = {};
  bool ready = false;
};
HostResources g_res[kMaxDevices];
std::mutex g_host_mu;

cudaError_t make_resources(HostResources *r) {
  cudaError_t err;
  if ((err = cudaStreamCreateWithFlags(&r->in, cudaStreamNonBlocking)) != cudaSuccess) return err;
  if ((err = cudaStreamCreateWithFlags(&r->out, cudaStreamNonBlocking)) != cudaSuccess) return err;
  if ((err = cudaEventCreateWithFlags(&r->start, cudaEventDisableTiming)) != cudaSuccess) return err;
  if ((err = cudaEventCreateWithFlags(&r->done, cudaEventDisableTiming)) != cudaSuccess) return err;
  for (int p = 0; p < kMaxParts; ++p) {
    if ((err = cudaEventCreateWithFlags(&r->in_done[p], cudaEventDisableTiming)) != cudaSuccess)
      return err;
    if ((err = cudaEventCreateWithFlags(&r->comp_done[p], cudaEventDisableTiming)) != cudaSuccess)
      return err;
  }
  r->ready = true;
  return cudaSuccess;
}

// Parts of the batch: as many as kMaxParts, at least one row each.
int num_parts(int B) { return B < kMaxParts ? B : kMaxParts; }
int part_rows(int B) { return (B + num_parts(B) - 1) / num_parts(B); }

// Device bytes: X and O for the whole batch, then the layer's workspace for
// the largest part.  0 when the arguments are invalid.
size_t host_bytes(int B, int T, int C, const flash_gau_weights *w, int causal, int dtype,
                  size_t *x_bytes, size_t *fwd_bytes) {
  if (!w || B <= 0 || T <= 0) return 0;
  const size_t fwd = flash_gau_workspace_bytes(part_rows(B), T, C, w, causal, dtype);
  if (fwd == 0) return 0;
  const size_t io = dtype == FLASH_GAU_BF16 ? 2 : 4;
  const size_t xb = (size_t)B * T * w->d * io;
  if (x_bytes) *x_bytes = xb;
  if (fwd_bytes) *fwd_bytes = fwd;
  return 2 * align_up(xb) + fwd;
}

}  // namespace
}  // namespace flashgau

using namespace flashgau;

extern "C" {

size_t flash_gau_forward_host_workspace_bytes(int B, int T, int C, const flash_gau_weights *w,
                                              int causal, int dtype) {
  return host_bytes(B, T, C, w, causal ? 1 : 0, dtype, nullptr, nullptr);
}

int flash_gau_forward_host(const void *X_host, const flash_gau_weights *w, int B, int T, int C,
                           int causal, int dtype, void *out_host, void *workspace,
                           size_t workspace_bytes, void *stream) {
  if (!X_host || !w || !out_host || !workspace) return FLASH_GAU_EINVAL;
  causal = causal ? 1 : 0;
  size_t xb = 0, fwd = 0;
  const size_t need = host_bytes(B, T, C, w, causal, dtype, &xb, &fwd);
  if (need == 0) {
    // the same status as the device-buffer forward for these arguments
    flash_gau_workspace_layout L;
    const int st = flash_gau_workspace_layout_query(B, T, C, w->d, w->e, w->s, causal, dtype, &L);
    return st != FLASH_GAU_OK ? st : FLASH_GAU_EINVAL;
  }
  if (workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % kAlign != 0)
    return FLASH_GAU_EWORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLASH_GAU_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return FLASH_GAU_EDEVICE;

  char *ws = static_cast<char *>(workspace);
  char *Xd = ws, *Od = ws + align_up(xb), *fws = ws + 2 * align_up(xb);
  const char *Xh = static_cast<const char *>(X_host);
  char *Oh = static_cast<char *>(out_host);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int parts = num_parts(B), rows = part_rows(B);
  const size_t row_bytes = xb / B;

  std::lock_guard<std::mutex> lock(g_host_mu);
  HostResources &r = g_res[dev];
  cudaError_t err;
  if (!r.ready && (err = make_resources(&r)) != cudaSuccess) return FLASH_GAU_ECUDA;
#define HOST_TRY(x) \
  do { \
    if ((err = (x)) != cudaSuccess) return FLASH_GAU_ECUDA; \
  } while (0)
  // everything after the work already queued on the caller's stream
  HOST_TRY(cudaEventRecord(r.start, st));
  HOST_TRY(cudaStreamWaitEvent(r.in, r.start, 0));
  HOST_TRY(cudaStreamWaitEvent(r.out, r.start, 0));
  for (int p = 0; p < parts; ++p) {
    const int b0 = p * rows, nb = b0 + rows <= B ? rows : B - b0;
    if (nb <= 0) break;
    HOST_TRY(cudaMemcpyAsync(Xd + b0 * row_bytes, Xh + b0 * row_bytes, nb * row_bytes,
                             cudaMemcpyHostToDevice, r.in));
    HOST_TRY(cudaEventRecord(r.in_done[p], r.in));
  }
  for (int p = 0; p < parts; ++p) {
    const int b0 = p * rows, nb = b0 + rows <= B ? rows : B - b0;
    if (nb <= 0) break;
    HOST_TRY(cudaStreamWaitEvent(st, r.in_done[p], 0));
    const int rc = flash_gau_forward(Xd + b0 * row_bytes, w, nb, T, C, causal, dtype,
                                     Od + b0 * row_bytes, fws, fwd, stream);
    if (rc != FLASH_GAU_OK) return rc;
    HOST_TRY(cudaEventRecord(r.comp_done[p], st));
    HOST_TRY(cudaStreamWaitEvent(r.out, r.comp_done[p], 0));
    HOST_TRY(cudaMemcpyAsync(Oh + b0 * row_bytes, Od + b0 * row_bytes, nb * row_bytes,
                             cudaMemcpyDeviceToHost, r.out));
  }
  HOST_TRY(cudaEventRecord(r.done, r.out));
  HOST_TRY(cudaStreamWaitEvent(st, r.done, 0));
#undef HOST_TRY
  return FLASH_GAU_OK;
}

}  // extern "C"
