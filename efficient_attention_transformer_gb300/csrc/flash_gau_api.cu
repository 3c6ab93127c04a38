// C ABI of libflashgau: argument validation, workspace layout and the stage
// schedule of one forward pass.  Every launch happens on the caller's stream.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "flash_gau_internal.h"

using namespace flashgau;

namespace {
thread_local char g_cuda_msg[256] = "no CUDA error recorded";
}  // namespace

int flashgau::record_cuda(cudaError_t err) {
  snprintf(g_cuda_msg, sizeof(g_cuda_msg), "CUDA error %d: %s", (int)err,
           cudaGetErrorString(err));
  return FLASH_GAU_ECUDA;
}

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Per-device facts looked up once: compute capability and SM count.
struct DeviceInfo {
  int checked = 0;
  int ok = 0;
  int num_sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(int *num_sms) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return record_cuda(err);
  if (dev < 0 || dev >= kMaxDevices) return FLASH_GAU_EDEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo &di = g_dev[dev];
  if (!di.checked) {
    int major = 0, minor = 0, sms = 0;
    if ((err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return record_cuda(err);
    di.ok = (major == 10 && minor == 3);
    di.num_sms = sms;
    di.checked = 1;
  }
  if (!di.ok) return FLASH_GAU_EDEVICE;
  *num_sms = di.num_sms;
  return FLASH_GAU_OK;
}

int check_shape(int B, int T, int C, int d, int e, int s, int dtype) {
  if (B <= 0 || T <= 0 || C <= 0 || d <= 0 || e <= 0 || s <= 0) return FLASH_GAU_EINVAL;
  if (T % C != 0) return FLASH_GAU_EINVAL;
  if (dtype != FLASH_GAU_FP32 && dtype != FLASH_GAU_BF16) return FLASH_GAU_EINVAL;
  if ((long long)B * T > (1LL << 30) || d > (1 << 16) || e > (1 << 16) || s > (1 << 16))
    return FLASH_GAU_ENOTSUP;
  if (C > 4096) return FLASH_GAU_ENOTSUP;
  if ((long long)B * (T / C) > 65535) return FLASH_GAU_ENOTSUP;
  if (dtype == FLASH_GAU_FP32) {
    if (s > 128) return FLASH_GAU_ENOTSUP;
  } else {
    if (d % 128 != 0 || e % 256 != 0 || s != 128 || C % 128 != 0) return FLASH_GAU_ENOTSUP;
  }
  return FLASH_GAU_OK;
}

int layout(int B, int T, int C, int d, int e, int s, int causal, int dtype,
           flash_gau_workspace_layout *L) {
  int st = check_shape(B, T, C, d, e, s, dtype);
  if (st != FLASH_GAU_OK) return st;
  const size_t io = dtype == FLASH_GAU_BF16 ? 2 : 4;
  const size_t M = (size_t)B * T, G = (size_t)(T / C);
  size_t off = 0;
  L->status = off;
  off = align_up(off + sizeof(int));
  L->U = off;
  off = align_up(off + M * e * io);
  L->V = off;
  off = align_up(off + M * e * io);
  L->heads = off;
  off = align_up(off + 4 * M * s * io);
  L->state = off;
  off = align_up(off + (size_t)B * G * s * e * io);
  L->prefix = off;
  off = align_up(off + (size_t)B * G * s * e * io);  // per chunk when segmented
  L->gated = off;
  off = align_up(off + M * e * io);
  L->bias = off;
  off = align_up(off + (2 * (size_t)C - 1) * sizeof(float));
  L->xn = off;
  off = align_up(off + M * d * io);
  L->rope = off;
  off = align_up(off + (size_t)T * (s / 2) * 4);
  L->total_bytes = off;
  return FLASH_GAU_OK;
}

// ---- backward workspace ----------------------------------------------------
// fp32 buffers, each 256-byte aligned; with base == nullptr only the size.
int backward_layout(int B, int T, int C, int d, int e, int s, int causal, int dtype, char *base,
                    BackwardLayout *L, size_t *total) {
  if (B <= 0 || T <= 0 || C <= 0 || d <= 0 || e <= 0 || s <= 0) return FLASH_GAU_EINVAL;
  if (T % C != 0) return FLASH_GAU_EINVAL;
  const long long M = (long long)B * T, G = T / C;
  // grid limits of the GEMM and the reductions: rows / 64 and B * G batches
  // in gridDim.y / z, 2C - 1 bias blocks
  if (M > 65535LL * 64 || (long long)B * G > 65535 || C > 4096 || s > (1 << 16) ||
      e > (1 << 16) || d > (1 << 16))
    return FLASH_GAU_ENOTSUP;
  const size_t f = sizeof(float), N = 2 * (size_t)e + s, se = (size_t)s * e;
  size_t off = 0;
  auto take = [&](float **p, size_t n) {
    if (p) *p = base ? reinterpret_cast<float *>(base + off) : nullptr;
    off = align_up(off + n * f);
  };
  BackwardLayout dummy;
  BackwardLayout &l = L ? *L : dummy;
  l.status = base ? reinterpret_cast<int *>(base) : nullptr;
  off = kAlign;
  take(&l.pre, M * N);
  take(&l.U, M * e);
  take(&l.V, M * e);
  take(&l.Z, M * s);
  take(&l.H, 4 * M * s);
  take(&l.S, B * G * C * C);
  take(&l.P, B * G * C * C);
  take(&l.Vh, M * e);
  take(&l.A, M * e);
  take(&l.state, B * G * se);
  take(&l.prefix, (causal ? B * G : B) * se);
  take(&l.dA, M * e);
  take(&l.dU, M * e);
  take(&l.dVh, M * e);
  take(&l.dV, M * e);
  take(&l.dP, B * G * C * C);
  take(&l.dH, 4 * M * s);
  take(&l.dprefix, B * G * se);
  take(&l.dZ, M * s);
  // bf16 operand copies for the tensor-core contractions (2 bytes each)
  float *a_io = nullptr, *dpre_io = nullptr;
  const size_t io_n = dtype == FLASH_GAU_BF16 ? 1 : 0;
  take(&a_io, io_n * (M * e + 1) / 2);
  take(&dpre_io, io_n * (M * N + 1) / 2);
  l.A_io = a_io;
  l.dpre_io = dpre_io;
  float *h_io = nullptr, *v_io = nullptr, *p_io = nullptr, *pre_io = nullptr;
  float *dvh_io = nullptr, *ds_io = nullptr, *dst_io = nullptr;
  take(&h_io, io_n * (4 * M * s + 1) / 2);
  take(&v_io, io_n * (M * e + 1) / 2);
  take(&p_io, io_n * (B * G * C * C + 1) / 2);
  take(&pre_io, io_n * ((causal ? B * G : B) * se + 1) / 2);
  take(&dvh_io, io_n * (M * e + 1) / 2);
  take(&ds_io, io_n * (B * G * C * C + 1) / 2);
  take(&dst_io, io_n * (B * G * se + 1) / 2);
  l.H_io = h_io;
  l.V_io = v_io;
  l.P_io = p_io;
  l.prefix_io = pre_io;
  l.dVh_io = dvh_io;
  l.dS_io = ds_io;
  l.dstate_io = dst_io;
  *total = off;
  return FLASH_GAU_OK;
}

// ---- decode state ----------------------------------------------------------
int decode_layout(int B, int C, int d, int e, int s, char *base, DecodeLayout *L, size_t *total) {
  if (B <= 0 || C <= 0 || d <= 0 || e <= 0 || s <= 0) return FLASH_GAU_EINVAL;
  // grid rows (sequences), the chunk's weights in shared memory, and the
  // 8-column (16-byte) weight loads
  if (B > 65535 || C > 4096 || s > 256 || d > 16384 || e > 16384) return FLASH_GAU_ENOTSUP;
  if (d % 8 != 0 || e % 8 != 0 || s % 8 != 0) return FLASH_GAU_ENOTSUP;
  const size_t N = 2 * (size_t)e + s;
  // slices of the CUDA-core split-K products, or of the tensor-core ones
  // (bf16), whichever is more
  const size_t sp = std::max(decode_slices(d, (int)N), decode_tc_slices(d, (int)N, nullptr));
  const size_t so = std::max(decode_slices(e, d), decode_tc_slices(e, d, nullptr));
  // the tensor-core products read the gated row in the io type (bf16)
  const size_t gio = (size_t)B * e * 2;
  size_t off = 0;
  auto take = [&](void **p, size_t bytes) {
    *p = base ? base + off : nullptr;
    off = align_up(off + bytes);
  };
  void *st, *pos, *pre, *kq, *kl, *vc, *proj, *g, *gb, *outp, *hd, *sc;
  const size_t f = sizeof(float);
  take(&st, sizeof(int));
  take(&pos, (size_t)B * sizeof(int));
  take(&pre, (size_t)B * s * e * f);
  take(&kq, (size_t)B * C * s * f);
  take(&kl, (size_t)B * C * s * f);
  take(&vc, (size_t)B * C * e * f);
  take(&proj, sp * B * N * f);
  take(&g, (size_t)B * e * f);
  take(&gb, gio);
  take(&outp, so * B * d * f);
  take(&hd, (size_t)B * 4 * s * f);
  take(&sc, (size_t)B * C * f);
  if (L) {
    L->status = (int *)st;
    L->pos = (int *)pos;
    L->prefix = (float *)pre;
    L->kq = (float *)kq;
    L->kl = (float *)kl;
    L->vc = (float *)vc;
    L->proj = (float *)proj;
    L->gated = (float *)g;
    L->gated_io = gb;
    L->outp = (float *)outp;
    L->heads = (float *)hd;
    L->score = (float *)sc;
  }
  *total = off;
  return FLASH_GAU_OK;
}

// ---- stage schedules ------------------------------------------------------
const Stage kStagesF32[] = {
    {"projection", simt_projection_f32},
    {"chunk_state", simt_chunk_state_f32},
    {"prefix_scan", simt_prefix_scan_f32},
    {"chunk_attention", simt_chunk_attention_f32},
    {"output", simt_output_f32},
};
const Stage kStagesBF16[] = {
    {"projection", tc_projection_bf16},
    {"chunk_state_scan", tc_chunk_state_scan_bf16},
    {"chunk_attention", tc_chunk_attention_bf16},
    {"output", tc_output_bf16},
};

const Stage *stages(int dtype, int /*causal*/, int *n) {
  if (dtype == FLASH_GAU_FP32) {
    *n = (int)(sizeof(kStagesF32) / sizeof(kStagesF32[0]));
    return kStagesF32;
  }
  if (dtype == FLASH_GAU_BF16) {
    *n = (int)(sizeof(kStagesBF16) / sizeof(kStagesBF16[0]));
    return kStagesBF16;
  }
  *n = 0;
  return nullptr;
}

}  // namespace

void flashgau::rope_table(RopeTable *tab, int s, float base) {
  const double two_pi = 6.283185307179586476925287;
  for (int i = 0; i < kMaxRopePairs; ++i) {
    const double phi = i < s / 2 ? pow((double)base, -2.0 * i / s) / two_pi : 0.0;
    const float hi = (float)phi;
    tab->phi[i] = make_float2(hi, (float)(phi - (double)hi));
  }
}

namespace {

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const char *pa = (const char *)a, *pb = (const char *)b;
  return pa < pb + nb && pb < pa + na;
}

// The two term factors: finite values only (an infinite factor would turn
// the masked zeros of the local term into NaN).
bool scales_finite(const flash_gau_weights *w) {
  return isfinite(w->lin_scale) && isfinite(w->local_scale);
}

int check_block(const flash_gau_block *blk, int s) {
  if (!blk) return FLASH_GAU_OK;
  if (blk->norm < FLASH_GAU_NORM_NONE || blk->norm > FLASH_GAU_NORM_SCALE) return FLASH_GAU_EINVAL;
  if (blk->norm != FLASH_GAU_NORM_NONE && (!blk->norm_g || !(blk->norm_eps > 0.f)))
    return FLASH_GAU_EINVAL;
  if (blk->rope && (s % 2 != 0 || !(blk->rope_base > 1.f))) return FLASH_GAU_EINVAL;
  if (blk->pos_offset < 0) return FLASH_GAU_EINVAL;
  return FLASH_GAU_OK;
}

}  // namespace

int flashgau::check_forward(const void *X, const flash_gau_weights *w, int B, int T, int C,
                            int causal, int dtype, const void *out, const void *workspace,
                            size_t workspace_bytes, flash_gau_workspace_layout *L,
                            int *num_sms) {
  if (!X || !w || !out || !w->W_uvz || !w->W_o || !w->gamma || !w->beta || !w->relpos ||
      !scales_finite(w))
    return FLASH_GAU_EINVAL;
  int st = layout(B, T, C, w->d, w->e, w->s, causal ? 1 : 0, dtype, L);
  if (st != FLASH_GAU_OK) return st;
  const size_t io = dtype == FLASH_GAU_BF16 ? 2 : 4;
  const size_t nx = (size_t)B * T * w->d * io;
  if (overlaps(out, nx, X, nx)) return FLASH_GAU_EINVAL;
  if (workspace) {
    if (workspace_bytes < L->total_bytes || ((uintptr_t)workspace % kAlign) != 0)
      return FLASH_GAU_EWORKSPACE;
    if (overlaps(out, nx, workspace, L->total_bytes)) return FLASH_GAU_EINVAL;
  }
  return device_info(num_sms);
}

namespace {

// One forward: the layer alone (blk == null) or the flash_block wrapper.
int run_forward(const void *X, const flash_gau_weights *w, const flash_gau_block *blk, int B,
                int T, int C, int causal, int dtype, void *out, void *workspace,
                size_t workspace_bytes, void *stream, void *const *stage_events,
                int n_events, const flash_gau_segments *seg = nullptr) {
  if (!workspace) return FLASH_GAU_EINVAL;
  if (n_events < 0 || (n_events > 0 && !stage_events)) return FLASH_GAU_EINVAL;
  causal = causal ? 1 : 0;
  if (w) {
    const int bst = check_block(blk, w->s);
    if (bst != FLASH_GAU_OK) return bst;
  }
  flash_gau_workspace_layout L;
  int num_sms = 0;
  const int st = check_forward(X, w, B, T, C, causal, dtype, out, workspace, workspace_bytes,
                               &L, &num_sms);
  if (st != FLASH_GAU_OK) return st;

  Problem p;
  p.B = B;
  p.T = T;
  p.C = C;
  p.G = T / C;
  p.d = w->d;
  p.e = w->e;
  p.s = w->s;
  p.causal = causal;
  p.dtype = dtype;
  p.M = (long long)B * T;
  p.lin_scale = w->lin_scale;
  p.local_scale = w->local_scale;
  p.seg_ids = seg ? seg->ids : nullptr;
  p.chunk_average = (seg && seg->average) ? 1 : 0;
  p.per_chunk = (causal || p.seg_ids) ? 1 : 0;
  p.lin_off = (dtype == FLASH_GAU_BF16 && !p.seg_ids && !p.chunk_average &&
               p.local_scale != 0.f && (p.lin_scale == 0.f || (causal && p.G == 1)))
                  ? 1
                  : 0;
  p.X = X;
  p.W_uvz = w->W_uvz;
  p.W_o = w->W_o;
  p.gamma = w->gamma;
  p.beta = w->beta;
  p.relpos = w->relpos;
  p.out = out;
  char *ws = (char *)workspace;
  p.status = (int *)(ws + L.status);
  p.U = ws + L.U;
  p.V = ws + L.V;
  p.heads = ws + L.heads;
  p.state = ws + L.state;
  p.prefix = ws + L.prefix;
  p.gated = ws + L.gated;
  p.bias = reinterpret_cast<float *>(ws + L.bias);
  p.xn = ws + L.xn;
  p.rope_cs = ws + L.rope;
  p.stream = (cudaStream_t)stream;
  p.num_sms = num_sms;
  p.norm = blk ? blk->norm : FLASH_GAU_NORM_NONE;
  p.norm_g = blk ? blk->norm_g : nullptr;
  p.norm_b = blk ? blk->norm_b : nullptr;
  p.norm_eps = blk ? blk->norm_eps : 0.f;
  p.rope = blk ? (blk->rope ? 1 : 0) : 0;
  p.rope_base = blk ? blk->rope_base : 0.f;
  p.pos_offset = blk ? blk->pos_offset : 0;
  p.residual = (blk && blk->residual) ? X : nullptr;
  p.A_in = p.norm != FLASH_GAU_NORM_NONE ? p.xn : X;
  if (p.rope) rope_table(&p.rope_tab, p.s, p.rope_base);

  int n = 0;
  const Stage *sched = stages(dtype, causal, &n);
  Stage full[8];
  int nf = 0;
  if (p.norm != FLASH_GAU_NORM_NONE) full[nf++] = {"norm", block_norm};
  if (p.rope && dtype == FLASH_GAU_BF16) full[nf++] = {"rope_table", rope_table_stage};
  for (int k = 0; k < n; ++k) {
    full[nf++] = sched[k];
    if (p.rope && dtype == FLASH_GAU_FP32 && strcmp(sched[k].name, "projection") == 0)
      full[nf++] = {"rope", simt_rope_heads_f32};
  }
  cudaError_t err;
  if (n_events > 0 &&
      (err = cudaEventRecord((cudaEvent_t)stage_events[0], p.stream)) != cudaSuccess)
    return record_cuda(err);
  for (int k = 0; k < nf; ++k) {
    if ((err = full[k].fn(p)) != cudaSuccess) return record_cuda(err);
    if (k + 1 < n_events &&
        (err = cudaEventRecord((cudaEvent_t)stage_events[k + 1], p.stream)) != cudaSuccess)
      return record_cuda(err);
  }
  return FLASH_GAU_OK;
}

}  // namespace

extern "C" {

int flash_gau_workspace_layout_query(int B, int T, int C, int d, int e, int s, int causal,
                                     int dtype, flash_gau_workspace_layout *out) {
  if (!out) return FLASH_GAU_EINVAL;
  return layout(B, T, C, d, e, s, causal, dtype, out);
}

size_t flash_gau_workspace_bytes(int B, int T, int C, const flash_gau_weights *w, int causal,
                                 int dtype) {
  if (!w) return 0;
  flash_gau_workspace_layout L;
  if (layout(B, T, C, w->d, w->e, w->s, causal, dtype, &L) != FLASH_GAU_OK) return 0;
  return L.total_bytes;
}

int flash_gau_num_stages(int dtype, int causal) {
  int n = 0;
  stages(dtype, causal, &n);
  return n;
}

const char *flash_gau_stage_name(int dtype, int causal, int k) {
  int n = 0;
  const Stage *st = stages(dtype, causal, &n);
  if (!st || k < 0 || k >= n) return nullptr;
  return st[k].name;
}

int flash_gau_forward_timed(const void *X, const flash_gau_weights *w, int B, int T, int C,
                            int causal, int dtype, void *out, void *workspace,
                            size_t workspace_bytes, void *stream, void *const *stage_events,
                            int n_events) {
  return run_forward(X, w, nullptr, B, T, C, causal, dtype, out, workspace, workspace_bytes,
                     stream, stage_events, n_events);
}

int flash_gau_rope_toeplitz_bias(const float *a, const float *b, int m, int C, float rope_base,
                                 float *relpos, void *stream) {
  if (!a || !b || !relpos) return FLASH_GAU_EINVAL;
  if (m < 2 || m % 2 != 0 || m > 128 || C < 1 || C > 4096 || !(rope_base > 1.f))
    return FLASH_GAU_EINVAL;
  const cudaError_t err =
      rope_toeplitz_bias(a, b, m, C, rope_base, relpos, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? FLASH_GAU_OK : record_cuda(err);
}

int flash_gau_block_forward(const void *X, const flash_gau_weights *w, const flash_gau_block *blk,
                            int B, int T, int C, int causal, int dtype, void *out,
                            void *workspace, size_t workspace_bytes, void *stream) {
  if (!blk) return FLASH_GAU_EINVAL;
  return run_forward(X, w, blk, B, T, C, causal, dtype, out, workspace, workspace_bytes, stream,
                     nullptr, 0);
}

int flash_gau_forward_segmented(const void *X, const flash_gau_weights *w,
                                const flash_gau_segments *seg, int B, int T, int C, int causal,
                                int dtype, void *out, void *workspace, size_t workspace_bytes,
                                void *stream) {
  return run_forward(X, w, nullptr, B, T, C, causal, dtype, out, workspace, workspace_bytes,
                     stream, nullptr, 0, seg);
}

size_t flash_gau_backward_workspace_bytes(int B, int T, int C, const flash_gau_weights *w,
                                          int causal, int dtype) {
  if (!w || (dtype != FLASH_GAU_FP32 && dtype != FLASH_GAU_BF16)) return 0;
  size_t total = 0;
  if (backward_layout(B, T, C, w->d, w->e, w->s, causal ? 1 : 0, dtype, nullptr, nullptr,
                      &total) !=
      FLASH_GAU_OK)
    return 0;
  return total;
}

int flash_gau_backward(const void *X, const void *dO, const flash_gau_weights *w, int B, int T,
                       int C, int causal, int dtype, const flash_gau_grads *g, void *workspace,
                       size_t workspace_bytes, void *stream) {
  if (!X || !dO || !w || !g || !workspace) return FLASH_GAU_EINVAL;
  if (!w->W_uvz || !w->W_o || !w->gamma || !w->beta || !w->relpos || !scales_finite(w))
    return FLASH_GAU_EINVAL;
  if (!g->dX || !g->dW_uvz || !g->dW_o || !g->dgamma || !g->dbeta || !g->drelpos)
    return FLASH_GAU_EINVAL;
  if (dtype != FLASH_GAU_FP32 && dtype != FLASH_GAU_BF16) return FLASH_GAU_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return FLASH_GAU_EWORKSPACE;
  causal = causal ? 1 : 0;
  BackwardProblem q;
  size_t total = 0;
  int st = backward_layout(B, T, C, w->d, w->e, w->s, causal, dtype,
                           static_cast<char *>(workspace), &q.L, &total);
  if (st != FLASH_GAU_OK) return st;
  if (workspace_bytes < total) return FLASH_GAU_EWORKSPACE;
  q.B = B;
  q.T = T;
  q.C = C;
  q.G = T / C;
  q.d = w->d;
  q.e = w->e;
  q.s = w->s;
  q.causal = causal;
  q.M = (long long)B * T;
  q.lin_scale = w->lin_scale;
  q.local_scale = w->local_scale;
  q.X = X;
  q.dO = dO;
  q.W_uvz = w->W_uvz;
  q.W_o = w->W_o;
  q.gamma = w->gamma;
  q.beta = w->beta;
  q.relpos = w->relpos;
  q.dX = g->dX;
  q.dW_uvz = g->dW_uvz;
  q.dW_o = g->dW_o;
  q.dgamma = g->dgamma;
  q.dbeta = g->dbeta;
  q.drelpos = g->drelpos;
  q.stream = static_cast<cudaStream_t>(stream);
  st = device_info(&q.num_sms);
  if (st != FLASH_GAU_OK) return st;
  // the status word of this workspace, read by flash_gau_workspace_status
  cudaError_t zerr = cudaMemsetAsync(workspace, 0, sizeof(int), q.stream);
  if (zerr != cudaSuccess) return record_cuda(zerr);
  const cudaError_t err = dtype == FLASH_GAU_BF16 ? backward_bf16(q) : backward_f32(q);
  return err == cudaSuccess ? FLASH_GAU_OK : record_cuda(err);
}

size_t flash_gau_decode_state_bytes(int B, int C, const flash_gau_weights *w, int dtype) {
  if (!w || (dtype != FLASH_GAU_FP32 && dtype != FLASH_GAU_BF16)) return 0;
  size_t total = 0;
  if (decode_layout(B, C, w->d, w->e, w->s, nullptr, nullptr, &total) != FLASH_GAU_OK) return 0;
  return total;
}

int flash_gau_decode_step(const void *x, const flash_gau_weights *w, int B, int C, int dtype,
                          void *state, size_t state_bytes, void *out, void *stream) {
  if (!x || !w || !state || !out) return FLASH_GAU_EINVAL;
  if (!w->W_uvz || !w->W_o || !w->gamma || !w->beta || !w->relpos || !scales_finite(w))
    return FLASH_GAU_EINVAL;
  if (dtype != FLASH_GAU_FP32 && dtype != FLASH_GAU_BF16) return FLASH_GAU_EINVAL;
  if (reinterpret_cast<uintptr_t>(state) % kAlign != 0) return FLASH_GAU_EWORKSPACE;
  DecodeProblem q;
  size_t total = 0;
  int st = decode_layout(B, C, w->d, w->e, w->s, static_cast<char *>(state), &q.L, &total);
  if (st != FLASH_GAU_OK) return st;
  if (state_bytes < total) return FLASH_GAU_EWORKSPACE;
  int num_sms = 0;  // the device check
  if ((st = device_info(&num_sms)) != FLASH_GAU_OK) return st;
  q.B = B;
  q.C = C;
  q.d = w->d;
  q.e = w->e;
  q.s = w->s;
  q.lin_scale = w->lin_scale;
  q.local_scale = w->local_scale;
  q.x = x;
  q.W_uvz = w->W_uvz;
  q.W_o = w->W_o;
  q.gamma = w->gamma;
  q.beta = w->beta;
  q.relpos = w->relpos;
  q.out = out;
  q.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t err = dtype == FLASH_GAU_BF16 ? decode_step_bf16(q) : decode_step_f32(q);
  return err == cudaSuccess ? FLASH_GAU_OK : record_cuda(err);
}

int flash_gau_forward(const void *X, const flash_gau_weights *w, int B, int T, int C, int causal,
                      int dtype, void *out, void *workspace, size_t workspace_bytes,
                      void *stream) {
  return flash_gau_forward_timed(X, w, B, T, C, causal, dtype, out, workspace, workspace_bytes,
                                 stream, nullptr, 0);
}

int flash_gau_workspace_status(void *workspace, void *stream) {
  if (!workspace) return FLASH_GAU_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  int word = 0;
  cudaError_t err = cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return record_cuda(err);
  if (word != 0) {
    int zero = 0;
    err = cudaMemcpyAsync(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice, s);
    if (err == cudaSuccess) err = cudaStreamSynchronize(s);
    if (err != cudaSuccess) return record_cuda(err);
  }
  return word;
}

const char *flash_gau_strerror(int status) {
  switch (status) {
    case FLASH_GAU_OK: return "success";
    case FLASH_GAU_EINVAL: return "invalid argument (null pointer, non-positive size, T % C != 0, "
                                  "unknown dtype or overlapping output)";
    case FLASH_GAU_ENOTSUP: return "shape not supported for this dtype";
    case FLASH_GAU_EWORKSPACE: return "workspace too small or not 256-byte aligned";
    case FLASH_GAU_ECUDA: return g_cuda_msg;
    case FLASH_GAU_EDEVICE: return "current CUDA device is not an sm_103 (GB300) GPU";
    case FLASH_GAU_ETIMEOUT: return "a kernel gave up a bounded wait (pipeline stalled)";
    default: return "unknown status";
  }
}

int flash_gau_version(void) { return 107; }

}  // extern "C"
