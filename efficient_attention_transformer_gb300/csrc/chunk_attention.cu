// Chunk attention of mixed chunk attention on tcgen05 tensor cores, bf16 with
// fp32 accumulation ("Transformer Quality in Linear Time", Method: local
// part, eq. 7/8 global part, display after eq. 8; flash_block pseudocode):
//
//   acc   = Q_lin Prefix_g                               (global term)
//   acc  += sum_kb relu^2(Q_quad K_quad[kb]^T / C + b) V[kb]   (local term)
//   gated = U * acc
//
// One CTA per (chunk, 128-query tile, 256-column value tile).  Key blocks of
// 128 are visited in order (only those at or below the diagonal when
// causal).  S = Q_quad K_quad^T of a key block lands in one of two TMEM
// buffers; four warps turn it into P = relu^2(S/C + b) (masked) in
// registers and write P as bf16 to shared memory in the 128-byte swizzled
// K-major layout, where it is the A operand of the next MMA.  The C x C
// score matrix never leaves the SM.  Because relu^2 has no row
// normalisation, the products of successive key blocks simply add.
//
// Shared memory (224 KB): Q_quad tile 32 KB; P slots 4 x 16 KB (Q_lin first
// occupies slots 0-1); K_quad ring 2 x 32 KB; B-operand ring 2 x 32 KB (the
// prefix state rows, then V rows, 64 rows x 256 columns per stage).
// TMEM: accumulator columns 0-255, S buffers 256-383 and 384-511.
#include <cuda_bf16.h>

#include "flash_gau_internal.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace flashgau {
namespace {

using namespace ptx;

constexpr int QT = 128;     // query rows per CTA
constexpr int KB = 128;     // keys per block
constexpr int ET = 256;     // value columns per CTA
constexpr int SD = 128;     // head width s
constexpr int NUM_THREADS = 192;

constexpr int Q_BYTES = QT * SD * 2;          // 32 KB (two 64-wide atoms)
constexpr int ATOM_BYTES = 128 * 64 * 2;      // 16 KB: 128 rows x 64 bf16
constexpr int P_SLOT_BYTES = ATOM_BYTES;      // 128 rows x 64 keys
constexpr int K_STAGE_BYTES = KB * SD * 2;    // 32 KB
constexpr int B_BOX_BYTES = 64 * 64 * 2;      // 64 rows x 64 columns: 8 KB
constexpr int B_STAGE_BYTES = 64 * ET * 2;    // 32 KB

constexpr int OFF_Q = 0;
constexpr int OFF_P = OFF_Q + Q_BYTES;                 // 4 slots
constexpr int OFF_K = OFF_P + 4 * P_SLOT_BYTES;        // 2 stages
constexpr int OFF_B = OFF_K + 2 * K_STAGE_BYTES;       // 2 stages
constexpr int TILE_BYTES = OFF_B + 2 * B_STAGE_BYTES;  // 224 KB
constexpr int SMEM_BYTES = TILE_BYTES + 1024 + 512;

constexpr uint32_t TM_ACC = 0, TM_S0 = 256;

struct Bars {
  uint64_t q_full, ql_full;
  uint64_t k_full[2], k_empty[2];
  uint64_t b_full[2], b_empty[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], p_free[2];
  uint64_t acc_full, drain, u_full;
  uint32_t tmem_base;
  volatile int abort_flag;
};

struct AttnParams {
  int C, G, e, causal;
  long long M;
  int pre_rows_per_batch;  // causal: prefix row block per chunk; else per batch
  float inv_c;
  const float *relpos;
  int *status;
};

__device__ __forceinline__ void raise_timeout(Bars *b, int *status) {
  b->abort_flag = 1;
  atomicExch(status, FLASH_GAU_ETIMEOUT);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// Ring position helper: stage index and the parity of its current phase.
struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  int n;
  __device__ explicit Ring(int n_) : n(n_) {}
  __device__ void next() {
    if (++stage == n) {
      stage = 0;
      phase ^= 1;
    }
  }
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
chunk_attention_kernel(const __grid_constant__ CUtensorMap tmQq,
                       const __grid_constant__ CUtensorMap tmKq,
                       const __grid_constant__ CUtensorMap tmQl,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmPre,
                       const __grid_constant__ CUtensorMap tmU,
                       const __grid_constant__ CUtensorMap tmG, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *tiles = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars *bar = reinterpret_cast<Bars *>(tiles + TILE_BYTES);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const int et = blockIdx.x;                 // value column tile
  const int qt = blockIdx.y;                 // query tile inside the chunk
  const int chunk = blockIdx.z;              // b * G + g
  const int b = chunk / p.G;
  const long long tok0 = (long long)chunk * p.C;  // first token of the chunk
  const int nkb = p.causal ? qt + 1 : p.C / KB;
  const int pre_row0 = p.causal ? chunk * SD : b * SD;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar->q_full), 1);
    mbar_init(smem_u32(&bar->ql_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar->k_full[i]), 1);
      mbar_init(smem_u32(&bar->k_empty[i]), 1);
      mbar_init(smem_u32(&bar->b_full[i]), 1);
      mbar_init(smem_u32(&bar->b_empty[i]), 1);
      mbar_init(smem_u32(&bar->s_full[i]), 1);
      mbar_init(smem_u32(&bar->s_free[i]), 128);
      mbar_init(smem_u32(&bar->p_full[i]), 128);
      mbar_init(smem_u32(&bar->p_free[i]), 1);
    }
    mbar_init(smem_u32(&bar->acc_full), 1);
    mbar_init(smem_u32(&bar->drain), 1);
    mbar_init(smem_u32(&bar->u_full), 1);
    bar->abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bar->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // setup above overlaps the previous kernel's tail; its outputs are read below
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tmem = bar->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (elect_one()) {
      const int qrow = (int)(tok0 + qt * QT);
      uint32_t fb = smem_u32(&bar->q_full);
      mbar_arrive_expect_tx(fb, Q_BYTES);
      tma_load_2d(smem_u32(tiles + OFF_Q), &tmQq, fb, 0, qrow);
      tma_load_2d(smem_u32(tiles + OFF_Q + ATOM_BYTES), &tmQq, fb, 64, qrow);
      Ring kr(2), br(2);
      bool ok = true;
      // K_quad block 0
      auto load_k = [&](int kb) -> bool {
        if (!mbar_wait(smem_u32(&bar->k_empty[kr.stage]), kr.phase ^ 1, &bar->abort_flag)) return false;
        const uint32_t f = smem_u32(&bar->k_full[kr.stage]);
        uint8_t *dst = tiles + OFF_K + kr.stage * K_STAGE_BYTES;
        mbar_arrive_expect_tx(f, K_STAGE_BYTES);
        const int krow = (int)(tok0 + kb * KB);
        tma_load_2d(smem_u32(dst), &tmKq, f, 0, krow);
        tma_load_2d(smem_u32(dst + ATOM_BYTES), &tmKq, f, 64, krow);
        kr.next();
        return true;
      };
      auto load_b = [&](const CUtensorMap *tm, int row) -> bool {
        if (!mbar_wait(smem_u32(&bar->b_empty[br.stage]), br.phase ^ 1, &bar->abort_flag)) return false;
        const uint32_t f = smem_u32(&bar->b_full[br.stage]);
        uint8_t *dst = tiles + OFF_B + br.stage * B_STAGE_BYTES;
        mbar_arrive_expect_tx(f, B_STAGE_BYTES);
#pragma unroll
        for (int j = 0; j < ET / 64; ++j)
          tma_load_2d(smem_u32(dst + j * B_BOX_BYTES), tm, f, et * ET + j * 64, row);
        br.next();
        return true;
      };
      ok = load_k(0);
      if (ok) {
        fb = smem_u32(&bar->ql_full);
        mbar_arrive_expect_tx(fb, Q_BYTES);
        tma_load_2d(smem_u32(tiles + OFF_P), &tmQl, fb, 0, qrow);
        tma_load_2d(smem_u32(tiles + OFF_P + P_SLOT_BYTES), &tmQl, fb, 64, qrow);
        ok = load_b(&tmPre, pre_row0) && load_b(&tmPre, pre_row0 + 64);
      }
      for (int kb = 0; ok && kb < nkb && !bar->abort_flag; ++kb) {
        if (kb + 1 < nkb) ok = load_k(kb + 1);
        const int vrow = (int)(tok0 + kb * KB);
        ok = ok && load_b(&tmV, vrow) && load_b(&tmV, vrow + 64);
      }
      // the U tile of the epilogue goes into the K_quad ring once the last
      // S product has read it: 4 row quarters x 4 column boxes of 32 x 64
      for (int i = 0; ok && i < 2; ++i) {
        ok = mbar_wait(smem_u32(&bar->k_empty[kr.stage]), kr.phase ^ 1, &bar->abort_flag);
        kr.next();
      }
      if (ok) {
        const uint32_t f = smem_u32(&bar->u_full);
        mbar_arrive_expect_tx(f, QT * ET * 2);
        for (int q = 0; q < 4; ++q)
          for (int j = 0; j < ET / 64; ++j)
            tma_load_2d(smem_u32(tiles + OFF_K + (q * 4 + j) * 4096), &tmU, f, et * ET + j * 64,
                        qrow + q * 32);
      }
      if (!ok) raise_timeout(bar, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (elect_one()) {
      const uint32_t idesc_s = idesc_bf16_f32(128, KB, 0, 0);
      const uint32_t idesc_v = idesc_bf16_f32(128, ET, 0, 1);
      const uint32_t sQ = smem_u32(tiles + OFF_Q);
      const uint32_t sP = smem_u32(tiles + OFF_P);
      const uint32_t sK = smem_u32(tiles + OFF_K);
      const uint32_t sB = smem_u32(tiles + OFF_B);
      Ring kr(2), br(2);
      bool ok = true;
      // S[kb] = Q_quad K_quad[kb]^T into TMEM buffer kb % 2
      auto issue_s = [&](int kb) -> bool {
        const int sb = kb & 1;
        if (kb >= 2 && !mbar_wait(smem_u32(&bar->s_free[sb]), ((kb >> 1) - 1) & 1, &bar->abort_flag)) return false;
        if (!mbar_wait(smem_u32(&bar->k_full[kr.stage]), kr.phase, &bar->abort_flag)) return false;
        tc_fence_after();
        const uint32_t kst = sK + kr.stage * K_STAGE_BYTES;
#pragma unroll
        for (int k = 0; k < SD / 16; ++k) {
          const uint32_t off = (k >> 2) * ATOM_BYTES + (k & 3) * 32;
          mma_f16_ss(tmem + TM_S0 + sb * KB, sw128_desc(sQ + off, 16, 1024),
                     sw128_desc(kst + off, 16, 1024), idesc_s, k != 0);
        }
        mma_commit(smem_u32(&bar->k_empty[kr.stage]));
        mma_commit(smem_u32(&bar->s_full[sb]));
        kr.next();
        return true;
      };
      // acc (+)= A[two or four 16-row K steps per stage] * B stage
      auto issue_b = [&](uint32_t a_atom, bool first) -> bool {
        if (!mbar_wait(smem_u32(&bar->b_full[br.stage]), br.phase, &bar->abort_flag)) return false;
        tc_fence_after();
        const uint32_t bst = sB + br.stage * B_STAGE_BYTES;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16_ss(tmem + TM_ACC, sw128_desc(a_atom + k * 32, 16, 1024),
                     sw128_desc(bst + k * 2048, B_BOX_BYTES, 1024), idesc_v, !(first && k == 0));
        mma_commit(smem_u32(&bar->b_empty[br.stage]));
        br.next();
        return true;
      };
      ok = mbar_wait(smem_u32(&bar->q_full), 0, &bar->abort_flag);
      ok = ok && issue_s(0);
      // global term first: acc = Q_lin Prefix (Q_lin sits in P slots 0-1)
      ok = ok && mbar_wait(smem_u32(&bar->ql_full), 0, &bar->abort_flag);
      ok = ok && issue_b(sP, true) && issue_b(sP + P_SLOT_BYTES, false);
      if (ok) mma_commit(smem_u32(&bar->p_free[0]));
      for (int kb = 0; ok && kb < nkb && !bar->abort_flag; ++kb) {
        if (kb + 1 < nkb) ok = issue_s(kb + 1);
        const int pp = kb & 1;
        ok = ok && mbar_wait(smem_u32(&bar->p_full[pp]), (kb >> 1) & 1, &bar->abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t pslot = sP + pp * 2 * P_SLOT_BYTES;
        ok = issue_b(pslot, false) && issue_b(pslot + P_SLOT_BYTES, false);
        if (ok) mma_commit(smem_u32(&bar->p_free[pp]));
      }
      if (ok) mma_commit(smem_u32(&bar->acc_full));
      else raise_timeout(bar, p.status);
      mma_commit(smem_u32(&bar->drain));
      if (!mbar_wait(smem_u32(&bar->drain), 0)) raise_timeout(bar, p.status);
    }
  } else {
    // ------------------------------------- relu^2 warps, then the epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;   // row inside the query tile
    const int i = qt * QT + r;           // row inside the chunk
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint8_t *sP = tiles + OFF_P;
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
      const int sb = kb & 1;
      if (!mbar_wait(smem_u32(&bar->s_full[sb]), (kb >> 1) & 1, &bar->abort_flag)) { ok = false; break; }
      tc_fence_after();
      // P slot pair kb&1 must be free (slot pair 0 first held Q_lin)
      const uint32_t pf_parity = (sb == 0) ? ((kb >> 1) & 1) : (((kb >> 1) & 1) ^ 1);
      if (!mbar_wait(smem_u32(&bar->p_free[sb]), pf_parity, &bar->abort_flag)) { ok = false; break; }
      const bool diag = p.causal && kb == qt;
      const float *bias_row = p.relpos + (kb * KB - i + p.C - 1);  // + key index j
#pragma unroll 1
      for (int c0 = 0; c0 < KB; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + TM_S0 + sb * KB + c0, v);
        tmem_ld_wait();
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float x0 = fmaf(__uint_as_float(v[j]), p.inv_c, __ldg(bias_row + c0 + j));
          float x1 = fmaf(__uint_as_float(v[j + 1]), p.inv_c, __ldg(bias_row + c0 + j + 1));
          x0 = fmaxf(x0, 0.f);
          x1 = fmaxf(x1, 0.f);
          x0 *= x0;
          x1 *= x1;
          if (diag) {
            if (c0 + j > r) x0 = 0.f;
            if (c0 + j + 1 > r) x1 = 0.f;
          }
          packed[j / 2] = pack_bf16(x0, x1);
        }
        // keys c0..c0+31 -> slot (c0 / 64), 16-byte chunks (c0 % 64)/8 .. +3
        uint8_t *slot = sP + (sb * 2 + (c0 >> 6)) * P_SLOT_BYTES + r * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk16 = ((c0 & 63) >> 3) + q;
          uint4 w = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                               packed[4 * q + 3]);
          *reinterpret_cast<uint4 *>(slot + ((chunk16 ^ (r & 7)) << 4)) = w;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar->s_free[sb]));
      mbar_arrive(smem_u32(&bar->p_full[sb]));
    }
    if (ok && mbar_wait(smem_u32(&bar->acc_full), 0, &bar->abort_flag) &&
        mbar_wait(smem_u32(&bar->u_full), 0, &bar->abort_flag)) {
      tc_fence_after();
      // U boxes sit in the K ring, the gated boxes are staged in the B ring
      // (free once every MMA has completed); both 32 rows x 128 bytes,
      // swizzled, one per (row quarter, 64-column block).
      for (int j = 0; j < ET / 64; ++j) {
        uint32_t va[32], vb[32];
        tmem_ld32(tmem + lane_off + TM_ACC + j * 64, va);
        tmem_ld32(tmem + lane_off + TM_ACC + j * 64 + 32, vb);
        tmem_ld_wait();
        const uint8_t *ubox = tiles + OFF_K + (quarter * 4 + j) * 4096;
        uint8_t *gbox = tiles + OFF_B + (quarter * 4 + j) * 4096;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 u4 = *reinterpret_cast<const uint4 *>(ubox + sw128_offset(lane, c));
          const __nv_bfloat162 *uh = reinterpret_cast<const __nv_bfloat162 *>(&u4);
          const uint32_t *src = c < 4 ? &va[8 * c] : &vb[8 * (c - 4)];
          uint4 w;
          uint32_t *wp = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float2 uf = __bfloat1622float2(uh[h]);
            wp[h] = pack_bf16(uf.x * __uint_as_float(src[2 * h]),
                              uf.y * __uint_as_float(src[2 * h + 1]));
          }
          *reinterpret_cast<uint4 *>(gbox + sw128_offset(lane, c)) = w;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int grow = (int)(tok0 + qt * QT + quarter * 32);
        for (int j = 0; j < ET / 64; ++j)
          tma_store_2d(&tmG, smem_u32(tiles + OFF_B + (quarter * 4 + j) * 4096), et * ET + j * 64,
                       grow);
        tma_store_commit();
        tma_store_wait<0>();
      }
      __syncwarp();
    } else {
      raise_timeout(bar, p.status);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t tc_chunk_attention_bf16(const Problem &pr) {
  const __nv_bfloat16 *heads = (const __nv_bfloat16 *)pr.heads;
  const long long Ms = pr.M * pr.s;
  CUtensorMap tQq, tKq, tQl, tV, tPre;
  cudaError_t err;
  if ((err = make_tmap_bf16_2d(&tQq, heads, pr.M, pr.s, pr.s, QT, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tKq, heads + Ms, pr.M, pr.s, pr.s, KB, 64)) != cudaSuccess)
    return err;
  if ((err = make_tmap_bf16_2d(&tQl, heads + 2 * Ms, pr.M, pr.s, pr.s, QT, 64)) != cudaSuccess)
    return err;
  if ((err = make_tmap_bf16_2d(&tV, pr.V, pr.M, pr.e, pr.e, 64, 64)) != cudaSuccess) return err;
  CUtensorMap tU, tG;
  if ((err = make_tmap_bf16_2d(&tU, pr.U, pr.M, pr.e, pr.e, 32, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tG, pr.gated, pr.M, pr.e, pr.e, 32, 64)) != cudaSuccess) return err;
  const long long pre_rows = (long long)(pr.causal ? pr.B * pr.G : pr.B) * pr.s;
  if ((err = make_tmap_bf16_2d(&tPre, pr.prefix, pre_rows, pr.e, pr.e, 64, 64)) != cudaSuccess)
    return err;

  static unsigned long long configured = 0;
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev < 64 && !(configured & (1ull << dev))) {
    err = cudaFuncSetAttribute(chunk_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SMEM_BYTES);
    if (err != cudaSuccess) return err;
    configured |= 1ull << dev;
  }
  AttnParams p;
  p.C = pr.C;
  p.G = pr.G;
  p.e = pr.e;
  p.causal = pr.causal;
  p.M = pr.M;
  p.pre_rows_per_batch = pr.s;
  p.inv_c = 1.0f / (float)pr.C;
  p.relpos = pr.relpos;
  p.status = pr.status;
  dim3 grid(pr.e / ET, pr.C / QT, pr.B * pr.G);
  return launch_pdl(chunk_attention_kernel, grid, dim3(NUM_THREADS), SMEM_BYTES, pr.stream, tQq,
                    tKq, tQl, tV, tPre, tU, tG, p);
}

}  // namespace flashgau
