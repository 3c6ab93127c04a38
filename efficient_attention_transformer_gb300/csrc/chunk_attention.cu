// Chunk attention of mixed chunk attention on tcgen05 tensor cores, bf16 with
// fp32 accumulation ("Transformer Quality in Linear Time", Method: local
// part, eq. 7/8 global part, display after eq. 8; flash_block pseudocode):
//
//   acc   = Q_lin Prefix_g                                      (global term)
//   acc  += sum_kb relu^2(Q_quad K_quad[kb]^T / C + b) V[kb]    (local term)
//   gated = U * acc
//
// Work unit: (chunk, 128-query tile, 128-column value tile).  One
// persistent CTA per SM; the producer takes units from a global atomic
// counter (dynamic scheduling: per chunk the query tiles with more key
// blocks first, value tile fastest, so the cheapest units come last and
// units sharing Q/K run on neighbouring SMs at the same time) and hands
// their indices to the other roles through a 4-entry queue.  Key
// blocks of 128 are visited in order, only those at or below the diagonal
// when causal.  Because relu^2 has no row normalisation, the products of
// successive key blocks simply add into one accumulator.
//
// Roles (448 threads):
//   warp 0     TMA producer: Q_quad, Q_lin, the K_quad ring, and a ring of
//              64-row x 128-column B operands (prefix state rows, then V
//              rows);
//   warp 1     MMA issuer: S = Q_quad K_quad^T into a 128-column TMEM
//              buffer (two buffers), acc = Q_lin Prefix (smem A), acc += P V
//              with P read from TMEM;
//   warps 2-9  relu^2, two per TMEM lane quarter, each for 64 of a block's
//              128 keys: read S with tcgen05.ld, compute relu^2(S/C + b)
//              (the bias table carries the causal mask as -inf, written by
//              the projection kernel), write P as packed bf16
//              over the start of the same S columns with tcgen05.st (keys
//              0-63 at packed columns 0-31, keys 64-127 at 64-95); the
//              C x C scores never leave TMEM and registers;
//   warps 10-13 epilogue: gated = U * acc, U boxes TMA-loaded into per-warp
//              double buffers, the product written in place and TMA-stored.
// Two accumulators alternate between units, so while the epilogue warps
// drain one, the MMAs of the next unit already fill the other.
//
// Shared memory (224 KB): Q_quad 32 KB, Q_lin 32 KB, K ring 2 x 32 KB,
// B ring 4 x 16 KB, epilogue boxes 4 warps x 2 x 4 KB.  TMEM: accumulators
// at columns 0 and 128, S/P buffers at 256 and 384 (128 columns each).
#include <cuda_bf16.h>

#include "flash_gau_internal.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace flashgau {
namespace {

using namespace ptx;

constexpr int QT = 128;  // query rows per unit
constexpr int KB = 128;  // keys per block
constexpr int ET = 128;  // value columns per unit
constexpr int SD = 128;  // head width s
constexpr int RELU_WARPS = 8;
constexpr int NUM_THREADS = 32 * (2 + RELU_WARPS + 4);

constexpr int ATOM_BYTES = 128 * 64 * 2;        // 128 rows x 64 bf16: 16 KB
constexpr int Q_BYTES = 2 * ATOM_BYTES;         // 32 KB
constexpr int K_STAGE_BYTES = 2 * ATOM_BYTES;   // 128 keys x 128: 32 KB
constexpr int B_BOX_BYTES = 64 * 64 * 2;        // 64 rows x 64 columns: 8 KB
constexpr int B_STAGES = 4;
constexpr int B_STAGE_BYTES = 2 * B_BOX_BYTES;  // 64 rows x 128 columns: 16 KB
constexpr int E_BOX_BYTES = 32 * 128;           // 32 rows x 64 bf16: 4 KB

constexpr int OFF_QQ = 0;
constexpr int OFF_QL = OFF_QQ + Q_BYTES;
constexpr int OFF_K = OFF_QL + Q_BYTES;
constexpr int OFF_B = OFF_K + 2 * K_STAGE_BYTES;
constexpr int OFF_E = OFF_B + B_STAGES * B_STAGE_BYTES;
constexpr int TILE_BYTES = OFF_E + 4 * 2 * E_BOX_BYTES;  // 224 KB
constexpr int SMEM_BYTES = TILE_BYTES + 1024 + 512;

constexpr uint32_t TM_ACC = 0, TM_S = 256;

struct Bars {
  uint64_t q_full, q_empty, ql_full, ql_empty;
  uint64_t k_full[2], k_empty[2];
  uint64_t b_full[B_STAGES], b_empty[B_STAGES];
  uint64_t s_full[2], p_full[2], sb_free[2];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t u_full[4][2];
  uint64_t uq_full[4], uq_empty[4];  // unit-index queue
  volatile int unit_q[4];
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
};

struct AttnParams {
  int C, G, causal;
  int n_et, n_qt, total;  // units (chunk, query tile, value tile), value tile fastest
  float inv_c;
  const float *bias;  // [2C-1] relpos, -inf at causally masked offsets
  int *status;
  int *next_unit;  // work counter, zeroed by the projection kernel
};

// Agents that consume each queued unit index: the MMA thread, the relu^2
// warps and the epilogue warps (one arrival per warp).
constexpr int QUEUE_AGENTS = 1 + 8 + 4;

struct Unit {
  int chunk, b, qt, et, nkb;
  long long tok0;  // first token of the chunk
};

__device__ __forceinline__ Unit unit_of(const AttnParams &p, int u) {
  Unit x;
  x.et = u % p.n_et;
  x.qt = p.n_qt - 1 - (u / p.n_et) % p.n_qt;  // more key blocks first
  x.chunk = u / (p.n_et * p.n_qt);
  x.b = x.chunk / p.G;
  x.tok0 = (long long)x.chunk * p.C;
  x.nkb = p.causal ? x.qt + 1 : p.C / KB;
  return x;
}

__device__ __forceinline__ void raise_timeout(Bars *b, int *status) {
  b->abort_flag = 1;
  atomicExch(status, FLASH_GAU_ETIMEOUT);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// Ring position: stage index and the parity of its current phase.
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

// Half `half` (64 keys) of one 128-key block of the local term, for this
// thread's query row r (row i = qt*128 + r of the chunk): reads the 64 S
// columns (fp32) at sbuf + 64*half, writes P = relu^2(S/C + b) as 32 packed
// bf16 columns over the start of those same columns.  The bias table holds
// -inf at the causally masked offsets, so the mask costs nothing here.  All
// 64 S values are in registers before the first store lands.
__device__ __forceinline__ void relu2_half(uint32_t sbuf, const AttnParams &p, int kb, int qt,
                                           int r, int half) {
  const int i = qt * QT + r;
  const int c0 = half * 64;
  const float *bias_row = p.bias + (kb * KB + c0 - i + p.C - 1);  // + key index j
  uint32_t va[32], vb[32];
  tmem_ld32(sbuf + c0, va);
  tmem_ld32(sbuf + c0 + 32, vb);
  tmem_ld_wait();
  uint32_t lo[16], hi[16];
#pragma unroll
  for (int j = 0; j < 64; j += 2) {
    const uint32_t s0 = j < 32 ? va[j] : vb[j - 32];
    const uint32_t s1 = j < 32 ? va[j + 1] : vb[j - 31];
    float x0 = fmaf(__uint_as_float(s0), p.inv_c, __ldg(bias_row + j));
    float x1 = fmaf(__uint_as_float(s1), p.inv_c, __ldg(bias_row + j + 1));
    x0 = fmaxf(x0, 0.f);
    x1 = fmaxf(x1, 0.f);
    x0 *= x0;
    x1 *= x1;
    if (j < 32) lo[j / 2] = pack_bf16(x0, x1);
    else hi[(j - 32) / 2] = pack_bf16(x0, x1);
  }
  tmem_st16(sbuf + c0, lo);
  tmem_st16(sbuf + c0 + 16, hi);
}

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
  const volatile int *abort = &bar->abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar->q_full), 1);
    mbar_init(smem_u32(&bar->q_empty), 1);
    mbar_init(smem_u32(&bar->ql_full), 1);
    mbar_init(smem_u32(&bar->ql_empty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar->k_full[i]), 1);
      mbar_init(smem_u32(&bar->k_empty[i]), 1);
      mbar_init(smem_u32(&bar->acc_full[i]), 1);
      mbar_init(smem_u32(&bar->acc_empty[i]), 128);
      mbar_init(smem_u32(&bar->s_full[i]), 1);
      mbar_init(smem_u32(&bar->p_full[i]), 32 * RELU_WARPS);
      mbar_init(smem_u32(&bar->sb_free[i]), 1);
      for (int w = 0; w < 4; ++w) mbar_init(smem_u32(&bar->u_full[w][i]), 1);
    }
    for (int i = 0; i < B_STAGES; ++i) {
      mbar_init(smem_u32(&bar->b_full[i]), 1);
      mbar_init(smem_u32(&bar->b_empty[i]), 1);
    }
    for (int q = 0; q < 4; ++q) {
      mbar_init(smem_u32(&bar->uq_full[q]), 1);
      mbar_init(smem_u32(&bar->uq_empty[q]), QUEUE_AGENTS);
    }
    mbar_init(smem_u32(&bar->drain), 1);
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
  // This kernel may start while the chunk-state/scan kernel launched before
  // it still runs: everything except the prefix states (U, V, the heads, the
  // zeroed work counter) was written by the projection, which completed
  // before any CTA of that kernel got past its own griddepcontrol.wait, and
  // the producer waits for that kernel itself just before its first prefix
  // load.
  griddep_launch_dependents();
  const uint32_t tmem = bar->tmem_base;
  // unit queue: entry q of this CTA's sequence sits in slot q & 3
  auto pop = [&](int q) -> int {  // unit index, -1 when done, -2 on timeout
    if (!mbar_wait(smem_u32(&bar->uq_full[q & 3]), (q >> 2) & 1, abort)) return -2;
    return bar->unit_q[q & 3];
  };
  auto release = [&](int q) { mbar_arrive(smem_u32(&bar->uq_empty[q & 3])); };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (elect_one()) {
      Ring kr(2), br(B_STAGES);
      bool ok = true;
      auto load_k = [&](long long krow) -> bool {
        if (!mbar_wait(smem_u32(&bar->k_empty[kr.stage]), kr.phase ^ 1, abort)) return false;
        const uint32_t f = smem_u32(&bar->k_full[kr.stage]);
        uint8_t *dst = tiles + OFF_K + kr.stage * K_STAGE_BYTES;
        mbar_arrive_expect_tx(f, K_STAGE_BYTES);
        tma_load_2d(smem_u32(dst), &tmKq, f, 0, (int)krow);
        tma_load_2d(smem_u32(dst + ATOM_BYTES), &tmKq, f, 64, (int)krow);
        kr.next();
        return true;
      };
      auto load_b = [&](const CUtensorMap *tm, int col0, long long row) -> bool {
        if (!mbar_wait(smem_u32(&bar->b_empty[br.stage]), br.phase ^ 1, abort)) return false;
        const uint32_t f = smem_u32(&bar->b_full[br.stage]);
        uint8_t *dst = tiles + OFF_B + br.stage * B_STAGE_BYTES;
        mbar_arrive_expect_tx(f, B_STAGE_BYTES);
#pragma unroll
        for (int j = 0; j < ET / 64; ++j)
          tma_load_2d(smem_u32(dst + j * B_BOX_BYTES), tm, f, col0 + j * 64, (int)row);
        br.next();
        return true;
      };
      // next unit: from the global counter, announced through the queue
      auto push = [&](int q, int u) -> bool {
        if (!mbar_wait(smem_u32(&bar->uq_empty[q & 3]), ((q >> 2) & 1) ^ 1, abort)) return false;
        bar->unit_q[q & 3] = u;
        mbar_arrive(smem_u32(&bar->uq_full[q & 3]));
        return true;
      };
      bool prefix_ready = false;
      int i = 0;
      for (;; ++i) {
        int u = atomicAdd(p.next_unit, 1);
        if (u >= p.total) u = -1;
        ok = push(i, u);
        if (!ok || u < 0) break;
        const Unit x = unit_of(p, u);
        const long long qrow = x.tok0 + x.qt * QT;
        const long long pre_row0 = (long long)(p.causal ? x.chunk : x.b) * SD;
        ok = mbar_wait(smem_u32(&bar->q_empty), (i & 1) ^ 1, abort);
        if (!ok) break;
        uint32_t f = smem_u32(&bar->q_full);
        mbar_arrive_expect_tx(f, Q_BYTES);
        tma_load_2d(smem_u32(tiles + OFF_QQ), &tmQq, f, 0, (int)qrow);
        tma_load_2d(smem_u32(tiles + OFF_QQ + ATOM_BYTES), &tmQq, f, 64, (int)qrow);
        ok = load_k(x.tok0);
        for (int kb = 0; ok && kb < x.nkb; ++kb) {
          if (kb + 1 < x.nkb) ok = load_k(x.tok0 + (kb + 1) * KB);
          ok = ok && load_b(&tmV, x.et * ET, x.tok0 + kb * KB) &&
               load_b(&tmV, x.et * ET, x.tok0 + kb * KB + 64);
        }
        // the global term last: the prefix states come from the kernel
        // launched just before this one, which may still be running
        if (ok && !prefix_ready) {
          griddep_wait();
          prefix_ready = true;
        }
        ok = ok && mbar_wait(smem_u32(&bar->ql_empty), (i & 1) ^ 1, abort);
        if (!ok) break;
        f = smem_u32(&bar->ql_full);
        mbar_arrive_expect_tx(f, Q_BYTES);
        tma_load_2d(smem_u32(tiles + OFF_QL), &tmQl, f, 0, (int)qrow);
        tma_load_2d(smem_u32(tiles + OFF_QL + ATOM_BYTES), &tmQl, f, 64, (int)qrow);
        ok = load_b(&tmPre, x.et * ET, pre_row0) && load_b(&tmPre, x.et * ET, pre_row0 + 64);
      }
      if (!ok) raise_timeout(bar, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (elect_one()) {
      const uint32_t idesc_s = idesc_bf16_f32(128, KB, 0, 0);
      const uint32_t idesc_v = idesc_bf16_f32(128, ET, 0, 1);
      const uint64_t dq = sw128_desc(smem_u32(tiles + OFF_QQ), 16, 1024);
      const uint32_t sQL = smem_u32(tiles + OFF_QL);
      const uint32_t sK = smem_u32(tiles + OFF_K);
      const uint32_t sB = smem_u32(tiles + OFF_B);
      Ring kr(2), br(B_STAGES);
      int n = 0;  // S blocks issued so far (all units): buffer n & 1
      uint32_t acc_col = TM_ACC;  // accumulator of the current unit
      bool ok = true;
      // S[n] = Q_quad K_quad^T into TMEM buffer n & 1
      auto issue_s = [&]() -> bool {
        const int sb = n & 1;
        if (n >= 2 && !mbar_wait(smem_u32(&bar->sb_free[sb]), ((n >> 1) - 1) & 1, abort))
          return false;
        if (!mbar_wait(smem_u32(&bar->k_full[kr.stage]), kr.phase, abort)) return false;
        tc_fence_after();
        const uint64_t dk = sw128_desc(sK + kr.stage * K_STAGE_BYTES, 16, 1024);
#pragma unroll
        for (int k = 0; k < SD / 16; ++k) {
          const uint32_t off = (k >> 2) * ATOM_BYTES + (k & 3) * 32;
          mma_f16_ss(tmem + TM_S + sb * KB, desc_advance(dq, off), desc_advance(dk, off), idesc_s,
                     k != 0);
        }
        mma_commit(smem_u32(&bar->k_empty[kr.stage]));
        mma_commit(smem_u32(&bar->s_full[sb]));
        kr.next();
        ++n;
        return true;
      };
      // acc (+)= A * B stage, A a 64-wide K-major atom in shared memory
      auto issue_b_smem = [&](uint32_t a_atom, bool first) -> bool {
        if (!mbar_wait(smem_u32(&bar->b_full[br.stage]), br.phase, abort)) return false;
        tc_fence_after();
        const uint64_t da = sw128_desc(a_atom, 16, 1024);
        const uint64_t db = sw128_desc(sB + br.stage * B_STAGE_BYTES, B_BOX_BYTES, 1024);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16_ss(tmem + acc_col, desc_advance(da, k * 32), desc_advance(db, k * 2048), idesc_v,
                     !(first && k == 0));
        mma_commit(smem_u32(&bar->b_empty[br.stage]));
        br.next();
        return true;
      };
      // acc += P * B stage, P: 64 keys = 32 packed columns of TMEM at a_col
      auto issue_b_tmem = [&](uint32_t a_col, bool first) -> bool {
        if (!mbar_wait(smem_u32(&bar->b_full[br.stage]), br.phase, abort)) return false;
        tc_fence_after();
        const uint64_t db = sw128_desc(sB + br.stage * B_STAGE_BYTES, B_BOX_BYTES, 1024);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16_ts(tmem + acc_col, tmem + a_col + k * 8, desc_advance(db, k * 2048), idesc_v,
                     !(first && k == 0));
        mma_commit(smem_u32(&bar->b_empty[br.stage]));
        br.next();
        return true;
      };
      for (int i = 0; ok; ++i) {
        const int u = pop(i);
        if (u < 0) {
          ok = u == -1;
          break;
        }
        const Unit x = unit_of(p, u);
        const int n0 = n;
        ok = mbar_wait(smem_u32(&bar->q_full), i & 1, abort) && issue_s();
        if (ok && x.nkb == 1) mma_commit(smem_u32(&bar->q_empty));
        // this unit's accumulator must have been drained by the epilogue of
        // the unit two before
        acc_col = TM_ACC + (i & 1) * ET;
        ok = ok && mbar_wait(smem_u32(&bar->acc_empty[i & 1]), ((i >> 1) & 1) ^ 1, abort);
        if (!ok) break;
        tc_fence_after();
        // local term first, global term (Q_lin Prefix) last
        for (int kb = 0; ok && kb < x.nkb; ++kb) {
          if (kb + 1 < x.nkb) {
            ok = issue_s();
            if (ok && kb + 2 == x.nkb) mma_commit(smem_u32(&bar->q_empty));
          }
          const int si = n0 + kb, sb = si & 1;
          ok = ok && mbar_wait(smem_u32(&bar->p_full[sb]), (si >> 1) & 1, abort);
          if (!ok) break;
          tc_fence_after();
          const uint32_t pcol = TM_S + sb * KB;
          ok = issue_b_tmem(pcol, kb == 0) && issue_b_tmem(pcol + 64, false);
          if (ok) mma_commit(smem_u32(&bar->sb_free[sb]));
        }
        ok = ok && mbar_wait(smem_u32(&bar->ql_full), i & 1, abort);
        if (!ok) break;
        tc_fence_after();
        ok = issue_b_smem(sQL, false) && issue_b_smem(sQL + ATOM_BYTES, false);
        if (ok) mma_commit(smem_u32(&bar->ql_empty));
        if (ok) mma_commit(smem_u32(&bar->acc_full[i & 1]));
        release(i);
      }
      if (!ok) raise_timeout(bar, p.status);
      mma_commit(smem_u32(&bar->drain));
      if (!mbar_wait(smem_u32(&bar->drain), 0)) raise_timeout(bar, p.status);
    }
  } else if (warp < 2 + RELU_WARPS) {
    // -------------------------------------------------- relu^2 warps
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;  // row inside the query tile
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int n = 0;
    bool ok = true;
    for (int q = 0; ok; ++q) {
      const int u = pop(q);
      if (u < 0) {
        ok = u == -1;
        break;
      }
      const Unit x = unit_of(p, u);
      for (int kb = 0; kb < x.nkb; ++kb, ++n) {
        const int sb = n & 1;
        if (!mbar_wait(smem_u32(&bar->s_full[sb]), (n >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        relu2_half(tmem + lane_off + TM_S + sb * KB, p, kb, x.qt, r, half);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar->p_full[sb]));
      }
      __syncwarp();
      if (lane == 0) release(q);
    }
    if (!ok) raise_timeout(bar, p.status);
  } else {
    // ------------------------------------------------------- epilogue
    const int quarter = warp & 3, w = warp - (2 + RELU_WARPS);
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint8_t *ebuf = tiles + OFF_E + w * 2 * E_BOX_BYTES;
    // U box of part j (64 value columns) of unit u into buffer b
    auto load_u = [&](int u, int j, int b) {
      if (lane != 0 || u < 0) return;
      const Unit x = unit_of(p, u);
      const uint32_t f = smem_u32(&bar->u_full[w][b]);
      mbar_arrive_expect_tx(f, E_BOX_BYTES);
      tma_load_2d(smem_u32(ebuf + b * E_BOX_BYTES), &tmU, f, x.et * ET + j * 64,
                  (int)(x.tok0 + x.qt * QT + quarter * 32));
    };
    bool ok = true;
    int cur = pop(0);
    ok = cur != -2;
    load_u(cur, 0, 0);
    load_u(cur, 1, 1);
    int c = 0;
    for (int i = 0; ok && cur >= 0; ++i) {
      // the next unit's index, to prefetch its U boxes (released later)
      const int nxt = pop(i + 1);
      if (nxt == -2 ||
          !mbar_wait(smem_u32(&bar->acc_full[i & 1]), (i >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      const Unit x = unit_of(p, cur);
      tc_fence_after();
      const int grow = (int)(x.tok0 + x.qt * QT + quarter * 32);
      for (int j = 0; j < ET / 64; ++j, ++c) {
        const int b = c & 1;
        if (!mbar_wait(smem_u32(&bar->u_full[w][b]), (c >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        uint32_t va[32], vb[32];
        const uint32_t acc = tmem + lane_off + TM_ACC + (i & 1) * ET + j * 64;
        tmem_ld32(acc, va);
        tmem_ld32(acc + 32, vb);
        tmem_ld_wait();
        if (j == ET / 64 - 1) {
          tc_fence_before();
          mbar_arrive(smem_u32(&bar->acc_empty[i & 1]));
        }
        uint8_t *box = ebuf + b * E_BOX_BYTES;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 *slot = reinterpret_cast<uint4 *>(box + sw128_offset(lane, q));
          const uint4 u4 = *slot;
          const __nv_bfloat162 *uh = reinterpret_cast<const __nv_bfloat162 *>(&u4);
          const uint32_t *src = q < 4 ? &va[8 * q] : &vb[8 * (q - 4)];
          uint4 g4;
          uint32_t *gp = reinterpret_cast<uint32_t *>(&g4);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float2 uf = __bfloat1622float2(uh[h]);
            gp[h] = pack_bf16(uf.x * __uint_as_float(src[2 * h]),
                              uf.y * __uint_as_float(src[2 * h + 1]));
          }
          *slot = g4;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmG, smem_u32(box), x.et * ET + j * 64, grow);
          tma_store_commit();
          tma_store_wait_read<0>();  // the box is refilled next
        }
        __syncwarp();
        load_u(nxt, j, b);
      }
      __syncwarp();
      if (lane == 0) release(i);
      cur = nxt;
    }
    if (lane == 0) tma_store_wait<0>();
    __syncwarp();
    if (!ok) raise_timeout(bar, p.status);
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
  CUtensorMap tQq, tKq, tQl, tV, tPre, tU, tG;
  cudaError_t err;
  if ((err = make_tmap_bf16_2d(&tQq, heads, pr.M, pr.s, pr.s, QT, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tKq, heads + Ms, pr.M, pr.s, pr.s, KB, 64)) != cudaSuccess)
    return err;
  if ((err = make_tmap_bf16_2d(&tQl, heads + 2 * Ms, pr.M, pr.s, pr.s, QT, 64)) != cudaSuccess)
    return err;
  if ((err = make_tmap_bf16_2d(&tV, pr.V, pr.M, pr.e, pr.e, 64, 64)) != cudaSuccess) return err;
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
  p.causal = pr.causal;
  p.n_et = pr.e / ET;
  p.n_qt = pr.C / QT;
  p.total = pr.B * pr.G * p.n_qt * p.n_et;
  p.inv_c = 1.0f / (float)pr.C;
  p.bias = pr.bias;
  p.status = pr.status;
  p.next_unit = pr.status + kNextUnitWord;
  const int grid = p.total < pr.num_sms ? p.total : pr.num_sms;
  return launch_pdl(chunk_attention_kernel, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, pr.stream,
                    tQq, tKq, tQl, tV, tPre, tU, tG, p);
}

}  // namespace flashgau
