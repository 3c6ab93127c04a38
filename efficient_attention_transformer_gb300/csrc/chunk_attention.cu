// Chunk attention of mixed chunk attention on tcgen05 tensor cores, bf16 with
// fp32 accumulation ("Transformer Quality in Linear Time", Method: local
// part, eq. 7/8 global part, display after eq. 8; flash_block pseudocode):
//
//   acc   = sum_kb relu^2(Q_quad K_quad[kb]^T / C + b) V[kb]    (local term)
//   acc  += Q_lin Prefix_g                                      (global term)
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
// Roles (576 threads):
//   warp 0     TMA producer: Q_lin, and one ring carrying Q_quad, K_quad,
//              V and prefix state tiles in the order the MMAs consume them;
//   warp 1     MMA issuer: S = Q_quad K_quad^T into a 128-column TMEM
//              buffer (two buffers), acc = P V with P read from TMEM, then
//              acc += Q_lin Prefix (smem A), so that the prefix states, which
//              the kernel launched before this one writes, are needed last;
//   warps 2-9  relu^2, two per TMEM lane quarter, each for 64 of a block's
//              128 keys: read S with tcgen05.ld, compute relu^2(S/C + b)
//              (the bias table carries the causal mask as -inf, written by
//              the projection kernel), write P as packed bf16
//              over the start of the same S columns with tcgen05.st (keys
//              0-63 at packed columns 0-31, keys 64-127 at 64-95); the
//              C x C scores never leave TMEM and registers;
//   warps 10-17 epilogue: gated = U * acc, two warps per TMEM lane quarter
//              (one per 64-column half of a value tile); U boxes TMA-loaded
//              into per-warp double buffers one value tile ahead, the
//              product written in place and TMA-stored.
// Two accumulators alternate between units, so while the epilogue warps
// drain one, the MMAs of the next unit already fill the other.
//
// The local term carries a factor local_scale (1 as written).  Any other
// non-zero value multiplies P in the relu^2 warps; 0 (global term only)
// gives every unit zero key blocks, so no Q_quad/K_quad/V tile is loaded
// and no score is formed: a unit is then acc = Q_lin Prefix and the gate.
//
// Shared memory (224 KB): Q_lin 32 KB, one ring of 8 x 16 KB stages for
// Q_quad and K_quad atoms and V / prefix half-blocks, epilogue boxes
// 8 warps x 2 x 4 KB.  TMEM: accumulators
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
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 32 * (2 + RELU_WARPS + EPI_WARPS);

constexpr int ATOM_BYTES = 128 * 64 * 2;  // 128 rows x 64 bf16: 16 KB
constexpr int Q_BYTES = 2 * ATOM_BYTES;   // 32 KB
constexpr int B_BOX_BYTES = 64 * 64 * 2;  // 64 rows x 64 columns: 8 KB
// One ring of 16 KB stages carries every streamed operand in the MMA
// issuer's order: a Q_quad or K_quad atom (128 rows x 64 columns) or half
// of a V / prefix block (64 rows x 128 columns, two 64 x 64 boxes).
constexpr int STAGE_BYTES = 16 * 1024;
constexpr int RING = 8;
constexpr int E_BOX_BYTES = 32 * 128;     // 32 rows x 64 bf16: 4 KB

constexpr int OFF_QL = 0;
constexpr int OFF_RING = OFF_QL + Q_BYTES;
constexpr int OFF_E = OFF_RING + RING * STAGE_BYTES;
constexpr int TILE_BYTES = OFF_E + EPI_WARPS * 2 * E_BOX_BYTES;  // 224 KB
constexpr int SMEM_BYTES = TILE_BYTES + 1024 + 512;

constexpr uint32_t TM_ACC = 0, TM_S = 256;

struct Bars {
  uint64_t ql_full, ql_empty;
  uint64_t full[RING], empty[RING];
  uint64_t s_full[2], p_full[2], sb_free[2];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t u_full[EPI_WARPS][2];
  uint64_t uq_full[4], uq_empty[4];  // unit-index queue
  volatile int unit_q[4];
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
};

struct AttnParams {
  int C, G, causal;
  int n_et, n_qt;   // value tiles (128 columns of e), query tiles per chunk
  int ng, n_vg;     // value tiles per grouped unit, groups per query tile
  int n_grouped;    // units (chunk, query tile, group of ng value tiles) of
                    // the first chunks, group fastest; after them, one
                    // unit per value tile (chunk, query tile, value tile)
                    // for the remaining chunks, so the schedule ends on
                    // small pieces of work
  int g_split;      // first chunk of the single-tile units
  int total;
  float inv_c;
  float local_scale;  // factor on P; 0: no key blocks at all
  int per_chunk;      // a prefix state per chunk (else one per batch row)
  const float *bias;  // [2C-1] relpos, -inf at causally masked offsets
  int *status;
  int *next_unit;  // work counter, zeroed by the projection kernel
  int lin_off;     // no global term: no Q_lin or prefix loads, no Q_lin Prefix MMA
  // chunks longer than the two S/P buffers (C > 256): a unit's value tiles
  // all take each key block's P in turn (key blocks outer), so that one S
  // and its relu^2 serve ng value tiles
  int kb_outer;
};

// Agents that consume each queued unit index: the MMA thread, the relu^2
// warps and the epilogue warps (one arrival per warp).
constexpr int QUEUE_AGENTS = 1 + RELU_WARPS + EPI_WARPS;

struct Unit {
  int chunk, b, qt, et0, ng, nkb;  // value tiles et0 .. et0 + ng - 1
  long long tok0;                  // first token of the chunk
  // Q_quad comes through the ring once per unit and stays until its last S
  // when the unit's last K block (ring position 4 (nkb - 1) + 1, counting
  // from Q) lands before the ring wraps onto Q; longer units load Q_quad
  // with every K block instead.
  bool q_per_block;
};

__device__ __forceinline__ Unit unit_of(const AttnParams &p, int u) {
  Unit x;
  int per_qt, chunk0 = 0;  // units per (chunk, query tile), first chunk
  if (u < p.n_grouped) {
    x.ng = p.ng;
    per_qt = p.n_vg;
  } else {
    u -= p.n_grouped;
    x.ng = 1;
    per_qt = p.n_et;
    chunk0 = p.g_split;
  }
  x.et0 = (u % per_qt) * x.ng;
  x.qt = p.n_qt - 1 - (u / per_qt) % p.n_qt;  // more key blocks first
  x.chunk = chunk0 + u / (per_qt * p.n_qt);
  x.b = x.chunk / p.G;
  x.tok0 = (long long)x.chunk * p.C;
  x.nkb = p.local_scale == 0.f ? 0 : p.causal ? x.qt + 1 : p.C / KB;
  x.q_per_block = 4 * (x.nkb - 1) + 1 >= RING;
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
// 64 S values are in registers before the first store lands.  SCALED: P is
// multiplied by local_scale.
template <bool SCALED>
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
    if (SCALED) {
      x0 *= p.local_scale;
      x1 *= p.local_scale;
    }
    if (j < 32) lo[j / 2] = pack_bf16(x0, x1);
    else hi[(j - 32) / 2] = pack_bf16(x0, x1);
  }
  tmem_st16(sbuf + c0, lo);
  tmem_st16(sbuf + c0 + 16, hi);
}

// KB_OUTER: chunks longer than 256 with key blocks outer (p.kb_outer); a
// separate instance, so that the other keeps its code as it is
template <bool KB_OUTER>
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
    mbar_init(smem_u32(&bar->ql_full), 1);
    mbar_init(smem_u32(&bar->ql_empty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar->acc_full[i]), 1);
      mbar_init(smem_u32(&bar->acc_empty[i]), 32 * EPI_WARPS);
      mbar_init(smem_u32(&bar->s_full[i]), 1);
      mbar_init(smem_u32(&bar->p_full[i]), 32 * RELU_WARPS);
      mbar_init(smem_u32(&bar->sb_free[i]), 1);
      for (int w = 0; w < EPI_WARPS; ++w) mbar_init(smem_u32(&bar->u_full[w][i]), 1);
    }
    for (int i = 0; i < RING; ++i) {
      mbar_init(smem_u32(&bar->full[i]), 1);
      mbar_init(smem_u32(&bar->empty[i]), 1);
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
    // Stages in the MMA issuer's order: per unit, Q_quad (two atoms) and
    // K block 0 (two atoms); then per value tile of the group, per key
    // block, the next K block (first value tile only, one block ahead of
    // its S; preceded by Q_quad again for units that stream it per block)
    // and the block's V rows (two halves), then the value tile's prefix
    // state rows (two halves).  Q_lin, read by every value tile of the
    // unit, has a buffer of its own.
    if (elect_one()) {
      Ring rr(RING);
      bool ok = true;
      // one stage: nbox boxes of map tm at columns x0, x0 + 64, .., row
      auto load = [&](const CUtensorMap *tm, int nbox, int x0, long long row) -> bool {
        if (!mbar_wait(smem_u32(&bar->empty[rr.stage]), rr.phase ^ 1, abort)) return false;
        const uint32_t f = smem_u32(&bar->full[rr.stage]);
        uint8_t *dst = tiles + OFF_RING + rr.stage * STAGE_BYTES;
        mbar_arrive_expect_tx(f, STAGE_BYTES);
        for (int j = 0; j < nbox; ++j)
          tma_load_2d(smem_u32(dst + j * (STAGE_BYTES / nbox)), tm, f, x0 + j * 64, (int)row);
        rr.next();
        return true;
      };
      auto load_atoms = [&](const CUtensorMap *tm, long long row) -> bool {
        return load(tm, 1, 0, row) && load(tm, 1, 64, row);
      };
      // next unit: from the global counter, announced through the queue
      auto push = [&](int q, int u) -> bool {
        if (!mbar_wait(smem_u32(&bar->uq_empty[q & 3]), ((q >> 2) & 1) ^ 1, abort)) return false;
        bar->unit_q[q & 3] = u;
        mbar_arrive(smem_u32(&bar->uq_full[q & 3]));
        return true;
      };
      // Without a global term the kernel before this one is the projection
      // itself (the chunk-state stage launches nothing): wait for it before
      // the first ticket, as the projection zeroes the work counter.
      bool prefix_ready = p.lin_off != 0;
      if (prefix_ready) griddep_wait();
      for (int i = 0;; ++i) {
        int u = atomicAdd(p.next_unit, 1);
        if (u >= p.total) u = -1;
        ok = push(i, u);
        if (!ok || u < 0) break;
        const Unit x = unit_of(p, u);
        const long long qrow = x.tok0 + x.qt * QT;
        const long long pre_row0 = (long long)(p.per_chunk ? x.chunk : x.b) * SD;
        const long long ncb = 2LL * p.n_et;  // 64-column blocks of e
        if (x.nkb > 0) ok = load_atoms(&tmQq, qrow) && load_atoms(&tmKq, x.tok0);
        if constexpr (KB_OUTER) {
          // per key block: the next K block, then this block's V rows of
          // every value tile; then Q_lin and every value tile's prefix
          for (int kb = 0; ok && kb < x.nkb; ++kb) {
            if (kb + 1 < x.nkb)
              ok = (!x.q_per_block || load_atoms(&tmQq, qrow)) &&
                   load_atoms(&tmKq, x.tok0 + (kb + 1) * KB);
            for (int t = 0; ok && t < x.ng; ++t) {
              const int col = (x.et0 + t) * ET;
              ok = load(&tmV, 1, 0, rb64_row(x.tok0 + kb * KB, col, ncb)) &&
                   load(&tmV, 1, 0, rb64_row(x.tok0 + kb * KB + 64, col, ncb));
            }
          }
          if (ok && !p.lin_off) {
            if (!prefix_ready) {
              griddep_wait();
              prefix_ready = true;
            }
            ok = mbar_wait(smem_u32(&bar->ql_empty), (i & 1) ^ 1, abort);
            if (!ok) break;
            const uint32_t f = smem_u32(&bar->ql_full);
            mbar_arrive_expect_tx(f, Q_BYTES);
            tma_load_2d(smem_u32(tiles + OFF_QL), &tmQl, f, 0, (int)qrow);
            tma_load_2d(smem_u32(tiles + OFF_QL + ATOM_BYTES), &tmQl, f, 64, (int)qrow);
            for (int t = 0; ok && t < x.ng; ++t) {
              const int col = (x.et0 + t) * ET;
              ok = load(&tmPre, 1, 0, rb64_row(pre_row0, col, ncb)) &&
                   load(&tmPre, 1, 0, rb64_row(pre_row0 + 64, col, ncb));
            }
          }
        } else {
        for (int t = 0; ok && t < x.ng; ++t) {
          const int col = (x.et0 + t) * ET;
          for (int kb = 0; ok && kb < x.nkb; ++kb) {
            if (t == 0 && kb + 1 < x.nkb)
              ok = (!x.q_per_block || load_atoms(&tmQq, qrow)) &&
                   load_atoms(&tmKq, x.tok0 + (kb + 1) * KB);
            ok = ok && load(&tmV, 1, 0, rb64_row(x.tok0 + kb * KB, col, ncb)) &&
                 load(&tmV, 1, 0, rb64_row(x.tok0 + kb * KB + 64, col, ncb));
          }
          if (p.lin_off) continue;  // local term only
          if (ok && t == 0) {
            // the global term last: the prefix states come from the kernel
            // launched just before this one, which may still be running
            if (!prefix_ready) {
              griddep_wait();
              prefix_ready = true;
            }
            ok = mbar_wait(smem_u32(&bar->ql_empty), (i & 1) ^ 1, abort);
            if (!ok) break;
            const uint32_t f = smem_u32(&bar->ql_full);
            mbar_arrive_expect_tx(f, Q_BYTES);
            tma_load_2d(smem_u32(tiles + OFF_QL), &tmQl, f, 0, (int)qrow);
            tma_load_2d(smem_u32(tiles + OFF_QL + ATOM_BYTES), &tmQl, f, 64, (int)qrow);
          }
          ok = ok && load(&tmPre, 1, 0, rb64_row(pre_row0, col, ncb)) &&
               load(&tmPre, 1, 0, rb64_row(pre_row0 + 64, col, ncb));
        }
        }
        if (!ok) break;
      }
      if (!ok) raise_timeout(bar, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (elect_one()) {
      const uint32_t idesc_s = idesc_bf16_f32(128, KB, 0, 0);
      const uint32_t idesc_v = idesc_bf16_f32(128, ET, 0, 1);
      const uint32_t sQL = smem_u32(tiles + OFF_QL);
      const uint32_t sRing = smem_u32(tiles + OFF_RING);
      Ring rr(RING);
      int n = 0;  // S blocks issued so far (all units): buffer n & 1
      int v = 0;  // value tiles issued so far (all units): accumulator v & 1
      uint32_t acc_col = TM_ACC;  // accumulator of the current value tile
      int q_stage[2] = {0, 0};    // ring stages of the unit's Q_quad atoms
      bool ok = true;
      // the next ring stage, once full: its index
      auto next_stage = [&](int &st) -> bool {
        if (!mbar_wait(smem_u32(&bar->full[rr.stage]), rr.phase, abort)) return false;
        st = rr.stage;
        rr.next();
        return true;
      };
      auto stage_addr = [&](int st) -> uint32_t { return sRing + st * STAGE_BYTES; };
      // S[n] = Q_quad K_quad^T into TMEM buffer n & 1.  Q_quad's atoms come
      // from the ring with the unit's first S and stay until its last, or
      // come with every S (q_per_block).
      auto issue_s = [&](bool q_new, bool q_done) -> bool {
        const int sb = n & 1;
        if (n >= 2 && !mbar_wait(smem_u32(&bar->sb_free[sb]), ((n >> 1) - 1) & 1, abort))
          return false;
        if (q_new && !(next_stage(q_stage[0]) && next_stage(q_stage[1]))) return false;
        int k_stage[2];
        if (!(next_stage(k_stage[0]) && next_stage(k_stage[1]))) return false;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < SD / 16; ++k) {
          const uint64_t dq = sw128_desc(stage_addr(q_stage[k >> 2]), 16, 1024);
          const uint64_t dk = sw128_desc(stage_addr(k_stage[k >> 2]), 16, 1024);
          mma_f16_ss(tmem + TM_S + sb * KB, desc_advance(dq, (k & 3) * 32),
                     desc_advance(dk, (k & 3) * 32), idesc_s, k != 0);
        }
        mma_commit(smem_u32(&bar->empty[k_stage[0]]));
        mma_commit(smem_u32(&bar->empty[k_stage[1]]));
        mma_commit(smem_u32(&bar->s_full[sb]));
        if (q_done) {
          mma_commit(smem_u32(&bar->empty[q_stage[0]]));
          mma_commit(smem_u32(&bar->empty[q_stage[1]]));
        }
        ++n;
        return true;
      };
      // acc (+)= A * B stage, A a 64-wide K-major atom in shared memory
      auto issue_b_smem = [&](uint32_t a_atom, bool first) -> bool {
        int st;
        if (!next_stage(st)) return false;
        tc_fence_after();
        const uint64_t da = sw128_desc(a_atom, 16, 1024);
        const uint64_t db = sw128_desc(stage_addr(st), B_BOX_BYTES, 1024);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16_ss(tmem + acc_col, desc_advance(da, k * 32), desc_advance(db, k * 2048), idesc_v,
                     !(first && k == 0));
        mma_commit(smem_u32(&bar->empty[st]));
        return true;
      };
      // acc += P * B stage, P: 64 keys = 32 packed columns of TMEM at a_col
      auto issue_b_tmem = [&](uint32_t a_col, bool first) -> bool {
        int st;
        if (!next_stage(st)) return false;
        tc_fence_after();
        const uint64_t db = sw128_desc(stage_addr(st), B_BOX_BYTES, 1024);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16_ts(tmem + acc_col, tmem + a_col + k * 8, desc_advance(db, k * 2048), idesc_v,
                     !(first && k == 0));
        mma_commit(smem_u32(&bar->empty[st]));
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
        if (x.nkb > 0) ok = issue_s(true, x.q_per_block || x.nkb == 1);
        if constexpr (KB_OUTER) {
          // every accumulator of the unit drained by the epilogue first (the
          // first S above overlaps that)
          for (int t = 0; ok && t < x.ng; ++t)
            ok = mbar_wait(smem_u32(&bar->acc_empty[(v + t) & 1]), (((v + t) >> 1) & 1) ^ 1, abort);
          if (!ok) break;
          tc_fence_after();
          for (int kb = 0; ok && kb < x.nkb; ++kb) {
            const int si = n0 + kb, sb = si & 1;
            if (kb + 1 < x.nkb) ok = issue_s(x.q_per_block, x.q_per_block || kb + 2 == x.nkb);
            ok = ok && mbar_wait(smem_u32(&bar->p_full[sb]), (si >> 1) & 1, abort);
            if (!ok) break;
            tc_fence_after();
            const uint32_t pcol = TM_S + sb * KB;
            for (int t = 0; ok && t < x.ng; ++t) {
              acc_col = TM_ACC + ((v + t) & 1) * ET;
              ok = issue_b_tmem(pcol, kb == 0) && issue_b_tmem(pcol + 64, false);
            }
            if (ok) mma_commit(smem_u32(&bar->sb_free[sb]));
          }
          if (ok && !p.lin_off) {
            ok = mbar_wait(smem_u32(&bar->ql_full), i & 1, abort);
            if (ok) tc_fence_after();
            for (int t = 0; ok && t < x.ng; ++t) {
              acc_col = TM_ACC + ((v + t) & 1) * ET;
              // with no key blocks the global term opens the accumulator
              ok = issue_b_smem(sQL, x.nkb == 0) && issue_b_smem(sQL + ATOM_BYTES, false);
            }
            if (ok) mma_commit(smem_u32(&bar->ql_empty));
          }
          if (!ok) break;
          for (int t = 0; t < x.ng; ++t) mma_commit(smem_u32(&bar->acc_full[(v + t) & 1]));
          v += x.ng;
        } else {
        // P of the unit's key blocks stays in TMEM for all its value tiles
        for (int t = 0; ok && t < x.ng; ++t, ++v) {
          const bool last_t = t + 1 == x.ng;
          // this value tile's accumulator must have been drained by the
          // epilogue of the value tile two before
          acc_col = TM_ACC + (v & 1) * ET;
          ok = mbar_wait(smem_u32(&bar->acc_empty[v & 1]), ((v >> 1) & 1) ^ 1, abort);
          if (!ok) break;
          tc_fence_after();
          // local term first, global term (Q_lin Prefix) last
          for (int kb = 0; ok && kb < x.nkb; ++kb) {
            const int si = n0 + kb, sb = si & 1;
            if (t == 0) {
              if (kb + 1 < x.nkb)
                ok = issue_s(x.q_per_block, x.q_per_block || kb + 2 == x.nkb);
              ok = ok && mbar_wait(smem_u32(&bar->p_full[sb]), (si >> 1) & 1, abort);
              if (!ok) break;
              tc_fence_after();
            }
            const uint32_t pcol = TM_S + sb * KB;
            ok = issue_b_tmem(pcol, kb == 0) && issue_b_tmem(pcol + 64, false);
            if (ok && last_t) mma_commit(smem_u32(&bar->sb_free[sb]));
          }
          if (!p.lin_off) {
            if (ok && t == 0) {
              ok = mbar_wait(smem_u32(&bar->ql_full), i & 1, abort);
              if (ok) tc_fence_after();
            }
            // with no key blocks the global term opens the accumulator
            ok = ok && issue_b_smem(sQL, x.nkb == 0) && issue_b_smem(sQL + ATOM_BYTES, false);
            if (!ok) break;
            if (last_t) mma_commit(smem_u32(&bar->ql_empty));
          }
          if (!ok) break;
          mma_commit(smem_u32(&bar->acc_full[v & 1]));
        }
        }
        if (!ok) break;
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
        if (p.local_scale == 1.f)
          relu2_half<false>(tmem + lane_off + TM_S + sb * KB, p, kb, x.qt, r, half);
        else
          relu2_half<true>(tmem + lane_off + TM_S + sb * KB, p, kb, x.qt, r, half);
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
    // Two warps per TMEM lane quarter, one per 64-column half of every
    // value tile.  A warp's two boxes alternate between value tiles: the U
    // box of the next value tile is requested when the current one starts,
    // the gated product is written over the current box and TMA-stored.
    const int w = warp - (2 + RELU_WARPS);
    const int quarter = warp & 3, half = w >> 2;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint8_t *ebuf = tiles + OFF_E + w * 2 * E_BOX_BYTES;
    // this warp's U box of value tile t of unit u into buffer b
    auto load_u = [&](int u, int t, int b) {
      if (lane != 0 || u < 0) return;
      const Unit x = unit_of(p, u);
      const uint32_t f = smem_u32(&bar->u_full[w][b]);
      mbar_arrive_expect_tx(f, E_BOX_BYTES);
      tma_load_2d(smem_u32(ebuf + b * E_BOX_BYTES), &tmU, f, (x.et0 + t) * ET + half * 64,
                  (int)(x.tok0 + x.qt * QT + quarter * 32));
    };
    bool ok = true;
    int cur = pop(0);
    ok = cur != -2;
    load_u(cur, 0, 0);
    int v = 0;
    for (int i = 0; ok && cur >= 0; ++i) {
      const Unit x = unit_of(p, cur);
      const int grow = (int)(x.tok0 + x.qt * QT + quarter * 32);
      int nxt = -1;
      for (int t = 0; ok && t < x.ng; ++t, ++v) {
        const int b = v & 1;
        // At the unit's last value tile, the next unit's index (released
        // later).  Not earlier: the producer announces it only after all of
        // this unit's loads, which need the earlier value tiles drained.
        if (t + 1 == x.ng) {
          nxt = pop(i + 1);
          if (nxt == -2) {
            ok = false;
            break;
          }
        }
        // the other box: its store (of the previous value tile) has read
        // it, refill it with the next value tile's U
        if (lane == 0) tma_store_wait_read<0>();
        __syncwarp();
        if (t + 1 < x.ng) load_u(cur, t + 1, b ^ 1);
        else load_u(nxt, 0, b ^ 1);
        if (!mbar_wait(smem_u32(&bar->acc_full[v & 1]), (v >> 1) & 1, abort) ||
            !mbar_wait(smem_u32(&bar->u_full[w][b]), (v >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t va[32], vb[32];
        const uint32_t acc = tmem + lane_off + TM_ACC + (v & 1) * ET + half * 64;
        tmem_ld32(acc, va);
        tmem_ld32(acc + 32, vb);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar->acc_empty[v & 1]));
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
          tma_store_2d(&tmG, smem_u32(box), (x.et0 + t) * ET + half * 64, grow);
          tma_store_commit();
        }
        __syncwarp();
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
  // V and the prefix states in 64 x 64 blocks (flat 128-byte rows): 64 rows
  // of a value tile are one contiguous 128-row box
  if ((err = make_tmap_bf16_2d(&tV, pr.V, pr.M * pr.e / 64, 64, 64, 128, 64)) != cudaSuccess)
    return err;
  if ((err = make_tmap_bf16_2d(&tU, pr.U, pr.M, pr.e, pr.e, 32, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tG, pr.gated, pr.M, pr.e, pr.e, 32, 64)) != cudaSuccess) return err;
  const long long pre_rows = (long long)(pr.per_chunk ? pr.B * pr.G : pr.B) * pr.s;
  if ((err = make_tmap_bf16_2d(&tPre, pr.prefix, pre_rows * pr.e / 64, 64, 64, 128, 64)) !=
      cudaSuccess)
    return err;

  static unsigned long long configured = 0;
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev < 64 && !(configured & (1ull << dev))) {
    err = cudaFuncSetAttribute(chunk_attention_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(chunk_attention_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (err != cudaSuccess) return err;
    configured |= 1ull << dev;
  }
  AttnParams p;
  p.C = pr.C;
  p.G = pr.G;
  p.causal = pr.causal;
  p.n_et = pr.e / ET;
  p.n_qt = pr.C / QT;
  // Value tiles per unit: the unit's P is computed once and stays in TMEM
  // for each of them, which takes a unit's key blocks fitting the two S/P
  // buffers (C <= 256); else one.  As many as divide the value tiles while
  // leaving at least one unit per SM (the single-tile units at the end of
  // the schedule balance the SMs' finishing times).
  const long long tiles = (long long)pr.B * pr.G * p.n_qt * p.n_et;
  p.ng = 1;
  for (int ng : {4, 3, 2})
    if (pr.C <= 2 * KB && p.n_et % ng == 0 && tiles / ng >= pr.num_sms) {
      p.ng = ng;
      break;
    }
  // Longer chunks: key blocks outer, two value tiles a unit (the two
  // accumulators), when that still leaves about two units per SM
  p.kb_outer = 0;
  if (pr.C > 2 * KB && p.n_et % 2 == 0 && tiles / 2 >= 2LL * pr.num_sms) {
    p.kb_outer = 1;
    p.ng = 2;
  }
  p.n_vg = p.n_et / p.ng;
  // the last chunks as single-tile units: about one for every two SMs (one
  // per SM, or two, ended the schedule later on the long workload)
  const int BG = pr.B * pr.G, per_chunk = p.n_qt * p.n_et;
  int singles = p.ng > 1 ? (pr.num_sms / 2 + per_chunk - 1) / per_chunk : BG;
  if (singles > BG) singles = BG;
  p.g_split = BG - singles;
  p.n_grouped = p.g_split * p.n_qt * p.n_vg;
  p.total = p.n_grouped + singles * per_chunk;
  p.inv_c = 1.0f / (float)pr.C;
  p.local_scale = pr.local_scale;
  p.per_chunk = pr.per_chunk;
  p.bias = pr.bias;
  p.status = pr.status;
  p.next_unit = pr.status + kNextUnitWord;
  p.lin_off = pr.lin_off;
  const int grid = p.total < pr.num_sms ? p.total : pr.num_sms;
  if (p.kb_outer)
    return launch_pdl(chunk_attention_kernel<true>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES,
                      pr.stream, tQq, tKq, tQl, tV, tPre, tU, tG, p);
  return launch_pdl(chunk_attention_kernel<false>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES,
                    pr.stream, tQq, tKq, tQl, tV, tPre, tU, tG, p);
}

}  // namespace flashgau
