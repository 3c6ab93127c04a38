// Pair (2-SM) tcgen05 GEMM with fused epilogues for the two large dense
// contractions of the FLASH GAU forward, bf16 in, fp32 accumulation:
//   projection   [U|V|Z] = swish(X W_uvz); the Z tile's epilogue writes the
//                four scale/offset heads Z*gamma_h + beta_h
//                ("Transformer Quality in Linear Time", Method, eq. 5 and
//                 the four heads of mixed chunk attention)
//   output       O = gated W_o                   (display after eq. 8)
// and for the backward pass's weight-sized ones: the recompute of X W_uvz
// (with V, Z and the heads), dA = dO W_o^T with the gate's gradient in its
// epilogue, and dX = dPre W_uvz^T (a K-major B).
//
// A cluster of two CTAs on neighbouring SMs computes 256 x 256 output tiles
// with tcgen05.mma.cta_group::2 (M = 256): each CTA holds its own 128 rows
// of A and half of the B columns of every 64-deep k-block (32 KB per stage,
// 6 stages), so each SM moves two thirds of the operand bytes a single-SM
// 128 x 256 tile needs.  The leader CTA's warp 1 issues the MMAs; both CTAs'
// TMA loads complete on the leader's stage barrier; the leader's commits
// release the stage, and announce a finished accumulator, in both CTAs.
// Each CTA's TMEM holds its own 128 rows (two 256-column accumulators); its
// eight epilogue warps (two per TMEM lane quarter, each half of the
// columns) drain them through tcgen05.ld into swizzled staging and TMA
// stores, and report the accumulator free to the leader.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <vector>

#include "flash_gau_internal.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace flashgau {
namespace {

using namespace ptx;

constexpr int BM = 128;                          // rows per CTA (256 per pair)
constexpr int BN = 256;                          // columns per pair tile
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;         // 8 KB: 64 columns x 64 k-rows
constexpr int STAGE_BYTES = A_BYTES + BN / 2 * BK * 2;  // 32 KB
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 2 * ACC_COLS;
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 32 * (2 + EPI_WARPS);  // producer, MMA issuer, epilogue
constexpr int STG_BYTES = 32 * 128;                // one 32-row x 128-byte store box
// Shared memory of an instance: the stage ring, then each epilogue warp's
// staging boxes (one; the gate-gradient epilogue three: its two operand
// boxes and a store box, with a shorter ring to make room)
constexpr uint16_t kPair = 0x3, kLeader = 0x1;

// EPI_PROJ_ROPE: the projection with the flash_block RoPE of the heads, a
// separate instance so that its register needs stay out of the plain one.
// EPI_RECOMPUTE: the backward pass's recompute of X W_uvz: Pre in bf16 for
// every column, and from its bf16 values the V activations (row-major bf16),
// Z (fp32) and the four heads (bf16) that the backward's contractions read.
// EPI_GATE_GRAD: the backward's dA = dO W_o^T, and from it in the epilogue
// (with Pre_u and Vh boxes loaded by TMA) the gate's gradient:
// dVh = dA * swish(Pre_u) and the U part of dPre = (dA * Vh) * swish'(Pre_u),
// the latter in place over Pre_u; dA itself is not stored.
enum Epi { EPI_PROJ = 0, EPI_STORE = 1, EPI_PROJ_ROPE = 2, EPI_RECOMPUTE = 3, EPI_GATE_GRAD = 4 };

template <int EPI>
struct Layout {
  static constexpr int stages = EPI == EPI_GATE_GRAD ? 4 : STAGES;
  static constexpr int boxes = EPI == EPI_GATE_GRAD ? 3 : 1;  // staging boxes per epilogue warp
  static constexpr int stg_off = stages * STAGE_BYTES;
  static constexpr int tile_bytes = stg_off + EPI_WARPS * boxes * STG_BYTES;
  static constexpr int smem_bytes = tile_bytes + 1024 /*align*/ + 256 /*barriers*/;
  static_assert(smem_bytes <= 227 * 1024, "shared memory of one CTA");
};

struct Params {
  int N, K;        // output columns, contraction depth
  int bn;          // columns per pair tile of the first rp_split row pairs: 256 or 128
  int m_tiles;     // 128-row tiles of the output
  int n_tiles;     // bn-column pair tiles per row pair
  // the row pairs from rp_split on (a last, partial round of tiles) in
  // 128-column tiles, n_tiles2 per row pair, from tile index t_split on
  int rp_split, n_tiles2, t_split;
  int total;       // pair tiles
  const float *gamma, *beta;
  int M_tokens;
  int e, s;
  int *status;
  int *sched;  // projection: the scheduling words of the workspace, zeroed here
  // projection: the attention kernel's bias table, written here
  const float *relpos;
  float *bias;
  int C, causal;
  // projection with RoPE (flash_block): heads rotated at positions
  // t + pos_offset
  int T_seq;
  const uint32_t *rope_cs;  // [s / 2][T] half2 (cos, sin)
  // output (flash_block): the shortcut added to O, or null
  const __nv_bfloat16 *residual;
  // recompute: Z in fp32, [M, s]
  float *zf;
};

struct Smem {
  uint64_t full[STAGES];   // leader: both CTAs' loads of a stage landed
  uint64_t empty[STAGES];  // both: the pair MMAs have read the stage
  uint64_t acc_full[2];    // both: an accumulator is ready
  uint64_t acc_empty[2];   // leader: both CTAs drained an accumulator
  uint64_t drain;
  uint64_t ebar[EPI_WARPS];  // gate gradient: an epilogue warp's operand boxes landed
  uint32_t tmem_base;
  volatile int abort_flag;
};

__device__ __forceinline__ void raise_timeout(Smem *sm, int *status) {
  sm->abort_flag = 1;
  atomicExch(status, FLASH_GAU_ETIMEOUT);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// Per-warp staged TMA store: the warp writes one 32-row x 128-byte box into
// its staging buffer (row = lane, swizzled), then lane 0 stores it.  The
// buffer is rewritten only after the previous store has finished reading
// shared memory.
struct Stager {
  uint8_t *buf;  // this warp's 4 KB
  int lane;
  int count = 0;
  __device__ uint8_t *begin() {
    if (lane == 0) tma_store_wait_read<0>();
    __syncwarp();
    return buf;
  }
  // row data: 8 x 16 bytes
  __device__ void put(uint8_t *b, const uint4 (&w)[8]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(b + sw128_offset(lane, c)) = w[c];
  }
  // keep: store with the L2 evict_last policy, for data the next kernels
  // read again
  __device__ void finish(uint8_t *b, const CUtensorMap *tm, int x, int y, bool keep = false) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (keep) tma_store_2d_hint(tm, smem_u32(b), x, y, l2_evict_last());
      else tma_store_2d(tm, smem_u32(b), x, y);
      tma_store_commit();
    }
    ++count;
  }
  __device__ void drain() {
    if (lane == 0) tma_store_wait<0>();
    __syncwarp();
  }
};

// 64 accumulator columns of this thread's row -> 8 x 16 bytes of bf16
template <typename F>
__device__ __forceinline__ void pack64(const uint32_t (&a)[32], const uint32_t (&b)[32], F f,
                                       uint4 (&w)[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t *src = c < 4 ? &a[8 * c] : &b[8 * (c - 4)];
    const int col = 8 * c;
    w[c].x = pack_bf16(f(__uint_as_float(src[0]), col + 0), f(__uint_as_float(src[1]), col + 1));
    w[c].y = pack_bf16(f(__uint_as_float(src[2]), col + 2), f(__uint_as_float(src[3]), col + 3));
    w[c].z = pack_bf16(f(__uint_as_float(src[4]), col + 4), f(__uint_as_float(src[5]), col + 5));
    w[c].w = pack_bf16(f(__uint_as_float(src[6]), col + 6), f(__uint_as_float(src[7]), col + 7));
  }
}

// B_KM: B is the transpose of a row-major [N, K] matrix (K-major), each
// CTA's half of the tile's columns one box of up to 128 rows x 64 k;
// otherwise B is a row-major [K, N] matrix (N-major), 64-column boxes.
// TAIL: the launch's last row pairs run 128-column tiles (plan_tiles); a
// separate instance, so that launches without one keep the plain mapping
template <int EPI, bool B_KM = false, bool TAIL = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC0,
                    const __grid_constant__ CUtensorMap tmC1,
                    const __grid_constant__ CUtensorMap tmC2, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *tiles = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using L = Layout<EPI>;
  Smem *sm = reinterpret_cast<Smem *>(tiles + L::tile_bytes);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rank = (int)cluster_ctarank();  // 0 = leader of the pair
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::stages; ++i) {
      mbar_init(smem_u32(&sm->full[i]), 1);
      mbar_init(smem_u32(&sm->empty[i]), 1);
    }
    for (int i = 0; i < EPI_WARPS; ++i) mbar_init(smem_u32(&sm->ebar[i]), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm->acc_full[i]), 1);
      mbar_init(smem_u32(&sm->acc_empty[i]), 2 * EPI_WARPS);  // all epilogue warps, 2 CTAs
    }
    mbar_init(smem_u32(&sm->drain), 1);
    sm->abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&sm->tmem_base), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers and TMEM exist before any remote access
  tc_fence_after();
  // setup above overlaps the previous kernel's tail; its outputs are read below
  griddep_wait();
  griddep_launch_dependents();
  // The chunk-state kernel's grid barrier and the chunk-attention kernel's
  // work counter start from zero.  Both kernels touch them only after this
  // grid has completed (the first after its griddepcontrol.wait, the second
  // once every CTA of the first has passed that wait), and the previous
  // forward's kernels had all completed before this one got past its wait.
  if ((EPI == EPI_PROJ || EPI == EPI_PROJ_ROPE) && blockIdx.x == 0) {
    if (threadIdx.x == 0) {
      p.sched[kNextUnitWord] = 0;
      p.sched[kGridBarrierWord] = 0;
    }
    // The relative-position bias as the attention kernel reads it.  Causal:
    // an offset j - i >= 1 (a later key) gets -inf, so that relu^2(S/C + b)
    // is exactly 0 there and no separate mask is applied.
    for (int k = threadIdx.x; k < 2 * p.C - 1; k += blockDim.x)
      p.bias[k] = (p.causal && k >= p.C) ? -INFINITY : p.relpos[k];
  }
  const uint32_t tmem_base = sm->tmem_base;
  const int kblocks = p.K / BK;
  const int first = blockIdx.x / 2, step = gridDim.x / 2;
  // Pair tile t: row pair rp, columns n0 .. n0 + nsz.  Tiles before t_split
  // are bn wide (row pairs in order, n-tiles fastest), the rest 128 wide.
  // The output projection walks the rows last first: the attention kernel
  // wrote the last rows of the gated product most recently, so they are
  // still in L2.
  auto geom = [&](int t, int &rp, int &n0, int &nsz) {
    int w;
    if (!TAIL || t < p.t_split) {
      rp = t / p.n_tiles;
      n0 = (t % p.n_tiles) * p.bn;
      w = p.bn;
    } else {
      const int u = t - p.t_split;
      rp = p.rp_split + u / p.n_tiles2;
      n0 = (u % p.n_tiles2) * (BN / 2);
      w = BN / 2;
    }
    nsz = min(w, p.N - n0);
    if (EPI == EPI_STORE) rp = (p.m_tiles + 1) / 2 - 1 - rp;
  };

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both)
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = first; t < p.total && !sm->abort_flag; t += step) {
        int rp, n0, nsz;
        geom(t, rp, n0, nsz);
        const int mt = rp * 2 + rank;
        // an overhanging CTA of the last pair re-reads the last valid rows
        // (its results are discarded) so every box is in bounds
        const int arow = min(mt, p.m_tiles - 1) * BM;
        const int half = nsz / 2, hboxes = half / 64;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, &sm->abort_flag)) {
            raise_timeout(sm, p.status);
            break;
          }
          const uint32_t full_own = smem_u32(&sm->full[stage]);
          const uint32_t full_leader = mapa_shared(full_own, 0);
          uint8_t *sA = tiles + stage * STAGE_BYTES;
          uint8_t *sB = sA + A_BYTES;
          // a K-major B box is always 128 rows (rows past the tile's half
          // are read and unused)
          const uint32_t b_bytes = B_KM ? 2 * B_BOX_BYTES : hboxes * B_BOX_BYTES;
          if (leader) mbar_arrive_expect_tx(full_own, 2 * (A_BYTES + b_bytes));
          tma_load_2d_pair(smem_u32(sA), &tmA, full_leader, kb * BK, arow);
          if (B_KM) {
            tma_load_2d_pair(smem_u32(sB), &tmB, full_leader, kb * BK, n0 + rank * half);
          } else {
            for (int j = 0; j < hboxes; ++j)
              tma_load_2d_pair(smem_u32(sB + j * B_BOX_BYTES), &tmB, full_leader,
                               n0 + rank * half + j * 64, kb * BK);
          }
          if (++stage == L::stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (leader)
    if (leader && elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int t = first; t < p.total && !sm->abort_flag; t += step, ++local) {
        int rp, n0, nsz;
        geom(t, rp, n0, nsz);
        const int acc = local & 1;
        if (!mbar_wait(smem_u32(&sm->acc_empty[acc]), ((local >> 1) & 1) ^ 1, &sm->abort_flag)) {
          raise_timeout(sm, p.status);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        const uint32_t idesc = idesc_bf16_f32(2 * BM, nsz, 0, B_KM ? 0 : 1);
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(smem_u32(&sm->full[stage]), phase, &sm->abort_flag)) {
            raise_timeout(sm, p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(tiles + stage * STAGE_BYTES);
          // A: K-major, 16 elements (32 B) per step inside the swizzle atom;
          // B: N-major, 16 rows of 128 B per step, 64-column boxes 8 KB
          // apart (or K-major like A)
          const uint64_t da = sw128_desc(sA, 16, 1024);
          const uint64_t db = B_KM ? sw128_desc(sA + A_BYTES, 16, 1024)
                                   : sw128_desc(sA + A_BYTES, B_BOX_BYTES, 1024);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_f16_ss_pair(d_tmem, desc_advance(da, k * 32),
                            desc_advance(db, B_KM ? k * 32 : k * 2048), idesc, (kb | k) != 0);
          mma_commit_pair_mc(smem_u32(&sm->empty[stage]), kPair);
          if (++stage == L::stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair_mc(smem_u32(&sm->acc_full[acc]), kPair);
      }
      // every MMA this thread issued has completed once `drain` flips
      mma_commit_pair_mc(smem_u32(&sm->drain), kLeader);
      if (!mbar_wait(smem_u32(&sm->drain), 0)) raise_timeout(sm, p.status);
    }
  } else {
    // -------------------------------------------------- epilogue (both)
    const int quarter = warp & 3;       // TMEM lanes 32*quarter .. +31
    const int half = (warp - 2) >> 2;   // which half of the tile's columns
    Stager st{tiles + L::stg_off + (warp - 2) * L::boxes * STG_BYTES, lane};
    if constexpr (EPI == EPI_GATE_GRAD) {
      // boxes: st.buf carries dVh; xb is Pre_u, then dPre_u in place; vb is Vh
      uint8_t *xb = st.buf + STG_BYTES, *vb = st.buf + 2 * STG_BYTES;
      const uint32_t ebar = smem_u32(&sm->ebar[warp - 2]);
      uint32_t e_issued = 0, e_used = 0;
      auto load_e = [&](int col, int row) {
        if (lane == 0) {
          tma_store_wait_read<0>();  // the previous box's stores have read xb
          mbar_arrive_expect_tx(ebar, 2 * STG_BYTES);
          tma_load_2d(smem_u32(xb), &tmC1, ebar, col, row);
          tma_load_2d(smem_u32(vb), &tmC2, ebar, col, row);
        }
        ++e_issued;
      };
      int local = 0;
      for (int t = first; t < p.total && !sm->abort_flag; t += step, ++local) {
        int rp, n0, nsz;
        geom(t, rp, n0, nsz);
        const int mt = rp * 2 + rank;
        const bool valid = mt < p.m_tiles;
        const int acc = local & 1;
        const int row0 = mt * BM + quarter * 32;
        const int cbeg = half * (nsz / 2), cend = (half + 1) * (nsz / 2);
        // the first box's operands load while the accumulator fills
        if (valid) load_e(n0 + cbeg, row0);
        if (!mbar_wait(smem_u32(&sm->acc_full[acc]), (local >> 1) & 1, &sm->abort_flag)) {
          raise_timeout(sm, p.status);
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * ACC_COLS;
        bool ok = true;
        for (int c0 = cbeg; c0 < cend; c0 += 64) {
          if (valid && c0 != cbeg) load_e(n0 + c0, row0);
          uint32_t ra[32], rb[32];
          tmem_ld32(taddr + c0, ra);
          tmem_ld32(taddr + c0 + 32, rb);
          tmem_ld_wait();
          if (c0 + 64 >= cend) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&sm->acc_empty[acc]), 0));
          }
          if (!valid) continue;
          if (!mbar_wait(ebar, e_used & 1, &sm->abort_flag)) {
            raise_timeout(sm, p.status);
            ok = false;
            break;
          }
          ++e_used;
          // dA as bf16 (as the separate kernel read it), with this row's Pre_u and Vh
          uint4 w[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t *src = q < 4 ? &ra[8 * q] : &rb[8 * (q - 4)];
            const uint4 xv = *reinterpret_cast<const uint4 *>(xb + sw128_offset(lane, q));
            const uint4 vv = *reinterpret_cast<const uint4 *>(vb + sw128_offset(lane, q));
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, vw[4] = {vv.x, vv.y, vv.z, vv.w};
            uint32_t dvh[4], dpu[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 a = __bfloat1622float2(__floats2bfloat162_rn(
                  __uint_as_float(src[2 * j]), __uint_as_float(src[2 * j + 1])));
              const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xw[j]));
              const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&vw[j]));
              dvh[j] = pack_bf16(a.x * swish_fast(x.x), a.y * swish_fast(x.y));
              dpu[j] = pack_bf16((a.x * v.x) * swish_grad_fast(x.x), (a.y * v.y) * swish_grad_fast(x.y));
            }
            w[q] = make_uint4(dvh[0], dvh[1], dvh[2], dvh[3]);
            *reinterpret_cast<uint4 *>(xb + sw128_offset(lane, q)) =
                make_uint4(dpu[0], dpu[1], dpu[2], dpu[3]);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4 *>(st.buf + sw128_offset(lane, q)) = w[q];
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC0, smem_u32(st.buf), n0 + c0, row0);
            tma_store_2d(&tmC1, smem_u32(xb), n0 + c0, row0);
            tma_store_commit();
          }
        }
        if (!ok) break;
      }
      // operands still in flight (an early exit) land before the shared
      // memory is given up
      if (e_issued > e_used) mbar_wait(ebar, e_used & 1);
      if (lane == 0) tma_store_wait<0>();
      __syncwarp();
    } else {
    int local = 0;
    for (int t = first; t < p.total && !sm->abort_flag; t += step, ++local) {
      int rp, n0, nsz;
      geom(t, rp, n0, nsz);
      const int mt = rp * 2 + rank;
      const bool valid = mt < p.m_tiles;
      const int acc = local & 1;
      if (!mbar_wait(smem_u32(&sm->acc_full[acc]), (local >> 1) & 1, &sm->abort_flag)) {
        raise_timeout(sm, p.status);
        break;
      }
      tc_fence_after();
      const int row0 = mt * BM + quarter * 32;  // first row of this warp's box
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * ACC_COLS;
      const int cend = (half + 1) * (nsz / 2);
      for (int c0 = half * (nsz / 2); c0 < cend; c0 += 64) {
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr + c0, ra);
        tmem_ld32(taddr + c0 + 32, rb);
        tmem_ld_wait();
        if (c0 + 64 >= cend) {
          // the accumulator is drained: tell the leader (one arrival per warp)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&sm->acc_empty[acc]), 0));
        }
        if (!valid) continue;
        if constexpr (EPI == EPI_RECOMPUTE) {
          const int n = n0 + c0;
          uint4 w[8];
          pack64(ra, rb, [](float x, int) { return x; }, w);
          {
            uint8_t *b = st.begin();
            st.put(b, w);
            st.finish(b, &tmC0, n, row0);
          }
          if (n >= p.e) {
            // swish of the bf16 Pre, with the backward's sigmoid
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float xa = __bfloat162float(__float2bfloat16_rn(__uint_as_float(ra[j])));
              const float xb = __bfloat162float(__float2bfloat16_rn(__uint_as_float(rb[j])));
              ra[j] = __float_as_uint(xa * __fdividef(1.0f, 1.0f + __expf(-xa)));
              rb[j] = __float_as_uint(xb * __fdividef(1.0f, 1.0f + __expf(-xb)));
            }
            if (n < 2 * p.e) {
              pack64(ra, rb, [](float x, int) { return x; }, w);
              uint8_t *b = st.begin();
              st.put(b, w);
              st.finish(b, &tmC1, n - p.e, row0);
            } else {
              const int c = n - 2 * p.e;  // column inside Z
              float4 *zr = reinterpret_cast<float4 *>(p.zf + (size_t)(row0 + lane) * p.s + c);
#pragma unroll
              for (int q = 0; q < 8; ++q) {  // columns 4q.. from ra, 32 + 4q.. from rb
                zr[q] = make_float4(__uint_as_float(ra[4 * q]), __uint_as_float(ra[4 * q + 1]),
                                    __uint_as_float(ra[4 * q + 2]), __uint_as_float(ra[4 * q + 3]));
                zr[8 + q] = make_float4(__uint_as_float(rb[4 * q]), __uint_as_float(rb[4 * q + 1]),
                                        __uint_as_float(rb[4 * q + 2]), __uint_as_float(rb[4 * q + 3]));
              }
#pragma unroll 1
              for (int h = 0; h < 4; ++h) {
                const float *g = p.gamma + h * p.s + c;
                const float *be = p.beta + h * p.s + c;
                pack64(ra, rb, [&](float z, int col) { return fmaf(z, __ldg(g + col), __ldg(be + col)); },
                       w);
                uint8_t *b = st.begin();
                st.put(b, w);
                st.finish(b, &tmC2, c, h * p.M_tokens + row0);
              }
            }
          }
        } else if constexpr (EPI == EPI_STORE) {
          uint4 w[8];
          if (p.residual) {
            // the block's shortcut: this thread's row, 64 columns of X
            const uint4 *xr = reinterpret_cast<const uint4 *>(
                p.residual + (size_t)(row0 + lane) * p.N + n0 + c0);
            uint4 xv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) xv[q] = __ldg(xr + q);
            const __nv_bfloat16 *xh = reinterpret_cast<const __nv_bfloat16 *>(xv);
            pack64(ra, rb, [&](float x, int col) { return x + __bfloat162float(xh[col]); }, w);
          } else {
            pack64(ra, rb, [](float x, int) { return x; }, w);
          }
          uint8_t *b = st.begin();
          st.put(b, w);
          st.finish(b, &tmC0, n0 + c0, row0);
        } else {
          const int n = n0 + c0;
          if (n < 2 * p.e) {
            uint4 w[8];
            pack64(ra, rb, [](float x, int) { return swish_tanh(x); }, w);
            uint8_t *b = st.begin();
            st.put(b, w);
            // V is read by the chunk-state and the attention kernels: kept in
            // L2 ahead of U, which only the attention reads
            if (n < p.e) st.finish(b, &tmC0, n, row0);
            else st.finish(b, &tmC1, 0, (int)rb64_row(row0, n - p.e, p.e / 64), true);
          } else {
            const int c = n - 2 * p.e;  // column inside Z
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              ra[j] = __float_as_uint(swish_tanh(__uint_as_float(ra[j])));
              rb[j] = __float_as_uint(swish_tanh(__uint_as_float(rb[j])));
            }
            if constexpr (EPI == EPI_PROJ_ROPE) {
              // flash_block RoPE: the (even, odd) column pairs of this row
              // rotated by the table's (cos, sin) at its position; the 32
              // pairs' entries, one coalesced load each, stay packed
              uint32_t csn[32];
              {
                const uint32_t *tab =
                    p.rope_cs + (size_t)(c / 2) * p.T_seq + (row0 + lane) % p.T_seq;
#pragma unroll
                for (int k = 0; k < 32; ++k) csn[k] = __ldg(tab + (size_t)k * p.T_seq);
              }
#pragma unroll 1
              for (int h = 0; h < 4; ++h) {
                const float *g = p.gamma + h * p.s + c;
                const float *be = p.beta + h * p.s + c;
                uint8_t *b = st.begin();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                  const uint32_t *src = hf == 0 ? ra : rb;  // columns 32 hf .. 32 hf + 31
                  uint4 w4[4];
                  uint32_t *wp = reinterpret_cast<uint32_t *>(w4);  // word k: pair 16 hf + k
#pragma unroll
                  for (int k2 = 0; k2 < 8; ++k2) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                      const int k = 2 * k2 + j, col = 32 * hf + 2 * k;
                      const float2 q = __half22float2(
                          *reinterpret_cast<const __half2 *>(&csn[16 * hf + k]));
                      const float cs = q.x, sn = q.y;
                      const float y0 = fmaf(__uint_as_float(src[2 * k]), __ldg(g + col), __ldg(be + col));
                      const float y1 = fmaf(__uint_as_float(src[2 * k + 1]), __ldg(g + col + 1),
                                            __ldg(be + col + 1));
                      wp[k] = pack_bf16(y0 * cs - y1 * sn, y0 * sn + y1 * cs);
                    }
                  }
#pragma unroll
                  for (int cc = 0; cc < 4; ++cc)
                    *reinterpret_cast<uint4 *>(b + sw128_offset(lane, 4 * hf + cc)) = w4[cc];
                }
                st.finish(b, &tmC2, c, h * p.M_tokens + row0);
              }
            } else {
#pragma unroll 1
              for (int h = 0; h < 4; ++h) {
                const float *g = p.gamma + h * p.s + c;
                const float *be = p.beta + h * p.s + c;
                uint4 w[8];
                pack64(ra, rb, [&](float z, int col) { return fmaf(z, __ldg(g + col), __ldg(be + col)); },
                       w);
                uint8_t *b = st.begin();
                st.put(b, w);
                st.finish(b, &tmC2, c, h * p.M_tokens + row0);
              }
            }
          }
        }
      }
    }
    st.drain();
    }
  }

  tc_fence_before();
  // neither CTA exits while its peer may still signal its barriers
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int EPI, bool B_KM = false, bool TAIL = false>
cudaError_t launch(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &c0,
                   const CUtensorMap &c1, const CUtensorMap &c2, const Params &p,
                   const Problem &pr) {
  // plain products may carry a tail of 128-column tiles (plan_tiles)
  if constexpr (!TAIL && (EPI == EPI_STORE || EPI == EPI_GATE_GRAD)) {
    if (p.t_split < p.total) return launch<EPI, B_KM, true>(tmA, tmB, c0, c1, c2, p, pr);
  }
  // per device: shared-memory attribute set, and how many pairs fit at once
  static int max_pairs[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kernel = tc_gemm_pair_kernel<EPI, B_KM, TAIL>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = Layout<EPI>::smem_bytes;
  cfg.stream = pr.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (max_pairs[dev] == 0) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Layout<EPI>::smem_bytes);
    if (err != cudaSuccess) return err;
    int n = 0;
    cfg.gridDim = dim3(2 * (pr.num_sms / 2));
    err = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (err != cudaSuccess) return err;
    max_pairs[dev] = n > 0 ? n : 1;
  }
  const int pairs = p.total < max_pairs[dev] ? p.total : max_pairs[dev];
  cfg.gridDim = dim3(2 * pairs);
  return cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, c0, c1, c2, p);
}

// The tile plan of a launch: bn-column tiles (256 or 128) for the first
// rp_split row pairs, 128-column tiles for the rest, chosen to minimise the
// busiest pair's work when tile t goes to pair t % pairs.  A 128-column
// tile counts about 0.6 of a 256-column one: it reads the same A block, and
// the mainloop is bound by shared-memory traffic rather than by the MMAs
// (measured on the output projection, 256 rows a pair, 768 columns, 1536
// deep).  So a last, partial round of 256-column tiles is cut into twice
// as many 128-column ones when they fit one round, or every tile is 128
// wide when that fills the rounds better.  Plain products only: the
// projection's epilogue makes its narrow tiles dearer (a 128-column tail
// measured slower there), so it keeps 256-column tiles.
struct Plan {
  int bn;
  int rp_split;
};

double plan_makespan(int row_pairs, int N, int pairs, int bn, int rp_split,
                     std::vector<double> &load) {
  load.assign(pairs, 0.0);
  long long t = 0;
  auto add = [&](int w, int rows) {
    for (int r = 0; r < rows; ++r)
      for (int n0 = 0; n0 < N; n0 += w, ++t) load[t % pairs] += (N - n0 >= BN) && w == BN ? 1.0 : 0.6;
  };
  add(bn, rp_split);
  add(BN / 2, row_pairs - rp_split);
  double m = 0.0;
  for (double v : load) m = v > m ? v : m;
  return m;
}

Plan plan_tiles(long long M, int N, int num_sms) {
  const int row_pairs = (int)((M / BM + 1) / 2), pairs = num_sms / 2 > 0 ? num_sms / 2 : 1;
  Plan best = {BN, row_pairs};
  if (N % (BN / 2) != 0) return best;
  const int n256 = (N + BN - 1) / BN, n128 = N / (BN / 2);
  // large launches: the last round is a small part of the work
  if ((long long)row_pairs * n256 > 16LL * pairs) return best;
  thread_local struct {
    long long M;
    int N, sms;
    Plan plan;
  } cache[8];
  thread_local int next = 0;
  for (const auto &c : cache)
    if (c.M == M && c.N == N && c.sms == num_sms) return c.plan;
  std::vector<double> load;
  double cost = plan_makespan(row_pairs, N, pairs, BN, row_pairs, load);
  auto consider = [&](int bn, int rp_split) {
    const double c = plan_makespan(row_pairs, N, pairs, bn, rp_split, load);
    if (c < cost - 1e-9) {
      cost = c;
      best = {bn, rp_split};
    }
  };
  consider(BN / 2, row_pairs);
  // a tail of row pairs in 128-column tiles, at most two rounds of them
  for (int k = 1; k <= row_pairs && (long long)k * n128 <= 2LL * pairs; ++k)
    consider(BN, row_pairs - k);
  cache[next] = {M, N, num_sms, best};
  next = (next + 1) % 8;
  return best;
}

Params base_params(const Problem &pr, int N, int K, Plan plan = {BN, 1 << 30}) {
  Params p = {};
  p.N = N;
  p.K = K;
  p.bn = plan.bn;
  p.m_tiles = (int)(pr.M / BM);
  const int row_pairs = (p.m_tiles + 1) / 2;
  p.n_tiles = (N + plan.bn - 1) / plan.bn;
  p.rp_split = plan.rp_split < row_pairs ? plan.rp_split : row_pairs;
  p.n_tiles2 = (N + BN / 2 - 1) / (BN / 2);
  p.t_split = p.rp_split * p.n_tiles;
  p.total = p.t_split + (row_pairs - p.rp_split) * p.n_tiles2;
  p.status = pr.status;
  p.M_tokens = (int)pr.M;
  p.e = pr.e;
  p.s = pr.s;
  return p;
}

}  // namespace

cudaError_t tc_projection_bf16(const Problem &pr) {
  const int N = 2 * pr.e + pr.s;
  CUtensorMap tmA, tmB, tU, tV, tH;
  cudaError_t err;
  // A: the input, or its normalised copy (flash_block pre-norm)
  if ((err = make_tmap_bf16_2d(&tmA, pr.A_in, pr.M, pr.d, pr.d, BM, 64)) != cudaSuccess)
    return err;
  if ((err = make_tmap_bf16_2d(&tmB, pr.W_uvz, pr.d, N, N, BK, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tU, pr.U, pr.M, pr.e, pr.e, 32, 64)) != cudaSuccess) return err;
  // V in 64 x 64 blocks (flat 128-byte rows), 32-row store boxes
  if ((err = make_tmap_bf16_2d(&tV, pr.V, pr.M * pr.e / 64, 64, 64, 32, 64)) != cudaSuccess)
    return err;
  if ((err = make_tmap_bf16_2d(&tH, pr.heads, 4 * pr.M, pr.s, pr.s, 32, 64)) != cudaSuccess)
    return err;
  Params p = base_params(pr, N, pr.d);
  p.gamma = pr.gamma;
  p.beta = pr.beta;
  p.sched = pr.status;
  p.T_seq = pr.T;
  p.rope_cs = (const uint32_t *)pr.rope_cs;
  p.relpos = pr.relpos;
  p.bias = pr.bias;
  p.C = pr.C;
  p.causal = pr.causal;
  if (pr.rope) return launch<EPI_PROJ_ROPE>(tmA, tmB, tU, tV, tH, p, pr);
  return launch<EPI_PROJ>(tmA, tmB, tU, tV, tH, p, pr);
}

cudaError_t pair_gemm_bf16(const void *A, const void *B, int b_km, void *C, int M, int N, int K,
                           int *status, int num_sms, cudaStream_t stream) {
  if (M % BM != 0 || N % (2 * 64) != 0 || K % BK != 0) return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB, tC;
  cudaError_t err;
  if ((err = make_tmap_bf16_2d(&tmA, A, M, K, K, BM, 64)) != cudaSuccess) return err;
  if (b_km) err = make_tmap_bf16_2d(&tmB, B, N, K, K, BN / 2, 64);
  else err = make_tmap_bf16_2d(&tmB, B, K, N, N, BK, 64);
  if (err != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tC, C, M, N, N, 32, 64)) != cudaSuccess) return err;
  Problem pr = {};
  pr.M = M;
  pr.status = status;
  pr.stream = stream;
  pr.num_sms = num_sms;
  const Params p = base_params(pr, N, K, plan_tiles(M, N, num_sms));
  if (b_km) return launch<EPI_STORE, true>(tmA, tmB, tC, tC, tC, p, pr);
  return launch<EPI_STORE>(tmA, tmB, tC, tC, tC, p, pr);
}

cudaError_t pair_gate_grad_bf16(const void *dO, const void *W_o, void *pre, const void *Vh,
                                void *dVh, int M, int e, int s, int d, int *status, int num_sms,
                                cudaStream_t stream) {
  const int N = 2 * e + s;  // Pre's row: U, V, Z
  if (M % BM != 0 || e % (2 * 64) != 0 || d % BK != 0) return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB, tD, tX, tV;
  cudaError_t err;
  if ((err = make_tmap_bf16_2d(&tmA, dO, M, d, d, BM, 64)) != cudaSuccess) return err;
  // B = W_o^T: the stored [e, d] W_o read K-major
  if ((err = make_tmap_bf16_2d(&tmB, W_o, e, d, d, BN / 2, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tD, dVh, M, e, e, 32, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tX, pre, M, e, N, 32, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tV, Vh, M, e, e, 32, 64)) != cudaSuccess) return err;
  Problem pr = {};
  pr.M = M;
  pr.status = status;
  pr.stream = stream;
  pr.num_sms = num_sms;
  const Params p = base_params(pr, e, d, plan_tiles(M, e, num_sms));
  return launch<EPI_GATE_GRAD, true>(tmA, tmB, tD, tX, tV, p, pr);
}

cudaError_t pair_recompute_bf16(const void *X, const void *W_uvz, const float *gamma,
                                const float *beta, void *pre, void *V_io, float *Z, void *H_io,
                                int M, int d, int e, int s, int *status, int num_sms,
                                cudaStream_t stream) {
  const int N = 2 * e + s;
  if (M % BM != 0 || e % BN != 0 || s != 128 || d % BK != 0) return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB, tP, tV, tH;
  cudaError_t err;
  if ((err = make_tmap_bf16_2d(&tmA, X, M, d, d, BM, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tmB, W_uvz, d, N, N, BK, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tP, pre, M, N, N, 32, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tV, V_io, M, e, e, 32, 64)) != cudaSuccess) return err;
  if ((err = make_tmap_bf16_2d(&tH, H_io, 4LL * M, s, s, 32, 64)) != cudaSuccess) return err;
  Problem pr = {};
  pr.M = M;
  pr.e = e;
  pr.s = s;
  pr.status = status;
  pr.stream = stream;
  pr.num_sms = num_sms;
  Params p = base_params(pr, N, d);
  p.gamma = gamma;
  p.beta = beta;
  p.zf = Z;
  return launch<EPI_RECOMPUTE>(tmA, tmB, tP, tV, tH, p, pr);
}

cudaError_t tc_output_bf16(const Problem &pr) {
  CUtensorMap tmA, tmB, tO;
  cudaError_t err;
  if ((err = make_tmap_bf16_2d(&tmA, pr.gated, pr.M, pr.e, pr.e, BM, 64)) != cudaSuccess)
    return err;
  if ((err = make_tmap_bf16_2d(&tmB, pr.W_o, pr.e, pr.d, pr.d, BK, 64)) != cudaSuccess)
    return err;
  if ((err = make_tmap_bf16_2d(&tO, pr.out, pr.M, pr.d, pr.d, 32, 64)) != cudaSuccess) return err;
  Params p = base_params(pr, pr.d, pr.e, plan_tiles(pr.M, pr.d, pr.num_sms));
  p.residual = (const __nv_bfloat16 *)pr.residual;
  return launch<EPI_STORE>(tmA, tmB, tO, tO, tO, p, pr);
}

}  // namespace flashgau
